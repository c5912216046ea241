"""Seeded synthetic workloads for the speculative-tree hot path.

This module is the one piece shared by the CUDA path's tests/bench and the CPU
oracle's tests: it draws random logits and uniforms and nothing else.  It holds
none of the method's arithmetic (no truncation, softmax, expansion, ranking or
verification).

Workload recipe (the pages publish no generator; this stands in for the draft /
target logits of an EAGLE-3 style drafter and its target model at vocab sizes
32K-152K):

* latent logits of a row:  l[v] = -a * ln(rank(v)) + N(0, noise_sd), where
  rank is a uniformly random permutation of 1..V (argsort of iid uniforms).
* draft row = latent row + N(0, sigma_draft), cast to the storage dtype.
* draft row e of tree b is the e-th expanded node in expansion order; its
  content is keyed by (tree, slot), not by the node's token path.
* target row of pruned node i = the latent row of its expansion slot when the
  node was expanded (root = slot 0), else a fresh latent row keyed by (tree, i).
* uniforms are U[0, 1) float32.

Presets mirror the five workloads of the RheoSampling / SMART notes:
tiny brute force (V=32, fp32), Vicuna-like (V=32000), LLaMA-3-vocab
(V=128256), RL-rollout large batch (V=151936) and the batch sweep with the
SMART builder.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    V: int
    dtype: str            # "bf16" | "f32"
    K: int
    m: int
    W: int
    depth: int
    R: int
    temperature: float
    zipf_a: float
    sigma_draft: float
    builder: str = "topr"   # "topr" | "smart"
    support: int = 128
    noise_sd: float = 0.5
    # SMART cost model (units of one target step)
    lam: float = 0.02
    beta: float = 0.0
    gamma: float = 0.5
    delta: float = 0.01
    rho: float = 1.3
    eta: float = 0.0
    alpha: float = 1.0
    verify_order: str = "rheo"  # "rheo" (probe first) | "rrsw" (probe last)

    @property
    def n_exp(self) -> int:
        """Expanded rows a tree consumes (top-R builder) / needs at most (SMART)."""
        if self.builder == "smart":
            return self.R + 1
        return 1 + (self.depth - 1) * self.W

    @property
    def n_cand(self) -> int:
        return self.K + (self.depth - 1) * self.W * self.K

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, V=32, dtype="f32", K=4, m=1, W=4, depth=3, R=8,
                     temperature=1.0, zipf_a=1.2, sigma_draft=1.0),
    "vicuna": Workload("vicuna", B=1, V=32000, dtype="bf16", K=8, m=1, W=8, depth=8, R=60,
                       temperature=1.0, zipf_a=1.2, sigma_draft=1.0),
    "llama3": Workload("llama3", B=8, V=128256, dtype="bf16", K=8, m=1, W=8, depth=8, R=60,
                       temperature=1.0, zipf_a=1.2, sigma_draft=0.8),
    "rl": Workload("rl", B=64, V=151936, dtype="bf16", K=6, m=1, W=6, depth=6, R=32,
                   temperature=0.7, zipf_a=1.0, sigma_draft=1.2),
    "sweep_smart": Workload("sweep_smart", B=64, V=128256, dtype="bf16", K=8, m=1, W=8, depth=8,
                            R=60, temperature=1.0, zipf_a=1.2, sigma_draft=1.0, builder="smart"),
}

# The throughput workload: LLaMA-3-vocab trees at batch 64.
BENCH_WORKLOAD = WORKLOADS["llama3"].with_(name="llama3_b64", B=64)


def _seed_of(*parts) -> int:
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 62) - 1)


def _gen(seed_parts, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed_of(*seed_parts))
    return g


def latent_rows(seed_parts: Sequence, n: int, V: int, a: float, noise_sd: float,
                device="cpu", chunk: int = 64) -> torch.Tensor:
    """[n][V] float32 latent logits -a*ln(rank) + N(0, noise_sd) over random ranks."""
    g = _gen(("latent",) + tuple(seed_parts), device)
    out = torch.empty((n, V), dtype=torch.float32, device=device)
    base = -a * torch.log(torch.arange(1, V + 1, dtype=torch.float32, device=device))
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        perm = torch.argsort(torch.rand((e - s, V), generator=g, device=device), dim=1)
        noise = torch.randn((e - s, V), generator=g, device=device) * noise_sd
        out[s:e] = base[perm] + noise
    return out


def cast_rows(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(dtype)


def draft_logits(wl: Workload, seed: int, n_rows: Optional[int] = None, device="cpu",
                 row_stride: Optional[int] = None, trees: Optional[Sequence[int]] = None):
    """Draft logits [B][n_rows][row_stride] (storage dtype) and latent rows [B][n_rows][V] fp32.

    Tree b's rows are keyed by (seed, b), so any subset `trees` of the batch
    can be generated alone (the result then has len(trees) trees).  Padding
    columns (row_stride > V) are filled with -inf; they are never read by a
    caller that passes V correctly.
    """
    n_rows = n_rows or wl.n_exp
    stride = row_stride or wl.V
    ids = list(range(wl.B)) if trees is None else list(trees)
    lat = torch.empty((len(ids), n_rows, wl.V), dtype=torch.float32, device=device)
    drf = torch.full((len(ids), n_rows, stride), float("-inf"),
                     dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32, device=device)
    for i, b in enumerate(ids):
        lat[i] = latent_rows((seed, "tree", b), n_rows, wl.V, wl.zipf_a, wl.noise_sd, device)
        g = _gen(("draftnoise", seed, b), device)
        noise = torch.randn((n_rows, wl.V), generator=g, device=device) * wl.sigma_draft
        drf[i, :, :wl.V] = cast_rows(lat[i] + noise, wl.dtype)
    return drf, lat


def uniforms(seed: int, tag: str, shape, device="cpu") -> torch.Tensor:
    g = _gen(("uniform", seed, tag), device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def build_uniforms(wl: Workload, seed: int, n_rows: Optional[int] = None, device="cpu"):
    return uniforms(seed, "probe", (wl.B, n_rows or wl.n_exp), device)


def verify_uniforms(wl: Workload, seed: int, device="cpu"):
    return (uniforms(seed, "verify", (wl.B, wl.depth, wl.K), device),
            uniforms(seed, "bonus", (wl.B,), device))


def target_logits(wl: Workload, seed: int, latent: torch.Tensor, node_exp_row: torch.Tensor,
                  n_nodes=None, device="cpu", row_stride: Optional[int] = None,
                  trees: Optional[Sequence[int]] = None):
    """Target logits [B][R+1][row_stride] for a built tree.

    node_exp_row[i][j] >= 0 gives the latent slot of an expanded node; other
    nodes (and unused entries) get a fresh latent row keyed by (tree, node).
    `trees` names the batch indices of the rows of `latent` / `node_exp_row`.
    """
    stride = row_stride or wl.V
    max_nodes = node_exp_row.shape[1]
    ids = list(range(node_exp_row.shape[0])) if trees is None else list(trees)
    out = torch.full((len(ids), max_nodes, stride), float("-inf"),
                     dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32, device=device)
    exp_row = node_exp_row.to("cpu")
    for i, b in enumerate(ids):
        rows = latent_rows((seed, "fresh", b), max_nodes, wl.V, wl.zipf_a, wl.noise_sd, device)
        sel = [(j, int(exp_row[i, j])) for j in range(max_nodes) if int(exp_row[i, j]) >= 0]
        if sel:
            dst = torch.tensor([j for j, _ in sel], device=device)
            src = torch.tensor([e for _, e in sel], device=latent.device)
            rows[dst] = latent[i].index_select(0, src).to(device)
        out[i, :, :wl.V] = cast_rows(rows, wl.dtype)
    return out


def path_keyed_rows(seed: int, paths: Sequence[tuple], V: int, a: float, noise_sd: float,
                    dtype: str = "f32") -> torch.Tensor:
    """One latent row per token path (a tuple of token ids), keyed by hash(seed, path).

    Used for losslessness checks: the target distribution of a node depends only
    on the tokens on its path, as for a real autoregressive target model.
    """
    rows = torch.empty((len(paths), V), dtype=torch.float32)
    for i, path in enumerate(paths):
        rows[i] = latent_rows((seed, "path") + tuple(int(t) for t in path), 1, V, a, noise_sd)[0]
    return cast_rows(rows, dtype)


def path_keyed_draft(seed: int, paths: Sequence[tuple], V: int, a: float, noise_sd: float,
                     sigma: float, dtype: str = "f32") -> torch.Tensor:
    """Draft rows correlated with path_keyed_rows (same latent + N(0, sigma))."""
    lat = path_keyed_rows(seed, paths, V, a, noise_sd, "f32")
    out = torch.empty_like(lat)
    for i, path in enumerate(paths):
        g = _gen(("pathnoise", seed) + tuple(int(t) for t in path), "cpu")
        out[i] = lat[i] + torch.randn((V,), generator=g) * sigma
    return cast_rows(out, dtype)


def bf16_bits(x: torch.Tensor):
    """uint16 numpy view of a bf16 tensor (exact bits, for the oracle)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def to_numpy_f64(x: torch.Tensor):
    """Exact float64 copy of a bf16/f32 tensor."""
    return x.detach().to("cpu").to(torch.float64).numpy()


def profile_timings(seed: int, sizes: Sequence[float], t_base: float = 1.0e-3, draft_per_token: float = 2.0e-5,
                    slope: float = 2.0e-3, knee: float = 96.0, curvature: float = 6.0e-5, noise: float = 0.02):
    """Synthetic profiled step times (seconds) of a device, standing in for timed model forward passes.

    A plain target step takes t_base; drafting a tree of n tokens takes about
    draft_per_token * n; verifying it takes t_base * (1 + slope * n +
    curvature * max(0, n - knee)^2): nearly flat while the target pass is
    memory-bound, growing faster past a compute knee.  Each time carries
    relative Gaussian noise of the given size.  Returns (t_draft, t_verify)
    as float64 numpy arrays.
    """
    rng = np.random.default_rng(_seed_of("profile", seed))
    n = np.asarray(sizes, dtype=np.float64)
    t_draft = draft_per_token * n * (1.0 + noise * rng.standard_normal(n.shape))
    t_verify = t_base * (1.0 + slope * n + curvature * np.maximum(0.0, n - knee) ** 2)
    t_verify = t_verify * (1.0 + noise * rng.standard_normal(n.shape))
    return np.maximum(t_draft, 0.0), np.maximum(t_verify, 0.0)
