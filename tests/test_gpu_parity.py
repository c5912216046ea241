"""CUDA path vs the CPU oracle, element by element, on seeded synthetic inputs.

Every call goes through the C ABI (libspec_tree.so) via the ctypes binding.
"""
import numpy as np
import pytest
import torch

from dynamic_tree_speculative_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

import parity  # noqa: E402  (loads the native library; fails loudly if absent)


def _report(name, out, replays_allowed=True):
    """Print the counts; where no near-tie replay is expected, fail with them."""
    msg = (f"{name}: build {out['build_exact']} equal, {out['build_replayed']} with adopted near-ties; "
           f"verify {out['verify_exact']} equal, {out['verify_replayed']} with adopted near-ties; "
           f"decisions {out['adopted'][:8]}")
    print(msg)
    if not replays_allowed:
        assert not out["adopted"], msg


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_parity(seed):
    wl = WL.WORKLOADS["tiny"].with_(B=256)
    out = parity.run_parity(wl, seed)
    _report("tiny", out)


@pytest.mark.parametrize("seed", [0, 1])
def test_vicuna_parity(seed):
    wl = WL.WORKLOADS["vicuna"].with_(B=4)
    _report("vicuna", parity.run_parity(wl, seed))


def test_llama3_parity():
    """LLaMA-3-vocab workload at its own batch (8 trees, V = 128256), every tree."""
    wl = WL.WORKLOADS["llama3"]
    _report("llama3", parity.run_parity(wl, 3))


def _full_batch(name, wl, seed, max_bonus):
    """Every tree of a full-size batch: the trees equal without any adopted decision; in verification
    only bonus draws may be near-ties.  A bonus draw over the whole vocabulary lands within 1e-6 of
    mass of a CDF boundary whenever it falls among tail tokens of probability ~1e-6, and the float32
    sums then decide some of them the other way; the oracle adopts the GPU's token there and the
    rest of the tree is compared as usual."""
    out = parity.run_parity(wl, seed)
    _report(name, out)
    assert out["build_exact"] == wl.B, out["adopted"]
    assert all(a[1] == "bonus" for a in out["adopted"]) and len(out["adopted"]) <= max_bonus, out["adopted"]


def test_rl_large_batch_every_tree():
    """RL-rollout workload at full size (64 trees, V = 151936, T = 0.7), every tree against the oracle
    (this seed: one bonus near-tie, tree 33)."""
    _full_batch("rl", WL.WORKLOADS["rl"], 4, 2)


def test_bench_workload_every_tree():
    """The timed workload (LLaMA-3 vocab, 64 trees) in the bench's launch configuration, every tree
    against the oracle (this seed: two bonus near-ties, trees 16 and 62)."""
    _full_batch("bench", WL.BENCH_WORKLOAD, 5, 3)


@pytest.mark.parametrize("builder", ["topr", "smart"])
def test_sweep_one_tree(builder):
    """The batch sweep's smallest batch (one tree: one row per select CTA, one verify cluster of 8 CTAs
    of 1024 threads), build and verify against the oracle."""
    base = WL.WORKLOADS["sweep_smart"] if builder == "smart" else WL.BENCH_WORKLOAD
    _report(f"sweep_{builder}_b1", parity.run_parity(base.with_(B=1), 31))


class _Trees:
    """Host copies of some trees of a device batch, indexed like the batch."""

    def __init__(self, x, idx):
        self.rows = {b: x[b].cpu() for b in idx}

    def __getitem__(self, k):
        if isinstance(k, tuple):
            return self.rows[k[0]][k[1:]]
        return self.rows[k]


@pytest.mark.parametrize("builder", ["topr", "smart"])
def test_sweep_256_trees_build_sampled(builder):
    """The batch sweep's largest batch (256 trees, 48 draft rows per select CTA handed out on demand),
    in the bench's launch configuration: inputs generated on the device, sampled trees' builds against
    the oracle on host copies of their rows."""
    from dynamic_tree_speculative_gb300 import binding as B
    base = WL.WORKLOADS["sweep_smart"] if builder == "smart" else WL.BENCH_WORKLOAD
    wl = base.with_(B=256)
    params = B.Params.from_workload(wl)
    n_rows = B.rows_needed(params)
    draft, _ = WL.draft_logits(wl, 41, n_rows=n_rows, device="cuda")
    u = WL.build_uniforms(wl, 41, n_rows=n_rows, device="cuda")
    tree = B.TreeBuffers(params, wl.B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.spec_tree_build(params, wl.V, draft, u, tree, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sample = [0, 85, 170, 255]
    case = parity.Case(wl, _Trees(draft, sample), None, _Trees(u, sample), None, None, wl.V)
    g = {k: getattr(tree, k).cpu().numpy() for k in (
        "node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "node_score",
        "n_nodes", "sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")}
    del draft
    out = parity.compare_case(g, case, sample)
    _report(f"sweep_{builder}_b256", out)
    assert out["build_exact"] + out["build_replayed"] == len(sample)


@pytest.mark.parametrize("seed", [0, 1])
def test_smart_parity(seed):
    wl = WL.WORKLOADS["sweep_smart"].with_(B=6, V=32000)
    _report("smart", parity.run_parity(wl, seed))


def test_smart_parity_with_fitted_costs():
    """SMART trees whose cost coefficients come from spec_tree_smart_fit on profiled step times."""
    from dynamic_tree_speculative_gb300 import binding as B
    sizes = [16, 64, 128, 256, 384]
    td, tv = WL.profile_timings(7, sizes)
    f = B.spec_tree_smart_fit(sizes, td, tv, 1.0e-3)
    wl = WL.WORKLOADS["sweep_smart"].with_(B=8, V=32000, lam=f.lam, beta=0.0, gamma=f.gamma, delta=f.delta,
                                           rho=f.rho, eta=0.0)
    out = parity.run_parity(wl, 13)
    sizes_built = out["gpu"]["n_nodes"] - 1
    print(f"fitted lam {f.lam:.4g} gamma {f.gamma:.4g} delta {f.delta:.4g} rho {f.rho:.4g}; "
          f"tree sizes {sizes_built.tolist()}")
    _report("smart_fitted", out)


def test_smart_parity_llama_vocab():
    wl = WL.WORKLOADS["sweep_smart"].with_(B=4)
    _report("smart128k", parity.run_parity(wl, 9))


EDGE = {
    "support_is_V": dict(V=100, K=8, m=1, W=4, depth=4, R=12, stride=104),
    "ragged_V": dict(V=1001, K=8, m=1, W=4, depth=4, R=20, stride=1008),
    "tiny_V_no_vector": dict(V=5, K=2, m=1, W=2, depth=3, R=6, stride=8),
    "f32_ragged": dict(V=4099, K=6, m=1, W=3, depth=3, R=10, dtype="f32", stride=4100),
    "m0": dict(V=3000, K=4, m=0, W=4, depth=4, R=16),
    "m2": dict(V=3000, K=6, m=2, W=3, depth=4, R=16),
    "m3": dict(V=3000, K=6, m=3, W=3, depth=4, R=16),
    "cold": dict(V=3000, K=6, m=1, W=3, depth=4, R=16, temperature=0.5),
    "hot": dict(V=3000, K=6, m=1, W=3, depth=4, R=16, temperature=1.7),
    "R1": dict(V=3000, K=4, m=1, W=2, depth=3, R=1),
    "R_over_all": dict(V=3000, K=4, m=1, W=3, depth=4, R=200),
    "depth1": dict(V=3000, K=8, m=1, W=8, depth=1, R=8),
    "support_32": dict(V=3000, K=4, m=1, W=3, depth=3, R=10, support=32),
    "wide": dict(V=9000, K=16, m=1, W=16, depth=3, R=100),
    # the pages' Top-K baseline: every child deterministic, no probe
    "topk_m_eq_K": dict(V=3000, K=4, m=4, W=4, depth=4, R=16),
    # probe-last verification (the pages' "Rheo + RRSw" ablation), with and without fillers
    "rrsw": dict(V=3000, K=4, m=1, W=4, depth=4, R=16, verify_order="rrsw"),
    "rrsw_no_fillers": dict(V=3000, K=2, m=1, W=2, depth=5, R=14, verify_order="rrsw"),
    "rrsw_m0": dict(V=3000, K=3, m=0, W=3, depth=4, R=14, verify_order="rrsw"),
    # the pages' support-size ablation (one CTA per row past 128 tokens)
    "support_256": dict(V=32000, K=8, m=1, W=4, depth=4, R=20, support=256),
    "support_512": dict(V=32000, K=8, m=1, W=4, depth=4, R=20, support=512),
    "support_1024": dict(V=32000, K=8, m=1, W=4, depth=4, R=20, support=1024),
    "support_1024_m0": dict(V=9000, K=4, m=0, W=4, depth=4, R=16, support=1024),
    "support_1024_rrsw": dict(V=9000, K=2, m=1, W=2, depth=5, R=14, support=1024, verify_order="rrsw"),
    "support_1024_f32": dict(V=5003, K=6, m=1, W=3, depth=3, R=10, dtype="f32", stride=5004, support=1024),
    "support_300_ragged": dict(V=4097, K=6, m=2, W=3, depth=3, R=12, stride=4104, support=300),
    # support >= V: the dense support of a small vocabulary
    "dense_small_vocab": dict(V=700, K=8, m=1, W=4, depth=4, R=20, stride=704, support=1024),
    # the cold limit: m = 0 reduces to Top-K (its tail starts at the top token, so
    # its tempered weight never underflows); m = 1 keeps its proxy, at a temperature
    # above the float32 underflow of exp((l_2 - l_1) / T) for these rows
    "cold_m0": dict(V=3000, K=4, m=0, W=4, depth=4, R=16, temperature=0.02),
    "cold_m1": dict(V=3000, K=4, m=1, W=4, depth=4, R=16, temperature=0.1),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name):
    kw = dict(EDGE[name])
    stride = kw.pop("stride", None)
    base = WL.WORKLOADS["vicuna"].with_(B=16)
    wl = base.with_(**kw)
    _report(name, parity.run_parity(wl, 11, row_stride=stride))


DENSE = 0x40000000  # support = the whole vocabulary (SPEC_TREE_SUPPORT_DENSE)

DENSE_CASES = {
    # the pages' "full dense" support at the pages' vocabularies
    "vicuna": dict(B=4),
    "m0": dict(B=6, V=20000, K=4, m=0, W=4, depth=4, R=16),
    "m2": dict(B=6, V=20000, K=6, m=2, W=3, depth=4, R=16),
    "probe_last_no_fillers": dict(B=8, V=20000, K=2, m=1, W=2, depth=5, R=14, verify_order="rrsw"),
    "probe_last": dict(B=6, V=20000, K=4, m=1, W=4, depth=4, R=16, verify_order="rrsw"),
    "f32_ragged": dict(B=4, V=5003, K=6, m=1, W=3, depth=3, R=10, dtype="f32", stride=5004),
    "bf16_ragged": dict(B=4, V=4099, K=6, m=1, W=3, depth=3, R=10, stride=4104),
    "cold": dict(B=6, V=20000, K=6, m=1, W=3, depth=4, R=16, temperature=0.5),
    "hot": dict(B=6, V=20000, K=6, m=1, W=3, depth=4, R=16, temperature=1.7),
    "topk_m_eq_K": dict(B=4, V=20000, K=4, m=4, W=4, depth=4, R=16),
    "smart": dict(B=6, V=32000, builder="smart"),
}


@pytest.mark.parametrize("name", sorted(DENSE_CASES))
def test_dense_support(name):
    """|S| = V (the support-size ablation's dense row): ranks 0..K-1 and the probe drawn from the whole
    tempered tail in rank order, verification against q~_T over the whole vocabulary."""
    kw = dict(DENSE_CASES[name])
    stride = kw.pop("stride", None)
    wl = WL.WORKLOADS["vicuna"].with_(support=DENSE, **kw)
    out = parity.run_parity(wl, 31, row_stride=stride)
    _report(f"dense_{name}", out)
    # the probes come from deep in the tail too, not only from the first 128 ranks
    pp = out["gpu"]["probe_pos"]
    if name == "vicuna":
        assert (pp >= 128).any(), pp.max()


def test_dense_support_llama_vocab():
    """The dense support at the LLaMA-3 vocabulary (V = 128256), every tree of a small batch."""
    wl = WL.WORKLOADS["llama3"].with_(B=3, support=DENSE)
    _report("dense_llama3", parity.run_parity(wl, 32))


def test_wide_support_llama_vocab():
    """Support 1024 at the LLaMA-3 vocabulary (V = 128256), every tree of a small batch."""
    wl = WL.WORKLOADS["llama3"].with_(B=4, support=1024)
    _report("llama3_support1024", parity.run_parity(wl, 17))


def test_heavy_ties_wide_support():
    """Integer-valued bf16 logits with support 512: ties at the |S|-th key take the smallest ids."""
    wl = WL.WORKLOADS["vicuna"].with_(B=4, V=20000, depth=3, R=12, K=6, W=3, support=512)
    n_rows = 1 + (wl.depth - 1) * wl.W
    g = torch.Generator().manual_seed(6)
    draft = torch.randint(-6, 3, (wl.B, n_rows, wl.V), generator=g).to(torch.bfloat16)
    draft[1] = 0.25
    ex, exm = _parity_on_draft(wl, draft)
    assert ex + exm == wl.B


def _parity_on_draft(wl, draft, seed=0):
    case = parity.make_case(wl, seed)
    case.draft = draft
    case.latent = draft.float()
    trees = parity.oracle_build(case, range(wl.B))
    g = parity.run_gpu(case, None)
    out = parity.compare_case(g, case, range(wl.B), None, trees)
    return out["build_exact"], out["build_replayed"]


def test_heavy_ties_and_constant_rows():
    """Integer-valued bf16 logits (massive ties) and a constant row: ids break ties ascending."""
    wl = WL.WORKLOADS["vicuna"].with_(B=4, V=20000, depth=3, R=12, K=6, W=3)
    n_rows = 1 + (wl.depth - 1) * wl.W
    g = torch.Generator().manual_seed(5)
    draft = torch.randint(-6, 3, (wl.B, n_rows, wl.V), generator=g).to(torch.bfloat16)
    draft[1] = 0.25
    draft[2, :, 5000:] = -3.0  # a long constant tail
    ex, exm = _parity_on_draft(wl, draft)
    assert ex + exm == wl.B


def test_rows_whose_cut_jumps():
    """Rows whose top-|S| cut jumps far from the previous rows' (scaled, shifted, integer-valued and
    constant rows mixed among normal ones), many rows per CTA: a threshold predicted from earlier
    rows is then too high, too low or floods the queue, and the exact path must take over."""
    wl = WL.WORKLOADS["vicuna"].with_(B=64, V=20000)
    case = parity.make_case(wl, 8)
    n_rows = case.draft.shape[1]
    g = torch.Generator().manual_seed(8)
    kind = torch.randint(0, 20, (wl.B, n_rows), generator=g)
    x = case.draft.float()
    scale = torch.ones((wl.B, n_rows))
    shift = torch.zeros((wl.B, n_rows))
    scale[(kind >= 8) & (kind < 11)] = 3.0
    scale[(kind >= 11) & (kind < 14)] = 0.3
    shift[(kind >= 14) & (kind < 16)] = 6.0
    shift[(kind >= 16) & (kind < 18)] = -6.0
    x = x * scale[..., None] + shift[..., None]
    ints = torch.randint(-6, 3, x.shape, generator=g).float()
    x = torch.where((kind == 18)[..., None], ints, x)
    x = torch.where((kind == 19)[..., None], torch.full_like(x, 0.25), x)
    case.draft = x.to(torch.bfloat16)
    sample = list(range(0, wl.B, 4))
    trees = parity.oracle_build(case, sample)
    out = parity.run_gpu(case, None)
    assert out["status"] == 0, out["status"]
    res = parity.compare_case(out, case, sample, None, trees)
    _report("cut jumps", res)


@pytest.mark.parametrize("support,V,stride,B", [(128, 32000, None, 8), (256, 32000, None, 8), (1024, 32000, None, 8),
                                                (256, 32001, 32008, 8), (128, 128256, None, 2)])
def test_cut_hint_from_the_previous_call(support, V, stride, B):
    """The row schedule keeps a cut key of the latest call (of the latest row, for supports above 128)
    as the predicted queue threshold of the next rows.  The second call's rows here differ wildly from
    the first's (scaled by 3, shifted by 5), so the hint lies far below their cut and the exact path must
    take over; a third call on the same rows hits it; a fourth on rows like the first's gets a hint far
    above their cut.  Every call equals the oracle.  A vocabulary that is not a multiple of the vector
    width sends its last elements through their own branch; two trees of the LLaMA-3 vocabulary (114
    rows, no more than SMs) run one CTA per SM with the deep ring."""
    from dynamic_tree_speculative_gb300 import binding
    wl = WL.WORKLOADS["vicuna"].with_(B=B, V=V, support=support)
    params = binding.Params.from_workload(wl)
    tree = binding.TreeBuffers(params, wl.B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i, (scale, shift) in enumerate([(1.0, 0.0), (3.0, 5.0), (3.0, 5.0), (1.0, 0.0)]):
        case = parity.make_case(wl, 70 + i, row_stride=stride)
        case.draft = (case.draft.float() * scale + shift).to(torch.bfloat16)
        binding.spec_tree_build(params, wl.V, case.draft.cuda(), case.u_probe.cuda(), tree, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        hint = int(tree.sched[2].item())
        assert hint != 0  # a cut was kept for the next call
        g = {k: getattr(tree, k).cpu().numpy() for k in (
            "node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "node_score",
            "n_nodes", "sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")}
        out = parity.compare_case(g, case, range(wl.B))
        assert out["build_exact"] + out["build_replayed"] == wl.B


def test_wide_support_queue_path_at_full_size():
    """|S| = 1024 at the LLaMA-3 vocabulary, 64 trees: the first call leaves a cut, so every row of the
    second call (the same rows) takes the predicted-threshold queue path; sampled trees of both calls
    equal the oracle."""
    from dynamic_tree_speculative_gb300 import binding as B
    wl = WL.BENCH_WORKLOAD.with_(support=1024)
    params = B.Params.from_workload(wl)
    tree = B.TreeBuffers(params, wl.B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    case = parity.make_case(wl, 23)
    sample = [0, 21, 42, 63]
    for _ in range(2):
        B.spec_tree_build(params, wl.V, case.draft.cuda(), case.u_probe.cuda(), tree, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert int(tree.sched[2].item()) != 0
        g = {k: getattr(tree, k).cpu().numpy() for k in (
            "node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "node_score",
            "n_nodes", "sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")}
        out = parity.compare_case(g, case, sample)
        assert out["build_exact"] + out["build_replayed"] == len(sample)


def test_queue_path_with_ragged_vocabulary():
    """Many rows per CTA (the predicted-threshold queue path and rows handed out on demand) on a
    vocabulary that is not a multiple of the vector width: the elements past the last whole vector
    join the candidates through their own branch."""
    wl = WL.WORKLOADS["vicuna"].with_(B=64, V=32001)
    out = parity.run_parity(wl, 19, sample=[0, 13, 29, 47, 63], row_stride=32008)
    _report("queue_ragged", out)


def test_verify_reads_target_rows_from_pinned_host_memory():
    """Target logits left in pinned host memory (unified addressing): verify reads the accepted
    path's rows over the host link and returns exactly what it returns from HBM."""
    from dynamic_tree_speculative_gb300 import binding as B
    wl = WL.WORKLOADS["llama3"].with_(B=8)
    case = parity.make_case(wl, 12)
    trees = parity.oracle_build(case, range(wl.B))
    target = parity.target_for(case, trees, 12)
    params = B.Params.from_workload(wl)
    dev = "cuda"
    tree = B.TreeBuffers(params, wl.B, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.spec_tree_build(params, wl.V, case.draft.to(dev), case.u_probe.to(dev), tree, status)
    outs = []
    for tgt in (target.to(dev), target.pin_memory()):
        out = B.VerifyOutputs(params, wl.B, device=dev)
        B.spec_tree_verify(params, wl.V, tgt, tree, case.u_verify.to(dev), case.u_bonus.to(dev), out.accept_len,
                           out.out_tok, out.out_node, out.margins, status)
        torch.cuda.synchronize()
        outs.append([x.cpu() for x in (out.accept_len, out.out_tok, out.out_node)])
    assert int(status.item()) == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_nan_row_sets_status_and_stays_in_bounds():
    from dynamic_tree_speculative_gb300 import binding as B
    wl = WL.WORKLOADS["vicuna"].with_(B=2, V=5000, depth=3, R=10, K=4, W=2)
    case = parity.make_case(wl, 0)
    case.draft[0, 1, 777] = float("nan")
    g = parity.run_gpu(case, None)
    assert g["status"] & B.S_NONFINITE_DRAFT
    # the other tree is untouched by the bad row
    trees = parity.oracle_build(case, [1])
    assert parity.compare_case(g, case, [1], None, trees)["build_exact"] == 1


def test_probe_survival_independent_of_identity_gpu():
    """Sweeping the root's probe uniform never moves the probe node (only tokens change)."""
    wl = WL.WORKLOADS["vicuna"].with_(B=32, V=4000, depth=4, R=14, K=4, W=3)
    case = parity.make_case(wl, 21)
    case.u_probe[:, 0] = torch.linspace(0.0, 0.999, wl.B)
    case.draft[:] = case.draft[0:1]          # same rows in every tree
    case.u_probe[:, 1:] = case.u_probe[0:1, 1:]
    g = parity.run_gpu(case, None)
    sig = set()
    for b in range(wl.B):
        kinds = g["node_kind"][b]
        parents = g["node_parent"][b]
        probe_nodes = [i for i in range(len(kinds)) if kinds[i] == 2 and parents[i] == 0]
        sig.add(tuple(probe_nodes))
    assert len(sig) == 1, sig


def test_gpu_losslessness_chi_square():
    """Tiny workload on the GPU path, path-keyed targets: first emitted token ~ p(root)."""
    from scipy.stats import chi2
    from dynamic_tree_speculative_gb300 import binding as B
    wl = WL.WORKLOADS["tiny"].with_(B=10000)
    params = B.Params.from_workload(wl)
    n_rows = B.rows_needed(params)
    base, _ = WL.draft_logits(wl.with_(B=1), 77, n_rows=n_rows)
    draft = base.expand(wl.B, -1, -1).contiguous()
    u_probe = WL.uniforms(77, "p", (wl.B, n_rows))
    uv, ub = WL.uniforms(77, "v", (wl.B, wl.depth, wl.K)), WL.uniforms(77, "b", (wl.B,))
    dev = "cuda"
    tree = B.TreeBuffers(params, wl.B, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.spec_tree_build(params, wl.V, draft.to(dev), u_probe.to(dev), tree, status)
    tok = tree.node_token.cpu().numpy()
    par = tree.node_parent.cpu().numpy()
    nn = tree.n_nodes.cpu().numpy()
    cache = {}
    rows = torch.empty((wl.B, wl.R + 1, wl.V), dtype=torch.float32)
    for b in range(wl.B):
        for i in range(wl.R + 1):
            path, j = [], i
            while j > 0:
                path.append(int(tok[b, j]))
                j = par[b, j]
            key = tuple(reversed(path)) if i < nn[b] else ("unused",)
            if key not in cache:
                cache[key] = WL.path_keyed_rows(123, [key if key != ("unused",) else (-7,)], wl.V, 1.2, 0.5)[0]
            rows[b, i] = cache[key]
    out = B.VerifyOutputs(params, wl.B, device=dev)
    B.spec_tree_verify(params, wl.V, rows.to(dev), tree, uv.to(dev), ub.to(dev), out.accept_len, out.out_tok,
                       out.out_node, out.margins, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    first = out.out_tok[:, 0].cpu().numpy()
    p = torch.softmax(cache[()].double(), 0).numpy()
    counts = np.bincount(first, minlength=wl.V)
    exp = p * wl.B
    keep = exp >= 5
    stat = ((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    rest_o, rest_e = counts[~keep].sum(), exp[~keep].sum()
    if rest_e > 0:
        stat += (rest_o - rest_e) ** 2 / rest_e
    dof = keep.sum() + (1 if rest_e > 0 else 0) - 1
    assert chi2.sf(stat, dof) > 1e-3


def _exact_level0_acceptance(rows, wl, target_row, mode):
    """Probability (over the probe draw and the accept uniforms) that the root accepts a child."""
    from oracle import spec_tree_oracle as O
    op = parity.oracle_params(wl)
    p_full = O.target_probs(WL.to_numpy_f64(target_row), wl.temperature)
    ex0 = O.expand_row(rows[0], op, 0.5)
    draws = [(1.0, 0.5)]
    if ex0.probe_pos >= 0:
        cum = np.cumsum(ex0.qT[op.m:])
        draws = []
        for s in range(op.m, len(ex0.q)):
            lo = cum[s - op.m - 1] if s > op.m else 0.0
            if ex0.qT[s] > 0:
                draws.append((ex0.qT[s] / ex0.zT, (lo + cum[s - op.m]) / 2.0 / ex0.zT))
    total = 0.0
    for wgt, u in draws:
        t = O.build(rows, np.array([u]), op)
        kids = O.children_in_order(t, 0, mode)
        steps, _, _ = O.level_thresholds(p_full, t.expansions[0], op.m, [int(t.token[j]) for j in kids],
                                         [int(t.kind[j]) for j in kids], mode)
        reach = 1.0
        for _, _, a, _, _ in steps:
            total += wgt * reach * a
            reach *= 1.0 - a
    return total


def test_depth1_acceptance_of_the_three_verifiers():
    """The pages' single-layer controlled experiment on the GPU path: one root with K = 2
    children verified probe first (RheoSampling), probe last (Rheo + RRSw) and as one-hot
    Top-K (m = K); each GPU acceptance rate over 20000 trees matches the oracle's exact
    expectation, and probe first never accepts less than probe last (Key design 3)."""
    from dynamic_tree_speculative_gb300 import binding as B
    n = 20000
    base = WL.WORKLOADS["tiny"].with_(B=n, K=2, m=1, W=2, depth=1, R=2)
    rows, _ = WL.draft_logits(base.with_(B=1), 31, n_rows=1)
    target_row = WL.latent_rows((31, "tgt-d1"), 1, base.V, 1.2, 0.5)[0]
    dev = "cuda"
    rates, exact = {}, {}
    for name, wl in (("rheo", base), ("rrsw", base.with_(verify_order="rrsw")), ("topk", base.with_(m=2))):
        params = B.Params.from_workload(wl)
        draft = rows.expand(n, -1, -1).contiguous()
        u_probe = WL.uniforms(41, "p", (n, 1))
        uv, ub = WL.uniforms(41, "v", (n, 1, wl.K)), WL.uniforms(41, "b", (n,))
        tree = B.TreeBuffers(params, n, device=dev)
        out = B.VerifyOutputs(params, n, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        B.spec_tree_build(params, wl.V, draft.to(dev), u_probe.to(dev), tree, status)
        target = target_row.reshape(1, 1, -1).expand(n, wl.R + 1, -1).contiguous()
        B.spec_tree_verify(params, wl.V, target.to(dev), tree, uv.to(dev), ub.to(dev), out.accept_len,
                           out.out_tok, out.out_node, None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        rates[name] = float((out.accept_len >= 1).float().mean())
        exact[name] = _exact_level0_acceptance(WL.to_numpy_f64(rows[0]), wl, target_row,
                                               "rrsw" if name == "rrsw" else "rheo")
        sd = (exact[name] * (1 - exact[name]) / n) ** 0.5
        assert abs(rates[name] - exact[name]) < 5 * sd + 1e-9, (name, rates[name], exact[name])
    print("depth-1 acceptance (gpu / exact):", {k: (round(rates[k], 4), round(exact[k], 4)) for k in rates})
    assert exact["rheo"] >= exact["rrsw"] - 1e-12
