"""GPU-vs-oracle comparison helpers for the parity tests.

Rules (float decisions on the two sides are taken in float32 on the GPU and
float64 in the oracle):
  * support ids, node topology, tokens, accept lengths: bit-exact;
  * probabilities, tail masses and scores: within 1e-5 absolute;
  * a tree may differ only if the oracle recorded a near-tie decision for it
    (a probe sample or accept test within 1e-6 of probability mass, a
    ranking gap below 1e-5 relative, a SMART test within 1e-5 relative); such
    trees are counted as exempt and reported.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from dynamic_tree_speculative_gb300 import binding as B
from dynamic_tree_speculative_gb300 import workloads as WL
from oracle import spec_tree_oracle as O

PROB_TOL = 1e-5


def oracle_params(wl: WL.Workload) -> O.Params:
    return O.Params(K=wl.K, m=wl.m, W=wl.W, depth=wl.depth, R=wl.R, temperature=wl.temperature,
                    support=wl.support, builder=wl.builder, lam=wl.lam, beta=wl.beta, gamma=wl.gamma,
                    delta=wl.delta, rho=wl.rho, eta=wl.eta, alpha=wl.alpha)


@dataclasses.dataclass
class Case:
    wl: WL.Workload
    draft: torch.Tensor      # host, [B][n_rows][stride]
    latent: torch.Tensor
    u_probe: torch.Tensor
    u_verify: torch.Tensor
    u_bonus: torch.Tensor
    row_stride: int


def make_case(wl: WL.Workload, seed: int, row_stride=None) -> Case:
    n_rows = B.rows_needed(B.Params.from_workload(wl))
    draft, latent = WL.draft_logits(wl, seed, n_rows=n_rows, row_stride=row_stride)
    uv, ub = WL.verify_uniforms(wl, seed)
    return Case(wl, draft, latent, WL.build_uniforms(wl, seed, n_rows=n_rows), uv, ub, row_stride or wl.V)


def oracle_build(case: Case, trees_idx):
    op = oracle_params(case.wl)
    V = case.wl.V
    out = {}
    for b in trees_idx:
        rows = WL.to_numpy_f64(case.draft[b, :, :V])
        out[b] = O.build(rows, case.u_probe[b].numpy().astype(np.float64), op)
    return out


def target_for(case: Case, trees: dict, seed: int):
    """Target rows [B][R+1][stride] keyed on the oracle trees' expansion slots."""
    wl = case.wl
    exp_row = torch.full((wl.B, wl.R + 1), -1, dtype=torch.int32)
    for b, t in trees.items():
        exp_row[b, :t.n_nodes] = torch.from_numpy(t.exp_row.astype(np.int32))
    return WL.target_logits(wl, seed, case.latent, exp_row, None, row_stride=case.row_stride)


def run_gpu(case: Case, target=None, device="cuda"):
    wl = case.wl
    params = B.Params.from_workload(wl)
    tree = B.TreeBuffers(params, wl.B, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    B.spec_tree_build(params, wl.V, case.draft.to(device), case.u_probe.to(device), tree, status)
    res = {"tree": tree, "status": status}
    if target is not None:
        out = B.VerifyOutputs(params, wl.B, device=device)
        B.spec_tree_verify(params, wl.V, target.to(device), tree, case.u_verify.to(device),
                           case.u_bonus.to(device), out.accept_len, out.out_tok, out.out_node, out.margins, status)
        res["verify"] = out
    torch.cuda.synchronize()
    host = {k: getattr(tree, k).cpu().numpy() for k in (
        "node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "node_score",
        "n_nodes", "sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")}
    if target is not None:
        host.update(accept_len=out.accept_len.cpu().numpy(), out_tok=out.out_tok.cpu().numpy(),
                    out_node=out.out_node.cpu().numpy(), margins=out.margins.cpu().numpy())
    host["status"] = int(status.item())
    # the support selection hands rows out from the tree's counter and leaves it at zero
    assert tree.sched.cpu().tolist() == [0, 0], tree.sched
    return host


def _tree_diffs(g, b, t: O.Tree, S: int):
    """List of mismatching fields of tree b (empty when the GPU equals the oracle)."""
    diffs = []
    n = t.n_nodes
    if int(g["n_nodes"][b]) != n:
        return ["n_nodes"]
    for name, ref in (("node_token", t.token), ("node_parent", t.parent), ("node_depth", t.depth),
                      ("node_kind", t.kind), ("node_slot", t.slot), ("node_exp_row", t.exp_row)):
        if not np.array_equal(g[name][b, :n].astype(np.int64), ref):
            diffs.append(name)
    if not np.allclose(g["node_score"][b, :n], t.score, atol=PROB_TOL, rtol=0):
        diffs.append("node_score")
    for e, ex in t.expansions.items():
        if not np.array_equal(g["sup_id"][b, e, :S].astype(np.int64), ex.sup_id):
            diffs.append(f"sup_id[{e}]")
        if not np.allclose(g["sup_q"][b, e, :S], ex.q, atol=PROB_TOL, rtol=0):
            diffs.append(f"sup_q[{e}]")
        if not np.allclose(g["sup_qT"][b, e, :S], ex.qT, atol=PROB_TOL, rtol=0):
            diffs.append(f"sup_qT[{e}]")
        if abs(g["sup_z"][b, e] - ex.z) > PROB_TOL or abs(g["sup_zT"][b, e] - ex.zT) > PROB_TOL:
            diffs.append(f"z[{e}]")
        if int(g["probe_pos"][b, e]) != ex.probe_pos:
            diffs.append(f"probe_pos[{e}]")
    return diffs


def compare_build(g, trees: dict, S: int):
    """Assert build parity; returns (exact, exempt) tree counts."""
    exact = exempt = 0
    for b, t in trees.items():
        d = _tree_diffs(g, b, t, S)
        if not d:
            exact += 1
            continue
        # support ids are integer work: never exempt
        assert not any(x.startswith("sup_id") for x in d), (b, d)
        assert t.margins.near > 0, f"tree {b} differs without a near-tie: {d[:6]} margins={t.margins.min}"
        exempt += 1
    return exact, exempt


def compare_verify(g, trees: dict, results: dict):
    exact = exempt = 0
    for b, r in results.items():
        t = trees[b]
        same = int(g["accept_len"][b]) == r.accept_len and \
            g["out_tok"][b, :r.accept_len + 1].tolist() == r.tokens and \
            g["out_node"][b, :r.accept_len].tolist() == r.nodes and \
            (g["out_tok"][b, r.accept_len + 1:] == -1).all()
        if same:
            exact += 1
            continue
        near = t.margins.near + r.margins.near
        assert near > 0, (f"tree {b} verify differs without a near-tie: gpu len {int(g['accept_len'][b])} "
                          f"tok {g['out_tok'][b].tolist()} oracle len {r.accept_len} tok {r.tokens} "
                          f"margins {r.margins.min}")
        exempt += 1
    return exact, exempt


def run_parity(wl: WL.Workload, seed: int, sample=None, row_stride=None, verify=True, max_exempt_frac=0.1):
    case = make_case(wl, seed, row_stride)
    idx = list(range(wl.B)) if sample is None else list(sample)
    trees = oracle_build(case, idx)
    target = target_for(case, trees, seed) if verify else None
    g = run_gpu(case, target)
    assert g["status"] == 0, f"status {g['status']}"
    S = min(wl.support, wl.V)
    ex, exm = compare_build(g, trees, S)
    out = {"build_exact": ex, "build_exempt": exm, "gpu": g, "trees": trees}
    if verify:
        op = oracle_params(wl)
        tnp = {b: WL.to_numpy_f64(target[b, :, :wl.V]) for b in idx}
        results = {b: O.verify(trees[b], tnp[b], case.u_verify[b].numpy(), float(case.u_bonus[b]), op,
                               mode=wl.verify_order)
                   for b in idx}
        vx, vxm = compare_verify(g, trees, results)
        out.update(verify_exact=vx, verify_exempt=vxm, results=results)
        assert vxm <= max_exempt_frac * len(idx) + 1, out
    assert exm <= max_exempt_frac * len(idx) + 1, out
    return out
