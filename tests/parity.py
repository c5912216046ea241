"""GPU-vs-oracle parity runs: seeded cases, the GPU path through the C ABI, the oracle beside it.

The comparison rules and the replay of near-tie decisions are in
tests/parity_compare.py: support ids, topology, tokens and accept lengths are
bit-exact except where a difference starts at a decision the oracle logged as
a near-tie (the oracle then adopts the GPU's choice and the comparison goes
on); probabilities, masses and scores agree within 1e-5 absolute.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from dynamic_tree_speculative_gb300 import binding as B
from dynamic_tree_speculative_gb300 import workloads as WL
from oracle import spec_tree_oracle as O

import parity_compare as PC

PROB_TOL = PC.PROB_TOL


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
    tree = B.TreeBuffers(params, wl.B, device=device, V=wl.V)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    draft = case.draft.to(device)
    B.spec_tree_build(params, wl.V, draft, case.u_probe.to(device), tree, status)
    res = {"tree": tree, "status": status}
    if target is not None:
        out = B.VerifyOutputs(params, wl.B, device=device)
        if B.is_dense(params, wl.V):
            B.spec_tree_verify_dense(params, wl.V, target.to(device), draft, tree, case.u_verify.to(device),
                                     case.u_bonus.to(device), out.accept_len, out.out_tok, out.out_node, out.margins,
                                     status)
        else:
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
    assert tree.sched.cpu().tolist()[:2] == [0, 0], tree.sched
    return host


def case_inputs(case: Case, idx):
    """{b: (draft rows as float64, probe uniforms)} for the oracle."""
    V = case.wl.V
    return {b: (WL.to_numpy_f64(case.draft[b, :, :V]), case.u_probe[b].numpy().astype(np.float64)) for b in idx}


def compare_case(g, case: Case, idx, target=None, built=None):
    """Compare the GPU outputs `g` for trees `idx` with the oracle, replaying near-ties (tests/parity_compare.py).

    With `target` ([B][R+1][stride] host tensor), verification is compared too.
    """
    wl = case.wl
    op = oracle_params(wl)
    vin = None
    if target is not None:
        vin = {b: (WL.to_numpy_f64(target[b, :, :wl.V]), case.u_verify[b].numpy(), float(case.u_bonus[b]))
               for b in idx}
    return PC.compare_batch(g, case_inputs(case, idx), op, min(wl.support, wl.V), vin, wl.verify_order, built)


def run_parity(wl: WL.Workload, seed: int, sample=None, row_stride=None, verify=True):
    """Build (and verify) on the GPU, compare trees `sample` (default: all) with the oracle.

    Target rows are keyed on the oracle's expansion slots of the compared trees.
    Any difference must start at a near-tie decision of the oracle, which then
    adopts the GPU's choice (counted in the returned dict's *_replayed fields).
    """
    case = make_case(wl, seed, row_stride)
    idx = list(range(wl.B)) if sample is None else list(sample)
    trees = oracle_build(case, idx)
    target = target_for(case, trees, seed) if verify else None
    g = run_gpu(case, target)
    assert g["status"] == 0, f"status {g['status']}"
    out = compare_case(g, case, idx, target, trees)
    out["gpu"] = g
    return out
