"""Tree-by-tree comparison of another implementation's outputs with the oracle, with replay.

Pure numpy + the oracle: no GPU and no native library here, so the comparison
logic itself is tested on the CPU (tests/test_parity_replay.py).

Rules (the other side takes its float decisions in float32, the oracle in
float64):
  * support ids are compared bit for bit and are never exempt;
  * node topology, tokens, kinds, slots, expansion rows, accepted tokens and
    nodes, accept lengths: bit for bit, except at a decision where the oracle
    itself logged a near-tie (a probe or bonus draw u * Z within 1e-6 * Z of a
    CDF boundary, an accept test with |u - ratio| < 1e-6, two path scores
    within 1e-5 relative, a SMART keep test within 1e-5 relative);
  * at such a decision the oracle adopts the other side's choice (replay mode,
    `oracle.Replay`) and the comparison goes on downstream, so a difference is
    exempt only at the decision where it starts, and only when that decision is
    a near-tie; the oracle refuses to adopt anything else;
  * probabilities, tail masses and scores: within 1e-5 absolute.

Every adopted decision is counted in `TALLY`, which the test session prints.
"""
from __future__ import annotations

import collections

import numpy as np

from oracle import spec_tree_oracle as O

PROB_TOL = 1e-5
MAX_REPLAYS = 16

# session-wide counts: trees compared, trees equal without replay, decisions adopted by kind
TALLY = {"build_trees": 0, "build_exact": 0, "verify_trees": 0, "verify_exact": 0,
         "adopted": collections.Counter()}


class ParityError(AssertionError):
    pass


# ------------------------------------------------------------------ build ---

def _support_diffs(g, b, t: O.Tree, S: int, K: int):
    """Rows of the oracle's tree whose support ids, probabilities or masses differ.

    A dense support of a vocabulary larger than the GPU's support arrays keeps
    support ranks 0..K-1 and, at entry K, the probe: those are compared.
    """
    ids, probs, probes = [], [], []
    dense = S > g["sup_id"].shape[2]
    n = K if dense else S
    for e, ex in t.expansions.items():
        if not np.array_equal(g["sup_id"][b, e, :n].astype(np.int64), ex.sup_id[:n]):
            ids.append(e)
        if not (np.allclose(g["sup_q"][b, e, :n], ex.q[:n], atol=PROB_TOL, rtol=0)
                and np.allclose(g["sup_qT"][b, e, :n], ex.qT[:n], atol=PROB_TOL, rtol=0)
                and abs(g["sup_z"][b, e] - ex.z) <= PROB_TOL and abs(g["sup_zT"][b, e] - ex.zT) <= PROB_TOL):
            probs.append(e)
        pp = int(g["probe_pos"][b, e])
        if pp != ex.probe_pos:
            probes.append(e)
        elif dense and pp >= 0:
            # the probe entry: the oracle's token, q and q_T at that rank
            if int(g["sup_id"][b, e, K]) != int(ex.sup_id[pp]):
                ids.append(e)
            elif abs(g["sup_q"][b, e, K] - ex.q[pp]) > PROB_TOL or abs(g["sup_qT"][b, e, K] - ex.qT[pp]) > PROB_TOL:
                probs.append(e)
    return ids, probs, probes


def _nodes_of(tok, par, dep, kind, slot, exp_row, n, W, builder):
    """Creation keys (depth, parent's frontier rank, slot) of nodes 1..n-1 and their ordering facts."""
    exp_rank = {}
    by_depth = collections.defaultdict(list)
    for i in range(1, n):
        if exp_row[i] >= 0:
            by_depth[int(dep[i])].append(i)
    for d, nodes in by_depth.items():
        nodes.sort(key=lambda i: int(exp_row[i]))
        for r, i in enumerate(nodes):
            exp_rank[i] = (int(exp_row[i]) - 1 - (d - 1) * W) if builder == "topr" else r
    keys = {}
    for i in range(1, n):
        p = int(par[i])
        keys[i] = (int(dep[i]), 0 if p == 0 else exp_rank.get(p, -1), int(slot[i]))
    canon = collections.defaultdict(list)       # per depth, canonical order
    for i in range(1, n):
        canon[int(dep[i])].append(keys[i])
    expanded = {d: [keys[i] for i in nodes] for d, nodes in by_depth.items()}
    return keys, canon, expanded


def _tree_fields_equal(g, b, t: O.Tree):
    n = t.n_nodes
    if int(g["n_nodes"][b]) != n:
        return False
    for name, ref in (("node_token", t.token), ("node_parent", t.parent), ("node_depth", t.depth),
                      ("node_kind", t.kind), ("node_slot", t.slot), ("node_exp_row", t.exp_row)):
        if not np.array_equal(g[name][b, :n].astype(np.int64), ref):
            return False
    return True


def _order_pairs(g_list, o_list, pairs):
    """(x, y) pairs that g_list places x before y while o_list places y before x."""
    pos = {k: i for i, k in enumerate(o_list)}
    common = [k for k in g_list if k in pos]
    for i in range(len(common)):
        for j in range(i + 1, len(common)):
            if pos[common[i]] > pos[common[j]]:
                pairs.add((common[i], common[j]))


def _infer_build_replay(g, b, t: O.Tree, op: O.Params, rp: O.Replay):
    """Add to `rp` the decisions on which the other side's tree differs from the oracle's."""
    ng = int(g["n_nodes"][b])
    gk, gcanon, gexp = _nodes_of(g["node_token"][b], g["node_parent"][b], g["node_depth"][b], g["node_kind"][b],
                                 g["node_slot"][b], g["node_exp_row"][b], ng, op.W, op.builder)
    ok, ocanon, oexp = _nodes_of(t.token, t.parent, t.depth, t.kind, t.slot, t.exp_row, t.n_nodes, op.W,
                                 op.builder)
    gset, oset = set(gk.values()), set(ok.values())
    pairs = set()
    for d in set(gexp) | set(oexp):
        ge, oe = gexp.get(d, []), oexp.get(d, [])
        _order_pairs(ge, oe, pairs)
        if op.builder == "topr":
            for x in ge:
                if x not in oe:
                    for y in oe:
                        if y not in ge:
                            pairs.add((x, y))
    for d in set(gcanon) | set(ocanon):
        _order_pairs(gcanon.get(d, []), ocanon.get(d, []), pairs)
    if op.builder == "topr":
        for x in gset - oset:
            for y in oset - gset:
                pairs.add((x, y))
    else:
        for x in gset - oset:
            rp.keep[x] = True
        for y in oset - gset:
            rp.keep[y] = False
    rp.before |= pairs


def compare_build_tree(g, b: int, rows, u_probe, op: O.Params, S: int, first: O.Tree = None):
    """Oracle tree for tree b, replaying near-ties until it equals the other side's outputs.

    Returns (oracle tree, adopted decisions).  Raises ParityError on any
    difference that does not start at a near-tie the oracle logged.  `first`
    is the oracle's tree without replay when it has been built already.
    """
    rp = O.Replay()
    for _ in range(MAX_REPLAYS):
        rp.adopted = []
        try:
            t = first if (first is not None and not rp) else O.build(rows, u_probe, op, rp if rp else None)
        except O.ReplayRefused as e:
            raise ParityError(f"tree {b}: difference not at a near-tie: {e}") from None
        ids, probs, probes = _support_diffs(g, b, t, S, op.K)
        if ids:
            raise ParityError(f"tree {b}: support ids differ in rows {ids[:8]}")
        if probs:
            raise ParityError(f"tree {b}: support probabilities differ in rows {probs[:8]}")
        new_probe = {e: int(g["probe_pos"][b, e]) for e in probes}
        if new_probe:
            if all(rp.probe.get(e) == v for e, v in new_probe.items()):
                raise ParityError(f"tree {b}: probe ranks differ in rows {probes[:8]} after replay")
            rp.probe.update(new_probe)
            continue
        if _tree_fields_equal(g, b, t):
            if not np.allclose(g["node_score"][b, :t.n_nodes], t.score, atol=PROB_TOL, rtol=0):
                raise ParityError(f"tree {b}: node scores differ beyond {PROB_TOL}")
            return t, list(rp.adopted)
        before = (set(rp.before), dict(rp.keep))
        _infer_build_replay(g, b, t, op, rp)
        if (rp.before, rp.keep) == before:
            raise ParityError(f"tree {b}: node arrays differ and no near-tie decision explains it "
                              f"(oracle near-ties: {t.margins.ties[:6]})")
    raise ParityError(f"tree {b}: still different after {MAX_REPLAYS} replays")


# ----------------------------------------------------------------- verify ---

def _verify_equal(g, b, r: O.VerifyResult):
    return (int(g["accept_len"][b]) == r.accept_len
            and g["out_tok"][b, :r.accept_len + 1].tolist() == r.tokens
            and g["out_node"][b, :r.accept_len].tolist() == r.nodes
            and bool((g["out_tok"][b, r.accept_len + 1:] == -1).all())
            and bool((g["out_node"][b, r.accept_len:] == -1).all()))


def compare_verify_tree(g, b: int, t: O.Tree, target_rows, u_verify, u_bonus: float, op: O.Params, mode: str):
    """Oracle verification of tree b, replaying near-tie decisions until it equals the other side's.

    Returns (oracle result, adopted decisions); raises ParityError otherwise.
    """
    rp = O.Replay()
    acc_g = int(g["accept_len"][b])
    nodes_g = [int(x) for x in g["out_node"][b, :max(acc_g, 0)]]
    for _ in range(MAX_REPLAYS):
        rp.adopted = []
        try:
            r = O.verify(t, target_rows, u_verify, u_bonus, op, mode=mode, replay=rp if rp else None)
        except O.ReplayRefused as e:
            raise ParityError(f"tree {b}: verification differs, not at a near-tie: {e}") from None
        if _verify_equal(g, b, r):
            return r, list(rp.adopted)
        # first level where the walks part
        lvl = 0
        while lvl < min(acc_g, r.accept_len) and nodes_g[lvl] == r.nodes[lvl]:
            lvl += 1
        node = 0 if lvl == 0 else r.nodes[lvl - 1]
        kids = O.children_in_order(t, node, mode)
        j_g = kids.index(nodes_g[lvl]) if lvl < acc_g and nodes_g[lvl] in kids else len(kids)
        j_o = kids.index(r.nodes[lvl]) if lvl < r.accept_len else len(kids)
        before = (dict(rp.accept), dict(rp.bonus))
        if j_g < j_o:
            rp.accept[(lvl, j_g)] = True
        elif j_o < j_g:
            rp.accept[(lvl, j_o)] = False
        else:
            rp.bonus[lvl] = int(g["out_tok"][b, lvl])
        if (rp.accept, rp.bonus) == before:
            raise ParityError(f"tree {b}: verification differs at level {lvl} after replay")
    raise ParityError(f"tree {b}: verification still different after {MAX_REPLAYS} replays")


# ------------------------------------------------------------------ batch ---

def compare_batch(g, trees_in: dict, op: O.Params, S: int, verify_inputs=None, mode="rheo", built=None):
    """Compare every tree of `trees_in` ({b: (rows, u_probe)}); optionally verification too.

    verify_inputs: {b: (target_rows, u_verify, u_bonus)} or None; built: {b: oracle
    tree without replay} where already built.  Returns a
    dict of counts and the oracle's trees/results; raises ParityError on the
    first tree that differs other than at a near-tie.
    """
    out = {"build_exact": 0, "build_replayed": 0, "verify_exact": 0, "verify_replayed": 0,
           "adopted": [], "trees": {}, "results": {}}
    for b, (rows, u) in trees_in.items():
        t, adopted = compare_build_tree(g, b, rows, u, op, S, (built or {}).get(b))
        out["trees"][b] = t
        TALLY["build_trees"] += 1
        if adopted:
            out["build_replayed"] += 1
            out["adopted"] += [(b,) + tuple(a) for a in adopted]
            TALLY["adopted"].update(a[0] for a in adopted)
        else:
            out["build_exact"] += 1
            TALLY["build_exact"] += 1
        if verify_inputs is not None:
            tgt, uv, ub = verify_inputs[b]
            r, vad = compare_verify_tree(g, b, t, tgt, uv, ub, op, mode)
            out["results"][b] = r
            TALLY["verify_trees"] += 1
            if vad:
                out["verify_replayed"] += 1
                out["adopted"] += [(b,) + tuple(a) for a in vad]
                TALLY["adopted"].update(a[0] for a in vad)
            else:
                out["verify_exact"] += 1
                TALLY["verify_exact"] += 1
    return out


def tally_line() -> str:
    a = dict(TALLY["adopted"])
    return (f"parity vs oracle: build {TALLY['build_exact']}/{TALLY['build_trees']} trees equal without replay, "
            f"verify {TALLY['verify_exact']}/{TALLY['verify_trees']}; near-tie decisions adopted: "
            f"{sum(a.values())} {a if a else ''}")
