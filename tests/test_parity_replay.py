"""The parity comparison and its replay mode, checked on the CPU against outputs made by the oracle.

The "other implementation" here is the oracle itself, run with a near-tie
decision taken the other way (which the oracle permits only at a near-tie),
or with an output edited by hand (a real mistake).  The comparison must
adopt the first kind at exactly that decision, count it, and refuse the
second kind.
"""
import numpy as np
import pytest

import parity_compare as PC
from oracle import spec_tree_oracle as O


def outputs(trees, results, p: O.Params, n_rows: int, S: int, rows=None, u=None):
    """The oracle's trees (and verification results) in the GPU path's output layout.

    Like the GPU path, every draft row's support is filled (from `rows`, `u` for
    rows the tree did not expand)."""
    B = len(trees)
    M = max(t.n_nodes for t in trees) + 4
    g = {k: np.full((B, M), -1, np.int32) for k in
         ("node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row")}
    g["node_score"] = np.zeros((B, M), np.float32)
    g["n_nodes"] = np.zeros(B, np.int32)
    g["sup_id"] = np.full((B, n_rows, S), -1, np.int32)
    for k in ("sup_q", "sup_qT"):
        g[k] = np.zeros((B, n_rows, S), np.float32)
    for k in ("sup_z", "sup_zT"):
        g[k] = np.zeros((B, n_rows), np.float32)
    g["probe_pos"] = np.full((B, n_rows), -1, np.int32)
    for b, t in enumerate(trees):
        n = t.n_nodes
        g["n_nodes"][b] = n
        for k, v in (("node_token", t.token), ("node_parent", t.parent), ("node_depth", t.depth),
                     ("node_kind", t.kind), ("node_slot", t.slot), ("node_exp_row", t.exp_row)):
            g[k][b, :n] = v
        g["node_score"][b, :n] = t.score
        exps = dict(t.expansions)
        if rows is not None:
            for e in range(n_rows):
                exps.setdefault(e, O.expand_row(rows[e], p, float(u[e])))
        for e, ex in exps.items():
            g["sup_id"][b, e] = ex.sup_id
            g["sup_q"][b, e], g["sup_qT"][b, e] = ex.q, ex.qT
            g["sup_z"][b, e], g["sup_zT"][b, e] = ex.z, ex.zT
            g["probe_pos"][b, e] = ex.probe_pos
    if results is not None:
        g["accept_len"] = np.array([r.accept_len for r in results], np.int32)
        g["out_tok"] = np.full((B, p.depth + 1), -1, np.int32)
        g["out_node"] = np.full((B, p.depth + 1), -1, np.int32)
        for b, r in enumerate(results):
            g["out_tok"][b, :len(r.tokens)] = r.tokens
            g["out_node"][b, :len(r.nodes)] = r.nodes
    return g


def _rows(seed, n, V):
    rng = np.random.default_rng(seed)
    return -1.2 * np.log(1 + rng.permutation(V)[None, :].repeat(n, 0)) + rng.normal(0, 0.5, (n, V))


P = O.Params(K=4, m=1, W=3, depth=3, R=9, support=32)


@pytest.fixture(autouse=True)
def _keep_session_tally():
    """These comparisons are oracle against oracle: keep them out of the session's GPU parity counts."""
    saved = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in PC.TALLY.items()}
    yield
    PC.TALLY.clear()
    PC.TALLY.update(saved)


def _case(seed=0):
    n_rows = 1 + (P.depth - 1) * P.W
    rows = _rows(seed, n_rows, 32)
    u = np.random.default_rng(seed + 100).random(n_rows)
    return rows, u, n_rows


def test_identical_outputs_compare_equal_without_replay():
    rows, u, n_rows = _case()
    t = O.build(rows, u, P)
    g = outputs([t], None, P, n_rows, 32)
    out = PC.compare_batch(g, {0: (rows, u)}, P, 32)
    assert out["build_exact"] == 1 and not out["adopted"]


def test_probe_draw_near_tie_is_adopted_at_its_row():
    rows, u, n_rows = _case(1)
    ex = O.expand_row(rows[0], P, 0.5)
    cum = np.cumsum(ex.qT[P.m:])
    # put the root's draw 1e-9 of mass above the boundary between tail ranks 2 and 3
    u[0] = (cum[1] + 1e-9) / ex.zT
    t = O.build(rows, u, P)
    assert t.expansions[0].probe_pos == P.m + 2
    other = O.build(rows, u, P, O.Replay(probe={0: P.m + 1}))
    g = outputs([other], None, P, n_rows, 32)
    out = PC.compare_batch(g, {0: (rows, u)}, P, 32)
    assert out["build_replayed"] == 1 and out["adopted"] == [(0, "probe", 0)]
    # the oracle refuses a rank that the draw does not reach
    with pytest.raises(O.ReplayRefused):
        O.build(rows, u, P, O.Replay(probe={0: P.m + 3}))


def test_probe_difference_away_from_a_tie_fails():
    rows, u, n_rows = _case(2)
    t = O.build(rows, u, P)
    g = outputs([t], None, P, n_rows, 32)
    k = t.expansions[0].probe_pos
    g["probe_pos"][0, 0] = k + 1 if k + 1 < 32 else k - 1
    with pytest.raises(PC.ParityError):
        PC.compare_batch(g, {0: (rows, u)}, P, 32)


def _near_tied_fillers(seed):
    """Rows whose root has two fillers with path scores 1e-9 apart (relative)."""
    rows, u, n_rows = _case(seed)
    order = np.argsort(-rows[0], kind="stable")
    rows[0, order[2]] = rows[0, order[1]] - 1e-9
    return rows, u, n_rows


def test_ranking_near_tie_is_adopted():
    rows, u, n_rows = _near_tied_fillers(3)
    u[0] = 0.999   # probe deep in the tail: the fillers are support ranks 1 and 2
    t = O.build(rows, u, P)
    fills = [int(t.slot[i]) for i in range(t.n_nodes) if t.kind[i] == O.FILL and t.depth[i] == 1]
    assert fills == [2, 3]
    a, b = (1, 0, 2), (1, 0, 3)    # the two near-tied fillers
    other = O.build(rows, u, P, O.Replay(before={(b, a)}))
    assert other.token.tolist() != t.token.tolist() or other.exp_row.tolist() != t.exp_row.tolist()
    g = outputs([other], None, P, n_rows, 32)
    out = PC.compare_batch(g, {0: (rows, u)}, P, 32)
    assert out["build_replayed"] == 1 and all(x[1] == "order" for x in out["adopted"]), (fills, out["adopted"])


def test_ranking_difference_away_from_a_tie_fails():
    rows, u, n_rows = _case(4)
    t = O.build(rows, u, P)
    g = outputs([t], None, P, n_rows, 32)
    with pytest.raises(PC.ParityError):     # an exact tie is broken by the creation index
        g2 = outputs([t], None, P, n_rows, 32)
        for k in ("node_token", "node_kind", "node_slot", "node_exp_row"):
            g2[k][0, [1, 2]] = g2[k][0, [2, 1]]
        assert t.score[1] == t.score[2]
        PC.compare_batch(g2, {0: (rows, u)}, P, 32)
    # swap two first-layer nodes of the canonical order whose scores are far apart
    d1 = [i for i in range(t.n_nodes) if t.depth[i] == 1]
    i, j = next((i, j) for i in d1 for j in d1 if j > i and t.score[i] - t.score[j] > 1e-3 * t.score[i])
    for k in ("node_token", "node_kind", "node_slot", "node_exp_row"):
        g[k][0, [i, j]] = g[k][0, [j, i]]
    with pytest.raises(PC.ParityError):
        PC.compare_batch(g, {0: (rows, u)}, P, 32)


def _verify_case(seed):
    rows, u, n_rows = _case(seed)
    t = O.build(rows, u, P)
    rng = np.random.default_rng(seed + 7)
    target = _rows(seed + 50, P.R + 1, 32)
    uv = rng.random((P.depth, P.K))
    return rows, u, n_rows, t, target, uv, float(rng.random())


def test_accept_test_near_tie_is_adopted():
    rows, u, n_rows, t, target, uv, ub = _verify_case(5)
    p_full = O.target_probs(target[0], 1.0)
    kids = O.children_in_order(t, 0)
    steps, _, _ = O.level_thresholds(p_full, t.expansions[0], P.m, [int(t.token[j]) for j in kids],
                                     [int(t.kind[j]) for j in kids])
    uv[0, 0] = steps[0][2] - 1e-9 if steps[0][2] < 1 else 0.5     # just below the first accept threshold
    r = O.verify(t, target, uv, ub, P)
    assert r.accept_len >= 1
    other = O.verify(t, target, uv, ub, P, replay=O.Replay(accept={(0, 0): False}))
    g = outputs([t], [other], P, n_rows, 32)
    out = PC.compare_batch(g, {0: (rows, u)}, P, 32, {0: (target, uv, ub)})
    assert out["verify_replayed"] == 1 and out["adopted"][0][1] == "accept"
    with pytest.raises(O.ReplayRefused):
        uv2 = uv.copy()
        uv2[0, 0] = 0.0
        O.verify(t, target, uv2, ub, P, replay=O.Replay(accept={(0, 0): False}))


def test_bonus_near_tie_is_adopted_and_a_wrong_bonus_fails():
    rows, u, n_rows, t, target, uv, ub = _verify_case(6)
    uv[:] = 0.999999   # reject every one-hot child; the walk ends where a probe ratio >= 1 stops accepting
    r = O.verify(t, target, uv, ub, P)
    lvl = r.accept_len
    node = r.nodes[-1] if r.nodes else 0
    p_full = O.target_probs(target[node], 1.0)
    kids = O.children_in_order(t, node)
    if kids:
        _, w, Zr = O.level_thresholds(p_full, t.expansions[int(t.exp_row[node])], P.m,
                                      [int(t.token[j]) for j in kids], [int(t.kind[j]) for j in kids])
    else:
        w, Zr = p_full, 1.0
    cum = np.cumsum(w)
    v = int(np.nonzero(w > 0)[0][3])
    ub = (cum[v] + 1e-9) / Zr          # a draw 1e-9 of mass above the end of token v's interval
    r = O.verify(t, target, uv, ub, P)
    assert r.accept_len == lvl and r.tokens[-1] != v
    other = O.verify(t, target, uv, ub, P, replay=O.Replay(bonus={lvl: v}))
    assert other.tokens[-1] == v
    g = outputs([t], [other], P, n_rows, 32)
    out = PC.compare_batch(g, {0: (rows, u)}, P, 32, {0: (target, uv, ub)})
    assert out["adopted"] == [(0, "bonus", lvl)]
    g["out_tok"][0, lvl] = (v + 5) % 32
    with pytest.raises(PC.ParityError):
        PC.compare_batch(g, {0: (rows, u)}, P, 32, {0: (target, uv, ub)})


def test_smart_keep_near_tie_is_adopted():
    rows, u, n_rows = _case(8)
    rows[0] *= 4.0          # a peaked root: q(x_1) > z, so the probe's proxy z is below the top child
    ex = O.expand_row(rows[0], P, u[0])
    top = max(c[4] for c in ex.children)
    assert sum(c[4] == top for c in ex.children) == 1
    # first test: keep iff alpha * P / lambda > 1; put lambda 1e-9 (relative) under P
    ps = O.Params(K=4, m=1, W=3, depth=3, R=9, support=32, builder="smart", lam=top / (1 + 1e-9), gamma=0.0)
    t = O.build(rows, u, ps)
    assert t.trace[0]["keep"]
    first = t.trace[0]["path"]
    key = (1, 0, [c[0] for c in ex.children if c[4] == top][0])
    other = O.build(rows, u, ps, O.Replay(keep={key: False}))
    assert other.n_nodes == 1 and first
    g = outputs([other], None, ps, n_rows, 32, rows, u)
    out = PC.compare_batch(g, {0: (rows, u)}, ps, 32)
    assert out["adopted"] == [(0, "smart", 1, key)]
