"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine on the same definition, brute force on tiny inputs, a closed form, an
invariant the pages state (the Local Ranking Preservation lemma), exact
enumeration of the output law (losslessness) or a hand-worked example.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import spec_tree_oracle as O
from dynamic_tree_speculative_gb300 import workloads as WL


def _bf16_row(rng, V, spread=6.0, ties=True):
    """Random bf16-valued row (as exact float64) with many exact ties."""
    x = rng.normal(0.0, spread, V)
    if ties:
        x = np.round(x * 4) / 4
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------- inputs ---

def test_bf16_bits_decode_matches_torch():
    rng = np.random.default_rng(0)
    x = torch.tensor(rng.normal(0, 30, 4096), dtype=torch.float32).to(torch.bfloat16)
    x[:4] = torch.tensor([0.0, -0.0, float("inf"), float("-inf")], dtype=torch.bfloat16)
    bits = WL.bf16_bits(x)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())


# ----------------------------------------------------------- truncation ---

@pytest.mark.parametrize("V,size", [(40, 128), (300, 128), (1000, 128), (257, 7),
                                    # the support-size ablation, and the dense support of a small vocabulary
                                    (3000, 256), (3000, 512), (5000, 1024), (700, 1024)])
def test_support_is_brute_force_top_by_logit_then_id(V, size):
    rng = np.random.default_rng(V)
    for _ in range(20):
        row = _bf16_row(rng, V)
        got = O.support_of(row, min(size, V))
        brute = sorted(range(V), key=lambda v: (-row[v], v))[:min(size, V)]
        assert list(got) == brute


def test_support_treats_signed_zeros_equal_and_nan_last():
    row = np.array([-0.0, 0.0, np.nan, -1.0, 0.0, np.inf * -1])
    assert list(O.support_of(row, 6)[:4]) == [0, 1, 4, 3]
    assert O.support_of(row, 6)[-1] == 2


def test_target_probs_match_scipy():
    """p = softmax(t / T) over the whole vocabulary (RheoSampling, training strategy: verification at
    temperature T), against scipy's softmax."""
    rng = np.random.default_rng(3)
    for T in (1.0, 0.7, 1.6):
        row = _bf16_row(rng, 5000)
        np.testing.assert_allclose(O.target_probs(row, T), scipy.special.softmax(row.astype(np.float64) / T),
                                   rtol=1e-12, atol=1e-15)


def test_truncated_softmax_matches_scipy():
    rng = np.random.default_rng(1)
    for T in (1.0, 0.7, 1.6):
        row = _bf16_row(rng, 5000)
        sup = O.support_of(row, 128)
        q, qT, _, _ = O.truncated_softmax(row[sup], T)
        np.testing.assert_allclose(q, scipy.special.softmax(row[sup]), rtol=1e-13, atol=0)
        np.testing.assert_allclose(qT, scipy.special.softmax(row[sup] / T), rtol=1e-13, atol=0)


# ------------------------------------------------ dual-identity expansion ---

@pytest.mark.parametrize("m", [0, 1, 2, 3])
@pytest.mark.parametrize("T", [1.0, 0.7, 1.5])
def test_local_ranking_preservation_lemma(m, T):
    """q_proxy(x_s) >= q(x_{m+1}) and <= q(x_m) at every expanded node (Key design 2)."""
    rng = np.random.default_rng(10 * m + int(T * 10))
    p = O.Params(K=8, m=m, W=8, depth=2, R=8, temperature=T)
    for i in range(200):
        row = _bf16_row(rng, 600, spread=rng.uniform(0.5, 8.0))
        ex = O.expand_row(row, p, rng.random())
        kids = {slot: (kind, rank, tok, lp) for slot, kind, rank, tok, lp in ex.children}
        assert kids[m][0] == O.PROBE
        proxy = kids[m][3]
        assert proxy >= ex.q[m]
        if m >= 1:
            assert proxy <= ex.q[m - 1]
        for slot in range(m + 1, 8):
            assert kids[slot][0] == O.FILL and kids[slot][3] <= proxy


def test_probe_law_is_the_tempered_tail():
    """The probe identity is distributed as q~_T = q_T / z_T over the tail."""
    rng = np.random.default_rng(3)
    row = _bf16_row(rng, 200, spread=2.0)
    for m, T in [(1, 1.0), (2, 0.7), (0, 1.3)]:
        p = O.Params(K=4, m=m, W=4, depth=2, R=4, temperature=T)
        n = 20000
        counts = {}
        for j in range(n):
            ex = O.expand_row(row, p, (j + 0.5) / n)
            counts[ex.probe_pos] = counts.get(ex.probe_pos, 0) + 1
        ex = O.expand_row(row, p, 0.5)
        for k in range(m, len(ex.q)):
            # grid quadrature of the inverse CDF: error at most one grid cell per side
            assert abs(counts.get(k, 0) / n - ex.qT[k] / ex.zT) <= 2.0 / n + 1e-12


def test_expansion_slots_and_fillers():
    row = np.array([5.0, 4.0, 3.0, 2.0, 1.0, 0.0, -1.0, -2.0])
    p = O.Params(K=5, m=1, W=2, depth=2, R=4)
    # force the probe to rank 2 (token 2): fillers skip it
    ex = O.expand_row(row, p, 0.0, force_probe_pos=2)
    assert [(s, k, tok) for s, k, _, tok, _ in ex.children] == \
        [(0, O.DET, 0), (1, O.PROBE, 2), (2, O.FILL, 1), (3, O.FILL, 3), (4, O.FILL, 4)]
    q = np.exp(row - 5.0) / np.exp(row - 5.0).sum()
    z = q[1:].sum()
    assert ex.children[1][4] == pytest.approx(min(q[0], z), rel=1e-14)
    # no tail weight -> no probe, fillers take every non-deterministic slot
    row2 = np.array([0.0, -np.inf, -np.inf, -np.inf, -np.inf])
    ex2 = O.expand_row(row2, O.Params(K=3, m=1, W=1, depth=1, R=3), 0.3)
    assert ex2.probe_pos == -1 and [k for _, k, _, _, _ in ex2.children] == [O.DET, O.FILL, O.FILL]


# --------------------------------------------------------------- building ---

def _tiny_rows(seed, n_rows, V=32, dtype="f32"):
    wl = WL.WORKLOADS["tiny"]
    drf, _ = WL.draft_logits(wl.with_(V=V, dtype=dtype), seed, n_rows=n_rows)
    return WL.to_numpy_f64(drf[0])


def test_full_tree_frontier_structure():
    """With R >= N_cand the tree holds every candidate: check the frontier rule."""
    p = O.Params(K=4, m=1, W=3, depth=4, R=10_000)
    n_rows = 1 + (p.depth - 1) * p.W
    for seed in range(5):
        rows = _tiny_rows(seed, n_rows)
        u = np.random.default_rng(seed).random(n_rows)
        t = O.build_topr(rows, u, p)
        assert t.n_nodes == 1 + p.K + (p.depth - 1) * p.W * p.K
        for d in range(1, p.depth):
            at_d = [i for i in range(t.n_nodes) if t.depth[i] == d]
            best = sorted(at_d, key=lambda i: (-t.score[i], i))[:p.W]
            expd = sorted([i for i in at_d if t.exp_row[i] >= 0], key=lambda i: t.exp_row[i])
            assert expd == best
            assert [t.exp_row[i] for i in expd] == [1 + (d - 1) * p.W + r for r in range(p.W)]
        for i in range(1, t.n_nodes):
            par = t.parent[i]
            assert t.depth[i] == t.depth[par] + 1
            # path score = product of local probabilities (proxy for probes)
            ex = t.expansions[t.exp_row[par]]
            lp = [c[4] for c in ex.children if c[0] == t.slot[i]][0]
            assert t.score[i] == t.score[par] * lp
            assert t.score[i] <= t.score[par]
        n_kids = np.bincount(t.parent[1:], minlength=t.n_nodes)
        for i in range(t.n_nodes):
            assert n_kids[i] == (p.K if (t.exp_row[i] >= 0) else 0)


def test_topr_is_the_top_r_subset_of_the_full_tree():
    p_full = O.Params(K=4, m=1, W=3, depth=4, R=10_000)
    n_rows = 1 + (p_full.depth - 1) * p_full.W
    for seed in range(5):
        rows = _tiny_rows(100 + seed, n_rows)
        u = np.random.default_rng(seed).random(n_rows)
        full = O.build_topr(rows, u, p_full)

        def path(t, i):
            out = []
            while i > 0:
                out.append((int(t.slot[i]),))
                i = t.parent[i]
            return tuple(reversed(out))

        for R in (1, 5, 8, 20, 37):
            t = O.build_topr(rows, u, O.Params(K=4, m=1, W=3, depth=4, R=R))
            assert t.n_nodes == R + 1
            keys = {path(full, i): (-full.score[i], full.depth[i], i) for i in range(1, full.n_nodes)}
            # creation order key: depth, then position in the full tree's canonical order is
            # (depth, score, parent rank, slot); break exact ties the same way
            want = sorted(keys, key=lambda k: keys[k])[:R]
            got = [path(t, i) for i in range(1, t.n_nodes)]
            assert sorted(got) == sorted(want)
            # canonical order: depth ascending, then score descending
            for i in range(1, t.n_nodes - 1):
                a, b = i, i + 1
                assert (t.depth[a], -t.score[a]) <= (t.depth[b], -t.score[b])
            # ancestor closed
            for i in range(1, t.n_nodes):
                assert 0 <= t.parent[i] < i


def test_probe_survival_is_independent_of_probe_identity():
    """Sweeping one row's probe uniform changes tokens but not the probe's rank (Key design 2)."""
    p = O.Params(K=4, m=1, W=3, depth=4, R=12)
    n_rows = 1 + (p.depth - 1) * p.W
    rows = _tiny_rows(7, n_rows)
    base_u = np.random.default_rng(7).random(n_rows)
    for row in (0, 1, 4):
        sigs = set()
        for g in np.linspace(0.0, 0.999, 40):
            u = base_u.copy()
            u[row] = g
            t = O.build_topr(rows, u, p)
            # find the probe child of the node expanded from `row`
            owner = [i for i in range(t.n_nodes) if t.exp_row[i] == row]
            if not owner:
                continue
            probe = [i for i in range(t.n_nodes) if t.parent[i] == owner[0] and t.kind[i] == O.PROBE]
            survives = bool(probe)
            pos = probe[0] if probe else -1
            exp_row = int(t.exp_row[probe[0]]) if probe else -2
            sigs.add((survives, pos, exp_row))
        assert len(sigs) <= 1, sigs


@pytest.mark.parametrize("seed", range(3))
def test_m0_with_probe_on_top1_is_deterministic_topk(seed):
    """m = 0 and u_probe = 0: the probe is x_1, so every node expands to its top-K (findings on m)."""
    p = O.Params(K=4, m=0, W=3, depth=3, R=12)
    n_rows = 1 + (p.depth - 1) * p.W
    rows = _tiny_rows(200 + seed, n_rows)
    t = O.build_topr(rows, np.zeros(n_rows), p)
    for i in range(t.n_nodes):
        if t.exp_row[i] < 0:
            continue
        row = rows[t.exp_row[i]]
        kids = [j for j in range(t.n_nodes) if t.parent[j] == i]
        topk = sorted(range(len(row)), key=lambda v: (-row[v], v))[:p.K]
        assert set(int(t.token[j]) for j in kids) <= set(topk)
        q = scipy.special.softmax(row)  # V = 32 < 128: the support is the whole row
        for j in kids:
            assert t.score[j] == pytest.approx(t.score[i] * q[int(t.token[j])], rel=1e-12)


# ------------------------------------------------------------------ SMART ---

def test_smart_cost_closed_forms():
    p = O.Params(K=8, m=1, W=8, depth=8, R=60)
    assert O.smart_cost(0, p) == 1.0
    assert O.smart_marginal_cost(0, p) == pytest.approx(0.02)
    # C(1) = 1 + 0.02 + 0.5*(e^0.01 - 1)
    assert O.smart_cost(1, p) == pytest.approx(1.02 + 0.5 * (math.exp(0.01) - 1), rel=1e-15)
    # C(10) = 1 + 0.2 + 0.5*(e^(0.01*10^1.3) - 1); 10^1.3 = 19.952623...
    assert O.smart_cost(10, p) == pytest.approx(1.2 + 0.5 * (math.exp(0.19952623149688797) - 1), rel=1e-14)
    # dC/dn is the derivative of C: central difference
    for n in (1.0, 5.0, 20.0, 60.0):
        h = 1e-5
        fd = (O.smart_cost(n + h, p) - O.smart_cost(n - h, p)) / (2 * h)
        assert O.smart_marginal_cost(n, p) == pytest.approx(fd, rel=1e-8)


def test_smart_first_keep_threshold_is_lambda():
    """Empty tree: C(0) = 1, dC(0) = lambda, L = 1, |P| = 1 => keep iff alpha * P > lambda."""
    p = O.Params(K=2, m=0, W=2, depth=1, R=5, builder="smart")
    for P_top, expect in [(0.019, False), (0.021, True), (0.5, True)]:
        keep, lhs, rhs = O.smart_keep(P_top, 0, 1.0, 1, p)
        assert keep == expect
        assert rhs == 1.0 and lhs == pytest.approx(P_top / 0.02)


def test_smart_tree_structure():
    p = O.Params(K=4, m=1, W=4, depth=4, R=6, builder="smart")
    rows = _tiny_rows(9, p.R + 1)
    u = np.random.default_rng(9).random(p.R + 1)
    t = O.build_smart(rows, u, p)
    assert 1 <= t.n_nodes <= p.R + 1
    for i in range(1, t.n_nodes):
        assert 0 <= t.parent[i] < i and t.depth[i] == t.depth[t.parent[i]] + 1
    # lambda huge: nothing is worth expanding
    t0 = O.build_smart(rows, u, O.Params(K=4, m=1, W=4, depth=4, R=6, builder="smart", lam=100.0))
    assert t0.n_nodes == 1
    # free nodes: every candidate is kept until the budget
    tf = O.build_smart(rows, u, O.Params(K=4, m=1, W=4, depth=4, R=6, builder="smart",
                                         lam=1e-12, gamma=0.0))
    assert tf.n_nodes == 7


# ------------------------------------------------------------ verification ---

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def _golden(name):
    import json
    import os
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_hand_worked_verification_level():
    """V = 4, one node, m = 1: the hand derivation in tests/golden/hand_worked_level.json."""
    g = _golden("hand_worked_level.json")
    row = np.log(np.array(g["draft_q"]))
    p = O.Params(K=g["K"], m=g["m"], W=1, depth=1, R=g["K"])
    ex = O.expand_row(row, p, 0.0, force_probe_pos=g["probe_rank"])
    assert ex.children[g["m"]][4] == pytest.approx(g["expected_proxy"], abs=1e-15)
    p_full = O.target_probs(np.log(np.array(g["target_p"])), 1.0)
    by_slot = sorted(ex.children)
    order = [by_slot[g["m"]]] + [c for c in by_slot if c[1] != O.PROBE]
    steps, w, Zr = O.level_thresholds(p_full, ex, g["m"], [c[3] for c in order], [c[1] for c in order])
    assert [[k, x] for k, x, *_ in steps] == g["expected_order"]  # [kind, token]
    np.testing.assert_allclose([s[2] for s in steps], g["expected_accept"], atol=1e-14)
    np.testing.assert_allclose([s[4] for s in steps], g["expected_Zr_before"], atol=1e-14)
    assert Zr == pytest.approx(g["expected_final_Zr"], abs=1e-14)
    np.testing.assert_allclose(w, g["expected_final_w"], atol=1e-14)


def test_smart_cost_golden_values():
    g = _golden("smart_cost.json")
    c = g["coefficients"]
    p = O.Params(K=8, m=1, W=8, depth=8, R=60, lam=c["lambda"], gamma=c["gamma"], delta=c["delta"],
                 rho=c["rho"], beta=c["beta"], eta=c["eta"])
    for n, val in g["C"].items():
        assert O.smart_cost(int(n), p) == pytest.approx(val, rel=1e-14)
    P = g["first_keep_threshold_P"]
    assert not O.smart_keep(P * 0.999, 0, 1.0, 1, p)[0]
    assert O.smart_keep(P * 1.001, 0, 1.0, 1, p)[0]


def check_smart_golden(O_mod):
    """The SMART builder against the hand-worked trees of tests/golden/smart_tree.json:
    every keep test (candidate, state n / L / |P|, lhs, rhs, decision) in order, the kept
    set in canonical order and each kept node's expansion row."""
    g = _golden("smart_tree.json")
    rows = np.log(np.array(g["draft_q"]))
    u = np.array(g["u_probe"])
    for case in g["cases"]:
        p = O_mod.Params(K=2, m=1, W=2, depth=3, R=case["R"], support=6, builder="smart", lam=case["lam"],
                         gamma=case["gamma"], delta=case["delta"], rho=case["rho"], alpha=case["alpha"])
        t = O_mod.build_smart(rows, u, p)
        got = [(e["layer"], list(e["path"]), e["n"], e["paths"], e["keep"]) for e in t.trace]
        want = [(e["layer"], e["path"], e["n"], e["paths"], e["keep"]) for e in case["expected_trace"]]
        assert got == want, (case["name"], got, want)
        for e, w in zip(t.trace, case["expected_trace"]):
            for k in ("score", "L", "lhs", "rhs"):
                assert e[k] == pytest.approx(w[k], rel=1e-12), (case["name"], w["path"], k)
        paths = []
        for i in range(1, t.n_nodes):
            path, j = [], i
            while j > 0:
                path.append(int(t.token[j]))
                j = int(t.parent[j])
            paths.append(list(reversed(path)))
        assert paths == [k["path"] for k in case["expected_kept"]], (case["name"], paths)
        assert t.exp_row[1:].tolist() == [k["exp_row"] for k in case["expected_kept"]], case["name"]
        assert t.exp_row[0] == 0


def test_smart_builder_hand_worked_trees():
    """SMART notes, flowchart and Key design 3: three hand-worked trees (linear cost, a budget
    reached mid-layer, convex cost with alpha = 0.8) with every keep test derived by hand."""
    check_smart_golden(O)


def _first_token_law(rows, u_rest, p, target_root, mode="rheo"):
    """Exact law of the first emitted token: sum over root probe identities s of
    q~(s) * P(token | s), where P(token | s) follows the accept probabilities of
    the oracle's level thresholds (reach probabilities multiply)."""
    V = rows.shape[1]
    p_full = O.target_probs(target_root, p.temperature)
    ex0 = O.expand_row(rows[0], p, 0.5)
    law = np.zeros(V)
    tail_mass = 0.0
    for s in range(p.m, len(ex0.q)):
        wgt = ex0.qT[s] / ex0.zT
        if wgt == 0.0:
            continue
        tail_mass += wgt
        # a u_probe inside rank s's CDF interval draws probe s
        cum = np.cumsum(ex0.qT[p.m:])
        lo = cum[s - p.m - 1] if s > p.m else 0.0
        u0 = (lo + cum[s - p.m]) / 2.0 / ex0.zT
        u = u_rest.copy()
        u[0] = u0
        t = O.build(rows, u, p)
        assert t.expansions[0].probe_pos == s
        kids = O.children_in_order(t, 0, mode)
        steps, w, Zr = O.level_thresholds(p_full, t.expansions[0], p.m, [int(t.token[j]) for j in kids],
                                          [int(t.kind[j]) for j in kids], mode)
        reach = 1.0
        for kind, x, a, _, _ in steps:
            law[x] += wgt * reach * a
            reach *= (1.0 - a)
        if Zr > 0:
            law += wgt * reach * w / Zr
    assert tail_mass == pytest.approx(1.0, abs=1e-12)
    return law, p_full


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("R,m,T", [(8, 1, 1.0), (2, 1, 1.0), (3, 2, 0.7), (8, 0, 1.4), (1, 1, 1.0)])
def test_losslessness_exact_first_token(seed, R, m, T):
    """Summed over probe identities, the first emitted token has law p exactly (Key design 3)."""
    p = O.Params(K=4, m=m, W=4, depth=3, R=R, temperature=T)
    n_rows = 1 + (p.depth - 1) * p.W
    rows = _tiny_rows(300 + seed, n_rows)
    u_rest = np.random.default_rng(seed).random(n_rows)
    target = WL.to_numpy_f64(WL.latent_rows((seed, "tgt"), 1, 32, 1.2, 0.5))[0]
    law, p_full = _first_token_law(rows, u_rest, p, target)
    np.testing.assert_allclose(law, p_full, atol=1e-12, rtol=0)


@pytest.mark.parametrize("m,T", [(1, 1.0), (0, 0.8), (2, 1.3)])
def test_losslessness_exact_first_token_dense_support(m, T):
    """The dense support (|S| = V = 300, a tail reaching past rank 128): summed over probe identities,
    the first emitted token has law p exactly (Key design 1's dense row with Key design 3)."""
    p = O.Params(K=4, m=m, W=4, depth=2, R=6, temperature=T, support=1 << 30)
    n_rows = 1 + (p.depth - 1) * p.W
    rows = _tiny_rows(500 + m, n_rows, V=300)
    u_rest = np.random.default_rng(m).random(n_rows)
    target = WL.to_numpy_f64(WL.latent_rows((m, "tgt-dense"), 1, 300, 1.2, 0.5))[0]
    ex = O.expand_row(rows[0], p, 0.5)
    assert len(ex.sup_id) == 300 and ex.qT[128:].sum() > 1e-3
    law, p_full = _first_token_law(rows, u_rest, p, target)
    np.testing.assert_allclose(law, p_full, atol=1e-12, rtol=0)


def test_rrsw_without_fillers_is_lossless():
    """Probe-last (RRSw schedule) is a valid sampler when the candidates do not depend on the probe.

    With K = m + 1 there are no fillers, so the one-hot stage sees a fixed
    candidate set and the probe, verified last against the renormalised
    remainder, is an ordinary rejection step.  (With fillers the candidate set
    depends on the probe identity and the probe-last schedule is not a valid
    sampler; the pages compare the schedules on the deterministic-prefix case.)
    """
    for seed in range(6):
        for m in (1, 2):
            p = O.Params(K=m + 1, m=m, W=m + 1, depth=1, R=m + 1, temperature=1.0)
            rows = _tiny_rows(400 + seed, 1)
            target = WL.to_numpy_f64(WL.latent_rows((seed, "tgt2"), 1, 32, 1.2, 0.5))[0]
            law_r, p_full = _first_token_law(rows, np.zeros(1), p, target, "rheo")
            law_s, _ = _first_token_law(rows, np.zeros(1), p, target, "rrsw")
            np.testing.assert_allclose(law_r, p_full, atol=1e-12)
            np.testing.assert_allclose(law_s, p_full, atol=1e-12)


def _accept_prob_level0(rows, p, target, mode):
    """Exact probability that level 0 accepts some child (not the bonus)."""
    p_full = O.target_probs(target, p.temperature)
    ex0 = O.expand_row(rows[0], p, 0.5)
    total = 0.0
    for s in range(p.m, len(ex0.q)):
        wgt = ex0.qT[s] / ex0.zT
        cum = np.cumsum(ex0.qT[p.m:])
        lo = cum[s - p.m - 1] if s > p.m else 0.0
        t = O.build(rows, np.array([(lo + cum[s - p.m]) / 2.0 / ex0.zT]), p)
        kids = O.children_in_order(t, 0, mode)
        steps, _, _ = O.level_thresholds(p_full, t.expansions[0], p.m, [int(t.token[j]) for j in kids],
                                         [int(t.kind[j]) for j in kids], mode)
        reach = 1.0
        for _, _, a, _, _ in steps:
            total += wgt * reach * a
            reach *= 1.0 - a
    return total


def test_depth1_acceptance_ordering():
    """Probe-first >= probe-last on the same candidates, always (OT dominance, Key design 3).

    The pages' controlled depth-1 experiment also reports one-hot Top-K below
    both (80.0 < 83.5 < 85.4 %); on these synthetic rows the averages keep that order.
    """
    rheo, rrsw, topk = [], [], []
    for seed in range(25):
        rows = _tiny_rows(500 + seed, 1)
        target = WL.to_numpy_f64(WL.latent_rows((seed, "tgt3"), 1, 32, 1.2, 0.5))[0]
        p = O.Params(K=2, m=1, W=2, depth=1, R=2)
        a = _accept_prob_level0(rows, p, target, "rheo")
        b = _accept_prob_level0(rows, p, target, "rrsw")
        assert a >= b - 1e-12
        # one-hot Top-K: the K best tokens, all deterministic: accept mass = sum of p over them
        top = O.support_of(rows[0], 32)[:2]
        c = float(O.target_probs(target, 1.0)[top].sum())
        rheo.append(a), rrsw.append(b), topk.append(c)
    assert np.mean(rheo) >= np.mean(rrsw) >= np.mean(topk) - 0.02


def _independent_onehot_walk(t, target_rows, u_verify, u_bonus, T):
    """Plain one-hot recursive rejection (EAGLE-style, draft prob 1), written independently."""
    node, level, out = 0, 0, []
    while True:
        tt = np.asarray(target_rows[node], dtype=np.float64) / T
        pr = np.exp(tt - tt.max())
        pr /= pr.sum()
        kids = sorted([j for j in range(t.n_nodes) if t.parent[j] == node], key=lambda j: t.slot[j])
        mass = 1.0
        nxt = -1
        for j, c in enumerate(kids):
            x = int(t.token[c])
            if u_verify[level][j] < pr[x] / mass:
                nxt = c
                break
            mass -= pr[x]
            pr[x] = 0.0
        if nxt < 0:
            c = np.cumsum(pr)
            v = int(np.searchsorted(c, u_bonus * mass, side="right"))
            return out, v
        out.append(nxt)
        node, level = nxt, level + 1


def test_no_probe_reduces_to_one_hot_recursive_rejection():
    """Trees where no probe survives verify exactly like one-hot recursive rejection."""
    checked = 0
    for seed in range(40):
        p = O.Params(K=4, m=3, W=2, depth=3, R=5, temperature=1.0)
        n_rows = 1 + (p.depth - 1) * p.W
        rows = _tiny_rows(600 + seed, n_rows)
        rng = np.random.default_rng(seed)
        t = O.build_topr(rows, rng.random(n_rows), p)
        if (t.kind == O.PROBE).any():
            continue
        checked += 1
        target = WL.to_numpy_f64(WL.latent_rows((seed, "tgt4"), t.n_nodes, 32, 1.2, 0.5))
        for trial in range(20):
            uv = rng.random((p.depth, p.K))
            ub = float(rng.random())
            res = O.verify(t, target, uv, ub, p)
            nodes, bonus = _independent_onehot_walk(t, target, uv, ub, 1.0)
            assert res.nodes == nodes and res.tokens[-1] == bonus
    assert checked >= 10


def test_m_equal_k_is_the_one_hot_topk_tree():
    """m = K: K deterministic children (ranks 0..K-1), no probe drawn, one-hot recursive
    rejection in verification, and the first emitted token still has law p exactly."""
    p = O.Params(K=4, m=4, W=2, depth=3, R=12, temperature=1.0)
    n_rows = 1 + (p.depth - 1) * p.W
    for seed in range(8):
        rows = _tiny_rows(700 + seed, n_rows)
        rng = np.random.default_rng(seed)
        t = O.build_topr(rows, rng.random(n_rows), p)
        assert not (t.kind == O.PROBE).any()
        for ex in t.expansions.values():
            assert ex.probe_pos == -1
            assert [(slot, kind, rank) for slot, kind, rank, _, _ in ex.children] == \
                [(k, O.DET, k) for k in range(p.K)]
        target = WL.to_numpy_f64(WL.latent_rows((seed, "tgt7"), t.n_nodes, 32, 1.2, 0.5))
        for trial in range(10):
            uv = rng.random((p.depth, p.K))
            ub = float(rng.random())
            res = O.verify(t, target, uv, ub, p)
            nodes, bonus = _independent_onehot_walk(t, target, uv, ub, 1.0)
            assert res.nodes == nodes and res.tokens[-1] == bonus
        # exact law of the first token at the root
        p_full = O.target_probs(target[0], p.temperature)
        kids = O.children_in_order(t, 0)
        steps, w, Zr = O.level_thresholds(p_full, t.expansions[0], p.m, [int(t.token[j]) for j in kids],
                                          [int(t.kind[j]) for j in kids])
        law, reach = np.zeros_like(p_full), 1.0
        for _, x, a, _, _ in steps:
            law[x] += reach * a
            reach *= 1.0 - a
        law += reach * w / Zr
        np.testing.assert_allclose(law, p_full, atol=1e-12, rtol=0)


# -------------------------------------------------------- multi-level chi^2 ---

def _chi2_pvalue(counts, probs, n):
    from scipy.stats import chi2
    exp = probs * n
    # pool bins with expected < 5
    order = np.argsort(exp)
    obs_b, exp_b = [], []
    acc_o = acc_e = 0.0
    for i in order:
        acc_o += counts[i]
        acc_e += exp[i]
        if acc_e >= 5:
            obs_b.append(acc_o), exp_b.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        if exp_b:
            obs_b[-1] += acc_o
            exp_b[-1] += acc_e
    obs_b, exp_b = np.array(obs_b), np.array(exp_b)
    stat = ((obs_b - exp_b) ** 2 / exp_b).sum()
    return chi2.sf(stat, len(exp_b) - 1)


@pytest.mark.parametrize("seed", [0, 1])
def test_losslessness_chi_square_two_levels(seed):
    """Tiny workload, path-keyed target rows: first token ~ p(root), second ~ p(first)."""
    wl = WL.WORKLOADS["tiny"]
    p = O.Params(K=wl.K, m=wl.m, W=wl.W, depth=wl.depth, R=wl.R, temperature=wl.temperature)
    n_rows = wl.n_exp
    rows = _tiny_rows(700 + seed, n_rows)
    cache = {}

    def row_for(path):
        if path not in cache:
            cache[path] = WL.to_numpy_f64(WL.path_keyed_rows(seed, [path], 32, 1.2, 0.5))[0]
        return cache[path]

    rng = np.random.default_rng(1000 + seed)
    n = 10000
    first = np.zeros(32)
    second = {}
    for _ in range(n):
        t = O.build_topr(rows, rng.random(n_rows), p)
        paths = []
        for i in range(t.n_nodes):
            pth, j = [], i
            while j > 0:
                pth.append(int(t.token[j]))
                j = t.parent[j]
            paths.append(tuple(reversed(pth)))
        target = np.stack([row_for(pt) for pt in paths])
        res = O.verify(t, target, rng.random((p.depth, p.K)), float(rng.random()), p)
        first[res.tokens[0]] += 1
        if res.accept_len >= 1:
            second.setdefault(res.tokens[0], np.zeros(32))
            second[res.tokens[0]][res.tokens[1]] += 1
    pv = _chi2_pvalue(first, O.target_probs(row_for(()), 1.0), n)
    assert pv > 1e-3
    v, c = max(second.items(), key=lambda kv: kv[1].sum())
    pv2 = _chi2_pvalue(c, O.target_probs(row_for((v,)), 1.0), int(c.sum()))
    assert pv2 > 1e-3


def test_topr_frontiers_are_the_expanded_nodes():
    """Each recorded frontier has min(W, layer size) entries; every kept node expanded from
    draft row 1 + (d-1)W + r is entry r of the frontier of layer d, with its parent's rank."""
    rng = np.random.default_rng(3)
    p = O.Params(K=3, m=1, W=4, depth=4, R=200)
    n_rows = 1 + (p.depth - 1) * p.W
    rows = rng.normal(size=(n_rows, 50)) * 2.0
    t = O.build(rows, rng.random(n_rows), p)
    sizes, ln = [], p.K
    for _ in range(1, p.depth):
        sizes.append(min(ln, p.W))
        ln = min(ln, p.W) * p.K
    assert [len(f) for f in t.frontiers] == sizes
    # R covers every candidate, so every frontier node is kept
    assert t.n_nodes == 1 + t.n_candidates
    seen = 0
    for i in range(1, t.n_nodes):
        if t.exp_row[i] < 0:
            continue
        d = int(t.depth[i])
        r = int(t.exp_row[i]) - (1 + (d - 1) * p.W)
        tok, prank = t.frontiers[d - 1][r]
        assert tok == t.token[i]
        par = int(t.parent[i])
        assert prank == (-1 if d == 1 else int(t.exp_row[par]) - (1 + (d - 2) * p.W))
        seen += 1
    assert seen == sum(sizes)


def _separated_rows(seed, n_rows, V=40, gap=0.6):
    """Rows whose sorted logits are gap apart (a random permutation of 0, gap, 2 gap, ...)."""
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(V).astype(np.float64) * gap for _ in range(n_rows)])


def _tree_sig(t):
    return t.token.tolist(), t.parent.tolist(), t.depth.tolist()


@pytest.mark.parametrize("seed", range(4))
def test_cold_limit_m0_is_the_topk_tree(seed):
    """T -> 0 with m = 0: the probe is always the top token (the tempered tail
    collapses on rank 0), so sampling and structure both reduce to Top-K."""
    kw = dict(K=4, W=3, depth=3, R=10)
    n_rows = 1 + (kw["depth"] - 1) * kw["W"]
    rows = _separated_rows(seed, n_rows)
    topk = O.build_topr(rows, np.full(n_rows, 0.5), O.Params(m=4, temperature=0.02, **kw))
    for u in (0.0, 0.37, 0.999):
        t = O.build_topr(rows, np.full(n_rows, u), O.Params(m=0, temperature=0.02, **kw))
        for ex in t.expansions.values():
            assert ex.probe_pos == 0
        assert _tree_sig(t) == _tree_sig(topk)


@pytest.mark.parametrize("seed", range(4))
def test_cold_limit_m1_keeps_a_proxy_difference(seed):
    """T -> 0 with m = 1: the probe is always the second token, so the children are
    Top-K's tokens, but the probe carries min(q(x_1), z) instead of q(x_2): the
    small structural difference from Top-K that the pages describe."""
    kw = dict(K=4, W=3, depth=3, R=10)
    n_rows = 1 + (kw["depth"] - 1) * kw["W"]
    rows = _separated_rows(seed, n_rows)
    p = O.Params(m=1, temperature=0.02, **kw)
    t = O.build_topr(rows, np.full(n_rows, 0.5), p)
    for e, ex in t.expansions.items():
        assert ex.probe_pos == 1
        order = np.argsort(-rows[e], kind="stable")
        assert [tok for _, _, _, tok, _ in ex.children] == order[:kw["K"]].tolist()
        lp_probe = [lp for _, kind, _, _, lp in ex.children if kind == O.PROBE][0]
        assert lp_probe == pytest.approx(min(ex.q[0], ex.z), rel=1e-15)
        assert lp_probe > ex.q[1]


def test_cold_limit_underflow_draws_no_probe():
    """Reading: once the tempered tail weight underflows (T = 1e-4 with gaps of
    0.6), there is no tail mass to sample, no probe is drawn, and m = 1 builds
    exactly the Top-K tree."""
    kw = dict(K=4, W=3, depth=3, R=10)
    n_rows = 1 + (kw["depth"] - 1) * kw["W"]
    rows = _separated_rows(9, n_rows)
    t1 = O.build_topr(rows, np.full(n_rows, 0.5), O.Params(m=1, temperature=1e-4, **kw))
    tk = O.build_topr(rows, np.full(n_rows, 0.5), O.Params(m=4, temperature=1e-4, **kw))
    for ex in t1.expansions.values():
        assert ex.zT == 0.0 and ex.probe_pos == -1
    assert _tree_sig(t1) == _tree_sig(tk)
    assert np.array_equal(t1.score, tk.score)
