"""Plain float64 CPU oracle for stochastic dynamic-tree speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The library (the CUDA path) never calls it,
and this module imports nothing from the library.

It restates, step by step and in float64, what the pages define:

* RheoSampling ("RheoSampling: Resolving the One-Hot Dilemma in Stochastic
  Dynamic-Tree Speculative Decoding", NeurIPS 2026 notes):
  - Method / Key design 1: top-128 truncation of the draft logits before the
    softmax;
  - Method / Key design 2: dual-identity expansion (top-m deterministic
    children, one probe from the renormalised tail carrying the proxy
    probability min{q(x_m), z}, q(x_1)+eps when m=0, fillers), with the
    Local Ranking Preservation lemma;
  - Method / overall framework + flowchart: cumulative path scores, global
    top-R pruning (expand-then-rerank, EAGLE-2/3 style);
  - Method / Key design 3: optimal-transport verification (probe first with
    min(1, p/q~), residual norm(max(0, p - q~)), recursive rejection of the
    remaining candidates, bonus token from the final residual);
  - the training-strategy paragraph: construction and pruning use the
    untempered draft probabilities, probe sampling and verification use T.
* SMART ("SMART: When is it Actually Worth Expanding a Speculative Tree?",
  ECCV 2026 notes), Method / Key designs 1-3 and the flowchart: the
  marginal-gain keep rule with the draft cost model lambda*|T| + beta and the
  verify cost model gamma*(exp(delta*|T|^rho) - 1) + eta.

Readings where the pages are silent or ambiguous are listed with the design
notes of the repository; each one is repeated at the point of use below.

Every decision that floating point takes (a sample from a CDF, an accept test,
a ranking comparison, a SMART keep test) also records its margin, so that a
comparison against another implementation can tell near-ties from errors.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

ROOT, DET, PROBE, FILL = 0, 1, 2, 3

# Decision margins below these values are near-ties (see `Margins`).
MASS_MARGIN = 1e-6      # |u - ratio| of an accept test; |u * Z - cumulative mass| / Z of a CDF draw
SCORE_MARGIN = 1e-5     # relative gap between two compared path scores
SMART_MARGIN = 1e-5     # |lhs - rhs| / rhs of the SMART keep test


@dataclasses.dataclass
class Params:
    K: int
    m: int
    W: int
    depth: int
    R: int
    temperature: float = 1.0
    support: int = 128
    builder: str = "topr"     # "topr" | "smart"
    lam: float = 0.02
    beta: float = 0.0
    gamma: float = 0.5
    delta: float = 0.01
    rho: float = 1.3
    eta: float = 0.0
    alpha: float = 1.0
    smart_paths: str = "leaves"   # "leaves" (|P| = #leaves) | "one" (|P| = 1)


class Margins:
    """Smallest margin seen per decision kind, the count of near-ties, and where each one sits.

    `ties` lists every near-tie as (kind, where, margin).  `where` names the
    decision: ("probe", row) for a probe draw, ("order", layer, i) for the gap
    between positions i and i+1 of a ranked layer (layer "final" for the top-R
    cut), ("smart", layer, creation key) for a keep test, ("accept", level, j)
    for the j-th accept test of a verification level, ("bonus", level) for the
    bonus draw.
    """

    def __init__(self):
        self.min = {}
        self.near = 0
        self.ties = []

    def add(self, kind: str, value: float, threshold: float, where=None):
        value = abs(float(value))
        if kind not in self.min or value < self.min[kind]:
            self.min[kind] = value
        if value < threshold:
            self.near += 1
            self.ties.append((kind, where, value))

    def merge(self, other: "Margins"):
        for k, v in other.min.items():
            if k not in self.min or v < self.min[k]:
                self.min[k] = v
        self.near += other.near
        self.ties.extend(other.ties)


class ReplayRefused(AssertionError):
    """A decision offered for replay was not a near-tie of this oracle."""


@dataclasses.dataclass
class Replay:
    """Decisions adopted from another implementation (the replay mode of a parity check).

    Where two implementations take a floating-point decision on opposite sides
    of a near-tie, the oracle can adopt the other side's choice and go on, so
    that everything downstream is still compared.  It adopts a choice only
    where its own margin for that decision is a near-tie (below the thresholds
    above) and raises ReplayRefused otherwise:

      probe[row]          = probe rank drawn for a draft row;
      before              = set of (a, b) creation keys, a ranked before b;
      keep[key]           = SMART keep decision of a candidate;
      accept[(level, j)]  = outcome of the j-th accept test of a level;
      bonus[level]        = bonus token drawn at a level.

    `adopted` lists the decisions that changed the oracle's result.
    """
    probe: dict = dataclasses.field(default_factory=dict)
    before: set = dataclasses.field(default_factory=set)
    keep: dict = dataclasses.field(default_factory=dict)
    accept: dict = dataclasses.field(default_factory=dict)
    bonus: dict = dataclasses.field(default_factory=dict)
    adopted: list = dataclasses.field(default_factory=list)

    def __bool__(self):
        return bool(self.probe or self.before or self.keep or self.accept or self.bonus)


# --------------------------------------------------------------------------
# Inputs
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bfloat16 bit patterns (uint16)."""
    u32 = bits.astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def as_f64(row) -> np.ndarray:
    a = np.asarray(row)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


# --------------------------------------------------------------------------
# Draft side: truncation, softmaxes, dual-identity expansion
# --------------------------------------------------------------------------

def support_of(row: np.ndarray, size: int) -> np.ndarray:
    """Top-|S| truncation (RheoSampling, Key design 1).

    The support S is the first |S| token ids when the row is ordered by logit
    descending, ties by token id ascending (a stable sort of -logit).  NaN
    logits sort last.
    """
    return np.argsort(-row, kind="stable")[:size]


def truncated_softmax(l_sorted: np.ndarray, temperature: float):
    """q over S at T=1 and q_T over S at temperature T (RheoSampling, Key design 1).

    Logits outside S are -inf, so both vanish there.  Returns the unnormalised
    weights too (e = exp(l - l_max), e_T = exp((l - l_max)/T)).
    """
    lmax = l_sorted[0]
    e = np.exp(l_sorted - lmax)
    eT = np.exp((l_sorted - lmax) / temperature)
    return e / e.sum(), eT / eT.sum(), e, eT


@dataclasses.dataclass
class Expansion:
    sup_id: np.ndarray      # [S] token ids in rank order
    q: np.ndarray           # [S] untempered truncated softmax
    qT: np.ndarray          # [S] tempered truncated softmax
    z: float                # untempered tail mass (ranks m..S-1)
    zT: float               # tempered tail mass
    probe_pos: int          # rank of the probe in S, -1 if there is none
    children: list          # [(slot, kind, rank, token, local_prob)]
    margins: Margins


def _draw_accepts(cum: np.ndarray, weights: np.ndarray, target: float, k: int, total: float) -> bool:
    """Whether index k is a choice of the inverse-CDF draw `target` = u * total within the near-tie margin.

    k is a valid choice of another implementation when its own cumulative
    interval [cum[k-1], cum[k]) holds the target up to MASS_MARGIN * total
    and its weight is positive.
    """
    if not 0 <= k < cum.shape[0] or not weights[k] > 0.0:
        return False
    lo = cum[k - 1] if k > 0 else 0.0
    return lo - MASS_MARGIN * total <= target < cum[k] + MASS_MARGIN * total


def expand_row(row, p: Params, u_probe: float, force_probe_pos: Optional[int] = None,
               row_index=None, replay: Optional[Replay] = None) -> Expansion:
    """Dual-identity expansion of one draft row (RheoSampling, Key design 2).

    * x_1..x_m: the m highest-q tokens (ranks 0..m-1), kind DET.
    * tail = ranks m..|S|-1; z = sum of q over the tail.  The pages write
      z = 1 - sum_{i<=m} q(x_i); the sum over the tail is the same number in
      exact arithmetic and keeps the lemma exact in floating point.
    * probe x_s ~ q~_T = q_T / z_T over the tail (tempered: the probe is
      sampled at T): the first tail rank k, in rank order, with
      u * z_T < sum_{j<=k} q_T(x_j).  If rounding leaves no such k, the last
      tail token of positive weight is taken.  No probe if the tail is empty
      or has zero tempered weight.
    * proxy = min{q(x_m), z} for m >= 1, and q(x_1) + eps (one ulp) for m = 0.
    * fillers: the next tail tokens in rank order, skipping x_s, until the
      node has min(K, |S|) children.
    * m = K is the one-hot Top-K node (the pages' Top-K baseline): K
      deterministic children and no probe (none is drawn).
    * slots: DET 0..m-1, PROBE m, FILL after; local probability q(child)
      (untempered), the proxy for the probe.

    `force_probe_pos` replaces the sampled probe by a given tail rank (used
    only to enumerate probe identities exactly).  `row_index` locates the
    draw's near-tie; `replay.probe[row_index]` adopts another implementation's
    probe rank where the draw is a near-tie.
    """
    row = as_f64(row)
    V = row.shape[0]
    S = min(p.support, V)
    if p.K > S or p.m > p.K or p.m < 0:
        raise ValueError("need 0 <= m <= K <= |S|")
    sup = support_of(row, S)
    l = row[sup]
    q, qT, _, _ = truncated_softmax(l, p.temperature)
    m = p.m
    z = float(q[m:].sum())
    zT = float(qT[m:].sum())
    mg = Margins()
    probe_pos = -1
    if m < p.K and m < S and zT > 0.0:
        if force_probe_pos is not None:
            probe_pos = int(force_probe_pos)
            assert m <= probe_pos < S and qT[probe_pos] > 0
        else:
            target = u_probe * zT
            cum = np.cumsum(qT[m:])
            k = int(np.searchsorted(cum, target, side="right"))  # first k with target < cum[k]
            if k >= cum.shape[0]:
                k = int(np.nonzero(qT[m:] > 0)[0][-1])
            probe_pos = m + k
            lo = cum[k - 1] if k > 0 else 0.0
            mg.add("probe_sample", min(target - lo, cum[k] - target) / zT, MASS_MARGIN, ("probe", row_index))
            if replay is not None and row_index in replay.probe and replay.probe[row_index] != probe_pos:
                other = int(replay.probe[row_index])
                if not _draw_accepts(cum, qT[m:], target, other - m, zT):
                    raise ReplayRefused(f"probe of row {row_index}: rank {other} is not a near-tie of {probe_pos}")
                probe_pos = other
                replay.adopted.append(("probe", row_index))
    children = []
    for s in range(m):
        children.append((s, DET, s, int(sup[s]), float(q[s])))
    if probe_pos >= 0:
        proxy = min(float(q[m - 1]), z) if m >= 1 else float(np.nextafter(q[0], np.inf))
        children.append((m, PROBE, probe_pos, int(sup[probe_pos]), proxy))
    fillers = [k for k in range(m, S) if k != probe_pos]
    need = min(p.K, S) - len(children)
    for k in fillers[:need]:
        children.append((len(children), FILL, k, int(sup[k]), float(q[k])))
    return Expansion(sup, q, qT, z, zT, probe_pos, children, mg)


# --------------------------------------------------------------------------
# Tree building
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Tree:
    token: np.ndarray       # [n] (root = -1)
    parent: np.ndarray      # [n] canonical index of the parent (root = -1)
    depth: np.ndarray
    kind: np.ndarray
    slot: np.ndarray
    exp_row: np.ndarray     # draft row expanded for the node, -1 if none
    score: np.ndarray       # cumulative path score (proxy for probes)
    expansions: dict        # draft row -> Expansion
    margins: Margins
    n_candidates: int
    # top-R builder: for each layer d < D, its frontier in rank order as
    # (token, rank of the parent in the previous frontier, -1 for the root)
    frontiers: list = dataclasses.field(default_factory=list)
    # SMART builder: every keep test in the order taken, as a dict with the
    # candidate's layer, token path, score and the state (n, L, |P|) it saw,
    # lhs, rhs and the decision
    trace: list = dataclasses.field(default_factory=list)

    @property
    def n_nodes(self) -> int:
        return int(self.token.shape[0])


class _Cand:
    __slots__ = ("depth", "parent", "prank", "slot", "kind", "token", "score", "exp_row", "idx")

    def __init__(self, depth, parent, prank, slot, kind, token, score):
        self.depth, self.parent, self.prank, self.slot = depth, parent, prank, slot
        self.kind, self.token, self.score = kind, token, score
        self.exp_row = -1
        self.idx = -1

    def key(self):
        """Ranking key: score descending, then creation index (depth, parent rank, slot).

        The token id never enters the key, so a probe's survival cannot depend
        on which token it drew (RheoSampling, Key design 2).
        """
        return (-self.score, self.depth, self.prank, self.slot)

    def ckey(self):
        """Creation index (depth, parent's rank in its frontier, slot)."""
        return (self.depth, self.prank, self.slot)

    def path(self):
        """Token path from the root's first child down to this candidate."""
        out, c = [], self
        while c.parent is not None:
            out.append(c.token)
            c = c.parent
        return tuple(reversed(out))


def _ranked(cands: Sequence[_Cand], replay: Optional[Replay], where) -> List[_Cand]:
    """Candidates in ranking-key order; with a replay, adopted near-tie orders applied.

    replay.before holds (a, b) creation-key pairs that another implementation
    ranked a before b.  Such a pair is adopted only when the two path scores
    differ, by at most SCORE_MARGIN (relative): equal scores are ordered by the
    creation index everywhere.
    """
    ordered = sorted(cands, key=_Cand.key)
    if not replay or not replay.before:
        return ordered
    import functools

    def cmp(a, b):
        ka, kb = a.ckey(), b.ckey()
        flip = (ka, kb) in replay.before or (kb, ka) in replay.before
        natural = -1 if a.key() < b.key() else (1 if a.key() > b.key() else 0)
        if not flip:
            return natural
        want = -1 if (ka, kb) in replay.before else 1
        if want != natural:
            # equal scores are ordered by the creation index on every implementation
            gap = abs(a.score - b.score)
            if not 0.0 < gap <= SCORE_MARGIN * max(a.score, b.score):
                raise ReplayRefused(f"order of {ka} and {kb} at {where}: scores {a.score} and {b.score}")
        return want
    out = sorted(cands, key=functools.cmp_to_key(cmp))
    if [c.ckey() for c in out] != [c.ckey() for c in ordered]:
        replay.adopted.append(("order", where))
    return out


def _record_order_margins(ordered: Sequence[_Cand], upto: int, mg: Margins, layer=None):
    """Relative gaps of adjacent scores in a ranked list, over the first `upto`+1 items.

    Exact ties (gap 0) are structural (equal logits under one parent, or a
    proxy equal to q(x_m)) and are broken by the creation index on any
    implementation, so they are not near-ties.
    """
    n = min(len(ordered) - 1, upto)
    for i in range(n):
        a, b = ordered[i].score, ordered[i + 1].score
        if a > 0 and a != b:
            mg.add("rank", (a - b) / a, SCORE_MARGIN, ("order", layer, i))


def _expand(rows, u_probe, p, row_idx, cache, mg, replay=None):
    if row_idx not in cache:
        if row_idx >= len(rows):
            raise ValueError(f"tree needs draft row {row_idx} but only {len(rows)} were given")
        ex = expand_row(rows[row_idx], p, float(u_probe[row_idx]), row_index=row_idx, replay=replay)
        mg.merge(ex.margins)
        cache[row_idx] = ex
    return cache[row_idx]


def _children(parent: _Cand, prank: int, ex: Expansion, depth: int) -> List[_Cand]:
    return [_Cand(depth, parent, prank, slot, kind, tok, parent.score * lp)
            for (slot, kind, _rank, tok, lp) in ex.children]


def _emit(selected: List[_Cand], root: _Cand, cache: dict, mg: Margins, n_cand: int,
          replay: Optional[Replay] = None) -> Tree:
    """Canonical order: root, then depth ascending, then ranking key."""
    depths = sorted({c.depth for c in selected})
    nodes = [root] + [c for d in depths
                      for c in _ranked([x for x in selected if x.depth == d], replay, ("canonical", d))]
    for i, c in enumerate(nodes):
        c.idx = i
    n = len(nodes)
    tree = Tree(token=np.full(n, -1, np.int64), parent=np.full(n, -1, np.int64),
                depth=np.zeros(n, np.int64), kind=np.zeros(n, np.int64),
                slot=np.full(n, -1, np.int64), exp_row=np.full(n, -1, np.int64),
                score=np.zeros(n, np.float64), expansions=cache, margins=mg, n_candidates=n_cand)
    for i, c in enumerate(nodes):
        tree.token[i] = c.token
        tree.parent[i] = -1 if c.parent is None else c.parent.idx
        if c.parent is not None and c.parent.idx < 0:
            raise AssertionError("pruned tree is not ancestor-closed")
        tree.depth[i] = c.depth
        tree.kind[i] = c.kind
        tree.slot[i] = c.slot
        tree.exp_row[i] = c.exp_row
        tree.score[i] = c.score
    return tree


def _new_root():
    root = _Cand(0, None, 0, -1, ROOT, -1, 1.0)
    root.exp_row = 0
    return root


def build_topr(rows, u_probe, p: Params, replay: Optional[Replay] = None) -> Tree:
    """Expand-then-rerank tree with global top-R pruning (RheoSampling, overall framework).

    Layer d = 1..D: the candidates are the children of every frontier node of
    layer d-1 (the root for d = 1), scored by parent score x local probability.
    For d < D the frontier of layer d is its top-W candidates by the ranking
    key; frontier rank r of layer d is expanded from draft row 1 + (d-1)*W + r.
    After layer D the whole candidate set is cut to its top-R by the same key
    (R counts draft nodes; the root is kept in addition).  Because a child's
    score never exceeds its parent's and ties go to the shallower node, the
    top-R set is ancestor-closed.

    `replay` (optional) adopts another implementation's choices at near-ties.
    """
    mg = Margins()
    cache = {}
    root = _new_root()
    frontier = [root]
    frontiers = []
    allc: List[_Cand] = []
    for d in range(1, p.depth + 1):
        layer = []
        for prank, node in enumerate(frontier):
            ex = _expand(rows, u_probe, p, node.exp_row, cache, mg, replay)
            layer.extend(_children(node, prank, ex, d))
        allc.extend(layer)
        if d < p.depth:
            _record_order_margins(sorted(layer, key=_Cand.key), p.W, mg, d)
            ordered = _ranked(layer, replay, ("frontier", d))
            frontier = ordered[:p.W]
            for r, c in enumerate(frontier):
                c.exp_row = 1 + (d - 1) * p.W + r
            frontiers.append([(c.token, -1 if d == 1 else c.prank) for c in frontier])
    _record_order_margins(sorted(allc, key=_Cand.key), p.R, mg, "final")
    ordered = _ranked(allc, replay, ("final",))
    tree = _emit(ordered[:p.R], root, cache, mg, len(allc), replay)
    tree.frontiers = frontiers
    return tree


def smart_cost(n: float, p: Params) -> float:
    """C(n) = c_T + C_draft + C_verify in units of one target step (SMART, Key designs 1-2).

    Reading: the denominator of the speedup R(T) includes the target step that
    runs anyway (c_T = 1), so an empty tree has R = 1.  The literal ratio with
    beta = eta = 0 is 0/0 at the empty tree and keeps no node.
    """
    return 1.0 + p.lam * n + p.beta + p.gamma * (math.exp(p.delta * n ** p.rho) - 1.0) + p.eta


def smart_marginal_cost(n: float, p: Params) -> float:
    """dC/dn = lambda + gamma*delta*rho*n^(rho-1)*exp(delta*n^rho) (SMART, Key design 3).

    The n^(rho-1) term is taken as 0 at n = 0 (rho > 1).
    """
    powterm = 0.0 if n == 0 else p.rho * n ** (p.rho - 1.0)
    return p.lam + p.gamma * p.delta * powterm * math.exp(p.delta * n ** p.rho)


def smart_keep(P_u: float, n: int, L: float, paths: int, p: Params):
    """Keep test alpha * dL(u)/dC(n) > L/C(n), dL(u) = P(u)/|P| (SMART, Key design 3).

    Returns (keep, lhs, rhs).
    """
    lhs = p.alpha * (P_u / paths) / smart_marginal_cost(n, p)
    rhs = L / smart_cost(n, p)
    return lhs > rhs, lhs, rhs


def build_smart(rows, u_probe, p: Params, replay: Optional[Replay] = None) -> Tree:
    """Layer-wise greedy SMART builder over dual-identity children (SMART, flowchart + Key design 3).

    State: n = kept draft nodes, L = 1 + sum of kept P(v) (expected accepted
    length), |P| = number of leaves (1 for the root-only tree).  Layer l: the
    candidates are the children of every kept node of layer l-1, visited in
    descending ranking key; each is kept iff the keep test holds and n < R
    (the budget).  After a keep, n and L grow and |P| grows by one unless the
    parent was still a leaf.  Building stops when a layer keeps nothing, the
    budget is reached or l = D; otherwise the kept nodes of the layer are
    expanded in key order from the next draft rows (1, 2, ...).

    Every keep test is recorded in `Tree.trace`.  `replay` (optional) adopts
    another implementation's choices at near-ties.
    """
    mg = Margins()
    trace = []
    cache = {}
    root = _new_root()
    active = [root]
    has_child = {id(root): False}
    n, L, paths = 0, 1.0, 1
    kept: List[_Cand] = []
    next_row = 1
    n_cand = 0
    for d in range(1, p.depth + 1):
        layer = []
        for prank, node in enumerate(active):
            ex = _expand(rows, u_probe, p, node.exp_row, cache, mg, replay)
            layer.extend(_children(node, prank, ex, d))
        n_cand += len(layer)
        _record_order_margins(sorted(layer, key=_Cand.key), len(layer), mg, d)
        layer = _ranked(layer, replay, ("layer", d))
        kept_layer = []
        for c in layer:
            if n >= p.R:
                break
            P_paths = paths if p.smart_paths == "leaves" else 1
            keep, lhs, rhs = smart_keep(c.score, n, L, P_paths, p)
            if rhs > 0:
                mg.add("smart", (lhs - rhs) / rhs, SMART_MARGIN, ("smart", d, c.ckey()))
            if replay is not None and c.ckey() in replay.keep and replay.keep[c.ckey()] != keep:
                if not (rhs > 0 and abs(lhs - rhs) < SMART_MARGIN * rhs):
                    raise ReplayRefused(f"keep test of {c.ckey()}: lhs {lhs} rhs {rhs}")
                keep = replay.keep[c.ckey()]
                replay.adopted.append(("smart", d, c.ckey()))
            trace.append(dict(layer=d, path=c.path(), score=c.score, n=n, L=L, paths=P_paths,
                              lhs=lhs, rhs=rhs, keep=bool(keep)))
            if keep:
                n += 1
                L += c.score
                if has_child.get(id(c.parent), False):
                    paths += 1
                has_child[id(c.parent)] = True
                has_child[id(c)] = False
                kept_layer.append(c)
        kept.extend(kept_layer)
        if not kept_layer or n >= p.R or d == p.depth:
            break
        for c in kept_layer:
            c.exp_row = next_row
            next_row += 1
        active = kept_layer
    tree = _emit(kept, root, cache, mg, n_cand, replay)
    tree.trace = trace
    return tree


def build(rows, u_probe, p: Params, replay: Optional[Replay] = None) -> Tree:
    """Build one tree from its draft rows [n_rows][V] and probe uniforms [n_rows]."""
    if p.builder == "smart":
        return build_smart(rows, u_probe, p, replay)
    return build_topr(rows, u_probe, p, replay)


# --------------------------------------------------------------------------
# Target side: verification
# --------------------------------------------------------------------------

def target_probs(row, temperature: float) -> np.ndarray:
    """p = softmax(t / T) over the full vocabulary."""
    t = as_f64(row)
    e = np.exp((t - t.max()) / temperature)
    return e / e.sum()


def children_in_order(tree: Tree, node: int, mode: str = "rheo") -> List[int]:
    """Children of a node in verification order.

    rheo: probe first, then the others by slot (DET then FILL, rank order).
    rrsw: deterministic / filler children by slot first, probe last.
    """
    kids = [int(j) for j in np.nonzero(tree.parent == node)[0]]
    kids.sort(key=lambda j: int(tree.slot[j]))
    probes = [j for j in kids if tree.kind[j] == PROBE]
    others = [j for j in kids if tree.kind[j] != PROBE]
    return probes + others if mode == "rheo" else others + probes


def tail_q_tilde(ex: Expansion, m: int, V: int) -> np.ndarray:
    """q~_T(v) = q_T(v) / z_T for v in the tail (ranks m..|S|-1), else 0 (Key design 2)."""
    qt = np.zeros(V)
    if ex.zT > 0:
        qt[ex.sup_id[m:]] = ex.qT[m:] / ex.zT
    return qt


def level_thresholds(p_full: np.ndarray, ex: Optional[Expansion], m: int, kids_tokens: Sequence[int],
                     kids_kinds: Sequence[int], mode: str = "rheo"):
    """The accept probabilities one verification level offers, in order (Key design 3).

    Returns a list of (kind, token, accept_probability_given_reached, w_before, Zr_before)
    and the final (w, Zr) after every candidate is rejected.  This is the
    closed-form law used both by `verify` (which draws each decision with a
    uniform) and by exact enumeration.

    rheo: probe first with min(1, p/q~); on rejection the residual
      w = max(0, p - q~) (w = p off the tail) with mass Zr = 1 - sum min(p, q~);
      then each remaining child x is a one-hot draft: accept with w(x)/Zr,
      else Zr -= w(x), w(x) = 0.  Without a probe w = p, Zr = 1.
    rrsw: one-hot children first under w = p, probe last with
      min(1, (w/Zr)/q~), residual norm(max(0, w/Zr - q~)).
    """
    V = p_full.shape[0]
    steps = []
    w = p_full.copy()
    Zr = 1.0
    qt = tail_q_tilde(ex, m, V) if ex is not None else None

    def probe_step(w, Zr):
        x = kids_tokens[0] if mode == "rheo" else kids_tokens[-1]
        ratio = (w[x] / Zr) / qt[x]
        a = min(1.0, ratio)
        steps.append((PROBE, x, a, w.copy(), Zr))
        wn = np.maximum(0.0, w / Zr - qt)
        Zn = 1.0 - float(np.minimum(w / Zr, qt).sum())
        return wn, Zn

    order = list(zip(kids_kinds, kids_tokens))
    if mode == "rheo" and order and order[0][0] == PROBE:
        w, Zr = probe_step(w, Zr)
        order = order[1:]
    tail_probe = mode == "rrsw" and order and order[-1][0] == PROBE
    for kind, x in (order[:-1] if tail_probe else order):
        if Zr <= 0.0:
            break
        a = w[x] / Zr
        steps.append((kind, x, a, w.copy(), Zr))
        Zr -= w[x]
        w[x] = 0.0
    if tail_probe and Zr > 0.0:
        w, Zr = probe_step(w, Zr)
    return steps, w, Zr


@dataclasses.dataclass
class VerifyResult:
    accept_len: int
    tokens: List[int]         # accepted tokens then the bonus token
    nodes: List[int]          # accepted node indices (the bonus has none)
    margins: Margins
    residual_empty: bool = False


def verify(tree: Tree, target_rows, u_verify, u_bonus: float, p: Params, mode: str = "rheo",
           replay: Optional[Replay] = None) -> VerifyResult:
    """Layer-by-layer verification of one tree (RheoSampling, Key design 3).

    From the root: p = softmax(t/T) of the node's target row over the full
    vocabulary.  The j-th decision at level l (the node's depth) uses
    u_verify[l][j] and accepts iff u < its accept probability (strict).  An
    accepted child becomes the node and the walk goes on.  When every child
    is rejected, or the node has none, the bonus token is the first token in
    id order with u_bonus * Zr < sum_{v' <= v} w(v'), and the walk ends.
    If rounding leaves the residual mass Zr <= 0, the bonus is drawn from p
    and `residual_empty` is set.

    `replay` (optional) adopts another implementation's accept outcomes
    (replay.accept[(level, j)]) and bonus tokens (replay.bonus[level]) where
    the decision is a near-tie.
    """
    mg = Margins()
    node, level = 0, 0
    toks, nodes = [], []
    empty = False
    while True:
        p_full = target_probs(target_rows[node], p.temperature)
        kids = children_in_order(tree, node, mode)
        accepted = -1
        if kids:
            ex = tree.expansions[int(tree.exp_row[node])]
            steps, w, Zr = level_thresholds(p_full, ex, p.m, [int(tree.token[j]) for j in kids],
                                            [int(tree.kind[j]) for j in kids], mode)
            for j, (kind, x, a, w_before, Z_before) in enumerate(steps):
                u = float(u_verify[level][j])
                # the near-tie margin of an accept test is |u - ratio|
                if kind == PROBE:
                    qt = tail_q_tilde(ex, p.m, p_full.shape[0])[x]
                    margin = u - (w_before[x] / Z_before) / qt
                else:
                    margin = u - w_before[x] / Z_before
                mg.add("accept", margin, MASS_MARGIN, ("accept", level, j))
                accept = u < a
                if replay is not None and (level, j) in replay.accept and replay.accept[(level, j)] != accept:
                    if not abs(margin) < MASS_MARGIN:
                        raise ReplayRefused(f"accept test {j} of level {level}: margin {margin}")
                    accept = replay.accept[(level, j)]
                    replay.adopted.append(("accept", level, j))
                if accept:
                    accepted = next(k for k in kids if int(tree.token[k]) == x and int(tree.kind[k]) == kind)
                    break
        else:
            w, Zr = p_full, 1.0
        if accepted >= 0:
            toks.append(int(tree.token[accepted]))
            nodes.append(accepted)
            node, level = accepted, level + 1
            continue
        if Zr <= 0.0:
            empty = True
            w, Zr = p_full, 1.0
        target = u_bonus * Zr
        cum = np.cumsum(w)
        v = int(np.searchsorted(cum, target, side="right"))
        if v >= cum.shape[0]:
            v = int(np.nonzero(w > 0)[0][-1])
        lo = cum[v - 1] if v > 0 else 0.0
        mg.add("bonus", min(target - lo, cum[v] - target) / Zr, MASS_MARGIN, ("bonus", level))
        if replay is not None and level in replay.bonus and replay.bonus[level] != v:
            other = int(replay.bonus[level])
            if not _draw_accepts(cum, w, target, other, Zr):
                raise ReplayRefused(f"bonus at level {level}: token {other} is not a near-tie of {v}")
            v = other
            replay.adopted.append(("bonus", level))
        toks.append(v)
        return VerifyResult(len(nodes), toks, nodes, mg, empty)


# --------------------------------------------------------------------------
# Batch drivers
# --------------------------------------------------------------------------

def build_batch(draft, u_probe, p: Params) -> List[Tree]:
    """draft: [B][n_rows][V] (float array or uint16 bf16 bits); u_probe: [B][n_rows]."""
    return [build(draft[b], u_probe[b], p) for b in range(len(draft))]


def verify_batch(trees: List[Tree], target, u_verify, u_bonus, p: Params) -> List[VerifyResult]:
    """target: [B][R+1][V]; u_verify: [B][D][K]; u_bonus: [B]."""
    return [verify(trees[b], target[b], u_verify[b], float(u_bonus[b]), p) for b in range(len(trees))]
