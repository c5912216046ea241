"""The oracle's pins have teeth: each planted mistake below fails at least one of them.

A mistake is planted by editing one line of the oracle's source text, executing
the edited text as a separate module and running pins from
tests/test_oracle_pins.py against that module instead of the oracle.  Nothing
here touches the CUDA path; everything runs on the CPU.

The mistakes are the plausible ones for each part of the method:
  * SMART builder (SMART notes, flowchart and Key design 3): |P| grown on every
    keep, L grown by the local probability instead of the path score, kept
    nodes expanded from the wrong draft rows, a layer scanned in ascending
    key order;
  * expansion and verification (RheoSampling notes, Key designs 2 and 3): q~
    formed from the untempered q, the probe's proxy replaced by its true
    probability, the token id inside the ranking key, the residual without
    max(0, .), the target p left untempered, the bonus drawn from p instead
    of the final residual;
  * truncation (Key design 1): ties at the cut broken by descending id.
"""
import pathlib
import sys
import types

import pytest

import test_oracle_pins as pins
from oracle import spec_tree_oracle

SRC = pathlib.Path(spec_tree_oracle.__file__).read_text()


def _mutant(old: str, new: str) -> types.ModuleType:
    assert SRC.count(old) == 1, f"mutation site not unique: {old!r}"
    name = "oracle_mutant"
    mod = types.ModuleType(name)
    sys.modules[name] = mod        # dataclasses look their module up while the class is made
    try:
        exec(compile(SRC.replace(old, new), name, "exec"), mod.__dict__)
    finally:
        del sys.modules[name]
    return mod


def _smart_golden():
    pins.check_smart_golden(pins.O)


def _lemma():
    for m in (1, 2):
        pins.test_local_ranking_preservation_lemma(m, 1.0)


def _support_brute_force():
    for V, size in [(300, 128), (3000, 256)]:
        pins.test_support_is_brute_force_top_by_logit_then_id(V, size)


def _chi_square():
    pins.test_losslessness_chi_square_two_levels(0)


def _lossless():
    for R, m, T in [(8, 1, 1.0), (3, 2, 0.7), (8, 0, 1.4)]:
        pins.test_losslessness_exact_first_token(0, R, m, T)


MUTANTS = {
    "smart_paths_every_keep": (
        "                if has_child.get(id(c.parent), False):\n                    paths += 1",
        "                if True:\n                    paths += 1",
        [_smart_golden]),
    "smart_L_local_q": (
        "                L += c.score\n",
        "                L += c.score / c.parent.score\n",
        [_smart_golden]),
    "smart_wrong_expansion_rows": (
        "        for c in kept_layer:\n            c.exp_row = next_row",
        "        for c in reversed(kept_layer):\n            c.exp_row = next_row",
        [_smart_golden]),
    "smart_ascending_scan": (
        '        layer = _ranked(layer, replay, ("layer", d))',
        '        layer = _ranked(layer, replay, ("layer", d))[::-1]',
        [_smart_golden]),
    "q_tilde_untempered": (
        "        qt[ex.sup_id[m:]] = ex.qT[m:] / ex.zT",
        "        qt[ex.sup_id[m:]] = ex.q[m:] / ex.z",
        [_lossless]),
    "proxy_is_true_probability": (
        "        children.append((m, PROBE, probe_pos, int(sup[probe_pos]), proxy))",
        "        children.append((m, PROBE, probe_pos, int(sup[probe_pos]), float(q[probe_pos])))",
        [_lemma, pins.test_probe_survival_is_independent_of_probe_identity]),
    "token_in_ranking_key": (
        "        return (-self.score, self.depth, self.prank, self.slot)",
        "        return (-self.score, self.token, self.depth, self.prank, self.slot)",
        [pins.test_probe_survival_is_independent_of_probe_identity, _lossless]),
    "residual_without_max0": (
        "        wn = np.maximum(0.0, w / Zr - qt)",
        "        wn = w / Zr - qt",
        [pins.test_hand_worked_verification_level, _lossless]),
    "support_ties_by_id_descending": (
        '    return np.argsort(-row, kind="stable")[:size]',
        '    return (len(row) - 1 - np.argsort(-row[::-1], kind="stable"))[:size]',
        [_support_brute_force]),
    "target_p_untempered": (
        "    e = np.exp((t - t.max()) / temperature)",
        "    e = np.exp(t - t.max())",
        [pins.test_target_probs_match_scipy]),
    "bonus_from_p_not_the_residual": (
        "        cum = np.cumsum(w)",
        "        cum = np.cumsum(p_full) * Zr",
        [_chi_square]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    old, new, checks = MUTANTS[name]
    monkeypatch.setattr(pins, "O", _mutant(old, new))
    failed = []
    for check in checks:
        try:
            check()
        except AssertionError as e:
            failed.append((check.__name__, str(e)[:120]))
    assert failed, f"planted mistake {name} passes every pin it was run against"


def test_unplanted_source_passes_the_same_pins(monkeypatch):
    """The copy executed the same way without an edit passes every check used above."""
    monkeypatch.setattr(pins, "O", _mutant("ROOT, DET, PROBE, FILL = 0, 1, 2, 3", "ROOT, DET, PROBE, FILL = 0, 1, 2, 3"))
    for _, _, checks in MUTANTS.values():
        for check in checks:
            check()
