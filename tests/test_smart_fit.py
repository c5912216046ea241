"""SMART cost-model fit: the oracle pinned to exact data and library least squares,
and the native fit (spec_tree_smart_fit, host only) against the oracle."""
import math

import numpy as np
import pytest

from dynamic_tree_speculative_gb300 import workloads as WL
from oracle import smart_fit_oracle as SO

# sizes reaching well past the synthetic profile's compute knee
SIZES = [16, 64, 128, 256, 384]


def _exact(n, lam, gamma, delta, rho, t_base=2.0e-3):
    """Timings that follow the cost model exactly (the definition, written out)."""
    n = np.asarray(n, dtype=np.float64)
    t_draft = t_base * lam * n
    t_verify = t_base * (1.0 + gamma * (np.exp(delta * n ** rho) - 1.0))
    return t_draft, t_verify, t_base


@pytest.fixture(scope="module")
def native():
    from dynamic_tree_speculative_gb300 import binding as B
    return B


KNOWN = [
    dict(lam=0.02, gamma=0.05, delta=0.01, rho=1.3, n=[10, 20, 40, 80, 160]),
    dict(lam=0.005, gamma=0.5, delta=2.0e-4, rho=2.1, n=[8, 32, 64, 96, 128]),
    dict(lam=0.1, gamma=0.01, delta=0.05, rho=1.0, n=[4, 8, 16, 32, 64]),
]


@pytest.mark.parametrize("k", range(len(KNOWN)))
def test_oracle_recovers_known_coefficients(k):
    c = KNOWN[k]
    td, tv, tb = _exact(c["n"], c["lam"], c["gamma"], c["delta"], c["rho"])
    f = SO.fit_smart_cost(c["n"], td, tv, tb)
    assert f.lam == pytest.approx(c["lam"], rel=1e-12)
    for name in ("gamma", "delta", "rho"):
        assert getattr(f, name) == pytest.approx(c[name], rel=1e-5), name
    assert f.sse_verify < 1e-20


def test_oracle_line_is_the_least_squares_slope():
    """The weighted slope through the origin equals numpy's least-squares solution."""
    rng = np.random.default_rng(4)
    n = np.array([3.0, 9.0, 20.0, 41.0, 77.0])
    td = 1e-5 * n * (1 + 0.1 * rng.standard_normal(5))
    w = np.array([1.0, 0.5, 2.0, 1.0, 0.25])
    f = SO.fit_smart_cost(n, td, 1e-3 * (1 + 0.001 * n), 1e-3, w)
    sw = np.sqrt(w)
    ref = np.linalg.lstsq((sw * n)[:, None], sw * td / 1e-3, rcond=None)[0][0]
    assert f.lam == pytest.approx(ref, rel=1e-12)


def test_oracle_curve_is_a_minimum():
    """No small move of (gamma, delta, rho) inside the domain lowers the residual (noisy data)."""
    td, tv = WL.profile_timings(3, SIZES)
    f = SO.fit_smart_cost(SIZES, td, tv, 1.0e-3)
    y = (tv - 1.0e-3) / 1.0e-3

    def sse(g, d, r):
        return float(np.sum((g * np.expm1(d * np.asarray(SIZES, float) ** r) - y) ** 2))

    base = sse(f.gamma, f.delta, f.rho)
    assert base == pytest.approx(f.sse_verify, rel=1e-9)
    for dg, dd, dr in ((1e-4, 0, 0), (-1e-4, 0, 0), (0, 1e-4, 0), (0, -1e-4, 0), (0, 0, 1e-4), (0, 0, -1e-4)):
        r = min(4.0, max(1.0, f.rho * (1 + dr)))
        assert sse(f.gamma * (1 + dg), f.delta * (1 + dd), r) >= base * (1 - 1e-9)


@pytest.mark.parametrize("k", range(len(KNOWN)))
def test_native_recovers_known_coefficients(native, k):
    c = KNOWN[k]
    td, tv, tb = _exact(c["n"], c["lam"], c["gamma"], c["delta"], c["rho"])
    f = native.spec_tree_smart_fit(c["n"], td, tv, tb)
    assert f.lam == pytest.approx(c["lam"], rel=1e-12)
    for name in ("gamma", "delta", "rho"):
        assert getattr(f, name) == pytest.approx(c[name], rel=1e-5), name
    assert f.rms_verify < 1e-9


def _compare(nf, of, sizes, tv, t_base, w=None):
    w = np.ones(len(sizes)) if w is None else np.asarray(w, float)
    assert nf.lam == pytest.approx(of.lam, rel=1e-12)
    sse_native = nf.rms_verify ** 2 * float(np.sum(w))
    # the native grid search reaches the oracle's optimum (or a better one)
    assert sse_native <= of.sse_verify * (1 + 1e-6) + 1e-18
    # the fitted curve at the profiled sizes is unique: compare it, not the coefficients
    y = (np.asarray(tv) - t_base) / t_base
    cn = SO.verify_cost(sizes, nf.gamma, nf.delta, nf.rho)
    co = SO.fitted_verify_curve(of, sizes)
    assert np.max(np.abs(cn - co)) <= 1e-5 * max(1.0, float(np.max(np.abs(y))))


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_oracle_on_noisy_profiles(native, seed):
    td, tv = WL.profile_timings(seed, SIZES, noise=0.03)
    nf = native.spec_tree_smart_fit(SIZES, td, tv, 1.0e-3)
    of = SO.fit_smart_cost(SIZES, td, tv, 1.0e-3)
    _compare(nf, of, SIZES, tv, 1.0e-3)


def test_native_matches_oracle_with_weights(native):
    """Decaying weights, as an online refit over a window of recent profiles would use."""
    sizes = SIZES + [32, 192, 320]
    td, tv = WL.profile_timings(11, sizes, noise=0.05)
    w = 0.8 ** np.arange(len(sizes))[::-1]
    nf = native.spec_tree_smart_fit(sizes, td, tv, 1.0e-3, w)
    of = SO.fit_smart_cost(sizes, td, tv, 1.0e-3, w)
    _compare(nf, of, sizes, tv, 1.0e-3, w)


def test_zero_weight_drops_a_point(native):
    sizes = SIZES + [200]
    td, tv = WL.profile_timings(5, sizes, noise=0.03)
    tv = tv.copy()
    tv[-1] *= 3.0  # an outlier, given no weight
    a = native.spec_tree_smart_fit(sizes, td, tv, 1.0e-3, [1, 1, 1, 1, 1, 0])
    b = native.spec_tree_smart_fit(SIZES, td[:5], tv[:5], 1.0e-3)
    assert a.lam == pytest.approx(b.lam, rel=1e-12)
    for name in ("gamma", "delta", "rho"):
        assert getattr(a, name) == pytest.approx(getattr(b, name), rel=1e-9), name


def test_flat_verification_gives_no_growth(native):
    """Verification no slower than the plain step: gamma = 0, the keep rule pays drafting only."""
    n = [8, 16, 32, 64, 128]
    f = native.spec_tree_smart_fit(n, [1e-5 * x for x in n], [1e-3] * 5, 1e-3)
    assert f.gamma == 0.0 and f.rms_verify == 0.0


def test_fitted_coefficients_are_valid_smart_params(native):
    td, tv = WL.profile_timings(2, SIZES)
    f = native.spec_tree_smart_fit(SIZES, td, tv, 1.0e-3)
    p = f.apply(native.Params(K=8, m=1, W=8, depth=8, R=60, builder=native.BUILDER_SMART))
    assert native.spec_tree_check_params(p, 128256) == native.OK
    assert p.beta == 0.0 and p.eta == 0.0 and p.rho >= 1.0


@pytest.mark.parametrize("bad", ["few", "zero_size", "neg_time", "nan", "base", "weights"])
def test_bad_inputs_are_refused(native, bad):
    n, td, tv, tb, w = [8, 16, 32, 64], [1e-4] * 4, [1e-3] * 4, 1e-3, None
    if bad == "few":
        n, td, tv = n[:2], td[:2], tv[:2]
    elif bad == "zero_size":
        n = [0, 16, 32, 64]
    elif bad == "neg_time":
        tv = [1e-3, -1.0, 1e-3, 1e-3]
    elif bad == "nan":
        td = [1e-4, math.nan, 1e-4, 1e-4]
    elif bad == "base":
        tb = 0.0
    elif bad == "weights":
        w = [0.0] * 4
    with pytest.raises(native.SpecTreeError):
        native.spec_tree_smart_fit(n, td, tv, tb, w)
