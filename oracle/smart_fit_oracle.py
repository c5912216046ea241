"""Plain float64 CPU oracle of the SMART cost-model fit.

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module; the library
never calls it, and it imports nothing from the library.

SMART ("SMART: When is it Actually Worth Expanding a Speculative Tree?", ECCV
2026 notes), Method / Key design 2: a one-off profiling of a few forward
passes on the target device fits the drafting cost as lambda*|T| + beta and
the verification cost as gamma*(exp(delta*|T|^rho) - 1) + eta by least
squares, with the biases beta and eta fixed at zero so that both pass through
the origin.

Reading (the pages give no units): costs are in units of one plain target
step t_base, the unit of the keep rule's C(n) = 1 + C_draft(n) + C_verify(n),
so the draft line is fitted to t_draft / t_base and the verification curve to
the time above the plain step, (t_verify - t_base) / t_base.  The search
domain is rho in [1, 4], gamma >= 0 and delta * max(n)^rho in [1e-6, 30]
(the curve's exponent at the largest profiled size).

The line is the textbook least-squares slope through the origin.  The curve is
fitted by brute force over a dense grid of (rho, log of that exponent), gamma
by linear least squares at each point, then polished by a library
least-squares solver (scipy's trust-region reflective method, bounded to the
domain) from the best grid points; the best result is kept.  Where the optimum is not unique (a flat valley of
gamma * delta at small exponents) the coefficients are not comparable; the
fitted curve at the profiled sizes is, and the tests compare that.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import scipy.optimize

RHO_LO, RHO_HI = 1.0, 4.0
LOGU_LO, LOGU_HI = float(np.log(1e-6)), float(np.log(30.0))


@dataclasses.dataclass
class CostFit:
    lam: float
    gamma: float
    delta: float
    rho: float
    sse_draft: float    # weighted sums of squared residuals, in units of t_base squared
    sse_verify: float


def draft_cost(n, lam: float):
    """C_draft(n) = lambda * n (beta = 0)."""
    return lam * np.asarray(n, dtype=np.float64)


def verify_cost(n, gamma: float, delta: float, rho: float):
    """C_verify(n) = gamma * (exp(delta * n^rho) - 1) (eta = 0)."""
    n = np.asarray(n, dtype=np.float64)
    return gamma * np.expm1(delta * n ** rho)


def fit_smart_cost(n: Sequence[float], t_draft: Sequence[float], t_verify: Sequence[float], t_base: float,
                   w: Optional[Sequence[float]] = None) -> CostFit:
    n = np.asarray(n, dtype=np.float64)
    w = np.ones_like(n) if w is None else np.asarray(w, dtype=np.float64)
    d = np.asarray(t_draft, dtype=np.float64) / t_base
    y = (np.asarray(t_verify, dtype=np.float64) - t_base) / t_base

    # drafting: minimise sum w (lambda n - d)^2 -> lambda = sum w n d / sum w n^2, kept >= 0
    lam = max(0.0, float(np.sum(w * n * d) / np.sum(w * n * n)))
    sse_d = float(np.sum(w * (draft_cost(n, lam) - d) ** 2))

    # verification, with u = delta * max(n)^rho (the exponent at the largest size):
    # brute force over a dense (rho, log u) grid, gamma >= 0 by linear least
    # squares at each point, then a library least-squares polish of
    # (gamma, log u, rho) within the domain from the best grid points
    n_max = float(n.max())
    x = n / n_max
    rhos = np.linspace(RHO_LO, RHO_HI, 121)
    logus = np.linspace(LOGU_LO, LOGU_HI, 801)
    F = np.expm1(np.exp(logus)[:, None, None] * x[None, None, :] ** rhos[None, :, None])  # [u][rho][i]
    sff = np.einsum("abi,i->ab", F * F, w)
    sfy = np.einsum("abi,i->ab", F, w * y)
    G = np.where(sff > 0, np.maximum(sfy / np.where(sff > 0, sff, 1.0), 0.0), 0.0)
    SSE = np.einsum("abi,i->ab", (G[:, :, None] * F - y[None, None, :]) ** 2, w)
    sw = np.sqrt(w)

    def resid(th):
        g, lu, r = th
        return sw * (g * np.expm1(np.exp(lu) * x ** r) - y)

    best = None
    for flat in np.argsort(SSE, axis=None)[:3]:
        ia, ib = np.unravel_index(flat, SSE.shape)
        x0 = [G[ia, ib], logus[ia], rhos[ib]]
        cand = [(float(SSE[ia, ib]), *x0)]
        if x0[0] > 0:
            res = scipy.optimize.least_squares(
                resid, x0=x0, bounds=([0.0, LOGU_LO, RHO_LO], [np.inf, LOGU_HI, RHO_HI]), method="trf",
                x_scale="jac", ftol=1e-15, xtol=1e-15, gtol=1e-15, max_nfev=2000)
            cand.append((float(np.sum(res.fun ** 2)), *res.x))
        for c in cand:
            if best is None or c[0] < best[0]:
                best = c
    sse_v, g, lu, r = best
    return CostFit(lam=lam, gamma=float(g), delta=float(np.exp(lu) / n_max ** r), rho=float(r), sse_draft=sse_d,
                   sse_verify=sse_v)


def fitted_verify_curve(fit: CostFit, n) -> np.ndarray:
    return verify_cost(n, fit.gamma, fit.delta, fit.rho)
