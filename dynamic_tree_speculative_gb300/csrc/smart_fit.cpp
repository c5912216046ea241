// SMART cost-model fit (host only): SMART notes, Method / Key design 2 (a
// one-off device profiling of a few forward passes fits the drafting cost as
// a line through the origin and the verification cost as a power-exponential
// curve through the origin, both by least squares).
//
// Costs are in units of one plain target step (t_base), the unit the keep
// rule's C(n) = 1 + C_draft(n) + C_verify(n) uses:
//   C_draft(n)  = lambda * n                     fitted to t_draft / t_base
//   C_verify(n) = gamma * (exp(delta n^rho) - 1) fitted to (t_verify - t_base) / t_base
// lambda has a closed form.  For fixed (delta, rho) the verification model is
// linear in gamma, which then has a closed form too, so only (delta, rho) are
// searched: rho in [1, 4] and u = delta * n_max^rho (the exponent at the
// largest profiled size) in [1e-6, 30].  The residual's valley in (log u, rho)
// is narrow and curved (the exponential makes it very sensitive to u), so the
// search is nested: for each rho, the best log u by a dense scan refined by
// repeated zooming; over rho, the same scan-and-zoom of that profile.  It is
// deterministic and needs no starting point.
#include <math.h>
#include <stddef.h>

#include "spec_tree.h"

namespace {

constexpr double RHO_LO = 1.0, RHO_HI = 4.0;
constexpr double LOGU_LO = -13.815510557964274;  // ln(1e-6)
constexpr double LOGU_HI = 3.4011973816621555;   // ln(30)

struct Points {
  int n;
  const double* x;  // tree sizes divided by the largest
  const double* y;  // verification cost above the plain step, in t_base
  const double* w;  // weights
};

// Weighted sum of squared residuals of the best gamma >= 0 for (log u, rho);
// the gamma is returned through *gamma.  The residuals are summed directly
// (not expanded), so that near-exact fits keep their resolution.
double sse_at(const Points& P, double logu, double rho, double* gamma) {
  const double u = exp(logu);
  double f[1024];
  double sfy = 0.0, sff = 0.0;
  for (int i = 0; i < P.n; ++i) {
    f[i] = expm1(u * pow(P.x[i], rho));
    sfy += P.w[i] * f[i] * P.y[i];
    sff += P.w[i] * f[i] * f[i];
  }
  double g = sff > 0.0 ? sfy / sff : 0.0;
  if (!(g > 0.0)) g = 0.0;
  *gamma = g;
  double sse = 0.0;
  for (int i = 0; i < P.n; ++i) {
    const double r = g * f[i] - P.y[i];
    sse += P.w[i] * r * r;
  }
  return sse;
}

// Minimum of f over [lo, hi]: a scan of n0 points, then 40 rounds that
// evaluate 7 points spread over +-h around the best so far and shrink h by 3.
// Writes the argument to *arg and calls on_best(x) whenever a new best is
// evaluated (right after f(x)).
template <typename F, typename B>
double zoom_min(double lo, double hi, int n0, F f, double* arg, B on_best) {
  double c = lo, best = 0.0;
  for (int i = 0; i < n0; ++i) {
    const double x = lo + (hi - lo) * i / (n0 - 1);
    const double e = f(x);
    if (i == 0 || e < best) {
      best = e;
      c = x;
      on_best(x);
    }
  }
  double h = (hi - lo) / (n0 - 1);
  for (int it = 0; it < 40; ++it) {
    const double c0 = c;
    for (int k = 0; k < 7; ++k) {
      double x = c0 + h * (k - 3) / 3.0;
      x = x < lo ? lo : (x > hi ? hi : x);
      const double e = f(x);
      if (e < best) {
        best = e;
        c = x;
        on_best(x);
      }
    }
    h /= 3.0;
  }
  *arg = c;
  return best;
}

}  // namespace

extern "C" int spec_tree_smart_fit(int npts, const double* n, const double* t_draft, const double* t_verify,
                                   double t_base, const double* w, spec_tree_params* p, double* coef,
                                   double* rms) {
  if (npts < 3 || npts > 1024 || n == nullptr || t_draft == nullptr || t_verify == nullptr) return SPEC_TREE_E_PARAM;
  if (!(t_base > 0.0) || !isfinite(t_base)) return SPEC_TREE_E_PARAM;
  double x_max = 0.0, w_sum = 0.0;
  for (int i = 0; i < npts; ++i) {
    const double wi = w ? w[i] : 1.0;
    if (!(n[i] > 0.0) || !isfinite(n[i]) || !(t_draft[i] >= 0.0) || !isfinite(t_draft[i]) ||
        !(t_verify[i] >= 0.0) || !isfinite(t_verify[i]) || !(wi >= 0.0) || !isfinite(wi))
      return SPEC_TREE_E_PARAM;
    x_max = n[i] > x_max ? n[i] : x_max;
    w_sum += wi;
  }
  if (!(w_sum > 0.0)) return SPEC_TREE_E_PARAM;

  double xs[1024], ys[1024], ws[1024];
  double snd = 0.0, snn = 0.0;
  for (int i = 0; i < npts; ++i) {
    ws[i] = w ? w[i] : 1.0;
    xs[i] = n[i] / x_max;
    ys[i] = (t_verify[i] - t_base) / t_base;
    snd += ws[i] * n[i] * (t_draft[i] / t_base);
    snn += ws[i] * n[i] * n[i];
  }
  // drafting: the weighted least-squares line through the origin
  double lambda = snn > 0.0 ? snd / snn : 0.0;
  if (!(lambda > 0.0)) lambda = 0.0;
  double sse_d = 0.0;
  for (int i = 0; i < npts; ++i) {
    const double r = lambda * n[i] - t_draft[i] / t_base;
    sse_d += ws[i] * r * r;
  }

  // verification: nested scan-and-zoom searches, log u inside, rho outside
  const Points P{npts, xs, ys, ws};
  double best_logu = LOGU_LO, best_g = 0.0;
  auto best_over_u = [&](double rho, double* logu_out, double* g_out) {
    double g;
    return zoom_min(LOGU_LO, LOGU_HI, 201, [&](double lu) { return sse_at(P, lu, rho, &g); }, logu_out,
                    [&](double) { *g_out = g; });
  };
  double best_rho = RHO_LO;
  zoom_min(RHO_LO, RHO_HI, 31, [&](double rho) {
    double lu, g;
    return best_over_u(rho, &lu, &g);
  }, &best_rho, [](double) {});
  const double best = best_over_u(best_rho, &best_logu, &best_g);
  const double delta = exp(best_logu) / pow(x_max, best_rho);
  if (coef) {
    coef[0] = lambda;
    coef[1] = best_g;
    coef[2] = delta;
    coef[3] = best_rho;
  }
  if (p) {
    p->lambda = static_cast<float>(lambda);
    p->beta = 0.0f;
    p->gamma = static_cast<float>(best_g);
    p->delta = static_cast<float>(delta);
    p->rho = static_cast<float>(best_rho);
    p->eta = 0.0f;
  }
  if (rms) {
    rms[0] = sqrt(sse_d / w_sum);
    rms[1] = sqrt(best / w_sum);
  }
  return SPEC_TREE_OK;
}
