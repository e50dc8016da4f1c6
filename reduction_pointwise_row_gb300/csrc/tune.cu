// Launch-configuration search of "Stax (4): GPU Codegen and Dynamic Shapes",
// section 9.6: the configuration space is a box of parameters that move by
// factors of two (Definition 9.2), the cost is a measured time (+inf for a
// configuration that cannot run), and coordinate descent (Algorithm 9.2)
// accepts a neighbour -- one parameter times or divided by 2 -- whenever it is
// faster by more than the factor (1 - eps).  Proposition 9.2 bounds the
// number of acceptances by min(|box|, ceil(log(t0 / tmin) / -log(1 - eps)))
// and guarantees that no single-coordinate neighbour of the result is faster
// by that factor.  Each configuration is measured once (memoised), so the
// cost behaves as the deterministic function the proposition assumes; with
// measurement noise |eta| <= eta_max, eps > 2 eta_max / (1 + eta_max) makes
// every acceptance a true improvement.
#include <cmath>
#include <map>
#include <vector>

#include "../../include/fr.h"
#include "launch.h"

namespace fr {

CdResult coordinate_descent(int p, const int *lo, const int *hi, int *c, double eps,
                            const std::function<double(const int *)> &cost) {
  std::map<std::vector<int>, double> memo;
  CdResult r{0, 0, 0.0};
  auto t_of = [&](const std::vector<int> &v) {
    auto it = memo.find(v);
    if (it != memo.end()) return it->second;
    const double t = cost(v.data());
    ++r.evaluations;
    memo.emplace(v, t);
    return t;
  };
  std::vector<int> cur(c, c + p);
  double t = t_of(cur);
  r.t = t;
  if (!std::isfinite(t)) return r;  // Proposition 9.2 needs a finite start
  bool improved = true;
  while (improved) {
    improved = false;
    for (int i = 0; i < p; ++i) {
      for (int step : {+1, -1}) {  // parameter i times 2, then divided by 2
        std::vector<int> nb = cur;
        nb[i] += step;
        if (nb[i] < lo[i] || nb[i] > hi[i]) continue;
        const double tn = t_of(nb);
        if (tn < (1.0 - eps) * t) {
          cur = nb;
          t = tn;
          ++r.acceptances;
          improved = true;
        }
      }
    }
  }
  for (int i = 0; i < p; ++i) c[i] = cur[i];
  r.t = t;
  return r;
}

}  // namespace fr

extern "C" fr_status fr_coordinate_descent(int32_t p, const int32_t *lo, const int32_t *hi,
                                           int32_t *c, double eps, fr_cost_fn cost, void *ctx,
                                           int32_t *acceptances, int32_t *evaluations) {
  if (p < 1 || p > FR_CD_MAX_PARAMS || !lo || !hi || !c || !cost) return FR_ERR_INVALID_ARG;
  if (!(eps > 0.0 && eps < 1.0)) return FR_ERR_INVALID_ARG;
  int l[FR_CD_MAX_PARAMS], h[FR_CD_MAX_PARAMS], v[FR_CD_MAX_PARAMS];
  for (int i = 0; i < p; ++i) {
    if (lo[i] > hi[i] || c[i] < lo[i] || c[i] > hi[i]) return FR_ERR_INVALID_ARG;
    l[i] = lo[i];
    h[i] = hi[i];
    v[i] = c[i];
  }
  const fr::CdResult r = fr::coordinate_descent(
      p, l, h, v, eps, [&](const int *q) {
        int32_t w[FR_CD_MAX_PARAMS];
        for (int i = 0; i < p; ++i) w[i] = q[i];
        return cost(w, ctx);
      });
  if (acceptances) *acceptances = r.acceptances;
  if (evaluations) *evaluations = r.evaluations;
  if (!std::isfinite(r.t)) return FR_ERR_INVALID_ARG;  // the start cannot run
  for (int i = 0; i < p; ++i) c[i] = v[i];
  return FR_OK;
}
