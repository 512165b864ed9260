// plan_select.cu -- SNIP's per-layer format selection (host code): the
// knapsack-like integer program that chooses FP8 or NVFP4 for each linear so
// as to minimise a quality-loss estimate while a target fraction of the GEMM
// FLOPs runs in FP4.
//
// Sources: "SNIP" (Pan et al.), Abstract and Figure 2 (statistics collected
// periodically feed an ILP that picks layer-wise precision to minimise the
// overall quality loss under an efficiency target; the pages call it
// knapsack-like) and Figure 3 (efficiency = the fraction of FP4 FLOPs).  The
// pages do not print the divergence formulas, so the per-layer cost of a
// format is the proxy computed by snip_plan_costs from the statistics pass.
//
// Exact solution by dynamic programming over the FP4 FLOPs in units of the
// greatest common divisor of the layers' FLOPs: dp[c] = least extra cost of a
// layer set whose FP4 FLOPs are exactly c units, then the best c at or above
// the target.  One decision bit per (layer, c) recovers the set.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "snip.h"

namespace {

constexpr double kMaxExactFlops = 9007199254740992.0;   // 2^53
constexpr uint64_t kMaxCells = 1ull << 28;              // decision bits of the table

uint64_t gcd_u64(uint64_t a, uint64_t b) {
  while (b) {
    const uint64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

}  // namespace

extern "C" {

snip_status snip_plan_costs(int n_layers, const double* raw_host, double* cost_fp8, double* cost_nvfp4) {
  if (n_layers < 0 || (n_layers > 0 && (!raw_host || !cost_fp8 || !cost_nvfp4))) return SNIP_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    double c8 = 0.0, c4 = 0.0;
    for (int t = 0; t < 3; ++t) {   // X, W, dY
      const double* r = raw_host + ((int64_t)l * 3 + t) * SNIP_STATS_NVALS;
      const double x2 = r[SNIP_ST_SUM_X2], e4 = r[SNIP_ST_NVFP4_ERR2], e8 = r[SNIP_ST_FP8_ERR2];
      if (!std::isfinite(x2) || !std::isfinite(e4) || !std::isfinite(e8)) return SNIP_ERR_NONFINITE;
      if (x2 > 0.0) {
        c4 += e4 / x2;
        c8 += e8 / x2;
      }
    }
    cost_fp8[l] = c8;
    cost_nvfp4[l] = c4;
  }
  return SNIP_OK;
}

snip_status snip_plan_select(int n_layers, const double* flops, const double* cost_fp8, const double* cost_nvfp4,
                             double fp4_fraction, int* fmt_out, double* fp4_fraction_out, double* cost_out) {
  if (n_layers < 0 || (n_layers > 0 && (!flops || !cost_fp8 || !cost_nvfp4 || !fmt_out))) return SNIP_ERR_INVALID_ARG;
  if (!(fp4_fraction >= 0.0 && fp4_fraction <= 1.0)) return SNIP_ERR_INVALID_ARG;
  // integral FLOPs, reduced by their common divisor
  uint64_t g = 0;
  for (int i = 0; i < n_layers; ++i) {
    const double f = flops[i];
    if (!(f >= 0.0 && f <= kMaxExactFlops) || f != std::floor(f)) return SNIP_ERR_INVALID_ARG;
    if (!std::isfinite(cost_fp8[i]) || !std::isfinite(cost_nvfp4[i])) return SNIP_ERR_INVALID_ARG;
    g = gcd_u64(g, (uint64_t)f);
  }
  if (g == 0) g = 1;
  std::vector<uint64_t> w(n_layers);
  uint64_t wt = 0;
  for (int i = 0; i < n_layers; ++i) {
    w[i] = (uint64_t)flops[i] / g;
    wt += w[i];
  }
  // required FP4 units: the fraction of the total, less a tolerance for the rounding of the fraction itself
  double need_d = std::ceil(fp4_fraction * (double)wt - 1e-9);
  if (need_d < 0.0) need_d = 0.0;
  const uint64_t need = need_d > (double)wt ? wt : (uint64_t)need_d;
  if ((uint64_t)n_layers * (wt + 1) > kMaxCells) return SNIP_ERR_SHAPE;

  const double inf = HUGE_VAL;
  std::vector<double> dp(wt + 1, inf);
  std::vector<uint8_t> take((size_t)n_layers * (wt + 1), 0);
  dp[0] = 0.0;
  for (int i = 0; i < n_layers; ++i) {
    const double delta = cost_nvfp4[i] - cost_fp8[i];
    uint8_t* ti = take.data() + (size_t)i * (wt + 1);
    // descending: each layer enters a set at most once (a zero-FLOP layer only where it lowers the cost)
    for (uint64_t c = wt + 1; c-- > w[i];) {
      const double src = dp[c - w[i]];
      if (src == inf) continue;
      const double cand = src + delta;
      if (cand < dp[c]) {
        dp[c] = cand;
        ti[c] = 1;
      }
    }
  }
  uint64_t best = wt + 1;
  for (uint64_t c = need; c <= wt; ++c)
    if (dp[c] < inf && (best > wt || dp[c] < dp[best])) best = c;
  if (best > wt) return SNIP_ERR_SHAPE;   // unreachable: the all-FP4 set always meets the target
  // walk the decisions back from the last layer
  uint64_t c = best;
  for (int i = n_layers - 1; i >= 0; --i) {
    const bool in = take[(size_t)i * (wt + 1) + c] != 0;
    fmt_out[i] = in ? SNIP_FMT_NVFP4 : SNIP_FMT_FP8_E4M3;
    if (in) c -= w[i];
  }
  double f4 = 0.0, ftot = 0.0, cost = 0.0;
  for (int i = 0; i < n_layers; ++i) {
    ftot += flops[i];
    if (fmt_out[i] == SNIP_FMT_NVFP4) {
      f4 += flops[i];
      cost += cost_nvfp4[i];
    } else {
      cost += cost_fp8[i];
    }
  }
  if (fp4_fraction_out) *fp4_fraction_out = ftot > 0.0 ? f4 / ftot : 0.0;
  if (cost_out) *cost_out = cost;
  return SNIP_OK;
}

}  // extern "C"
