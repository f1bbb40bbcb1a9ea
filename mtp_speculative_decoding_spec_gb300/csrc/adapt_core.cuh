// Adaptive width: the update of one request's width state from its cycle's result (see
// spec_adapt_width in spec.h), shared by the width kernel and by the LM-head kernel's last
// block when the greedy acceptance and the width update are fused into it.
#pragma once
#include "params.cuh"

namespace spec {

constexpr float kFitVarMin = 0.25f;  // variance of the widths a usable fit needs
constexpr float kFitOutlier = 4.f;   // costs above this many times the fitted one are skipped

// The usable fit (a, b) of c ~ a + b*k from the moving averages, or false.
__device__ __forceinline__ bool fit_model(const float* f, float& a, float& b) {
  const float var = __fsub_rn(f[1], __fmul_rn(f[0], f[0]));
  if (!(var >= kFitVarMin)) return false;
  b = __fdiv_rn(__fsub_rn(f[3], __fmul_rn(f[0], f[2])), var);
  a = __fsub_rn(f[2], __fmul_rn(b, f[0]));
  return a > 0.f && b > 0.f;
}

// Request b's update from its cycle's result o: per-depth rates, the cycle-cost fit and the
// next width, written to state[b], k_next[b] and (when set) k_mirror[b]. One thread.
__device__ __forceinline__ void adapt_request(const AdaptParams& p, int b,
                                              const spec_accept_out& o) {
  spec_width_state s = p.state[b];
  const int k = p.k_used[b];
  // the cycle's cost: given, or the device time since this request's previous call
  float cost = 0.f;
  if (p.cycle_cost) {
    cost = p.cycle_cost[b];
  } else {
    const uint32_t now = static_cast<uint32_t>(globaltimer_ns() >> 10) | 1u;
    if (s.t_last != 0u) cost = static_cast<float>(now - s.t_last);  // modulo 2^32
    s.t_last = now;
  }
  // beliefs: an observed depth's rate, else the belief of the depth above (0.5 for depth 1)
  float bel[kMaxRows];
  bel[0] = 0.5f;
  for (int d = 1; d < kMaxRows; ++d)
    bel[d] = ((s.seen >> d) & 1u) ? s.rate[d] : (d > 1 ? bel[d - 1] : 0.5f);
  if (o.status == SPEC_REQ_OK && k >= 0 && k <= kMaxRows - 1) {
    uint32_t obs = 0u;  // depths observed in this cycle
    for (int d = 1; d <= k; ++d) {
      float x;
      if (d <= o.n_accept)
        x = 1.f;
      else if (d == o.n_accept + 1 && !o.eos_hit)
        x = 0.f;
      else
        break;
      s.rate[d] = __fadd_rn(bel[d], __fmul_rn(p.alpha, __fsub_rn(x, bel[d])));
      s.seen |= 1u << d;
      obs |= 1u << d;
    }
    // a depth seen before but not in this cycle relaxes towards the updated belief of the
    // depth above, in increasing depth, so that one that looked poor is tried again
    float above = ((s.seen >> 1) & 1u) ? s.rate[1] : 0.5f;
    for (int d = 2; d < kMaxRows; ++d) {
      const bool was_seen = (s.seen >> d) & 1u;
      if (was_seen && !((obs >> d) & 1u))
        s.rate[d] = __fadd_rn(s.rate[d], __fmul_rn(p.alpha, __fsub_rn(above, s.rate[d])));
      above = was_seen ? s.rate[d] : above;
    }
    s.cycles += 1u;
    // the cycle-cost fit: moving averages of k, k^2, c and k*c
    if (cost > 0.f) {
      const float kf = static_cast<float>(k);
      const float x[4] = {kf, __fmul_rn(kf, kf), cost, __fmul_rn(kf, cost)};
      float a, bb;
      if (!(s.seen & 1u)) {
        for (int i = 0; i < 4; ++i) s.fit[i] = x[i];
        s.seen |= 1u;
      } else if (!(fit_model(s.fit, a, bb) &&
                   cost > __fmul_rn(kFitOutlier, __fadd_rn(a, __fmul_rn(bb, kf))))) {
        for (int i = 0; i < 4; ++i)
          s.fit[i] = __fadd_rn(s.fit[i], __fmul_rn(p.alpha, __fsub_rn(x[i], s.fit[i])));
      }
      if (fit_model(s.fit, a, bb)) s.rate[0] = __fdiv_rn(bb, a);
    }
  }
  // expected tokens E(k) = 1 + sum_j prod_{i<=j} rate[i]; the best E(k) / cost(k) over
  // k in [1, k_max] (never 0: the first draft is always tried, so depth 1 stays observed)
  for (int d = 1; d < kMaxRows; ++d)  // beliefs after this cycle's update
    bel[d] = ((s.seen >> d) & 1u) ? s.rate[d] : (d > 1 ? bel[d - 1] : 0.5f);
  const float ratio = s.rate[0];
  float e = 1.f, run = 1.f, best = -1.f;
  const int lo = p.k_max < 1 ? p.k_max : 1;
  int kb = lo;
  for (int kk = 0; kk <= p.k_max; ++kk) {
    if (kk > 0) {
      run = __fmul_rn(run, bel[kk]);
      e = __fadd_rn(e, run);
    }
    const float c = ratio > 0.f ? __fadd_rn(1.f, __fmul_rn(ratio, static_cast<float>(kk)))
                                : p.cost[kk];
    const float v = __fdiv_rn(e, c);
    if (kk >= lo && v > best) {
      best = v;
      kb = kk;
    }
  }
  s.k = kb;
  p.state[b] = s;
  p.k_next[b] = kb;
  if (p.k_mirror) p.k_mirror[b] = kb;
}

}  // namespace spec
