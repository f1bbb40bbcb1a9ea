// Block epilogue shared by the LM-head kernels of 1..8 rows (CUDA-core and tensor-core
// variants): each block has its rows' logits for its vocabulary run in shared memory (ztile);
// it reduces per-row partial statistics, and the last block to finish combines them and, for
// the draft head, draws the token.
#pragma once

#include <math.h>

#include "params.cuh"

namespace spec {

// Rows [v0, v1) of block `blk`: a contiguous run of `band_rows`-row bands, balanced to one band.
__device__ __forceinline__ void block_rows(int blk, int nblk, int64_t nbands, int band_rows,
                                           int64_t V, int64_t& v0, int64_t& v1) {
  const int64_t b0 = static_cast<int64_t>(blk) * nbands / nblk;
  const int64_t b1 = static_cast<int64_t>(blk + 1) * nbands / nblk;
  v0 = b0 * band_rows;
  v1 = min(b1 * band_rows, V);
  if (v1 < v0) v1 = v0;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Weight of one logit in the tile's integer sum: exp((z - m) / T) in [0, 1], in 2^-40 units.
// The same expression is evaluated in the tile pass and in the draw's rescan, with explicit
// round-to-nearest operations (no contraction), so both see identical integers.
__device__ __forceinline__ unsigned long long tile_weight(float z, float m, float invT) {
  return quantise(expf(__fmul_rn(__fsub_rn(z, m), invT)));
}

// Per-block partials, ticket and (last block) the combine and the draft draw. All `nwarps`
// warps of the block call it after a __syncthreads that publishes ztile; `scratch` needs
// nwarps * 2 * gridDim.x doubles; flags[1] is a free shared int.
static __device__ __forceinline__ void gemv_block_epilogue(const GemvParams& p, const float* ztile,
                                                           int64_t v0, int nt, uint8_t* scratch,
                                                           int* flags, int nwarps) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int GR = gridDim.x, blk = blockIdx.x;
  const int NWALL = nwarps;
  // ---------------- per-block partial statistics of each row ----------------
  for (int q = warp; q < p.nrows; q += NWALL) {
    const float T = p.temperature[q / p.rows_per_req];
    const float invT = __fdiv_rn(1.f, T > 0.f ? T : 1.f);
    const float* zr = ztile + static_cast<size_t>(q) * p.tile_cap;
    Top2 t = top2_empty();
    int bad = 0;
    for (int j = lane; j < nt; j += 32) {
      const float z = zr[j];
      if (isnan(z) || z == INFINITY)
        bad = 1;
      else
        top2_push(t, z, static_cast<int32_t>(v0 + j));
    }
    t = warp_top2(t);
    bad = __any_sync(0xffffffffu, bad);
    unsigned long long ssum = 0ull;
    if (t.idx != kNoIndex && t.best != -INFINITY) {
      for (int j = lane; j < nt; j += 32) {
        const float z = zr[j];
        if (!(isnan(z) || z == INFINITY)) ssum += tile_weight(z, t.best, invT);
      }
    }
    ssum = warp_sum_u64(ssum);
    if (lane == 0) {
      GemvPartial pp;
      pp.m = t.best;
      pp.second = t.second;
      pp.idx = (t.idx == kNoIndex) ? -1 : t.idx;
      pp.flags = bad;
      pp.s = ssum;
      pp.pad = 0ull;
      p.part[static_cast<size_t>(blk) * kMaxRows + q] = pp;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&p.hdr->gemv_ticket, 1u);
    flags[1] = (ticket == static_cast<unsigned>(GR) - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!flags[1]) return;
  __threadfence();

  // ---------------- last block: combine the partials of every block ----------------
  // The scratch (free shared memory) holds per-block weights and scale factors.
  double* blk_w = reinterpret_cast<double*>(scratch) + static_cast<size_t>(warp) * 2 * GR;
  double* blk_f = blk_w + GR;
  for (int q = warp; q < p.nrows; q += NWALL) {
    const float T = p.temperature[q / p.rows_per_req];
    const float Te = T > 0.f ? T : 1.f;
    const float invT = __fdiv_rn(1.f, Te);
    Top2 t = top2_empty();
    int bad = 0;
    for (int cc = lane; cc < GR; cc += 32) {
      const GemvPartial* pp = p.part + static_cast<size_t>(cc) * kMaxRows + q;
      bad |= __ldcg(&pp->flags);
      const int32_t idx = __ldcg(&pp->idx);
      if (idx >= 0) t = top2_merge(t, Top2{__ldcg(&pp->m), __ldcg(&pp->second), idx});
    }
    t = warp_top2(t);
    bad = __any_sync(0xffffffffu, bad);
    const bool nonfinite = bad || t.idx == kNoIndex || t.best == -INFINITY;
    const float M = t.best;
    double S = 0.0;
    for (int cc = lane; cc < GR; cc += 32) {
      const GemvPartial* pp = p.part + static_cast<size_t>(cc) * kMaxRows + q;
      const float mc = __ldcg(&pp->m);
      const unsigned long long sc = __ldcg(&pp->s);
      double f = 0.0;
      if (!nonfinite && __ldcg(&pp->idx) >= 0 && mc != -INFINITY)  // fp32 factor, fp64 sums
        f = static_cast<double>(expf(__fmul_rn(__fsub_rn(mc, M), invT)));
      blk_f[cc] = f;
      blk_w[cc] = static_cast<double>(sc) * f;
      S += blk_w[cc];
    }
    S = warp_sum_f64(S);
    spec_rowstats st;
    if (nonfinite) {
      st.max = __int_as_float(0x7fc00000);
      st.log_norm = st.max;
      st.gap = st.max;
      st.argmax = -1;
    } else {
      st.max = M;
      st.log_norm = static_cast<float>(log(S) - 27.725887222397812);  // log(S * 2^-40)
      st.gap = __fsub_rn(M, t.second);
      st.argmax = t.idx;
    }
    if (lane == 0 && p.stats) p.stats[q] = st;

    if (p.draft) {
      int32_t tok = -1;
      if (!nonfinite && !(T > 0.f)) tok = t.idx;
      if (!nonfinite && T > 0.f && p.logits) {
        // inverse CDF: first block whose cumulative weight exceeds u*S, then the first token
        // inside it whose cumulative integer weight exceeds the remainder
        __syncwarp();
        const uint32_t u24 = uniform_u24(p.seed[q], p.pos[q] + p.pos_offset, PURPOSE_DRAFT);
        const double target = static_cast<double>(u24) * 5.9604644775390625e-08 * S;
        int cstar = -1;
        unsigned long long tt = 0ull;
        if (lane == 0) {
          double cum = 0.0;
          int last_nz = -1;
          for (int cc = 0; cc < GR; ++cc) {
            const double w = blk_w[cc];
            if (w > 0.0) last_nz = cc;
            if (w > 0.0 && cum + w > target) {
              cstar = cc;
              break;
            }
            cum += w;
          }
          const GemvPartial* pp;
          if (cstar >= 0) {
            pp = p.part + static_cast<size_t>(cstar) * kMaxRows + q;
            const unsigned long long sc = __ldcg(&pp->s);
            double rem = (target - cum) / blk_f[cstar];
            if (!(rem >= 0.0)) rem = 0.0;
            tt = static_cast<unsigned long long>(rem);
            if (tt >= sc) tt = sc - 1ull;
          } else {
            cstar = last_nz;
            if (cstar >= 0) {
              pp = p.part + static_cast<size_t>(cstar) * kMaxRows + q;
              tt = __ldcg(&pp->s) - 1ull;
            }
          }
        }
        cstar = __shfl_sync(0xffffffffu, cstar, 0);
        tt = __shfl_sync(0xffffffffu, tt, 0);
        if (cstar >= 0) {
          int64_t c0, c1;
          block_rows(cstar, GR, p.nbands, p.band_rows, p.V, c0, c1);
          const float mc = __ldcg(&(p.part + static_cast<size_t>(cstar) * kMaxRows + q)->m);
          const float* yrow = p.logits + static_cast<size_t>(q) * p.logits_stride;
          unsigned long long carry = 0ull;
          for (int64_t base = c0; base < c1 && tok < 0; base += 32) {
            const int64_t v = base + lane;
            unsigned long long w = 0ull;
            if (v < c1) {
              const float z = __ldcg(yrow + v);
              if (!(isnan(z) || z == INFINITY)) w = tile_weight(z, mc, invT);
            }
            unsigned long long incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const unsigned long long up = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += up;
            }
            const bool hit = (w > 0ull) && (carry + incl > tt);
            const unsigned mask = __ballot_sync(0xffffffffu, hit);
            if (mask) tok = static_cast<int32_t>(base + __ffs(mask) - 1);
            carry += __shfl_sync(0xffffffffu, incl, 31);
          }
        }
      }
      if (lane == 0) p.token_out[static_cast<size_t>(q) * p.token_stride] = tok;
    }
  }
  if (tid == 0) p.hdr->gemv_ticket = 0u;
}

}  // namespace spec
