// LM-head projection of 1..8 rows (verify rows, or one draft row per request) with the row
// statistics and, for the draft head, the token choice fused in.
//
// Shape of the work (lucebox-hub PR #15 "MTP speculative decoding", section "What": the trunk
// verifies k drafts in one batched forward of k+1 rows through the shared LM head; the draft
// head covers the first 64,000 vocabulary rows and picks its token on the GPU): z = H W^T with
// W [V, d] bf16 (or fp32) streamed once from HBM, H [rows <= 8, d] tiny. This is a streaming
// GEMV: the weight bytes bound it, so the design is about keeping HBM busy:
//   * one persistent block per SM; block c owns the contiguous rows [c*V/G, (c+1)*V/G)
//     (balanced to one row, no wave tail);
//   * a producer warp streams groups of whole weight rows (contiguous bytes) into a ring of
//     shared-memory stages with 1-D bulk (TMA) copies completed on mbarriers;
//   * each consumer thread owns one 16-byte chunk of the hidden dimension and holds the
//     matching slice of every H row in registers, so a weight byte is read from shared memory
//     once and used for all rows; partial dot products are combined by a fixed butterfly
//     (xor 16, 8, 4, 2, 1) and then across the warps of a row in ascending order. That order
//     does not depend on how many rows share the call, so every row's logits are bitwise
//     batch-invariant (section "Exactness": verify stays batch-invariant up to eight rows);
//   * the block keeps its tile of logits in shared memory, reduces max / argmax / top-2 and a
//     sum of exp((z - m)/T) quantised to 2^-40 units in 64-bit integers (exact, so the sum
//     does not depend on order either), and the last block to finish combines the per-block
//     partials; for the draft head at T > 0 it also draws the token by inverse CDF and writes
//     it to device memory.
#include <math.h>

#include "params.cuh"

namespace spec {


// Reduce-scatter of SIZE values per lane over the warp: after the call lane l holds, in v[0],
// the full warp sum of value index l / (32 / SIZE_initial). The pairing order is the fixed
// butterfly xor 16, 8, 4, 2, 1 for every value, whatever the number of values.
template <int SIZE, int OFF>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (OFF > 0) {
      if constexpr (SIZE > 1) {
        constexpr int H = SIZE / 2;
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
        }
        ReduceScatter<H, OFF / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
        ReduceScatter<1, OFF / 2>::run(v, lane);
      }
    }
  }
};

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <bool BF16>
__device__ __forceinline__ void unpack16(const uint4 w, float* f) {
  if constexpr (BF16) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(u[k] << 16);
      f[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
    }
  } else {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
  }
}

// Weight of one logit in the tile's integer sum: exp((z - m) / T) in [0, 1], in 2^-40 units.
// The same expression is evaluated in the tile pass and in the draw's rescan, with explicit
// round-to-nearest operations (no contraction), so both see identical integers.
__device__ __forceinline__ unsigned long long tile_weight(float z, float m, float invT) {
  return quantise(expf(__fmul_rn(__fsub_rn(z, m), invT)));
}

// Rows of the weight matrix each row group handles per stage: the reduction of G*RP partial
// sums per lane costs about the same for any G*RP <= 32, so G shrinks as the rows grow.
template <int RP>
struct RowsPerStage {
  static constexpr int G = (RP >= 8) ? 4 : 8;
};

template <int RP, bool BF16>
__global__ void __launch_bounds__(448, 1) gemv_rows_kernel(const GemvParams p) {
  constexpr int EPC = BF16 ? 8 : 4;       // elements per 16-byte chunk
  constexpr int G = RowsPerStage<RP>::G;  // weight rows per row group per stage
  constexpr int NV = G * RP;              // partial sums per lane per stage
  constexpr int SPREAD = 32 / NV;         // lanes holding the same value after the reduction
  static_assert(NV <= 32 && 32 % NV == 0, "reduction layout");
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, NW = p.nw;
  const int PRODUCER = NW, REDUCER = NW + 1;
  uint8_t* stage_base = smem;
  float* red = reinterpret_cast<float*>(smem + p.ring_bytes);  // [S][NW][32]
  float* ztile = red + static_cast<size_t>(S) * NW * 32;
  uint64_t* full = reinterpret_cast<uint64_t*>(ztile + static_cast<size_t>(RP) * p.tile_cap);
  uint64_t* empty = full + S;
  uint64_t* redbar = empty + S;  // [S][ng]
  int* flags = reinterpret_cast<int*>(redbar + S * p.ng);  // [0] abort, [1] last block

  const int GR = gridDim.x, blk = blockIdx.x;
  const int64_t v0 = static_cast<int64_t>(blk) * p.V / GR;
  const int64_t v1 = static_cast<int64_t>(blk + 1) * p.V / GR;
  const int nt = static_cast<int>(v1 - v0);
  const int nst = (nt + p.stage_rows - 1) / p.stage_rows;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW + 1);  // every consumer warp and the reducer
    }
    for (int s = 0; s < S * p.ng; ++s) mbar_init(&redbar[s], p.wpr);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == PRODUCER) {
    // ---------------- producer: stream whole weight rows into the stage ring ----------------
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < nst; ++it) {
        const int s = it % S;
        if (it >= S && !mbar_wait_bounded(&empty[s], ((it / S) - 1) & 1)) {
          atomicOr(&p.hdr->error, ERR_GEMV_WAIT_EMPTY);
          atomicExch(&flags[0], 1);
          break;
        }
        const int rows = min(p.stage_rows, nt - it * p.stage_rows);
        const uint32_t bytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(p.row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(stage_base + static_cast<size_t>(s) * p.stage_bytes,
                 p.W + static_cast<size_t>(v0 + static_cast<int64_t>(it) * p.stage_rows) *
                           p.row_bytes,
                 bytes, &full[s]);
        issued = it + 1;
      }
      // every issued copy must have landed before this block may exit
      for (int it = max(0, issued - S); it < issued; ++it) {
        if (!mbar_wait_bounded(&full[it % S], (it / S) & 1)) {
          atomicOr(&p.hdr->error, ERR_GEMV_DRAIN);
          break;
        }
      }
    }
  } else if (warp == REDUCER) {
    // ---------------- reducer: sum each row's per-warp partials in ascending warp order -------
    float tq[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r)
      tq[r] = (r < p.nrows && p.logits) ? p.temperature[r / p.rows_per_req] : 0.f;
    for (int it = 0; it < nst; ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      const int rows = min(p.stage_rows, nt - it * p.stage_rows);
      bool ok = true;
      for (int gi = 0; gi < p.ng; ++gi) {
        if (!mbar_wait_bounded(&redbar[s * p.ng + gi], ph)) {
          atomicOr(&p.hdr->error, ERR_GEMV_WAIT_RED);
          atomicExch(&flags[0], 1);
          ok = false;
          break;
        }
        if (lane < NV) {
          const int g = lane / RP, r = lane % RP;
          const int lr = gi * G + g;
          if (r < p.nrows && lr < rows) {
            const float* src = red + (static_cast<size_t>(s) * NW + gi * p.wpr) * 32 + lane;
            float z = 0.f;
            for (int w2 = 0; w2 < p.wpr; ++w2) z += src[w2 * 32];
            const int local = it * p.stage_rows + lr;
            ztile[static_cast<size_t>(r) * p.tile_cap + local] = z;
            float tr = 0.f;
#pragma unroll
            for (int rr = 0; rr < RP; ++rr)
              if (rr == r) tr = tq[rr];
            if (tr > 0.f) p.logits[static_cast<size_t>(r) * p.logits_stride + v0 + local] = z;
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage's partial sums are consumed
    }
  } else {
    // ---------------- consumers: dot products against register-resident H ----------------
    const int gi = warp / p.wpr, wi = warp - gi * p.wpr;
    const int chunk = wi * 32 + lane;
    const bool active = chunk < p.cpr;
    float h[RP][EPC];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      uint4 hv = make_uint4(0u, 0u, 0u, 0u);
      if (active && r < p.nrows)
        hv = *reinterpret_cast<const uint4*>(p.H + static_cast<size_t>(r) * p.h_row_bytes +
                                             static_cast<size_t>(chunk) * 16);
      unpack16<BF16>(hv, h[r]);
    }

    for (int it = 0; it < nst; ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      if (!mbar_wait_bounded(&full[s], ph)) {
        atomicOr(&p.hdr->error, ERR_GEMV_WAIT_FULL);
        atomicExch(&flags[0], 1);
        break;
      }
      const int rows = min(p.stage_rows, nt - it * p.stage_rows);
      float v[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = 0.f;
      if (active) {
        const uint8_t* sp = stage_base + static_cast<size_t>(s) * p.stage_bytes +
                            static_cast<size_t>(gi * G) * p.row_bytes +
                            static_cast<size_t>(chunk) * 16;
        uint4 w[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
          w[g] = (gi * G + g < rows) ? lds128(sp + static_cast<size_t>(g) * p.row_bytes)
                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float wf[EPC];
          unpack16<BF16>(w[g], wf);
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            // packed fp32x2 FMAs: even and odd elements accumulate separately, then add
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EPC; e += 2)
              a = __ffma2_rn(make_float2(wf[e], wf[e + 1]), make_float2(h[r][e], h[r][e + 1]), a);
            v[g * RP + r] = a.x + a.y;
          }
        }
      }
      ReduceScatter<NV, 16>::run(v, lane);
      float* rb = red + (static_cast<size_t>(s) * NW + warp) * 32;
      if ((lane % SPREAD) == 0) rb[lane / SPREAD] = v[0];
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&redbar[s * p.ng + gi]);
        mbar_arrive(&empty[s]);
      }
    }
  }
  __syncthreads();

  // ---------------- per-block partial statistics of each row ----------------
  const int NWALL = NW + 2;
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
  // The stage ring is free now; it holds per-block weights and scale factors.
  double* blk_w = reinterpret_cast<double*>(stage_base) + static_cast<size_t>(warp) * 2 * GR;
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
      if (!nonfinite && __ldcg(&pp->idx) >= 0 && mc != -INFINITY)
        f = exp((static_cast<double>(mc) - static_cast<double>(M)) / static_cast<double>(Te));
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
          const int64_t c0 = static_cast<int64_t>(cstar) * p.V / GR;
          const int64_t c1 = static_cast<int64_t>(cstar + 1) * p.V / GR;
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

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

template <int RP, bool BF16>
static cudaError_t launch_variant(const GemvLaunch& L, cudaStream_t stream) {
  auto kern = gemv_rows_kernel<RP, BF16>;
  static int configured_smem = 0;  // largest dynamic smem size set so far for this variant
  if (L.smem > configured_smem) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (e != cudaSuccess) return e;
    configured_smem = L.smem;
  }
  kern<<<L.grid, L.threads, L.smem, stream>>>(L.p);
  return cudaGetLastError();
}

cudaError_t gemv_dispatch(const GemvLaunch& L, bool bf16, int rp, cudaStream_t stream) {
  if (bf16) {
    switch (rp) {
      case 1: return launch_variant<1, true>(L, stream);
      case 2: return launch_variant<2, true>(L, stream);
      case 4: return launch_variant<4, true>(L, stream);
      default: return launch_variant<8, true>(L, stream);
    }
  }
  switch (rp) {
    case 1: return launch_variant<1, false>(L, stream);
    case 2: return launch_variant<2, false>(L, stream);
    case 4: return launch_variant<4, false>(L, stream);
    default: return launch_variant<8, false>(L, stream);
  }
}

}  // namespace spec
