// Block epilogue shared by the LM-head kernels of 1..8 rows (CUDA-core and tensor-core
// variants): each block has its rows' logits for its vocabulary run in shared memory (ztile);
// it reduces per-row partial statistics, and the last block to finish combines them and, for
// the draft head, draws the token.
#pragma once

#include <math.h>

#include "adapt_core.cuh"
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

// Draft head with device-chosen widths: true when no row of this launch needs the step (every
// k_active[b] <= pos_offset). Waits for the previous kernel first: the widths are written by
// it. Uniform across the block (every thread reads the same values).
__device__ __forceinline__ bool draft_step_idle(const GemvParams& p) {
  if (p.kact == nullptr) return false;
  pdl_wait();
  for (int r = 0; r < p.nrows && r < kMaxRows; ++r)
    if (p.kact[r] > p.pos_offset) return false;
  return true;
}

// Vocabulary id of projected row r (-1 stays -1).
__device__ __forceinline__ int32_t row_id(const GemvParams& p, int64_t r) {
  return static_cast<int32_t>(r < p.lo_rows ? r : p.hi_row0 + (r - p.lo_rows));
}
// Weight row of the TMA box that starts at projected row y (boxes never straddle lo_rows).
__device__ __forceinline__ int box_row(const GemvParams& p, int y) {
  return static_cast<int>(y < p.lo_rows ? y : p.hi_row0 + (y - p.lo_rows));
}

// Per-row inputs of the statistics and the draw, read once at the start of the kernel (after
// its dependency wait) so that the last block's finish does not wait on global loads.
struct RowInputs {
  float invT[kMaxRows];     // 1 / T (1 at T <= 0)
  float T[kMaxRows];        // the row's request temperature
  uint64_t seed[kMaxRows];  // draft head only
  int64_t pos[kMaxRows];    // draft head only
};
static_assert(sizeof(RowInputs) == 192, "row inputs");

// Called by threads r = 0..7 of the block (each fills its row; rows past nrows get T = 1).
__device__ __forceinline__ void load_row_inputs(const GemvParams& p, RowInputs* ri, int r) {
  const bool live = r < p.nrows;
  const float T = live ? p.temperature[r / p.rows_per_req] : 1.f;
  ri->T[r] = T;
  ri->invT[r] = __fdiv_rn(1.f, T > 0.f ? T : 1.f);
  ri->seed[r] = (live && p.draft) ? p.seed[r] : 0ull;
  ri->pos[r] = (live && p.draft) ? p.pos[r] : 0;
}

// uint64 (below 2^53) to fp32 from its two 32-bit halves: 32-bit conversions only.
__device__ __forceinline__ float u64_to_f32(unsigned long long v) {
  return __fmaf_rn(__uint2float_rn(static_cast<uint32_t>(v >> 32)), 4294967296.f,
                   __uint2float_rn(static_cast<uint32_t>(v)));
}

// Weight of one logit in the tile's integer sum: exp((z - m) / T) in [0, 1], in 2^-40 units.
// The same expression is evaluated in the tile pass and in the draw's rescan, with explicit
// round-to-nearest operations (no contraction), so both see identical integers.
__device__ __forceinline__ unsigned long long tile_weight(float z, float m, float invT) {
  return quantise(expf(__fmul_rn(__fsub_rn(z, m), invT)));
}

// One block's partial statistics of each row from its logit tile in shared memory: top-2 and
// NaN / +Inf flag, and the exact integer sum of tile_weight(z, m) relative to the block max m.
// Called by all `nwarps` warps after a __syncthreads that publishes ztile.
static __device__ __forceinline__ void gemv_block_partials(const GemvParams& p, const float* ztile,
                                                           int64_t v0, int nt, int nwarps,
                                                           const RowInputs* ri) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q = warp; q < p.nrows; q += nwarps) {
    const float invT = ri->invT[q];
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
      p.part[static_cast<size_t>(blockIdx.x) * kMaxRows + q] = pp;
    }
  }
}

// Greedy acceptance of request b by one warp, from its verify rows' statistics st[b*R + r]:
// the rule and status codes of spec_accept at T <= 0 (lucebox-hub PR #15, "Exactness": accept
// d_i while it is the argmax of row i - 1, emit the argmax at the first mismatch or the bonus
// argmax of row k after all k; EOS ends the block). Lane i holds draft i and row i.
//
// What it reads from global memory (k, the drafts, the 14 counter words, one a lane) is loaded
// by greedy_prefetch when the last block starts its combine, so that those loads overlap it;
// after the decision every lane stores its own counter word: no chain of round trips.
struct GreedyPre {
  int k, x_any;
  unsigned long long cnt;  // counter word `lane` of the request (lane < 14)
};
static __device__ __forceinline__ GreedyPre greedy_prefetch(const GemvParams& p, int b,
                                                            int lane) {
  GreedyPre g;
  g.k = p.acc_k[b];
  g.x_any = (lane < p.acc_k_max) ? p.acc_drafts[static_cast<size_t>(b) * p.acc_k_max + lane]
                                 : -1;
  g.cnt = (p.acc_counters && lane < 14)
              ? reinterpret_cast<const unsigned long long*>(p.acc_counters + b)[lane]
              : 0ull;
  return g;
}
static __device__ void greedy_accept_warp(const GemvParams& p, int b, int R,
                                          const spec_rowstats* st_rows, int lane,
                                          const GreedyPre& g) {
  const int k = g.k;
  const int kmax = p.acc_k_max;
  int status = SPEC_REQ_OK;
  const bool kbad = (k < 0 || k > kmax || k + 1 > R);
  if (kbad) status = SPEC_REQ_BAD_K;
  spec_rowstats st_any{0.f, 0.f, 0.f, -1};
  if (lane < R) st_any = st_rows[b * R + lane];
  int x = -1;
  bool xbad = false;
  if (!kbad && lane < k) {
    x = g.x_any;
    xbad = (x < 0 || static_cast<int64_t>(x) >= p.V);
  }
  if (status == SPEC_REQ_OK && __any_sync(0xffffffffu, xbad)) status = SPEC_REQ_BAD_TOKEN;
  spec_rowstats st{0.f, 0.f, 0.f, -1};
  bool nf = false;
  if (status == SPEC_REQ_OK) {
    if (lane <= k) {
      st = st_any;
      nf = isnan(st.max);
    }
    if (__any_sync(0xffffffffu, nf)) status = SPEC_REQ_NONFINITE;
  }
  const bool acc = status == SPEC_REQ_OK && lane < k && x == st.argmax;
  const unsigned accmask = __ballot_sync(0xffffffffu, acc);
  // the decision, worked out by every lane alike (status and k are the same in all lanes)
  int ntok = 0, nacc = 0, eos_hit = 0, mytok = -1;  // mytok: the token at position `lane`
  if (status == SPEC_REQ_OK) {
    bool stop = false;
    for (int i = 0; i < k && !stop; ++i) {
      const int xi = __shfl_sync(0xffffffffu, x, i);
      const int ai = __shfl_sync(0xffffffffu, st.argmax, i);
      const int t = ((accmask >> i) & 1u) ? xi : ai;
      if (lane == ntok) mytok = t;
      ++ntok;
      if ((accmask >> i) & 1u) {
        ++nacc;
        if (p.acc_eos >= 0 && xi == p.acc_eos) {
          eos_hit = 1;
          stop = true;
        }
      } else {
        if (p.acc_eos >= 0 && ai == p.acc_eos) eos_hit = 1;
        stop = true;
      }
    }
    if (!stop) {
      const int ak = __shfl_sync(0xffffffffu, st.argmax, k);
      if (lane == ntok) mytok = ak;
      ++ntok;
      if (p.acc_eos >= 0 && ak == p.acc_eos) eos_hit = 1;
    }
  }
  // the result record: lanes 0..7 its tokens, lane 8 the header fields
  spec_accept_out* o = p.acc_out + b;
  if (lane < 8) o->tokens[lane] = lane < ntok ? mytok : -1;
  if (lane == 8) {
    o->status = status;
    o->n_accept = nacc;
    o->n_emit = ntok;
    o->eos_hit = eos_hit;
    o->sample_kind = 0;
    o->sample_row = -1;
    o->reserved[0] = 0;
    o->reserved[1] = 0;
  }
  if (p.acc_counters && lane < 14) {  // word `lane`: cycles, drafted, accepted, emitted, eos,
    unsigned long long add = 0ull;    // errors, depth[0..7]
    const bool ok = status == SPEC_REQ_OK;
    if (lane == 0) add = 1ull;
    else if (lane == 1 && ok) add = static_cast<unsigned long long>(k);
    else if (lane == 2 && ok) add = static_cast<unsigned long long>(nacc);
    else if (lane == 3 && ok) add = static_cast<unsigned long long>(ntok);
    else if (lane == 4 && ok) add = static_cast<unsigned long long>(eos_hit);
    else if (lane == 5 && !ok) add = 1ull;
    else if (lane >= 6 && ok && lane - 6 == (nacc & 7)) add = 1ull;
    reinterpret_cast<unsigned long long*>(p.acc_counters + b)[lane] = g.cnt + add;
  }
  if (p.ad_state && lane == 0) {  // the width update of spec_adapt_width_mirror, fused
    AdaptParams ap;
    ap.B = 0;  // unused by the update of one request
    ap.k_max = p.acc_k_max;
    ap.out = p.acc_out;
    ap.k_used = p.acc_k;
    ap.cost = p.ad_cost;
    ap.cycle_cost = p.ad_cycle_cost;
    ap.alpha = p.ad_alpha;
    ap.state = p.ad_state;
    ap.k_next = p.ad_k_next;
    ap.k_mirror = p.ad_k_mirror;
    spec_accept_out r;  // the fields of this cycle's record the update reads
    r.status = status;
    r.n_accept = nacc;
    r.n_emit = ntok;
    r.eos_hit = eos_hit;
    adapt_request(ap, b, r);
  }
}

// After every block has written its partials: the ticket, and in the last block the combine
// of each row's partials into its statistics and, for the draft head, the token. All `nwarps`
// (>= 8) warps call it; `scratch` (free shared memory, 8-byte aligned) needs
// gemv_finish_scratch_bytes(gridDim.x) bytes; flags[1] is a free shared int.
static __device__ __forceinline__ void gemv_finish(const GemvParams& p, uint8_t* scratch,
                                                   int* flags, int nwarps, const RowInputs* ri) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int GR = gridDim.x;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&p.hdr->gemv_ticket, 1u);
    flags[1] = (ticket == static_cast<unsigned>(GR) - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!flags[1]) return;
  __threadfence();

  // the fused greedy acceptance's global reads, issued now so that they overlap the combine
  GreedyPre gpre{0, -1, 0ull};
  if (p.acc_out && warp < min(p.nrows, kMaxRows) / max(p.rows_per_req, 1))
    gpre = greedy_prefetch(p, warp, lane);

  // ---------------- last block: combine the partials of every block ----------------
  // All threads first copy the partials of every (block, row) into shared memory in one round
  // of loads. Row q's region of the scratch holds blk_s (uint64 integer sums), blk_m (block
  // maxima, later the scale factors f = exp((m_c - M)/T)), blk_w (runners-up, later the block
  // weights s_c * f) and blk_i (argmax indices). The combine runs in fp32 (a fixed order, so
  // deterministic; relative error ~1e-6), keeping the 64-bit work on the integer units.
  const int nr = min(p.nrows, kMaxRows);
  const size_t rstride = gemv_finish_row_bytes(GR);
  int* s_rbad = reinterpret_cast<int*>(scratch + kMaxRows * rstride);  // [8]
  // [8]: the rows' statistics, for the fused greedy acceptance
  spec_rowstats* s_st = reinterpret_cast<spec_rowstats*>(scratch + kMaxRows * rstride + 64);
  if (tid < kMaxRows) s_rbad[tid] = 0;
  __syncthreads();
  for (int i = tid; i < GR * nr; i += blockDim.x) {
    const int cc = i / nr, q = i - cc * nr;
    const uint4* pp = reinterpret_cast<const uint4*>(p.part + static_cast<size_t>(cc) * kMaxRows + q);
    const uint4 a = __ldcg(pp), b = __ldcg(pp + 1);
    uint8_t* base = scratch + q * rstride;
    const int32_t idx = static_cast<int32_t>(a.z);
    reinterpret_cast<unsigned long long*>(base)[cc] = (static_cast<unsigned long long>(b.y) << 32) | b.x;
    reinterpret_cast<float*>(base + 8 * GR)[cc] = (idx >= 0) ? __uint_as_float(a.x) : -INFINITY;
    reinterpret_cast<float*>(base + 12 * GR)[cc] = __uint_as_float(a.y);
    reinterpret_cast<int32_t*>(base + 16 * GR)[cc] = idx;
    if (a.w) atomicOr(&s_rbad[q], 1);
  }
  __syncthreads();
  for (int q = warp; q < nr; q += nwarps) {
    uint8_t* base = scratch + q * rstride;
    unsigned long long* blk_s = reinterpret_cast<unsigned long long*>(base);
    float* blk_m = reinterpret_cast<float*>(base + 8 * GR);
    float* blk_w = reinterpret_cast<float*>(base + 12 * GR);
    const int32_t* blk_i = reinterpret_cast<const int32_t*>(base + 16 * GR);
    const float T = ri->T[q];
    const float invT = ri->invT[q];
    const uint64_t seed_q = ri->seed[q];
    const int64_t pos_q = ri->pos[q];
    Top2 t = top2_empty();
    for (int cc = lane; cc < GR; cc += 32) {
      const int32_t idx = blk_i[cc];
      if (idx >= 0) t = top2_merge(t, Top2{blk_m[cc], blk_w[cc], idx});
    }
    int bad = s_rbad[q];
    t = warp_top2(t);
    const bool nonfinite = bad || t.idx == kNoIndex || t.best == -INFINITY;
    const float M = t.best;
    float S = 0.f;
    for (int cc = lane; cc < GR; cc += 32) {  // entries this lane read above
      const float mc = blk_m[cc];
      float f = 0.f;
      if (!nonfinite && mc != -INFINITY) f = expf(__fmul_rn(__fsub_rn(mc, M), invT));
      blk_m[cc] = f;
      blk_w[cc] = __fmul_rn(u64_to_f32(blk_s[cc]), f);
      S = __fadd_rn(S, blk_w[cc]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, o));
    spec_rowstats st;
    if (nonfinite) {
      st.max = __int_as_float(0x7fc00000);
      st.log_norm = st.max;
      st.gap = st.max;
      st.argmax = -1;
    } else {
      st.max = M;
      st.log_norm = __fsub_rn(logf(S), 27.725887222397812f);  // log(S * 2^-40)
      st.gap = __fsub_rn(M, t.second);
      st.argmax = t.idx < 0 ? t.idx : row_id(p, t.idx);
    }
    if (lane == 0 && p.stats) p.stats[q] = st;
    if (lane == 0) s_st[q] = st;

    if (p.draft) {
      int32_t tok = -1;
      if (!nonfinite && !(T > 0.f)) tok = t.idx;
      if (!nonfinite && T > 0.f && p.logits) {
        // inverse CDF: the first block whose cumulative weight exceeds u*S, then the first token
        // inside it whose cumulative integer weight exceeds the remainder. Each lane walks a
        // contiguous chunk of blocks from its exclusive prefix; the first lane with a hit wins.
        __syncwarp();
        const uint32_t u24 = uniform_u24(seed_q, pos_q + p.pos_offset, PURPOSE_DRAFT);
        const float target = __fmul_rn(__fmul_rn(static_cast<float>(u24), 5.9604644775390625e-08f), S);
        const int nb = (GR + 31) / 32;
        const int b_lo = min(GR, lane * nb), b_hi = min(GR, b_lo + nb);
        float lsum = 0.f;
        for (int cc = b_lo; cc < b_hi; ++cc) lsum = __fadd_rn(lsum, blk_w[cc]);
        float incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl = __fadd_rn(incl, up);
        }
        float cum = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) cum = 0.f;
        int hit = -1, last_nz = -1;
        float cum_hit = 0.f;
        for (int cc = b_lo; cc < b_hi; ++cc) {
          const float w = blk_w[cc];
          if (w > 0.f) last_nz = cc;
          if (hit < 0 && w > 0.f && __fadd_rn(cum, w) > target) {
            hit = cc;
            cum_hit = cum;
          }
          cum = __fadd_rn(cum, w);
        }
        const unsigned hmask = __ballot_sync(0xffffffffu, hit >= 0);
        int cstar;
        float frac = 1.f;  // the target's position inside the chosen block, as a fraction of it
        if (hmask) {
          const int L = __ffs(hmask) - 1;
          cstar = __shfl_sync(0xffffffffu, hit, L);
          cum_hit = __shfl_sync(0xffffffffu, cum_hit, L);
          frac = __fdiv_rn(__fsub_rn(target, cum_hit), blk_w[cstar]);
          if (!(frac >= 0.f)) frac = 0.f;
        } else {  // rounding left u*S past the total: the last block with weight
          cstar = last_nz;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) cstar = max(cstar, __shfl_xor_sync(0xffffffffu, cstar, o));
        }
        if (cstar >= 0) {
          // the block's logits in per-lane chunks: exact integer weights against the block max,
          // an inclusive scan of the chunk sums (its last entry is the block's integer total I),
          // the target tt = floor(frac * I), then the warp walks the one chunk that holds it
          int64_t c0, c1;
          block_rows(cstar, GR, p.nbands, p.band_rows, p.V, c0, c1);
          const float mc = __ldcg(&(p.part + static_cast<size_t>(cstar) * kMaxRows + q)->m);
          const float* yrow = p.logits + static_cast<size_t>(q) * p.logits_stride;
          const int64_t n2 = (c1 - c0 + 31) / 32;
          const int64_t lo = min(c1, c0 + lane * n2), hi = min(c1, lo + n2);
          unsigned long long lw = 0ull;
          for (int64_t base = lo; base < hi; base += 8) {  // eight loads in flight per lane
            float z[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) z[u] = (base + u < hi) ? __ldcg(yrow + base + u) : -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              if (base + u < hi && !(isnan(z[u]) || z[u] == INFINITY))
                lw += tile_weight(z[u], mc, invT);
          }
          unsigned long long inc = lw;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long up = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += up;
          }
          const unsigned long long I = __shfl_sync(0xffffffffu, inc, 31);
          unsigned long long tt = I - 1ull;  // I >= 2^40: the block max itself weighs 2^40
          if (frac < 1.f) {
            const unsigned long long t2 = __float2ull_rd(__fmul_rn(frac, u64_to_f32(I)));
            tt = t2 < tt ? t2 : tt;
          }
          const unsigned lmask = __ballot_sync(0xffffffffu, lw > 0ull && inc > tt);
          if (lmask) {
            // the whole warp walks the winning lane's chunk, 32 tokens per round
            const int L = __ffs(lmask) - 1;
            unsigned long long carry = __shfl_sync(0xffffffffu, inc - lw, L);  // exact
            const int64_t clo = __shfl_sync(0xffffffffu, lo, L);
            const int64_t chi = __shfl_sync(0xffffffffu, hi, L);
            for (int64_t base = clo; base < chi && tok < 0; base += 32) {
              const int64_t v = base + lane;
              unsigned long long w = 0ull;
              if (v < chi) {
                const float z = __ldcg(yrow + v);
                if (!(isnan(z) || z == INFINITY)) w = tile_weight(z, mc, invT);
              }
              unsigned long long incl = w;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long up = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += up;
              }
              const unsigned mask = __ballot_sync(0xffffffffu, w > 0ull && carry + incl > tt);
              if (mask) tok = static_cast<int32_t>(base + __ffs(mask) - 1);
              carry += __shfl_sync(0xffffffffu, incl, 31);
            }
          }
        }
      }
      if (lane == 0)
        p.token_out[static_cast<size_t>(q) * p.token_stride] = tok < 0 ? tok : row_id(p, tok);
    }
  }
  if (p.acc_out) {  // the fused greedy acceptance, one warp per request
    __syncthreads();
    const int R = max(p.rows_per_req, 1);
    if (warp < nr / R) greedy_accept_warp(p, warp, R, s_st, lane, gpre);  // B <= 8 <= nwarps
  }
  if (tid == 0) p.hdr->gemv_ticket = 0u;
}

// Partials from the block's logit tile, then gemv_finish.
static __device__ __forceinline__ void gemv_block_epilogue(const GemvParams& p, const float* ztile,
                                                           int64_t v0, int nt, uint8_t* scratch,
                                                           int* flags, int nwarps,
                                                           const RowInputs* ri) {
  gemv_block_partials(p, ztile, v0, nt, nwarps, ri);
  gemv_finish(p, scratch, flags, nwarps, ri);
}

}  // namespace spec
