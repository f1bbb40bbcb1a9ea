// Acceptance, residual correction, bonus token and EOS truncation for B requests.
//
// Rules (lucebox-hub PR #15 "MTP speculative decoding", section "Exactness": a greedy draft
// is accepted only if it equals the trunk's token; DS4Server issue #98 "Add Qwen3.8 Flash Next
// native MTP speculation", section "Implementation" and closing comment: a draft is kept when
// u*q <= p, a rejection is replaced by a draw from max(0, p - q), zero and non-finite
// probabilities get defined outcomes, an EOS among the drafts ends the block) -- see
// spec_accept in spec.h for the exact statement.
//
// Work layout: grid (slices, B), one block per 1,024-entry slice of the vocabulary of one
// request. Every block first takes the O(k) decision for its request (identical in every
// block); when the decision needs a draw over the whole vocabulary (residual at the first
// rejection, or the bonus at temperature > 0) each block sums its slice's weights, quantised
// to 2^-40 units, in exact 64-bit integers; the last block of the request (a per-request
// ticket, no inter-block waiting) picks the slice holding the target and rescans it. Integer
// sums make the drawn token independent of block scheduling and summation order.
//
// Filtered mode (spec_accept_filtered: top-k / top-p target, one-hot q): each block reduces
// every verify row of its slice to the slice's best top_k entries (a 64-bit key orders by
// logit, then by lower id; one warp per row: a threshold cut and a bitonic sort of the keys
// above it); the last block merges the slices' sorted lists, one warp per row (a tournament
// over their heads), then row by row cuts at top-p and takes the decisions and draws on the
// <= 32 survivors in exact integer weights.
#include <math.h>

#include "adapt_core.cuh"
#include "params.cuh"

namespace spec {

constexpr int kAcceptSumSlots = kMaxRows;  // per-slice integer sums: one per verify row
// shared memory for one row's candidate keys in the filtered mode's last block (40 KB: up to
// 160 slices x 32, or V = 151,936 at any top-k); larger rows are merged from L2
constexpr int kFilterStageKeys = 5120;


struct Decision {
  int status, n_accept, ntok, eos_hit;
  int tokens[8];
  int need;  // 0 none, 1 residual draw, 2 bonus draw, 3 exact-match draws (rows 0..srow),
             // 4 filtered decisions (rows 0..srow)
  int srow;  // verify row of the draw
  int xrej;  // the rejected draft (one-hot q)
  int pad;
};

// Draft row holding vocabulary id x: x below lo, lo + x - hi0 from hi0 while inside the Vd
// draft rows, -1 for ids the draft set does not cover (q = 0 there).
__device__ __forceinline__ int64_t draft_row_of(int64_t x, int64_t lo, int64_t hi0, int64_t Vd) {
  if (x < lo) return x;
  const int64_t r = lo + (x - hi0);
  return (x >= hi0 && r < Vd) ? r : -1;
}

// p(v) = exp((z - max)/T) * exp(-log_norm), every operation rounded on its own.
__device__ __forceinline__ float prob_of(float z, float mx, float invT, float inv_norm) {
  return __fmul_rn(expf(__fmul_rn(__fsub_rn(z, mx), invT)), inv_norm);
}

struct DrawCtx {
  const float* prow;  // verify logits row of the draw
  float pmax, pinvT, pinv_norm;
  const float* qrow;  // draft logits row (residual with q_logits), else null
  float qmax, qinv_norm;
  int64_t Vd, qlo, qhi0;  // draft rows and their map (draft_row_of)
  int xrej;        // one-hot q position (residual without q_logits), else -1
  bool residual;
};

// The two integer weights of vocabulary entry j: residual max(0, p - q) and p itself. The
// logit and draft rows are read-only in this kernel, so they are read through L1.
__device__ __forceinline__ void entry_weights(const DrawCtx& c, int64_t j,
                                              unsigned long long& wr,
                                              unsigned long long& wp) {
  const float pj = prob_of(__ldg(c.prow + j), c.pmax, c.pinvT, c.pinv_norm);
  wp = quantise(pj);
  if (!c.residual) {
    wr = wp;
    return;
  }
  float qj = 0.f;
  if (c.qrow) {
    const int64_t jr = draft_row_of(j, c.qlo, c.qhi0, c.Vd);
    if (jr >= 0) qj = prob_of(__ldg(c.qrow + jr), c.qmax, c.pinvT, c.qinv_norm);
  } else {
    qj = (j == c.xrej) ? 1.f : 0.f;
  }
  wr = quantise(fmaxf(0.f, __fsub_rn(pj, qj)));
}

// Weights of the four contiguous entries jb..jb+3 (zero past V): p's if use_p, else the
// residual's. The loads of all four entries are issued before any is used.
__device__ __forceinline__ unsigned long long entry_weights4(const DrawCtx& c, int64_t jb,
                                                             int64_t V, bool use_p,
                                                             unsigned long long* w) {
  float z[4], y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    z[e] = (jb + e < V) ? __ldg(c.prow + jb + e) : -INFINITY;
    y[e] = -INFINITY;
    if (c.residual && c.qrow && jb + e < V) {
      const int64_t jr = draft_row_of(jb + e, c.qlo, c.qhi0, c.Vd);
      if (jr >= 0) y[e] = __ldg(c.qrow + jr);
    }
  }
  unsigned long long t = 0ull;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int64_t j = jb + e;
    unsigned long long we = 0ull;
    if (j < V) {
      const float pj = prob_of(z[e], c.pmax, c.pinvT, c.pinv_norm);
      if (use_p || !c.residual) {
        we = quantise(pj);
      } else {
        float qj = 0.f;
        if (c.qrow)
          qj = (y[e] == -INFINITY) ? 0.f : prob_of(y[e], c.qmax, c.pinvT, c.qinv_norm);
        else
          qj = (j == c.xrej) ? 1.f : 0.f;
        we = quantise(fmaxf(0.f, __fsub_rn(pj, qj)));
      }
    }
    w[e] = we;
    t += we;
  }
  return t;
}

// Block sums of two values at once (one pair of barriers); sh holds 2 per warp.
__device__ __forceinline__ void block_sum2_u64(unsigned long long& a, unsigned long long& b,
                                               unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum_u64(a);
  b = warp_sum_u64(b);
  __syncthreads();
  if (lane == 0) {
    sh[2 * warp] = a;
    sh[2 * warp + 1] = b;
  }
  __syncthreads();
  unsigned long long ta = 0ull, tb = 0ull;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
    ta += sh[2 * w];
    tb += sh[2 * w + 1];
  }
  a = ta;
  b = tb;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  unsigned long long t = 0ull;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += sh[w];
  return t;
}

// Inclusive scan of one value per thread across the block (ascending thread order); returns
// the thread's inclusive prefix and, through *total, the block total.
__device__ __forceinline__ unsigned long long block_incl_scan_u64(unsigned long long w,
                                                                  unsigned long long* sh,
                                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long up = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += up;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  unsigned long long before = 0ull, t = 0ull;
  for (int w2 = 0; w2 < static_cast<int>(blockDim.x >> 5); ++w2) {
    if (w2 < warp) before += sh[w2];
    t += sh[w2];
  }
  *total = t;
  return before + incl;
}

// The draw context of verify row `row` of request b: p at temperature T, and for a residual
// the draft distribution (q rows, or one-hot at the rejected draft `xrej`). pst / qst: the
// request's verify-row and draft-row statistics, copied to shared memory by the decision.
__device__ __forceinline__ DrawCtx draw_ctx(const AcceptParams& p, int b, int row, bool residual,
                                            int xrej, float T, const spec_rowstats* pst,
                                            const spec_rowstats* qst) {
  DrawCtx c;
  const size_t prow = static_cast<size_t>(b) * p.R + row;
  c.prow = p.logits + prow * p.V;
  c.pmax = pst[row].max;
  c.pinvT = __fdiv_rn(1.f, T);
  c.pinv_norm = expf(-pst[row].log_norm);
  c.residual = residual;
  c.qrow = nullptr;
  c.qmax = 0.f;
  c.qinv_norm = 0.f;
  c.Vd = p.Vd;
  c.qlo = p.q_lo;
  c.qhi0 = p.q_hi0;
  c.xrej = -1;
  if (residual) {
    if (p.q_logits) {
      const size_t qr = static_cast<size_t>(row) * p.B + b;
      c.qrow = p.q_logits + qr * p.q_stride;
      c.qmax = qst[row].max;
      c.qinv_norm = expf(-qst[row].log_norm);
    } else {
      c.xrej = xrej;
    }
  }
  return c;
}

// Inverse-CDF draw over request b's vocabulary from slot `slot` of its slice sums (the exact
// integer weights the context defines: p if use_p, else the residual): the slice whose
// cumulative weight first exceeds u*total by a block-parallel scan, then the token inside it by
// rescanning the slice. Called by every thread of the block; returns the token (-1 only if the
// total is zero, which the callers exclude).
__device__ int draw_token(const AcceptParams& p, int b, const DrawCtx& c, bool use_p, int slot,
                          uint32_t u24, unsigned long long* sh, int* s_slice,
                          unsigned long long* s_before, int* s_tok) {
  const int tid = threadIdx.x;
  const unsigned long long* rs = p.sums + static_cast<size_t>(b) * p.NS * kAcceptSumSlots;
  unsigned long long tot = 0ull;
  for (int i = tid; i < p.NS; i += kAcceptThreads) tot += __ldcg(rs + kAcceptSumSlots * i + slot);
  tot = block_sum_u64(tot, sh);
  const unsigned long long target = cdf_target(u24, tot);
  if (tid == 0) {
    *s_slice = -1;
    *s_tok = -1;
  }
  {
    unsigned long long carry = 0ull;
    for (int base = 0; base < p.NS; base += kAcceptThreads) {
      const int i = base + tid;
      const unsigned long long w = (i < p.NS) ? __ldcg(rs + kAcceptSumSlots * i + slot) : 0ull;
      unsigned long long round_total;
      const unsigned long long cum = carry + block_incl_scan_u64(w, sh, &round_total);
      if (w > 0ull && cum > target && cum - w <= target) {
        *s_slice = i;
        *s_before = cum - w;
      }
      carry += round_total;
      __syncthreads();
      if (*s_slice >= 0) break;
    }
  }
  if (*s_slice >= 0) {
    const int64_t base = static_cast<int64_t>(*s_slice) * kAcceptSlice;
    unsigned long long carry = *s_before;
    for (int e = 0; e < kAcceptSlice / kAcceptThreads; ++e) {
      const int64_t j = base + e * kAcceptThreads + tid;
      unsigned long long w = 0ull;
      if (j < p.V) {
        unsigned long long wr, wp;
        entry_weights(c, j, wr, wp);
        w = use_p ? wp : wr;
      }
      unsigned long long round_total;
      const unsigned long long cum = carry + block_incl_scan_u64(w, sh, &round_total);
      if (w > 0ull && cum > target && cum - w <= target) *s_tok = static_cast<int>(j);
      carry += round_total;
      __syncthreads();
      if (*s_tok >= 0) break;
    }
  }
  __syncthreads();
  return *s_tok;
}

// Inverse-CDF draw for a vocabulary of at most kAcceptThreads slices, thread i holding slice
// i's integer weight w_i (0 from NS on): one block scan finds the slice whose cumulative weight
// first exceeds floor(u * total), one pass over its 1,024 entries (four contiguous entries a
// thread, all loads in flight together) and a second scan find the token. Two scans and one
// round of loads, against a round per 256 entries in draw_token. Called by every thread;
// returns the token (-1 when the total is zero).
__device__ int draw_in_slices(const AcceptParams& p, const DrawCtx& c, bool use_p,
                              unsigned long long w_i, uint32_t u24, unsigned long long* sh,
                              int* s_slice, unsigned long long* s_before, int* s_tok) {
  const int tid = threadIdx.x;
  unsigned long long tot;
  const unsigned long long incl = block_incl_scan_u64(w_i, sh, &tot);
  if (tot == 0ull) return -1;  // uniform: every thread holds the same total
  const unsigned long long target = cdf_target(u24, tot);
  if (tid == 0) *s_tok = -1;
  if (w_i > 0ull && incl > target && incl - w_i <= target) {  // exactly one thread
    *s_slice = tid;
    *s_before = incl - w_i;
  }
  __syncthreads();
  const int64_t jb = static_cast<int64_t>(*s_slice) * kAcceptSlice + 4 * tid;
  const unsigned long long before = *s_before;
  unsigned long long w[4];
  const unsigned long long ts = entry_weights4(c, jb, p.V, use_p, w);
  unsigned long long tt;
  unsigned long long cum = before + block_incl_scan_u64(ts, sh, &tt) - ts;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (w[e] > 0ull && cum <= target && cum + w[e] > target) *s_tok = static_cast<int>(jb + e);
    cum += w[e];
  }
  __syncthreads();
  return *s_tok;
}

// ---------------------------------------------------------------------- filtered acceptance
// Order-preserving 64-bit key of (logit, id): larger logit first, then lower id; -0 counts as
// +0. Real keys are never 0 (that would need a NaN logit), so 0 marks "no entry".
__device__ __forceinline__ unsigned long long rank_key(float z, int64_t id) {
  uint32_t u = __float_as_uint(z == 0.f ? 0.f : z);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) |
         (0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t u = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ int key_id(unsigned long long key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v,
                                                            unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  unsigned long long t = 0ull;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t = sh[w] > t ? sh[w] : t;
  return t;
}

// One compare-exchange step of a descending bitonic sort over a warp's elements i = lane + 32 h
// (block size kb, stride j < 32): the lower index of a pair keeps the larger key in a
// descending block ((i & kb) == 0), the smaller in an ascending one.
__device__ __forceinline__ unsigned long long bitonic_step(unsigned long long v, int i, int kb,
                                                           int j) {
  const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
  const bool desc = (i & kb) == 0, lower = (i & j) == 0;
  const unsigned long long hi = v > o ? v : o, lo = v > o ? o : v;
  return (desc == lower) ? hi : lo;
}

// The K (<= 32) largest of 64 keys, two per lane (positions lane and lane + 32), sorted
// descending into positions 0..K-1: a bitonic sort over the warp.
__device__ __forceinline__ void warp_sort64_desc(unsigned long long& a, unsigned long long& b) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kb = 2; kb <= 64; kb <<= 1) {
#pragma unroll
    for (int j = kb >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // the pair (lane, lane + 32) sits in one lane
        const bool desc = (lane & kb) == 0;
        const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
        a = desc ? hi : lo;
        b = desc ? lo : hi;
      } else {
        a = bitonic_step(a, lane, kb, j);
        b = bitonic_step(b, lane + 32, kb, j);
      }
    }
  }
}

// The best K keys of verify row `row` of request b over slice sl, descending, written to the
// workspace (0 past the last entry). Called by one warp: lane l holds entries l + 32 i.
// A threshold cut first: the K-th largest of the 32 lane maxima bounds the slice's K-th key
// from below (those K maxima are keys), so only keys at or above it can be in the top K;
// when at most 64 are, they are gathered in `buf` (64 keys of shared memory for this warp) and
// sorted. Otherwise (keys concentrated in a few lanes) K rounds of a warp maximum select them.
__device__ __forceinline__ void slice_topk_warp(const AcceptParams& p, int b, int sl, int row, int K,
                                                unsigned long long* buf) {
  const int lane = threadIdx.x & 31;
  const float* z = p.logits + (static_cast<size_t>(b) * p.R + row) * p.V;
  const int64_t j0 = static_cast<int64_t>(sl) * kAcceptSlice;
  unsigned long long key[kAcceptSlice / 32];
#pragma unroll
  for (int e = 0; e < kAcceptSlice / 32; ++e) {
    const int64_t j = j0 + e * 32 + lane;
    key[e] = (j < p.V) ? rank_key(__ldcg(z + j), j) : 0ull;
  }
  unsigned long long* out =
      p.cand + ((static_cast<size_t>(b) * p.NS + sl) * kMaxRows + row) * kMaxTopK;
  {
    unsigned long long t[kAcceptSlice / 64];  // the lane's maximum by a 5-level tree
#pragma unroll
    for (int e = 0; e < kAcceptSlice / 64; ++e)
      t[e] = key[2 * e] > key[2 * e + 1] ? key[2 * e] : key[2 * e + 1];
#pragma unroll
    for (int w = kAcceptSlice / 128; w >= 1; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) t[e] = t[e] > t[e + w] ? t[e] : t[e + w];
    unsigned long long mx = t[0];  // sort the 32 lane maxima descending: position K-1 = L
#pragma unroll
    for (int kb = 2; kb <= 32; kb <<= 1)
#pragma unroll
      for (int j = kb >> 1; j > 0; j >>= 1) mx = bitonic_step(mx, lane, kb, j);
    const unsigned long long L = __shfl_sync(0xffffffffu, mx, K - 1);
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kAcceptSlice / 32; ++e) cnt += (key[e] != 0ull && key[e] >= L) ? 1 : 0;
    int incl = cnt;  // inclusive prefix of the counts over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    const int n = __shfl_sync(0xffffffffu, incl, 31);
    if (L != 0ull && n <= 64) {
      int at = incl - cnt;
#pragma unroll
      for (int e = 0; e < kAcceptSlice / 32; ++e)
        if (key[e] != 0ull && key[e] >= L) buf[at++] = key[e];
      __syncwarp();
      unsigned long long a = lane < n ? buf[lane] : 0ull;
      unsigned long long c = lane + 32 < n ? buf[lane + 32] : 0ull;
      __syncwarp();  // buf is free again for the warp's next row
      warp_sort64_desc(a, c);
      if (lane < K) out[lane] = a;  // K <= 32: positions 0..K-1 are all in a
      return;
    }
  }
  for (int r = 0; r < K; ++r) {
    // the lane's largest key by a 5-level tree (a linear scan is a 31-deep dependent chain)
    unsigned long long t[kAcceptSlice / 64];
#pragma unroll
    for (int e = 0; e < kAcceptSlice / 64; ++e)
      t[e] = key[2 * e] > key[2 * e + 1] ? key[2 * e] : key[2 * e + 1];
#pragma unroll
    for (int w = kAcceptSlice / 128; w >= 1; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) t[e] = t[e] > t[e + w] ? t[e] : t[e + w];
    const unsigned long long wm = warp_max_u64(t[0]);
    if (lane == 0) out[r] = wm;
#pragma unroll
    for (int e = 0; e < kAcceptSlice / 32; ++e)
      if (key[e] == wm) key[e] = 0ull;  // keys are unique: only the winner matches
  }
}

// The best K keys of row `row` over the whole vocabulary: a tournament over the slices' sorted
// lists (each thread holds the heads of slices tid + 256 m, m < 4). When the row's NS x K keys
// fit in `stage` (dynamic shared memory) they are first copied there in one coalesced pass, so
// that a round's winner reads its next key from shared memory: read from L2 instead, that load
// sits on the critical path of every round. Called by every thread.
__device__ __forceinline__ void merge_rows_topk(const AcceptParams& p, int b, int row, int K,
                                unsigned long long* s_top, unsigned long long* sh,
                                unsigned long long* stage, int stage_keys) {
  const int tid = threadIdx.x;
  const unsigned long long* base = p.cand + static_cast<size_t>(b) * p.NS * kMaxRows * kMaxTopK;
  const bool staged = p.NS * K <= stage_keys;
  if (staged) {
    for (int i = tid; i < p.NS * K; i += kAcceptThreads) {
      const int s = i / K, j = i - s * K;
      stage[i] = __ldcg(base + (static_cast<size_t>(s) * kMaxRows + row) * kMaxTopK + j);
    }
    __syncthreads();
  }
  auto at = [&](int s, int j) {
    return staged ? stage[s * K + j]
                  : __ldcg(base + (static_cast<size_t>(s) * kMaxRows + row) * kMaxTopK + j);
  };
  int ptr[4];
  unsigned long long head[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int s = tid + kAcceptThreads * m;
    ptr[m] = 0;
    head[m] = (s < p.NS) ? at(s, 0) : 0ull;
  }
  for (int r = 0; r < K; ++r) {
    unsigned long long m = head[0];
#pragma unroll
    for (int i = 1; i < 4; ++i) m = head[i] > m ? head[i] : m;
    const unsigned long long bm = block_max_u64(m, sh);
    if (tid == 0) s_top[r] = bm;
    if (bm != 0ull) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (head[i] == bm) {
          const int s = tid + kAcceptThreads * i;
          ++ptr[i];
          head[i] = (ptr[i] < K) ? at(s, ptr[i]) : 0ull;
        }
      }
    }
  }
  __syncthreads();
}

// The same top-K of row `row` by one warp, for at most 32 * kWarpMergeLists slices: lane l
// holds the head and the next key of slices l + 32 i in registers; a round is the lane maxima's
// warp maximum, and the winning lane moves its slice to the prefetched next key and loads the
// one after (needed no earlier than that slice's next win). Keys are unique, so the result is
// the block tournament's. With one warp per row all rows merge at once (the block tournament
// ran the rows one after another, two block barriers a round).
constexpr int kWarpMergeLists = 8;
__device__ __forceinline__ void merge_row_topk_warp(const AcceptParams& p, int b, int row, int K,
                                                    unsigned long long* out) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* base = p.cand + static_cast<size_t>(b) * p.NS * kMaxRows * kMaxTopK;
  auto at = [&](int s, int j) {
    return __ldcg(base + (static_cast<size_t>(s) * kMaxRows + row) * kMaxTopK + j);
  };
  unsigned long long head[kWarpMergeLists], next[kWarpMergeLists];
  int ptr[kWarpMergeLists];
#pragma unroll
  for (int i = 0; i < kWarpMergeLists; ++i) {
    const int s = lane + 32 * i;
    ptr[i] = 0;
    head[i] = (s < p.NS) ? at(s, 0) : 0ull;
    next[i] = (s < p.NS && K > 1) ? at(s, 1) : 0ull;
  }
  for (int r = 0; r < K; ++r) {
    unsigned long long m = head[0];
#pragma unroll
    for (int i = 1; i < kWarpMergeLists; ++i) m = head[i] > m ? head[i] : m;
    const unsigned long long wm = warp_max_u64(m);
    if (lane == 0) out[r] = wm;
    if (wm == 0ull) continue;  // every list is exhausted: the rest of out is 0 too
#pragma unroll
    for (int i = 0; i < kWarpMergeLists; ++i) {
      if (head[i] == wm) {
        const int s = lane + 32 * i;
        ++ptr[i];
        head[i] = next[i];
        next[i] = (ptr[i] + 1 < K) ? at(s, ptr[i] + 1) : 0ull;
      }
    }
  }
}

// u * W <= w * 2^24 for u = u24 * 2^-24, exactly (128-bit products).
__device__ __forceinline__ bool u_le_ratio(uint32_t u24, unsigned long long W,
                                           unsigned long long w) {
  const unsigned long long lh = __umul64hi(static_cast<unsigned long long>(u24), W);
  const unsigned long long ll = static_cast<unsigned long long>(u24) * W;
  const unsigned long long rh = w >> 40, rl = w << 24;
  return lh < rh || (lh == rh && ll <= rl);
}

// Inverse-CDF draw over (id, weight) pairs in ascending id: the first entry whose cumulative
// weight exceeds floor(u * total); -1 if the total is 0.
__device__ int small_draw(int* id, unsigned long long* w, int n, uint32_t u24) {
  for (int i = 1; i < n; ++i) {  // insertion sort by id (n <= 32)
    const int ki = id[i];
    const unsigned long long kw = w[i];
    int j = i - 1;
    while (j >= 0 && id[j] > ki) {
      id[j + 1] = id[j];
      w[j + 1] = w[j];
      --j;
    }
    id[j + 1] = ki;
    w[j + 1] = kw;
  }
  unsigned long long tot = 0ull;
  for (int i = 0; i < n; ++i) tot += w[i];
  if (tot == 0ull) return -1;
  const unsigned long long target = cdf_target(u24, tot);
  unsigned long long cum = 0ull;
  for (int i = 0; i < n; ++i) {
    cum += w[i];
    if (w[i] > 0ull && cum > target) return id[i];
  }
  return -1;
}

// The counters of one cycle; eos_too = false leaves the EOS count to the caller (the ratio
// rule counts everything else as soon as its decision is known, before the draw).
__device__ void count_cycle(const AcceptParams& p, int b, const Decision& D, int k, int ntok,
                            bool eos_too) {
  if (!p.counters) return;
  spec_counters* c = p.counters + b;
  c->cycles += 1ull;
  if (D.status == SPEC_REQ_OK) {
    c->drafted += static_cast<unsigned long long>(k);
    c->accepted += static_cast<unsigned long long>(D.n_accept);
    c->emitted += static_cast<unsigned long long>(ntok);
    if (eos_too) c->eos += static_cast<unsigned long long>(D.eos_hit);
    c->depth[D.n_accept & 7] += 1ull;
  } else {
    c->errors += 1ull;
  }
}

__device__ void write_result(const AcceptParams& p, int b, const Decision& D) {
  spec_accept_out o;
  o.status = D.status;
  o.n_accept = D.n_accept;
  o.n_emit = D.ntok;
  o.eos_hit = D.eos_hit;
  for (int i = 0; i < 8; ++i) o.tokens[i] = i < D.ntok ? D.tokens[i] : -1;
  o.sample_kind = D.need;
  o.sample_row = D.need ? D.srow : -1;
  o.reserved[0] = 0;
  o.reserved[1] = 0;
  p.out[b] = o;
}

__device__ void finalize(const AcceptParams& p, int b, const Decision& D, int k) {
  write_result(p, b, D);
  count_cycle(p, b, D, k, D.ntok, true);
}

// kFiltered: the instantiation for spec_accept_filtered. The ratio-rule and exact-match modes
// run the other one, which leaves the filtered path's registers out: with them every mode held
// 80-92 registers instead of 62, and 32-request acceptances (thousands of blocks) ran ~25%
// slower for the lost residency.
template <bool kFiltered>
__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(const AcceptParams p) {
  __shared__ Decision D;
  __shared__ int sx[8], sam[8];
  __shared__ spec_rowstats s_pst[kMaxRows], s_qst[kMaxRows];
  __shared__ unsigned long long sh[kAcceptThreads / 32];
  __shared__ unsigned long long s2[2 * (kAcceptThreads / 32)];
  __shared__ int s_last, s_slice, s_tok;
  __shared__ unsigned long long s_before;
  pdl_trigger();
  pdl_wait();  // everything below reads what the LM-head kernels wrote

  const int b = blockIdx.y, sl = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j0 = static_cast<int64_t>(sl) * kAcceptSlice;
  const int k = p.k[b];
  const float T = p.temperature[b];

  // ---------------- the O(k) decision (same in every block of the request) ----------------
  if (warp == 0) {
    int status = SPEC_REQ_OK;
    const bool kbad = (k < 0 || k > p.k_max || k + 1 > p.R);
    if (kbad) status = SPEC_REQ_BAD_K;
    // this lane's draft, verify-row and draft-row statistics, loaded together whatever k is
    // (the indices stay inside the arrays' k_max and R rows): one round of loads
    const int x_any = (lane < p.k_max) ? p.drafts[static_cast<size_t>(b) * p.k_max + lane] : -1;
    spec_rowstats st_any{0.f, 0.f, 0.f, -1}, qs_any{0.f, 0.f, 0.f, -1};
    if (lane < p.R) st_any = p.stats[static_cast<size_t>(b) * p.R + lane];
    if (p.q_logits && lane < p.k_max) qs_any = p.q_stats[static_cast<size_t>(lane) * p.B + b];
    if (lane < kMaxRows) {
      s_pst[lane] = st_any;
      s_qst[lane] = qs_any;
    }
    int x = -1;
    bool xbad = false;
    if (!kbad && lane < k) {
      x = x_any;
      xbad = (x < 0 || static_cast<int64_t>(x) >= p.V);
    }
    if (status == SPEC_REQ_OK && __any_sync(0xffffffffu, xbad)) status = SPEC_REQ_BAD_TOKEN;
    if (status == SPEC_REQ_OK && T > 0.f &&
        (p.logits == nullptr || (p.q_logits != nullptr && p.q_stats == nullptr)))
      status = SPEC_REQ_NO_LOGITS;
    const bool filt = kFiltered && T > 0.f;  // filtered mode: decided in the last block
    if (status == SPEC_REQ_OK && filt) {
      const int tk = p.top_k[b];
      const float tp = p.top_p[b];
      if (tk < 1 || tk > kMaxTopK || !(tp > 0.f && tp <= 1.f)) status = SPEC_REQ_BAD_FILTER;
    }
    spec_rowstats st{0.f, 0.f, 0.f, -1};
    bool nf = false;
    if (status == SPEC_REQ_OK) {
      if (lane <= k) {
        st = st_any;
        nf = isnan(st.max);
      }
      if (T > 0.f && p.q_logits && lane < k) nf = nf || isnan(qs_any.max);
      if (__any_sync(0xffffffffu, nf)) status = SPEC_REQ_NONFINITE;
    }
    const bool exact = p.exact && T > 0.f;  // exact-match mode: decided by the draws below
    bool acc = false;
    if (status == SPEC_REQ_OK && lane < k && !exact && !filt) {
      if (!(T > 0.f)) {
        acc = (x == st.argmax);
      } else {
        const float invT = __fdiv_rn(1.f, T);
        const size_t row = static_cast<size_t>(b) * p.R + lane;
        const float px = prob_of(__ldcg(p.logits + row * p.V + x), st.max, invT,
                                 expf(-st.log_norm));
        float qx = 1.f;
        if (p.q_logits) {
          qx = 0.f;
          const int64_t xr = draft_row_of(x, p.q_lo, p.q_hi0, p.Vd);
          if (xr >= 0) {
            const size_t qr = static_cast<size_t>(lane) * p.B + b;
            qx = prob_of(__ldcg(p.q_logits + qr * p.q_stride + xr), qs_any.max, invT,
                         expf(-qs_any.log_norm));
          }
        }
        const float u = u24_to_float(uniform_u24(p.seed[b], p.pos_base[b] + lane, PURPOSE_ACCEPT));
        acc = (px > 0.f) && (__fmul_rn(u, qx) <= px);
      }
    }
    const unsigned accmask = __ballot_sync(0xffffffffu, acc);
    if (lane < 8) {
      sx[lane] = x;
      sam[lane] = st.argmax;
    }
    __syncwarp();
    if (lane == 0) {
      Decision d;
      d.status = status;
      d.n_accept = 0;
      d.ntok = 0;
      d.eos_hit = 0;
      d.need = 0;
      d.srow = -1;
      d.xrej = -1;
      d.pad = 0;
      if (status == SPEC_REQ_OK && (exact || filt)) {
        d.need = exact ? 3 : 4;
        d.srow = k;
      } else if (status == SPEC_REQ_OK) {
        bool stop = false;
        for (int i = 0; i < k && !stop; ++i) {
          if ((accmask >> i) & 1u) {
            d.tokens[d.ntok++] = sx[i];
            d.n_accept++;
            if (p.eos >= 0 && sx[i] == p.eos) {
              d.eos_hit = 1;
              stop = true;
            }
          } else {
            if (!(T > 0.f)) {
              d.tokens[d.ntok++] = sam[i];
              if (p.eos >= 0 && sam[i] == p.eos) d.eos_hit = 1;
            } else {
              d.need = 1;
              d.srow = i;
              d.xrej = sx[i];
            }
            stop = true;
          }
        }
        if (!stop) {
          if (!(T > 0.f)) {
            d.tokens[d.ntok++] = sam[k];
            if (p.eos >= 0 && sam[k] == p.eos) d.eos_hit = 1;
          } else {
            d.need = 2;
            d.srow = k;
          }
        }
      }
      D = d;
    }
  }
  __syncthreads();

  if (D.need == 0) {
    if (sl == 0 && tid == 0) finalize(p, b, D, k);
    return;
  }
  // the ratio rule's counters are known now except whether the drawn token is EOS
  if ((D.need == 1 || D.need == 2) && sl == 0 && tid == 0) count_cycle(p, b, D, k, D.ntok + 1, false);

  // ---------------- slice sums of the draws' integer weights ----------------
  unsigned long long* mysum = p.sums + (static_cast<size_t>(b) * p.NS + sl) * kAcceptSumSlots;
  if (kFiltered && D.need == 4) {
    // filtered: the slice's best top_k keys of every row 0..k, one warp per row
    __shared__ unsigned long long s_cut[kMaxRows][64];  // each row warp's threshold cut
    if (warp <= k) slice_topk_warp(p, b, sl, warp, p.top_k[b], s_cut[warp]);
  } else if (D.need == 3) {
    // exact-match: the p weights of every row 0..k over this slice, slots 0..k
    unsigned long long sp[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) sp[r] = 0ull;
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r <= k) {
        unsigned long long w[4];
        sp[r] = entry_weights4(draw_ctx(p, b, r, false, -1, T, s_pst, s_qst), j0 + 4 * tid, p.V, true, w);
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r <= k) {
        const unsigned long long t = block_sum_u64(sp[r], sh);
        if (tid == 0) mysum[r] = t;
      }
    }
  } else {
    const DrawCtx c = draw_ctx(p, b, D.srow, D.need == 1, D.xrej, T, s_pst, s_qst);
    unsigned long long w[4];
    unsigned long long sr = entry_weights4(c, j0 + 4 * tid, p.V, false, w);
    unsigned long long sp = sr;
    if (c.residual) sp = entry_weights4(c, j0 + 4 * tid, p.V, true, w);  // loads hit L1
    block_sum2_u64(sr, sp, s2);
    if (tid == 0) {
      mysum[0] = sr;
      mysum[1] = sp;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(p.tickets + b, 1u);
    s_last = (t == static_cast<unsigned>(p.NS) - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---------------- last block of the request: the draws ----------------
  if (D.need == 3) {
    // exact-match: the trunk's own token row by row (U(pos_base + r, BONUS)); keep drafts while
    // they equal it, emit it at the first mismatch, or as the bonus after row k
    __shared__ int s_stop;
    __shared__ Decision E;
    if (tid == 0) {
      E = D;
      s_stop = 0;
    }
    const bool fast = p.NS <= kAcceptThreads;
    const unsigned long long* rs = p.sums + static_cast<size_t>(b) * p.NS * kAcceptSumSlots;
    __syncthreads();
    for (int r = 0; r <= k; ++r) {
      const DrawCtx c = draw_ctx(p, b, r, false, -1, T, s_pst, s_qst);
      const uint32_t u24 = uniform_u24(p.seed[b], p.pos_base[b] + r, PURPOSE_BONUS);
      const unsigned long long wr =
          (fast && tid < p.NS) ? __ldcg(rs + kAcceptSumSlots * tid + r) : 0ull;
      const int tok = fast ? draw_in_slices(p, c, true, wr, u24, sh, &s_slice, &s_before, &s_tok)
                           : draw_token(p, b, c, true, r, u24, sh, &s_slice, &s_before, &s_tok);
      if (tid == 0) {
        E.srow = r;
        E.tokens[E.ntok++] = tok;
        const bool is_eos = (p.eos >= 0 && tok == p.eos);
        if (r < k && tok == sx[r]) {
          E.n_accept++;
          if (is_eos) {
            E.eos_hit = 1;
            s_stop = 1;
          }
        } else {
          if (is_eos) E.eos_hit = 1;
          s_stop = 1;
        }
      }
      __syncthreads();
      if (s_stop) break;
    }
    if (tid == 0) {
      finalize(p, b, E, k);
      p.tickets[b] = 0u;
    }
    return;
  }

  if (kFiltered && D.need == 4) {
    // filtered: row by row, the top-k set (tournament over the slices' lists), the top-p cut,
    // then the ratio test of the draft against p' (q one-hot), a residual draw at the first
    // rejection, or the bonus draw after row k
    __shared__ unsigned long long s_topr[kMaxRows][kMaxTopK];  // each row's top-k, descending
    __shared__ Decision F;
    const int K = p.top_k[b];
    const double tp = static_cast<double>(p.top_p[b]);
    const float invT = __fdiv_rn(1.f, T);
    if (tid == 0) {
      F = D;
      F.need = 0;
      F.srow = -1;
    }
    // every row's top-k set first: one warp per row, all rows at once (up to 256 slices);
    // the block tournament row by row above that
    if (p.NS <= 32 * kWarpMergeLists) {
      if (warp <= k) merge_row_topk_warp(p, b, warp, K, s_topr[warp]);
    } else {
      extern __shared__ unsigned long long f_stage[];  // kFilterStageKeys when launched filtered
      for (int r = 0; r <= k; ++r) {
        merge_rows_topk(p, b, r, K, s_topr[r], sh, f_stage, p.filtered ? kFilterStageKeys : 0);
      }
    }
    __syncthreads();
    // Each row's target p' at once, one warp per row (lane j: the row's j-th key): the weights
    // quantise(exp((z_j - z_top) / T)), their exact integer sum W, the top-p cut (key j is kept
    // while the weight ahead of it, a warp prefix sum, is below top_p * W; the prefix only
    // grows, so the kept keys are the leading ones), the kept mass Wk, and the draft's place in
    // the kept set. Integer sums are exact in any order: the same values the row-by-row loop
    // below once computed itself.
    __shared__ unsigned long long f_w[kMaxRows][kMaxTopK], f_Wk[kMaxRows], f_wx[kMaxRows];
    __shared__ int f_id[kMaxRows][kMaxTopK], f_n[kMaxRows], f_jx[kMaxRows];
    if (warp <= k) {
      const int r = warp;
      const unsigned long long key = lane < K ? s_topr[r][lane] : 0ull;
      const unsigned zero = __ballot_sync(0xffffffffu, key == 0ull);
      const int nk = zero ? __ffs(zero) - 1 : 32;  // the leading non-empty keys
      const float ztop = key_logit(s_topr[r][0]);
      const int id = key_id(key);
      const unsigned long long w =
          lane < nk ? quantise(expf(__fmul_rn(__fsub_rn(key_logit(key), ztop), invT))) : 0ull;
      unsigned long long incl = w;  // inclusive prefix sum over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned long long W = __shfl_sync(0xffffffffu, incl, 31);
      const double cut = tp * static_cast<double>(W);
      const bool kept = lane < nk && static_cast<double>(incl - w) < cut;
      const unsigned keptm = __ballot_sync(0xffffffffu, kept);
      unsigned long long wk = kept ? w : 0ull;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) wk += __shfl_xor_sync(0xffffffffu, wk, o);
      const int x = r < k ? sx[r] : -1;
      const unsigned hit = __ballot_sync(0xffffffffu, kept && id == x);
      const int jx = hit ? 31 - __clz(hit) : -1;  // ids are distinct: at most one hit
      f_w[r][lane] = w;
      f_id[r][lane] = id;
      if (lane == 0) {
        f_n[r] = __popc(keptm);
        f_Wk[r] = wk;
        f_jx[r] = jx;
      }
      const unsigned long long wx = __shfl_sync(0xffffffffu, w, jx >= 0 ? jx : 0);
      if (lane == 0) f_wx[r] = jx >= 0 ? wx : 0ull;
    }
    __syncthreads();
    // the decisions, row after row: the ratio test of the draft against p' (q one-hot), a
    // residual draw at the first rejection, or the bonus draw after row k
    if (tid == 0) {
      for (int r = 0; r <= k; ++r) {
        const int n = f_n[r];
        int id[kMaxTopK];
        unsigned long long w[kMaxTopK];
        bool emitted_draw = false;
        int tok = -1;
        if (r < k) {
          const int x = sx[r];
          const int jx = f_jx[r];
          const uint32_t ua = uniform_u24(p.seed[b], p.pos_base[b] + r, PURPOSE_ACCEPT);
          if (f_wx[r] > 0ull && u_le_ratio(ua, f_Wk[r], f_wx[r])) {
            F.tokens[F.ntok++] = x;
            F.n_accept++;
            if (p.eos >= 0 && x == p.eos) {
              F.eos_hit = 1;
              break;
            }
            continue;
          }
          // residual: p' without the draft (p' itself if nothing else is left)
          int m = 0;
          unsigned long long rest = 0ull;
          for (int j = 0; j < n; ++j) {
            if (j == jx) continue;
            id[m] = f_id[r][j];
            w[m] = f_w[r][j];
            rest += w[m];
            ++m;
          }
          if (rest == 0ull) {
            for (int j = 0; j < n; ++j) {
              id[j] = f_id[r][j];
              w[j] = f_w[r][j];
            }
            m = n;
          }
          tok = small_draw(id, w, m,
                           uniform_u24(p.seed[b], p.pos_base[b] + r, PURPOSE_RESIDUAL));
          F.need = 1;
          emitted_draw = true;
        } else {
          for (int j = 0; j < n; ++j) {
            id[j] = f_id[r][j];
            w[j] = f_w[r][j];
          }
          tok = small_draw(id, w, n, uniform_u24(p.seed[b], p.pos_base[b] + k, PURPOSE_BONUS));
          F.need = 2;
          emitted_draw = true;
        }
        if (emitted_draw) {
          if (tok < 0) tok = f_id[r][0];  // unreachable: the cut set always has weight
          F.srow = r;
          F.tokens[F.ntok++] = tok;
          if (p.eos >= 0 && tok == p.eos) F.eos_hit = 1;
          break;
        }
      }
    }
    if (tid == 0) {
      finalize(p, b, F, k);
      p.tickets[b] = 0u;
    }
    return;
  }

  // ratio rule: one draw, from the residual (p if the residual is empty) or the bonus row
  const DrawCtx c = draw_ctx(p, b, D.srow, D.need == 1, D.xrej, T, s_pst, s_qst);
  const unsigned long long* rs = p.sums + static_cast<size_t>(b) * p.NS * kAcceptSumSlots;
  const uint32_t purpose = (D.need == 1) ? PURPOSE_RESIDUAL : PURPOSE_BONUS;
  const uint32_t u24 = uniform_u24(p.seed[b], p.pos_base[b] + D.srow, purpose);
  int tok;
  if (p.NS <= kAcceptThreads) {
    // slot 0 holds the residual's slice sums, slot 1 p's: both in one round of loads
    const unsigned long long w_r = (tid < p.NS) ? __ldcg(rs + kAcceptSumSlots * tid) : 0ull;
    const unsigned long long w_p = (tid < p.NS) ? __ldcg(rs + kAcceptSumSlots * tid + 1) : 0ull;
    tok = draw_in_slices(p, c, D.need == 2, D.need == 2 ? w_p : w_r, u24, sh, &s_slice,
                         &s_before, &s_tok);
    if (tok < 0 && D.need == 1)  // the residual sums to zero: draw from p
      tok = draw_in_slices(p, c, true, w_p, u24, sh, &s_slice, &s_before, &s_tok);
  } else {
    unsigned long long tr = 0ull;
    for (int i = tid; i < p.NS; i += kAcceptThreads) tr += __ldcg(rs + kAcceptSumSlots * i);
    tr = block_sum_u64(tr, sh);
    const bool use_p = (D.need == 2) || (tr == 0ull);
    tok = draw_token(p, b, c, use_p, use_p ? 1 : 0, u24, sh, &s_slice, &s_before, &s_tok);
  }
  if (tid == 0) {
    Decision d = D;
    if (tok < 0) tok = s_pst[D.srow].argmax;  // unreachable
    d.tokens[d.ntok++] = tok;
    if (p.eos >= 0 && tok == p.eos) d.eos_hit = 1;
    write_result(p, b, d);
    if (p.counters && d.eos_hit) p.counters[b].eos += 1ull;
    p.tickets[b] = 0u;
  }
}

// ------------------------------------------------------------------------------------------
// Adaptive width: one thread per request updates the per-depth acceptance rates and the cycle-
// cost fit from the cycle's result and picks the next width (see spec_adapt_width in spec.h).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) adapt_width_kernel(const AdaptParams p) {
  pdl_trigger();
  pdl_wait();  // reads the acceptance results of the previous kernel
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  adapt_request(p, b, p.out[b]);
}

// The select node of a width graph: the switch's value for this launch is the largest width
// any request chose (clamped to the bodies there are).
__global__ void width_select_kernel(cudaGraphConditionalHandle h, const int32_t* k_next, int B,
                                    int n_bodies) {
  if (threadIdx.x != 0) return;
  int w = 0;
  for (int b = 0; b < B; ++b) w = max(w, k_next[b]);
  w = min(max(w, 0), n_bodies - 1);
  cudaGraphSetConditional(h, static_cast<unsigned>(w));
}

const void* width_select_function() { return reinterpret_cast<const void*>(width_select_kernel); }

cudaError_t adapt_launch(const AdaptParams& prm, cudaStream_t stream) {
  return launch_pdl(adapt_width_kernel, dim3((prm.B + 127) / 128), dim3(128), 0, stream, prm);
}

cudaError_t accept_launch(const AcceptParams& prm, cudaStream_t stream) {
  dim3 grid(prm.NS, prm.B);
  if (prm.filtered) {
    // the stage of candidate keys, dynamic, on top of the static arrays: past 48 KB together
    constexpr int kStage = kFilterStageKeys * static_cast<int>(sizeof(unsigned long long));
    static SmemAllowance allowed;
    const cudaError_t e = allow_dynamic_smem(accept_kernel<true>, kStage, allowed);
    if (e != cudaSuccess) return e;
    return launch_pdl(accept_kernel<true>, grid, dim3(kAcceptThreads), kStage, stream, prm);
  }
  return launch_pdl(accept_kernel<false>, grid, dim3(kAcceptThreads), 0, stream, prm);
}

}  // namespace spec
