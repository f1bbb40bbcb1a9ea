// Batched LM-head projection on the tcgen05 tensor cores: z = H W^T for 9..256 verify rows
// (e.g. 32 requests x 8 rows) with the per-row statistics fused into the epilogue.
//
// At 256 rows the LM head is a dense contraction (2 * 256 * 2560 * 151,936 = 199 GFLOP over
// 778 MB of weights, ~256 flop per weight byte), so it runs on the 5th-generation tensor cores
// (lucebox-hub PR #15 "MTP speculative decoding", section "What": one batched verify through
// the shared LM head; here batched over requests as well as rows):
//   * one persistent CTA per SM walks vocabulary tiles of 128 rows;
//   * a producer warp loads, per 64-wide k-block, the two 128-row halves of H and the 128-row
//     weight tile with 2-D TMA (128-byte swizzle) into a 4-stage ring;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128 token rows,
//     N = 128 vocabulary rows, K = 16) into two TMEM accumulators, one per half of H, and
//     commits each stage back to the producer and each finished tile to the epilogue; the
//     accumulators are double-buffered (2 x 2 x 128 of the 512 TMEM columns), so the epilogue
//     of one tile overlaps the MMAs of the next;
//   * eight epilogue warps (two per TMEM lane quadrant, one per 64-column half of the tile)
//     read the accumulators with tcgen05.ld: TMEM lane = token row, so each thread owns one
//     token row; it writes the row's logits when its temperature is > 0 and folds the tile's
//     max / argmax / runner-up (a register tree) and sum of exp((z - m)/T) into running
//     statistics over the CTA's tiles, stored once as a per-(row, CTA, column half) partial;
//   * a second small kernel combines the partials of each row (one block per row).
#include <math.h>

#include "params.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kTcTileN = 128;       // vocabulary rows per tile (MMA N)
constexpr int kTcHalfM = 128;       // token rows per accumulator (MMA M)
constexpr int kTcKBlock = 64;       // bf16 elements per k-block (one 128-byte swizzle row)
constexpr int kTcStages = 4;
constexpr int kTcABytes = kTcHalfM * kTcKBlock * 2;   // 16 KB per half of H
constexpr int kTcBBytes = kTcTileN * kTcKBlock * 2;   // 16 KB per weight tile
constexpr int kTcStageBytes = 2 * kTcABytes + kTcBBytes;
constexpr int kTcThreads = 10 * 32;  // producer, MMA, 8 epilogue warps
constexpr int kTcEpiWarps = 8;      // two per TMEM lane quadrant, 64 columns each
constexpr int kTcSubTiles = 2;      // per-row partials per tile (one per column half)
constexpr int kTcMaxParts = 1024;   // partials per row the combine kernel holds (<= 512 CTAs)
constexpr uint32_t kTmemCols = 512;

// Top-2 of two candidates where every index of `a` is below every index of `b`, so ties go to
// `a` (the lower vocabulary index) without comparing indices.
__device__ __forceinline__ Top2 top2_merge_lr(const Top2& a, const Top2& b) {
  const bool bw = b.best > a.best;
  return Top2{bw ? b.best : a.best, bw ? fmaxf(b.second, a.best) : fmaxf(a.second, b.best),
              bw ? b.idx : a.idx};
}

// Top-2 (value, lowest index of the maximum, runner-up value) of 64 register values by a balanced
// tree: six levels of independent merges instead of a 64-long dependent chain.
__device__ __forceinline__ Top2 top2_of_64(const float* v) {
  Top2 t[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = v[2 * i], b = v[2 * i + 1];
    const bool bw = b > a;
    t[i] = Top2{bw ? b : a, bw ? a : b, bw ? 2 * i + 1 : 2 * i};
  }
#pragma unroll
  for (int n = 16; n >= 1; n >>= 1) {
#pragma unroll
    for (int i = 0; i < n; ++i) t[i] = top2_merge_lr(t[2 * i], t[2 * i + 1]);
  }
  return t[0];
}

// --------------------------------------------------------------------------- main kernel
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_rows_tc_kernel(const __grid_constant__ CUtensorMap hmap,
                        const __grid_constant__ CUtensorMap wmap, const GemmParams p) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzle tiles, whatever the base alignment
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStageBytes);
  uint64_t* empty = full + kTcStages;
  uint64_t* tmem_full = empty + kTcStages;  // [2]: one per accumulator buffer
  uint64_t* tmem_empty = tmem_full + 2;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = p.d / kTcKBlock;
  const int nhalf = (p.nrows > kTcHalfM) ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kTcEpiWarps);  // one arrive per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // allocate the accumulators (all 512 columns; one CTA per SM)
    tmem_alloc(tmem_slot, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t bytes = static_cast<uint32_t>((nhalf == 2 ? 2 : 1) * kTcABytes + kTcBBytes);
      int s = 0;
      uint32_t eph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < p.ntiles && !*reinterpret_cast<volatile int*>(abort_flag);
           tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          if (it >= kTcStages && !mbar_wait_bounded(&empty[s], eph)) {
            atomicOr(&p.hdr->error, ERR_TC_WAIT);
            atomicExch(abort_flag, 1);
            break;
          }
          uint8_t* st = stages + s * kTcStageBytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          tc_tma_load_2d(st, &hmap, kb * kTcKBlock, 0, &full[s]);
          if (nhalf == 2) tc_tma_load_2d(st + kTcABytes, &hmap, kb * kTcKBlock, kTcHalfM, &full[s]);
          tc_tma_load_2d(st + 2 * kTcABytes, &wmap, kb * kTcKBlock, tile * kTcTileN, &full[s]);
          if (++s == kTcStages) {
            s = 0;
            if (it + 1 > kTcStages) eph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(kTcHalfM, kTcTileN);
      int s = 0;
      uint32_t fph = 0;
      int tcount = 0;
      const uint64_t stages_desc = smem_desc_sw128(smem_u32(stages));
      for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tcount) {
        // accumulator buffer of this tile: the epilogue of the previous tile drains the other
        const int buf = tcount & 1, use = tcount >> 1;
        if (use > 0 && !mbar_wait_bounded(&tmem_empty[buf], (use - 1) & 1)) {
          atomicOr(&p.hdr->error, ERR_TC_WAIT);
          atomicExch(abort_flag, 1);
          break;
        }
        tc_fence_after();
        const uint32_t dacc = tmem_base + static_cast<uint32_t>(buf * 2 * kTcTileN);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&full[s], fph)) {
            atomicOr(&p.hdr->error, ERR_TC_WAIT);
            atomicExch(abort_flag, 1);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t st = desc_advance(stages_desc, static_cast<uint32_t>(s * kTcStageBytes));
#pragma unroll
          for (int ks = 0; ks < kTcKBlock / 16; ++ks) {
            const uint64_t bdesc = desc_advance(st, 2 * kTcABytes + ks * 32);
            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
            tc_mma(dacc, desc_advance(st, ks * 32), bdesc, idesc, acc);
            if (nhalf == 2)
              tc_mma(dacc + kTcTileN, desc_advance(st, kTcABytes + ks * 32), bdesc, idesc, acc);
          }
          tc_commit(&empty[s]);  // frees the stage when these MMAs have read it
          if (++s == kTcStages) {
            s = 0;
            fph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tmem_full[tcount & 1]);  // the tile's accumulators are complete
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp & 3;                // TMEM lane quadrant this warp may access
    const int ch = (warp - 2) / 4;          // column half of every tile: [64*ch, 64*ch + 64)
    const int row_in_half = ew * 32 + lane;
    // running statistics of this thread's rows over the CTA's tiles, in tile order: exact
    // top-2; the normaliser S = sum exp((z - M)/T) relative to the running max M, rescaled
    // when M grows (a fixed order, so the result is deterministic)
    Top2 run[2] = {top2_empty(), top2_empty()};
    int run_bad[2] = {0, 0};
    double run_s[2] = {0.0, 0.0};
    float run_T[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = h * kTcHalfM + row_in_half;
      run_T[h] = (q < p.nrows) ? p.temperature[q / p.rows_per_req] : 0.f;
    }
    int tcount = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tcount) {
      const int buf = tcount & 1;
      if (!mbar_wait_bounded(&tmem_full[buf], (tcount >> 1) & 1)) {
        atomicOr(&p.hdr->error, ERR_TC_WAIT);
        atomicExch(abort_flag, 1);
        break;
      }
      tc_fence_after();
      const int64_t v0 = static_cast<int64_t>(tile) * kTcTileN + ch * (kTcTileN / 2);
      const int nv = static_cast<int>(
          max(static_cast<int64_t>(0), min(static_cast<int64_t>(kTcTileN / 2), p.V - v0)));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h >= nhalf) break;
        const int q = h * kTcHalfM + row_in_half;  // token row of this thread
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                               static_cast<uint32_t>((buf * 2 + h) * kTcTileN + ch * (kTcTileN / 2));
        const bool live = q < p.nrows;
        const float T = run_T[h];
        float* lrow = (live && T > 0.f && p.logits)
                          ? p.logits + static_cast<size_t>(q) * p.logits_stride + v0
                          : nullptr;
        float v[kTcTileN / 2];
        tmem_ld64(taddr, v);  // every lane takes part (the load is warp-collective)
        if (nv <= 0) continue;  // column half past the vocabulary (uniform across the warp)
        if (lrow) {
          if (p.vec_store && nv == kTcTileN / 2) {
            float4* dst = reinterpret_cast<float4*>(lrow);
#pragma unroll
            for (int j = 0; j < kTcTileN / 8; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < kTcTileN / 2; ++j)
              if (j < nv) lrow[j] = v[j];
          }
        }
        if (nv < kTcTileN / 2) {  // ragged last tile: columns past V take no part
#pragma unroll
          for (int j = 0; j < kTcTileN / 2; ++j)
            if (j >= nv) v[j] = -INFINITY;
        }
        bool bad = false;
#pragma unroll
        for (int j = 0; j < kTcTileN / 2; ++j) bad |= !(v[j] < INFINITY);  // NaN or +inf
        Top2 t = top2_of_64(v);
        t.idx += static_cast<int32_t>(v0);
        run_bad[h] |= bad ? 1 : 0;
        if (t.best != -INFINITY && !bad) {
          // the tile's sum of exp((z - m_tile)/T) in fp32 (64 terms in eight chains), folded
          // into the running fp64 sum with an fp32 rescale factor when the running max moves
          const float k2 = __fmul_rn(__fdiv_rn(1.f, T > 0.f ? T : 1.f), 1.4426950408889634f);
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < kTcTileN / 2; ++j)
            acc[j & 7] += exp2f(__fmul_rn(__fsub_rn(v[j], t.best), k2));
          const double st = static_cast<double>(((acc[0] + acc[1]) + (acc[2] + acc[3])) +
                                                ((acc[4] + acc[5]) + (acc[6] + acc[7])));
          if (run[h].idx == kNoIndex || run[h].best == -INFINITY) {
            run_s[h] = st;
          } else if (t.best > run[h].best) {
            run_s[h] = run_s[h] * static_cast<double>(exp2f(__fmul_rn(__fsub_rn(run[h].best, t.best), k2))) + st;
          } else {
            run_s[h] += st * static_cast<double>(exp2f(__fmul_rn(__fsub_rn(t.best, run[h].best), k2)));
          }
        }
        run[h] = top2_merge(run[h], t);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[buf]);
    }
    // one partial per (row, CTA, column half)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = h * kTcHalfM + row_in_half;
      if (h < nhalf && q < p.nrows) {
        GemmPartial pp;
        pp.m = run[h].best;
        pp.second = run[h].second;
        pp.idx = (run[h].idx == kNoIndex) ? -1 : run[h].idx;
        pp.flags = run_bad[h];
        pp.s = run_s[h];
        pp.pad = 0.0;
        p.part[(static_cast<size_t>(q) * gridDim.x + blockIdx.x) * kTcSubTiles + ch] = pp;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  pdl_trigger();  // the combine may be scheduled now
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// --------------------------------------------------------------------------- row combine
// One block per row: combine the row's per-tile partials in a fixed order (thread-strided,
// then a fixed tree), exactly like the last block of the GEMV.
__global__ void __launch_bounds__(256) gemm_rows_combine_kernel(const GemmParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm_best[8], sm_second[8], sm_sum[8];
  __shared__ int sm_idx[8], sm_bad[8];
  __shared__ float sm_m[kTcMaxParts], sm_s[kTcMaxParts];  // each partial's max and sum, loaded once
  const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nparts = p.nblocks * kTcSubTiles;  // <= kTcMaxParts (checked on the host)
  const GemmPartial* row = p.part + static_cast<size_t>(q) * nparts;
  const float T = p.temperature[q / p.rows_per_req];
  const float k2 = __fmul_rn(__fdiv_rn(1.f, T > 0.f ? T : 1.f), 1.4426950408889634f);
  Top2 t = top2_empty();
  int bad = 0;
  for (int i = tid; i < nparts; i += blockDim.x) {
    const uint4* pp = reinterpret_cast<const uint4*>(row + i);
    const uint4 a = __ldcg(pp), b = __ldcg(pp + 1);  // {m, second, idx, flags}, {s (double), pad}
    const int32_t idx = static_cast<int32_t>(a.z);
    bad |= static_cast<int>(a.w);
    if (idx >= 0) t = top2_merge(t, Top2{__uint_as_float(a.x), __uint_as_float(a.y), idx});
    sm_m[i] = (idx >= 0) ? __uint_as_float(a.x) : -INFINITY;
    sm_s[i] = static_cast<float>(__hiloint2double(static_cast<int>(b.y), static_cast<int>(b.x)));
  }
  t = warp_top2(t);
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sm_best[warp] = t.best;
    sm_second[warp] = t.second;
    sm_idx[warp] = t.idx;
    sm_bad[warp] = bad;
  }
  __syncthreads();
  Top2 all = top2_empty();
  int anybad = 0;
  for (int w = 0; w < 8; ++w) {
    all = top2_merge(all, Top2{sm_best[w], sm_second[w], sm_idx[w]});
    anybad |= sm_bad[w];
  }
  const bool nonfinite = anybad || all.idx == kNoIndex || all.best == -INFINITY;
  const float M = all.best;
  // the normaliser in fp32: thread sums in index order, then fixed trees (deterministic)
  float S = 0.f;
  if (!nonfinite) {
    for (int i = tid; i < nparts; i += blockDim.x) {  // entries this thread wrote above
      const float mc = sm_m[i], sc = sm_s[i];
      if (mc != -INFINITY && sc > 0.f)
        S = __fadd_rn(S, __fmul_rn(sc, exp2f(__fmul_rn(__fsub_rn(mc, M), k2))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, o));
  if (lane == 0) sm_sum[warp] = S;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot = __fadd_rn(tot, sm_sum[w]);
    spec_rowstats st;
    if (nonfinite) {
      st.max = __int_as_float(0x7fc00000);
      st.log_norm = st.max;
      st.gap = st.max;
      st.argmax = -1;
    } else {
      st.max = M;
      st.log_norm = logf(tot);
      st.gap = __fsub_rn(M, all.second);
      st.argmax = all.idx;
    }
    p.stats[q] = st;
  }
}

// --------------------------------------------------------------------------- host side
cudaError_t gemm_tc_launch(const GemmLaunch& L, cudaStream_t stream) {
  static SmemAllowance allowed;
  cudaError_t e = allow_dynamic_smem(gemm_rows_tc_kernel, L.smem, allowed);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, gemm_rows_tc_kernel, kTcThreads,
                                                    L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorLaunchOutOfResources;
  e = launch_pdl(gemm_rows_tc_kernel, dim3(L.grid), dim3(kTcThreads), L.smem, stream, L.hmap, L.wmap,
                 L.p);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_rows_combine_kernel, dim3(L.p.nrows), dim3(256), 0, stream, L.p);
}

int gemm_tc_smem_bytes() { return kTcStages * kTcStageBytes + 1024 + 128; }
int gemm_tc_tile_rows() { return kTcTileN; }
int gemm_tc_max_ctas() { return kTcMaxParts / kTcSubTiles; }
int gemm_tc_subtiles() { return kTcSubTiles; }
int gemm_tc_kblock() { return kTcKBlock; }

}  // namespace spec
