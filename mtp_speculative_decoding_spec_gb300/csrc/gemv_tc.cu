// LM-head projection of 1..8 rows (verify rows, or one draft row per request) on the tcgen05
// tensor cores, for bf16 weights, with the same fused row statistics and draft draw as the
// CUDA-core kernel in gemv.cu.
//
// The projection z = H W^T streams W [V, d] once from HBM (lucebox-hub PR #15 "MTP speculative
// decoding", section "What": the trunk verifies k drafts in one batched forward of k+1 rows
// through the shared LM head). On the CUDA cores every weight costs one fp32 FMA per row, so at
// 5..8 rows the FMA pipe, not HBM, sets the pace; here the multiply-adds go to the tensor cores
// and the kernel is left with streaming alone:
//   * one persistent CTA per SM owns a contiguous run of 32-row bands of the vocabulary and
//     walks it in tiles of 128 rows (the last one partial: its stages carry more k-blocks, so
//     that it takes fewer of them);
//   * a producer warp loads, per stage, 512 contiguous bytes of each of the tile's weight rows
//     (four 64-wide k-blocks as 2-D TMA boxes of 32 rows, 128-byte swizzle; only the boxes the
//     tile needs) and the matching 16-row H blocks (rows past the live ones read as zero) into
//     a ring of shared-memory stages. Requests of 512 contiguous bytes per row keep HBM far
//     busier than 128-byte ones. The weight lines carry an evict-first L2 policy: the matrix
//     is far larger than L2 and read once, and without the hint it pushes the logits written
//     during the stream out to HBM just before the acceptance reads them back;
//   * one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32, M = 128 weight rows,
//     N = 16 H rows, K = 16); every tile of the block has its own 16-column TMEM accumulator,
//     so the shared memory goes to the stages alone (three of 72 KB at any row count);
//   * four warps (one per TMEM lane quadrant) read each finished accumulator with tcgen05.ld
//     (lane = vocabulary row, column = H row), write the logits of rows at T > 0 (coalesced)
//     and fold the tile into each row's running statistics while the next tiles stream in: the
//     top-2, and the sum of exp((z - m)/T) kept as (M, S) -- the exact integer sum of
//     rint(exp((z - m_q)/T) 2^40) over the tile's 32 rows of the warp, against their own max
//     m_q, scaled onto the running max M in fp32 (a fixed order of separately rounded
//     operations). A tile takes ~14 us to stream and its statistics well under one, so when
//     streaming is over only the four quadrants remain to be merged;
//   * then the same finish as the CUDA-core kernel: the last block's combine and the draft
//     draw.
// Batch invariance (section "Exactness": up to eight rows, a row's verify logits may not depend
// on how many rows are verified together): every
// call with bf16 weights runs this kernel whatever the number of rows, H row r always sits in
// MMA column r, and a column's result depends only on that column's operands.
#include "gemv_epilogue.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kSkTileRows = 128;  // weight rows per tile (MMA M)
constexpr int kSkBoxRows = 32;    // rows per TMA box (and the band of the block partition)
constexpr int kSkN = 16;          // H rows per MMA (N); rows past the live ones are zero
constexpr int kSkKBlock = 64;     // bf16 elements per k-block (one 128-byte swizzle row)
constexpr int kSkKB = 4;          // k-blocks per stage: 512 contiguous bytes of each weight row
constexpr int kSkBoxBytes = kSkBoxRows * kSkKBlock * 2;  // 4 KB
constexpr int kSkWBytes = kSkTileRows * kSkKBlock * 2;   // 16 KB per k-block
constexpr int kSkHBytes = kSkN * kSkKBlock * 2;          // 2 KB per k-block
constexpr int kSkStageBytes = kSkKB * (kSkWBytes + kSkHBytes);  // 72 KB, a multiple of 1024

// k-blocks per stage of a tile that holds nbox of the four boxes. A stage's round trip costs
// about the same whatever it carries (a block's last tile of one box took ~10 us over its ten
// stages, against ~12-14 us for a full tile), so a partial tile packs more k-blocks into each
// stage: 12, 7 and 5 for one, two and three boxes, and runs in 4, 6 or 8 stages instead of 10.
// In a stage the k-blocks' weight boxes sit back to back (nbox * 4 KB each), then their H
// blocks; the MMA still reads a 128-row operand at each k-block's start, so the largest start
// plus 16 KB must stay inside the stage (the rows past the tile's boxes are other k-blocks'
// bytes, in lanes nobody reads). The MMAs keep their k order, so the results do not change.
__host__ __device__ constexpr int tile_kblocks(int nbox) {
  return (kSkStageBytes / (nbox * kSkBoxBytes + kSkHBytes)) <
                 ((kSkStageBytes - kSkWBytes) / (nbox * kSkBoxBytes) + 1)
             ? kSkStageBytes / (nbox * kSkBoxBytes + kSkHBytes)
             : (kSkStageBytes - kSkWBytes) / (nbox * kSkBoxBytes) + 1;
}
static_assert(tile_kblocks(4) == kSkKB, "a full tile keeps the 4-k-block stage");
static_assert(tile_kblocks(1) == 12 && tile_kblocks(2) == 7 && tile_kblocks(3) == 5,
              "the packed stages of a partial tile");
constexpr int kSkThreads = 8 * 32;  // producer, MMA issuer, two idle warps, four drain warps
constexpr int kSkDrainWarp0 = 4;    // warps 4..7: TMEM lane quadrants 0..3
constexpr int kSkMaxTiles = 16;     // tiles per block: 16 x 16 = 256 TMEM columns at most
constexpr int kSkStatBytes = 1024;  // start of the idle ring: per-quadrant top-2, row sums

__global__ void __launch_bounds__(kSkThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                   const __grid_constant__ CUtensorMap hmap, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (draft_step_idle(p)) return;  // before any setup: nothing allocated, nothing in flight
  if (threadIdx.x == 0) {  // the tensor maps' descriptors, ahead of the first copies
    asm volatile("prefetch.tensormap [%0];" ::"l"(&wmap) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&hmap) : "memory");
  }
  const int S = p.stages;
  // the ring of stages; once streaming is over it holds the block's statistics and then the
  // combine's scratch
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.ring_bytes);
  uint64_t* empty = full + S;
  uint64_t* tile_done = empty + S;  // [kSkMaxTiles]: one phase each
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_done + kSkMaxTiles);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] last block
  float* s_temp = reinterpret_cast<float*>(flags + 4);  // [8] T of rows whose logits are written
  RowInputs* ri = reinterpret_cast<RowInputs*>(
      (reinterpret_cast<uintptr_t>(s_temp + kMaxRows) + 7) & ~static_cast<uintptr_t>(7));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t v0, v1;
  block_rows(blockIdx.x, gridDim.x, p.nbands, kSkBoxRows, p.V, v0, v1);
  const int nt = static_cast<int>(v1 - v0);
  const int ntile = (nt + kSkTileRows - 1) / kSkTileRows;
  const int nkb = (p.d + kSkKBlock - 1) / kSkKBlock;  // k-blocks per row
  const int nks = (nkb + kSkKB - 1) / kSkKB;           // stages per full tile
  const int nr = min(p.nrows, kMaxRows);
  // one 16-column accumulator per tile of the block, all resident until the end
  const int ntile_cap = (p.tile_cap + kSkTileRows - 1) / kSkTileRows;
  uint32_t tcols = 32;
  while (tcols < static_cast<uint32_t>(ntile_cap * kSkN)) tcols <<= 1;

  // The stage schedule: iterations [0, full_it) cover the full tiles, tile it / nks and stage
  // it % nks; the rest cover the last tile, whose nbox_last boxes take kpb_last k-blocks a
  // stage (four boxes: the same stages as any other tile).
  const int nbox_last =
      ntile > 0 ? (nt - (ntile - 1) * kSkTileRows + kSkBoxRows - 1) / kSkBoxRows : 0;
  const int kpb_last = ntile > 0 ? tile_kblocks(nbox_last) : kSkKB;
  const int full_it = ntile > 0 ? (ntile - 1) * nks : 0;
  const int total_it = ntile > 0 ? full_it + (nkb + kpb_last - 1) / kpb_last : 0;
  struct StageMap {
    int t, ks, nbox, kpb, nk;  // tile, its stage, boxes, k-blocks a stage, k-blocks in this one
  };
  auto stage_of = [&](int it) {
    StageMap m;
    if (it < full_it) {
      m.t = it / nks;
      m.ks = it - m.t * nks;
      m.nbox = kSkTileRows / kSkBoxRows;
      m.kpb = kSkKB;
    } else {
      m.t = ntile - 1;
      m.ks = it - full_it;
      m.nbox = nbox_last;
      m.kpb = kpb_last;
    }
    m.nk = min(m.kpb, nkb - m.ks * m.kpb);
    return m;
  };
  // weight rows of a tile's four 32-row boxes, worked out once per stage in 32-bit arithmetic
  // (V < 2^24): the producer's issue loop sets this kernel's pace, and mapping every box there
  // measured ~5% slower
  const int lo_rows = static_cast<int>(p.lo_rows);
  const int hi_shift = static_cast<int>(p.hi_row0 - p.lo_rows);
  const uint64_t wpol = l2_policy_evict_first();  // the weights: read once, never kept in L2
  auto box_rows = [&](int y, int* yb) {
#pragma unroll
    for (int b = 0; b < kSkTileRows / kSkBoxRows; ++b) {
      const int r = y + b * kSkBoxRows;
      yb[b] = r < lo_rows ? r : r + hi_shift;
    }
  };
  auto issue_w = [&](int it, int s) {  // the weight boxes of iteration it into stage s
    const StageMap m = stage_of(it);
    const int y = static_cast<int>(v0) + m.t * kSkTileRows;
    uint8_t* st = ring + static_cast<size_t>(s) * kSkStageBytes;
    int yb[kSkTileRows / kSkBoxRows];
    box_rows(y, yb);
    mbar_arrive_expect_tx(&full[s],
                          static_cast<uint32_t>(m.nk * (m.nbox * kSkBoxBytes + kSkHBytes)));
    for (int kk = 0; kk < m.nk; ++kk)
#pragma unroll
      for (int b = 0; b < kSkTileRows / kSkBoxRows; ++b)
        if (b < m.nbox)
          tc_tma_load_2d_hint(st + (kk * m.nbox + b) * kSkBoxBytes, &wmap,
                              (m.ks * m.kpb + kk) * kSkKBlock, yb[b], &full[s], wpol);
  };
  auto issue_h = [&](int it, int s) {  // the H blocks of iteration it into stage s
    const StageMap m = stage_of(it);
    uint8_t* st = ring + static_cast<size_t>(s) * kSkStageBytes + m.kpb * m.nbox * kSkBoxBytes;
    for (int kk = 0; kk < m.nk; ++kk)
      tc_tma_load_2d(st + kk * kSkHBytes, &hmap, (m.ks * m.kpb + kk) * kSkKBlock, 0, &full[s]);
  };
  // Steady state: per k-block its weight boxes, then its H block. This order (k-block outer,
  // 32-row boxes inner, H between k-blocks) streamed measurably faster than issuing all weight
  // boxes first or walking each row band's 512 bytes first.
  auto issue_all = [&](int it, int s) {
    const StageMap m = stage_of(it);
    const int y = static_cast<int>(v0) + m.t * kSkTileRows;
    uint8_t* st = ring + static_cast<size_t>(s) * kSkStageBytes;
    uint8_t* sh = st + m.kpb * m.nbox * kSkBoxBytes;
    int yb[kSkTileRows / kSkBoxRows];
    box_rows(y, yb);
    mbar_arrive_expect_tx(&full[s],
                          static_cast<uint32_t>(m.nk * (m.nbox * kSkBoxBytes + kSkHBytes)));
    for (int kk = 0; kk < m.nk; ++kk) {
      const int x = (m.ks * m.kpb + kk) * kSkKBlock;
#pragma unroll
      for (int b = 0; b < kSkTileRows / kSkBoxRows; ++b)
        if (b < m.nbox)
          tc_tma_load_2d_hint(st + (kk * m.nbox + b) * kSkBoxBytes, &wmap, x, yb[b], &full[s],
                              wpol);
      tc_tma_load_2d(sh + kk * kSkHBytes, &hmap, x, 0, &full[s]);
    }
  };
  // The weights are never written by the path: the first stages stream in before the wait for
  // the previous kernel, whose tail they overlap, and before the tensor memory is allocated.
  // H, the temperatures, the outputs and the workspace are only touched after the wait.
  const int pre = min(S, total_it);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < kSkMaxTiles; ++t) mbar_init(&tile_done[t], 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();  // the barriers' initialisation before the copies that complete on them
    for (int it = 0; it < pre; ++it) issue_w(it, it);
  }
  if (warp == 1) tmem_alloc(tmem_slot, tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  if (tid == 0)
    for (int it = 0; it < pre; ++it) issue_h(it, it);  // the first MMAs wait on nothing else
  if (tid >= 32 && tid < 32 + kMaxRows) {  // lanes of the MMA warp, idle until the barrier
    const int r = tid - 32;
    load_row_inputs(p, ri, r);
    s_temp[r] = (r < p.nrows && p.logits) ? ri->T[r] : 0.f;
  }
  __syncthreads();
  // running top-2 and NaN / +Inf flag of each row over this warp's TMEM lane quadrant (drain
  // warps only)
  Top2 run[kMaxRows];
  int rbad[kMaxRows];
  float rM[kMaxRows], rS[kMaxRows];  // running max and exp-sum (2^-40 units) against it
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    run[r] = top2_empty();
    rbad[r] = 0;
    rM[r] = -INFINITY;
    rS[r] = 0.f;
  }

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int it = pre, s = pre % S;
      for (; it < total_it && !*reinterpret_cast<volatile int*>(&flags[0]); ++it) {
        // stage s is reused every S iterations: wait until the MMAs of its last use are done
        if (!mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((it / S) & 1) ^ 1))) {
          atomicOr(&p.hdr->error, ERR_TC_WAIT);
          atomicExch(&flags[0], 1);
          break;
        }
        issue_all(it, s);
        if (++s == S) s = 0;
      }
      // every issued copy must have landed before the ring is reused or the block exits
      for (int j = max(0, it - S); j < it; ++j) {
        if (!mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1))) {
          atomicOr(&p.hdr->error, ERR_GEMV_DRAIN);
          break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(kSkTileRows, kSkN);
      const uint64_t ring_desc = smem_desc_sw128(smem_u32(ring));
      int it = 0, s = 0;
      for (int t = 0; t < ntile; ++t) {
        const uint32_t dacc = tmem_base + static_cast<uint32_t>(t * kSkN);
        bool ok = true;
        const int it_end = (t + 1 < ntile) ? it + nks : total_it;  // this tile's stages
        for (; it < it_end; ++it) {
          if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((it / S) & 1))) {
            atomicOr(&p.hdr->error, ERR_TC_WAIT);
            atomicExch(&flags[0], 1);
            ok = false;
            break;
          }
          tc_fence_after();
          const StageMap m = stage_of(it);
          const uint64_t st = desc_advance(ring_desc, static_cast<uint32_t>(s * kSkStageBytes));
          const uint32_t wstep = static_cast<uint32_t>(m.nbox * kSkBoxBytes);  // per k-block
          const uint32_t hbase = static_cast<uint32_t>(m.kpb) * wstep;
          for (int kk = 0; kk < m.nk; ++kk) {
            const uint64_t a = desc_advance(st, static_cast<uint32_t>(kk) * wstep);
            const uint64_t b = desc_advance(st, hbase + static_cast<uint32_t>(kk * kSkHBytes));
#pragma unroll
            for (int k16 = 0; k16 < kSkKBlock / 16; ++k16)
              tc_mma(dacc, desc_advance(a, k16 * 32), desc_advance(b, k16 * 32), idesc,
                     (m.ks > 0 || kk > 0 || k16 > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);  // frees the stage once these MMAs have read it
          if (++s == S) s = 0;
        }
        if (!ok) break;
        tc_commit(&tile_done[t]);  // the tile's accumulator is complete
      }
    }
  } else if (warp >= kSkDrainWarp0) {
    // -------------- per finished tile: logits of rows at T > 0, running top-2 of each row
    const int ew = warp & 3;  // TMEM lane quadrant this warp may access
    bool hot = false;
    for (int r = 0; r < nr; ++r) hot |= s_temp[r] > 0.f;
    for (int t = 0; t < ntile; ++t) {
      if (!mbar_wait_bounded(&tile_done[t], 0u)) {
        atomicOr(&p.hdr->error, ERR_TC_WAIT);
        atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      float v[8];
      tmem_ld8(tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                   static_cast<uint32_t>(t * kSkN),
               v);  // warp-collective: every lane takes part
      const int local = t * kSkTileRows + ew * 32 + lane;
      const bool valid = local < nt;
      if (hot && valid) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          if (r < nr && s_temp[r] > 0.f)
            p.logits[static_cast<size_t>(r) * p.logits_stride + v0 + local] = v[r];
      }
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < nr) {
          const float z = v[r];
          const bool nf = isnan(z) || z == INFINITY;
          Top2 c = (valid && !nf) ? Top2{z, -INFINITY, static_cast<int32_t>(v0 + local)}
                                  : top2_empty();
          c = warp_top2(c);
          rbad[r] |= __any_sync(0xffffffffu, valid && nf) ? 1 : 0;
          run[r] = top2_merge(run[r], c);
          const float mq = c.best;  // warp-uniform: the max of this warp's rows of the tile
          if (mq != -INFINITY) {
            const float invT = ri->invT[r];
            const unsigned long long w = (valid && !nf) ? tile_weight(z, mq, invT) : 0ull;
            const float sq = u64_to_f32(warp_sum_u64(w));
            if (mq > rM[r]) {
              rS[r] = __fadd_rn(__fmul_rn(rS[r], expf(__fmul_rn(__fsub_rn(rM[r], mq), invT))), sq);
              rM[r] = mq;
            } else {
              rS[r] = __fadd_rn(rS[r], __fmul_rn(sq, expf(__fmul_rn(__fsub_rn(mq, rM[r]), invT))));
            }
          }
        }
      }
    }
  }

  // every tile's MMAs have completed (the drain warps waited for each) and every copy has
  // landed (the producer waited for each): the ring is free for the block's statistics and the
  // accumulators are no longer needed. The next kernel may now be scheduled into this kernel's
  // tail (not earlier: blocks parked in its wait during the stream cost bandwidth).
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
  Top2* s_top = reinterpret_cast<Top2*>(ring);                             // [4 quadrants][8]
  int* s_bad = reinterpret_cast<int*>(ring + 4 * kMaxRows * sizeof(Top2));  // [4][8]
  float2* s_ms = reinterpret_cast<float2*>(ring + 512);                     // [4][8] (M, S)
  if (warp >= kSkDrainWarp0 && lane == 0) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      s_top[(warp & 3) * kMaxRows + r] = run[r];
      s_bad[(warp & 3) * kMaxRows + r] = rbad[r];
      s_ms[(warp & 3) * kMaxRows + r] = make_float2(rM[r], rS[r]);
    }
  }
  __syncthreads();
  if (tid < nr) {
    // the quadrants merged in a fixed order: top-2, NaN / +Inf flag, and the exp-sum against
    // the block max M (the integer weights' scale, 2^-40 units)
    Top2 m = top2_empty();
    int bad = 0;
    for (int w = 0; w < 4; ++w) {
      m = top2_merge(m, s_top[w * kMaxRows + tid]);
      bad |= s_bad[w * kMaxRows + tid];
    }
    const float invT = ri->invT[tid];
    float S = 0.f;
    if (!*reinterpret_cast<volatile int*>(&flags[0]) && m.best != -INFINITY) {
      for (int w = 0; w < 4; ++w) {
        const float2 q = s_ms[w * kMaxRows + tid];
        if (q.x != -INFINITY)
          S = __fadd_rn(S, __fmul_rn(q.y, expf(__fmul_rn(__fsub_rn(q.x, m.best), invT))));
      }
    }
    GemvPartial pp;
    pp.m = m.best;
    pp.second = m.second;
    pp.idx = (m.idx == kNoIndex) ? -1 : m.idx;
    pp.flags = bad;
    pp.s = __float2ull_rn(S);
    pp.pad = 0ull;
    p.part[static_cast<size_t>(blockIdx.x) * kMaxRows + tid] = pp;
  }
  gemv_finish(p, ring + kSkStatBytes, flags, kSkThreads / 32, ri);
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

int gemv_tc_band_rows() { return kSkBoxRows; }
int gemv_tc_box_rows() { return kSkBoxRows; }
int gemv_tc_kblock() { return kSkKBlock; }
int gemv_tc_h_rows() { return kSkN; }
int gemv_tc_stage_bytes() { return kSkStageBytes; }
int gemv_tc_threads() { return kSkThreads; }
int gemv_tc_max_block_rows() { return kSkMaxTiles * kSkTileRows; }
int gemv_tc_stat_bytes() { return kSkStatBytes; }

cudaError_t gemv_tc_launch(const GemvTcLaunch& L, cudaStream_t stream) {
  static SmemAllowance allowed;
  cudaError_t e = allow_dynamic_smem(gemv_tc_kernel, L.smem, allowed);
  if (e != cudaSuccess) return e;
  int fit = 0;  // shared memory must admit one block per SM
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, gemv_tc_kernel, kSkThreads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorLaunchOutOfResources;
  return launch_pdl(gemv_tc_kernel, dim3(L.grid), dim3(kSkThreads), L.smem, stream, L.wmap, L.hmap,
                    L.p);
}

}  // namespace spec
