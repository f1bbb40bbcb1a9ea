// LM-head projection of 1..8 rows over 4-bit affine weights in groups of 32 (DS4Server issue
// #98, closing comment: the MTP head's weights are 4-bit affine values in groups of 32), on the
// tcgen05 tensor cores, with the same fused row statistics and draft draw as the bf16 kernels.
//
// Row layout (5d/8 bytes per vocabulary row, d a multiple of 128): d/2 bytes of codes, then one
// (scale, bias) bf16 pair per 32-element group. In each little-endian 32-bit word of 8
// consecutive codes e0..e7, e_{2i} sits in bits 4i..4i+3 and e_{2i+1} in bits 16+4i..16+4i+3.
// The dequantised weight is bf16(s*q + b), rounded once, so z = H w^T is a bf16 projection.
//
// The weights are a quarter of the bf16 bytes plus the pairs (1,600 against 5,120 bytes per row
// at d = 2560), so HBM still bounds the kernel, but each weight now costs ALU work before the
// tensor core can use it, and the MMA's A operand has to be written by threads:
//   * a producer warp loads, per stage, 256 code bytes and 64 pair bytes of each of the tile's
//     rows (2-D TMA boxes of 32 rows; the codes with 128-byte swizzle, so the 16-byte reads
//     below hit distinct banks) and the matching [16 x 64] blocks of H;
//   * twelve dequantisation warps (thread = vocabulary row of a 32-row quarter of the tile)
//     turn each code word into four bf16 pairs with a mask, an exact subtraction and one
//     fma.rn.bf16x2 (s*q + b, rounded once), and write them to a ring of shared-memory A
//     buffers of 128 elements x 128 rows in the MMA's K-major 128-byte-swizzle layout (the
//     layout TMA gives the bf16 kernel's weight tiles). A task is 128 elements: each one pays
//     two barrier waits, a proxy fence and an arrival, which at 64 elements cost more than the
//     arithmetic. A from tensor memory was measured
//     first: with N = 16 each such MMA took ~120 cycles against ~8 from shared memory;
//   * three threads issue tcgen05.mma kind::f16 (M = 128 weight rows, N = 16 H rows, K = 16),
//     each taking every third K block into its own 16-column TMEM accumulator per tile, and
//     release each A buffer, and each stage's H blocks, with tcgen05.commit. One thread could
//     not keep up: at N = 16 an MMA does ~8 cycles of math, but a thread issues one every ~54
//     cycles at best and ~170 with its waits and commits beside busy warps (measured);
//   * after the stream all sixteen warps read the accumulators (the three partial sums added
//     in a fixed order): logits of rows at T > 0 and each row's top-2, then the exact integer
//     sums against the block max; then the shared finish, as in the bf16 tensor-core kernel.
// Batch invariance: one kernel for 1..8 rows with H row r in MMA column r, as for bf16.
#include "gemv_epilogue.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kQTileRows = 128;   // weight rows per tile (MMA M)
constexpr int kQBoxRows = 32;     // rows per TMA box (and the band of the block partition)
constexpr int kQN = 16;           // H rows per MMA (N); rows past the live ones are zero
constexpr int kQStageElems = 512;                  // elements of each row per stage
constexpr int kQChunkBytes = 128;                  // code bytes per box row (256 elements)
constexpr int kQChunks = kQStageElems / 256;       // code boxes per row per stage: 2
constexpr int kQCodeBox = kQBoxRows * kQChunkBytes;          // 4 KB
constexpr int kQCodeTile = kQTileRows * kQChunkBytes;        // 16 KB per chunk of a tile
constexpr int kQPairRowBytes = kQStageElems / 32 * 4;        // 64 bytes of pairs per row
constexpr int kQPairBox = kQBoxRows * kQPairRowBytes;        // 2 KB
constexpr int kQPairOff = kQChunks * kQCodeTile;             // 32 KB
constexpr int kQHBlock = kQN * 128;                          // [16 rows x 64] bf16: 2 KB
constexpr int kQHOff = kQPairOff + kQTileRows * kQPairRowBytes;  // 40 KB
constexpr int kQStageBytes = kQHOff + (kQStageElems / 64) * kQHBlock;  // 56 KB
constexpr int kQThreads = 16 * 32;
constexpr int kQDeqWarp0 = 4;     // warps 4..15: dequantisation, row quarter = warp & 3
constexpr int kQDeqSlots = 3;     // dequantisation warps per row quarter
constexpr int kQTaskElems = 128;  // one task: 128 elements (two 64-wide K blocks) of every row
constexpr int kQTasksPerStage = kQStageElems / kQTaskElems;  // 4
constexpr int kQKBlockBytes = kQTileRows * 128;              // one K block of A: 16 KB
constexpr int kQABufs = 3;
constexpr int kQABufBytes = 2 * kQKBlockBytes;               // 32 KB
constexpr int kQIssuers = 3;      // MMA-issuing threads (warps 1..3), one accumulator set each
constexpr int kQMaxTiles = 8;     // tiles per block: issuer j's accumulators in TMEM columns
constexpr int kQAccCols = kQMaxTiles * kQN;  // [128 j, 128 j + 128)
constexpr uint32_t kQTmemCols = 512;
constexpr int kQStatBytes = 4096; // per-warp top-2 and flags, row sums; then the finish scratch

static_assert(kQStageBytes % 1024 == 0 && kQABufBytes % 1024 == 0,
              "stages and A buffers keep the 1024-byte swizzle alignment");
static_assert(kQABufs >= kQDeqSlots, "a task's A-buffer wait is never two phases ahead");
static_assert(kQABufs % kQIssuers == 0, "every A buffer belongs to one issuer");

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Codes of one 32-element group (four words) and its (scale, bias) pair -> 16 bf16 pairs, in
// element order (column c of the group holds elements 2c and 2c+1).
__device__ __forceinline__ void dequant_group(const uint4 w, uint32_t sb, uint32_t* out) {
  const uint32_t s2 = __byte_perm(sb, sb, 0x1010);  // {s, s}
  const uint32_t b2 = __byte_perm(sb, sb, 0x3232);  // {b, b}
  const uint32_t one2 = 0x3F803F80u, m128 = 0xC300C300u;  // {1, 1}, {-128, -128}
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // bf16 pair (128 + e_{2j}, 128 + e_{2j+1}): the code lands in the low mantissa bits of
      // 128 = 0x4300, where one unit is 1
      const uint32_t t = ((words[i] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
      const uint32_t q = bf16x2_fma(t, one2, m128);     // exact: the codes 0..15
      out[4 * i + j] = bf16x2_fma(q, s2, b2);           // s*q + b, rounded once
    }
  }
}

__global__ void __launch_bounds__(kQThreads, 1)
    gemv_q4_kernel(const __grid_constant__ CUtensorMap cmap,
                   const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap hmap, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (draft_step_idle(p)) return;  // before any setup: nothing allocated, nothing in flight
  const int S = p.stages;
  uint8_t* ring = smem;                      // stages; afterwards statistics and scratch
  uint8_t* abufs = smem + p.ring_bytes;      // [kQABufs][128 rows][128 B], swizzled
  uint64_t* full = reinterpret_cast<uint64_t*>(abufs + p.hs_bytes);
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;              // [kQABufs]
  uint64_t* a_empty = a_full + kQABufs;      // [kQABufs]
  uint64_t* mma_done = a_empty + kQABufs;    // one phase: every MMA of the block has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] last block
  float* s_temp = reinterpret_cast<float*>(flags + 4);
  RowInputs* ri = reinterpret_cast<RowInputs*>(
      (reinterpret_cast<uintptr_t>(s_temp + kMaxRows) + 7) & ~static_cast<uintptr_t>(7));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t v0, v1;
  block_rows(blockIdx.x, gridDim.x, p.nbands, kQBoxRows, p.V, v0, v1);
  const int nt = static_cast<int>(v1 - v0);
  const int ntile = (nt + kQTileRows - 1) / kQTileRows;
  const int d = p.d;
  const int nks = (d + kQStageElems - 1) / kQStageElems;  // stages per tile
  const int last_tasks = (d - (nks - 1) * kQStageElems) / kQTaskElems;  // in a tile's last stage
  const int nr = min(p.nrows, kMaxRows);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      // every dequantisation warp once, and each issuer's MMAs on the stage's H blocks
      mbar_init(&empty[s], kQDeqSlots * 4 + kQIssuers);
    }
    for (int b = 0; b < kQABufs; ++b) {
      mbar_init(&a_full[b], 4);
      mbar_init(&a_empty[b], 1);
    }
    mbar_init(mma_done, kQIssuers);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kQTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_it = ntile * nks;
  const uint64_t wpol = l2_policy_evict_first();  // codes and pairs: read once, not kept in L2
  auto stage_tasks = [&](int ks) { return ks == nks - 1 ? last_tasks : kQTasksPerStage; };
  auto issue_w = [&](int it, int s) {  // codes, pairs (and the byte count of H) of iteration it
    const int t = it / nks, ks = it - t * nks;
    const int rows = min(kQTileRows, nt - t * kQTileRows);
    const int nbox = (rows + kQBoxRows - 1) / kQBoxRows;
    const int y = static_cast<int>(v0) + t * kQTileRows;
    const int x0 = ks * (kQStageElems / 2);              // first code byte of the stage
    const int nch = min(kQChunks, (d / 2 - x0 + kQChunkBytes - 1) / kQChunkBytes);
    uint8_t* st = ring + static_cast<size_t>(s) * kQStageBytes;
    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nbox * (nch * kQCodeBox + kQPairBox) +
                                                          stage_tasks(ks) * 2 * kQHBlock));
    for (int c = 0; c < nch; ++c)
      for (int b = 0; b < nbox; ++b)
        tc_tma_load_2d_hint(st + c * kQCodeTile + b * kQCodeBox, &cmap, x0 + c * kQChunkBytes,
                            box_row(p, y + b * kQBoxRows), &full[s], wpol);
    for (int b = 0; b < nbox; ++b)
      tc_tma_load_2d_hint(st + kQPairOff + b * kQPairBox, &smap, ks * kQPairRowBytes,
                          box_row(p, y + b * kQBoxRows), &full[s], wpol);
  };
  auto issue_h = [&](int it, int s) {  // the H blocks of iteration it
    const int ks = it % nks;
    uint8_t* st = ring + static_cast<size_t>(s) * kQStageBytes;
    for (int hb = 0; hb < 2 * stage_tasks(ks); ++hb)
      tc_tma_load_2d(st + kQHOff + hb * kQHBlock, &hmap, ks * kQStageElems + hb * 64, 0,
                     &full[s]);
  };
  // The weights are never written by the path: the first stages' codes and pairs stream in
  // before the wait for the previous kernel; H only after it.
  const int pre = min(S, total_it);
  if (warp == 0 && lane == 0) {
    for (int it = 0; it < pre; ++it) issue_w(it, it);
    pdl_wait();
    for (int it = 0; it < pre; ++it) issue_h(it, it);
  } else {
    pdl_wait();
  }
  if (tid >= 32 && tid < 32 + kMaxRows) {
    const int r = tid - 32;
    load_row_inputs(p, ri, r);
    s_temp[r] = (r < p.nrows && p.logits) ? ri->T[r] : 0.f;
  }
  __syncthreads();
  volatile int* vflag = &flags[0];

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int it = pre, s = pre % S;
      for (; it < total_it && !*vflag; ++it) {
        if (!mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((it / S) & 1) ^ 1))) {
          atomicOr(&p.hdr->error, ERR_TC_WAIT);
          atomicExch(&flags[0], 1);
          break;
        }
        issue_w(it, s);
        issue_h(it, s);
        if (++s == S) s = 0;
      }
      for (int j = max(0, it - S); j < it; ++j) {  // every issued copy lands before exit
        if (!mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1))) {
          atomicOr(&p.hdr->error, ERR_GEMV_DRAIN);
          break;
        }
      }
    }
  } else if (warp <= kQIssuers) {
    // ------------------------------------------------------------------ MMA issuers
    // Task n (global order): K block jt of stage ks of tile t, A buffer n % kQABufs, issued by
    // thread n % 3 into its own accumulator of tile t. Every issuer visits every stage in
    // order (the full phase gives the H blocks) and releases it once.
    if (lane == 0) {
      const int j0 = warp - 1;
      const uint32_t idesc = tc_idesc(kQTileRows, kQN);
      const uint64_t adesc = smem_desc_sw128(smem_u32(abufs));
      const uint64_t ring_desc = smem_desc_sw128(smem_u32(ring));
      int n = 0;
      bool ok = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const uint32_t dacc = tmem_base + static_cast<uint32_t>(j0 * kQAccCols + t * kQN);
        uint32_t acc = 0u;  // the first MMA of this issuer in the tile starts the sum
        for (int ks = 0; ks < nks && ok; ++ks) {
          const int it = t * nks + ks, s = it % S;
          if (*vflag || !mbar_wait_bounded(&full[s], static_cast<uint32_t>((it / S) & 1))) {
            ok = false;
            break;
          }
          const uint64_t hst =
              desc_advance(ring_desc, static_cast<uint32_t>(s * kQStageBytes + kQHOff));
          const int cnt = stage_tasks(ks);
          for (int jt = (j0 - n % kQIssuers + kQIssuers) % kQIssuers; jt < cnt;
               jt += kQIssuers) {
            const int nn = n + jt, buf = nn % kQABufs;
            if (*vflag ||
                !mbar_wait_bounded(&a_full[buf], static_cast<uint32_t>((nn / kQABufs) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a = desc_advance(adesc, static_cast<uint32_t>(buf * kQABufBytes));
            const uint64_t b = desc_advance(hst, static_cast<uint32_t>(2 * jt * kQHBlock));
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
              for (int k16 = 0; k16 < 4; ++k16) {
                tc_mma(dacc, desc_advance(a, c * kQKBlockBytes + k16 * 32),
                       desc_advance(b, c * kQHBlock + k16 * 32), idesc, acc);
                acc = 1u;
              }
            }
            tc_commit(&a_empty[buf]);  // the A buffer is free once these MMAs have read it
          }
          if (ok) tc_commit(&empty[s]);  // and the stage's H blocks
          n += cnt;
        }
      }
      if (!ok) {
        atomicOr(&p.hdr->error, ERR_TC_WAIT);
        atomicExch(&flags[0], 1);
      }
      tc_commit(mma_done);  // arrives once every MMA this thread issued has completed
    }
  } else if (warp >= kQDeqWarp0) {
    // ------------------------------------------------------------------ dequantisation
    // Task n goes to slot n % 3 of every row quarter; the four warps of a task each write 32
    // rows of its A buffer and arrive on a_full (count 4). Every warp waits on every stage's
    // full phase in order and releases every stage once, so no warp is ever two phases away
    // from a stage barrier, whatever tasks it skips.
    const int quarter = warp & 3, slot = (warp - kQDeqWarp0) >> 2;
    const int r = quarter * 32 + lane;  // tile row
    int n = 0;  // global index of the current stage's first task
    bool ok = true;
    for (int t = 0; t < ntile && ok; ++t) {
      for (int ks = 0; ks < nks && ok; ++ks) {
        const int it = t * nks + ks, s = it % S;
        const int cnt = stage_tasks(ks);
        // every lane waits (each needs the barrier's acquire of the copied bytes); the warp
        // goes on only if all of them saw the phase complete. (Lane 0 alone waiting, the others
        // held at a shuffle, measured slower.)
        if (!__all_sync(0xffffffffu, !*vflag && mbar_wait_bounded(
                                         &full[s], static_cast<uint32_t>((it / S) & 1)))) {
          ok = false;
          break;
        }
        const uint8_t* st = ring + static_cast<size_t>(s) * kQStageBytes;
        const int first = (slot - n % kQDeqSlots + kQDeqSlots) % kQDeqSlots;
        if (first >= cnt) {  // no task here: release the stage at once
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        for (int jt = first; jt < cnt; jt += kQDeqSlots) {
          const int nn = n + jt, buf = nn % kQABufs;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&a_empty[buf], static_cast<uint32_t>(
                                                              ((nn / kQABufs) & 1) ^ 1)))) {
            ok = false;
            break;
          }
          // the task's 128 elements: code units 4 (jt & 1) .. +3 of chunk jt / 2 of the row (one
          // group each) and pairs 4 jt .. 4 jt + 3 of the stage
          const uint8_t* crow = st + (jt >> 1) * kQCodeTile + r * kQChunkBytes;
          const uint4 sbv =
              *reinterpret_cast<const uint4*>(st + kQPairOff + r * kQPairRowBytes + jt * 16);
          uint4 w[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int u = (jt & 1) * 4 + g;
            w[g] = *reinterpret_cast<const uint4*>(crow + ((u ^ (r & 7)) << 4));
          }
          if (jt + kQDeqSlots >= cnt) {  // this warp's last task of the stage: its bytes are in
            __syncwarp();                // registers, so the codes and pairs may be replaced
            if (lane == 0) mbar_arrive(&empty[s]);
          }
          const uint32_t sbw[4] = {sbv.x, sbv.y, sbv.z, sbv.w};
          // row r of K block c of the A buffer: 16-byte unit u (elements 8u .. 8u+7) at
          // c*16384 + r*128 + ((u ^ (r & 7)) << 4)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            dequant_group(w[2 * c], sbw[2 * c], o);
            dequant_group(w[2 * c + 1], sbw[2 * c + 1], o + 16);
            uint8_t* arow = abufs + static_cast<size_t>(buf) * kQABufBytes + c * kQKBlockBytes +
                            r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(arow + ((u ^ (r & 7)) << 4)) =
                  make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[buf]);
        }
        n += cnt;
      }
    }
    if (!ok && lane == 0) {
      atomicOr(&p.hdr->error, ERR_TC_WAIT);
      atomicExch(&flags[0], 1);
    }
  }

  // Streaming is over for every role; wait for the block's last MMAs, then the ring is free.
  // The next kernel may now be scheduled into this kernel's tail (not earlier: blocks parked in
  // its wait during the stream cost bandwidth).
  __syncthreads();
  const bool mmas_done = mbar_wait_bounded(mma_done, 0u);
  tc_fence_after();
  if (!mmas_done && tid == 0) {
    atomicOr(&p.hdr->error, ERR_TC_WAIT);
    atomicExch(&flags[0], 1);
  }
  pdl_trigger();
  Top2* s_top = reinterpret_cast<Top2*>(ring);                              // [16 warps][8]
  int* s_bad = reinterpret_cast<int*>(ring + 16 * kMaxRows * sizeof(Top2));  // [16][8]
  unsigned long long* s_sum = reinterpret_cast<unsigned long long*>(ring + 2560);  // [8]
  static_assert(16 * kMaxRows * (sizeof(Top2) + sizeof(int)) <= 2560, "statistics layout");
  const int ew = warp & 3, quarter = warp >> 2;  // lane quadrant; four warps per quadrant
  const bool go = mmas_done && !*vflag;
  const int tpt = (nks - 1) * kQTasksPerStage + last_tasks;  // tasks per tile
  // logit rows 0..7 of tile t for this warp's 32 lanes: the issuers' partial sums in a fixed
  // order (an issuer with no task in the tile, possible only below three tasks a tile, has
  // nothing there)
  auto tile_logits = [&](int t, float* v) {
    const uint32_t base = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                          static_cast<uint32_t>(t * kQN);
    bool any = false;
#pragma unroll
    for (int j = 0; j < kQIssuers; ++j) {
      // issuer j has a task in tile t: the first task index >= t * tpt that is j mod 3 falls
      // inside the tile (always so from three tasks a tile)
      if (tpt >= kQIssuers || ((j - t * tpt) % kQIssuers + kQIssuers) % kQIssuers < tpt) {
        float w[8];
        tmem_ld8(base + static_cast<uint32_t>(j * kQAccCols), w);  // warp-uniform branch
#pragma unroll
        for (int r = 0; r < 8; ++r) v[r] = any ? __fadd_rn(v[r], w[r]) : w[r];
        any = true;
      }
    }
  };
  // pass 1: logits of rows at T > 0 and each row's top-2 over the tiles of this warp
  {
    Top2 run[kMaxRows];
    int rbad[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      run[r] = top2_empty();
      rbad[r] = 0;
    }
    bool hot = false;
    for (int r = 0; r < nr; ++r) hot |= s_temp[r] > 0.f;
    for (int t = quarter; go && t < ntile; t += 4) {
      float v[8];
      tile_logits(t, v);
      const int local = t * kQTileRows + ew * 32 + lane;
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
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        s_top[warp * kMaxRows + r] = run[r];
        s_bad[warp * kMaxRows + r] = rbad[r];
      }
    }
  }
  if (tid < kMaxRows) s_sum[tid] = 0ull;
  __syncthreads();

  // pass 2: exact integer sums of the block's logits against the block max; the four warps of
  // a lane quadrant take every fourth tile
  if (go) {
    float mref[kMaxRows], invT[kMaxRows];
    bool dosum[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      Top2 m = top2_empty();
      for (int w = 0; w < 16; ++w) m = top2_merge(m, s_top[w * kMaxRows + r]);
      mref[r] = m.best;
      dosum[r] = r < nr && m.idx != kNoIndex && m.best != -INFINITY;
      invT[r] = ri->invT[r];
    }
    unsigned long long acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0ull;
    for (int t = quarter; t < ntile; t += 4) {
      float v[8];
      tile_logits(t, v);
      const int local = t * kQTileRows + ew * 32 + lane;
      const bool ok = local < nt;
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < nr) {
          const float z = v[r];
          const unsigned long long w = tile_weight(z, mref[r], invT[r]);
          acc[r] += (ok && dosum[r] && !(isnan(z) || z == INFINITY)) ? w : 0ull;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < nr) {
        const unsigned long long a = warp_sum_u64(acc[r]);
        if (lane == 0) atomicAdd(&s_sum[r], a);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kQTmemCols);
  }
  if (tid < nr) {
    Top2 m = top2_empty();
    int bad = 0;
    for (int w = 0; w < 16; ++w) {
      m = top2_merge(m, s_top[w * kMaxRows + tid]);
      bad |= s_bad[w * kMaxRows + tid];
    }
    GemvPartial pp;
    pp.m = m.best;
    pp.second = m.second;
    pp.idx = (m.idx == kNoIndex) ? -1 : m.idx;
    pp.flags = bad;
    pp.s = s_sum[tid];
    pp.pad = 0ull;
    p.part[static_cast<size_t>(blockIdx.x) * kMaxRows + tid] = pp;
  }
  gemv_finish(p, ring + kQStatBytes, flags, kQThreads / 32, ri);
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

int gemv_q4_band_rows() { return kQBoxRows; }
int gemv_q4_stage_bytes() { return kQStageBytes; }
int gemv_q4_max_block_rows() { return kQMaxTiles * kQTileRows; }
int gemv_q4_stat_bytes() { return kQStatBytes; }
int gemv_q4_code_box_bytes() { return kQChunkBytes; }
int gemv_q4_pair_box_bytes() { return kQPairRowBytes; }
int gemv_q4_box_rows() { return kQBoxRows; }
int gemv_q4_h_rows() { return kQN; }
int gemv_q4_h_box_elems() { return 64; }
// the A buffers, plus barriers, TMEM slot, flags, temperatures, row inputs and alignment
size_t gemv_q4_abuf_bytes() { return static_cast<size_t>(kQABufs) * kQABufBytes; }
size_t gemv_q4_fixed_bytes(int) { return gemv_q4_abuf_bytes() + 2048; }

cudaError_t gemv_q4_launch(const GemvQ4Launch& L, cudaStream_t stream) {
  static SmemAllowance allowed;
  cudaError_t e = allow_dynamic_smem(gemv_q4_kernel, L.smem, allowed);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, gemv_q4_kernel, kQThreads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorLaunchOutOfResources;
  return launch_pdl(gemv_q4_kernel, dim3(L.grid), dim3(kQThreads), L.smem, stream, L.cmap, L.smap,
                    L.hmap, L.p);
}

}  // namespace spec
