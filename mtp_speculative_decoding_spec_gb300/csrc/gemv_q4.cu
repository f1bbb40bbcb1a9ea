// LM-head projection of 1..8 rows over 4-bit affine weights in groups of 32 (DS4Server issue
// #98, closing comment: the MTP head's weights are 4-bit affine values in groups of 32), with
// the same fused row statistics and draft draw as the bf16 kernels.
//
// Row layout (5d/8 bytes per vocabulary row, d a multiple of 128): d/2 bytes of codes, then one
// (scale, bias) bf16 pair per 32-element group. In each little-endian 32-bit word of 8
// consecutive codes e0..e7, e_{2i} sits in bits 4i..4i+3 and e_{2i+1} in bits 16+4i..16+4i+3.
// The dequantised weight is bf16(s*q + b), rounded once, so z = H w^T is a bf16 projection.
//
// Design. The weights are a quarter of the bf16 bytes plus the pairs (1,600 against 5,120 bytes
// per row at d = 2560), and every weight costs ALU work before anything can use it. Measured on
// this part: bf16x2 FMAs and the integer ALU ops (shift, LOP3, PRMT) issue at 64 lanes a cycle
// per SM, so exact dequantisation (two bf16x2 FMAs and ~2 ALU ops per weight pair) is the cost
// to minimise, and every further instruction per weight counts:
//   * a tcgen05 form needs the dequantised weights in shared memory (A from shared memory or
//     tensor memory) with a handshake per block of A between the writing warps and the issuing
//     thread; such a version of this kernel measured ~123 us for 2 rows;
//   * a CUDA-core form (each thread one row, the bf16 pairs widened to fp32 and multiplied into
//     fp32 sums with packed FMAs) spends ~1.5 more instructions per weight and row on the
//     widening and the FMAs; it measured ~112 us for 2 rows and ~234 us for 8;
//   * here the dequantised pairs go straight from registers into warp-level MMAs
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate): a bf16x2 pair of consecutive elements of
//     one row is exactly one register of the MMA's A fragment, so each thread dequantises only
//     the elements its fragment holds, and one MMA per 8 weights of a thread replaces the
//     widening and all the FMAs, for any number of rows up to 8 (the 8 H rows are the MMA's N).
// The MMA's throughput is not the question here (an 8-row projection is a few percent of what
// the tensor cores can do); its register operands are.
//   * sixteen warps own one 32-row box each (512 rows a pass, up to two passes a block), as two
//     16-row MMA tiles; each warp streams its box through a ring of its own (two slots): a stage
//     is 128 code bytes and 32 pair bytes (256 elements) of each of its rows, two 2-D TMA boxes
//     (the codes with 128-byte swizzle, so the 16-byte reads of 8 consecutive rows hit distinct
//     banks) under an evict-first L2 policy, issued by the warp itself. Measured alternatives:
//     one ring shared by all warps (refilled by the last warp out of a stage) held every warp to
//     the slowest one (~135 us); 128-element stages (64-byte code rows) with four slots, 92 us;
//     8 or 12 warps with deeper rings, 90 / 84 us; the same boxes by per-lane cp.async, 86 us;
//     L2 prefetch of later stages, 84 us. At ~2 stages in flight a warp waits ~1 us a stage for
//     its next slot: the loads take ~4 us, which is the bytes in flight over the ~4.6 TB/s this
//     access pattern (128 + 32 bytes of every 1,600-byte row per stage) gets from HBM.
//   * the k order inside each 32-element group is permuted, the same way in A and B (the same
//     products are summed; only the order of the MMA's fp32 additions changes, and it is the
//     same for every row and every row count): thread c of a quad takes the four pairs of code
//     word c (elements 8c .. 8c + 7), so one 32-bit shared load gives a thread a row's word and
//     the four pairs come out of it by constant shifts;
//   * H (the block's up to 8 rows, rows past nrows zero) is copied once to shared memory as
//     [d/32 groups][8 rows][32 bf16] (natural order inside a group): under that permutation one
//     16-byte load gives thread (g, c) its B registers for a group, elements 8c .. 8c + 7 of H
//     row g;
//   * after the stream a thread holds, per pass, the logits of 4 vocabulary rows for 2 H rows
//     (in registers); the logits of rows at T > 0 are stored, and the row statistics and the
//     shared finish run as in the bf16 kernels.
// Batch invariance: column n of an MMA depends only on H row n (column n of B), and every row
// goes through the same MMAs in the same order whatever the number of rows, so the logits of a
// row are bitwise the same for 1..8 rows.
#include "gemv_epilogue.cuh"
#include "tcgen05.cuh"

namespace spec {

constexpr int kQWarps = 16;                        // every warp consumes; no producer warp
constexpr int kQThreads = 32 * kQWarps;            // 512
constexpr int kQBoxRows = 32;                      // rows per TMA box, and the partition's band
constexpr int kQPassRows = kQBoxRows * kQWarps;    // 512
constexpr int kQMaxPasses = 2;
constexpr int kQStageElems = 256;                  // elements of each row per stage
constexpr int kQGroups = kQStageElems / 32;        // 32-element groups per stage
constexpr int kQCodeRow = kQStageElems / 2;        // 128 code bytes of a row per stage
constexpr int kQPairRow = kQGroups * 4;            // 32 bytes of (scale, bias) pairs
constexpr int kQCodeBox = kQBoxRows * kQCodeRow;   // 4 KB
constexpr int kQPairBox = kQBoxRows * kQPairRow;   // 1 KB
constexpr int kQSlotBytes = kQCodeBox + kQPairBox;  // one warp's stage: its box's codes, pairs
constexpr int kQVals = 8;  // logits a thread holds per pass: 2 tiles x 2 rows x 2 H rows
constexpr int kQStatBytes = 4096;  // per-warp top-2 and flags, row sums; then the finish scratch

static_assert(kQCodeRow == 64 || kQCodeRow == 128, "code rows use the 64- or 128-byte swizzle");
static_assert(kQCodeBox % (8 * kQCodeRow) == 0 && kQSlotBytes % (8 * kQCodeRow) == 0,
              "code boxes keep the alignment of their swizzle pattern (8 rows)");

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// D += A B for one 16 x 8 tile over k = 16: A [16 rows][16] bf16 (row-major fragment), B
// [16][8] bf16 (column-major fragment), D fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_addr(const void* a) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(a));
}
__device__ __forceinline__ uint32_t lds4(uint32_t a) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(a));
  return v;
}

// (s, s) and (b, b) from a (scale, bias) pair, by unpacking the two bf16 halves and packing
// each twice. Measured against a byte permute per splat: 76.4 -> 71.9 us for the 2-row verify.
__device__ __forceinline__ void splat_pair(uint32_t sb, uint32_t& s2, uint32_t& b2) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tmov.b32 %0, {lo, lo};\n\t"
      "mov.b32 %1, {hi, hi};\n\t}"
      : "=r"(s2), "=r"(b2)
      : "r"(sb));
}

// One A-fragment register: a pair of consecutive elements of an 8-element code word, its two
// codes at bits 0..3 and 16..19 of v (the word shifted right by 4 j for pair j), dequantised:
// the bf16 pair (128 + e, 128 + e') (the code lands in the low mantissa bits of 128 = 0x4300,
// where one unit is 1), minus 128 (exact), times s plus b, rounded once.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t v, uint32_t s2, uint32_t b2) {
  const uint32_t t = (v & 0x000F000Fu) | 0x43004300u;
  const uint32_t q = bf16x2_fma(t, 0x3F803F80u, 0xC300C300u);
  return bf16x2_fma(q, s2, b2);
}

// The word's four pairs, in order (pair j = elements 2j, 2j + 1): constant shifts.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2,
                                             uint32_t (&o)[4]) {
  o[0] = dequant_pair(w, s2, b2);
  o[1] = dequant_pair(w >> 4, s2, b2);
  o[2] = dequant_pair(w >> 8, s2, b2);
  o[3] = dequant_pair(w >> 12, s2, b2);
}

__global__ void __launch_bounds__(kQThreads, 1)
    gemv_q4_kernel(const __grid_constant__ CUtensorMap cmap,
                   const __grid_constant__ CUtensorMap smap, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (draft_step_idle(p)) return;  // before any setup: nothing in flight
  const int S = p.stages;              // slots of each warp's ring
  uint8_t* ring = smem;                // [16 warps][S][slot]; afterwards statistics and scratch
  uint8_t* hs = smem + p.ring_bytes;   // H: [d/32 groups][8 rows][32 bf16]
  uint64_t* full = reinterpret_cast<uint64_t*>(hs + p.hs_bytes);  // [8 warps][S]
  int* flags = reinterpret_cast<int*>(full + kQWarps * S);  // [0] abort, [1] last block
  float* s_temp = reinterpret_cast<float*>(flags + 4);
  RowInputs* ri = reinterpret_cast<RowInputs*>(
      (reinterpret_cast<uintptr_t>(s_temp + kMaxRows) + 7) & ~static_cast<uintptr_t>(7));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;  // MMA fragment coordinates: row group, column pair
  int64_t v0, v1;
  block_rows(blockIdx.x, gridDim.x, p.nbands, kQBoxRows, p.V, v0, v1);
  const int nt = static_cast<int>(v1 - v0);
  const int npass = (nt + kQPassRows - 1) / kQPassRows;
  const int d = p.d;
  const int nks = (d + kQStageElems - 1) / kQStageElems;  // a last half stage reads zeros
  const int nr = min(p.nrows, kMaxRows);
  // this warp's box: rows warp*32 .. warp*32 + 31 of each pass; the passes where it has rows
  const int wrow0 = warp * kQBoxRows;
  const int wpass = nt > wrow0 ? (nt - wrow0 + kQPassRows - 1) / kQPassRows : 0;
  const int wtotal = wpass * nks;  // this warp's stages
  uint64_t* wfull = full + warp * S;
  uint8_t* wring = ring + static_cast<size_t>(warp) * S * kQSlotBytes;

  if (tid == 0) {
    for (int s = 0; s < kQWarps * S; ++s) mbar_init(&full[s], 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t wpol = l2_policy_evict_first();  // codes and pairs: read once, not kept in L2
  auto issue = [&](int it) {  // this warp's codes and pairs of its stage it, into slot it % S
    const int pass = it / nks, ks = it - pass * nks, s = it % S;
    const int row = box_row(p, static_cast<int>(v0) + pass * kQPassRows + wrow0);
    uint8_t* st = wring + static_cast<size_t>(s) * kQSlotBytes;
    mbar_arrive_expect_tx(&wfull[s], static_cast<uint32_t>(kQSlotBytes));
    tc_tma_load_2d_hint(st, &cmap, ks * kQCodeRow, row, &wfull[s], wpol);
    tc_tma_load_2d_hint(st + kQCodeBox, &smap, ks * kQPairRow, row, &wfull[s], wpol);
  };

  // The weights are never written by the path: the first stages stream in before the wait for
  // the previous kernel; H and the row inputs only after it.
  int issued = min(S, wtotal);  // this warp's stages issued so far (tracked by lane 0)
  if (lane == 0)
    for (int it = 0; it < issued; ++it) issue(it);
  pdl_wait();
  {
    // 16-byte unit (G*8 + n)*4 + c = H row n at elements 32 G + 8 c .. 32 G + 8 c + 7: thread
    // (g, c) of a warp reads its B fragments of group G (n = g) in one 16-byte load; groups
    // past d (the rest of a last half stage) are zero. Every load of a thread is issued before
    // its stores (word-by-word loads serialised into ~5 us here).
    uint4* hu = reinterpret_cast<uint4*>(hs);
    const int nchunk = nks * kQGroups * 4;  // 16-byte chunks of a row, whole stages
    const int total = kMaxRows * nchunk;
    constexpr int kPer = 4;  // chunks a thread loads per round
    for (int i0 = tid; i0 < total; i0 += kPer * kQThreads) {
      uint4 v[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = i0 + u * kQThreads, n = i / nchunk, j = i - n * nchunk;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (i < total && n < nr && j < d / 8)
          v[u] = __ldg(reinterpret_cast<const uint4*>(p.H + static_cast<size_t>(n) *
                                                                p.h_row_bytes) + j);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = i0 + u * kQThreads, n = i / nchunk, j = i - n * nchunk;
        if (i < total) hu[((j >> 2) * 8 + n) * 4 + (j & 3)] = v[u];
      }
    }
  }
  if (tid < kMaxRows) {
    load_row_inputs(p, ri, tid);
    s_temp[tid] = (tid < p.nrows && p.logits) ? ri->T[tid] : 0.f;
  }
  __syncthreads();
  volatile int* vflag = &flags[0];

  // ------------------------------------------------------------------------ the stream
  // Each warp streams its own 32-row box through its own ring of S slots: it waits for a slot,
  // computes, and refills the slot with its stage it + S, so no warp ever waits for another.
  // Thread (g, c) holds A-fragment rows g and g + 8 of the box's two 16-row tiles (box rows
  // 16 mt + 8 h + g) and accumulates their logits for H rows 2c and 2c + 1. The MMA's k order
  // within a group is permuted (A and B alike): thread c's fragment registers take the four
  // pairs of code word c (elements 8c .. 8c + 7), so every shift is a constant and its B
  // fragments are 16 contiguous bytes of the H row.
  float zv[kQMaxPasses][kQVals];  // each pass's logits, [mt][h][j]
#pragma unroll
  for (int ps = 0; ps < kQMaxPasses; ++ps)
#pragma unroll
    for (int v = 0; v < kQVals; ++v) zv[ps][v] = 0.f;
  {
    const uint32_t wring_s = smem_addr(wring), hs_s = smem_addr(hs);
    // the swizzle of box rows 16 mt + 8 h + g: 16-byte unit u sits at u ^ (row & 7) (128-byte
    // rows) or u ^ ((row >> 1) & 3) (64-byte rows)
    const int swz = (kQCodeRow == 128 ? g : (g >> 1) & 3) << 4;
    float acc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mt][q] = 0.f;
    int it = 0;
#pragma unroll 1
    for (; it < wtotal; ++it) {
      const int pass = it / nks, ks = it - pass * nks, s = it % S;
      const uint32_t ph = static_cast<uint32_t>((it / S) & 1);
      // every lane waits (each needs the barrier's acquire of the copied bytes)
      if (!__all_sync(0xffffffffu, !*vflag && mbar_wait_bounded(&wfull[s], ph))) break;
      const uint32_t st = wring_s + static_cast<uint32_t>(s * kQSlotBytes);
      uint4 pr[2][2][kQGroups / 4];  // the stage's (scale, bias) pairs of this thread's rows
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int u = 0; u < kQGroups / 4; ++u)
            pr[mt][h][u] = lds16(st + kQCodeBox + (mt * 16 + h * 8 + g) * kQPairRow + 16 * u);
      const uint32_t hk = hs_s + static_cast<uint32_t>(ks * kQGroups * 512);
#pragma unroll
      for (int gg = 0; gg < kQGroups; ++gg) {  // group gg: elements 32 gg .. 32 gg + 31
        const uint4 hb = lds16(hk + gg * 512 + (g * 4 + c) * 16);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // code word c of the group in rows 16 mt + g and 16 mt + 8 + g (the same swizzle)
          const uint32_t ra = st + (mt * 16 + g) * kQCodeRow + ((gg << 4) ^ swz) + 4 * c;
          const uint32_t wa = lds4(ra), wb = lds4(ra + 8 * kQCodeRow);
          const uint4 pa = pr[mt][0][gg >> 2], pb = pr[mt][1][gg >> 2];
          const int gq = gg & 3;
          const uint32_t sa = gq == 0 ? pa.x : gq == 1 ? pa.y : gq == 2 ? pa.z : pa.w;
          const uint32_t sb = gq == 0 ? pb.x : gq == 1 ? pb.y : gq == 2 ? pb.z : pb.w;
          uint32_t sa2, ba2, sb2, bb2;
          splat_pair(sa, sa2, ba2);
          splat_pair(sb, sb2, bb2);
          uint32_t da[4], db[4];
          dequant_word(wa, sa2, ba2, da);
          dequant_word(wb, sb2, bb2, db);
          // pairs 0, 1 of the word in the first k16 step (with H elements 8c .. 8c + 3), 2, 3
          // in the second (8c + 4 .. 8c + 7)
          mma_bf16_16816(acc[mt], da[0], db[0], da[1], db[1], hb.x, hb.y);
          mma_bf16_16816(acc[mt], da[2], db[2], da[3], db[3], hb.z, hb.w);
        }
      }
      // every lane's reads of the slot are done: order them before the copy that refills it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0 && issued < wtotal) issue(issued++);
      if (ks == nks - 1) {  // the pass's rows are complete
#pragma unroll
        for (int ps = 0; ps < kQMaxPasses; ++ps)
          if (ps == pass)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int q = 0; q < 4; ++q) zv[ps][mt * 4 + q] = acc[mt][q];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[mt][q] = 0.f;
      }
    }
    if (it < wtotal) {  // a wait ran out or another warp gave up
      if (lane == 0) {
        atomicOr(&p.hdr->error, ERR_TC_WAIT);
        atomicExch(&flags[0], 1);
      }
    }
    // every copy this warp issued lands before the ring is reused (on the normal path each one
    // has been waited for already)
    if (lane == 0) {
      for (int j = it; j < issued; ++j) {
        if (!mbar_wait_bounded(&wfull[j % S], static_cast<uint32_t>((j / S) & 1))) {
          atomicOr(&p.hdr->error, ERR_GEMV_DRAIN);
          break;
        }
      }
    }
  }
  __syncthreads();
  // The next kernel may now be scheduled into this kernel's tail.
  pdl_trigger();
  Top2* s_top = reinterpret_cast<Top2*>(ring);                              // [16 warps][8]
  int* s_bad = reinterpret_cast<int*>(ring + 16 * kMaxRows * sizeof(Top2));  // [16][8]
  unsigned long long* s_sum = reinterpret_cast<unsigned long long*>(ring + 2560);  // [8]
  static_assert(16 * kMaxRows * (sizeof(Top2) + sizeof(int)) <= 2560, "statistics layout");
  const bool go = !*vflag;
  // value v = 4 mt + 2 h + j of pass ps: box row 16 mt + 8 h + g, H row 2c + j
  auto zlocal = [&](int ps, int v) {
    return ps * kQPassRows + wrow0 + (v >> 2) * 16 + ((v >> 1) & 1) * 8 + g;
  };
  // H row n lives in the lanes with c = n / 2, so a thread's values cover H rows 2c and 2c + 1,
  // and one reduction over the eight lanes of equal c (xor 4, 8, 16) serves all 8 rows at once.
  Top2* s_mtop = reinterpret_cast<Top2*>(ring + 2560 + 64);  // [8]: the block's top-2 per row
  static_assert(2560 + 64 + kMaxRows * sizeof(Top2) <= kQStatBytes, "statistics layout");
  // pass 1: logits of rows at T > 0, and each row's top-2 and NaN / +Inf flag per warp
  {
    Top2 t[2] = {top2_empty(), top2_empty()};
    int bad[2] = {0, 0};
    if (go) {
#pragma unroll
      for (int ps = 0; ps < kQMaxPasses; ++ps) {
#pragma unroll
        for (int v = 0; v < kQVals; ++v) {
          const int j = v & 1, n = 2 * c + j, local = zlocal(ps, v);
          if (ps < npass && n < nr && local < nt) {
            const float z = zv[ps][v];
            if (s_temp[n] > 0.f)
              p.logits[static_cast<size_t>(n) * p.logits_stride + v0 + local] = z;
            if (isnan(z) || z == INFINITY)
              bad[j] = 1;
            else
              top2_push(t[j], z, static_cast<int32_t>(v0 + local));
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        Top2 u;
        u.best = __shfl_xor_sync(0xffffffffu, t[j].best, o);
        u.second = __shfl_xor_sync(0xffffffffu, t[j].second, o);
        u.idx = __shfl_xor_sync(0xffffffffu, t[j].idx, o);
        t[j] = top2_merge(t[j], u);
        bad[j] |= __shfl_xor_sync(0xffffffffu, bad[j], o);
      }
    }
    if (lane < 4) {  // lane c: rows 2c, 2c + 1
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        s_top[warp * kMaxRows + 2 * lane + j] = t[j];
        s_bad[warp * kMaxRows + 2 * lane + j] = bad[j];
      }
    }
  }
  if (tid < kMaxRows) s_sum[tid] = 0ull;
  __syncthreads();
  if (tid < kMaxRows) {  // the block's top-2 of row tid, over the warps in order
    Top2 m = top2_empty();
    for (int w = 0; w < kQWarps; ++w) m = top2_merge(m, s_top[w * kMaxRows + tid]);
    s_mtop[tid] = m;
  }
  __syncthreads();

  // pass 2: exact integer sums of the block's logits against the block max
  if (go) {
    float mref[2], invT[2];
    bool dosum[2];
    unsigned long long a[2] = {0ull, 0ull};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = 2 * c + j;
      const Top2 m = s_mtop[n];
      mref[j] = m.best;
      dosum[j] = n < nr && m.idx != kNoIndex && m.best != -INFINITY;
      invT[j] = ri->invT[n];
    }
#pragma unroll
    for (int ps = 0; ps < kQMaxPasses; ++ps) {
#pragma unroll
      for (int v = 0; v < kQVals; ++v) {
        const int j = v & 1;
        const float z = zv[ps][v];
        if (ps < npass && dosum[j] && zlocal(ps, v) < nt && !(isnan(z) || z == INFINITY))
          a[j] += tile_weight(z, mref[j], invT[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) a[j] += __shfl_xor_sync(0xffffffffu, a[j], o);
    }
    if (lane < 4) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (2 * lane + j < nr) atomicAdd(&s_sum[2 * lane + j], a[j]);
    }
  }
  __syncthreads();
  if (tid < nr) {
    const Top2 m = s_mtop[tid];
    int bad = 0;
    for (int w = 0; w < kQWarps; ++w) bad |= s_bad[w * kMaxRows + tid];
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
// one slot of every warp's ring (the host sizes the ring in these units)
int gemv_q4_stage_bytes() { return kQWarps * kQSlotBytes; }
int gemv_q4_max_block_rows() { return kQMaxPasses * kQPassRows; }
int gemv_q4_stat_bytes() { return kQStatBytes; }
int gemv_q4_code_box_bytes() { return kQCodeRow; }
int gemv_q4_pair_box_bytes() { return kQPairRow; }
int gemv_q4_box_rows() { return kQBoxRows; }
// H in shared memory, grouped by 32 elements: 8 rows (rows past nrows zero) of d bf16 values,
// padded with zeros to whole stages
size_t gemv_q4_h_bytes(int d) {
  return static_cast<size_t>((d + kQStageElems - 1) / kQStageElems) * kQStageElems * 16;
}
// barriers, flags, temperatures, row inputs and alignment
size_t gemv_q4_fixed_bytes() { return 3072; }

cudaError_t gemv_q4_launch(const GemvQ4Launch& L, cudaStream_t stream) {
  static SmemAllowance allowed;
  cudaError_t e = allow_dynamic_smem(gemv_q4_kernel, L.smem, allowed);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, gemv_q4_kernel, kQThreads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorLaunchOutOfResources;
  return launch_pdl(gemv_q4_kernel, dim3(L.grid), dim3(kQThreads), L.smem, stream, L.cmap,
                    L.smap, L.p);
}

}  // namespace spec
