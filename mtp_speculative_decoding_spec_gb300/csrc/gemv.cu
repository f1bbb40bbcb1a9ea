// LM-head projection of 1..8 rows (verify rows, or one draft row per request) on the CUDA
// cores, for fp32 weights (bf16 weights run on the tensor cores, gemv_tc.cu), with the row
// statistics and, for the draft head, the token choice fused in.
//
// Shape of the work (lucebox-hub PR #15 "MTP speculative decoding", section "What": the trunk
// verifies k drafts in one batched forward of k+1 rows through the shared LM head; the draft
// head spans the first 64,000 vocabulary rows and chooses its token on the GPU): z = H W^T with
// W [V, d] streamed once from HBM, H [rows <= 8, d] tiny. This is a streaming GEMV: the weight
// bytes bound it, so the design is about keeping HBM busy with few instructions per weight
// byte (the kernel is templated on the weight type; only fp32 is instantiated):
//   * one persistent block per SM; the vocabulary is cut into 60-row bands and block c owns a
//     contiguous run of bands (balanced to one band, no wave tail, the same cut for any number
//     of rows);
//   * a producer warp streams each band as k-slabs of [60 rows x 512 bytes] with 2-D TMA
//     tensor copies into a ring of shared-memory stages completed on mbarriers;
//   * fifteen consumer warps each own 4 rows of the band and compute their full dot products:
//     lane l takes bytes [16 l, 16 l + 16) of every slab row, and the H rows sit in shared
//     memory as fp32 pairs laid out so that one conflict-free 128-bit load feeds packed
//     fp32x2 FMAs for two H rows; one butterfly (xor 16, 8, 4, 2, 1) per band finishes each
//     dot product. Every step of a row's sum is fixed by k alone, so every row's logits are
//     bitwise batch-invariant (section "Exactness": up to eight rows, a row's verify logits may
//     not depend on how many rows are verified together);
//   * the block keeps its tile of logits in shared memory, reduces max / argmax / top-2 and a
//     sum of exp((z - m)/T) quantised to 2^-40 units in 64-bit integers (exact, so the sum
//     does not depend on order either), and the last block to finish combines the per-block
//     partials; for the draft head at T > 0 it also draws the token by inverse CDF and writes
//     it to device memory (gemv_epilogue.cuh, shared with the tensor-core kernel).
#include <math.h>

#include "gemv_epilogue.cuh"

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

// 15 consumer warps + 1 producer: 16 warps put 4 on each SM sub-partition (more latency
// hiding), whose 16K registers then allow up to 128 per thread.
constexpr int kBandWarps = 15;                     // consumer warps per block
constexpr int kRowsPerWarp = 4;                    // weight rows per consumer warp per band
constexpr int kBandRows = kBandWarps * kRowsPerWarp;  // 60
constexpr int kSlabBytes = 512;                    // bytes of one weight row per k-slab

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
      : "memory");
}

template <int RP>
__global__ void __maxnreg__(128)
    gemv_rows_kernel(const __grid_constant__ CUtensorMap wmap, const GemvParams p) {
  pdl_wait();
  if (draft_step_idle(p)) return;
  constexpr int EPC = 4;                    // fp32 elements per 16-byte chunk
  constexpr int PP = EPC / 2;               // element pairs per chunk
  constexpr int RH = RP >= 2 ? RP / 2 : 1;  // H row pairs held per 128-bit load
  constexpr int G = kRowsPerWarp;
  constexpr int NV = G * RP;                // dot products finished per warp per band
  constexpr int SPREAD = 32 / NV;           // lanes holding the same value after the reduction
  static_assert(NV <= 32 && 32 % NV == 0, "reduction layout");
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, NW = kBandWarps, PRODUCER = kBandWarps;
  uint8_t* stage_base = smem;                                     // ring, [S][60 rows][512 B]
  float4* hs = reinterpret_cast<float4*>(smem + p.ring_bytes);   // H pairs
  float* ztile = reinterpret_cast<float*>(smem + p.ring_bytes + p.hs_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(ztile + static_cast<size_t>(RP) * p.tile_cap);
  uint64_t* empty = full + S;
  int* flags = reinterpret_cast<int*>(empty + S);  // [0] abort, [1] last block
  float* s_temp = reinterpret_cast<float*>(flags + 4);  // [8] T of rows whose logits are written
  RowInputs* ri = reinterpret_cast<RowInputs*>(
      (reinterpret_cast<uintptr_t>(s_temp + kMaxRows) + 7) & ~static_cast<uintptr_t>(7));

  const int GR = gridDim.x, blk = blockIdx.x;
  int64_t v0, v1;
  block_rows(blk, GR, p.nbands, kBandRows, p.V, v0, v1);
  const int nt = static_cast<int>(v1 - v0);
  const int nb = (nt + kBandRows - 1) / kBandRows;  // bands of this block
  const int niter = nb * p.nslab;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (tid < kMaxRows)
    s_temp[tid] = (tid < p.nrows && p.logits) ? p.temperature[tid / p.rows_per_req] : 0.f;
  if (tid < kMaxRows) load_row_inputs(p, ri, tid);
  // H rows -> shared memory as fp32 pairs: entry ((s*PP + q)*RH + rr)*32 + l holds
  // (h[2rr][k], h[2rr][k+1], h[2rr+1][k], h[2rr+1][k+1]) with k = s*slab_elems + l*EPC + 2q.
  {
    const int total = p.nslab * PP * RH * 32;
    for (int i = tid; i < total; i += blockDim.x) {
      const int l = i & 31, rr = (i >> 5) % RH, q = (i / (32 * RH)) % PP, s = i / (32 * RH * PP);
      const int k = s * p.slab_elems + l * EPC + 2 * q;
      float h4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = 2 * rr + (u >> 1), kk = k + (u & 1);
        float hv = 0.f;
        if (r < p.nrows && kk < p.d) {
          hv = reinterpret_cast<const float*>(p.H + static_cast<size_t>(r) * p.h_row_bytes)[kk];
        }
        h4[u] = hv;
      }
      hs[i] = make_float4(h4[0], h4[1], h4[2], h4[3]);
    }
  }
  __syncthreads();

  if (warp == PRODUCER) {
    // ---------------- producer: stream k-slabs of 60-row bands into the stage ring ---------
    if (lane == 0) {
      int issued = 0;
      const int y0 = static_cast<int>(v0);
      int s = 0, band = 0, slab = 0;
      uint32_t eph = 0;  // parity of the empty-barrier phase to wait for (second lap onwards)
      for (int it = 0; it < (p.stall ? 0 : niter); ++it) {
        if (it >= S && !mbar_wait_bounded(&empty[s], eph)) {
          atomicOr(&p.hdr->error, ERR_GEMV_WAIT_EMPTY);
          atomicExch(&flags[0], 1);
          break;
        }
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(p.stage_bytes));
        tma_load_2d(stage_base + static_cast<size_t>(s) * p.stage_bytes, &wmap,
                    slab * p.slab_elems, y0 + band * kBandRows, &full[s]);
        issued = it + 1;
        if (++slab == p.nslab) {
          slab = 0;
          ++band;
        }
        if (++s == S) {
          s = 0;
          if (it + 1 > S) eph ^= 1u;  // laps 2, 3, ... wait on phases 0, 1, 0, ...
        }
      }
      // every issued copy must have landed before this block may exit
      for (int it = max(0, issued - S); it < issued; ++it) {
        if (!mbar_wait_bounded(&full[it % S], (it / S) & 1)) {
          atomicOr(&p.hdr->error, ERR_GEMV_DRAIN);
          break;
        }
      }
    }
  } else {
    // ---------------- consumers: 4 rows per warp, full dot products ----------------
    const int wrow = warp * G;  // first row of this warp within a band
    // acc[g][r]: packed (even-element, odd-element) partial sums of row g against H row r
    unsigned long long acc[G][RP];
    const uint64_t ring_wait = p.ring_wait_ns ? p.ring_wait_ns : 2000000000ull;
    int s = 0, band = 0, slab = 0;
    uint32_t ph = 0;
    for (int it = 0; it < niter; ++it) {
      if (slab == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int r = 0; r < RP; ++r) acc[g][r] = 0ull;
      }
      if (!mbar_wait_bounded(&full[s], ph, ring_wait)) {
        atomicOr(&p.hdr->error, ERR_GEMV_WAIT_FULL);
        atomicExch(&flags[0], 1);
        break;
      }
      uint4 w[G];
      const uint8_t* sp = stage_base + static_cast<size_t>(s) * p.stage_bytes +
                          static_cast<size_t>(wrow) * kSlabBytes + lane * 16;
#pragma unroll
      for (int g = 0; g < G; ++g) w[g] = lds128(sp + g * kSlabBytes);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // release orders the loads above before reuse

      const float4* hp = hs + static_cast<size_t>(slab) * PP * RH * 32 + lane;
#pragma unroll
      for (int q = 0; q < PP; ++q) {
        unsigned long long wp[G];  // element pair q of each row: (w[2q], w[2q+1]) as fp32
#pragma unroll
        for (int g = 0; g < G; ++g) {
          wp[g] = (q == 0) ? pack2(w[g].x, w[g].y) : pack2(w[g].z, w[g].w);
        }
#pragma unroll
        for (int rr = 0; rr < RH; ++rr) {
          unsigned long long h0, h1;  // (h[2rr][k], h[2rr][k+1]), (h[2rr+1][k], h[2rr+1][k+1])
          lds128_b64(hp + (q * RH + rr) * 32, h0, h1);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            ffma2_acc(acc[g][2 * rr], wp[g], h0);
            if (2 * rr + 1 < RP) ffma2_acc(acc[g][2 * rr + 1], wp[g], h1);
          }
        }
      }

      if (slab == p.nslab - 1) {
        // the band's dot products are complete in each lane's k-range: sum across the warp
        float v[NV];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int r = 0; r < RP; ++r) v[g * RP + r] = sum2(acc[g][r]);
        ReduceScatter<NV, 16>::run(v, lane);
        if ((lane % SPREAD) == 0) {
          const int i = lane / SPREAD, g = i / RP, r = i % RP;
          const int local = band * kBandRows + wrow + g;
          if (r < p.nrows && local < nt) {
            ztile[static_cast<size_t>(r) * p.tile_cap + local] = v[0];
            if (s_temp[r] > 0.f)
              p.logits[static_cast<size_t>(r) * p.logits_stride + v0 + local] = v[0];
          }
        }
      }
      if (++slab == p.nslab) {
        slab = 0;
        ++band;
      }
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  __syncthreads();

  pdl_trigger();
  gemv_block_epilogue(p, ztile, v0, nt, stage_base, flags, NW + 1, ri);
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

template <int RP>
static cudaError_t launch_variant(const GemvLaunch& L, cudaStream_t stream) {
  auto kern = gemv_rows_kernel<RP>;
  static SmemAllowance allowed;  // per variant
  cudaError_t e = allow_dynamic_smem(kern, L.smem, allowed);
  if (e != cudaSuccess) return e;
  int fit = 0;  // registers and shared memory must admit one block per SM
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kern, L.threads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorLaunchOutOfResources;
  return launch_pdl(kern, dim3(L.grid), dim3(L.threads), L.smem, stream, L.wmap, L.p);
}

cudaError_t gemv_dispatch(const GemvLaunch& L, int rp, cudaStream_t stream) {
  switch (rp) {
    case 1: return launch_variant<1>(L, stream);
    case 2: return launch_variant<2>(L, stream);
    case 4: return launch_variant<4>(L, stream);
    default: return launch_variant<8>(L, stream);
  }
}

}  // namespace spec
