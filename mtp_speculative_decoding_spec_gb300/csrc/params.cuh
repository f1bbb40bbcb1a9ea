// Launch parameter blocks of the kernels (passed by value to each kernel).
#pragma once

#include <cuda.h>

#include <mutex>
#include <utility>

#include "common.cuh"

namespace spec {

struct GemvParams {
  int64_t V;        // rows projected (the verify vocabulary, or the draft rows)
  int d;            // hidden size
  int nslab;        // 512-byte k-slabs per weight row
  int slab_elems;   // elements per slab
  int64_t nbands;   // bands of band_rows rows over V (the unit of the block partition)
  int band_rows;    // 60 (CUDA-core kernel) or 32 (tensor-core kernel)
  int stages;
  int stage_bytes;  // one slab of one band: 60 rows x 512 bytes
  int ring_bytes;   // >= stages * stage_bytes; the last block reuses it as scratch
  int hs_bytes;     // shared-memory copy of H as fp32 pairs
  int tile_cap;     // max rows per block tile
  const uint8_t* H;
  int h_row_bytes;
  int nrows;
  int rows_per_req;
  const float* temperature;
  float* logits;  // nullable
  int64_t logits_stride;
  spec_rowstats* stats;  // nullable
  int draft;
  const uint64_t* seed;
  const int64_t* pos;
  int pos_offset;
  int32_t* token_out;
  int token_stride;
  const int32_t* kact;  // draft head: row b needs this step only if kact[b] > pos_offset (nullable)
  // projected row r (r < V) is weight row r below lo_rows and hi_row0 + r - lo_rows from there
  // (a draft set of two ranges; lo_rows = V when the rows are simply [0, V))
  int64_t lo_rows, hi_row0;
  WsHeader* hdr;
  GemvPartial* part;
  // failure-detection test of the bounded waits (CUDA-core kernel only): when stall is set the
  // producer issues no copy, and the consumers' waits for a stage give up after ring_wait_ns
  uint64_t ring_wait_ns;  // 0: the default limit
  int stall;
  // greedy acceptance fused into the last block's finish (spec_verify_accept_greedy) when
  // acc_out is set: drafts [B][acc_k_max], k [B], results and counters per request
  const int32_t* acc_k;
  const int32_t* acc_drafts;
  spec_accept_out* acc_out;
  spec_counters* acc_counters;
  int acc_k_max;
  int acc_eos;
  // and after it, when ad_state is set, the width update of spec_adapt_width_mirror (k_used =
  // acc_k; ad_k_mirror nullable)
  const float* ad_cost;
  const float* ad_cycle_cost;
  float ad_alpha;
  spec_width_state* ad_state;
  int32_t* ad_k_next;
  int32_t* ad_k_mirror;
};

// The greedy acceptance (and width update) a GEMV launch may carry (see GemvParams::acc_out).
struct GreedyAcc {
  const int32_t* k;
  const int32_t* drafts;
  spec_accept_out* out;
  spec_counters* counters;
  int k_max;
  int eos;
  const float* cost;
  const float* cycle_cost;
  float alpha;
  spec_width_state* state;  // null: no width update
  int32_t* k_next;
  int32_t* k_mirror;
};
inline void set_greedy(GemvParams& p, const GreedyAcc* g) {
  if (!g) return;
  p.acc_k = g->k;
  p.acc_drafts = g->drafts;
  p.acc_out = g->out;
  p.acc_counters = g->counters;
  p.acc_k_max = g->k_max;
  p.acc_eos = g->eos;
  p.ad_cost = g->cost;
  p.ad_cycle_cost = g->cycle_cost;
  p.ad_alpha = g->alpha;
  p.ad_state = g->state;
  p.ad_k_next = g->k_next;
  p.ad_k_mirror = g->k_mirror;
}

// Shared memory the last block's combine needs: per row, for each block, its integer sum (8
// bytes), max / scale factor, runner-up / weight and argmax (4 bytes each), rounded up; then
// one flag per row.
__host__ __device__ constexpr size_t gemv_finish_row_bytes(int nblocks) {
  return 24 * static_cast<size_t>(nblocks);
}
__host__ __device__ constexpr size_t gemv_finish_scratch_bytes(int nblocks) {
  return kMaxRows * gemv_finish_row_bytes(nblocks) + 64 + kMaxRows * sizeof(spec_rowstats);
}

struct GemvLaunch {
  int grid, threads, smem;
  CUtensorMap wmap;  // W as a 2-D tensor [V rows][d], box [60 rows][512 bytes]
  GemvParams p;
};

struct AcceptParams {
  int B, k_max, R, NS;
  const int32_t* k;
  const int32_t* drafts;
  const float* logits;
  const spec_rowstats* stats;
  int64_t V;
  const float* q_logits;
  const spec_rowstats* q_stats;
  int64_t Vd;
  int64_t q_stride;
  const float* temperature;
  int eos;
  const uint64_t* seed;
  const int64_t* pos_base;
  spec_accept_out* out;
  spec_counters* counters;
  uint32_t* tickets;         // [B]
  unsigned long long* sums;  // [B][NS][8]: ratio rule: residual, p; exact-match: p of rows 0..k
  int exact;                 // exact-match acceptance at T > 0
  int filtered;              // top-k / top-p filtered target at T > 0 (one-hot q)
  const int32_t* top_k;      // [B] in [1, kMaxTopK]
  const float* top_p;        // [B] in (0, 1]
  unsigned long long* cand;  // [B][NS][8 rows][kMaxTopK] each slice's best keys, descending
  // draft row of vocabulary id x: x below q_lo, q_lo + x - q_hi0 in [q_hi0, q_hi0 + Vd - q_lo),
  // none elsewhere (q_lo = Vd when the draft rows are [0, Vd))
  int64_t q_lo, q_hi0;
};

constexpr int kMaxTopK = 32;               // largest top-k of the filtered acceptance
constexpr int64_t kMaxFilteredV = 1 << 20;  // its vocabulary limit: at most 4 slices a thread

struct CommitParams {
  spec_state_desc st;
  const spec_accept_out* acc;
  const int32_t* k;
  int mode;
  int32_t* commit_status;
};

// Batched tensor-core path (9..256 rows): see gemm_tc.cu.
struct GemmPartial {  // a row's statistics over one CTA's tiles and one column half (32 bytes)
  float m;            // largest finite logit (-inf if none)
  float second;
  int32_t idx;        // -1 if none
  int32_t flags;      // bit 0: NaN or +Inf seen
  double s;           // sum of exp((z - m)/T)
  double pad;
};
static_assert(sizeof(GemmPartial) == 32, "partial is 32 bytes");

struct GemmParams {
  int64_t V;
  int d;
  int nrows;
  int rows_per_req;
  int ntiles;     // 128-row vocabulary tiles
  int nblocks;    // CTAs of the tensor-core kernel (partials per row = 2 * nblocks)
  int vec_store;  // logits rows 16-byte aligned (V % 4 == 0)
  const float* temperature;
  float* logits;  // nullable
  int64_t logits_stride;
  spec_rowstats* stats;
  WsHeader* hdr;
  GemmPartial* part;  // [nrows][nblocks][2]
};

struct GemmLaunch {
  int grid, smem;
  CUtensorMap hmap;  // H [nrows][d] bf16, box [128 rows][64], 128-byte swizzle
  CUtensorMap wmap;  // W [V][d] bf16, box [128 rows][64], 128-byte swizzle
  GemmParams p;
};

// Launch with programmatic stream serialization: the kernel may be scheduled while the previous
// kernel of the stream is still running; it calls pdl_wait before touching that kernel's data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A kernel's dynamic shared-memory limit, raised per device (the attribute belongs to the
// device's copy of the kernel) and only when a launch needs more than has been allowed there.
// The mutex keeps two threads' first launches from lowering each other's setting.
struct SmemAllowance {
  static constexpr int kDevices = 64;
  std::mutex mu;
  int bytes[kDevices] = {};
};

template <typename... KArgs>
inline cudaError_t allow_dynamic_smem(void (*kernel)(KArgs...), int bytes, SmemAllowance& a) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < SmemAllowance::kDevices;
  std::lock_guard<std::mutex> lock(a.mu);
  if (tracked && bytes <= a.bytes[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) a.bytes[dev] = bytes;
  return e;
}

cudaError_t gemm_tc_launch(const GemmLaunch& L, cudaStream_t stream);
int gemm_tc_smem_bytes();
int gemm_tc_tile_rows();
int gemm_tc_kblock();
int gemm_tc_subtiles();
int gemm_tc_max_ctas();

cudaError_t gemv_dispatch(const GemvLaunch& L, int rp, cudaStream_t stream);

// Tensor-core variant of the 1..8-row projection for bf16 weights: see gemv_tc.cu.
struct GemvTcLaunch {
  int grid, smem;
  CUtensorMap wmap;  // W [V][d] bf16, box [32 rows][64], 128-byte swizzle
  CUtensorMap hmap;  // H [nrows][d] bf16, box [16 rows][64], 128-byte swizzle
  GemvParams p;
};

cudaError_t gemv_tc_launch(const GemvTcLaunch& L, cudaStream_t stream);

struct GemvQ4Launch {
  int grid, smem;
  CUtensorMap cmap;  // codes: [V rows][d/2 bytes], row pitch 5d/8, box [32 rows][64 B], swizzled
  CUtensorMap smap;  // (scale, bias) pairs: [V rows][d/8 bytes] from byte d/2, box [32][16 B]
  GemvParams p;      // hs_bytes = the shared-memory copy of H
};

cudaError_t gemv_q4_launch(const GemvQ4Launch& L, cudaStream_t stream);
int gemv_q4_band_rows();
int gemv_q4_stage_bytes();
int gemv_q4_max_block_rows();
int gemv_q4_stat_bytes();
int gemv_q4_code_box_bytes();
int gemv_q4_pair_box_bytes();
int gemv_q4_box_rows();
size_t gemv_q4_h_bytes(int d);
size_t gemv_q4_fixed_bytes();
int gemv_tc_band_rows();
int gemv_tc_box_rows();
int gemv_tc_kblock();
int gemv_tc_h_rows();
int gemv_tc_stage_bytes();
int gemv_tc_threads();
int gemv_tc_max_block_rows();
int gemv_tc_stat_bytes();
cudaError_t accept_launch(const AcceptParams& prm, cudaStream_t stream);
cudaError_t commit_launch(const CommitParams& prm, int B, int blocks_per_request,
                          cudaStream_t stream);
int commit_replay_rows(const spec_state_desc& st);

struct AdaptParams {
  int B, k_max;
  const spec_accept_out* out;
  const int32_t* k_used;
  const float* cost;
  const float* cycle_cost;  // [B] or null: timed on the device
  float alpha;
  spec_width_state* state;
  int32_t* k_next;
  int32_t* k_mirror;  // [B] or null: a second copy of the chosen widths (e.g. host-mapped)
};
cudaError_t adapt_launch(const AdaptParams& prm, cudaStream_t stream);
const void* width_select_function();  // the select kernel of a width graph (see abi.cu)

}  // namespace spec
