// extern "C" entry points of libspec.so: argument validation, workspace layout, launch
// configuration. Every call validates on the host, then enqueues on the caller's stream; no
// call allocates memory or synchronises.
#include <stdint.h>
#include <string.h>

#include <atomic>

#include <cuda.h>

#include "params.cuh"


namespace spec {
namespace {

constexpr int kBandRows = 60;         // GEMV band: 15 consumer warps x 4 rows
constexpr int kMaxBandsPerBlock = 34;  // per-block tile of the GEMV (logits kept in smem)
constexpr int kGemvThreads = 16 * 32;  // 15 consumer warps + 1 producer

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the CUDA driver API, fetched through the runtime (no -lcuda).
EncodeTiledFn lookup_encode_tiled() {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<EncodeTiledFn>(ptr);
  return nullptr;
}

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = lookup_encode_tiled();  // looked up once, by the first caller
  return fn;
}

struct DevAttr {
  int sms = 0;
  int smem_optin = 0;
};

// Per-device attributes, queried on first use. Calls may come from several host threads: the
// cache is atomic (sms is published last, so a non-zero sms implies smem_optin is set).
DevAttr dev_attr() {
  struct Slot {
    std::atomic<int> sms{0};
    std::atomic<int> smem_optin{0};
  };
  static Slot cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevAttr{};
  DevAttr a;
  a.sms = cache[dev].sms.load(std::memory_order_acquire);
  if (a.sms != 0) {
    a.smem_optin = cache[dev].smem_optin.load(std::memory_order_relaxed);
    return a;
  }
  if (cudaDeviceGetAttribute(&a.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&a.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
    return DevAttr{};
  cache[dev].smem_optin.store(a.smem_optin, std::memory_order_relaxed);
  cache[dev].sms.store(a.sms, std::memory_order_release);
  return a;
}

int64_t gemv_bands(int64_t V) { return (V + kBandRows - 1) / kBandRows; }

int gemv_grid(int64_t V, int sms) {
  int64_t g = sms;
  const int64_t need = (gemv_bands(V) + kMaxBandsPerBlock - 1) / kMaxBandsPerBlock;
  if (need > g) g = need;
  return static_cast<int>(g);
}

int accept_slices(int64_t V) { return static_cast<int>((V + kAcceptSlice - 1) / kAcceptSlice); }

// Workspace layout. The zero-initialised counters sit at offsets that no call's batch moves:
// the GEMV ticket in the header, the accept tickets at the END of the caller's buffer. The
// regions between them hold only values written before they are read within one call, so their
// batch-dependent offsets may overlap from one call to the next:
//   [0, 256)                    header (GEMV ticket, error word)
//   [256, part_end)             GEMV per-block partials (grid of the vocabulary size)
//   [part_end, sums_end)        accept per-slice sums (B * slices * 8 * 8 bytes)
//   [sums_end, gemm_end)        batched path: per-(row, 256-row tile) partials (no counters)
//   [gemm_end, cand_end)        filtered accept: per-(request, slice, row) top-k keys
//   [ws_bytes - tickets, end)   accept tickets, one per request
struct WsLayout {
  size_t part, sums, gemm, cand, tickets_bytes, total;
};

int gemm_rows_max(int32_t max_batch) {
  const int64_t r = 8 * static_cast<int64_t>(max_batch);
  return r > kMaxRows ? static_cast<int>(r < 256 ? r : 256) : 0;
}

WsLayout ws_layout(int64_t V, int32_t max_batch, int sms) {
  WsLayout w;
  w.part = sizeof(WsHeader);
  w.sums = w.part + align_up(sizeof(GemvPartial) * kMaxRows * gemv_grid(V, sms), 256);
  w.gemm = w.sums + align_up(sizeof(unsigned long long) * kMaxRows * static_cast<size_t>(max_batch) *
                                 accept_slices(V),
                             256);
  const int64_t ntiles = (V + 127) / 128;  // batched path: 128-row vocabulary tiles
  w.tickets_bytes = align_up(sizeof(uint32_t) * static_cast<size_t>(max_batch), 256);
  w.cand = w.gemm +
           align_up(sizeof(GemvPartial) * static_cast<size_t>(gemm_rows_max(max_batch)) * ntiles * 2,
                    256);
  // the filtered acceptance's candidate keys exist only for vocabularies it accepts
  const size_t ncand = (V <= kMaxFilteredV) ? static_cast<size_t>(max_batch) * accept_slices(V) *
                                                  kMaxRows * kMaxTopK
                                            : 0;
  w.total = w.cand + align_up(sizeof(unsigned long long) * ncand, 256) + w.tickets_bytes;
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool known_wdt(spec_dtype w) { return w == SPEC_BF16 || w == SPEC_F32 || w == SPEC_Q4A32; }

int next_pow2_rows(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

// The tensor-core variant (bf16 weights, 16-byte aligned W and H): same parameters, same grid
// and workspace as the CUDA-core kernel, the vocabulary partitioned in 32-row bands.
spec_status run_gemv_tc(const void* W, int64_t V, int64_t d, const void* H, int nrows,
                        int rows_per_req, const float* temperature, float* logits,
                        int64_t logits_stride, spec_rowstats* stats, int draft,
                        const uint64_t* seed, const int64_t* pos, int pos_offset,
                        int32_t* token_out, int token_stride, const int32_t* kact,
                        void* workspace, const WsLayout& wl, int grid, const DevAttr& a,
                        EncodeTiledFn encode, cudaStream_t stream, int64_t lo_rows,
                        int64_t hi_row0, int64_t V_rows, const GreedyAcc* ga) {
  GemvTcLaunch L;
  memset(&L, 0, sizeof(L));
  GemvParams& p = L.p;
  const int band = gemv_tc_band_rows();
  const int64_t nbands = (V + band - 1) / band;
  const int tile_cap = static_cast<int>(((nbands + grid - 1) / grid) * band);
  if (tile_cap > gemv_tc_max_block_rows()) return SPEC_ERR_UNSUPPORTED;
  // after streaming, the ring holds the per-block statistics and then the combine's scratch
  const size_t after =
      static_cast<size_t>(gemv_tc_stat_bytes()) + gemv_finish_scratch_bytes(grid);
  // barriers (2 per stage + 16), TMEM slot, flags, temperatures, per-row inputs; alignment slack
  const size_t fixed = 1024 + 1024;
  const size_t budget = static_cast<size_t>(a.smem_optin);
  int stages = 16;
  size_t ring = 0, smem_total = 0;
  for (; stages >= 2; --stages) {
    ring = static_cast<size_t>(stages) * gemv_tc_stage_bytes();
    if (ring < after) ring = align_up(after, 1024);
    smem_total = ring + fixed;
    if (smem_total <= budget) break;
  }
  if (stages < 2) return SPEC_ERR_UNSUPPORTED;

  const int64_t row_bytes = d * 2;
  const cuuint32_t estride[2] = {1, 1};
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(V_rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gemv_tc_kblock()),
                               static_cast<cuuint32_t>(gemv_tc_box_rows())};
    if (encode(&L.wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), gdim, gstride,
               box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_CUDA;
  }
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(nrows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gemv_tc_kblock()),
                               static_cast<cuuint32_t>(gemv_tc_h_rows())};
    if (encode(&L.hmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(H), gdim, gstride,
               box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_CUDA;
  }
  p.V = V;
  p.d = static_cast<int>(d);
  p.nbands = nbands;
  p.band_rows = band;
  p.stages = stages;
  p.stage_bytes = gemv_tc_stage_bytes();
  p.ring_bytes = static_cast<int>(ring);
  p.tile_cap = tile_cap;
  p.H = static_cast<const uint8_t*>(H);
  p.h_row_bytes = static_cast<int>(row_bytes);
  p.nrows = nrows;
  p.rows_per_req = rows_per_req;
  p.temperature = temperature;
  p.logits = logits;
  p.logits_stride = logits_stride;
  p.stats = stats;
  p.draft = draft;
  p.seed = seed;
  p.pos = pos;
  p.pos_offset = pos_offset;
  p.token_out = token_out;
  p.token_stride = token_stride;
  p.kact = kact;
  p.lo_rows = lo_rows;
  p.hi_row0 = hi_row0;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.part = reinterpret_cast<GemvPartial*>(static_cast<uint8_t*>(workspace) + wl.part);
  set_greedy(p, ga);
  L.grid = grid;
  L.smem = static_cast<int>(smem_total);
  const cudaError_t e = gemv_tc_launch(L, stream);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// The 4-bit affine variant: rows of 5d/8 bytes (d/2 of codes, then d/32 bf16 (scale, bias)
// pairs), the same grid, partials and finish as the bf16 tensor-core kernel.
spec_status run_gemv_q4(const void* W, int64_t V, int64_t d, const void* H, int nrows,
                        int rows_per_req, const float* temperature, float* logits,
                        int64_t logits_stride, spec_rowstats* stats, int draft,
                        const uint64_t* seed, const int64_t* pos, int pos_offset,
                        int32_t* token_out, int token_stride, const int32_t* kact,
                        void* workspace, const WsLayout& wl, int grid, const DevAttr& a,
                        EncodeTiledFn encode, cudaStream_t stream, int64_t lo_rows,
                        int64_t hi_row0, int64_t V_rows, const GreedyAcc* ga) {
  GemvQ4Launch L;
  memset(&L, 0, sizeof(L));
  GemvParams& p = L.p;
  const int band = gemv_q4_band_rows();
  const int64_t nbands = (V + band - 1) / band;
  const int tile_cap = static_cast<int>(((nbands + grid - 1) / grid) * band);
  if (tile_cap > gemv_q4_max_block_rows()) return SPEC_ERR_UNSUPPORTED;
  const size_t h_bytes = align_up(gemv_q4_h_bytes(static_cast<int>(d)), 1024);
  const size_t after =
      static_cast<size_t>(gemv_q4_stat_bytes()) + gemv_finish_scratch_bytes(grid);
  const size_t fixed = h_bytes + gemv_q4_fixed_bytes();
  const size_t budget = static_cast<size_t>(a.smem_optin);
  int stages = 6;
  size_t ring = 0, smem_total = 0;
  for (; stages >= 2; --stages) {
    ring = static_cast<size_t>(stages) * gemv_q4_stage_bytes();
    if (ring < after) ring = align_up(after, 1024);
    smem_total = ring + fixed;
    if (smem_total <= budget) break;
  }
  if (stages < 2) return SPEC_ERR_UNSUPPORTED;

  const cuuint64_t pitch[1] = {static_cast<cuuint64_t>(5 * d / 8)};
  const cuuint32_t estride[2] = {1, 1};
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d / 2), static_cast<cuuint64_t>(V_rows)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gemv_q4_code_box_bytes()),
                               static_cast<cuuint32_t>(gemv_q4_box_rows())};
    const CUtensorMapSwizzle sw = gemv_q4_code_box_bytes() == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                                  : CU_TENSOR_MAP_SWIZZLE_64B;
    if (encode(&L.cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), gdim, pitch, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_CUDA;
  }
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d / 8), static_cast<cuuint64_t>(V_rows)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gemv_q4_pair_box_bytes()),
                               static_cast<cuuint32_t>(gemv_q4_box_rows())};
    void* pairs = static_cast<uint8_t*>(const_cast<void*>(W)) + d / 2;  // 16-byte aligned
    if (encode(&L.smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pairs, gdim, pitch, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_CUDA;
  }
  p.V = V;
  p.d = static_cast<int>(d);
  p.nbands = nbands;
  p.band_rows = band;
  p.stages = stages;
  p.stage_bytes = gemv_q4_stage_bytes();
  p.ring_bytes = static_cast<int>(ring);
  p.hs_bytes = static_cast<int>(h_bytes);
  p.tile_cap = tile_cap;
  p.H = static_cast<const uint8_t*>(H);
  p.h_row_bytes = static_cast<int>(2 * d);
  p.nrows = nrows;
  p.rows_per_req = rows_per_req;
  p.temperature = temperature;
  p.logits = logits;
  p.logits_stride = logits_stride;
  p.stats = stats;
  p.draft = draft;
  p.seed = seed;
  p.pos = pos;
  p.pos_offset = pos_offset;
  p.token_out = token_out;
  p.token_stride = token_stride;
  p.kact = kact;
  p.lo_rows = lo_rows;
  p.hi_row0 = hi_row0;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.part = reinterpret_cast<GemvPartial*>(static_cast<uint8_t*>(workspace) + wl.part);
  set_greedy(p, ga);
  L.grid = grid;
  L.smem = static_cast<int>(smem_total);
  const cudaError_t e = gemv_q4_launch(L, stream);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Configure and launch the GEMV for `nrows` rows over the first V rows of W.
spec_status run_gemv(const void* W, spec_dtype wdt, int64_t V, int64_t d, const void* H,
                     int nrows, int rows_per_req, const float* temperature, float* logits,
                     int64_t logits_stride, spec_rowstats* stats, int draft,
                     const uint64_t* seed, const int64_t* pos, int pos_offset,
                     int32_t* token_out, int token_stride, const int32_t* kact, void* workspace,
                     size_t workspace_bytes, int32_t batch_for_ws, cudaStream_t stream,
                     int64_t lo_rows = -1, int64_t hi_row0 = -1, uint64_t ring_wait_ns = 0,
                     int stall = 0, const GreedyAcc* ga = nullptr) {
  // rows [0, V) are weight rows [0, V), or [0, lo_rows) then hi_row0.. (a two-range draft set)
  if (lo_rows < 0 || lo_rows >= V) {
    lo_rows = V;
    hi_row0 = V;
  }
  const int64_t V_rows = hi_row0 + (V - lo_rows);  // weight rows the tensor maps span
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return SPEC_ERR_CUDA;
  const int elt = (wdt == SPEC_BF16) ? 2 : 4;
  const int64_t row_bytes = d * elt;
  if (wdt == SPEC_Q4A32) {
    if (d % 128 != 0) return SPEC_ERR_INVALID;  // whole words of codes, 16-byte row pitch
    if (d > 4096) return SPEC_ERR_UNSUPPORTED;
  } else {
    if (row_bytes % 16 != 0) return SPEC_ERR_INVALID;
    if (d > (wdt == SPEC_BF16 ? 3072 : 1536)) return SPEC_ERR_UNSUPPORTED;
  }
  // batch_for_ws = 0: a scratch that holds only what the LM head uses (header and partials,
  // which come first in every layout); otherwise the caller's full workspace
  const WsLayout wl = ws_layout(V, batch_for_ws > 0 ? batch_for_ws : 1, a.sms);
  if (workspace_bytes < (batch_for_ws > 0 ? wl.total : wl.sums)) return SPEC_ERR_INVALID;
  EncodeTiledFn encode = encode_tiled();
  if (!encode) return SPEC_ERR_CUDA;

  const int grid = gemv_grid(V, a.sms);
  if (wdt == SPEC_Q4A32)  // every entry point has checked that W and H are 16-byte aligned
    return run_gemv_q4(W, V, d, H, nrows, rows_per_req, temperature, logits, logits_stride, stats,
                       draft, seed, pos, pos_offset, token_out, token_stride, kact, workspace, wl,
                       grid, a, encode, stream, lo_rows, hi_row0, V_rows, ga);
  if (wdt == SPEC_BF16)  // every entry point has checked that W and H are 16-byte aligned
    return run_gemv_tc(W, V, d, H, nrows, rows_per_req, temperature, logits, logits_stride, stats,
                       draft, seed, pos, pos_offset, token_out, token_stride, kact, workspace, wl,
                       grid, a, encode, stream, lo_rows, hi_row0, V_rows, ga);
  if (lo_rows != V) return SPEC_ERR_UNSUPPORTED;  // the fp32 kernel's 60-row bands: [0, V) only

  GemvLaunch L;
  memset(&L, 0, sizeof(L));
  GemvParams& p = L.p;
  const int rp = next_pow2_rows(nrows);
  const int slab_elems = 512 / elt;
  const int nslab = static_cast<int>((d + slab_elems - 1) / slab_elems);
  const int64_t nbands = gemv_bands(V);
  const int tile_cap = static_cast<int>(((nbands + grid - 1) / grid) * kBandRows);
  const int stage_bytes = kBandRows * 512;
  const int pairs = (elt == 2) ? 4 : 2;
  const int row_pairs = rp >= 2 ? rp / 2 : 1;
  const size_t hs_bytes = static_cast<size_t>(nslab) * pairs * row_pairs * 32 * 16;
  // the last block reuses the stage ring for the combine's scratch
  const size_t scratch = gemv_finish_scratch_bytes(grid);
  // + flags, temperatures, per-row inputs (with alignment)
  const size_t fixed = hs_bytes + static_cast<size_t>(rp) * tile_cap * 4 + 512;
  const size_t budget = static_cast<size_t>(a.smem_optin);
  int stages = 8;
  size_t ring = 0, smem_total = 0;
  for (; stages >= 2; --stages) {
    ring = static_cast<size_t>(stages) * stage_bytes;
    if (ring < scratch) ring = align_up(scratch, 128);
    smem_total = ring + fixed + static_cast<size_t>(stages) * 16;
    if (smem_total <= budget) break;
  }
  if (stages < 2) return SPEC_ERR_UNSUPPORTED;

  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(V)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(slab_elems), static_cast<cuuint32_t>(kBandRows)};
  const cuuint32_t estride[2] = {1, 1};
  if (encode(&L.wmap, elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             2, const_cast<void*>(W), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SPEC_ERR_CUDA;

  p.V = V;
  p.d = static_cast<int>(d);
  p.nslab = nslab;
  p.slab_elems = slab_elems;
  p.nbands = nbands;
  p.band_rows = kBandRows;
  p.stages = stages;
  p.stage_bytes = stage_bytes;
  p.ring_bytes = static_cast<int>(ring);
  p.hs_bytes = static_cast<int>(hs_bytes);
  p.tile_cap = tile_cap;
  p.H = static_cast<const uint8_t*>(H);
  p.h_row_bytes = static_cast<int>(row_bytes);
  p.nrows = nrows;
  p.rows_per_req = rows_per_req;
  p.temperature = temperature;
  p.logits = logits;
  p.logits_stride = logits_stride;
  p.stats = stats;
  p.draft = draft;
  p.seed = seed;
  p.pos = pos;
  p.pos_offset = pos_offset;
  p.token_out = token_out;
  p.token_stride = token_stride;
  p.kact = kact;
  p.lo_rows = V;
  p.hi_row0 = V;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.part = reinterpret_cast<GemvPartial*>(static_cast<uint8_t*>(workspace) + wl.part);
  p.ring_wait_ns = ring_wait_ns;
  p.stall = stall;
  set_greedy(p, ga);
  L.grid = grid;
  L.threads = kGemvThreads;
  L.smem = static_cast<int>(smem_total);
  const cudaError_t e = gemv_dispatch(L, rp, stream);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// The batched tensor-core path (9..256 rows, bf16, d a multiple of 64).
spec_status run_gemm(const void* W, int64_t V, int64_t d, const void* H, int nrows,
                     int rows_per_req, const float* temperature, float* logits,
                     int64_t logits_stride, spec_rowstats* stats, void* workspace,
                     size_t workspace_bytes, int32_t batch_for_ws, cudaStream_t stream) {
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return SPEC_ERR_CUDA;
  if (d % gemm_tc_kblock() != 0 || nrows > 256) return SPEC_ERR_UNSUPPORTED;
  const WsLayout wl = ws_layout(V, batch_for_ws, a.sms);
  if (workspace_bytes < wl.total || gemm_rows_max(batch_for_ws) < nrows) return SPEC_ERR_INVALID;
  if (gemm_tc_smem_bytes() > a.smem_optin) return SPEC_ERR_UNSUPPORTED;
  EncodeTiledFn encode = encode_tiled();
  if (!encode) return SPEC_ERR_CUDA;
  GemmLaunch L;
  memset(&L, 0, sizeof(L));
  const cuuint64_t hdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(nrows)};
  const cuuint64_t wdim[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(V)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(d * 2)};
  const cuuint32_t hbox[2] = {static_cast<cuuint32_t>(gemm_tc_kblock()), 128};
  const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(gemm_tc_kblock()),
                              static_cast<cuuint32_t>(gemm_tc_tile_rows())};
  const cuuint32_t estride[2] = {1, 1};
  if (encode(&L.hmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(H), hdim, gstride,
             hbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SPEC_ERR_CUDA;
  if (encode(&L.wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), wdim, gstride,
             wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SPEC_ERR_CUDA;
  GemmParams& p = L.p;
  p.V = V;
  p.d = static_cast<int>(d);
  p.nrows = nrows;
  p.rows_per_req = rows_per_req;
  p.ntiles = static_cast<int>((V + gemm_tc_tile_rows() - 1) / gemm_tc_tile_rows());
  p.vec_store = (logits_stride % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) ? 1 : 0;
  p.temperature = temperature;
  p.logits = logits;
  p.logits_stride = logits_stride;
  p.stats = stats;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.part = reinterpret_cast<GemmPartial*>(static_cast<uint8_t*>(workspace) + wl.gemm);
  L.grid = p.ntiles < a.sms ? p.ntiles : a.sms;
  if (L.grid > gemm_tc_max_ctas()) L.grid = gemm_tc_max_ctas();  // the combine's partial limit
  p.nblocks = L.grid;
  L.smem = gemm_tc_smem_bytes();
  const cudaError_t e = gemm_tc_launch(L, stream);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// spec_accept and spec_accept_exact: validation, workspace layout, launch.
spec_status run_accept(int32_t B, int32_t k_max, const int32_t* k, const int32_t* drafts,
                       const float* logits, const spec_rowstats* stats, int64_t V, int32_t R,
                       const float* q_logits, const spec_rowstats* q_stats, int64_t V_draft,
                       int64_t q_stride, const float* temperature, int32_t eos_id,
                       const uint64_t* seed, const int64_t* pos_base, spec_accept_out* out,
                       spec_counters* counters, void* workspace, size_t workspace_bytes,
                       spec_stream_t stream, int exact, const int32_t* top_k = nullptr,
                       const float* top_p = nullptr, int64_t q_lo = -1, int64_t q_hi0 = -1) {
  if (B < 1 || k_max < 0 || k_max > kMaxRows - 1 || R < 1 || R > kMaxRows) return SPEC_ERR_INVALID;
  if (!k || (k_max > 0 && !drafts) || !stats || !temperature || !seed || !pos_base || !out ||
      !workspace)
    return SPEC_ERR_INVALID;
  if (V < 1 || V >= (int64_t(1) << 24)) return SPEC_ERR_INVALID;
  if (q_logits && (!q_stats || V_draft < 1 || V_draft > V || q_stride < V_draft))
    return SPEC_ERR_INVALID;
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return SPEC_ERR_CUDA;
  const WsLayout wl = ws_layout(V, B, a.sms);
  if (workspace_bytes < wl.total) return SPEC_ERR_INVALID;
  AcceptParams p;
  memset(&p, 0, sizeof(p));
  p.B = B;
  p.k_max = k_max;
  p.R = R;
  p.NS = accept_slices(V);
  p.k = k;
  p.drafts = drafts;
  p.logits = logits;
  p.stats = stats;
  p.V = V;
  p.q_logits = q_logits;
  p.q_stats = q_stats;
  p.Vd = q_logits ? V_draft : 0;
  // draft rows [0, Vd) are ids [0, Vd), or [0, q_lo) then q_hi0.. (a two-range draft set)
  if (q_lo < 0 || q_lo >= p.Vd) {
    q_lo = p.Vd;
    q_hi0 = p.Vd;
  }
  if (q_hi0 < q_lo || q_hi0 + (p.Vd - q_lo) > V) return SPEC_ERR_INVALID;
  p.q_lo = q_lo;
  p.q_hi0 = q_hi0;
  p.q_stride = q_stride;
  p.temperature = temperature;
  p.eos = eos_id;
  p.seed = seed;
  p.pos_base = pos_base;
  p.out = out;
  p.counters = counters;
  p.exact = exact;
  if (top_k) {  // filtered acceptance
    if (!top_p) return SPEC_ERR_INVALID;
    if (V > kMaxFilteredV) return SPEC_ERR_UNSUPPORTED;
    p.filtered = 1;
    p.top_k = top_k;
    p.top_p = top_p;
    p.cand = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + wl.cand);
  }
  // tickets: the last 4*B bytes of the buffer, its end rounded down to 4 bytes (see WsLayout)
  const size_t end4 = workspace_bytes & ~static_cast<size_t>(3);
  p.tickets = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + end4 -
                                          sizeof(uint32_t) * static_cast<size_t>(B));
  p.sums = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + wl.sums);
  const cudaError_t e = accept_launch(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace
}  // namespace spec

using namespace spec;

namespace spec {

// Copy of n 16-byte vectors from mapped host memory to device memory: each thread reads its
// vectors (at most four) at once, then waits for the stream's previous kernel before writing.
__global__ void __launch_bounds__(256) copy_from_host_kernel(uint4* __restrict__ dst,
                                                             const uint4* __restrict__ src,
                                                             int64_t n) {
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (i0 + u * step < n) v[u] = src[i0 + u * step];
  pdl_wait();
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (i0 + u * step < n) dst[i0 + u * step] = v[u];
}

// Device-accessible address of p, or nullptr: device or managed memory as it is, pinned host
// memory through its device alias.
void* device_accessible(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error this lookup may leave
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
    return const_cast<void*>(p);
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

}  // namespace spec

extern "C" {

size_t spec_workspace_bytes(int64_t V, int32_t max_batch) {
  if (V < 1 || max_batch < 1) return 0;
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return 0;
  return ws_layout(V, max_batch, a.sms).total;
}

const char* spec_status_str(spec_status s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID: return "SPEC_ERR_INVALID";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
  }
  return "SPEC_ERR_UNKNOWN";
}

int32_t spec_batched_supported(void) { return 1; }

spec_status spec_host_alias(const void* host_ptr, void** dev_ptr) {
  if (!host_ptr || !dev_ptr) return SPEC_ERR_INVALID;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host_ptr) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_INVALID;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return SPEC_ERR_INVALID;
  *dev_ptr = at.devicePointer;
  return SPEC_OK;
}

spec_status spec_copy_from_host(void* dst, const void* src_host, size_t bytes,
                                spec_stream_t stream) {
  if (bytes == 0) return SPEC_OK;
  if (!dst || !src_host || bytes % 16 != 0 || reinterpret_cast<uintptr_t>(dst) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(src_host) % 16 != 0)
    return SPEC_ERR_INVALID;
  void* src = nullptr;
  if (spec_host_alias(src_host, &src) != SPEC_OK) return SPEC_ERR_INVALID;
  void* d = spec::device_accessible(dst);
  if (!d) return SPEC_ERR_INVALID;
  const int64_t n = static_cast<int64_t>(bytes / 16);
  const int64_t grid = (n + 4 * 256 - 1) / (4 * 256);
  if (grid > 65535) return SPEC_ERR_UNSUPPORTED;  // 64 MiB per call
  const cudaError_t e = spec::launch_pdl(spec::copy_from_host_kernel, dim3(static_cast<unsigned>(grid)),
                                         dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                                         static_cast<uint4*>(d), static_cast<const uint4*>(src), n);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_lmhead_verify(const void* W, spec_dtype wdt, int64_t V, int64_t d,
                               const void* H, int32_t B, int32_t R, const float* temperature,
                               float* logits, spec_rowstats* stats, void* workspace,
                               size_t workspace_bytes, spec_stream_t stream) {
  if (!W || !H || !temperature || !stats || !workspace) return SPEC_ERR_INVALID;
  if (!known_wdt(wdt)) return SPEC_ERR_INVALID;
  if (V < 1 || V >= (int64_t(1) << 24) || d < 1 || B < 1 || R < 1 || R > kMaxRows)
    return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(H) || !aligned16(workspace)) return SPEC_ERR_INVALID;
  if (static_cast<int64_t>(B) * R > kMaxRows) {
    if (wdt != SPEC_BF16 || static_cast<int64_t>(B) * R > 256) return SPEC_ERR_UNSUPPORTED;
    return run_gemm(W, V, d, H, B * R, R, temperature, logits, V, stats, workspace,
                    workspace_bytes, B, reinterpret_cast<cudaStream_t>(stream));
  }
  return run_gemv(W, wdt, V, d, H, B * R, R, temperature, logits, V, stats, 0, nullptr,
                  nullptr, 0, nullptr, 0, nullptr, workspace, workspace_bytes, B,
                  reinterpret_cast<cudaStream_t>(stream));
}

spec_status spec_verify_accept_greedy(const void* W, spec_dtype wdt, int64_t V, int64_t d,
                                      const void* H, int32_t B, int32_t R,
                                      const float* temperature, float* logits,
                                      spec_rowstats* stats, int32_t k_max, const int32_t* k,
                                      const int32_t* drafts, int32_t eos_id,
                                      spec_accept_out* out, spec_counters* counters,
                                      const float* cost, const float* cycle_cost, float alpha,
                                      spec_width_state* state, int32_t* k_next,
                                      int32_t* k_mirror, void* workspace,
                                      size_t workspace_bytes, spec_stream_t stream) {
  if (!W || !H || !temperature || !stats || !workspace || !k || !out) return SPEC_ERR_INVALID;
  if (state && (!cost || !k_next || !(alpha > 0.f && alpha <= 1.f))) return SPEC_ERR_INVALID;
  if (!known_wdt(wdt)) return SPEC_ERR_INVALID;
  if (V < 1 || V >= (int64_t(1) << 24) || d < 1 || B < 1 || R < 1 || R > kMaxRows)
    return SPEC_ERR_INVALID;
  if (k_max < 0 || k_max > kMaxRows - 1 || (k_max > 0 && !drafts)) return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(H) || !aligned16(workspace)) return SPEC_ERR_INVALID;
  if (static_cast<int64_t>(B) * R > kMaxRows) return SPEC_ERR_UNSUPPORTED;  // the GEMV path only
  GreedyAcc ga;
  ga.k = k;
  ga.drafts = drafts;
  ga.out = out;
  ga.counters = counters;
  ga.k_max = k_max;
  ga.eos = eos_id;
  ga.cost = cost;
  ga.cycle_cost = cycle_cost;
  ga.alpha = alpha;
  ga.state = state;
  ga.k_next = k_next;
  ga.k_mirror = k_mirror;
  return run_gemv(W, wdt, V, d, H, B * R, R, temperature, logits, V, stats, 0, nullptr,
                  nullptr, 0, nullptr, 0, nullptr, workspace, workspace_bytes, B,
                  reinterpret_cast<cudaStream_t>(stream), -1, -1, 0, 0, &ga);
}

spec_status spec_draft_argmax(const void* W, spec_dtype wdt, int64_t V_draft, int64_t d,
                              const void* h, int32_t B, const float* temperature,
                              const uint64_t* seed, const int64_t* pos, int32_t pos_offset,
                              int32_t* token_out, int32_t token_stride, float* q_logits,
                              int64_t q_stride, spec_rowstats* q_stats, const int32_t* k_active,
                              void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  if (!W || !h || !temperature || !seed || !pos || !token_out || !workspace)
    return SPEC_ERR_INVALID;
  if (!known_wdt(wdt)) return SPEC_ERR_INVALID;
  if (V_draft < 1 || V_draft >= (int64_t(1) << 24) || d < 1 || B < 1 || B > kMaxRows)
    return SPEC_ERR_INVALID;
  if (token_stride < 1 || (q_logits && q_stride < V_draft)) return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(h) || !aligned16(workspace)) return SPEC_ERR_INVALID;
  return run_gemv(W, wdt, V_draft, d, h, B, 1, temperature, q_logits, q_stride, q_stats, 1,
                  seed, pos, pos_offset, token_out, token_stride, k_active, workspace,
                  workspace_bytes, B, reinterpret_cast<cudaStream_t>(stream));
}

spec_status spec_draft_argmax_rows(const void* W, spec_dtype wdt, int64_t n_low, int64_t hi_first,
                                   int64_t n_high, int64_t d, const void* h, int32_t B,
                                   const float* temperature, const uint64_t* seed,
                                   const int64_t* pos, int32_t pos_offset, int32_t* token_out,
                                   int32_t token_stride, float* q_logits, int64_t q_stride,
                                   spec_rowstats* q_stats, const int32_t* k_active,
                                   void* workspace, size_t workspace_bytes,
                                   spec_stream_t stream) {
  if (!W || !h || !temperature || !seed || !pos || !token_out || !workspace)
    return SPEC_ERR_INVALID;
  if (!known_wdt(wdt)) return SPEC_ERR_INVALID;
  if (n_low < 0 || n_high < 0 || hi_first < n_low || n_low + n_high < 1 ||
      hi_first + n_high >= (int64_t(1) << 24) || d < 1 || B < 1 || B > kMaxRows)
    return SPEC_ERR_INVALID;
  if (n_high > 0 && (wdt == SPEC_F32 || n_low % gemv_tc_box_rows() != 0))
    return SPEC_ERR_UNSUPPORTED;  // whole 32-row TMA boxes on the tensor-core kernels only
  const int64_t V_draft = n_low + n_high;
  if (token_stride < 1 || (q_logits && q_stride < V_draft)) return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(h) || !aligned16(workspace)) return SPEC_ERR_INVALID;
  return run_gemv(W, wdt, V_draft, d, h, B, 1, temperature, q_logits, q_stride, q_stats, 1,
                  seed, pos, pos_offset, token_out, token_stride, k_active, workspace,
                  workspace_bytes, B, reinterpret_cast<cudaStream_t>(stream),
                  n_high > 0 ? n_low : -1, hi_first);
}

spec_status spec_accept_rows(int32_t B, int32_t k_max, const int32_t* k, const int32_t* drafts,
                             const float* logits, const spec_rowstats* stats, int64_t V,
                             int32_t R, const float* q_logits, const spec_rowstats* q_stats,
                             int64_t n_low, int64_t hi_first, int64_t n_high, int64_t q_stride,
                             const float* temperature, int32_t eos_id, const uint64_t* seed,
                             const int64_t* pos_base, spec_accept_out* out,
                             spec_counters* counters, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream) {
  if (n_low < 0 || n_high < 0 || hi_first < n_low) return SPEC_ERR_INVALID;
  return spec::run_accept(B, k_max, k, drafts, logits, stats, V, R, q_logits, q_stats,
                          n_low + n_high, q_stride, temperature, eos_id, seed, pos_base, out,
                          counters, workspace, workspace_bytes, stream, 0, nullptr, nullptr,
                          n_high > 0 ? n_low : -1, hi_first);
}

spec_status spec_accept(int32_t B, int32_t k_max, const int32_t* k, const int32_t* drafts,
                        const float* logits, const spec_rowstats* stats, int64_t V, int32_t R,
                        const float* q_logits, const spec_rowstats* q_stats, int64_t V_draft,
                        int64_t q_stride, const float* temperature, int32_t eos_id,
                        const uint64_t* seed, const int64_t* pos_base, spec_accept_out* out,
                        spec_counters* counters, void* workspace, size_t workspace_bytes,
                        spec_stream_t stream) {
  return spec::run_accept(B, k_max, k, drafts, logits, stats, V, R, q_logits, q_stats, V_draft,
                          q_stride, temperature, eos_id, seed, pos_base, out, counters, workspace,
                          workspace_bytes, stream, 0);
}

namespace spec {
spec_status run_adapt(int32_t B, int32_t k_max, const spec_accept_out* out,
                      const int32_t* k_used, const float* cost, const float* cycle_cost,
                      float alpha, spec_width_state* state, int32_t* k_next, int32_t* k_mirror,
                      spec_stream_t stream) {
  if (B < 1 || k_max < 0 || k_max > kMaxRows - 1) return SPEC_ERR_INVALID;
  if (!out || !k_used || !cost || !state || !k_next) return SPEC_ERR_INVALID;
  if (!(alpha > 0.f && alpha <= 1.f)) return SPEC_ERR_INVALID;
  AdaptParams p;
  p.B = B;
  p.k_max = k_max;
  p.out = out;
  p.k_used = k_used;
  p.cost = cost;
  p.cycle_cost = cycle_cost;
  p.alpha = alpha;
  p.state = state;
  p.k_next = k_next;
  p.k_mirror = k_mirror;
  const cudaError_t e = adapt_launch(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
}  // namespace spec

spec_status spec_adapt_width(int32_t B, int32_t k_max, const spec_accept_out* out,
                             const int32_t* k_used, const float* cost, const float* cycle_cost,
                             float alpha, spec_width_state* state, int32_t* k_next,
                             spec_stream_t stream) {
  return spec::run_adapt(B, k_max, out, k_used, cost, cycle_cost, alpha, state, k_next, nullptr,
                         stream);
}

spec_status spec_adapt_width_mirror(int32_t B, int32_t k_max, const spec_accept_out* out,
                                    const int32_t* k_used, const float* cost,
                                    const float* cycle_cost, float alpha,
                                    spec_width_state* state, int32_t* k_next, int32_t* k_mirror,
                                    spec_stream_t stream) {
  if (!k_mirror) return SPEC_ERR_INVALID;
  return spec::run_adapt(B, k_max, out, k_used, cost, cycle_cost, alpha, state, k_next, k_mirror,
                         stream);
}

spec_status spec_accept_exact(int32_t B, int32_t k_max, const int32_t* k, const int32_t* drafts,
                              const float* logits, const spec_rowstats* stats, int64_t V,
                              int32_t R, const float* temperature, int32_t eos_id,
                              const uint64_t* seed, const int64_t* pos_base,
                              spec_accept_out* out, spec_counters* counters, void* workspace,
                              size_t workspace_bytes, spec_stream_t stream) {
  return spec::run_accept(B, k_max, k, drafts, logits, stats, V, R, nullptr, nullptr, 0, 0,
                          temperature, eos_id, seed, pos_base, out, counters, workspace,
                          workspace_bytes, stream, 1);
}

spec_status spec_accept_filtered(int32_t B, int32_t k_max, const int32_t* k,
                                 const int32_t* drafts, const float* logits,
                                 const spec_rowstats* stats, int64_t V, int32_t R,
                                 const float* temperature, const int32_t* top_k,
                                 const float* top_p, int32_t eos_id, const uint64_t* seed,
                                 const int64_t* pos_base, spec_accept_out* out,
                                 spec_counters* counters, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream) {
  if (!top_k || !top_p) return SPEC_ERR_INVALID;
  return spec::run_accept(B, k_max, k, drafts, logits, stats, V, R, nullptr, nullptr, 0, 0,
                          temperature, eos_id, seed, pos_base, out, counters, workspace,
                          workspace_bytes, stream, 0, top_k, top_p);
}

spec_status spec_width_graph_create(int32_t n_bodies, const int32_t* k_next, int32_t B,
                                    void** graph, void** bodies) {
  if (n_bodies < 1 || n_bodies > 64 || !k_next || B < 1 || B > 128 || !graph || !bodies)
    return SPEC_ERR_INVALID;
  cudaGraph_t g = nullptr;
  if (cudaGraphCreate(&g, 0) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaGraphConditionalHandle h;
  if (cudaGraphConditionalHandleCreate(&h, g, 0, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return SPEC_ERR_CUDA;
  }
  // node 1: the select kernel (sets the switch from the widths when the graph runs)
  const int32_t* kn = k_next;
  int nb = n_bodies, bb = B;
  void* args[] = {&h, &kn, &bb, &nb};
  cudaKernelNodeParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.func = const_cast<void*>(width_select_function());
  kp.gridDim = dim3(1);
  kp.blockDim = dim3(32);
  kp.kernelParams = args;
  cudaGraphNode_t sel;
  if (cudaGraphAddKernelNode(&sel, g, nullptr, 0, &kp) != cudaSuccess) {
    cudaGraphDestroy(g);
    return SPEC_ERR_CUDA;
  }
  // node 2: the switch over the bodies
  // (the struct's union has no default constructor: zeroed storage instead)
  alignas(cudaGraphNodeParams) unsigned char cp_storage[sizeof(cudaGraphNodeParams)];
  memset(cp_storage, 0, sizeof(cp_storage));
  cudaGraphNodeParams& cp = *reinterpret_cast<cudaGraphNodeParams*>(cp_storage);
  cp.type = cudaGraphNodeTypeConditional;
  cp.conditional.handle = h;
  cp.conditional.type = cudaGraphCondTypeSwitch;
  cp.conditional.size = static_cast<unsigned>(n_bodies);
  cudaGraphNode_t sw;
  if (cudaGraphAddNode(&sw, g, &sel, nullptr, 1, &cp) != cudaSuccess) {
    cudaGraphDestroy(g);
    return SPEC_ERR_CUDA;
  }
  for (int i = 0; i < n_bodies; ++i) bodies[i] = cp.conditional.phGraph_out[i];
  *graph = g;
  return SPEC_OK;
}

spec_status spec_graph_capture_begin(void* body, spec_stream_t stream) {
  if (!body || !stream) return SPEC_ERR_INVALID;  // the legacy stream cannot be captured
  return cudaStreamBeginCaptureToGraph(reinterpret_cast<cudaStream_t>(stream),
                                       static_cast<cudaGraph_t>(body), nullptr, nullptr, 0,
                                       cudaStreamCaptureModeRelaxed) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status spec_graph_capture_end(spec_stream_t stream) {
  if (!stream) return SPEC_ERR_INVALID;
  cudaGraph_t g = nullptr;
  return cudaStreamEndCapture(reinterpret_cast<cudaStream_t>(stream), &g) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status spec_graph_instantiate(void* graph, void** exec) {
  if (!graph || !exec) return SPEC_ERR_INVALID;
  cudaGraphExec_t e = nullptr;
  if (cudaGraphInstantiate(&e, static_cast<cudaGraph_t>(graph), 0) != cudaSuccess)
    return SPEC_ERR_CUDA;
  *exec = e;
  return SPEC_OK;
}

spec_status spec_graph_launch(void* exec, spec_stream_t stream) {
  if (!exec) return SPEC_ERR_INVALID;
  return cudaGraphLaunch(static_cast<cudaGraphExec_t>(exec),
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status spec_graph_destroy(void* graph, void* exec) {
  bool ok = true;
  if (exec) ok = cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(exec)) == cudaSuccess && ok;
  if (graph) ok = cudaGraphDestroy(static_cast<cudaGraph_t>(graph)) == cudaSuccess && ok;
  return ok ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_test_verify_stalled(const void* W, int64_t V, int64_t d, const void* H,
                                     int32_t B, int32_t R, const float* temperature,
                                     float* logits, spec_rowstats* stats, uint32_t wait_limit_us,
                                     void* workspace, size_t workspace_bytes,
                                     spec_stream_t stream) {
  if (!W || !H || !temperature || !stats || !workspace) return SPEC_ERR_INVALID;
  if (V < 1 || V >= (int64_t(1) << 24) || d < 1 || B < 1 || R < 1 || R > kMaxRows ||
      static_cast<int64_t>(B) * R > kMaxRows)
    return SPEC_ERR_INVALID;
  if (wait_limit_us < 1 || wait_limit_us > 1000000) return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(H) || !aligned16(workspace)) return SPEC_ERR_INVALID;
  return run_gemv(W, SPEC_F32, V, d, H, B * R, R, temperature, logits, V, stats, 0, nullptr,
                  nullptr, 0, nullptr, 0, nullptr, workspace, workspace_bytes, B,
                  reinterpret_cast<cudaStream_t>(stream), -1, -1,
                  static_cast<uint64_t>(wait_limit_us) * 1000ull, 1);
}

spec_status spec_commit_rollback(int32_t B, const spec_state_desc* st,
                                 const spec_accept_out* acc, const int32_t* k, int32_t mode,
                                 int32_t* commit_status, spec_stream_t stream) {
  if (B < 1 || !st || !acc || !k) return SPEC_ERR_INVALID;
  if (mode != SPEC_COMMIT_SNAPSHOT && mode != SPEC_COMMIT_REPLAY && mode != SPEC_COMMIT_INDEX)
    return SPEC_ERR_INVALID;
  if (st->n_slots < 2) return SPEC_ERR_INVALID;
  if (st->kv_layers < 0 || st->rec_layers < 0 || st->conv_rows < 0) return SPEC_ERR_INVALID;
  if (st->kv_layers > 0) {
    if (!st->kv || !st->kv_len || st->kv_capacity < 1 || st->kv_row_bytes < 16 ||
        st->kv_row_bytes % 16 != 0 || st->kv_request_stride % 16 != 0 || !aligned16(st->kv))
      return SPEC_ERR_INVALID;
    if (st->kv_request_stride < 2 * st->kv_layers * st->kv_capacity * st->kv_row_bytes &&
        B > 1)
      return SPEC_ERR_INVALID;
  }
  if (st->rec_layers > 0 && mode == SPEC_COMMIT_INDEX) {
    if (!st->live_slot) return SPEC_ERR_INVALID;  // the state itself is not touched
  } else if (st->rec_layers > 0) {
    if (st->rec_heads < 1 || st->rec_dk < 1 || st->rec_dv < 4 || st->rec_dv % 4 != 0)
      return SPEC_ERR_INVALID;
    // the kernels index one request's state in 16-byte vectors with 32-bit integers
    const int64_t rec_vec = static_cast<int64_t>(st->rec_layers) * st->rec_heads * st->rec_dk *
                            st->rec_dv / 4;
    const int64_t conv_vec =
        static_cast<int64_t>(st->rec_layers) * st->conv_rows * st->conv_width / 4;
    if (rec_vec >= (int64_t(1) << 31) || conv_vec >= (int64_t(1) << 31)) return SPEC_ERR_INVALID;
    if (!st->rec_live || !st->rec_slots || !aligned16(st->rec_live) || !aligned16(st->rec_slots))
      return SPEC_ERR_INVALID;
    if (mode == SPEC_COMMIT_REPLAY &&
        (!st->step_a || !st->step_b || !st->step_c || !aligned16(st->step_c)))
      return SPEC_ERR_INVALID;
    if (st->conv_rows > 0) {
      if (st->conv_width < 4 || st->conv_width % 4 != 0 || !st->conv_live || !st->conv_slots ||
          !aligned16(st->conv_live) || !aligned16(st->conv_slots))
        return SPEC_ERR_INVALID;
      if (mode == SPEC_COMMIT_REPLAY && (!st->conv_in || !aligned16(st->conv_in)))
        return SPEC_ERR_INVALID;
    }
  }
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return SPEC_ERR_CUDA;
  CommitParams p;
  memset(&p, 0, sizeof(p));
  p.st = *st;
  p.acc = acc;
  p.k = k;
  p.mode = mode;
  p.commit_status = commit_status;
  // the replay stages a head's step inputs in at most 48 KB of shared memory
  if (mode == SPEC_COMMIT_REPLAY && st->rec_layers > 0 && commit_replay_rows(*st) < 1)
    return SPEC_ERR_UNSUPPORTED;
  // blocks resident per SM: 4 for the copy, 3 for the replay (their launch bounds)
  const int per_sm = (mode == SPEC_COMMIT_SNAPSHOT) ? 4 : 3;
  int per_req = (per_sm * a.sms + B - 1) / B;
  if (st->rec_layers == 0) per_req = 1;
  if (per_req < 1) per_req = 1;
  const cudaError_t e = commit_launch(p, B, per_req, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Allocation-free variant of spec_lmhead_verify. Its scratch (the cross-block ticket, the error
// word and the per-block partial statistics) lives in a fixed device array that every GPU
// loading this library holds until the process exits. Host code must not pass the array's
// name to a kernel: in host code that name is only a stand-in, not a device address. The device
// address is fetched once per device with cudaGetSymbolAddress, with that device current.
// ------------------------------------------------------------------------------------------
namespace spec {
namespace {

constexpr size_t kNoAllocScratchBytes = 128 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (nullptr on failure).
void* noalloc_scratch() {
  static std::atomic<void*> addr[64];  // zero-initialised (static storage)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace
}  // namespace spec

extern "C" size_t spec_noalloc_scratch_bytes(void) { return spec::kNoAllocScratchBytes; }

extern "C" spec_status spec_noalloc_error_word(uint32_t* error_out, spec_stream_t stream) {
  if (!error_out) return SPEC_ERR_INVALID;
  void* scratch = spec::noalloc_scratch();
  if (!scratch) return SPEC_ERR_CUDA;
  // the error word sits at byte offset 4 of the scratch, as in a caller's workspace
  const cudaError_t e = cudaMemcpyAsync(error_out, static_cast<uint8_t*>(scratch) + 4,
                                        sizeof(uint32_t), cudaMemcpyDefault,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" spec_status spec_lmhead_verify_noalloc(const void* W, spec_dtype wdt, int64_t V,
                                                  int64_t d, const void* H, int32_t B, int32_t R,
                                                  const float* temperature, float* logits,
                                                  spec_rowstats* stats, spec_stream_t stream) {
  if (!W || !H || !temperature || !stats) return SPEC_ERR_INVALID;
  if (!known_wdt(wdt)) return SPEC_ERR_INVALID;
  if (V < 1 || V >= (int64_t(1) << 24) || d < 1 || B < 1 || R < 1 || R > kMaxRows)
    return SPEC_ERR_INVALID;
  if (!aligned16(W) || !aligned16(H)) return SPEC_ERR_INVALID;
  if (static_cast<int64_t>(B) * R > kMaxRows) return SPEC_ERR_UNSUPPORTED;
  const DevAttr a = dev_attr();
  if (a.sms <= 0) return SPEC_ERR_CUDA;
  // the fixed scratch must hold the GEMV's part of the workspace layout (header and per-block
  // partials); a batch-1 layout covers it for any B*R <= 8
  if (ws_layout(V, 1, a.sms).sums > kNoAllocScratchBytes) return SPEC_ERR_UNSUPPORTED;
  void* scratch = noalloc_scratch();
  if (!scratch) return SPEC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the ticket and the error word must start at zero (a previous call may have been cut short)
  if (cudaMemsetAsync(scratch, 0, sizeof(WsHeader), s) != cudaSuccess) return SPEC_ERR_CUDA;
  return run_gemv(W, wdt, V, d, H, B * R, R, temperature, logits, V, stats, 0, nullptr, nullptr,
                  0, nullptr, 0, nullptr, scratch, kNoAllocScratchBytes, 0, s);
}
