// Commit of the accepted prefix and rollback of the rest, in KV cache and recurrent state,
// entirely on the device.
//
// DS4Server issue #98 "Add Qwen3.8 Flash Next native MTP speculation", section
// "Implementation": the recurrent state is snapshotted at every verify row, attention rows of
// rejected tokens are dropped and only the accepted prefix is kept, with re-running the
// ordinary forward as the fallback. llama.cpp PR #28104 (its commits on whole-state
// checkpoints, on a replay that looped forever and on device-resident checkpoints): go back to
// the checkpoint taken before the round and re-apply the accepted tokens without checking them
// a second time, with checkpoints that never leave the device.
//
// m = n_emit of the request (0 when its acceptance failed) is read from device memory, so no
// host round-trip sits between acceptance and commit. Block 0 of each request trims the KV
// rows [P+m, P+k+1) and moves the length; all blocks stream the recurrent state with 16-byte
// loads and stores. Two kernels, one per mode: the copy (snapshot mode: slot m) and the replay
// (slot 0 advanced over rows 0..m-1 in registers, head by head, one pass over the state
// whatever m is). Index mode moves no state: the forward pass keeps the live state in a slot
// (live_slot) and writes each verify row's snapshot into the slots after it, so the commit
// only makes the kept prefix's slot the live one.
#include "params.cuh"

namespace spec {


// Grid-stride copy of n (< 2^31) 16-byte vectors with eight loads in flight per thread, the
// last batch predicated rather than copied one vector at a time (a remainder loop of single
// loads puts up to seven memory latencies in a row on the threads that run it); 32-bit
// indices keep the eight addresses out of 64-bit registers.
__device__ __forceinline__ void copy_vec8(float4* __restrict__ dst, const float4* __restrict__ src,
                                          int n, int gt, int gs) {
#pragma unroll 1
  for (int i = gt; i < n; i += 8 * gs) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i + u * gs < n) v[u] = __ldcs(src + (i + u * gs));
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i + u * gs < n) __stcs(dst + (i + u * gs), v[u]);
  }
}

// KV trim of request b by one block: zero rows [P+m, P+k+1) and set the length to P+m.
__device__ __forceinline__ void kv_trim(const CommitParams& p, int b, int m, int kk, bool kvalid) {
  const spec_state_desc& st = p.st;
  const int tid = threadIdx.x;
  int cst = SPEC_REQ_OK;
  if (st.kv_layers > 0) {
    const int64_t P = st.kv_len[b];
    const int64_t cap = st.kv_capacity;
    int64_t lo = P + m;
    int64_t hi = kvalid ? P + kk + 1 : lo;
    if (hi > cap) cst = SPEC_REQ_KV_OVERFLOW;
    lo = max(static_cast<int64_t>(0), min(lo, cap));
    hi = max(lo, min(hi, cap));
    uint8_t* base = static_cast<uint8_t*>(st.kv) + static_cast<size_t>(b) * st.kv_request_stride;
    const int64_t nvec = (hi - lo) * st.kv_row_bytes / 16;
    const int planes = 2 * st.kv_layers;
    for (int pl = 0; pl < planes; ++pl) {
      uint4* dst =
          reinterpret_cast<uint4*>(base + (static_cast<size_t>(pl) * cap + lo) * st.kv_row_bytes);
      for (int64_t i = tid; i < nvec; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (tid == 0) st.kv_len[b] = P + m;
  }
  if (tid == 0 && p.commit_status) p.commit_status[b] = cst;
}

// m = number of rows the request keeps (0 when its acceptance failed or k is out of range).
__device__ __forceinline__ int kept_rows(const CommitParams& p, int b, int& kk, bool& kvalid) {
  const int ns = p.st.n_slots;
  const int status = p.acc[b].status;
  kk = p.k[b];
  kvalid = kk >= 0 && kk <= ns - 2;
  int m = (status == SPEC_REQ_OK && kvalid) ? p.acc[b].n_emit : 0;
  return max(0, min(m, kvalid ? kk + 1 : 0));
}

// Snapshot mode: live <- slot m, for the recurrent and the conv state. A pure copy: four
// blocks per SM with eight 16-byte loads in flight per thread (128 KB per SM).
__global__ void __launch_bounds__(256, 4) commit_snapshot_kernel(const __grid_constant__ CommitParams p) {
  pdl_wait();
  const int b = blockIdx.y;
  const spec_state_desc& st = p.st;
  const int ns = st.n_slots;
  int kk;
  bool kvalid;
  const int m = kept_rows(p, b, kk, kvalid);
  if (blockIdx.x == 0) kv_trim(p, b, m, kk, kvalid);
  const int gt = blockIdx.x * blockDim.x + threadIdx.x;  // grid and state sizes checked < 2^31
  const int gs = gridDim.x * blockDim.x;
  if (st.rec_layers > 0) {
    const int64_t elems =
        static_cast<int64_t>(st.rec_layers) * st.rec_heads * st.rec_dk * st.rec_dv;
    copy_vec8(reinterpret_cast<float4*>(st.rec_live + static_cast<size_t>(b) * elems),
              reinterpret_cast<const float4*>(st.rec_slots + (static_cast<size_t>(b) * ns + m) * elems),
              static_cast<int>(elems / 4), gt, gs);
    if (st.conv_rows > 0) {
      const int64_t celems = static_cast<int64_t>(st.rec_layers) * st.conv_rows * st.conv_width;
      copy_vec8(reinterpret_cast<float4*>(st.conv_live + static_cast<size_t>(b) * celems),
                reinterpret_cast<const float4*>(st.conv_slots +
                                                (static_cast<size_t>(b) * ns + m) * celems),
                static_cast<int>(celems / 4), gt, gs);
    }
  }
}

// Index mode: one block per request trims the KV rows and moves live_slot[b] by the m kept rows
// (mod n_slots): that slot holds the state snapshot mode would copy into rec_live and conv_live.
__global__ void __launch_bounds__(256) commit_index_kernel(const __grid_constant__ CommitParams p) {
  pdl_wait();
  const int b = blockIdx.x;
  int kk;
  bool kvalid;
  const int m = kept_rows(p, b, kk, kvalid);
  kv_trim(p, b, m, kk, kvalid);  // every thread: it holds a block barrier
  if (threadIdx.x == 0 && p.st.rec_layers > 0) {
    const int ns = p.st.n_slots;
    const int live = p.st.live_slot[b];
    if (live >= 0 && live < ns)
      p.st.live_slot[b] = (live + m) % ns;
    else if (p.commit_status)
      p.commit_status[b] = SPEC_REQ_BAD_K;
  }
}

// Replay mode: live <- slot 0 advanced over rows 0..m-1 (S <- a S + b c^T, every operation
// separately rounded); conv rows <- the last rows of (slot-0 conv rows, conv inputs of rows
// 0..m-1). One block per (layer, head, chunk of 1,024 state vectors): it stages that head's step
// inputs of the kept rows in shared memory (c[0..dv), b[0..dk), a per row, up to `srows` rows
// at once; c first so that a thread reads its four c values as one 16-byte load), then every
// thread advances eight 16-byte state vectors through them: the state is read and written once
// with eight loads in flight, and no step input costs a memory latency per step.
constexpr int kReplayThreads = 128;
constexpr int kReplayVecs = 8;  // state vectors per thread: a chunk is 1,024 vectors

__host__ __device__ inline int replay_row_floats(int dk, int dv) {
  return (dv + dk + 1 + 3) & ~3;  // c[dv], b[dk], a, padded so that every row's c is aligned
}

__global__ void __launch_bounds__(kReplayThreads, 4)
    commit_replay_kernel(const __grid_constant__ CommitParams p, int srows, int chunks_per_head) {
  extern __shared__ __align__(16) float s_step[];  // [srows][replay_row_floats]
  pdl_wait();
  const int b = blockIdx.y;
  const spec_state_desc& st = p.st;
  const int ns = st.n_slots;
  const int tid = threadIdx.x;
  int kk;
  bool kvalid;
  const int m = kept_rows(p, b, kk, kvalid);
  if (blockIdx.x == 0) kv_trim(p, b, m, kk, kvalid);
  if (st.rec_layers <= 0) return;
  const int dv = st.rec_dv, dk = st.rec_dk, dv4 = dv / 4;
  const int LH = st.rec_layers * st.rec_heads;
  const int lh = static_cast<int>(blockIdx.x) / chunks_per_head;  // uniform in the block
  if (lh < LH) {
    const int64_t elems = static_cast<int64_t>(LH) * dk * dv;
    const int ph4 = dk * dv4;  // 16-byte vectors of one head's state
    const int vbase = (static_cast<int>(blockIdx.x) - lh * chunks_per_head) *
                      (kReplayVecs * kReplayThreads);
    float4* lv = reinterpret_cast<float4*>(st.rec_live + static_cast<size_t>(b) * elems) +
                 static_cast<size_t>(lh) * ph4;
    const float4* s0 = reinterpret_cast<const float4*>(st.rec_slots +
                                                       static_cast<size_t>(b) * ns * elems) +
                       static_cast<size_t>(lh) * ph4;
    const int rows = ns - 1;
    const float* A = st.step_a + static_cast<size_t>(b) * rows * LH;
    const float* Bv = st.step_b + static_cast<size_t>(b) * rows * LH * dk;
    const float* Cv = st.step_c + static_cast<size_t>(b) * rows * LH * dv;
    const int SR = replay_row_floats(dk, dv);
    float4 sv[kReplayVecs];
    int brow[kReplayVecs], ccol[kReplayVecs];  // the vector's row i and column group j / 4
#pragma unroll
    for (int u = 0; u < kReplayVecs; ++u) {
      const int vi = vbase + tid + u * kReplayThreads;
      if (vi < ph4) sv[u] = __ldcs(s0 + vi);
      const int vc = min(vi, ph4 - 1);
      brow[u] = vc / dv4;
      ccol[u] = vc - brow[u] * dv4;
    }
    int t0 = 0;
    // rows [t0, t0 + nt) of the kept ones; m is the same in every thread, so every thread
    // passes the barriers the same number of times
    while (t0 < m) {
      const int nt = min(srows, m - t0);
      __syncthreads();  // the previous rows' inputs are no longer read
      // a column r of the staged rows per thread and trip, all nt (<= 8) rows' loads in flight
      // before any store (a load-store loop would wait out a memory latency per element)
      for (int r = tid; r < dv + dk + 1; r += kReplayThreads) {
        float v[kMaxRows];
#pragma unroll
        for (int t = 0; t < kMaxRows; ++t) {
          if (t < nt) {
            const int64_t rl = static_cast<int64_t>(t0 + t) * LH + lh;
            v[t] = (r < dv) ? __ldg(Cv + rl * dv + r)
                            : (r < dv + dk ? __ldg(Bv + rl * dk + (r - dv)) : __ldg(A + rl));
          }
        }
#pragma unroll
        for (int t = 0; t < kMaxRows; ++t)
          if (t < nt) s_step[t * SR + r] = v[t];
      }
      __syncthreads();
      for (int t = 0; t < nt; ++t) {
        const float* in = s_step + t * SR;
        const float a = in[dv + dk];
#pragma unroll
        for (int u = 0; u < kReplayVecs; ++u) {
          const float bb = in[dv + brow[u]];
          const float4 c = reinterpret_cast<const float4*>(in)[ccol[u]];
          sv[u].x = __fadd_rn(__fmul_rn(a, sv[u].x), __fmul_rn(bb, c.x));
          sv[u].y = __fadd_rn(__fmul_rn(a, sv[u].y), __fmul_rn(bb, c.y));
          sv[u].z = __fadd_rn(__fmul_rn(a, sv[u].z), __fmul_rn(bb, c.z));
          sv[u].w = __fadd_rn(__fmul_rn(a, sv[u].w), __fmul_rn(bb, c.w));
        }
      }
      t0 += srows;
    }
#pragma unroll
    for (int u = 0; u < kReplayVecs; ++u) {
      const int vi = vbase + tid + u * kReplayThreads;
      if (vi < ph4) __stcs(lv + vi, sv[u]);
    }
  }
  if (st.conv_rows > 0) {
    const int C = st.conv_rows, W = st.conv_width;
    const int64_t celems = static_cast<int64_t>(st.rec_layers) * C * W;
    float* live = st.conv_live + static_cast<size_t>(b) * celems;
    const float* slot0 = st.conv_slots + static_cast<size_t>(b) * ns * celems;
    const int64_t rows = ns - 1;
    const int64_t L = st.rec_layers;
    const float* X = st.conv_in + static_cast<size_t>(b) * rows * L * W;
    const int per_layer = C * W;
    const int n4 = static_cast<int>(celems / 4);
    const int gt = blockIdx.x * kReplayThreads + tid, gs = gridDim.x * kReplayThreads;
    for (int i0 = gt; i0 < n4; i0 += 8 * gs) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * gs;
        if (i < n4) {
          const int64_t e = static_cast<int64_t>(i) * 4;
          const int64_t l = e / per_layer;
          const int rem = static_cast<int>(e - l * per_layer);
          const int cr = rem / W, w = rem - cr * W;
          const int srcrow = m + cr;  // row of (conv rows of slot 0, then conv_in rows)
          const float* src = (srcrow < C) ? slot0 + (l * C + srcrow) * W + w
                                          : X + (static_cast<int64_t>(srcrow - C) * L + l) * W + w;
          v[u] = __ldcs(reinterpret_cast<const float4*>(src));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * gs < n4) __stcs(reinterpret_cast<float4*>(live) + i0 + u * gs, v[u]);
    }
  }
}

// Rows of step inputs the replay stages in shared memory at once (48 KB at most); 0 when one
// row of a head's inputs does not fit.
int commit_replay_rows(const spec_state_desc& st) {
  const int64_t row_bytes = 4 * static_cast<int64_t>(replay_row_floats(st.rec_dk, st.rec_dv));
  int64_t r = (48 * 1024) / row_bytes;
  if (r > kMaxRows) r = kMaxRows;  // a cycle keeps at most 8 rows
  if (r > st.n_slots - 1) r = st.n_slots - 1;
  return static_cast<int>(r);
}

cudaError_t commit_launch(const CommitParams& prm, int B, int blocks_per_request,
                          cudaStream_t stream) {
  if (prm.mode == SPEC_COMMIT_SNAPSHOT)
    return launch_pdl(commit_snapshot_kernel, dim3(blocks_per_request, B), dim3(256), 0, stream,
                      prm);
  if (prm.mode == SPEC_COMMIT_INDEX)
    return launch_pdl(commit_index_kernel, dim3(B), dim3(256), 0, stream, prm);
  // the replay: one block per (layer, head, chunk of the head's state), at least enough blocks
  // for the conv rows and the KV trim
  const spec_state_desc& st = prm.st;
  int srows = 1, chunks = 1;
  int64_t units = blocks_per_request;
  size_t smem = 0;
  if (st.rec_layers > 0) {
    srows = commit_replay_rows(st);
    const int64_t ph4 = static_cast<int64_t>(st.rec_dk) * (st.rec_dv / 4);
    chunks = static_cast<int>((ph4 + kReplayVecs * kReplayThreads - 1) /
                              (kReplayVecs * kReplayThreads));
    units = static_cast<int64_t>(st.rec_layers) * st.rec_heads * chunks;
    smem = static_cast<size_t>(srows) * 4 * replay_row_floats(st.rec_dk, st.rec_dv);
  }
  if (units < 1) units = 1;
  if (units > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_pdl(commit_replay_kernel, dim3(static_cast<unsigned>(units), B),
                    dim3(kReplayThreads), smem, stream, prm, srows, chunks);
}

}  // namespace spec
