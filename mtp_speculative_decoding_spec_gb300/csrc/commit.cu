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
// loads and stores. Two kernels, one per mode, so that the copy (snapshot mode: slot m) does
// not carry the registers of the replay (slot 0 advanced over rows 0..m-1 in registers, one
// pass over the state whatever m is).
#include "params.cuh"

namespace spec {


// Grid-stride copy of n (< 2^31) 16-byte vectors with eight loads in flight per thread; 32-bit
// indices keep the eight addresses out of 64-bit registers.
__device__ __forceinline__ void copy_vec8(float4* __restrict__ dst, const float4* __restrict__ src,
                                          int n, int gt, int gs) {
  int i = gt;
#pragma unroll 1
  for (; i < n - 7 * gs; i += 8 * gs) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(src + (i + u * gs));
#pragma unroll
    for (int u = 0; u < 8; ++u) __stcs(dst + (i + u * gs), v[u]);
  }
#pragma unroll 1
  for (; i < n; i += gs) __stcs(dst + i, __ldcs(src + i));
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

// Replay mode: live <- slot 0 advanced over rows 0..m-1 (S <- a S + b c^T, every operation
// separately rounded), two state vectors per thread per step for more loads in flight; conv
// rows <- the last rows of (slot-0 conv rows, conv inputs of rows 0..m-1).
__global__ void __launch_bounds__(256, 2) commit_replay_kernel(const __grid_constant__ CommitParams p) {
  pdl_wait();
  const int b = blockIdx.y;
  const spec_state_desc& st = p.st;
  const int ns = st.n_slots;
  int kk;
  bool kvalid;
  const int m = kept_rows(p, b, kk, kvalid);
  if (blockIdx.x == 0) kv_trim(p, b, m, kk, kvalid);
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gs = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (st.rec_layers <= 0) return;
  {
    const int dv = st.rec_dv, dk = st.rec_dk;
    const int64_t elems = static_cast<int64_t>(st.rec_layers) * st.rec_heads * dk * dv;
    float4* live = reinterpret_cast<float4*>(st.rec_live + static_cast<size_t>(b) * elems);
    const float4* slot0 = reinterpret_cast<const float4*>(st.rec_slots + static_cast<size_t>(b) * ns * elems);
    const int rows = ns - 1;
    const int LH = st.rec_layers * st.rec_heads;
    const float* A = st.step_a + static_cast<size_t>(b) * rows * LH;
    const float* Bv = st.step_b + static_cast<size_t>(b) * rows * LH * dk;
    const float* Cv = st.step_c + static_cast<size_t>(b) * rows * LH * dv;
    // 32-bit vector indices (the host checks a request's state is below 2^31 vectors)
    const int n4 = static_cast<int>(elems / 4), dv4 = dv / 4, per_head4 = dk * dv4;
    const int gt4 = blockIdx.x * blockDim.x + threadIdx.x, gs4 = gridDim.x * blockDim.x;
    for (int i0 = gt4; i0 < n4; i0 += 2 * gs4) {
      float4 sv[2];
      int lh[2], ii[2], jj[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = min(i0 + u * gs4, n4 - 1);  // a duplicate of the last vector is harmless
        lh[u] = i / per_head4;                    // layer * heads + head
        const int rem = i - lh[u] * per_head4;
        ii[u] = rem / dv4;
        jj[u] = (rem - ii[u] * dv4) * 4;
        sv[u] = __ldcs(slot0 + i);
      }
      for (int t = 0; t < m; ++t) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t rl = static_cast<int64_t>(t) * LH + lh[u];
          const float a = __ldg(A + rl);
          const float bb = __ldg(Bv + rl * dk + ii[u]);
          const float4 c = __ldg(reinterpret_cast<const float4*>(Cv + rl * dv + jj[u]));
          sv[u].x = __fadd_rn(__fmul_rn(a, sv[u].x), __fmul_rn(bb, c.x));
          sv[u].y = __fadd_rn(__fmul_rn(a, sv[u].y), __fmul_rn(bb, c.y));
          sv[u].z = __fadd_rn(__fmul_rn(a, sv[u].z), __fmul_rn(bb, c.z));
          sv[u].w = __fadd_rn(__fmul_rn(a, sv[u].w), __fmul_rn(bb, c.w));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (i0 + u * gs4 < n4) __stcs(live + i0 + u * gs4, sv[u]);
    }
  }
  if (st.conv_rows > 0) {
    const int C = st.conv_rows, W = st.conv_width;
    const int64_t elems = static_cast<int64_t>(st.rec_layers) * C * W;
    float* live = st.conv_live + static_cast<size_t>(b) * elems;
    const float* slot0 = st.conv_slots + static_cast<size_t>(b) * ns * elems;
    const int64_t rows = ns - 1;
    const int64_t L = st.rec_layers;
    const float* X = st.conv_in + static_cast<size_t>(b) * rows * L * W;
    const int per_layer = C * W;
    for (int64_t i = gt; i < elems / 4; i += gs) {
      const int64_t e = i * 4;
      const int64_t l = e / per_layer;
      const int rem = static_cast<int>(e - l * per_layer);
      const int cr = rem / W, w = rem - cr * W;
      const int srcrow = m + cr;  // row of (conv rows of slot 0, then conv_in rows)
      const float* src = (srcrow < C) ? slot0 + (l * C + srcrow) * W + w
                                      : X + (static_cast<int64_t>(srcrow - C) * L + l) * W + w;
      __stcs(reinterpret_cast<float4*>(live + e), __ldcs(reinterpret_cast<const float4*>(src)));
    }
  }
}

cudaError_t commit_launch(const CommitParams& prm, int B, int blocks_per_request,
                          cudaStream_t stream) {
  dim3 grid(blocks_per_request, B);
  if (prm.mode == SPEC_COMMIT_SNAPSHOT)
    return launch_pdl(commit_snapshot_kernel, grid, dim3(256), 0, stream, prm);
  return launch_pdl(commit_replay_kernel, grid, dim3(256), 0, stream, prm);
}

}  // namespace spec
