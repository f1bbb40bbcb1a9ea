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
// loads and stores (snapshot mode: a copy of slot m; replay mode: slot 0 advanced over rows
// 0..m-1 in registers, one pass over the state whatever m is).
#include "params.cuh"

namespace spec {


// Grid-stride copy of n 16-byte vectors with four loads in flight per thread.
__device__ __forceinline__ void copy_vec4(float4* __restrict__ dst, const float4* __restrict__ src,
                                          int64_t n, int64_t gt, int64_t gs) {
  int64_t i = gt;
  for (; i + 3 * gs < n; i += 4 * gs) {
    const float4 a = __ldcs(src + i), b = __ldcs(src + i + gs), c = __ldcs(src + i + 2 * gs),
                 d = __ldcs(src + i + 3 * gs);
    __stcs(dst + i, a);
    __stcs(dst + i + gs, b);
    __stcs(dst + i + 2 * gs, c);
    __stcs(dst + i + 3 * gs, d);
  }
  for (; i < n; i += gs) __stcs(dst + i, __ldcs(src + i));
}

__global__ void __launch_bounds__(256) commit_kernel(const CommitParams p) {
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const spec_state_desc& st = p.st;
  const int ns = st.n_slots;
  const int status = p.acc[b].status;
  const int kk = p.k[b];
  const bool kvalid = kk >= 0 && kk <= ns - 2;
  int m = (status == SPEC_REQ_OK && kvalid) ? p.acc[b].n_emit : 0;
  m = max(0, min(m, kvalid ? kk + 1 : 0));

  // ---------------- KV trim (block 0 of the request) ----------------
  if (blockIdx.x == 0) {
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
        uint4* dst = reinterpret_cast<uint4*>(
            base + (static_cast<size_t>(pl) * cap + lo) * st.kv_row_bytes);
        for (int64_t i = tid; i < nvec; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
      if (tid == 0) st.kv_len[b] = P + m;
    }
    if (tid == 0 && p.commit_status) p.commit_status[b] = cst;
  }

  const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
  const int64_t gs = static_cast<int64_t>(gridDim.x) * blockDim.x;

  // ---------------- recurrent state ----------------
  if (st.rec_layers > 0) {
    const int dv = st.rec_dv, dk = st.rec_dk;
    const int64_t elems = static_cast<int64_t>(st.rec_layers) * st.rec_heads * dk * dv;
    float* live = st.rec_live + static_cast<size_t>(b) * elems;
    if (p.mode == SPEC_COMMIT_SNAPSHOT) {
      copy_vec4(reinterpret_cast<float4*>(live),
                reinterpret_cast<const float4*>(st.rec_slots + (static_cast<size_t>(b) * ns + m) * elems),
                elems / 4, gt, gs);
    } else {
      const float* slot0 = st.rec_slots + static_cast<size_t>(b) * ns * elems;
      const int64_t rows = ns - 1;
      const int64_t LH = static_cast<int64_t>(st.rec_layers) * st.rec_heads;
      const float* A = st.step_a + static_cast<size_t>(b) * rows * LH;
      const float* Bv = st.step_b + static_cast<size_t>(b) * rows * LH * dk;
      const float* Cv = st.step_c + static_cast<size_t>(b) * rows * LH * dv;
      const int per_head = dk * dv;  // < 2^31 for any supported shape
      for (int64_t i = gt; i < elems / 4; i += gs) {
        const int64_t e = i * 4;
        const int64_t lh = e / per_head;  // layer * heads + head
        const int rem = static_cast<int>(e - lh * per_head);
        const int ii = rem / dv, j = rem - ii * dv;
        float4 sv = __ldcs(reinterpret_cast<const float4*>(slot0 + e));
        for (int t = 0; t < m; ++t) {
          const int64_t rl = static_cast<int64_t>(t) * LH + lh;
          const float a = __ldg(A + rl);
          const float bb = __ldg(Bv + rl * dk + ii);
          const float4 c = __ldg(reinterpret_cast<const float4*>(Cv + rl * dv + j));
          sv.x = __fadd_rn(__fmul_rn(a, sv.x), __fmul_rn(bb, c.x));
          sv.y = __fadd_rn(__fmul_rn(a, sv.y), __fmul_rn(bb, c.y));
          sv.z = __fadd_rn(__fmul_rn(a, sv.z), __fmul_rn(bb, c.z));
          sv.w = __fadd_rn(__fmul_rn(a, sv.w), __fmul_rn(bb, c.w));
        }
        __stcs(reinterpret_cast<float4*>(live + e), sv);
      }
    }
  }

  // ---------------- conv rows ----------------
  if (st.rec_layers > 0 && st.conv_rows > 0) {
    const int C = st.conv_rows, W = st.conv_width;
    const int64_t elems = static_cast<int64_t>(st.rec_layers) * C * W;
    float* live = st.conv_live + static_cast<size_t>(b) * elems;
    if (p.mode == SPEC_COMMIT_SNAPSHOT) {
      copy_vec4(reinterpret_cast<float4*>(live),
                reinterpret_cast<const float4*>(st.conv_slots + (static_cast<size_t>(b) * ns + m) * elems),
                elems / 4, gt, gs);
    } else {
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
}

cudaError_t commit_launch(const CommitParams& prm, int B, int blocks_per_request,
                          cudaStream_t stream) {
  dim3 grid(blocks_per_request, B);
  commit_kernel<<<grid, 256, 0, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace spec
