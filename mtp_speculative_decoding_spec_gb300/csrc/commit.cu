// Commit of the accepted prefix and rollback of the rest, in KV cache and recurrent state,
// entirely on the device.
//
// DS4Server issue #98 "Add Qwen3.8 Flash Next native MTP speculation", section
// "Implementation": capture verification-row recurrent snapshots, trim rejected attention
// rows, commit only accepted rows, keep an ordinary-forward repair fallback. llama.cpp PR
// #28104 ("full checkpoints for MTP rollback", the replay-livelock fix, "keep speculative
// checkpoints on device"): restore the pre-round checkpoint and replay the accepted tokens
// without verifying them again, with checkpoints that never leave the device.
//
// m = n_emit of the request (0 when its acceptance failed) is read from device memory, so no
// host round-trip sits between acceptance and commit. Block 0 of each request trims the KV
// rows [P+m, P+k+1) and moves the length; all blocks stream the recurrent state with 16-byte
// loads and stores (snapshot mode: a copy of slot m; replay mode: slot 0 advanced over rows
// 0..m-1 in registers, one pass over the state whatever m is).
#include "params.cuh"

namespace spec {


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
    const int64_t L = st.rec_layers, H = st.rec_heads, dk = st.rec_dk, dv = st.rec_dv;
    const int64_t elems = L * H * dk * dv;
    float* live = st.rec_live + static_cast<size_t>(b) * elems;
    if (p.mode == SPEC_COMMIT_SNAPSHOT) {
      const float4* src =
          reinterpret_cast<const float4*>(st.rec_slots + (static_cast<size_t>(b) * ns + m) * elems);
      float4* dst = reinterpret_cast<float4*>(live);
      for (int64_t i = gt; i < elems / 4; i += gs) dst[i] = __ldcs(src + i);
    } else {
      const float* slot0 = st.rec_slots + static_cast<size_t>(b) * ns * elems;
      const int64_t rows = ns - 1;
      for (int64_t i = gt; i < elems / 4; i += gs) {
        const int64_t e = i * 4;
        const int64_t j = e % dv;
        const int64_t ii = (e / dv) % dk;
        const int64_t lh = e / (dv * dk);  // layer * H + head
        float4 s = __ldcs(reinterpret_cast<const float4*>(slot0 + e));
        for (int t = 0; t < m; ++t) {
          const int64_t rl = (static_cast<int64_t>(b) * rows + t) * L * H + lh;
          const float a = __ldg(st.step_a + rl);
          const float bb = __ldg(st.step_b + rl * dk + ii);
          const float4 c = __ldg(reinterpret_cast<const float4*>(st.step_c + rl * dv + j));
          s.x = __fadd_rn(__fmul_rn(a, s.x), __fmul_rn(bb, c.x));
          s.y = __fadd_rn(__fmul_rn(a, s.y), __fmul_rn(bb, c.y));
          s.z = __fadd_rn(__fmul_rn(a, s.z), __fmul_rn(bb, c.z));
          s.w = __fadd_rn(__fmul_rn(a, s.w), __fmul_rn(bb, c.w));
        }
        *reinterpret_cast<float4*>(live + e) = s;
      }
    }
  }

  // ---------------- conv rows ----------------
  if (st.rec_layers > 0 && st.conv_rows > 0) {
    const int64_t L = st.rec_layers, C = st.conv_rows, W = st.conv_width;
    const int64_t elems = L * C * W;
    float* live = st.conv_live + static_cast<size_t>(b) * elems;
    if (p.mode == SPEC_COMMIT_SNAPSHOT) {
      const float4* src = reinterpret_cast<const float4*>(
          st.conv_slots + (static_cast<size_t>(b) * ns + m) * elems);
      float4* dst = reinterpret_cast<float4*>(live);
      for (int64_t i = gt; i < elems / 4; i += gs) dst[i] = __ldcs(src + i);
    } else {
      const float* slot0 = st.conv_slots + static_cast<size_t>(b) * ns * elems;
      const int64_t rows = ns - 1;
      for (int64_t i = gt; i < elems / 4; i += gs) {
        const int64_t e = i * 4;
        const int64_t w = e % W;
        const int64_t cr = (e / W) % C;
        const int64_t l = e / (W * C);
        const int64_t srcrow = m + cr;  // row index into (conv rows of slot 0, conv_in rows)
        const float* src;
        if (srcrow < C)
          src = slot0 + (l * C + srcrow) * W + w;
        else
          src = st.conv_in + ((static_cast<int64_t>(b) * rows + (srcrow - C)) * L + l) * W + w;
        *reinterpret_cast<float4*>(live + e) = __ldcs(reinterpret_cast<const float4*>(src));
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
