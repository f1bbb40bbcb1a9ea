/*
 * spec.h -- C ABI of libspec.so: the per-cycle verify step of MTP speculative decoding on one
 * GB300 (sm_103a).
 *
 * One decode cycle (lucebox-hub PR #15 "MTP speculative decoding", section "What"): the MTP
 * head proposes up to seven drafts, each picked on the GPU over the first 64,000 vocabulary
 * rows and fed to the next draft from device memory; the trunk verifies the k drafts in one
 * batched pass of k+1 rows through the shared LM head; the accepted prefix is committed and
 * the rest rolled back bit-exactly (section "Exactness"). DS4Server issue #98 ("Add Qwen3.8
 * Flash Next native MTP speculation", section "Implementation") adds the sampled variant: a
 * draft is kept when u*q(x) <= p(x), a rejection is replaced by a draw from max(0, p - q), an
 * EOS among the drafts ends the block, the state is snapshotted per verify row and rejected
 * rows are dropped. llama.cpp PR #28104 moved its speculative checkpoints into device memory to
 * save host copies per token; in the same spirit no call here reads a result back to the host.
 *
 * Conventions for every call
 *   - All array arguments are DEVICE pointers unless stated; the caller owns and allocates
 *     every buffer (weights, activations, outputs, state, workspace). The library allocates
 *     no memory and keeps no state beyond cached device attributes (and the fixed scratch
 *     array that spec_lmhead_verify_noalloc uses in place of a workspace).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Nothing synchronises with the host.
 *   - Host-detectable errors (null required pointer, sizes out of range, misalignment) return
 *     SPEC_ERR_INVALID or SPEC_ERR_UNSUPPORTED before anything is enqueued. A failed launch
 *     returns SPEC_ERR_CUDA. Data-dependent problems never trap: they are written to the
 *     per-request status (spec_accept_out.status) and that request commits nothing.
 *   - Workspace: calls that reduce across thread blocks take a caller-allocated workspace of
 *     at least spec_workspace_bytes() bytes, 256-byte aligned, ZERO-FILLED ONCE before its
 *     first use. Every call leaves it reusable (its counters back at zero). Calls that may run
 *     concurrently (different streams) need separate workspaces. Byte offset 4 of the
 *     workspace holds a 32-bit error word that kernels set (never clear) if an internal
 *     bounded wait gives up; 0 means no error.
 *   - Limits: 1..8 verify rows per request (k = 0..7 drafts), at most 8 rows in total per
 *     spec_lmhead_verify / spec_draft_argmax call on the GEMV path; hidden size d with
 *     d * element_size a multiple of 16 bytes and d <= 3072 (bf16) / 1536 (fp32), or d a
 *     multiple of 128 up to 4096 (SPEC_Q4A32); V < 2^24. The GEMV path's last block combines
 *     every block's partials in shared memory, which bounds V at about 2.4 million rows for
 *     bf16 and fp32 weights; SPEC_Q4A32 keeps at most 1,024 rows per block, so V <= 1,024 x
 *     the device's SM count (155,648 on a 152-SM GB300). Beyond these the calls return
 *     SPEC_ERR_UNSUPPORTED.
 */
#ifndef SPEC_H
#define SPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *spec_stream_t; /* same type as cudaStream_t */

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID = 1,     /* bad argument: nothing enqueued */
  SPEC_ERR_UNSUPPORTED = 2, /* valid but outside what this build implements */
  SPEC_ERR_CUDA = 3         /* a CUDA runtime call or kernel launch failed */
} spec_status;

/*
 * LM-head weight formats. SPEC_BF16 and SPEC_F32: [V, d] row-major. SPEC_Q4A32: 4-bit affine
 * weights in groups of 32 (DS4Server issue #98, closing comment; the byte layout is this
 * library's): each vocabulary row is 5d/8 bytes, d a multiple of 128 and at most 4096. Bytes
 * [0, d/2) hold the codes q in 0..15: the codes of elements 8w..8w+7 (e0..e7) form the
 * little-endian 32-bit word w, e_{2i} in bits 4i..4i+3 and e_{2i+1} in bits 16+4i..16+4i+3.
 * Bytes [d/2, 5d/8) hold, per group g of elements 32g..32g+31, the bf16 scale s_g then the
 * bf16 bias b_g. The weight the projection uses is bf16(s_g * q + b_g), rounded once to nearest
 * even; H rows are bf16. The first V_draft rows of such a matrix are themselves a complete
 * matrix, so the draft head reads the same buffer. The 9..256-row batched path takes bf16 only.
 */
typedef enum { SPEC_BF16 = 0, SPEC_F32 = 1, SPEC_Q4A32 = 2 } spec_dtype;

/* Per-request status written by spec_accept / spec_commit_rollback. */
enum {
  SPEC_REQ_OK = 0,
  SPEC_REQ_NONFINITE = 1,   /* NaN or +Inf in a logit row the decision needs (or a row of -Inf) */
  SPEC_REQ_BAD_K = 2,       /* k outside [0, k_max] or k + 1 > verify rows */
  SPEC_REQ_KV_OVERFLOW = 3, /* commit: P + k + 1 exceeds the KV capacity (trim clipped) */
  SPEC_REQ_NO_LOGITS = 4,   /* temperature > 0 but the needed logits/q_logits were not given */
  SPEC_REQ_BAD_TOKEN = 5,   /* a draft id outside [0, V) */
  SPEC_REQ_BAD_FILTER = 6   /* spec_accept_filtered: top_k outside [1, 32] or top_p outside (0, 1] */
};

/* Statistics of one logit row z[0..V) at the row's temperature T (T <= 0 means greedy and the
 * normaliser is taken at T = 1):
 *   max      = max_v z[v]                              (NaN if any z[v] is NaN or +Inf)
 *   log_norm = log sum_v exp((z[v] - max) / T)
 *   gap      = max - (largest z[v] over v != argmax)   (top-2 gap; +Inf when V == 1)
 *   argmax   = lowest v with z[v] == max
 * The temperature-T distribution is p[v] = exp((z[v] - max) / T - log_norm). */
typedef struct {
  float max;
  float log_norm;
  float gap;
  int32_t argmax;
} spec_rowstats;

/* Result of one cycle for one request (64 bytes). tokens[0..n_emit) are the emitted tokens
 * t_1..t_m; unused entries are -1. sample_kind: 0 no draw, 1 residual draw, 2 bonus draw;
 * sample_row = the verify row the draw used (-1 if none); spec_accept_exact reports kind 3
 * (the trunk's own draws) with the row of the last draw. */
typedef struct {
  int32_t status;
  int32_t n_accept; /* drafts accepted */
  int32_t n_emit;   /* m = tokens emitted; the state keeps exactly m rows */
  int32_t eos_hit;  /* 1 if the last emitted token is the EOS id */
  int32_t tokens[8];
  int32_t sample_kind;
  int32_t sample_row;
  int32_t reserved[2];
} spec_accept_out;

/* Per-request telemetry accumulated by spec_accept (DS4Server issue #98, "Implementation"
 * asks for counts of drafted and accepted tokens, of verify passes, and for how deep the
 * acceptance went). */
typedef struct {
  uint64_t cycles;   /* verify passes */
  uint64_t drafted;  /* sum of k */
  uint64_t accepted; /* sum of n_accept */
  uint64_t emitted;  /* sum of n_emit */
  uint64_t eos;      /* cycles that ended on EOS */
  uint64_t errors;   /* cycles with status != 0 */
  uint64_t depth[8]; /* histogram of n_accept = 0..7 */
} spec_counters;

/* Where the state to commit lives (a HOST struct holding DEVICE pointers). Any part may be
 * absent: kv_layers = 0, rec_layers = 0 or conv_rows = 0 disables it.
 *
 *   KV cache: request b owns the bytes kv + b*kv_request_stride, laid out
 *             [kv_layers][2 (K, V)][kv_capacity][kv_row_bytes]; kv_len[b] = P, the number of
 *             valid positions before this cycle's k+1 verify rows (written at P..P+k).
 *   recurrent:rec_live  [B][rec_layers][rec_heads][rec_dk][rec_dv] float32
 *             rec_slots [B][n_slots][rec_layers][rec_heads][rec_dk][rec_dv] float32;
 *             slot 0 = the state before the cycle, slot r+1 = after verify row r.
 *   conv rows:conv_live [B][rec_layers][conv_rows][conv_width] float32, oldest row first;
 *             conv_slots[B][n_slots][rec_layers][conv_rows][conv_width] float32.
 *   replay inputs (mode SPEC_COMMIT_REPLAY only), per verify row r < n_slots-1:
 *             step_a [B][n_slots-1][rec_layers][rec_heads]         decay
 *             step_b [B][n_slots-1][rec_layers][rec_heads][rec_dk]
 *             step_c [B][n_slots-1][rec_layers][rec_heads][rec_dv]
 *             conv_in[B][n_slots-1][rec_layers][conv_width]         conv input of row r
 *   index mode (SPEC_COMMIT_INDEX only): live_slot [B] int32, the slot of rec_slots (and of
 *             conv_slots) that holds request b's live state; the cycle's verify forward read
 *             it there and wrote the state after verify row r into slot
 *             (live_slot[b] + r + 1) mod n_slots. rec_live and conv_live are not used.
 * n_slots >= k_max + 2. All float arrays 16-byte aligned; rec_dv, conv_width multiples of 4;
 * kv_row_bytes and kv_request_stride multiples of 16; one request's recurrent state
 * (rec_layers*rec_heads*rec_dk*rec_dv) and conv state (rec_layers*conv_rows*conv_width) each
 * below 2^33 floats (SPEC_ERR_INVALID otherwise). */
typedef struct {
  void *kv;
  int64_t kv_request_stride;
  int32_t kv_layers;
  int64_t kv_capacity;
  int64_t kv_row_bytes;
  int64_t *kv_len;
  int32_t rec_layers, rec_heads, rec_dk, rec_dv;
  float *rec_live;
  const float *rec_slots;
  int32_t conv_rows, conv_width;
  float *conv_live;
  const float *conv_slots;
  int32_t n_slots;
  const float *step_a;
  const float *step_b;
  const float *step_c;
  const float *conv_in;
  int32_t *live_slot;
} spec_state_desc;

enum { SPEC_COMMIT_SNAPSHOT = 0, SPEC_COMMIT_REPLAY = 1, SPEC_COMMIT_INDEX = 2 };

/* Workspace bytes needed by any call of this library on the current device for vocabularies
 * up to V rows and up to max_batch requests per call. */
size_t spec_workspace_bytes(int64_t V, int32_t max_batch);

/* Human-readable name of a spec_status. */
const char *spec_status_str(spec_status s);

/*
 * spec_lmhead_verify -- the shared LM head over the verify rows (lucebox-hub PR #15, "What":
 * all drafts are checked by one batched trunk forward; "Exactness": up to eight rows, a row's
 * verify logits may not depend on how many rows are verified together).
 *
 *   W           [V, d] LM-head weights, row-major (vocabulary-major), bf16 or fp32, or V rows
 *               of 4-bit codes and pairs (`wdt`, see spec_dtype).
 *   H           [B*R, d] verify hidden rows, same dtype as W (bf16 for SPEC_Q4A32); row
 *               b*R + r is request b's row r.
 *   temperature [B] float; <= 0 means greedy for that request.
 *   logits      [B*R, V] float32 or NULL. Rows of requests with temperature > 0 receive
 *               z = H W^T; rows of greedy requests are left untouched. NULL = statistics only.
 *   stats       [B*R] spec_rowstats of each row at its request's temperature.
 * B*R <= 8 runs the streaming GEMV (any wdt): there each row's logits and statistics are
 * bitwise independent of how many rows share the call (batch invariance). 9..256 rows run the
 * batched tensor-core GEMM (bf16 weights, d a multiple of 64, spec_batched_supported() == 1,
 * workspace sized for max_batch >= B); it accumulates in another order and is not bitwise
 * equal to the GEMV. Other combinations return SPEC_ERR_UNSUPPORTED.
 *   workspace   spec_workspace_bytes(V, max_batch) bytes (see the conventions above).
 */
spec_status spec_lmhead_verify(const void *W, spec_dtype wdt, int64_t V, int64_t d,
                               const void *H, int32_t B, int32_t R, const float *temperature,
                               float *logits, spec_rowstats *stats, void *workspace,
                               size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_draft_argmax -- draft-head projection over the first V_draft rows of the same LM head
 * with the token choice fused in; the token stays in device memory for the next draft
 * (lucebox-hub PR #15, "What": the draft head spans the first 64,000 vocabulary rows, chooses
 * its token on the GPU and hands it to the next draft without a trip to the host).
 *
 *   W, wdt, d   as for spec_lmhead_verify; only rows [0, V_draft) are read.
 *   h           [B, d] draft hidden rows (one per request), B <= 8.
 *   temperature [B]: <= 0 -> token = argmax (lowest index on ties); > 0 -> token drawn from
 *               softmax(y / T) by inverse CDF with the uniform U(seed[b], pos[b]+pos_offset,
 *               DRAFT) (Philox4x32-10; see spec_accept for the uniform's definition).
 *   seed [B] uint64, pos [B] int64: the request's Philox key and the absolute position the
 *               draft predicts is pos[b] + pos_offset.
 *   token_out   written at token_out[b * token_stride] (int32).
 *   q_logits    [B, q_stride] float32 (row b at q_logits + b*q_stride, first V_draft used) or
 *               NULL; required when any temperature > 0 (a request with T > 0 and no q_logits
 *               gets token -1). q_stats [B] or NULL.
 *   k_active    [B] int32 device array or NULL: this call is draft pos_offset + 1 of the cycle,
 *               and request b needs it only if k_active[b] > pos_offset. When no request needs
 *               it the launch returns at once and writes nothing, so a host can always enqueue
 *               k_max draft steps and let widths chosen on the device (spec_adapt_width) decide
 *               how many do work. Outputs of requests that do not need the step are not used.
 */
spec_status spec_draft_argmax(const void *W, spec_dtype wdt, int64_t V_draft, int64_t d,
                              const void *h, int32_t B, const float *temperature,
                              const uint64_t *seed, const int64_t *pos, int32_t pos_offset,
                              int32_t *token_out, int32_t token_stride, float *q_logits,
                              int64_t q_stride, spec_rowstats *q_stats, const int32_t *k_active,
                              void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_draft_argmax_rows -- spec_draft_argmax over a draft set of two row ranges (lucebox-hub
 * PR #15, "What": the draft head covers the control and special tokens plus the lowest ids).
 * Draft row r (r < n_low + n_high) is vocabulary row r for r < n_low and row
 * hi_first + r - n_low after; the special tokens a tokenizer keeps at the top of the vocabulary
 * form the second range. q_logits/q_stats are in draft-row order (V_draft = n_low + n_high
 * columns); token_out and q_stats.argmax are vocabulary ids. n_high = 0 is spec_draft_argmax.
 * Requires hi_first >= n_low, hi_first + n_high <= the rows of W, and, when n_high > 0, bf16 or
 * SPEC_Q4A32 weights with n_low a multiple of 32 (whole 32-row boxes); else
 * SPEC_ERR_INVALID / SPEC_ERR_UNSUPPORTED. Other arguments as for spec_draft_argmax.
 */
spec_status spec_draft_argmax_rows(const void *W, spec_dtype wdt, int64_t n_low, int64_t hi_first,
                                   int64_t n_high, int64_t d, const void *h, int32_t B,
                                   const float *temperature, const uint64_t *seed,
                                   const int64_t *pos, int32_t pos_offset, int32_t *token_out,
                                   int32_t token_stride, float *q_logits, int64_t q_stride,
                                   spec_rowstats *q_stats, const int32_t *k_active,
                                   void *workspace, size_t workspace_bytes,
                                   spec_stream_t stream);

/*
 * spec_accept -- acceptance, residual correction, bonus token and EOS truncation for B
 * requests (greedy rule: lucebox-hub PR #15, "Exactness"; ratio rule, residual, zero and
 * non-finite handling, EOS: DS4Server issue #98, "Implementation" and closing comment).
 *
 * For request b with k = k[b] drafts d_i = drafts[b*k_max + i-1] (i = 1..k), verify row r at
 * logits/stats row b*R + r (row r predicts position pos_base[b] + r):
 *   T <= 0: accept d_i while d_i == argmax z_{i-1}; the first mismatch emits argmax z_{i-1};
 *           all k accepted emits the bonus argmax z_k.
 *   T  > 0: p_r = softmax(z_r / T); q_i = softmax(y_i / T) over the draft rows, 0 beyond them,
 *           or one-hot at d_i when q_logits is NULL. Accept d_i while p_{i-1}(d_i) > 0 and
 *           u*q_i(d_i) <= p_{i-1}(d_i), u = U(pos_base+i-1, ACCEPT); at the first rejection
 *           emit an inverse-CDF draw from r = max(0, p_{i-1} - q_i) (from p_{i-1} if r sums to
 *           zero) with U(pos_base+i-1, RESIDUAL); all k accepted emits a draw from p_k with
 *           U(pos_base+k, BONUS).
 *   An emitted EOS (eos_id >= 0) ends the block; nothing after it is emitted.
 * Uniforms: U(pos, purpose) = (w0 >> 8) * 2^-24 where w0 is the first word of
 * Philox4x32-10(counter = (pos mod 2^32, pos >> 32, 0, purpose), key = (seed mod 2^32,
 * seed >> 32)) (Salmon et al., SC'11); purposes DRAFT = 1, ACCEPT = 2, RESIDUAL = 3, BONUS = 4.
 * Inverse CDF: the smallest token id whose cumulative weight exceeds u * total, with weights
 * quantised to multiples of 2^-40 and summed exactly in 64-bit integers.
 *
 *   logits [B*R, V] float32: needed for requests with T > 0 (status SPEC_REQ_NO_LOGITS if
 *          NULL); stats [B*R] from spec_lmhead_verify.
 *   q_logits [k_max*B, q_stride] float32, draft-major: draft i of request b at row
 *          (i-1)*B + b (what spec_draft_argmax writes for draft i when given q_logits + (i-1)*B
 *          rows), or NULL; q_stats [k_max*B] alongside it (required when q_logits is given).
 *   out [B]: results. counters [B] or NULL: accumulated telemetry.
 */
spec_status spec_accept(int32_t B, int32_t k_max, const int32_t *k, const int32_t *drafts,
                        const float *logits, const spec_rowstats *stats, int64_t V, int32_t R,
                        const float *q_logits, const spec_rowstats *q_stats, int64_t V_draft,
                        int64_t q_stride, const float *temperature, int32_t eos_id,
                        const uint64_t *seed, const int64_t *pos_base, spec_accept_out *out,
                        spec_counters *counters, void *workspace, size_t workspace_bytes,
                        spec_stream_t stream);

/*
 * spec_accept_rows -- spec_accept with q over the two-range draft set of
 * spec_draft_argmax_rows: q_i(x) is read from draft row x (x < n_low) or n_low + x - hi_first
 * (hi_first <= x < hi_first + n_high), and is zero at every other id, in the ratio test and in
 * the residual max(0, p - q). q_logits rows hold n_low + n_high columns in draft-row order.
 * Requires hi_first >= n_low and hi_first + n_high <= V. n_high = 0 is spec_accept.
 */
spec_status spec_accept_rows(int32_t B, int32_t k_max, const int32_t *k, const int32_t *drafts,
                             const float *logits, const spec_rowstats *stats, int64_t V,
                             int32_t R, const float *q_logits, const spec_rowstats *q_stats,
                             int64_t n_low, int64_t hi_first, int64_t n_high, int64_t q_stride,
                             const float *temperature, int32_t eos_id, const uint64_t *seed,
                             const int64_t *pos_base, spec_accept_out *out,
                             spec_counters *counters, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/*
 * spec_accept_exact -- exact-match acceptance at temperature (lucebox-hub PR #15,
 * "Exactness" and "Notes": a draft counts only if it is the token the trunk itself samples, so
 * the emitted text is the same as decoding without drafts for the same seed).
 *
 * For request b at T > 0 the trunk's token at position pos_base[b] + r is the inverse-CDF draw
 * of p_r = softmax(z_r / T) with U(pos_base + r, BONUS) -- the draw decoding without drafts
 * makes there. For i = 1..k: while d_i equals the trunk's token of row i-1 it is kept (an EOS
 * ends the block); the first mismatch emits the trunk's token and stops; all k kept emits the
 * trunk's token of row k. T <= 0 is greedy acceptance, exactly as spec_accept. No draft logits
 * are read. out[b].sample_kind = 3 for these draws and sample_row = the row of the last one.
 * Arguments, layouts, workspace, status codes and counters as for spec_accept.
 */
spec_status spec_accept_exact(int32_t B, int32_t k_max, const int32_t *k, const int32_t *drafts,
                              const float *logits, const spec_rowstats *stats, int64_t V,
                              int32_t R, const float *temperature, int32_t eos_id,
                              const uint64_t *seed, const int64_t *pos_base,
                              spec_accept_out *out, spec_counters *counters, void *workspace,
                              size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_accept_filtered -- acceptance against a top-k / top-p filtered target (llama.cpp PR
 * #28104, "Result": the trunk samples at temperature 1.0 with top-p 0.95 and top-k 20).
 *
 * For request b at T > 0 the target of verify row r is p'_r: the temperature-T distribution of
 * the row kept to its top_k[b] tokens (largest logits, ties to the lower id), then to the
 * smallest prefix of those, in descending probability, whose mass over the top-k set reaches
 * top_p[b], renormalised. Drafts are taken as the draft head's argmax picks with q one-hot at
 * each draft (run spec_draft_argmax at temperature 0), so: d_i is kept when
 * u <= p'_{i-1}(d_i) with u = U(pos_base + i - 1, ACCEPT); the first rejection emits a draw
 * from p'_{i-1} without d_i (RESIDUAL); all k kept emits a draw from p'_k (BONUS). The emitted
 * tokens then follow the filtered target exactly. Weights are exp((z - max)/T) quantised to
 * 2^-40 units; the ratio test compares u * sum(kept) with the draft's weight exactly, the top-p
 * cut compares the integer mass ahead with top_p times the top-k total, and the draws are
 * inverse CDFs in ascending token id. T <= 0 is greedy acceptance, exactly as spec_accept.
 *   top_k [B] int32 in [1, 32]; top_p [B] float in (0, 1]; otherwise the request gets status
 *   SPEC_REQ_BAD_FILTER. V at most 2^20 (else SPEC_ERR_UNSUPPORTED). No draft logits are read.
 *   Other arguments, layouts, workspace, status codes and counters as for spec_accept
 *   (sample_kind 1 residual, 2 bonus).
 */
spec_status spec_accept_filtered(int32_t B, int32_t k_max, const int32_t *k,
                                 const int32_t *drafts, const float *logits,
                                 const spec_rowstats *stats, int64_t V, int32_t R,
                                 const float *temperature, const int32_t *top_k,
                                 const float *top_p, int32_t eos_id, const uint64_t *seed,
                                 const int64_t *pos_base, spec_accept_out *out,
                                 spec_counters *counters, void *workspace,
                                 size_t workspace_bytes, spec_stream_t stream);

/* Adaptive width state of one request (64 bytes, zero-filled before the first cycle). */
typedef struct {
  float rate[8];    /* rate[d], d = 1..7: moving average of "draft d accepted, given 1..d-1 were";
                       rate[0]: the last usable fitted cost ratio b / a (0 = none yet) */
  uint32_t seen;    /* bit d set once depth d has been observed (until then it is believed to
                       do as well as depth d - 1; depth 1 starts at 0.5); bit 0 once the cost fit
                       holds an observation */
  uint32_t cycles;  /* cycles observed */
  int32_t k;        /* the width chosen for the next cycle */
  uint32_t t_last;  /* %globaltimer / 1024 (ns) at the previous call that timed the cycle itself;
                       0 = none */
  float fit[4];     /* moving averages of k, k^2, cost and k * cost over the observed cycles */
} spec_width_state;

/*
 * spec_adapt_width -- choose each request's next verify width on the device (lucebox-hub PR
 * #15, "What" and "Speed": the default width adapts, following the acceptance seen at each
 * draft depth and a fit of the request's cycle cost; the controller's form is this library's,
 * the pages give none).
 *
 * From request b's result out[b] of a cycle run at width k_used[b]: depths 1..n_accept were
 * accepted, depth n_accept + 1 (if <= k_used and the block did not end at an accepted EOS) was
 * rejected, deeper ones were not observed. Each observed depth moves its rate by
 * alpha * (x - rate) (x = 1 accepted, 0 rejected). A depth not yet observed is believed to do
 * as well as the depth above it (0.5 for depth 1), so widths grow while drafts keep being
 * accepted; a depth observed before but not in this cycle relaxes by the same alpha towards
 * the belief of the depth above it, so a depth that looked poor is tried again.
 * The cycle's cost c (cycle_cost[b], or, when cycle_cost is NULL, the %globaltimer time since
 * this request's previous call, in units of 1,024 ns) joins the request's cost fit c ~ a + b*k:
 * the moving averages (rate alpha; the first observation sets them) of k, k^2, c and k*c give
 * var = E[k^2] - E[k]^2, b = (E[kc] - E[k]E[c]) / var, a = E[c] - b E[k]. The fit is usable
 * when var >= 1/4 and a, b > 0, and its ratio b / a is then kept in rate[0]; a cost above four
 * times the usable fit's a + b*k is not folded in, nor a cost <= 0. A request whose status is
 * not OK keeps its state (t_last still moves). Then, with E(k) = 1 + sum_{j<=k} prod_{i<=j}
 * belief[i] the expected tokens of a cycle at width k and cost(k) = 1 + rate[0] * k once a
 * ratio is kept (the caller's cost[k] before), the next width is the k in [1, k_max] maximising
 * E(k) / cost(k) (the smallest on ties; never 0, so depth 1 stays observed and a request whose
 * drafts start failing can recover), written to k_next[b] and state[b].k.
 *   cost       [k_max + 1] float device array: the prior relative cost of a cycle at each width.
 *   cycle_cost [B] float device array or NULL (measure on the device, see above).
 *   alpha      in (0, 1].  k_used and k_next may be the same array.
 */
spec_status spec_adapt_width(int32_t B, int32_t k_max, const spec_accept_out *out,
                             const int32_t *k_used, const float *cost, const float *cycle_cost,
                             float alpha, spec_width_state *state, int32_t *k_next,
                             spec_stream_t stream);

/*
 * spec_adapt_width_mirror -- spec_adapt_width that also writes each chosen width to
 * k_mirror[b] (int32 [B], any memory the device can write: device memory, or the device alias
 * of pinned host memory from spec_host_alias). No counterpart on the pages: it lets a host
 * learn the widths without a copy on the stream, so that it can enqueue a later cycle at
 * exactly the chosen width (no graph, no idle draft step). The mirror holds the values once
 * the launch has completed (an event recorded after it). k_mirror NULL: SPEC_ERR_INVALID;
 * other arguments and errors as for spec_adapt_width.
 */
spec_status spec_adapt_width_mirror(int32_t B, int32_t k_max, const spec_accept_out *out,
                                    const int32_t *k_used, const float *cost,
                                    const float *cycle_cost, float alpha,
                                    spec_width_state *state, int32_t *k_next, int32_t *k_mirror,
                                    spec_stream_t stream);

/*
 * spec_verify_accept_greedy -- spec_lmhead_verify followed by the greedy acceptance of
 * spec_accept (lucebox-hub PR #15, "Exactness": a draft is kept while it is the verify row's
 * argmax), fused: the LM-head kernel's last block, which combines every row's statistics,
 * also takes each request's decision from them, so the cycle runs one kernel instead of two.
 * Every request is decided by the greedy rule whatever its temperature (the temperature still
 * sets its statistics and logits as in spec_lmhead_verify; use spec_accept for sampled
 * acceptance). out[b], counters[b] (nullable) and the status codes are exactly those
 * spec_accept writes at temperature <= 0 for the same k, drafts [B, k_max] and eos_id; the
 * stats (and logits) are those of spec_lmhead_verify. B*R <= 8 (the GEMV path) and
 * k_max <= 7; otherwise SPEC_ERR_UNSUPPORTED / SPEC_ERR_INVALID. Other arguments as for
 * spec_lmhead_verify and spec_accept.
 * With state non-NULL the width update of spec_adapt_width_mirror follows in the same block,
 * with k_used = k and the arguments cost, cycle_cost, alpha, state, k_next and k_mirror
 * (nullable) as there: state, k_next and k_mirror get the bytes that call writes (a cycle
 * timed on the device, cycle_cost NULL, is timed to this kernel's last block instead of to the
 * width kernel). state NULL: no width update (cost ... k_mirror ignored).
 */
spec_status spec_verify_accept_greedy(const void *W, spec_dtype wdt, int64_t V, int64_t d,
                                      const void *H, int32_t B, int32_t R,
                                      const float *temperature, float *logits,
                                      spec_rowstats *stats, int32_t k_max, const int32_t *k,
                                      const int32_t *drafts, int32_t eos_id,
                                      spec_accept_out *out, spec_counters *counters,
                                      const float *cost, const float *cycle_cost, float alpha,
                                      spec_width_state *state, int32_t *k_next,
                                      int32_t *k_mirror, void *workspace,
                                      size_t workspace_bytes, spec_stream_t stream);

/*
 * Adaptive-width cycles as one CUDA graph (no counterpart on the pages: it lets the width
 * chosen on the device decide how much work a cycle enqueues, with no host round trip and no
 * idle draft steps).
 *
 * spec_width_graph_create builds a graph of two nodes: a select kernel that reads k_next[0..B)
 * (B <= 128; the widths spec_adapt_width writes) when the graph runs and sets a switch to
 * w = max_b k_next[b] clamped to [0, n_bodies - 1], then a CUDA switch node that runs body w.
 * *graph receives the cudaGraph_t; bodies[0..n_bodies) the (empty) body graphs, each to be
 * filled by capturing this library's calls on a stream between spec_graph_capture_begin and
 * spec_graph_capture_end (a body for width w typically holds w draft steps, a verify of w + 1
 * rows, the acceptance, the commit and spec_adapt_width). Then spec_graph_instantiate, and
 * spec_graph_launch once per cycle; spec_graph_destroy releases both. The graph records the
 * device pointers of every captured call: the buffers must stay in place while it is used.
 * Errors: SPEC_ERR_INVALID for bad arguments, SPEC_ERR_CUDA if a CUDA graph call fails.
 */
spec_status spec_width_graph_create(int32_t n_bodies, const int32_t *k_next, int32_t B,
                                    void **graph, void **bodies);
spec_status spec_graph_capture_begin(void *body, spec_stream_t stream);
spec_status spec_graph_capture_end(spec_stream_t stream);
spec_status spec_graph_instantiate(void *graph, void **exec);
spec_status spec_graph_launch(void *exec, spec_stream_t stream);
spec_status spec_graph_destroy(void *graph, void *exec);

/*
 * spec_commit_rollback -- keep the accepted prefix, drop the rest, on the device (DS4Server
 * issue #98, "Implementation": rejected rows are dropped and only the accepted rows of the
 * recurrent state are committed or replayed; llama.cpp PR #28104: go back to a whole-state
 * checkpoint and replay the accepted tokens without checking them again, with the checkpoints
 * in device memory).
 *
 * With m = out[b].n_emit (m = 0 if out[b].status != 0) and P = kv_len[b] read on the device:
 *   KV rows [P+m, P+k[b]+1) are zero-filled (clipped to capacity), kv_len[b] = P + m;
 *   SPEC_COMMIT_SNAPSHOT: rec_live <- rec_slots[m], conv_live <- conv_slots[m];
 *   SPEC_COMMIT_REPLAY:   rec_live <- slot 0 advanced over rows 0..m-1 by
 *                         S = fl32(fl32(a*S) + fl32(b_i*c_j)) per layer and head, each
 *                         operation rounded separately; conv_live <- the last conv_rows rows
 *                         of (conv_slots[0] rows, conv_in rows 0..m-1).
 *   SPEC_COMMIT_INDEX:    live_slot[b] <- (live_slot[b] + m) mod n_slots: the slot that holds
 *                         the state snapshot commit would copy becomes the live one, and no
 *                         state byte moves (this library's form, not the pages': it needs the
 *                         forward pass to read and write the state through live_slot). A
 *                         live_slot[b] outside [0, n_slots) is left as it is, with
 *                         commit_status[b] = SPEC_REQ_BAD_K.
 * The snapshot and replay modes produce identical bytes when the slots were captured with the
 * same step; index mode selects those same bytes in place.
 *   k [B] the cycle's draft counts; commit_status [B] int32 or NULL (SPEC_REQ_KV_OVERFLOW).
 */
spec_status spec_commit_rollback(int32_t B, const spec_state_desc *st,
                                 const spec_accept_out *acc, const int32_t *k, int32_t mode,
                                 int32_t *commit_status, spec_stream_t stream);

/* 1 if this build has the batched tensor-core path for more than 8 verify rows per call. */
int32_t spec_batched_supported(void);

/*
 * Host transfers inside the chain of kernels (no counterpart on the pages: a deployment
 * convenience). A cudaMemcpyAsync between two of this library's kernels ends their programmatic
 * overlap (the second kernel no longer starts in the first one's tail); these two calls move a
 * cycle's inputs and results without one, through pinned host memory that is mapped into the
 * device's address space (cudaHostAlloc / cudaMallocHost memory on a 64-bit system).
 *
 * spec_host_alias -- *dev_ptr = the device address of pinned, mapped host memory host_ptr.
 *   A result pointer of this library's calls (for example spec_accept's `out`) may be such an
 *   alias: the kernel then writes the result straight into host memory, readable after the
 *   stream is synchronised. SPEC_ERR_INVALID if host_ptr is not such memory (pageable memory,
 *   device memory, or NULL). Enqueues nothing.
 *
 * spec_copy_from_host -- copy `bytes` (a multiple of 16, src and dst 16-byte aligned) from
 *   pinned, mapped host memory `src_host` to device memory `dst`, by a kernel on `stream`
 *   launched as a programmatic dependent like the library's other kernels: it reads the host
 *   bytes at once and writes `dst` only after the stream's previous kernel has finished, so a
 *   buffer that kernel reads may be refilled. The host must not change src_host until the
 *   copy has run. SPEC_ERR_INVALID for misalignment, a size that is not a multiple of 16, or a
 *   source that is not pinned mapped host memory; bytes = 0 enqueues nothing.
 */
spec_status spec_host_alias(const void *host_ptr, void **dev_ptr);
spec_status spec_copy_from_host(void *dst, const void *src_host, size_t bytes,
                                spec_stream_t stream);

/*
 * spec_lmhead_verify_noalloc -- spec_lmhead_verify for callers that cannot allocate device
 * memory. (The pages have no counterpart: this is a deployment convenience of this library.)
 *
 * Some callers cannot call cudaMalloc at all: a plugin handed only pre-allocated tensors by a
 * host framework that owns the device memory budget and forbids allocations after start-up, or
 * code that must not risk the implicit device synchronisation an allocation can cause. This
 * entry point takes the same inputs and outputs as spec_lmhead_verify but no workspace: its
 * scratch is a fixed device array of spec_noalloc_scratch_bytes() bytes (128 KiB) compiled into
 * the library, which every GPU that loads the library holds until the process exits. It
 * allocates nothing and calls no allocating routine.
 *
 *   - The first call on a device looks up the array's device address with that device current
 *     (one cudaGetSymbolAddress per device); make that first call before any stream capture.
 *   - Every call shares the one array and clears its counters at the start (an asynchronous
 *     memset on `stream`); calls whose work overlaps on the GPU (different streams, or several
 *     host threads) race on it and must be serialised by the caller.
 *   - A vocabulary whose scratch would exceed the array returns SPEC_ERR_UNSUPPORTED (at 152
 *     SMs that is beyond about 1,040,000 vocabulary rows); everything else validates and fails
 *     like spec_lmhead_verify (more than 8 rows in total: SPEC_ERR_UNSUPPORTED).
 */
spec_status spec_lmhead_verify_noalloc(const void *W, spec_dtype wdt, int64_t V, int64_t d,
                                       const void *H, int32_t B, int32_t R,
                                       const float *temperature, float *logits,
                                       spec_rowstats *stats, spec_stream_t stream);

/* Size of the fixed scratch array used by spec_lmhead_verify_noalloc. */
size_t spec_noalloc_scratch_bytes(void);

/*
 * spec_noalloc_error_word -- the error word of spec_lmhead_verify_noalloc's fixed scratch
 * array: the bits its kernels set if an internal bounded wait gave up (0 = no error; the same
 * bits as byte offset 4 of a caller's workspace). Enqueues on `stream` a 4-byte copy of the word
 * into *error_out, which may be device or host memory (pinned host memory keeps the copy
 * asynchronous). Each spec_lmhead_verify_noalloc call clears the word when it starts, so read
 * it after the call and before the next one on the same device; a call whose word is non-zero
 * returned SPEC_OK but its statistics and logits are not to be used. Allocates nothing.
 */
spec_status spec_noalloc_error_word(uint32_t *error_out, spec_stream_t stream);

/*
 * spec_test_verify_stalled -- failure-detection test of the bounded waits (no counterpart on
 * the pages; not part of the method). Runs the fp32 verify LM head (the CUDA-core kernel, which
 * holds no tensor memory) with its producer warp issuing no copy at all, so every consumer's
 * wait for the first stage runs out after wait_limit_us microseconds (1..1,000,000). Each block
 * then sets bit 0 of the workspace error word, skips the rest of its stream and finishes;
 * nothing is in flight when the kernel exits, the workspace counters are back at zero and the
 * statistics written are meaningless. Arguments as spec_lmhead_verify with wdt = SPEC_F32 and
 * at most 8 rows in total; the call itself returns SPEC_OK.
 */
spec_status spec_test_verify_stalled(const void *W, int64_t V, int64_t d, const void *H,
                                     int32_t B, int32_t R, const float *temperature,
                                     float *logits, spec_rowstats *stats, uint32_t wait_limit_us,
                                     void *workspace, size_t workspace_bytes,
                                     spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_H */
