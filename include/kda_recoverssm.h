/*
 * kda_recoverssm.h -- C ABI of libkda_recoverssm.so, the GB300 (sm_103a)
 * KDA RecoverSSM step of speculative decoding: replay the accepted tokens of
 * the previous window into the checkpoint state, verify this window's draft
 * tokens in chunked (WY) form, write the checkpoint back at most once and
 * store the new records.
 *
 * Sources (page titles of the vLLM kimi_k3 documentation):
 *  - "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.fused"
 *    (module docstring: deferred RecoverSSM steps 1-3, precision and layout
 *    notes; class KdaFused and its decay / quad_sum helpers);
 *  - "vllm.models.kimi_k3.nvidia.recoverssm.cutedsl.commit" (module
 *    docstring: the closed-form commit and the align boundary state; class
 *    KdaCommit: its argument list);
 *  - "vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.kernels"
 *    (kda_recoverssm_verify and its argument checks; _defer_commit_kernel;
 *    _prepare_flush_plan_kernel).
 *
 * Conventions shared by every entry point
 *  - K = V = 128 (key and value channels per head).  Other sizes return
 *    KDA_ERR_UNSUPPORTED.
 *  - Every pointer is DEVICE memory owned by the caller (the one exception:
 *    the per-layer address and stride arrays of kda_replay_verify_layers
 *    are host arrays, read during the call).  The library never
 *    allocates or frees, and only kda_check_status synchronises (with its
 *    own stream); every other call enqueues its kernels on `stream` (a
 *    cudaStream_t passed as void*, NULL = the legacy default stream) and
 *    returns at once.
 *  - BF16 tensors are passed as raw bit patterns (kda_bf16, uint16_t).
 *  - Activations are token-major, [n_tokens, H, 128].  Without
 *    query_start_loc, token b*Q + t is token t of request b's window and
 *    n_tokens = B*Q.  With query_start_loc ([B + 1] int32, the stock
 *    wrapper's argument), request b's window is tokens query_start_loc[b]
 *    .. query_start_loc[b + 1] - 1, of length q_b <= Q, and n_tokens <= B*Q
 *    (its activation-capacity check).  A request whose window does not lie
 *    in 0 .. n_tokens or is longer than Q is reported as KDA_ERR_ARG in the
 *    status word and nothing of it is read or written.  Only a window's q_b
 *    tokens are verified and only their outputs and records are written;
 *    the replay of pending tokens does not depend on the window.
 *  - A state slot is inert when slot <= null_slot (the pages use 0).  A
 *    record row < 0 means the request has none.
 *  - Live slots, destinations, boundary slots and record rows must be
 *    pairwise distinct across the requests of one call (the pages leave
 *    duplicates undefined).
 *  - `status` (nullable) is a device int32.  The caller sets it to 0; a
 *    kernel that meets an index outside its pool (slot >= n_slots, row >=
 *    n_rows), a misaligned per-layer address or a device wait that gave up
 *    writes the first such error code there (KDA_ERR_ARG, KDA_ERR_ALIGN,
 *    KDA_ERR_TIMEOUT) and skips the offending item instead of faulting.
 *  - Host-side checks return before anything is launched:
 *      KDA_ERR_ARG          a required pointer is NULL, or a size / count /
 *                           window / split is out of range;
 *      KDA_ERR_ALIGN        a pointer is not 16-byte aligned, or a slot /
 *                           row stride is not a multiple of 16 bytes;
 *      KDA_ERR_UNSUPPORTED  unknown state dtype, or K / V != 128;
 *      KDA_ERR_CUDA         the launch itself failed.
 *  - B == 0 is a no-op that returns KDA_OK whatever the other arguments;
 *    so is n_tokens == 0 once the arguments pass the checks (the stock
 *    wrapper returns early on zero tokens).
 */
#ifndef KDA_RECOVERSSM_H
#define KDA_RECOVERSSM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_OK 0
#define KDA_ERR_ARG (-1)
#define KDA_ERR_ALIGN (-2)
#define KDA_ERR_UNSUPPORTED (-3)
#define KDA_ERR_CUDA (-4)
#define KDA_ERR_TIMEOUT (-5)
#define KDA_ERR_SCRATCH (-6)

#define KDA_STATE_F32 0
#define KDA_STATE_BF16 1

#define KDA_HEAD_DIM 128
#define KDA_MAX_WINDOW 8
#define KDA_MAX_LAYERS 64

typedef uint16_t kda_bf16;

/* Version of this ABI (bumped on any signature change). */
int kda_abi_version(void);

/* A static, human-readable name for a status code. */
const char *kda_error_string(int status);

/*
 * kda_check_status -- reads back a device status word (the `status`
 * argument of the other calls).  Enqueues a 4-byte device-to-host copy of
 * *status on `stream`, waits for that stream, and returns the code it held
 * (KDA_OK when no kernel reported a problem).  Unlike every other entry
 * point it synchronises, with `stream` only; it allocates nothing and does
 * not reset the word.  Returns KDA_ERR_ARG for a NULL status and
 * KDA_ERR_CUDA if the copy or the wait fails (for instance after an earlier
 * fault on the stream).
 */
int kda_check_status(const int32_t *status, void *stream);

/*
 * kda_verify -- the stock RecoverSSM verify of one window, from the
 * checkpoint; the checkpoint is only read (page
 * "vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.kernels",
 * kda_recoverssm_verify docstring).
 *
 * Per (request b, head h) with slot = state_slots[b] > null_slot and
 * S = state_pool[slot, h] ([V=128 rows, K=128 columns]), for t < Q:
 *   d_t  = exp(lower_bound * sigmoid(exp(A_log[h]) * (raw_g_t + dt_bias[h])))
 *   kn_t = k_t * rsqrt(sum k_t^2 + 1e-6)
 *   qn_t = q_t * rsqrt(sum q_t^2 + 1e-6) * q_scale
 *   S <- S diag(d_t); u_t = sigmoid(raw_beta_t) (v_t - S kn_t);
 *   S <- S + u_t kn_t^T; o_t = S qn_t
 * computed in the equivalent chunked form of the "kda.fused" page (step 2):
 * the state is only read.  (With query_start_loc, t < q_b and token
 * query_start_loc[b] + t replace t < Q and token b*Q + t.)  Writes
 * out[b*Q + t, h, :] = BF16(o_t) and, when
 * the record row r (record_rows[b], or b when record_rows is NULL) is >= 0,
 * corr[r, h, t, :] = u_t (FP32), key_gate[r, h, t, 0:128] = k_t and
 * key_gate[r, h, t, 128:256] = raw_g_t (BF16 copies).  Inert requests
 * write zeros to `out` only.
 *
 *   q, k, raw_g   [n_tokens, H, 128] BF16;  v [n_tokens, H, 128] BF16
 *   raw_beta      [n_tokens, H] BF16
 *   query_start_loc [B + 1] int32 or NULL (see the conventions above)
 *   A_log [H] FP32; dt_bias [H, 128] FP32
 *   state_pool    [n_slots, H, 128, 128] of state_dtype, slot stride
 *                 `slot_stride` elements (>= H*128*128)
 *   state_slots   [B] int32; record_rows [B] int32 or NULL
 *   corr          [n_rows, H, rq, 128] FP32, row stride corr_row_stride
 *   key_gate      [n_rows, H, rq, 256] BF16, row stride kg_row_stride
 *   out           [n_tokens, H, 128] BF16
 *   1 <= Q <= rq <= 8; H >= 1; -10 <= lower_bound <= 10 (a bounded gate:
 *   the chunked form divides by prod_{r<=t} d_r, which must stay inside
 *   FP32; KDA_ERR_UNSUPPORTED otherwise).
 */
int kda_verify(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
               const kda_bf16 *raw_g, const kda_bf16 *raw_beta,
               const float *A_log, const float *dt_bias, float lower_bound,
               float q_scale, const void *state_pool, int state_dtype,
               int64_t slot_stride, int n_slots, const int32_t *state_slots,
               const int32_t *query_start_loc, int n_tokens,
               const int32_t *record_rows, float *corr, kda_bf16 *key_gate,
               int64_t corr_row_stride, int64_t kg_row_stride, int n_rows,
               int rq, kda_bf16 *out, int B, int H, int Q, int null_slot,
               int32_t *status, void *stream);

/*
 * kda_replay_verify -- the fused deferred RecoverSSM step ("kda.fused" page,
 * module docstring steps 1-3; class KdaFused).  Per (request b, head h) with
 * slot = state_slots[b] > null_slot, r = record_rows[b] and
 * n = r >= 0 ? clamp(pending[r], 0, rq) : 0:
 *  1. S_n = S_0 diag(D_n) + sum_{t<n} u_t (kn_t * P_t)^T from the request's
 *     records (u_t = corr[r, h, t, :], kn_t the normalised recorded key,
 *     d_t the decay of the recorded raw gate, D_n = prod_{s<n} d_s,
 *     P_t = prod_{t<s<n} d_s), written back to state_pool[slot, h] iff n > 0;
 *     with boundary_slots given and m = boundary_lens[b] > 0,
 *     boundary_slots[b] > null_slot and n > 0, S_min(m, n) is also written
 *     to state_pool[boundary_slots[b], h] (the commit page's align state);
 *  2. the chunked verify of this window from S_n, exactly as kda_verify;
 *  3. the new records, after every old record of the item has been read.
 * `pending` is only read (the defer step after sampling writes it).
 * `state_pool` is FP32.  split = 0 picks the launch shape; 1 is one
 * persistent CTA per SM streaming whole items; 2 or 4 splits each item's
 * rows across a thread-block cluster of that many CTAs (for small batches),
 * whose key-norm and pair-product partial sums are exchanged through
 * distributed shared memory.
 */
int kda_replay_verify(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                      const kda_bf16 *raw_g, const kda_bf16 *raw_beta,
                      const float *A_log, const float *dt_bias,
                      float lower_bound, float q_scale, float *state_pool,
                      int64_t slot_stride, int n_slots,
                      const int32_t *state_slots,
                      const int32_t *query_start_loc, int n_tokens,
                      const int32_t *record_rows,
                      const int32_t *pending, float *corr, kda_bf16 *key_gate,
                      int64_t corr_row_stride, int64_t kg_row_stride,
                      int n_rows, int rq, const int32_t *boundary_slots,
                      const int32_t *boundary_lens, kda_bf16 *out, int B,
                      int H, int Q, int null_slot, int split, int32_t *status,
                      void *stream);

/*
 * kda_replay_verify_layers -- kda_replay_verify over L layers in one launch
 * (persistent CTAs over the (layer, request, head) items, layer-major),
 * with per-layer base addresses and strides as the commit page's KdaCommit
 * takes them (its argument list: per-layer state / correction / key-gate
 * bases and their slot / row strides).  Layer l computes exactly what
 * kda_replay_verify computes on layer l's operands; the layers share the
 * index arrays, as the layers of one model share a request's slot, record
 * row and accepted count:
 *
 *   q, k, v, raw_g  [L, B*Q, H, 128] BF16, layer-stacked (layer l at
 *                   l*B*Q*H*128 elements); raw_beta [L, B*Q, H] BF16
 *   A_log [L, H]; dt_bias [L, H, 128] FP32
 *   state_pools, corrs, key_gates  HOST arrays [L] of DEVICE addresses:
 *                   layer l's FP32 pool [n_slots, H, 128, 128], corrections
 *                   [n_rows, H, rq, 128] FP32 and key/gate records
 *                   [n_rows, H, rq, 256] BF16, each 16-byte aligned
 *   slot_strides, corr_row_strides, kg_row_strides  HOST arrays [L] of
 *                   element strides (at least one slot's / row's extent,
 *                   multiples of 16 bytes)
 *   state_slots, record_rows [B], pending [n_rows] int32, device, shared
 *   out             [L, B*Q, H, 128] BF16, layer-stacked
 *   1 <= L <= KDA_MAX_LAYERS; 1 <= Q <= rq <= 8; uniform windows (b*Q + t);
 *   no boundary states; -10 <= lower_bound <= 10.
 * The host arrays are read during the call and their values become kernel
 * parameters (so a captured launch keeps them); everything else is as in
 * kda_replay_verify with split = 1.  Bad host values return KDA_ERR_ARG /
 * KDA_ERR_ALIGN before any launch; device-side index errors go to status.
 */
int kda_replay_verify_layers(const kda_bf16 *q, const kda_bf16 *k,
                             const kda_bf16 *v, const kda_bf16 *raw_g,
                             const kda_bf16 *raw_beta, const float *A_log,
                             const float *dt_bias, float lower_bound,
                             float q_scale, float *const *state_pools,
                             const int64_t *slot_strides, int n_slots,
                             const int32_t *state_slots,
                             const int32_t *record_rows,
                             const int32_t *pending, float *const *corrs,
                             kda_bf16 *const *key_gates,
                             const int64_t *corr_row_strides,
                             const int64_t *kg_row_strides, int n_rows,
                             int rq, kda_bf16 *out, int L, int B, int H,
                             int Q, int null_slot, int32_t *status,
                             void *stream);

/*
 * kda_commit -- the standalone closed-form commit over L layers (commit
 * page; KdaCommit argument list).  Per (layer l, request b, head h) with
 * n = min(commit_lens[b], Q), src = sources[b], dst = destinations[b],
 * r = record_rows[b] (or b when record_rows is NULL) and
 * live = n > 0 && src > null_slot && dst > null_slot && r >= 0:
 *   dst page <- S_n of the src page replayed from record row r (as in
 *   kda_replay_verify step 1), rounded once to the state dtype;
 *   with boundaries given, m = min(boundary_lens[b], Q) > 0 and
 *   boundaries[b] > null_slot: boundary page <- S_min(m, n).
 * Nothing is written for a request that is not live.  dst == src commits in
 * place.
 *
 *   state_ptrs, corr_ptrs, kg_ptrs  [L] device tables of device addresses
 *                 (uint64) of layer l's state pool [slots, H, 128, 128],
 *                 corrections [rows, H, Q, 128] FP32 and key/gate records
 *                 [rows, H, Q, 256] BF16; each address 16-byte aligned
 *   state_strides, corr_strides, kg_strides  [L] device int64 tables:
 *                 elements per slot / per record row, multiples of 16
 *                 bytes and at least one slot's / row's extent:
 *                 state >= H*128*128, corr >= H*Q*128, key/gate >= H*Q*256
 *   A_log [L, H], dt_bias [L, H, 128] FP32
 *   sources, commit_lens, destinations [B] int32
 *   boundaries, boundary_lens [B] int32 or both NULL (align off)
 *   record_rows [B] int32 or NULL
 *   state_dtype KDA_STATE_BF16 or KDA_STATE_F32; 1 <= Q <= 8;
 *   -10 <= lower_bound <= 10 (the boundary state divides by a product of
 *   up to Q decays, which must stay inside FP32; KDA_ERR_UNSUPPORTED
 *   otherwise).
 * The per-layer tables are device data, so they are checked by the kernel:
 * a layer whose address or stride is misaligned (KDA_ERR_ALIGN) or whose
 * stride is below the minimum or negative (KDA_ERR_ARG) is reported in
 * status and its items are skipped, never written.
 */
int kda_commit(const uint64_t *state_ptrs, const uint64_t *corr_ptrs,
               const uint64_t *kg_ptrs, const int64_t *state_strides,
               const int64_t *corr_strides, const int64_t *kg_strides,
               const float *A_log, const float *dt_bias,
               const int32_t *sources, const int32_t *commit_lens,
               const int32_t *destinations, const int32_t *boundaries,
               const int32_t *boundary_lens, const int32_t *record_rows,
               int state_dtype, float lower_bound, int null_slot, int L, int H,
               int B, int Q, int n_slots, int n_rows, int32_t *status,
               void *stream);

/*
 * kda_defer_commit -- after sampling, per request b (_defer_commit_kernel):
 * if record_rows[b] < 0 or state_slots[b] <= null_slot nothing changes;
 * else if eager && eager[b] != 0: pending[record_rows[b]] = 0 and the
 * commit length is kept (the row is committed now); otherwise
 * pending[record_rows[b]] = commit_lens[b] and commit_lens[b] = 0.
 * eager [B] uint8 or NULL.  Record rows >= n_rows are reported in status
 * and skipped.
 */
int kda_defer_commit(const int32_t *state_slots, int32_t *commit_lens,
                     const int32_t *record_rows, int32_t *pending,
                     const uint8_t *eager, int B, int null_slot, int n_rows,
                     int32_t *status, void *stream);

/*
 * kda_flush_plan -- the in-place commit plan of the pending replays
 * (_prepare_flush_plan_kernel), per request b:
 *   len = record_rows[b] >= 0 ? pending[record_rows[b]] : 0, clamped to
 *   [0, Q]; commit_lens[b] = (state_slots[b] > null_slot && len > 0) ? len
 *   : 0; final_slots[b] = state_slots[b]; boundary_slots[b] = null_slot;
 *   boundary_lens[b] = 0.
 * `pending` is only read.
 */
int kda_flush_plan(const int32_t *state_slots, const int32_t *record_rows,
                   const int32_t *pending, int32_t *commit_lens,
                   int32_t *final_slots, int32_t *boundary_slots,
                   int32_t *boundary_lens, int B, int Q, int null_slot,
                   int n_rows, int32_t *status, void *stream);

/*
 * kda_selftest_wait_timeout -- failure-detection self-test.  Launches one
 * small kernel whose bounded wait on a barrier that nothing completes runs
 * out after the library's fixed wait limit (about 2 s); the kernel then
 * writes KDA_ERR_TIMEOUT to *status (device int32, set to 0 by the caller)
 * and returns, leaving the context usable -- the same path every device
 * wait of the step and commit kernels takes when a copy or a hand-off never
 * arrives.  Returns KDA_ERR_ARG for a NULL status, KDA_ERR_CUDA if the
 * launch fails.
 */
int kda_selftest_wait_timeout(int32_t *status, void *stream);

/*
 * kda_layer_prologue -- the model layer's operands for the step ("kda.fused"
 * page, KdaFused.kernel: the convolution operands, convolution and SiLU,
 * gate projection, the window written last).  Per (request b, head h) with
 * slot = state_slots[b] > null_slot, r = record_rows[b] (or b when NULL) and
 * n = (pending && r >= 0) ? clamp(pending[r], 0, rq) : 0, for each channel
 * ch = part*D + h*128 + c of q (part 0), k (1) and v (2), D = H*128:
 *   s = [W[off], W[off+1], W[off+2], x_0 .. x_{Q-1}], W = conv_state[slot, ch],
 *       off = n - 1 when n > 0 else 0, x_t = x[b*Q + t, ch];
 *   out_t = BF16(silu(bias[ch] + sum_{i<4} conv_weight[part, i, h*128 + c] *
 *           s[t + i])), silu(z) = z / (1 + e^-z), written to q / k / v
 *           [b*Q + t, h, c];
 *   raw_g[b*Q + t, h, f] = BF16(sum_j f_b[h*128 + f, j] * f_a[b*Q + t, j]);
 *   W <- [W[off+1], W[off+2], x_0 .. x_{Q-1}] (entries from 2 + Q kept).
 * Inert requests are skipped (nothing read or written; the step writes
 * their zero outputs); a slot >= n_slots is reported as KDA_ERR_ARG in
 * status and skipped.  The sums run in FP32 (the convolution in tap order,
 * the projection on the tensor cores, in their order) and round once to
 * BF16.
 *
 *   x             [B*Q, 3*D] BF16 (q | k | v channels before the convolution)
 *   conv_weight   [3, 4, D] BF16 (tap 3 multiplies the current token)
 *   conv_bias     [3*D] BF16 or NULL
 *   conv_state    [n_slots, 3*D, rq + 2] BF16, slot stride conv_slot_stride
 *                 elements (>= 3*D*(rq+2), a multiple of 8); 16-byte
 *                 aligned; read and rewritten
 *   f_a           [B*Q, 128] BF16;  f_b [D, 128] BF16, 16-byte aligned
 *   q, k, v, raw_g  [B*Q, H, 128] BF16 outputs (the step's inputs), 16-byte
 *                 aligned
 *   pending       [n_rows] int32 or NULL (no replay pending: off = 0)
 *   1 <= Q <= rq <= 8.
 */
int kda_layer_prologue(const kda_bf16 *x, const kda_bf16 *conv_weight,
                       const kda_bf16 *conv_bias, kda_bf16 *conv_state,
                       int64_t conv_slot_stride, const kda_bf16 *f_a,
                       const kda_bf16 *f_b, const int32_t *state_slots,
                       const int32_t *record_rows, const int32_t *pending,
                       int n_slots, int n_rows, int rq, kda_bf16 *q, kda_bf16 *k,
                       kda_bf16 *v, kda_bf16 *raw_g, int B, int H, int Q,
                       int null_slot, int32_t *status, void *stream);

/*
 * kda_layer_epilogue -- the gated RMSNorm of the step's outputs ("kda.fused"
 * page, the kernel's end).  For every token t and head h, over the 128
 * value rows r of o[t, h, :] (the step's BF16 outputs):
 *   out[t, h*128 + r] = BF16(o * rsqrt(sum_r o^2 / 128 + eps) * norm_weight[r]
 *                            * sigmoid(gate[t, h*128 + r]))
 * in FP32.  o [n_tokens, H, 128] BF16; gate, out [n_tokens, H*128] BF16;
 * norm_weight [128] FP32; eps >= 0.  All four pointers 16-byte aligned.
 */
int kda_layer_epilogue(const kda_bf16 *o, const kda_bf16 *gate,
                       const float *norm_weight, float eps, kda_bf16 *out,
                       int n_tokens, int H, void *stream);

/*
 * kda_layer_step_workspace_bytes -- the workspace kda_layer_step needs for
 * B requests, H heads and windows of Q tokens: the step's operands q, k, v
 * and raw_g, 4 * B*Q * H * 128 BF16 values.  -1 for sizes out of range.
 */
int64_t kda_layer_step_workspace_bytes(int B, int H, int Q);

/*
 * kda_layer_step -- one model-layer step of the KDA RecoverSSM ("kda.fused"
 * page, KdaFused.kernel: the convolution operands, convolution and SiLU,
 * gate projection, the recurrence, and the gated RMSNorm at the kernel's
 * end).  Computes what kda_layer_prologue, kda_replay_verify and
 * kda_layer_epilogue compute one after the other, in two launches: the
 * prologue writes the step's q, k, v, raw_g into `workspace`, and the step
 * kernel folds the gated RMSNorm into its row solve, so the recurrence
 * outputs o never leave the chip:
 *   out[t, h*128 + r] = BF16(o * rsqrt(sum_r o^2 / 128 + eps) *
 *                            norm_weight[r] * sigmoid(gate[t, h*128 + r]))
 * with o the BF16-rounded recurrence output of token t, head h, row r.
 *   x, conv_weight, conv_bias, conv_state, conv_slot_stride, f_a, f_b  as in
 *                 kda_layer_prologue (the window is rolled by the pending
 *                 count and rewritten)
 *   raw_beta, A_log, dt_bias, lower_bound, q_scale, state_pool,
 *   slot_stride, n_slots, state_slots, record_rows, pending, corr,
 *   key_gate, corr_row_stride, kg_row_stride, n_rows, rq  as in
 *                 kda_replay_verify (uniform windows, no boundary states;
 *                 records and pending required)
 *   gate [B*Q, H*128] BF16; norm_weight [128] FP32; eps >= 0
 *   out  [B*Q, H*128] BF16 (inert requests: zeros)
 *   workspace  device, 16-byte aligned, at least
 *              kda_layer_step_workspace_bytes(B, H, Q) bytes, owned by the
 *              caller; its contents are overwritten (after the call it holds
 *              the step's q, k, v, raw_g, [B*Q, H, 128] BF16 each, in that
 *              order)
 * Returns KDA_ERR_ARG for a missing or short workspace, as well as every
 * code of the three calls it stands for.
 */
int kda_layer_step(const kda_bf16 *x, const kda_bf16 *conv_weight,
                   const kda_bf16 *conv_bias, kda_bf16 *conv_state,
                   int64_t conv_slot_stride, const kda_bf16 *f_a,
                   const kda_bf16 *f_b, const kda_bf16 *raw_beta,
                   const float *A_log, const float *dt_bias, float lower_bound,
                   float q_scale, float *state_pool, int64_t slot_stride,
                   int n_slots, const int32_t *state_slots,
                   const int32_t *record_rows, const int32_t *pending,
                   float *corr, kda_bf16 *key_gate, int64_t corr_row_stride,
                   int64_t kg_row_stride, int n_rows, int rq,
                   const kda_bf16 *gate, const float *norm_weight, float eps,
                   kda_bf16 *out, void *workspace, int64_t workspace_bytes,
                   int B, int H, int Q, int null_slot, int32_t *status,
                   void *stream);

/*
 * kda_layer_step_noalloc -- kda_layer_step for callers that cannot allocate
 * device memory when they call it (the pages have no counterpart: this is
 * for this library's users).  A serving runtime that reserves all device
 * memory in its own pool at start-up, or a plugin whose host framework owns
 * every device allocation, may not call cudaMalloc on the decode path.
 * This entry point takes the same arguments as kda_layer_step except the
 * workspace: the step's operands go to a fixed array of device memory that
 * belongs to the library, KDA_LAYER_STEP_NOALLOC_MAX_BYTES bytes, held on
 * every GPU that loads the library until the process exits.  It allocates
 * and frees nothing.
 *  - Sizes: kda_layer_step_workspace_bytes(B, H, Q) must not exceed
 *    KDA_LAYER_STEP_NOALLOC_MAX_BYTES (B * Q * H <= 16384 (token, head)
 *    rows); larger calls return KDA_ERR_SCRATCH before anything is launched.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address, a runtime query; make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents.  Nothing in it needs clearing (each call writes the
 *    operands it then reads), but calls whose work overlaps on the GPU (on
 *    different streams, or from different threads) race on it: order them.
 *  - Every other argument, result and status code is kda_layer_step's.
 */
#define KDA_LAYER_STEP_NOALLOC_MAX_BYTES (16 * 1024 * 1024)
int kda_layer_step_noalloc(const kda_bf16 *x, const kda_bf16 *conv_weight,
                           const kda_bf16 *conv_bias, kda_bf16 *conv_state,
                           int64_t conv_slot_stride, const kda_bf16 *f_a,
                           const kda_bf16 *f_b, const kda_bf16 *raw_beta,
                           const float *A_log, const float *dt_bias,
                           float lower_bound, float q_scale, float *state_pool,
                           int64_t slot_stride, int n_slots,
                           const int32_t *state_slots,
                           const int32_t *record_rows, const int32_t *pending,
                           float *corr, kda_bf16 *key_gate,
                           int64_t corr_row_stride, int64_t kg_row_stride,
                           int n_rows, int rq, const kda_bf16 *gate,
                           const float *norm_weight, float eps, kda_bf16 *out,
                           int B, int H, int Q, int null_slot, int32_t *status,
                           void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_RECOVERSSM_H */
