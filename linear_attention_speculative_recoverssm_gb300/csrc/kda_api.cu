// C ABI of libkda_recoverssm.so: argument checks (after the stock wrapper
// kda_recoverssm_verify on page "vllm.models.kimi_k3.nvidia.
// specialized_decode.recoverssm.kernels"), launch-shape choice, dispatch to
// the kernels.  No allocation, no synchronisation, no CPU fallback.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kda_recoverssm.h"
#include "kda_launch.h"
#include "kda_step.cuh"

namespace kda {

int launch_step_q1(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q2(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q3(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q4(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q5(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q6(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q7(const StepParams &, int, int, int, cudaStream_t);
int launch_step_q8(const StepParams &, int, int, int, cudaStream_t);
int launch_step_layers_q1(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q2(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q3(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q4(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q5(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q6(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q7(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_layers_q8(const StepParams &, const LayerBases &, int, cudaStream_t);
int launch_step_varlen_q1(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q2(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q3(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q4(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q5(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q6(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q7(const StepParams &, int, int, int, cudaStream_t);
int launch_step_varlen_q8(const StepParams &, int, int, int, cudaStream_t);

namespace {
std::atomic<int> g_sm_count[64];
}

int device_sm_count(int dev) {
  const int slot = dev & 63;
  int v = g_sm_count[slot].load();
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 1;
    g_sm_count[slot].store(v);
  }
  return v;
}

int launch_step(const StepParams &p, int n_items, int Q, int variant, int split,
                cudaStream_t stream) {
  // windows from query_start_loc: instances of their own
  if (p.qsl != nullptr) {
    switch (Q) {
      case 1: return launch_step_varlen_q1(p, n_items, variant, split, stream);
      case 2: return launch_step_varlen_q2(p, n_items, variant, split, stream);
      case 3: return launch_step_varlen_q3(p, n_items, variant, split, stream);
      case 4: return launch_step_varlen_q4(p, n_items, variant, split, stream);
      case 5: return launch_step_varlen_q5(p, n_items, variant, split, stream);
      case 6: return launch_step_varlen_q6(p, n_items, variant, split, stream);
      case 7: return launch_step_varlen_q7(p, n_items, variant, split, stream);
      case 8: return launch_step_varlen_q8(p, n_items, variant, split, stream);
      default: return KDA_ERR_ARG;
    }
  }
  switch (Q) {
    case 1: return launch_step_q1(p, n_items, variant, split, stream);
    case 2: return launch_step_q2(p, n_items, variant, split, stream);
    case 3: return launch_step_q3(p, n_items, variant, split, stream);
    case 4: return launch_step_q4(p, n_items, variant, split, stream);
    case 5: return launch_step_q5(p, n_items, variant, split, stream);
    case 6: return launch_step_q6(p, n_items, variant, split, stream);
    case 7: return launch_step_q7(p, n_items, variant, split, stream);
    case 8: return launch_step_q8(p, n_items, variant, split, stream);
    default: return KDA_ERR_ARG;
  }
}

int launch_step_layers(const StepParams &p, const LayerBases &lay, int n_items, int Q,
                       cudaStream_t stream) {
  switch (Q) {
    case 1: return launch_step_layers_q1(p, lay, n_items, stream);
    case 2: return launch_step_layers_q2(p, lay, n_items, stream);
    case 3: return launch_step_layers_q3(p, lay, n_items, stream);
    case 4: return launch_step_layers_q4(p, lay, n_items, stream);
    case 5: return launch_step_layers_q5(p, lay, n_items, stream);
    case 6: return launch_step_layers_q6(p, lay, n_items, stream);
    case 7: return launch_step_layers_q7(p, lay, n_items, stream);
    case 8: return launch_step_layers_q8(p, lay, n_items, stream);
    default: return KDA_ERR_ARG;
  }
}

}  // namespace kda

namespace {

// check_step_args: the call is valid but has no work (B == 0).
constexpr int kNothingToDo = 1;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The step kernels divide by Gamma_s = prod_{r<=s} d_r >= e^{Q * lower_bound}
// (the pair-product rows k_s / Gamma_s); a gate bound of at most 10 in size
// keeps that and its inverse inside FP32 for Q <= 8.
inline bool gate_bound_ok(float lower_bound) {
  return lower_bound >= -10.0f && lower_bound <= 10.0f;  // false for NaN
}

// Checks shared by kda_verify and kda_replay_verify.
int check_step_args(const void *q, const void *k, const void *v, const void *g,
                    const void *beta, const void *A_log, const void *dt_bias,
                    const void *state_pool, int state_bytes, int64_t slot_stride, int n_slots,
                    const void *state_slots, const void *corr, const void *key_gate,
                    int64_t corr_row_stride, int64_t kg_row_stride, int n_rows, int rq,
                    const void *out, int B, int H, int Q, const void *query_start_loc,
                    int n_tokens) {
  if (B < 0 || H < 1 || Q < 1 || Q > KDA_MAX_WINDOW || rq < Q || rq > KDA_MAX_WINDOW)
    return KDA_ERR_ARG;
  if (B == 0) return kNothingToDo;  // no requests: empty buffers may be NULL
  // the activations hold n_tokens rows: B*Q without query_start_loc, at most
  // B*Q with it (the stock wrapper's activation-capacity check)
  if (n_tokens < 0 || (long long)n_tokens > (long long)B * Q) return KDA_ERR_ARG;
  if (query_start_loc == nullptr && (long long)n_tokens != (long long)B * Q) return KDA_ERR_ARG;
  if (n_tokens == 0) return kNothingToDo;  // zero tokens
  if (!q || !k || !v || !g || !beta || !A_log || !dt_bias || !state_pool || !state_slots ||
      !corr || !key_gate || !out)
    return KDA_ERR_ARG;
  if (n_slots < 1 || n_rows < 0) return KDA_ERR_ARG;
  if (slot_stride < (int64_t)H * KDA_HEAD_DIM * KDA_HEAD_DIM) return KDA_ERR_ARG;
  if (corr_row_stride < (int64_t)H * rq * KDA_HEAD_DIM ||
      kg_row_stride < (int64_t)H * rq * 2 * KDA_HEAD_DIM)
    return KDA_ERR_ARG;
  if ((long long)B * H > 0x7fffffffLL) return KDA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) ||
      !aligned16(state_pool) || !aligned16(corr) || !aligned16(key_gate) || !aligned16(out) ||
      !aligned16(dt_bias))
    return KDA_ERR_ALIGN;
  if (((slot_stride * state_bytes) & 15) != 0 || ((corr_row_stride * 4) & 15) != 0 ||
      ((kg_row_stride * 2) & 15) != 0)
    return KDA_ERR_ALIGN;
  return KDA_OK;
}

kda::StepParams make_params(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                            const kda_bf16 *raw_g, const kda_bf16 *raw_beta, const float *A_log,
                            const float *dt_bias, float lower_bound, float q_scale, void *state,
                            int64_t slot_stride, int n_slots, const int32_t *state_slots,
                            const int32_t *query_start_loc, int n_tokens,
                            const int32_t *record_rows, const int32_t *pending, float *corr,
                            kda_bf16 *key_gate, int64_t corr_row_stride, int64_t kg_row_stride,
                            int n_rows, int rq, const int32_t *boundary_slots,
                            const int32_t *boundary_lens, kda_bf16 *out, int B, int H,
                            int null_slot, int32_t *status) {
  kda::StepParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = raw_g;
  p.beta = raw_beta;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.lower_bound = lower_bound;
  p.q_scale = q_scale;
  p.state = state;
  p.slot_stride = slot_stride;
  p.n_slots = n_slots;
  p.state_slots = state_slots;
  p.qsl = query_start_loc;
  p.n_tokens = n_tokens;
  p.record_rows = record_rows;
  p.pending = pending;
  p.bnd_slots = boundary_slots;
  p.bnd_lens = boundary_lens;
  p.corr = corr;
  p.kg = key_gate;
  p.corr_row_stride = corr_row_stride;
  p.kg_row_stride = kg_row_stride;
  p.n_rows = n_rows;
  p.rq = rq;
  p.out = out;
  p.B = B;
  p.H = H;
  p.null_slot = null_slot;
  p.status = status;
  p.gate = nullptr;
  p.norm_w = nullptr;
  p.norm_eps = 0.f;
  kda::set_head_divisor(p);
  return p;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return 2; }

const char *kda_error_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_ARG: return "invalid argument";
    case KDA_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_CUDA: return "CUDA launch failed";
    case KDA_ERR_TIMEOUT: return "device wait timed out";
    case KDA_ERR_SCRATCH: return "call larger than the library's fixed scratch memory";
    default: return "unknown status";
  }
}

int kda_check_status(const int32_t *status, void *stream) {
  if (!status) return KDA_ERR_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  // pageable destination: the copy completes before the call returns
  if (cudaMemcpyAsync(&host, status, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
  return host;
}

int kda_verify(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *raw_g,
               const kda_bf16 *raw_beta, const float *A_log, const float *dt_bias,
               float lower_bound, float q_scale, const void *state_pool, int state_dtype,
               int64_t slot_stride, int n_slots, const int32_t *state_slots,
               const int32_t *query_start_loc, int n_tokens, const int32_t *record_rows,
               float *corr, kda_bf16 *key_gate, int64_t corr_row_stride,
               int64_t kg_row_stride, int n_rows, int rq, kda_bf16 *out, int B, int H, int Q,
               int null_slot, int32_t *status, void *stream) {
  if (state_dtype != KDA_STATE_F32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_UNSUPPORTED;
  if (!gate_bound_ok(lower_bound)) return KDA_ERR_UNSUPPORTED;
  const int sb = state_dtype == KDA_STATE_F32 ? 4 : 2;
  int rc = check_step_args(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pool, sb,
                           slot_stride, n_slots, state_slots, corr, key_gate, corr_row_stride,
                           kg_row_stride, n_rows, rq, out, B, H, Q, query_start_loc, n_tokens);
  if (rc == kNothingToDo) return KDA_OK;
  if (rc != KDA_OK) return rc;
  const kda::StepParams p = make_params(
      q, k, v, raw_g, raw_beta, A_log, dt_bias, lower_bound, q_scale,
      const_cast<void *>(state_pool), slot_stride, n_slots, state_slots, query_start_loc,
      n_tokens, record_rows, nullptr,
      corr, key_gate, corr_row_stride, kg_row_stride, n_rows, rq, nullptr, nullptr, out, B, H,
      null_slot, status);
  return kda::launch_step(p, B * H, Q, state_dtype == KDA_STATE_F32 ? 0 : 1, 1,
                          static_cast<cudaStream_t>(stream));
}

int kda_replay_verify(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                      const kda_bf16 *raw_g, const kda_bf16 *raw_beta, const float *A_log,
                      const float *dt_bias, float lower_bound, float q_scale, float *state_pool,
                      int64_t slot_stride, int n_slots, const int32_t *state_slots,
                      const int32_t *query_start_loc, int n_tokens,
                      const int32_t *record_rows, const int32_t *pending, float *corr,
                      kda_bf16 *key_gate, int64_t corr_row_stride, int64_t kg_row_stride,
                      int n_rows, int rq, const int32_t *boundary_slots,
                      const int32_t *boundary_lens, kda_bf16 *out, int B, int H, int Q,
                      int null_slot, int split, int32_t *status, void *stream) {
  if (!gate_bound_ok(lower_bound)) return KDA_ERR_UNSUPPORTED;
  int rc = check_step_args(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pool, 4, slot_stride,
                           n_slots, state_slots, corr, key_gate, corr_row_stride, kg_row_stride,
                           n_rows, rq, out, B, H, Q, query_start_loc, n_tokens);
  if (split != 0 && split != 1 && split != 2 && split != 4) return KDA_ERR_ARG;
  if (rc == kNothingToDo) return KDA_OK;
  if (rc != KDA_OK) return rc;
  if (!record_rows || !pending) return KDA_ERR_ARG;
  if ((boundary_slots == nullptr) != (boundary_lens == nullptr)) return KDA_ERR_ARG;
  const int items = B * H;
  if (split == 0) {
    // Split each item's rows over a cluster only while every CTA of the
    // split grid still has an SM of its own (measured on GB300: a 4-way
    // split cuts the latency of 32 items by ~25%, while 128 items are
    // fastest whole on persistent CTAs); otherwise whole items.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    const int sms = kda::device_sm_count(dev);
    split = items * 4 <= sms ? 4 : (items * 2 <= sms ? 2 : 1);
  }
  if (split > 1 && items > 65535) split = 1;
  const kda::StepParams p = make_params(
      q, k, v, raw_g, raw_beta, A_log, dt_bias, lower_bound, q_scale, state_pool, slot_stride,
      n_slots, state_slots, query_start_loc, n_tokens, record_rows, pending, corr, key_gate,
      corr_row_stride, kg_row_stride, n_rows, rq, boundary_slots, boundary_lens, out, B, H,
      null_slot, status);
  return kda::launch_step(p, items, Q, boundary_slots ? 3 : 2, split,
                          static_cast<cudaStream_t>(stream));
}

int kda_replay_verify_layers(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                             const kda_bf16 *raw_g, const kda_bf16 *raw_beta,
                             const float *A_log, const float *dt_bias, float lower_bound,
                             float q_scale, float *const *state_pools,
                             const int64_t *slot_strides, int n_slots,
                             const int32_t *state_slots, const int32_t *record_rows,
                             const int32_t *pending, float *const *corrs,
                             kda_bf16 *const *key_gates, const int64_t *corr_row_strides,
                             const int64_t *kg_row_strides, int n_rows, int rq, kda_bf16 *out,
                             int L, int B, int H, int Q, int null_slot, int32_t *status,
                             void *stream) {
  if (!gate_bound_ok(lower_bound)) return KDA_ERR_UNSUPPORTED;
  if (L < 1 || L > KDA_MAX_LAYERS) return KDA_ERR_ARG;
  if (!state_pools || !slot_strides || !corrs || !key_gates || !corr_row_strides ||
      !kg_row_strides)
    return KDA_ERR_ARG;
  // every layer's pool and records, checked like the one-layer call's
  // (layer 0's stand in for the pointers the shared checks look at)
  const long long n_tok = (long long)B * Q;
  int rc = check_step_args(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pools[0], 4,
                           slot_strides[0], n_slots, state_slots, corrs[0], key_gates[0],
                           corr_row_strides[0], kg_row_strides[0], n_rows, rq, out, B, H, Q,
                           nullptr, (int)(n_tok > 0x7fffffffLL ? -1 : n_tok));
  if (rc == kNothingToDo) return KDA_OK;
  if (rc != KDA_OK) return rc;
  if (!record_rows || !pending) return KDA_ERR_ARG;
  if ((long long)L * B * H > 0x7fffffffLL) return KDA_ERR_ARG;
  kda::LayerBases lay;
  lay.L = L;
  lay.act_stride = n_tok * H * KDA_HEAD_DIM;
  lay.beta_stride = n_tok * H;
  for (int l = 0; l < L; ++l) {
    if (!state_pools[l] || !corrs[l] || !key_gates[l]) return KDA_ERR_ARG;
    if (slot_strides[l] < (int64_t)H * KDA_HEAD_DIM * KDA_HEAD_DIM ||
        corr_row_strides[l] < (int64_t)H * rq * KDA_HEAD_DIM ||
        kg_row_strides[l] < (int64_t)H * rq * 2 * KDA_HEAD_DIM)
      return KDA_ERR_ARG;
    if (!aligned16(state_pools[l]) || !aligned16(corrs[l]) || !aligned16(key_gates[l]))
      return KDA_ERR_ALIGN;
    if (((slot_strides[l] * 4) & 15) != 0 || ((corr_row_strides[l] * 4) & 15) != 0 ||
        ((kg_row_strides[l] * 2) & 15) != 0)
      return KDA_ERR_ALIGN;
    lay.state[l] = reinterpret_cast<uint64_t>(state_pools[l]);
    lay.corr[l] = reinterpret_cast<uint64_t>(corrs[l]);
    lay.kg[l] = reinterpret_cast<uint64_t>(key_gates[l]);
    lay.slot_stride[l] = slot_strides[l];
    lay.corr_stride[l] = corr_row_strides[l];
    lay.kg_stride[l] = kg_row_strides[l];
  }
  // layer 0's pool and records are also the StepParams' (the kernel reads
  // the layer bases for every layer)
  const kda::StepParams p = make_params(
      q, k, v, raw_g, raw_beta, A_log, dt_bias, lower_bound, q_scale, state_pools[0],
      slot_strides[0], n_slots, state_slots, nullptr, (int)n_tok, record_rows, pending, corrs[0],
      key_gates[0], corr_row_strides[0], kg_row_strides[0], n_rows, rq, nullptr, nullptr, out, B,
      H, null_slot, status);
  return kda::launch_step_layers(p, lay, L * B * H, Q, static_cast<cudaStream_t>(stream));
}

int64_t kda_layer_step_workspace_bytes(int B, int H, int Q) {
  if (B < 0 || H < 1 || Q < 1 || Q > KDA_MAX_WINDOW) return -1;
  return 4LL * B * Q * H * KDA_HEAD_DIM * (int64_t)sizeof(kda_bf16);
}

int kda_layer_step(const kda_bf16 *x, const kda_bf16 *conv_weight, const kda_bf16 *conv_bias,
                   kda_bf16 *conv_state, int64_t conv_slot_stride, const kda_bf16 *f_a,
                   const kda_bf16 *f_b, const kda_bf16 *raw_beta, const float *A_log,
                   const float *dt_bias, float lower_bound, float q_scale, float *state_pool,
                   int64_t slot_stride, int n_slots, const int32_t *state_slots,
                   const int32_t *record_rows, const int32_t *pending, float *corr,
                   kda_bf16 *key_gate, int64_t corr_row_stride, int64_t kg_row_stride,
                   int n_rows, int rq, const kda_bf16 *gate, const float *norm_weight,
                   float eps, kda_bf16 *out, void *workspace, int64_t workspace_bytes, int B,
                   int H, int Q, int null_slot, int32_t *status, void *stream) {
  if (!gate_bound_ok(lower_bound)) return KDA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f)) return KDA_ERR_ARG;  // (false for NaN)
  const int64_t need = kda_layer_step_workspace_bytes(B, H, Q);
  if (need < 0) return KDA_ERR_ARG;
  if (B == 0) return KDA_OK;
  if (!workspace || workspace_bytes < need || !gate || !norm_weight || !record_rows || !pending)
    return KDA_ERR_ARG;
  if (!aligned16(workspace) || !aligned16(gate) || !aligned16(norm_weight)) return KDA_ERR_ALIGN;
  // the step's operands q, k, v, raw_g, made by the prologue in the workspace
  const int64_t part = need / 4 / (int64_t)sizeof(kda_bf16);
  kda_bf16 *wq = static_cast<kda_bf16 *>(workspace);
  kda_bf16 *wk = wq + part, *wv = wk + part, *wg = wv + part;
  const int n_tokens = B * Q;
  int rc = check_step_args(wq, wk, wv, wg, raw_beta, A_log, dt_bias, state_pool, 4, slot_stride,
                           n_slots, state_slots, corr, key_gate, corr_row_stride, kg_row_stride,
                           n_rows, rq, out, B, H, Q, nullptr, n_tokens);
  if (rc == kNothingToDo) return KDA_OK;
  if (rc != KDA_OK) return rc;
  rc = kda_layer_prologue(x, conv_weight, conv_bias, conv_state, conv_slot_stride, f_a, f_b,
                          state_slots, record_rows, pending, n_slots, n_rows, rq, wq, wk, wv, wg,
                          B, H, Q, null_slot, status, stream);
  if (rc != KDA_OK) return rc;
  kda::StepParams p = make_params(wq, wk, wv, wg, raw_beta, A_log, dt_bias, lower_bound,
                                  q_scale, state_pool, slot_stride, n_slots, state_slots, nullptr,
                                  n_tokens, record_rows, pending, corr, key_gate,
                                  corr_row_stride, kg_row_stride, n_rows, rq, nullptr, nullptr,
                                  out, B, H, null_slot, status);
  p.gate = gate;
  p.norm_w = norm_weight;
  p.norm_eps = eps;
  return kda::launch_step(p, B * H, Q, 4, 1, static_cast<cudaStream_t>(stream));
}

int kda_commit(const uint64_t *state_ptrs, const uint64_t *corr_ptrs, const uint64_t *kg_ptrs,
               const int64_t *state_strides, const int64_t *corr_strides,
               const int64_t *kg_strides, const float *A_log, const float *dt_bias,
               const int32_t *sources, const int32_t *commit_lens, const int32_t *destinations,
               const int32_t *boundaries, const int32_t *boundary_lens,
               const int32_t *record_rows, int state_dtype, float lower_bound, int null_slot,
               int L, int H, int B, int Q, int n_slots, int n_rows, int32_t *status,
               void *stream) {
  if (state_dtype != KDA_STATE_F32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_UNSUPPORTED;
  // the align boundary state divides the partial replay sum by
  // prod_{m<=s<n} d_s, which must stay inside FP32
  if (!gate_bound_ok(lower_bound)) return KDA_ERR_UNSUPPORTED;
  if (L < 0 || H < 1 || B < 0 || Q < 1 || Q > KDA_MAX_WINDOW || n_slots < 1 || n_rows < 0)
    return KDA_ERR_ARG;
  if (!state_ptrs || !corr_ptrs || !kg_ptrs || !state_strides || !corr_strides || !kg_strides ||
      !A_log || !dt_bias || !sources || !commit_lens || !destinations)
    return KDA_ERR_ARG;
  if ((boundaries == nullptr) != (boundary_lens == nullptr)) return KDA_ERR_ARG;
  if (L == 0 || B == 0) return KDA_OK;
  return kda::launch_commit(state_ptrs, corr_ptrs, kg_ptrs, state_strides, corr_strides,
                            kg_strides, A_log, dt_bias, sources, commit_lens, destinations,
                            boundaries, boundary_lens, record_rows, state_dtype, lower_bound,
                            null_slot, L, H, B, Q, n_slots, n_rows, status,
                            static_cast<cudaStream_t>(stream));
}

int kda_defer_commit(const int32_t *state_slots, int32_t *commit_lens, const int32_t *record_rows,
                     int32_t *pending, const uint8_t *eager, int B, int null_slot, int n_rows,
                     int32_t *status, void *stream) {
  if (B < 0 || n_rows < 0) return KDA_ERR_ARG;
  if (!state_slots || !commit_lens || !record_rows || !pending) return KDA_ERR_ARG;
  if (B == 0) return KDA_OK;
  return kda::launch_defer_commit(state_slots, commit_lens, record_rows, pending, eager, B,
                                  null_slot, n_rows, status, static_cast<cudaStream_t>(stream));
}

int kda_flush_plan(const int32_t *state_slots, const int32_t *record_rows, const int32_t *pending,
                   int32_t *commit_lens, int32_t *final_slots, int32_t *boundary_slots,
                   int32_t *boundary_lens, int B, int Q, int null_slot, int n_rows,
                   int32_t *status, void *stream) {
  if (B < 0 || Q < 1 || Q > KDA_MAX_WINDOW || n_rows < 0) return KDA_ERR_ARG;
  if (!state_slots || !record_rows || !pending || !commit_lens || !final_slots ||
      !boundary_slots || !boundary_lens)
    return KDA_ERR_ARG;
  if (B == 0) return KDA_OK;
  return kda::launch_flush_plan(state_slots, record_rows, pending, commit_lens, final_slots,
                                boundary_slots, boundary_lens, B, Q, null_slot, n_rows, status,
                                static_cast<cudaStream_t>(stream));
}

}  // extern "C"

int kda_selftest_wait_timeout(int32_t *status, void *stream) {
  if (!status) return KDA_ERR_ARG;
  return kda::launch_selftest_timeout(status, static_cast<cudaStream_t>(stream));
}
