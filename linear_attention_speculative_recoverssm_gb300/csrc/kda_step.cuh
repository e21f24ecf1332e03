// Definitions shared by the KDA RecoverSSM step kernels (the warp-specialised
// persistent kernel and the cluster-split kernel): the launch parameters, the
// per-item metadata (slot, record row, clamped pending count, boundary) and
// the state-page addressing -- page "vllm.models.kimi_k3.nvidia.
// specialized_decode.cutedsl.kda.fused", module docstring steps 1-3.
//
// No tensor cores: per item the work is a [128 x 128] x [128 x 2Q] mat-vec
// (Q <= 8) against 64 KB of state read once and written at most once, so the
// step is bound by HBM bandwidth, with FP32 FMAs on the CUDA cores.
#pragma once

#include "kda_device.cuh"

namespace kda {

constexpr int kThreads = 256;

struct StepParams {
  const uint16_t *q, *k, *v, *g, *beta;  // BF16 bits
  const float *A_log, *dt_bias;
  float lower_bound, q_scale;
  void *state;            // pool base (FP32 or BF16 bits)
  long long slot_stride;  // elements per slot
  int n_slots;
  const int32_t *state_slots, *record_rows, *pending;
  // request b's window: tokens qsl[b] .. qsl[b + 1] - 1 of the n_tokens
  // activation rows (qsl == nullptr: tokens b*Q .. b*Q + Q - 1)
  const int32_t *qsl;
  int n_tokens;
  const int32_t *bnd_slots, *bnd_lens;
  float *corr;
  uint16_t *kg;
  long long corr_row_stride, kg_row_stride;
  int n_rows, rq;
  uint16_t *out;
  int B, H, null_slot;
  int32_t *status;
  // the gated RMSNorm folded into the step (the NORM instances only):
  // out[t, h*128 + r] = BF16(o * rsqrt(mean_r o^2 + norm_eps) * norm_w[r] *
  // sigmoid(gate[t, h*128 + r])), o the BF16-rounded recurrence output
  const uint16_t *gate;  // [n_tokens, H*128] BF16 bits
  const float *norm_w;   // [128]
  float norm_eps;
  // n / H by a multiply and shifts (set_head_divisor)
  uint32_t h_mul;
  int h_sh1, h_sh2;
};

// Division of an item index by the head count H, an invariant of the call,
// by a multiply and two shifts (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, the unsigned
// round-up method): with l = ceil(log2 H) and m = floor(2^32 (2^l - H) / H)
// + 1, n / H = (t + ((n - t) >> 1)) >> (l - 1) where t = mulhi(m, n), for
// every 32-bit n (H = 1: m = 1 and both shifts 0).
inline void set_head_divisor(StepParams &p) {
  const uint32_t H = (uint32_t)p.H;
  int l = 0;
  while ((1ull << l) < H) ++l;
  p.h_mul = (uint32_t)((((1ull << 32) * ((1ull << l) - H)) / H) + 1);
  p.h_sh1 = l > 0 ? 1 : 0;
  p.h_sh2 = l > 0 ? l - 1 : 0;
}

__device__ __forceinline__ int div_heads(const StepParams &p, int n) {
  const uint32_t u = (uint32_t)n;
  const uint32_t t = __umulhi(p.h_mul, u);
  return (int)((t + ((u - t) >> p.h_sh1)) >> p.h_sh2);
}

// The multi-layer step: one launch over L layers whose items are
// (layer, request, head), layer-major.  Every layer has its own state pool,
// corrections and key / gate records (addresses and strides, passed by value
// as kernel parameters); the index arrays (state slots, record rows, pending
// counts) are shared by the layers, and the activations and outputs of all
// layers are stacked, layer l's at l * act_stride elements (raw_beta at
// l * beta_stride).  A_log is [L, H] and dt_bias [L, H, 128].
constexpr int kMaxLayers = KDA_MAX_LAYERS;
struct LayerBases {
  int L;
  long long act_stride, beta_stride;
  uint64_t state[kMaxLayers], corr[kMaxLayers], kg[kMaxLayers];
  long long slot_stride[kMaxLayers], corr_stride[kMaxLayers], kg_stride[kMaxLayers];
};

// Number of scalars the token half reduces over channels: sum k_t^2,
// sum q_t^2 (Q each) and the Q*Q raw pair products (B_ts at t*Q + s for
// s <= t, A_ts at s*Q + t for s < t).
template <int Q>
struct Red {
  static constexpr int kN = 2 * Q + Q * Q;
  static constexpr int kPad = round_up(kN, 32);
};

// ---------------------------------------------------------------------------
// per-item metadata (uniform across the CTA)
// ---------------------------------------------------------------------------

struct ItemMeta {
  int b, h;
  int l;      // layer (the multi-layer step; 0 otherwise)
  int tok0;   // first token of the window
  int qb;     // window length, 0 .. Q
  int slot;   // < 0: inert
  int rec;    // < 0: no records
  int n;      // pending tokens to replay
  int bslot;  // boundary slot, < 0: none
  int m;      // boundary length (min(m, n))
};

// A request's window from query_start_loc: valid when it lies inside the
// activations and holds at most Q tokens.
__device__ __forceinline__ bool window_ok(const StepParams &p, int q0, int q1, int Q) {
  return q0 >= 0 && q1 >= q0 && q1 <= p.n_tokens && q1 - q0 <= Q;
}

template <bool REPLAY, bool BOUNDARY, bool VARLEN>
__device__ __forceinline__ ItemMeta item_meta(const StepParams &p, int item, int Q,
                                              bool report_errors) {
  ItemMeta it;
  it.b = item / p.H;
  it.h = item - it.b * p.H;
  it.l = 0;
  int slot = p.state_slots[it.b];
  if (slot >= p.n_slots) {
    if (report_errors) report(p.status, KDA_ERR_ARG);
    slot = -1;
  }
  it.slot = slot > p.null_slot ? slot : -1;
  it.tok0 = it.b * Q;
  it.qb = Q;
  if constexpr (VARLEN) {
    const int q0 = p.qsl[it.b], q1 = p.qsl[it.b + 1];
    if (window_ok(p, q0, q1, Q)) {
      it.tok0 = q0;
      it.qb = q1 - q0;
    } else {  // nothing of the request is read or written
      if (report_errors) report(p.status, KDA_ERR_ARG);
      it.slot = -1;
      it.tok0 = 0;
      it.qb = 0;
    }
  }
  int rec = p.record_rows != nullptr ? p.record_rows[it.b] : it.b;
  if (rec >= p.n_rows) {
    if (report_errors && it.slot >= 0) report(p.status, KDA_ERR_ARG);
    rec = -1;
  }
  it.rec = rec;
  int n = 0;
  if (REPLAY && rec >= 0) {
    n = p.pending[rec];
    n = n < 0 ? 0 : (n > p.rq ? p.rq : n);
  }
  it.n = n;
  it.bslot = -1;
  it.m = 0;
  if (BOUNDARY && n > 0 && p.bnd_slots != nullptr) {
    const int bs = p.bnd_slots[it.b];
    const int m = p.bnd_lens[it.b];
    if (bs >= p.n_slots) {
      if (report_errors) report(p.status, KDA_ERR_ARG);
    } else if (m > 0 && bs > p.null_slot) {
      it.bslot = bs;
      it.m = m < n ? m : n;
    }
  }
  return it;
}

template <typename ST>
__device__ __forceinline__ const ST *page_ptr(const StepParams &p, int slot,
                                              int h) {
  return reinterpret_cast<const ST *>(p.state) +
         (long long)slot * p.slot_stride + (long long)h * (kDim * kDim);
}

}  // namespace kda
