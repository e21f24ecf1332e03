// The KDA RecoverSSM step kernel: replay of the pending recorded tokens into
// the checkpoint, chunked (WY) verify of this window, write-back of S_n and
// of the new records -- page "vllm.models.kimi_k3.nvidia.specialized_decode.
// cutedsl.kda.fused", module docstring steps 1-3.
//
// Design (one GPU, sm_103a):
//  * Persistent CTAs, one per SM (the stage ring takes ~190 KB of shared
//    memory).  CTA i walks the (request, head) items i, i + grid, ...
//  * Thread 0 streams each item's state page (64 KB FP32, or 32 KB BF16,
//    contiguous [V=128 rows][K=128]) into a ring of NS shared-memory stages
//    with one bulk copy (cp.async.bulk, completing on an mbarrier), NS items
//    ahead of the compute, so HBM reads stay in flight while the CTA works.
//  * Prologue per item (no state needed): threads 0-127 own key channel
//    c = tid for this window's tokens (decays, Gamma_t k_t and Gamma_t q_t,
//    sums of squares, raw A / B pair products reduced over channels with a
//    warp reduce-scatter); threads 128-255 own channel c for the recorded
//    tokens (decays, suffix products P_t, D_n, the recorded corrections, v,
//    beta).  Keys and queries stay unnormalised in shared memory: their
//    rsqrt norms are per-token scalars folded into the corrections (replay)
//    and into the dot products / pair products (verify).
//  * Main loop: thread (g = tid / 4, l = tid % 4) holds rows g and g + 64
//    and keys 4 (l + 4 c') .. +3 for 8 chunks c' (c' rotated by g & 1 or
//    g & 3 so a warp's shared loads hit distinct banks): replay S_n =
//    S_0 D_n + sum_t u_t kp_t in registers, store S_n (n > 0) straight to
//    global memory, and accumulate the 2Q row dot products.  A
//    reduce-scatter over the 4 lanes of a row leaves each lane Q finished
//    dots.
//  * Row solve: thread r < 128 owns state row r: forward substitution for
//    u_t, outputs o_t (BF16), corrections u_t (FP32).
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
  const int32_t *bnd_slots, *bnd_lens;
  float *corr;
  uint16_t *kg;
  long long corr_row_stride, kg_row_stride;
  int n_rows, rq;
  uint16_t *out;
  int B, H, null_slot;
  int32_t *status;
};

template <typename ST>
struct StateTraits;
template <>
struct StateTraits<float> {
  static constexpr int kBytes = 4;
  // FP32 rows are 512 B: rotating chunk parity by row group keeps the 8
  // lanes of a quarter-warp on distinct banks.
  static constexpr int kRotate = 1;
  __device__ static float4 load4(const float *page, int row, int key) {
    return lds4(page + row * kDim + key);
  }
};
template <>
struct StateTraits<uint16_t> {
  static constexpr int kBytes = 2;
  static constexpr int kRotate = 3;
  __device__ static float4 load4(const uint16_t *page, int row, int key) {
    const uint2 w = *reinterpret_cast<const uint2 *>(page + row * kDim + key);
    return make_float4(__uint_as_float(w.x << 16),
                       __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xffff0000u));
  }
};

// Number of scalars the token half reduces over channels: sum k_t^2,
// sum q_t^2 (Q each) and the Q*Q raw pair products (B_ts at t*Q + s for
// s <= t, A_ts at s*Q + t for s < t).
template <int Q>
struct Red {
  static constexpr int kN = 2 * Q + Q * Q;
  static constexpr int kPad = round_up(kN, 32);
};

template <int Q, typename ST, int NS, bool BOUNDARY>
struct StepSmem {
  ST stage[NS][kDim * kDim];
  union {
    struct {
      float xk[Q][kDim];  // Gamma_t * k_t (unnormalised)
      float xq[Q][kDim];  // Gamma_t * q_t (unnormalised)
    } x;
    float dots[2 * Q][kDim];  // after the main loop: w (j < Q), y (j >= Q)
  } xd;
  float kp[kMaxQ][kDim];    // recorded k_t * P_t (unnormalised)
  float dn[kDim];           // D_n
  float kpb[BOUNDARY ? kMaxQ : 1][kDim];  // the same for S_min(m, n)
  float db[BOUNDARY ? 1 : 1][kDim];
  float uold[kMaxQ][kDim];  // recorded corrections u_t
  float vv[2][Q][kDim];     // v_t (double-buffered by item parity)
  float beta[2][kMaxQ];
  float red_tok[4][Red<Q>::kPad];
  float red_rec[4][kMaxQ];
  float scal[Red<Q>::kN];   // rsk[Q], rsq[Q] (with q_scale), A / B
  uint64_t full[NS];
};

template <typename ST>
__host__ __device__ constexpr int default_stages() {
  return sizeof(ST) == 4 ? 3 : 6;
}

// ---------------------------------------------------------------------------
// per-item metadata (uniform across the CTA)
// ---------------------------------------------------------------------------

struct ItemMeta {
  int b, h;
  int slot;   // < 0: inert
  int rec;    // < 0: no records
  int n;      // pending tokens to replay
  int bslot;  // boundary slot, < 0: none
  int m;      // boundary length (min(m, n))
};

template <bool REPLAY, bool BOUNDARY>
__device__ __forceinline__ ItemMeta item_meta(const StepParams &p, int item,
                                              bool report_errors) {
  ItemMeta it;
  it.b = item / p.H;
  it.h = item - it.b * p.H;
  int slot = p.state_slots[it.b];
  if (slot >= p.n_slots) {
    if (report_errors) report(p.status, KDA_ERR_ARG);
    slot = -1;
  }
  it.slot = slot > p.null_slot ? slot : -1;
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

// ---------------------------------------------------------------------------
// the persistent kernel
// ---------------------------------------------------------------------------

template <int Q, typename ST, bool REPLAY, bool BOUNDARY>
__global__ void __launch_bounds__(kThreads, 1)
    kda_step_persistent(const StepParams p, int n_items) {
  constexpr int NS = default_stages<ST>();
  using Smem = StepSmem<Q, ST, NS, BOUNDARY>;
  constexpr uint32_t kPageBytes = kDim * kDim * sizeof(ST);
  constexpr int NR = Red<Q>::kN;
  constexpr int NRP = Red<Q>::kPad;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int first = blockIdx.x, stride = gridDim.x;
  const int count = first < n_items ? (n_items - first + stride - 1) / stride : 0;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&sm.full[s], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // Producer: the state page of this CTA's j-th item into stage j % NS.
  auto issue = [&](int j) {
    const int item = first + j * stride;
    const int b = item / p.H;
    const int h = item - b * p.H;
    const int slot = p.state_slots[b];
    uint64_t *bar = &sm.full[j % NS];
    if (slot > p.null_slot && slot < p.n_slots) {
      mbar_arrive_expect_tx(bar, kPageBytes);
      bulk_g2s(sm.stage[j % NS], page_ptr<ST>(p, slot, h), kPageBytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  if (tid == 0) {
    for (int j = 0; j < NS && j < count; ++j) issue(j);
  }

  const int g = tid >> 2, l = tid & 3;  // main-loop row group and lane
  const bool token_half = tid < kDim;
  const int c = tid & (kDim - 1);       // prologue channel

  for (int j = 0; j < count; ++j) {
    const int item = first + j * stride;
    const ItemMeta it = item_meta<REPLAY, BOUNDARY>(p, item, tid == 0);
    const int par = j & 1;
    const long long tok0 = (long long)it.b * Q;  // first token of request b

    if (it.slot < 0) {
      // Inert request: zero outputs only.  Its stage was never loaded.
      for (int e = tid; e < Q * kDim; e += kThreads) {
        const int t = e / kDim, ch = e - t * kDim;
        p.out[((tok0 + t) * p.H + it.h) * kDim + ch] = 0;
      }
      if (tid == 0 && j + NS < count) issue(j + NS);
      // Keeps the record half from running two items ahead of the row solve
      // (the double-buffered v / beta would be overwritten).
      __syncthreads();
      continue;
    }

    // ---------------- prologue ----------------
    uint16_t kbits[Q], gbits[Q];
    if (token_half) {
      const float a = __expf(p.A_log[it.h]);
      const float dt = p.dt_bias[it.h * kDim + c];
      float kk[Q], qq[Q], dd[Q];
      float red[NRP];
#pragma unroll
      for (int i = 0; i < NRP; ++i) red[i] = 0.f;
      float gam = 1.f;
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        const long long off = ((tok0 + t) * p.H + it.h) * kDim + c;
        kbits[t] = p.k[off];
        gbits[t] = p.g[off];
        kk[t] = bf16_bits_to_f32(kbits[t]);
        qq[t] = bf16_bits_to_f32(p.q[off]);
        dd[t] = gate_decay(a, bf16_bits_to_f32(gbits[t]), dt, p.lower_bound);
        gam *= dd[t];
        sm.xd.x.xk[t][c] = gam * kk[t];
        sm.xd.x.xq[t][c] = gam * qq[t];
        red[t] = kk[t] * kk[t];
        red[Q + t] = qq[t] * qq[t];
      }
      // raw pair products: B(t, s) = k_s . P(s, t) q_t (s <= t) and
      // A(t, s) = k_s . P(s, t) k_t (s < t), P(s, t) = prod_{s<r<=t} d_r
#pragma unroll
      for (int s = 0; s < Q; ++s) {
        red[2 * Q + s * Q + s] = kk[s] * qq[s];
        float pr = 1.f;
#pragma unroll
        for (int t = s + 1; t < Q; ++t) {
          pr *= dd[t];
          const float w = kk[s] * pr;
          red[2 * Q + t * Q + s] = w * qq[t];
          red[2 * Q + s * Q + t] = w * kk[t];
        }
      }
      reduce_scatter<NRP, 32>(red, lane);
#pragma unroll
      for (int i = 0; i < NRP / 32; ++i) sm.red_tok[warp][lane * (NRP / 32) + i] = red[i];
    } else {
      // records of the previous window (read before any is overwritten)
      if (REPLAY && it.n > 0) {
        const float a = __expf(p.A_log[it.h]);
        const float dt = p.dt_bias[it.h * kDim + c];
        const long long cbase = (long long)it.rec * p.corr_row_stride +
                                (long long)it.h * p.rq * kDim + c;
        const long long kbase = (long long)it.rec * p.kg_row_stride +
                                (long long)it.h * p.rq * (2 * kDim) + c;
        float kr[kMaxQ], dr[kMaxQ];
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          kr[t] = 0.f;
          dr[t] = 1.f;
          if (t < it.n) {
            sm.uold[t][c] = p.corr[cbase + t * kDim];
            kr[t] = bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim]);
            dr[t] = gate_decay(a, bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim + kDim]),
                               dt, p.lower_bound);
          }
        }
        // suffix products: kp_t = k_t * prod_{t<s<n} d_s, D_n = prod_{s<n} d_s
        float fd = 1.f;
#pragma unroll
        for (int t = kMaxQ - 1; t >= 0; --t) {
          if (t < it.n) {
            sm.kp[t][c] = kr[t] * fd;
            fd *= dr[t];
          }
        }
        sm.dn[c] = fd;
        if constexpr (BOUNDARY) if (it.bslot >= 0) {
          float fb = 1.f;
#pragma unroll
          for (int t = kMaxQ - 1; t >= 0; --t) {
            if (t < it.m) {
              sm.kpb[t][c] = kr[t] * fb;
              fb *= dr[t];
            }
          }
          sm.db[0][c] = fb;
        }
        float sq[kMaxQ];
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) sq[t] = kr[t] * kr[t];
        reduce_scatter<kMaxQ, 8>(sq, lane & 7);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 8);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);
        if (lane < kMaxQ) sm.red_rec[warp - 4][lane] = sq[0];
      }
      const long long voff = (tok0 * p.H + it.h) * kDim + c;
#pragma unroll
      for (int t = 0; t < Q; ++t)
        sm.vv[par][t][c] = bf16_bits_to_f32(p.v[voff + (long long)t * p.H * kDim]);
      if (c < Q)
        sm.beta[par][c] = sigmoidf_fast(bf16_bits_to_f32(p.beta[(tok0 + c) * p.H + it.h]));
    }

    // The state page of this item must have landed; the wait is bounded and
    // its outcome made uniform with the barrier.
    const bool ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        report(p.status, KDA_ERR_TIMEOUT);
        // let this CTA's own copies in flight land before it exits
        for (int jj = j; jj < j + NS && jj < count; ++jj)
          mbar_wait_bounded(&sm.full[jj % NS], (uint32_t)((jj / NS) & 1));
      }
      __syncthreads();
      return;
    }

    // New key / gate records: the old ones were read before the barrier.
    if (token_half && it.rec >= 0) {
      const long long kbase = (long long)it.rec * p.kg_row_stride +
                              (long long)it.h * p.rq * (2 * kDim) + c;
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        p.kg[kbase + t * 2 * kDim] = kbits[t];
        p.kg[kbase + t * 2 * kDim + kDim] = gbits[t];
      }
    }

    // ---------------- main loop: replay + 2Q dots per row ----------------
    const int v0 = g, v1 = g + 64;
    float u0[kMaxQ], u1[kMaxQ], ub0[kMaxQ], ub1[kMaxQ];
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
      u0[t] = u1[t] = ub0[t] = ub1[t] = 0.f;
      if (REPLAY && t < it.n) {
        const float tot = (sm.red_rec[0][t] + sm.red_rec[2][t]) +
                          (sm.red_rec[1][t] + sm.red_rec[3][t]);
        const float rs = rsqrtf(tot + kNormEps);
        u0[t] = sm.uold[t][v0] * rs;
        u1[t] = sm.uold[t][v1] * rs;
        if (BOUNDARY && t < it.m) {
          ub0[t] = u0[t];
          ub1[t] = u1[t];
        }
      }
    }
    const ST *page = sm.stage[j % NS];
    float *gout = nullptr;
    float *gbnd = nullptr;
    if (REPLAY) {
      gout = reinterpret_cast<float *>(p.state) + (long long)it.slot * p.slot_stride +
             (long long)it.h * (kDim * kDim);
      if (BOUNDARY && it.bslot >= 0)
        gbnd = reinterpret_cast<float *>(p.state) + (long long)it.bslot * p.slot_stride +
               (long long)it.h * (kDim * kDim);
    }
    float acc[2][2 * Q];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int jj = 0; jj < 2 * Q; ++jj) acc[r][jj] = 0.f;

#pragma unroll
    for (int cc0 = 0; cc0 < 8; ++cc0) {
      const int cc = cc0 ^ (g & StateTraits<ST>::kRotate);
      const int key = 4 * (l + 4 * cc);
      float4 s0 = StateTraits<ST>::load4(page, v0, key);
      float4 s1 = StateTraits<ST>::load4(page, v1, key);
      if (REPLAY && it.n > 0) {
        if constexpr (BOUNDARY) if (gbnd != nullptr) {
          const float4 d4 = lds4(&sm.db[0][key]);
          float4 b0 = make_float4(s0.x * d4.x, s0.y * d4.y, s0.z * d4.z, s0.w * d4.w);
          float4 b1 = make_float4(s1.x * d4.x, s1.y * d4.y, s1.z * d4.z, s1.w * d4.w);
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t) {
            if (t < it.m) {
              const float4 k4 = lds4(&sm.kpb[t][key]);
              b0.x = fmaf(ub0[t], k4.x, b0.x); b0.y = fmaf(ub0[t], k4.y, b0.y);
              b0.z = fmaf(ub0[t], k4.z, b0.z); b0.w = fmaf(ub0[t], k4.w, b0.w);
              b1.x = fmaf(ub1[t], k4.x, b1.x); b1.y = fmaf(ub1[t], k4.y, b1.y);
              b1.z = fmaf(ub1[t], k4.z, b1.z); b1.w = fmaf(ub1[t], k4.w, b1.w);
            }
          }
          stg4(gbnd + v0 * kDim + key, b0);
          stg4(gbnd + v1 * kDim + key, b1);
        }
        const float4 d4 = lds4(&sm.dn[key]);
        s0 = make_float4(s0.x * d4.x, s0.y * d4.y, s0.z * d4.z, s0.w * d4.w);
        s1 = make_float4(s1.x * d4.x, s1.y * d4.y, s1.z * d4.z, s1.w * d4.w);
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          if (t < it.n) {
            const float4 k4 = lds4(&sm.kp[t][key]);
            s0.x = fmaf(u0[t], k4.x, s0.x); s0.y = fmaf(u0[t], k4.y, s0.y);
            s0.z = fmaf(u0[t], k4.z, s0.z); s0.w = fmaf(u0[t], k4.w, s0.w);
            s1.x = fmaf(u1[t], k4.x, s1.x); s1.y = fmaf(u1[t], k4.y, s1.y);
            s1.z = fmaf(u1[t], k4.z, s1.z); s1.w = fmaf(u1[t], k4.w, s1.w);
          }
        }
        stg4(gout + v0 * kDim + key, s0);
        stg4(gout + v1 * kDim + key, s1);
      }
#pragma unroll
      for (int jj = 0; jj < Q; ++jj) {
        const float4 x = lds4(&sm.xd.x.xk[jj][key]);
        acc[0][jj] = fmaf(s0.x, x.x, fmaf(s0.y, x.y, fmaf(s0.z, x.z, fmaf(s0.w, x.w, acc[0][jj]))));
        acc[1][jj] = fmaf(s1.x, x.x, fmaf(s1.y, x.y, fmaf(s1.z, x.z, fmaf(s1.w, x.w, acc[1][jj]))));
      }
#pragma unroll
      for (int jj = 0; jj < Q; ++jj) {
        const float4 x = lds4(&sm.xd.x.xq[jj][key]);
        acc[0][Q + jj] = fmaf(s0.x, x.x, fmaf(s0.y, x.y, fmaf(s0.z, x.z, fmaf(s0.w, x.w, acc[0][Q + jj]))));
        acc[1][Q + jj] = fmaf(s1.x, x.x, fmaf(s1.y, x.y, fmaf(s1.z, x.z, fmaf(s1.w, x.w, acc[1][Q + jj]))));
      }
    }

    // Reduce the 4 lanes of each row: lane l keeps (row v_{l>>1},
    // dots (l & 1) * Q .. +Q).
    float vals[4 * Q];
#pragma unroll
    for (int jj = 0; jj < 2 * Q; ++jj) {
      vals[jj] = acc[0][jj];
      vals[2 * Q + jj] = acc[1][jj];
    }
    reduce_scatter<4 * Q, 4>(vals, l);
    __syncthreads();  // every thread is done with xk / xq and the stage
    if (tid == 0 && j + NS < count) issue(j + NS);
    {
      const int row = (l >> 1) ? v1 : v0;
      const int jb = (l & 1) * Q;
#pragma unroll
      for (int i = 0; i < Q; ++i) sm.xd.dots[jb + i][row] = vals[i];
    }
    // Final scalars: norms and the normalised pair products.
    if (tid < NR) {
      auto tot = [&](int i) {
        return (sm.red_tok[0][i] + sm.red_tok[2][i]) + (sm.red_tok[1][i] + sm.red_tok[3][i]);
      };
      const float x = tot(tid);
      float val;
      if (tid < Q) {
        val = rsqrtf(x + kNormEps);
      } else if (tid < 2 * Q) {
        val = rsqrtf(x + kNormEps) * p.q_scale;
      } else {
        const int pi = tid - 2 * Q;
        const int a = pi / Q, bb = pi - a * Q;
        if (bb <= a) {  // B(t = a, s = bb)
          val = x * rsqrtf(tot(bb) + kNormEps) * (rsqrtf(tot(Q + a) + kNormEps) * p.q_scale);
        } else {        // A(t = bb, s = a)
          val = x * rsqrtf(tot(a) + kNormEps) * rsqrtf(tot(bb) + kNormEps);
        }
      }
      sm.scal[tid] = val;
    }
    __syncthreads();

    // ---------------- row solve (threads 0..127, one state row each) -----
    if (token_half) {
      const int row = tid;
      float u[Q];
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        float acc_t = sm.vv[par][t][row] - sm.xd.dots[t][row] * sm.scal[t];
#pragma unroll
        for (int s = 0; s < t; ++s) acc_t = fmaf(-sm.scal[2 * Q + s * Q + t], u[s], acc_t);
        u[t] = sm.beta[par][t] * acc_t;
      }
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        float o = sm.xd.dots[Q + t][row] * sm.scal[Q + t];
#pragma unroll
        for (int s = 0; s <= t; ++s) o = fmaf(sm.scal[2 * Q + t * Q + s], u[s], o);
        p.out[((tok0 + t) * p.H + it.h) * kDim + row] = f32_to_bf16_bits(o);
      }
      if (it.rec >= 0) {
        const long long cbase = (long long)it.rec * p.corr_row_stride +
                                (long long)it.h * p.rq * kDim + row;
#pragma unroll
        for (int t = 0; t < Q; ++t) p.corr[cbase + t * kDim] = u[t];
      }
      // dots alias xk / xq, which the next item's prologue rewrites
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
  }
}

}  // namespace kda
