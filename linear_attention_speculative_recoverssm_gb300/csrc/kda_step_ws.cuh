// Warp-specialised persistent kernel of the KDA RecoverSSM step: replay of
// the pending recorded tokens into the checkpoint, chunked (WY) verify of
// this window, write-back of S_n and of the new records -- page
// "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.fused", module
// docstring steps 1-3.
//
// One CTA per SM, 384 threads, items (request, head) strided over the grid.
//
//  * Prologue warpgroup (warps 0-3, thread c <-> key channel c) builds each
//    item's operands into one of two shared "ops" buffers, one item ahead of
//    the main warpgroups: the decays of this window and of the recorded
//    tokens, Gamma_t * k_t and Gamma_t * q_t, the replay coefficients
//    k_t * P_t and D_n, the sums of squares and raw A / B pair products
//    reduced over the 128 channels (warp reduce-scatter), the rsqrt norms and
//    normalised pair products, beta, v, and the recorded corrections scaled
//    by their key's rsqrt norm.  It also writes the new key / gate records,
//    after reading the old ones.  Its global loads overlap the main work.
//  * Main warpgroups (warps 4-11): a bulk copy (cp.async.bulk + mbarrier)
//    has brought the item's 64 KB state page into one of NS stages.  Thread
//    (row group rg = 0..15, lane l = 0..15) owns 8 keys of rows rg + 16 i:
//      pass A (n > 0): S_n = S_0 diag(D_n) + sum_t u_t (k_t P_t)^T, stored
//        to HBM and back into the stage in place;
//      pass B: the 2Q dot products of every row with Gamma_t k_t and
//        Gamma_t q_t, the dot vectors held in registers (Q at a time) so the
//        state is the only operand streamed from shared memory; packed FP32
//        FMAs; a reduce-scatter over the 16 lanes of a row;
//      row solve (threads of warpgroup 1, one row each): the forward
//        substitution u_t = beta_t (v_t - w_t - sum_s A_ts u_s), the outputs
//        o_t = y_t + sum_s B_ts u_s (BF16) and the corrections u_t (FP32).
//    When a stage is done the next page is requested into it (NS ahead).
//  * Hand-offs: mbarriers full[stage] (bulk copy landed), opfull[buf] (ops
//    ready), opempty[buf] (ops consumed).  Every wait is bounded; its
//    outcome is made uniform across the warpgroup with bar.red.or, and a
//    timeout is reported in the status word instead of hanging.
#pragma once

#include <cstddef>

#include "kda_step.cuh"

namespace kda {

constexpr int kWsThreads = 384;
constexpr int kBarPro = 1;   // named barrier of the prologue warpgroup
constexpr int kBarMain = 2;  // named barrier of the two main warpgroups

template <int Q>
struct WsRed {
  // reduced per item: sum k_t^2 (Q), sum q_t^2 (Q), sum of the recorded
  // keys' squares (8), then the Q*Q raw pair products
  static constexpr int kRec = 2 * Q;
  static constexpr int kPair = 2 * Q + kMaxQ;
  static constexpr int kN = kPair + Q * Q;
  static constexpr int kPad = round_up(kN, 32);
};

// 16-byte aligned so that ops[1] (and every float4 member) stays aligned.
template <int Q, bool BOUNDARY>
struct alignas(16) WsOps {
  float xk[Q][kDim];  // Gamma_t * k_t (unnormalised)
  float xq[Q][kDim];  // Gamma_t * q_t (unnormalised)
  float kp[kMaxQ][kDim];
  float dn[kDim];
  float kpb[BOUNDARY ? kMaxQ : 1][kDim];
  float db[BOUNDARY ? kDim : 4];
  float u[kMaxQ][kDim];  // recorded u_t[row] * rsqrt norm of its key
  float vv[Q][kDim];
  float beta[kMaxQ];
  // [rsk Q][rsq * q_scale Q][rs of recorded keys 8][pairs Q*Q]
  float scal[WsRed<Q>::kN];
  int meta[8];  // b, h, slot, rec, n, bslot, m
};

template <typename ST>
__host__ __device__ constexpr int ws_stages() {
  return sizeof(ST) == 4 ? 2 : 4;
}

template <int Q, typename ST, bool BOUNDARY>
struct WsSmem {
  static constexpr int NS = ws_stages<ST>();
  ST stage[NS][kDim * kDim];
  WsOps<Q, BOUNDARY> ops[2];
  float dots[kDim][2 * Q + 1];  // [row][w_0..w_Q-1, y_0..y_Q-1] (odd pitch)
  float red[4][WsRed<Q>::kPad];
  uint64_t full[NS];
  uint64_t opfull[2];
  uint64_t opempty[2];
};

// Every member read or written as float4 (or as a bulk-copy target) must sit
// on a 16-byte boundary; the barriers on 8.
template <int Q, typename ST, bool BOUNDARY>
struct WsLayoutCheck {
  using S = WsSmem<Q, ST, BOUNDARY>;
  using O = WsOps<Q, BOUNDARY>;
  static_assert(sizeof(O) % 16 == 0, "ops buffers must stay 16-byte aligned");
  static_assert(offsetof(S, stage) % 128 == 0 && offsetof(S, ops) % 16 == 0, "stage / ops");
  static_assert(offsetof(O, xk) % 16 == 0 && offsetof(O, xq) % 16 == 0 &&
                offsetof(O, kp) % 16 == 0 && offsetof(O, dn) % 16 == 0 &&
                offsetof(O, kpb) % 16 == 0 && offsetof(O, db) % 16 == 0,
                "float4-read ops members");
  static_assert(offsetof(S, full) % 8 == 0 && offsetof(S, opfull) % 8 == 0 &&
                offsetof(S, opempty) % 8 == 0, "mbarriers");
  static constexpr bool ok = true;
};

// The 8 keys of lane l (0..15) in a state row, as two groups of 4: FP32 rows
// are read as 16 B at 4l and at 64 + 4l (each quarter-warp reads 128
// contiguous bytes); BF16 rows as 16 B holding keys 8l .. 8l + 7.
template <typename ST>
struct WsKeys;
template <>
struct WsKeys<float> {
  __device__ static int a(int l) { return 4 * l; }
  __device__ static int b(int l) { return 64 + 4 * l; }
  __device__ static void load(const float *page, int row, int l, float4 &sa, float4 &sb) {
    sa = lds4(page + row * kDim + 4 * l);
    sb = lds4(page + row * kDim + 64 + 4 * l);
  }
};
template <>
struct WsKeys<uint16_t> {
  __device__ static int a(int l) { return 8 * l; }
  __device__ static int b(int l) { return 8 * l + 4; }
  __device__ static void load(const uint16_t *page, int row, int l, float4 &sa, float4 &sb) {
    const uint4 w = *reinterpret_cast<const uint4 *>(page + row * kDim + 8 * l);
    sa = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    sb = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                     __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
  }
};

// Rows whose dot products are reduced together: enough for the 16 lanes.
template <int Q>
struct WsGroup {
  static constexpr int kRows = Q >= 8 ? 2 : (Q >= 4 ? 4 : 8);
  static constexpr int kVals = round_up(kRows * Q, 16);
};

template <int Q, typename ST, bool REPLAY, bool BOUNDARY>
__global__ void __launch_bounds__(kWsThreads, 1)
    kda_step_ws(const StepParams p, int n_items) {
  using Smem = WsSmem<Q, ST, BOUNDARY>;
  using Ops = WsOps<Q, BOUNDARY>;
  static_assert(WsLayoutCheck<Q, ST, BOUNDARY>::ok, "layout");
  constexpr int NS = Smem::NS;
  constexpr uint32_t kPageBytes = kDim * kDim * sizeof(ST);
  constexpr int NR = WsRed<Q>::kN;
  constexpr int NRP = WsRed<Q>::kPad;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int first = blockIdx.x, stride = gridDim.x;
  const int count = first < n_items ? (n_items - first + stride - 1) / stride : 0;

  auto item_slot = [&](int j) {
    const int b = (first + j * stride) / p.H;
    const int s = p.state_slots[b];
    return (s > p.null_slot && s < p.n_slots) ? s : -1;
  };
  // State page of this CTA's j-th item into stage j % NS (thread 128 only).
  auto issue = [&](int j, int slot) {
    uint64_t *bar = &sm.full[j % NS];
    if (slot >= 0) {
      const int h = (first + j * stride) % p.H;
      mbar_arrive_expect_tx(bar, kPageBytes);
      bulk_g2s(sm.stage[j % NS], page_ptr<ST>(p, slot, h), kPageBytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&sm.full[s], 1);
    mbar_init(&sm.opfull[0], 1);
    mbar_init(&sm.opfull[1], 1);
    mbar_init(&sm.opempty[0], 1);
    mbar_init(&sm.opempty[1], 1);
    mbar_init_fence();
  }
  __syncthreads();

  if (warp < 4) {
    // =====================================================================
    // prologue warpgroup: thread c owns key channel c
    // =====================================================================
    const int c = tid;
    for (int j = 0; j < count; ++j) {
      const int item = first + j * stride;
      const ItemMeta it = item_meta<REPLAY, BOUNDARY>(p, item, c == 0);
      Ops &op = sm.ops[j & 1];
      const long long tok0 = (long long)it.b * Q;
      const bool live = it.slot >= 0;

      float kk[Q], qq[Q], vq[Q], gam[Q], inv[Q];
      uint16_t kbits[Q], gbits[Q];
      float kr[kMaxQ], ur[kMaxQ], dr[kMaxQ];
      float braw = 0.f;
      if (live) {
        // ---- global loads of this item (independent, issued together) ----
        const float a = __expf(p.A_log[it.h]);
        const float dt = p.dt_bias[it.h * kDim + c];
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          const long long off = ((tok0 + t) * p.H + it.h) * kDim + c;
          kbits[t] = p.k[off];
          gbits[t] = p.g[off];
          qq[t] = bf16_bits_to_f32(p.q[off]);
          vq[t] = bf16_bits_to_f32(p.v[off]);
        }
        if (c < Q) braw = bf16_bits_to_f32(p.beta[(tok0 + c) * p.H + it.h]);
        const long long cbase = (long long)it.rec * p.corr_row_stride +
                                (long long)it.h * p.rq * kDim + c;
        const long long kbase = (long long)it.rec * p.kg_row_stride +
                                (long long)it.h * p.rq * (2 * kDim) + c;
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          kr[t] = 0.f;
          ur[t] = 0.f;
          dr[t] = 1.f;
          if (REPLAY && t < it.n) {
            ur[t] = p.corr[cbase + t * kDim];
            kr[t] = bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim]);
            dr[t] = gate_decay(a, bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim + kDim]), dt,
                               p.lower_bound);
          }
        }
        float g = 1.f;
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          kk[t] = bf16_bits_to_f32(kbits[t]);
          g *= gate_decay(a, bf16_bits_to_f32(gbits[t]), dt, p.lower_bound);
          gam[t] = g;
          inv[t] = __fdividef(1.f, g);
        }
        // ---- channel reductions, 32 values at a time ----
#pragma unroll
        for (int ch = 0; ch < NRP / 32; ++ch) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int idx = ch * 32 + i;
            float val = 0.f;
            if (idx < Q) {
              val = kk[idx] * kk[idx];
            } else if (idx < 2 * Q) {
              val = qq[idx - Q] * qq[idx - Q];
            } else if (idx < WsRed<Q>::kPair) {
              val = kr[idx - 2 * Q] * kr[idx - 2 * Q];
            } else if (idx < NR) {
              const int pi = idx - WsRed<Q>::kPair;
              const int ra = pi / Q, rb = pi - (pi / Q) * Q;
              if (rb <= ra) {  // B(t = ra, s = rb) = k_s . P(s, t) q_t
                val = kk[rb] * (gam[ra] * inv[rb]) * qq[ra];
              } else {         // A(t = rb, s = ra) = k_s . P(s, t) k_t
                val = kk[ra] * (gam[rb] * inv[ra]) * kk[rb];
              }
            }
            v[i] = val;
          }
          reduce_scatter<32, 32>(v, lane);
          sm.red[warp][ch * 32 + lane] = v[0];
        }
      }

      // ---- the ops buffer of item j - 2 must have been consumed ----
      if (j >= 2) {
        const bool ok = mbar_wait_bounded(&sm.opempty[j & 1], (uint32_t)(((j >> 1) - 1) & 1));
        if (named_bar_or(kBarPro, 128, !ok)) {
          if (c == 0) report(p.status, KDA_ERR_TIMEOUT);
          break;
        }
      }
      if (c == 0) {
        op.meta[0] = it.b;
        op.meta[1] = it.h;
        op.meta[2] = it.slot;
        op.meta[3] = it.rec;
        op.meta[4] = it.n;
        op.meta[5] = it.bslot;
        op.meta[6] = it.m;
      }
      if (live) {
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          op.xk[t][c] = gam[t] * kk[t];
          op.xq[t][c] = gam[t] * qq[t];
          op.vv[t][c] = vq[t];
        }
        if (c < Q) op.beta[c] = sigmoidf_fast(braw);
        if (REPLAY && it.n > 0) {
          float fd = 1.f;
#pragma unroll
          for (int t = kMaxQ - 1; t >= 0; --t) {
            if (t < it.n) {
              op.kp[t][c] = kr[t] * fd;
              fd *= dr[t];
            }
          }
          op.dn[c] = fd;
          if constexpr (BOUNDARY) {
            if (it.bslot >= 0) {
              float fb = 1.f;
#pragma unroll
              for (int t = kMaxQ - 1; t >= 0; --t) {
                if (t < it.m) {
                  op.kpb[t][c] = kr[t] * fb;
                  fb *= dr[t];
                }
              }
              op.db[c] = fb;
            }
          }
        }
        named_bar(kBarPro, 128);
        // ---- final scalars ----
        if (c < NR) {
          auto tot = [&](int i) {
            return (sm.red[0][i] + sm.red[2][i]) + (sm.red[1][i] + sm.red[3][i]);
          };
          const float x = tot(c);
          float val;
          if (c < Q) {
            val = rsqrtf(x + kNormEps);
          } else if (c < 2 * Q) {
            val = rsqrtf(x + kNormEps) * p.q_scale;
          } else if (c < WsRed<Q>::kPair) {
            val = rsqrtf(x + kNormEps);
          } else {
            const int pi = c - WsRed<Q>::kPair;
            const int ra = pi / Q, rb = pi - (pi / Q) * Q;
            if (rb <= ra) {  // B(t = ra, s = rb)
              val = x * rsqrtf(tot(rb) + kNormEps) * (rsqrtf(tot(Q + ra) + kNormEps) * p.q_scale);
            } else {         // A(t = rb, s = ra)
              val = x * rsqrtf(tot(ra) + kNormEps) * rsqrtf(tot(rb) + kNormEps);
            }
          }
          op.scal[c] = val;
        }
        named_bar(kBarPro, 128);
        if (REPLAY) {
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t)
            if (t < it.n) op.u[t][c] = ur[t] * op.scal[WsRed<Q>::kRec + t];
        }
        // New key / gate records: the old ones were read above.
        if (it.rec >= 0) {
          const long long kbase = (long long)it.rec * p.kg_row_stride +
                                  (long long)it.h * p.rq * (2 * kDim) + c;
#pragma unroll
          for (int t = 0; t < Q; ++t) {
            p.kg[kbase + t * 2 * kDim] = kbits[t];
            p.kg[kbase + t * 2 * kDim + kDim] = gbits[t];
          }
        }
      }
      named_bar(kBarPro, 128);
      if (c == 0) mbar_arrive(&sm.opfull[j & 1]);
    }
    return;
  }

  // =======================================================================
  // main warpgroups
  // =======================================================================
  const int mt = tid - 128;
  const int rg = mt >> 4, l = mt & 15;
  const bool leader = mt == 0;
  const int ka = WsKeys<ST>::a(l), kb = WsKeys<ST>::b(l);
  int issued = 0;   // pages requested (leader)
  int consumed = 0;  // items whose page wait was reached
  if (leader) {
    for (; issued < NS && issued < count; ++issued) issue(issued, item_slot(issued));
  }
  for (int j = 0; j < count; ++j) {
    // prefetch the slot of the item whose page will reuse this stage
    int next_slot = -1;
    if (leader && j + NS < count) next_slot = item_slot(j + NS);

    consumed = j;
    bool ok = mbar_wait_bounded(&sm.opfull[j & 1], (uint32_t)((j >> 1) & 1));
    if (named_bar_or(kBarMain, 256, !ok)) {
      if (leader) report(p.status, KDA_ERR_TIMEOUT);
      break;
    }
    const Ops &op = sm.ops[j & 1];
    const int b = op.meta[0], h = op.meta[1], slot = op.meta[2], rec = op.meta[3];
    const int n = op.meta[4], bslot = op.meta[5], m = op.meta[6];
    const long long tok0 = (long long)b * Q;

    if (slot < 0) {
      for (int e = mt; e < Q * kDim; e += 256) {
        const int t = e / kDim, ch = e - t * kDim;
        p.out[((tok0 + t) * p.H + h) * kDim + ch] = 0;
      }
      named_bar(kBarMain, 256);
      if (leader) {
        mbar_arrive(&sm.opempty[j & 1]);
        if (j + NS < count) {
          issue(j + NS, next_slot);
          ++issued;
        }
      }
      consumed = j + 1;  // an inert item's stage phase completed on issue
      continue;
    }

    ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
    if (named_bar_or(kBarMain, 256, !ok)) {
      if (leader) report(p.status, KDA_ERR_TIMEOUT);
      break;
    }
    consumed = j + 1;
    ST *page = sm.stage[j % NS];

    // ---------------- pass A: replay, write-back (n > 0) ----------------
    if constexpr (REPLAY) {
      if (n > 0) {
        float *gpage = reinterpret_cast<float *>(p.state) + (long long)slot * p.slot_stride +
                       (long long)h * (kDim * kDim);
        float *gbnd = nullptr;
        if (BOUNDARY && bslot >= 0)
          gbnd = reinterpret_cast<float *>(p.state) + (long long)bslot * p.slot_stride +
                 (long long)h * (kDim * kDim);
        float4 kpa[kMaxQ], kpb4[kMaxQ];
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          if (t < n) {
            kpa[t] = lds4(&op.kp[t][ka]);
            kpb4[t] = lds4(&op.kp[t][kb]);
          }
        }
        const float4 da = lds4(&op.dn[ka]), dbv = lds4(&op.dn[kb]);
        float *fpage = reinterpret_cast<float *>(page);
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
          const int row = rg + 16 * i;
          const float4 s0a = lds4(fpage + row * kDim + ka);
          const float4 s0b = lds4(fpage + row * kDim + kb);
          if constexpr (BOUNDARY) {
            if (gbnd != nullptr) {
              float4 ba = fmul4(s0a, lds4(&op.db[ka]));
              float4 bb = fmul4(s0b, lds4(&op.db[kb]));
#pragma unroll
              for (int t = 0; t < kMaxQ; ++t) {
                if (t < m) {
                  const float u = op.u[t][row];
                  ba = ffma4s(u, lds4(&op.kpb[t][ka]), ba);
                  bb = ffma4s(u, lds4(&op.kpb[t][kb]), bb);
                }
              }
              stg4(gbnd + row * kDim + ka, ba);
              stg4(gbnd + row * kDim + kb, bb);
            }
          }
          float4 sa = fmul4(s0a, da), sb = fmul4(s0b, dbv);
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t) {
            if (t < n) {
              const float u = op.u[t][row];
              sa = ffma4s(u, kpa[t], sa);
              sb = ffma4s(u, kpb4[t], sb);
            }
          }
          stg4(gpage + row * kDim + ka, sa);
          stg4(gpage + row * kDim + kb, sb);
          sts4(fpage + row * kDim + ka, sa);
          sts4(fpage + row * kDim + kb, sb);
        }
      }
    }

    // ---------------- pass B: 2Q dots per row, Q vectors at a time -------
    constexpr int RB = WsGroup<Q>::kRows;
    constexpr int NV = WsGroup<Q>::kVals;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float4 xa[Q], xb[Q];
#pragma unroll
      for (int jj = 0; jj < Q; ++jj) {
        const float *x = half == 0 ? op.xk[jj] : op.xq[jj];
        xa[jj] = lds4(x + ka);
        xb[jj] = lds4(x + kb);
      }
#pragma unroll 1
      for (int i0 = 0; i0 < 8; i0 += RB) {
        float vals[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) vals[e] = 0.f;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const int row = rg + 16 * (i0 + r);
          float4 sa, sb;
          WsKeys<ST>::load(page, row, l, sa, sb);
#pragma unroll
          for (int jj = 0; jj < Q; ++jj) {
            float2 acc = make_float2(0.f, 0.f);
            acc = dot4_acc(sa, xa[jj], acc);
            acc = dot4_acc(sb, xb[jj], acc);
            vals[r * Q + jj] = acc.x + acc.y;
          }
        }
        reduce_scatter<NV, 16>(vals, l);
#pragma unroll
        for (int e = 0; e < NV / 16; ++e) {
          const int idx = l * (NV / 16) + e;
          if (idx < RB * Q) {
            const int r = idx / Q, jj = idx - (idx / Q) * Q;
            sm.dots[rg + 16 * (i0 + r)][half * Q + jj] = vals[e];
          }
        }
      }
    }
    if (REPLAY && n > 0) fence_proxy_async_smem();  // pass A wrote the stage
    named_bar(kBarMain, 256);  // dots complete, the stage is free
    if (leader && j + NS < count) {
      issue(j + NS, next_slot);
      ++issued;
    }

    // ---------------- row solve: warpgroup 1, one state row each --------
    if (mt < kDim) {
      const int row = mt;
      float u[Q];
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        float a_t = op.vv[t][row] - sm.dots[row][t] * op.scal[t];
#pragma unroll
        for (int s = 0; s < t; ++s)
          a_t = fmaf(-op.scal[WsRed<Q>::kPair + s * Q + t], u[s], a_t);
        u[t] = op.beta[t] * a_t;
      }
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        float o = sm.dots[row][Q + t] * op.scal[Q + t];
#pragma unroll
        for (int s = 0; s <= t; ++s) o = fmaf(op.scal[WsRed<Q>::kPair + t * Q + s], u[s], o);
        p.out[((tok0 + t) * p.H + h) * kDim + row] = f32_to_bf16_bits(o);
      }
      if (rec >= 0) {
        const long long cbase = (long long)rec * p.corr_row_stride +
                                (long long)h * p.rq * kDim + row;
#pragma unroll
        for (int t = 0; t < Q; ++t) p.corr[cbase + t * kDim] = u[t];
      }
    }
    named_bar(kBarMain, 256);  // ops and dots consumed
    if (leader) mbar_arrive(&sm.opempty[j & 1]);
    consumed = j + 1;
  }
  // After a timeout, copies requested but never waited for may still be in
  // flight: let them land (bounded) before this CTA's shared memory goes.
  if (leader) {
    for (int jj = consumed; jj < issued; ++jj)
      mbar_wait_bounded(&sm.full[jj % NS], (uint32_t)((jj / NS) & 1));
  }
}

}  // namespace kda
