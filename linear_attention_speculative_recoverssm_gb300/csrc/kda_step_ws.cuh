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
//    k_t * P_t and D_n, the squared norms of q_t and of the recorded keys
//    reduced over the 128 channels, beta, v, and the recorded corrections
//    scaled by their key's rsqrt norm.  The pair products come from Q rows
//    k_s / Gamma_s dotted with the same vectors as the state rows:
//    A_ts = (k_s / Gamma_s) . (Gamma_t k_t) (s < t), B_ts = (k_s / Gamma_s)
//    . (Gamma_t q_t) (s <= t), and the diagonal (k_s / Gamma_s) . (Gamma_s
//    k_s) is |k_s|^2; the warpgroup normalises them itself.  It also writes
//    the new key / gate records, after reading the old ones.  Its inputs
//    arrive by bulk copies one item ahead, so it never waits on HBM.
//  * Main warpgroups (warps 4-11): a bulk copy (cp.async.bulk + mbarrier)
//    has brought the item's 64 KB state page into one of NS stages.  Thread
//    (row group rg = 0..15, lane l = 0..15) owns 8 keys of rows rg + 16 i:
//      pass A (n > 0): S_n = S_0 diag(D_n) + sum_t u_t (k_t P_t)^T, stored
//        to HBM and back into the stage in place;
//      pass B: the 2Q dot products of every row with Gamma_t k_t and
//        Gamma_t q_t, the dot vectors held in registers (Q at a time) so the
//        state is the only operand streamed from shared memory; packed FP32
//        FMAs; a reduce-scatter over the 16 lanes of a row.  Lanes load
//        their vectors and rows in a lane-XOR-permuted order so the
//        reduce-scatter needs no selects (one shuffle and one add per pair);
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

// Reduced over channels by the prologue per item: sum q_t^2 (Q values),
// then the recorded keys' sums of squares (8 values).
constexpr int kWsRed = 16;

// 16-byte aligned so that ops[1] (and every float4 member) stays aligned.
template <int Q, bool BOUNDARY>
struct alignas(16) WsOps {
  float xk[Q][kDim];  // Gamma_t * k_t (unnormalised)
  float xq[Q][kDim];  // Gamma_t * q_t (unnormalised)
  float ex[Q][kDim];  // k_s / Gamma_s (unnormalised): the pair-product rows
  float kp[kMaxQ][kDim];
  float dn[kDim];
  // boundary: 1 / prod_{m <= s < n} d_s, turning the first m replay terms
  // of S_n's sum into S_m
  float ir[BOUNDARY ? kDim : 4];
  float u[kMaxQ][kDim];  // recorded u_t[row] * rsqrt norm of its key
  float vv[Q][kDim];
  float beta[kMaxQ];
  float rsq[Q];          // rsqrt(|q_t|^2 + eps) * q_scale
  float rsrec[kMaxQ];    // rsqrt(|recorded k_t|^2 + eps)
  float rsk[Q];          // rsqrt(|k_t|^2 + eps)
  float fin_a[Q][Q];     // normalised A_ts (s < t)
  float fin_b[Q][Q];     // normalised B_ts (s <= t)
  int meta[8];  // b, h, slot, rec, n, bslot, m
};

// One item's inputs, staged by bulk copies one item ahead of the prologue.
template <int Q>
struct alignas(16) WsIn {
  uint16_t tok[4][Q][kDim];      // q, k, raw_g, v rows of this window (BF16)
  uint16_t kg[kMaxQ][2 * kDim];  // recorded key / raw gate rows (first n)
  float corr[kMaxQ][kDim];       // recorded corrections (first n)
  int meta[8];                   // b, h, slot, rec, n, bslot, m
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
  WsIn<Q> in[2];
  float dots[kDim][2 * Q + 1];  // [row][w_0..w_Q-1, y_0..y_Q-1] (odd pitch)
  float dots_ex[Q][2 * Q + 1];  // prologue: the pair-product rows' dots
  float red[4][kWsRed];
  uint64_t full[NS];
  uint64_t opfull[2];
  uint64_t opempty[2];
  uint64_t infull[2];
  int next_meta[8];  // resolved index chain of the next item to request
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
                offsetof(O, ex) % 16 == 0 && offsetof(O, ir) % 16 == 0,
                "float4-read ops members");
  static_assert(sizeof(WsIn<Q>) % 16 == 0 && offsetof(S, in) % 16 == 0 &&
                offsetof(WsIn<Q>, tok) % 16 == 0 && offsetof(WsIn<Q>, kg) % 16 == 0 &&
                offsetof(WsIn<Q>, corr) % 16 == 0, "bulk-copy targets");
  static_assert(offsetof(S, full) % 8 == 0 && offsetof(S, opfull) % 8 == 0 &&
                offsetof(S, opempty) % 8 == 0 && offsetof(S, infull) % 8 == 0, "mbarriers");
  static_assert(sizeof(S) <= 232448, "shared memory per CTA");
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

// Rows whose dot products are reduced together.  For Q = 8 a group holds
// 32 values (two per lane after the reduction), for Q = 2 and 4 sixteen:
// then lane l computes value v at position v ^ (l << kShift) and every
// reduction step is a plain shuffle-and-add (kXor).  Other Q reduce with
// per-lane selects.
template <int Q>
struct WsGroup {
  static constexpr int kRows = Q >= 4 ? 4 : 8;
  static constexpr int kVals = round_up(kRows * Q, 16);
  static constexpr bool kXor = (Q == 2 || Q == 4 || Q == 8) && (kRows * Q == 16 || kRows * Q == 32);
  static constexpr int kShift = kRows * Q == 32 ? 1 : 0;
};

// The dots of `rows` state-like rows (RB of them, in the lane-permuted
// order) with Q vectors held in registers, reduced over the 16 lanes of a
// row; `emit(r, jj, value)` receives each finished dot.
template <int Q, typename Load, typename Emit>
__device__ __forceinline__ void ws_dot_group(const float4 (&xa)[Q], const float4 (&xb)[Q],
                                             int l, Load load, Emit emit) {
  using G = WsGroup<Q>;
  constexpr int RB = G::kRows;
  constexpr int NV = G::kVals;
  const int lp = G::kXor ? (l << G::kShift) : 0;
  const int rperm = lp / Q;         // slot r holds row r ^ rperm
  const int xperm = lp & (Q - 1);   // x slot jj holds vector jj ^ xperm (set by the caller)
  (void)xperm;
  float vals[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) vals[e] = 0.f;
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    float4 sa, sb;
    load(r ^ rperm, sa, sb);
#pragma unroll
    for (int jj = 0; jj < Q; ++jj) {
      float2 acc = make_float2(0.f, 0.f);
      acc = dot4_acc(sa, xa[jj], acc);
      acc = dot4_acc(sb, xb[jj], acc);
      vals[r * Q + jj] = acc.x + acc.y;
    }
  }
  if constexpr (G::kXor) {
    constexpr int W = 1 << G::kShift;  // values left per lane
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
#pragma unroll
      for (int i = 0; i < o * W; ++i) vals[i] += __shfl_xor_sync(0xffffffffu, vals[o * W + i], o);
    }
#pragma unroll
    for (int e = 0; e < W; ++e) {
      const int v = lp + e;  // value index: row v / Q, dot v % Q
      emit(v / Q, v & (Q - 1), vals[e]);
    }
  } else {
    reduce_scatter<NV, 16>(vals, l);
#pragma unroll
    for (int e = 0; e < NV / 16; ++e) {
      const int idx = l * (NV / 16) + e;
      if (idx < RB * Q) emit(idx / Q, idx - (idx / Q) * Q, vals[e]);
    }
  }
}

// The x-register permutation that goes with ws_dot_group.
template <int Q>
__device__ __forceinline__ int ws_xperm(int l) {
  using G = WsGroup<Q>;
  return G::kXor ? ((l << G::kShift) & (Q - 1)) : 0;
}

// Pass A for NT pending tokens: S_n = S_0 diag(D_n) + sum_{t<NT} u_t kp_t^T
// on this thread's 8 rows x 8 keys, stored to HBM and back into the stage;
// with a boundary slot, S_m (= the partial sum after m terms times
// 1 / prod_{m<=s<n} d_s) is stored too.  Fully unrolled: no per-token tests.
template <int NT, bool BOUNDARY, typename Ops>
__device__ __forceinline__ void ws_replay_rows(const Ops &op, float *fpage, float *gpage,
                                               float *gbnd, int m, int rg, int ka, int kb) {
#pragma unroll 1
  for (int grp = 0; grp < 2; ++grp) {
    const int key = grp == 0 ? ka : kb;
    float4 kpr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) kpr[t] = lds4(&op.kp[t][key]);
    const float4 d4 = lds4(&op.dn[key]);
    float4 ir4 = make_float4(1.f, 1.f, 1.f, 1.f);
    if (BOUNDARY && gbnd != nullptr) ir4 = lds4(&op.ir[key]);
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
      const int row = rg + 16 * i;
      float u[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) u[t] = op.u[t][row];
      float4 sn = fmul4(lds4(fpage + row * kDim + key), d4);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        sn = ffma4s(u[t], kpr[t], sn);
        if constexpr (BOUNDARY) {
          if (gbnd != nullptr && t == m - 1) stg4(gbnd + row * kDim + key, fmul4(sn, ir4));
        }
      }
      stg4(gpage + row * kDim + key, sn);
      sts4(fpage + row * kDim + key, sn);
    }
  }
}

template <int Q, typename ST, bool REPLAY, bool BOUNDARY>
__global__ void __launch_bounds__(kWsThreads, 1)
    kda_step_ws(const StepParams p, int n_items) {
  using Smem = WsSmem<Q, ST, BOUNDARY>;
  using Ops = WsOps<Q, BOUNDARY>;
  static_assert(WsLayoutCheck<Q, ST, BOUNDARY>::ok, "layout");
  constexpr int NS = Smem::NS;
  constexpr uint32_t kPageBytes = kDim * kDim * sizeof(ST);

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
    mbar_init(&sm.infull[0], 128);  // one asynchronous arrival per prologue thread
    mbar_init(&sm.infull[1], 128);
    mbar_init_fence();
  }
  __syncthreads();

  if (warp < 4) {
    // =====================================================================
    // prologue warpgroup: thread c owns key channel c
    // =====================================================================
    const int c = tid;
    // The index chain slot / record row -> pending count -> records runs two
    // items ahead in thread 0; warp 0 requests item j + 1's inputs while
    // item j is built, so the warpgroup itself never waits on HBM latency.
    int rs_slot = -1, rs_rec = -1, rs_bslot = -1, rs_blen = 0, rs_pend = 0;  // item j + 2
    auto publish_next = [&](const ItemMeta &m) {  // item j + 1, read by warp 0
      sm.next_meta[0] = m.b;
      sm.next_meta[1] = m.h;
      sm.next_meta[2] = m.slot;
      sm.next_meta[3] = m.rec;
      sm.next_meta[4] = m.n;
      sm.next_meta[5] = m.bslot;
      sm.next_meta[6] = m.m;
    };
    auto load_raw = [&](int i) {
      const int b = (first + i * stride) / p.H;
      rs_slot = p.state_slots[b];
      rs_rec = p.record_rows != nullptr ? p.record_rows[b] : b;
      rs_bslot = -1;
      rs_blen = 0;
      if (BOUNDARY && p.bnd_slots != nullptr) {
        rs_bslot = p.bnd_slots[b];
        rs_blen = p.bnd_lens[b];
      }
    };
    auto load_pending = [&]() {
      rs_pend = 0;
      if (REPLAY && rs_rec >= 0 && rs_rec < p.n_rows && rs_slot > p.null_slot &&
          rs_slot < p.n_slots)
        rs_pend = p.pending[rs_rec];
    };
    auto resolve = [&](int i) {  // item_meta from the loaded raw values
      ItemMeta it;
      it.b = (first + i * stride) / p.H;
      it.h = (first + i * stride) - it.b * p.H;
      int slot = rs_slot;
      if (slot >= p.n_slots) {
        report(p.status, KDA_ERR_ARG);
        slot = -1;
      }
      it.slot = slot > p.null_slot ? slot : -1;
      int rec = rs_rec;
      if (rec >= p.n_rows) {
        if (it.slot >= 0) report(p.status, KDA_ERR_ARG);
        rec = -1;
      }
      it.rec = rec;
      it.n = (REPLAY && rec >= 0) ? (rs_pend < 0 ? 0 : (rs_pend > p.rq ? p.rq : rs_pend)) : 0;
      it.bslot = -1;
      it.m = 0;
      if (BOUNDARY && it.n > 0 && p.bnd_slots != nullptr) {
        if (rs_bslot >= p.n_slots) {
          report(p.status, KDA_ERR_ARG);
        } else if (rs_blen > 0 && rs_bslot > p.null_slot) {
          it.bslot = rs_bslot;
          it.m = rs_blen < it.n ? rs_blen : it.n;
        }
      }
      return it;
    };
    // All prologue threads: item i's inputs into in[i & 1] with 16-byte
    // cp.async copies (the load/store path: they do not queue behind the state
    // pages in the bulk-copy engine); each thread then arrives on infull once
    // its own copies have landed.
    auto request_inputs = [&](int i) {
      ItemMeta m;
      m.b = sm.next_meta[0];
      m.h = sm.next_meta[1];
      m.slot = sm.next_meta[2];
      m.rec = sm.next_meta[3];
      m.n = sm.next_meta[4];
      m.bslot = sm.next_meta[5];
      m.m = sm.next_meta[6];
      WsIn<Q> &in = sm.in[i & 1];
      if (c == 0) {
        in.meta[0] = m.b;
        in.meta[1] = m.h;
        in.meta[2] = m.slot;
        in.meta[3] = m.rec;
        in.meta[4] = m.n;
        in.meta[5] = m.bslot;
        in.meta[6] = m.m;
      }
      if (m.slot >= 0) {
        const long long tok0 = (long long)m.b * Q;
        const int nrec = (m.rec >= 0) ? m.n : 0;
        constexpr int kTok = 4 * Q * 16;  // 16-byte chunks of the token rows
        const int total = kTok + nrec * 64;
        for (int e = c; e < total; e += 128) {
          if (e < kTok) {
            const int x = e / (Q * 16), t = (e / 16) % Q, part = e & 15;
            const uint16_t *src = x == 0 ? p.q : (x == 1 ? p.k : (x == 2 ? p.g : p.v));
            cp_async16(&in.tok[x][t][part * 8], src + ((tok0 + t) * p.H + m.h) * kDim + part * 8);
          } else if (e < kTok + nrec * 32) {
            const int f = e - kTok;  // key / gate rows: 32 chunks each
            cp_async16(&in.kg[f >> 5][(f & 31) * 8],
                       p.kg + (long long)m.rec * p.kg_row_stride +
                           (long long)m.h * p.rq * (2 * kDim) + (long long)f * 8);
          } else {
            const int f = e - kTok - nrec * 32;  // corrections: 32 chunks each
            cp_async16(&in.corr[f >> 5][(f & 31) * 4],
                       p.corr + (long long)m.rec * p.corr_row_stride +
                           (long long)m.h * p.rq * kDim + (long long)f * 4);
          }
        }
      }
      cp_async_arrive(&sm.infull[i & 1]);
    };
    // per-head / per-token scalars of an item, prefetched one item ahead
    // (kept raw: converting here would wait for the loads at once)
    float dt_n = 0.f, alog_n = 0.f;
    uint32_t beta_n = 0;
    auto load_small = [&](int i) {
      const int b = (first + i * stride) / p.H;
      const int h = (first + i * stride) - b * p.H;
      dt_n = p.dt_bias[h * kDim + c];
      alog_n = p.A_log[h];
      if (c < Q) beta_n = p.beta[((long long)b * Q + c) * p.H + h];
    };

    int requested = 0;  // items whose inputs were requested (warp 0)
    int taken = 0;      // items whose inputs were waited for
    if (count > 0) {
      requested = 1;
      if (c == 0) {
        load_raw(0);
        load_pending();
        publish_next(resolve(0));
      }
      named_bar(kBarPro, 128);  // next_meta published
      request_inputs(0);
      named_bar(kBarPro, 128);  // next_meta read by every thread
      if (c == 0 && count > 1) {
        load_raw(1);
        load_pending();
        publish_next(resolve(1));
        if (count > 2) load_raw(2);
      }
      named_bar(kBarPro, 128);  // next_meta published
      load_small(0);
    }

    for (int j = 0; j < count; ++j) {
      Ops &op = sm.ops[j & 1];
      const WsIn<Q> &in = sm.in[j & 1];
      const float dt = dt_n, a_log_h = alog_n;
      const uint32_t braw_bits = beta_n;
      if (j + 1 < count) {
        request_inputs(j + 1);
        requested = j + 2;
        load_small(j + 1);
      }
      if (c == 0 && j + 2 < count) load_pending();  // item j + 2 (its row is loaded)

      bool ok = mbar_wait_bounded(&sm.infull[j & 1], (uint32_t)((j >> 1) & 1));
      if (named_bar_or(kBarPro, 128, !ok)) {
        if (c == 0) report(p.status, KDA_ERR_TIMEOUT);
        break;
      }
      taken = j + 1;
      ItemMeta it;
      it.b = in.meta[0];
      it.h = in.meta[1];
      it.slot = in.meta[2];
      it.rec = in.meta[3];
      it.n = in.meta[4];
      it.bslot = in.meta[5];
      it.m = in.meta[6];
      const bool live = it.slot >= 0;

      // (inputs are re-read from the stage where needed: fewer live registers)
      float kk[Q], qq[Q], gam[Q], inv[Q];
      float kr[kMaxQ], dr[kMaxQ];
      const float a = __expf(a_log_h);
      if (live) {
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          kr[t] = 0.f;
          dr[t] = 1.f;
          if (REPLAY && t < it.n) {
            kr[t] = bf16_bits_to_f32(in.kg[t][c]);
            dr[t] = gate_decay(a, bf16_bits_to_f32(in.kg[t][kDim + c]), dt, p.lower_bound);
          }
        }
        float g = 1.f;
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          qq[t] = bf16_bits_to_f32(in.tok[0][t][c]);
          kk[t] = bf16_bits_to_f32(in.tok[1][t][c]);
          g *= gate_decay(a, bf16_bits_to_f32(in.tok[2][t][c]), dt, p.lower_bound);
          gam[t] = g;
          inv[t] = __fdividef(1.f, g);
        }
        // ---- channel reductions: |q_t|^2 and |recorded k_t|^2 ----
        {
          float v[kWsRed];
#pragma unroll
          for (int i = 0; i < kWsRed; ++i) {
            float val = 0.f;
            if (i < Q) val = qq[i] * qq[i];
            else if (i < Q + kMaxQ) val = kr[i - Q] * kr[i - Q];
            v[i] = val;
          }
          reduce_scatter<kWsRed, 16>(v, lane & 15);
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
          if (lane < kWsRed) sm.red[warp][lane] = v[0];
        }
      }
      // thread 0: the index chain of item j + 2, then the row of item j + 3
      if (c == 0 && j + 2 < count) {
        publish_next(resolve(j + 2));
        if (j + 3 < count) load_raw(j + 3);
      }

      // ---- the ops buffer of item j - 2 must have been consumed ----
      if (j >= 2) {
        ok = mbar_wait_bounded(&sm.opempty[j & 1], (uint32_t)(((j >> 1) - 1) & 1));
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
          op.ex[t][c] = kk[t] * inv[t];
          op.vv[t][c] = bf16_bits_to_f32(in.tok[3][t][c]);
        }
        if (c < Q) op.beta[c] = sigmoidf_fast(bf16_bits_to_f32(braw_bits));
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
              float rm = 1.f;  // prod_{m <= s < n} d_s
#pragma unroll
              for (int t = kMaxQ - 1; t >= 0; --t)
                if (t >= it.m && t < it.n) rm *= dr[t];
              op.ir[c] = __fdividef(1.f, rm);
            }
          }
        }
        named_bar(kBarPro, 128);
        // ---- norms of q and of the recorded keys ----
        if (c < Q + kMaxQ) {
          const float x = (sm.red[0][c] + sm.red[2][c]) + (sm.red[1][c] + sm.red[3][c]);
          if (c < Q) op.rsq[c] = rsqrtf(x + kNormEps) * p.q_scale;
          else op.rsrec[c - Q] = rsqrtf(x + kNormEps);
        }
        // ---- raw pair products: rows k_s / Gamma_s dotted with the vectors.
        // The (half, vector chunk) combinations are spread over the four
        // warps; each warp's two row groups hold the Q rows. ----
        {
          constexpr int QV = Q == 8 ? 4 : Q;  // vectors per dot call
          constexpr int RB = WsGroup<QV>::kRows;
          constexpr int NCHUNK = 2 * (Q / QV);  // (half, chunk) combinations
          const int prg = (c >> 4) & 1, pl = c & 15;
          const int pka = WsKeys<float>::a(pl), pkb = WsKeys<float>::b(pl);
          const int xp = ws_xperm<QV>(pl);
#pragma unroll 1
          for (int chunk = warp; chunk < NCHUNK; chunk += 4) {
            const int half = chunk / (Q / QV);
            const int v0 = (chunk - half * (Q / QV)) * QV;  // first vector of the chunk
            float4 xa[QV], xb[QV];
#pragma unroll
            for (int jj = 0; jj < QV; ++jj) {
              const float *x = half == 0 ? op.xk[v0 + (jj ^ xp)] : op.xq[v0 + (jj ^ xp)];
              xa[jj] = lds4(x + pka);
              xb[jj] = lds4(x + pkb);
            }
            // both row groups of the warp run every trip (full-warp shuffles);
            // rows past Q are zeros
#pragma unroll 1
            for (int b2 = 0; b2 < Q; b2 += 2 * RB) {
              const int base = b2 + prg * RB;
              ws_dot_group<QV>(
                  xa, xb, pl,
                  [&](int rr, float4 &sa, float4 &sb) {
                    const int srow = base + rr;
                    if (srow < Q) {
                      sa = lds4(&op.ex[srow][pka]);
                      sb = lds4(&op.ex[srow][pkb]);
                    } else {
                      sa = sb = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                  },
                  [&](int r, int jj, float v) {
                    if (base + r < Q) sm.dots_ex[base + r][half * Q + v0 + jj] = v;
                  });
            }
          }
        }
        named_bar(kBarPro, 128);
        if (REPLAY) {
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t)
            if (t < it.n) op.u[t][c] = in.corr[t][c] * op.rsrec[t];
        }
        if (c < Q * Q) {
          const int t = c / Q, s2 = c - (c / Q) * Q;
          const float rks = rsqrtf(sm.dots_ex[s2][s2] + kNormEps);
          if (s2 < t)
            op.fin_a[t][s2] = sm.dots_ex[s2][t] * rks * rsqrtf(sm.dots_ex[t][t] + kNormEps);
          if (s2 <= t) op.fin_b[t][s2] = sm.dots_ex[s2][Q + t] * rks * op.rsq[t];
          if (s2 == t) op.rsk[t] = rks;
        }
        // New key / gate records: the old ones were read above.
        if (it.rec >= 0) {
          const long long kbase = (long long)it.rec * p.kg_row_stride +
                                  (long long)it.h * p.rq * (2 * kDim) + c;
#pragma unroll
          for (int t = 0; t < Q; ++t) {
            p.kg[kbase + t * 2 * kDim] = in.tok[1][t][c];
            p.kg[kbase + t * 2 * kDim + kDim] = in.tok[2][t][c];
          }
        }
      }
      named_bar(kBarPro, 128);  // in[j & 1] read, ops[j & 1] complete
      if (c == 0) mbar_arrive(&sm.opfull[j & 1]);
    }
    // After a timeout: input copies requested but never waited for must
    // land (bounded) before this CTA's shared memory goes.
    if (c == 0) {
      for (int i = taken; i < requested; ++i)
        mbar_wait_bounded(&sm.infull[i & 1], (uint32_t)((i >> 1) & 1));
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
        // disjoint shared arrays: the stage (read S_0, write S_n in place) and
        // the corrections; saying so lets the loads run ahead of the stores
        float *fpage = reinterpret_cast<float *>(page);
        // n is uniform per item: one predicate-free instance per count
        switch (n) {
          case 1: ws_replay_rows<1, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 2: ws_replay_rows<2, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 3: ws_replay_rows<3, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 4: ws_replay_rows<4, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 5: ws_replay_rows<5, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 6: ws_replay_rows<6, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          case 7: ws_replay_rows<7, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
          default: ws_replay_rows<8, BOUNDARY>(op, fpage, gpage, gbnd, m, rg, ka, kb); break;
        }
      }
    }

    // keep pass B's vector loads from being hoisted into pass A (registers)
    asm volatile("" ::: "memory");
    // ---------------- pass B: 2Q dots per row, Q vectors at a time -------
    {
      constexpr int RB = WsGroup<Q>::kRows;
      const int xp = ws_xperm<Q>(l);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float4 xa[Q], xb[Q];
#pragma unroll
        for (int jj = 0; jj < Q; ++jj) {
          const float *x = half == 0 ? op.xk[jj ^ xp] : op.xq[jj ^ xp];
          xa[jj] = lds4(x + ka);
          xb[jj] = lds4(x + kb);
        }
        const ST *__restrict__ pg = page;                // disjoint from dots
        float *__restrict__ dp = &sm.dots[0][0];
        // unrolled: one group's loads and FMAs overlap the previous group's
        // shuffle chain
#pragma unroll
        for (int i0 = 0; i0 < 8; i0 += RB) {
          ws_dot_group<Q>(
              xa, xb, l,
              [&](int rr, float4 &sa, float4 &sb) {
                WsKeys<ST>::load(pg, rg + 16 * (i0 + rr), l, sa, sb);
              },
              [&](int r, int jj, float v) {
                dp[(rg + 16 * (i0 + r)) * (2 * Q + 1) + half * Q + jj] = v;
              });
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
        float a_t = op.vv[t][row] - sm.dots[row][t] * op.rsk[t];
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) a_t = fmaf(-op.fin_a[t][s2], u[s2], a_t);
        u[t] = op.beta[t] * a_t;
      }
#pragma unroll
      for (int t = 0; t < Q; ++t) {
        float o = sm.dots[row][Q + t] * op.rsq[t];
#pragma unroll
        for (int s2 = 0; s2 <= t; ++s2) o = fmaf(op.fin_b[t][s2], u[s2], o);
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
