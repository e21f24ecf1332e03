// Warp-specialised persistent kernel of the KDA RecoverSSM step: replay of
// the pending recorded tokens into the checkpoint, chunked (WY) verify of
// this window, write-back of S_n and of the new records -- page
// "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.fused", module
// docstring steps 1-3.
//
// One CTA per SM, 384 threads, items (request, head) strided over the grid.
//
//  * Prologue warpgroup (warps 0-3, thread c <-> key channel c) builds each
//    item's operands into one of three shared "ops" buffers, up to three
//    items ahead of the main warpgroups: the decays of this window and of the recorded
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
//    has brought the item's state page into one of NS stages.  Thread (main
//    warp w, lane 8 rs + c) owns rows 16 w + 4 rs .. + 3 and keys 32 i + 4 c
//    .. + 3 (i = 0..3) of them, and reads those 64 values into registers;
//    the last warp to do so requests the next page into the stage.
//      pass A (n > 0): S_n = S_0 diag(D_n) + sum_t u_t (k_t P_t)^T in
//        registers, stored to HBM (and the boundary state S_m);
//      pass B: the 2Q dot products of every row with Gamma_t k_t and
//        Gamma_t q_t straight from those registers, the vectors read from
//        shared memory 8 at a time; packed FP32 FMAs; a reduce-scatter over
//        the 8 lanes of a row group, each lane reading its vectors in a
//        lane-XOR-permuted order so every step is one shuffle and one add;
//      row solve, in registers: the forward substitution u_t = beta_t (v_t -
//        w_t - sum_s A_ts u_s) with u_s broadcast by shuffles within the row
//        group, the outputs o_t = y_t + sum_s B_ts u_s (BF16) and the
//        corrections u_t (FP32).
//    Main warps synchronise only through mbarriers, never a CTA barrier.
//    An inert item's stage phase is a bare arrival; the main warps still
//    wait for it before counting their read of the stage, so a warp that
//    runs ahead cannot count its read among the previous item's.
//  * Windows: request b's window is tokens b*Q .. b*Q + Q - 1, or, in the
//    VARLEN instances, the q_b <= Q tokens query_start_loc[b] .. whose
//    bounds the index chain loads and checks; only the window's tokens get
//    outputs and records.
//  * Hand-offs: mbarriers full[stage] (bulk copy landed), opfull[buf] (ops
//    ready), opempty[buf] (ops consumed by every main warp), and a counter
//    per stage whose eighth reader requests the next page into it.  Every
//    wait is bounded; its outcome is
//    made uniform across the warp (main) or warpgroup (prologue, with
//    bar.red.or), and a timeout is reported in the status word instead of
//    hanging.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <type_traits>

#include "kda_step.cuh"

namespace kda {

constexpr int kWsThreads = 384;
// Registers per thread: launched with 168 (the most 384 threads can have);
// the prologue warpgroup gives some up to the two main warpgroups, whose
// state tile, partial dots and vectors live in registers.  The split adds up
// to the launch total: 128 x 136 + 256 x 184 = 384 x 168.
constexpr int kWsRegsLaunch = 168;
constexpr int kWsRegsProlog = 136;
constexpr int kWsRegsMain = 184;
static_assert(128 * kWsRegsProlog + 256 * kWsRegsMain <= kWsThreads * kWsRegsLaunch,
              "register split exceeds the launch allocation");
constexpr int kBarPro = 1;   // named barrier of the prologue warpgroup
// Operand buffers between the prologue and the main warpgroups: the prologue
// may run up to this many items ahead, which absorbs the per-item jitter of
// either side.
constexpr int kWsOpsBufs = 3;
// The index chain runs in lanes 0 .. kWsChain - 1 of the prologue's warp 0,
// kWsChain items at a time (one per lane), every kWsChain items, into a ring
// of 2 kWsChain slots of meta words.
constexpr int kWsChain = 16;

// Reduced over channels by the prologue per item: sum q_t^2 (Q values),
// then the recorded keys' sums of squares (8 values).
constexpr int kWsRed = 16;

// Dot vectors of the verify, padded to whole groups of 8 (zeros).
template <int Q>
__host__ __device__ constexpr int ws_vectors() {
  return (2 * Q + 7) / 8 * 8;
}

// 16-byte aligned so that ops[1] (and every float4 member) stays aligned.
template <int Q, bool BOUNDARY>
struct alignas(16) WsOps {
  // x[t] = Gamma_t * k_t and x[Q + t] = Gamma_t * q_t (unnormalised), then
  // zero rows up to a multiple of 8 (written once, at kernel start)
  float x[ws_vectors<Q>()][kDim];
  float kp[kMaxQ][kDim];
  float dn[kDim];
  // boundary: 1 / prod_{m <= s < n} d_s, turning the first m replay terms
  // of S_n's sum into S_m
  float ir[BOUNDARY ? kDim : 4];
  float u[kMaxQ][kDim];  // recorded u_t[row] * rsqrt norm of its key
  uint16_t vv[Q][kDim];  // v_t[row] (BF16 bits, as staged)
  float beta[kMaxQ];
  float rsq[Q];          // rsqrt(|q_t|^2 + eps) * q_scale
  float rsrec[kMaxQ];    // rsqrt(|recorded k_t|^2 + eps)
  float rsk[Q];          // rsqrt(|k_t|^2 + eps)
  float fin_a[Q][Q];     // normalised A_ts (s < t), 0 for s >= t
  float fin_b[Q][Q];     // normalised B_ts (s <= t), 0 for s > t
  alignas(16) int meta[8];  // b (tok0 with VARLEN), h, slot, rec, n, bslot, m, qb (VARLEN)
};

// Tensor maps of the four token-major BF16 inputs [B*Q, H, 128], in the
// order q, k, raw_g, v, each as a 3-D tensor (128 channels, H heads, B*Q
// tokens) whose (128, 1, Q) box is one item's rows of the window.
struct WsMaps {
  CUtensorMap tok[4];
};

// The multi-layer instances take the layers' bases (LayerBases) as a kernel
// parameter; the others an empty stand-in.
template <bool LAYERS>
struct WsLayers {
  int unused;
};
template <>
struct WsLayers<true> : LayerBases {};

// One item's inputs, staged by tensor / bulk copies one item ahead of the
// prologue (128-byte aligned: tensor-copy destinations).
template <int Q>
struct alignas(128) WsIn {
  uint16_t tok[4][Q][kDim];      // q, k, raw_g, v rows of this window (BF16)
  uint16_t kg[kMaxQ][2 * kDim];  // recorded key / raw gate rows (first n)
  float corr[kMaxQ][kDim];       // recorded corrections (first n)
  alignas(16) int meta[8];       // as in WsOps
};

template <typename ST>
__host__ __device__ constexpr int ws_stages() {
  return sizeof(ST) == 4 ? 2 : 4;
}

template <int Q, typename ST, bool BOUNDARY>
struct WsSmemBase {
  static constexpr int NS = ws_stages<ST>();
  ST stage[NS][kDim * kDim];
  WsOps<Q, BOUNDARY> ops[kWsOpsBufs];
  WsIn<Q> in[2];
  float ex[Q][kDim];            // prologue: k_s / Gamma_s, the pair-product rows
  float dots_ex[Q][2 * Q + 1];  // prologue: the pair-product rows' dots
  float red[4][kWsRed];
  uint64_t full[NS];
  uint32_t sreads[NS];  // main-warp reads of each stage (8 per use)
  uint64_t opfull[kWsOpsBufs];
  uint64_t opempty[kWsOpsBufs];
  uint64_t infull[2];
  // the resolved index chain of item i in slot i % (2 kWsChain)
  alignas(16) int meta_ring[2 * kWsChain][8];
};

// The NORM instances add the folded gated RMSNorm's exchange: each main
// warp's sum of squares of its 16 rows of every token's outputs, per ops
// buffer, completed on nred[buf] (one arrival per main warp); and the norm
// weights.
template <int Q, typename ST, bool BOUNDARY>
struct WsSmemNorm : WsSmemBase<Q, ST, BOUNDARY> {
  uint64_t nred[kWsOpsBufs];
  alignas(16) float nsq[kWsOpsBufs][kMaxQ][8];  // [buf][token][main warp]
  alignas(16) float norm_w[kDim];  // read as float4
};

template <int Q, typename ST, bool BOUNDARY, bool NORM = false>
using WsSmem = std::conditional_t<NORM, WsSmemNorm<Q, ST, BOUNDARY>, WsSmemBase<Q, ST, BOUNDARY>>;

// Every member read or written as float4 (or as a bulk-copy target) must sit
// on a 16-byte boundary; the barriers on 8.
template <int Q, typename ST, bool BOUNDARY>
struct WsLayoutCheck {
  using S = WsSmemBase<Q, ST, BOUNDARY>;
  using SN = WsSmemNorm<Q, ST, BOUNDARY>;
  using O = WsOps<Q, BOUNDARY>;
  static_assert(sizeof(O) % 16 == 0, "ops buffers must stay 16-byte aligned");
  static_assert(offsetof(S, stage) % 128 == 0 && offsetof(S, ops) % 16 == 0, "stage / ops");
  static_assert(offsetof(O, x) % 16 == 0 && offsetof(O, u) % 16 == 0 &&
                offsetof(O, vv) % 16 == 0 &&
                offsetof(O, kp) % 16 == 0 && offsetof(O, dn) % 16 == 0 &&
                offsetof(O, vv) % 8 == 0 && offsetof(O, ir) % 16 == 0 &&
                offsetof(S, ex) % 16 == 0,
                "float4-read ops members");
  static_assert(sizeof(WsIn<Q>) % 128 == 0 && offsetof(S, in) % 128 == 0 &&
                offsetof(WsIn<Q>, tok) % 16 == 0 && offsetof(WsIn<Q>, kg) % 16 == 0 &&
                offsetof(WsIn<Q>, corr) % 16 == 0, "bulk-copy targets");
  static_assert(offsetof(S, full) % 8 == 0 && offsetof(S, opfull) % 8 == 0 &&
                offsetof(S, opempty) % 8 == 0 && offsetof(S, infull) % 8 == 0, "mbarriers");
  static_assert(offsetof(SN, nred) % 8 == 0 && offsetof(SN, norm_w) % 16 == 0 &&
                offsetof(SN, nsq) % 16 == 0 &&
                sizeof(SN) <= 232448, "the norm's barriers and float4-read weights");
  static_assert(sizeof(S) <= 232448, "shared memory per CTA");
  static constexpr bool ok = true;
};

// The prologue's pair-product dots: lane l (0..15) of a row takes the 8 keys
// 4l .. 4l + 3 and 64 + 4l .. 64 + 4l + 3 (each quarter-warp reads 128
// contiguous bytes).
struct WsKeys {
  __device__ static int a(int l) { return 4 * l; }
  __device__ static int b(int l) { return 64 + 4 * l; }
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

// ---------------------------------------------------------------------------
// Main warpgroups.  Thread (main warp w = 0..7, lane = 8 rs + c) owns state
// rows R0 .. R0 + 3 with R0 = 16 w + 4 rs, and the 16 keys 32 i + 4 c .. + 3
// (i = 0..3) of each: every warp access to a key chunk covers 128 contiguous
// bytes per row, and the 8 lanes c of a row group split the 128 keys.
// ---------------------------------------------------------------------------

// The thread's 4 x 16 state values from a stage (FP32 or BF16 page).
template <typename ST>
struct WsTile;
template <>
struct WsTile<float> {
  __device__ static void load(const float *page, int R0, int c, float4 (&s)[4][4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[r][i] = lds4(page + (R0 + r) * kDim + 32 * i + 4 * c);
  }
};
template <>
struct WsTile<uint16_t> {
  __device__ static void load(const uint16_t *page, int R0, int c, float4 (&s)[4][4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint2 w = *reinterpret_cast<const uint2 *>(page + (R0 + r) * kDim + 32 * i + 4 * c);
        s[r][i] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                              __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
      }
  }
};

// Pass A for NT pending tokens, in registers:
// S_n = S_0 diag(D_n) + sum_{t<NT} u_t kp_t^T, stored to HBM; with a boundary
// slot, S_m (= the partial sum after m terms times 1 / prod_{m<=s<n} d_s) is
// stored too.  Fully unrolled: no per-token tests but the boundary's.
template <int NT, bool BOUNDARY, typename Ops>
__device__ __forceinline__ void ws_replay(float4 (&s)[4][4], const Ops &op, float *gpage,
                                          float *gbnd, int m, int R0, int c) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 d4 = lds4(&op.dn[32 * i + 4 * c]);
#pragma unroll
    for (int r = 0; r < 4; ++r) s[r][i] = fmul4(s[r][i], d4);
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float4 u4 = lds4(&op.u[t][R0]);
    const float ur[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 k4 = lds4(&op.kp[t][32 * i + 4 * c]);
#pragma unroll
      for (int r = 0; r < 4; ++r) s[r][i] = ffma4s(ur[r], k4, s[r][i]);
    }
    if constexpr (BOUNDARY) {
      if (gbnd != nullptr && t == m - 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 ir4 = lds4(&op.ir[32 * i + 4 * c]);
#pragma unroll
          for (int r = 0; r < 4; ++r)
            stg4(gbnd + (R0 + r) * kDim + 32 * i + 4 * c, fmul4(s[r][i], ir4));
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) stg4(gpage + (R0 + r) * kDim + 32 * i + 4 * c, s[r][i]);
}

// Pass B: the dots of the thread's 4 rows with the dot vectors, 8 vectors
// (one group) at a time, reduced over the 8 lanes c of the row group.  Lane
// c takes vector 8 g + (j ^ c) in register slot j, so value (slot j, row r)
// at position 4 j + r is the logical value (4 j + r) ^ 4 c, and every step of
// the reduce-scatter is one shuffle and one add; lane c ends with the dots
// of vector 8 g + c with its 4 rows: d[g][r].
template <int NG>
__device__ __forceinline__ void ws_dots(const float4 (&s)[4][4], const float *__restrict__ xv,
                                        int c, float (&d)[NG][4]) {
  // vectors of the next slot are loaded while the current slot's FMAs run
  auto load_slot = [&](int v, float4 (&x4)[4]) {
    const float *x = xv + (8 * (v >> 3) + ((v & 7) ^ c)) * kDim + 4 * c;
#pragma unroll
    for (int i = 0; i < 4; ++i) x4[i] = lds4(x + 32 * i);
  };
  float4 xa[4], xb[4];
  load_slot(0, xa);
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float p[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int v = 8 * g + j;
      float4(&cur)[4] = (v & 1) ? xb : xa;
      float4(&nxt)[4] = (v & 1) ? xa : xb;
      if (v + 1 < 8 * NG) load_slot(v + 1, nxt);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float2 acc = fmul2(make_float2(s[r][0].x, s[r][0].y), make_float2(cur[0].x, cur[0].y));
        acc = ffma2(make_float2(s[r][0].z, s[r][0].w), make_float2(cur[0].z, cur[0].w), acc);
#pragma unroll
        for (int i = 1; i < 4; ++i) acc = dot4_acc(s[r][i], cur[i], acc);
        p[4 * j + r] = acc.x + acc.y;
      }
    }
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) {
#pragma unroll
      for (int i = 0; i < 4 * o; ++i) p[i] += __shfl_xor_sync(0xffffffffu, p[4 * o + i], o);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) d[g][r] = p[r];
  }
}

// Row solve of the thread's 4 rows, in registers.  After pass B lane c
// holds w_c (c < Q) in group 0 and y_t for t = 8 g + c - Q (when that is in
// 0 .. Q-1) in group g.  For s = 0 .. Q-1 the lane holding w_s has finished
// its residual v_s - w_s rsk_s - sum_{s'<s} A_ss' u_s'; u_s = beta_s times it
// is broadcast to the row group and folded into every lane's residual (the
// A coefficient is 0 for s >= t) and outputs (the B coefficient is 0 for
// s > t).  Writes o_t (BF16) and, with a record row, u_t (FP32).
// NORM: the outputs are not stored; the lane's BF16-rounded outputs (at
// most one token per lane) go to obf / tout (-1: none) for the norm.
template <int Q, int NG, bool VARLEN, bool NORM, typename Ops>
__device__ __forceinline__ void ws_solve(const float (&d)[NG][4], const Ops &op,
                                         const StepParams &p, uint16_t *out, float *corr,
                                         long long corr_row_stride, long long tok0, int qb,
                                         int h, int rec, int R0, int c, int lane,
                                         float (&obf)[4], int &tout) {
  const int cw = c < Q ? c : Q - 1;  // lanes without a w role compute unused values
  const uint2 vb = *reinterpret_cast<const uint2 *>(&op.vv[cw][R0]);
  const float4 v4 = make_float4(__uint_as_float(vb.x << 16), __uint_as_float(vb.x & 0xffff0000u),
                                __uint_as_float(vb.y << 16), __uint_as_float(vb.y & 0xffff0000u));
  const float rk = op.rsk[cw], bt = op.beta[cw];
  float res[4] = {fmaf(-d[0][0], rk, v4.x), fmaf(-d[0][1], rk, v4.y), fmaf(-d[0][2], rk, v4.z),
                  fmaf(-d[0][3], rk, v4.w)};
  float acoef[Q];
#pragma unroll
  for (int s2 = 0; s2 < Q; ++s2) acoef[s2] = op.fin_a[cw][s2];
  bool hy[NG];
  int ty[NG];
  float oacc[NG][4], bcoef[NG][Q];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int V = 8 * g + c;
    hy[g] = V >= Q && V < 2 * Q;
    ty[g] = hy[g] ? V - Q : 0;
    const float rq = op.rsq[ty[g]];
#pragma unroll
    for (int r = 0; r < 4; ++r) oacc[g][r] = d[g][r] * rq;
#pragma unroll
    for (int s2 = 0; s2 < Q; ++s2) bcoef[g][s2] = op.fin_b[ty[g]][s2];
  }
  const int base = lane & ~7;
#pragma unroll
  for (int s2 = 0; s2 < Q; ++s2) {
    float us[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) us[r] = __shfl_sync(0xffffffffu, bt * res[r], base + s2);
#pragma unroll
    for (int r = 0; r < 4; ++r) res[r] = fmaf(-acoef[s2], us[r], res[r]);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int r = 0; r < 4; ++r) oacc[g][r] = fmaf(bcoef[g][s2], us[r], oacc[g][r]);
  }
  if constexpr (NORM) {
    tout = -1;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if (hy[g]) {  // (a lane holds at most one output token)
        tout = ty[g];
#pragma unroll
        for (int r = 0; r < 4; ++r) obf[r] = bf16_bits_to_f32(f32_to_bf16_bits(oacc[g][r]));
      }
    }
  } else {
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if (hy[g] && (!VARLEN || ty[g] < qb)) {
        const uint2 o2 = make_uint2(pack_bf16x2(oacc[g][0], oacc[g][1]),
                                    pack_bf16x2(oacc[g][2], oacc[g][3]));
        *reinterpret_cast<uint2 *>(out + ((tok0 + ty[g]) * p.H + h) * kDim + R0) = o2;
      }
    }
  }
  if ((VARLEN ? c < qb : c < Q) && rec >= 0) {
    const long long cbase = (long long)rec * corr_row_stride + ((long long)h * p.rq + c) * kDim;
    stg4(corr + cbase + R0, make_float4(bt * res[0], bt * res[1], bt * res[2], bt * res[3]));
  }
}

// VARLEN: windows from query_start_loc (p.qsl, non-null), each of q_b <= Q
// tokens; otherwise request b's window is tokens b*Q .. b*Q + Q - 1.  The
// meta words carry b (uniform) or the window's first token and length.
// LAYERS: items (layer, request, head) over the layers of `lay` (uniform
// windows, FP32 state, no boundary states); the meta words carry the layer
// in place of the window length.
// NORM: the model layer's gated RMSNorm folded into the row solve (uniform
// windows, FP32 state, no boundary states): the main warps exchange their
// rows' sums of squares per token through shared memory (nred), and write
// the normed, gated outputs instead of o.
template <int Q, typename ST, bool REPLAY, bool BOUNDARY, bool VARLEN, bool LAYERS,
          bool NORM = false>
__global__ void __launch_bounds__(kWsThreads, 1)
    kda_step_ws(const StepParams p, const __grid_constant__ WsMaps maps,
                const __grid_constant__ WsLayers<LAYERS> lay, int n_items) {
  static_assert(!LAYERS || (!VARLEN && !BOUNDARY && REPLAY && sizeof(ST) == 4),
                "the multi-layer step: uniform windows, FP32 state, no boundary");
  static_assert(!NORM || (!VARLEN && !BOUNDARY && !LAYERS && REPLAY && sizeof(ST) == 4),
                "the folded norm: uniform windows, FP32 state, one layer, no boundary");
  using Smem = WsSmem<Q, ST, BOUNDARY, NORM>;
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

  // item index -> request and layer (layer-major over LAYERS' layers)
  auto req_of = [&](int idx) { return LAYERS ? (idx / p.H) % p.B : idx / p.H; };
  auto layer_of = [&](int idx) { return LAYERS ? idx / (p.H * p.B) : 0; };
  auto item_slot = [&](int j) {
    const int b = req_of(first + j * stride);
    const int s = p.state_slots[b];
    return (s > p.null_slot && s < p.n_slots) ? s : -1;
  };
  // State page of this CTA's j-th item into stage j % NS (thread 128 only).
  auto issue = [&](int j, int slot) {
    uint64_t *bar = &sm.full[j % NS];
    if (slot >= 0) {
      const int h = (first + j * stride) % p.H;
      mbar_arrive_expect_tx(bar, kPageBytes);
      if constexpr (LAYERS) {
        const int l = layer_of(first + j * stride);
        const float *page = reinterpret_cast<const float *>(lay.state[l]) +
                            (long long)slot * lay.slot_stride[l] + (long long)h * (kDim * kDim);
        bulk_g2s(sm.stage[j % NS], page, kPageBytes, bar);
      } else {
        bulk_g2s(sm.stage[j % NS], page_ptr<ST>(p, slot, h), kPageBytes, bar);
      }
    } else {
      mbar_arrive(bar);
    }
  };

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      sm.sreads[s] = 0;
    }
    for (int b = 0; b < kWsOpsBufs; ++b) {
      mbar_init(&sm.opfull[b], 1);
      mbar_init(&sm.opempty[b], 8);  // one arrival per main warp
    }
    mbar_init(&sm.infull[0], 1);  // thread 0's arrival with the copies' byte count
    mbar_init(&sm.infull[1], 1);
    if constexpr (NORM) {
      for (int b = 0; b < kWsOpsBufs; ++b) mbar_init(&sm.nred[b], 8);  // one per main warp
    }
    mbar_init_fence();
  }
  if constexpr (NORM) {
    if (tid < kDim) sm.norm_w[tid] = p.norm_w[tid];
  }
  // the padding dot vectors (rows 2Q .. of x) stay zero in both ops buffers
  constexpr int kPadFloats = (ws_vectors<Q>() - 2 * Q) * kDim;
  if constexpr (kPadFloats > 0) {
    for (int e = tid; e < kWsOpsBufs * kPadFloats; e += kWsThreads)
      sm.ops[e / kPadFloats].x[2 * Q + (e % kPadFloats) / kDim][e % kDim] = 0.f;
  }
  __syncthreads();

  if (warp < 4) {
    warpgroup_reg_dealloc<kWsRegsProlog>();
    // =====================================================================
    // prologue warpgroup: thread c owns key channel c
    // =====================================================================
    const int c = tid;
    // The index chain slot / record row -> pending count -> records runs two
    // items ahead in thread 0; thread 32 requests item j + 1's inputs while
    // item j is built, so the warpgroup itself never waits on HBM latency.
    // Raw per-request values of an item (no branch on them, so the loads stay
    // in flight) and its pending count, loaded a step later from its row.
    struct Raw {
      int slot = -1, rec = -1, bslot = -1, blen = 0, pend = 0, q0 = 0, q1 = 0;
    };
    // Lane l < kWsChain of warp 0 resolves item g kWsChain + l of every
    // group g: ra holds the row and pending count of its item in the next
    // group to resolve, rb the row of its item in the group after.
    Raw ra, rb;
    auto publish = [&](int i, const ItemMeta &m) {
      int *w = sm.meta_ring[i % (2 * kWsChain)];
      w[0] = VARLEN ? m.tok0 : m.b;
      w[1] = m.h;
      w[2] = m.slot;
      w[3] = m.rec;
      w[4] = m.n;
      w[5] = m.bslot;
      w[6] = m.m;
      w[7] = VARLEN ? m.qb : (LAYERS ? m.l : 0);
    };
    auto load_raw = [&](int i, Raw &r) {
      const int b = req_of(first + i * stride);
      r.slot = p.state_slots[b];
      r.rec = p.record_rows != nullptr ? p.record_rows[b] : b;
      r.bslot = -1;
      r.blen = 0;
      if (BOUNDARY && p.bnd_slots != nullptr) {
        r.bslot = p.bnd_slots[b];
        r.blen = p.bnd_lens[b];
      }
      r.pend = 0;
    };
    // item i's pending count and (VARLEN) window bounds, a step after its row
    auto load_pending = [&](int i, Raw &r) {
      r.pend = 0;
      if (REPLAY && r.rec >= 0 && r.rec < p.n_rows && r.slot > p.null_slot && r.slot < p.n_slots)
        r.pend = p.pending[r.rec];
      if constexpr (VARLEN) {
        const int b = div_heads(p, first + i * stride);
        r.q0 = p.qsl[b];
        r.q1 = p.qsl[b + 1];
      }
    };
    auto resolve = [&](int i, const Raw &r) {  // item_meta from the loaded raw values
      const int rs_slot = r.slot, rs_rec = r.rec, rs_bslot = r.bslot, rs_blen = r.blen,
                rs_pend = r.pend;
      ItemMeta it;
      if constexpr (LAYERS) {
        it.b = req_of(first + i * stride);
        it.h = (first + i * stride) % p.H;
        it.l = layer_of(first + i * stride);
      } else {
        it.b = div_heads(p, first + i * stride);
        it.h = (first + i * stride) - it.b * p.H;
        it.l = 0;
      }
      int slot = rs_slot;
      if (slot >= p.n_slots) {
        report(p.status, KDA_ERR_ARG);
        slot = -1;
      }
      it.slot = slot > p.null_slot ? slot : -1;
      it.tok0 = it.b * Q;
      it.qb = Q;
      if constexpr (VARLEN) {
        if (window_ok(p, r.q0, r.q1, Q)) {
          it.tok0 = r.q0;
          it.qb = r.q1 - r.q0;
        } else {  // nothing of the request is read or written
          report(p.status, KDA_ERR_ARG);
          it.slot = -1;
          it.tok0 = 0;
          it.qb = 0;
        }
      }
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
    // Thread 32 (warp 1: warp 0's lanes run the index chain): item i's
    // inputs into in[i & 1]: the window's q, k, raw_g and v rows by four
    // tensor copies, the first n recorded key / gate rows and corrections by
    // one bulk copy each, all completing on infull[i & 1].
    auto request_inputs = [&](int i) {
      if (c != 32) return;
      // the meta words move 16 bytes at a time: the ring slot and in.meta
      // have the same layout
      const int4 *w4 = reinterpret_cast<const int4 *>(sm.meta_ring[i % (2 * kWsChain)]);
      const int4 w0 = w4[0], w1 = w4[1];
      ItemMeta m;
      m.b = m.tok0 = w0.x;
      m.h = w0.y;
      m.slot = w0.z;
      m.rec = w0.w;
      m.n = w1.x;
      m.bslot = w1.y;
      m.m = w1.z;
      m.qb = VARLEN ? w1.w : Q;
      m.l = LAYERS ? w1.w : 0;
      WsIn<Q> &in = sm.in[i & 1];
      reinterpret_cast<int4 *>(in.meta)[0] = w0;
      reinterpret_cast<int4 *>(in.meta)[1] = w1;
      uint64_t *bar = &sm.infull[i & 1];
      if (m.slot < 0) {
        mbar_arrive(bar);
        return;
      }
      const int nrec = (m.rec >= 0) ? m.n : 0;
      constexpr uint32_t kTokBytes = 4u * Q * kDim * 2u;
      const uint32_t rec_bytes = (uint32_t)nrec * kDim * 4u;  // per record tensor
      mbar_arrive_expect_tx(bar, kTokBytes + 2u * rec_bytes);
#pragma unroll
      // (rows past the window or the activations arrive as zeros or as other
      // requests' tokens; nothing computed from them is written)
      for (int x = 0; x < 4; ++x) {
        if constexpr (LAYERS)
          tma_load_4d(&in.tok[x][0][0], &maps.tok[x], 0, m.h, m.b * Q, m.l, bar);
        else
          tma_load_3d(&in.tok[x][0][0], &maps.tok[x], 0, m.h, VARLEN ? m.tok0 : m.b * Q, bar);
      }
      if (nrec > 0) {
        const uint16_t *kg = p.kg;
        const float *corr = p.corr;
        long long kgs = p.kg_row_stride, cs = p.corr_row_stride;
        if constexpr (LAYERS) {
          kg = reinterpret_cast<const uint16_t *>(lay.kg[m.l]);
          corr = reinterpret_cast<const float *>(lay.corr[m.l]);
          kgs = lay.kg_stride[m.l];
          cs = lay.corr_stride[m.l];
        }
        bulk_g2s(&in.kg[0][0], kg + (long long)m.rec * kgs + (long long)m.h * p.rq * (2 * kDim),
                 rec_bytes, bar);
        bulk_g2s(&in.corr[0][0], corr + (long long)m.rec * cs + (long long)m.h * p.rq * kDim,
                 rec_bytes, bar);
      }
    };
    // per-head / per-token scalars of an item, prefetched one item ahead
    // (kept raw: converting here would wait for the loads at once)
    float dt_n = 0.f, alog_n = 0.f;
    uint32_t beta_n = 0;
    // (with VARLEN item i's window is read from its meta words)
    auto load_small = [&](int i) {
      if constexpr (LAYERS) {
        const int idx = first + i * stride;
        const int b = req_of(idx), h = idx % p.H, l = layer_of(idx);
        dt_n = p.dt_bias[((long long)l * p.H + h) * kDim + c];
        alog_n = p.A_log[l * p.H + h];
        beta_n = 0;
        if (c < Q) beta_n = p.beta[l * lay.beta_stride + ((long long)b * Q + c) * p.H + h];
        return;
      }
      const int b = div_heads(p, first + i * stride);
      const int h = (first + i * stride) - b * p.H;
      dt_n = p.dt_bias[h * kDim + c];
      alog_n = p.A_log[h];
      if constexpr (VARLEN) {
        const int *w = sm.meta_ring[i % (2 * kWsChain)];
        const long long tok = w[0];
        beta_n = 0;
        if (c < w[7]) beta_n = p.beta[(tok + c) * p.H + h];
      } else {
        if (c < Q) beta_n = p.beta[((long long)b * Q + c) * p.H + h];
      }
    };

    int requested = 0;  // items whose inputs were requested (thread 32)
    int taken = 0;      // items whose inputs were waited for
    if (count > 0) {
      requested = 1;
      // groups 0 and 1 resolved now; group 2's rows and pending counts and
      // group 3's rows loaded for the first turns below
      if (c < kWsChain) {
        for (int g = 0; g < 2; ++g) {
          const int i = g * kWsChain + c;
          if (i < count) {
            Raw r0;
            load_raw(i, r0);
            load_pending(i, r0);
            publish(i, resolve(i, r0));
          }
        }
        if (2 * kWsChain + c < count) {
          load_raw(2 * kWsChain + c, ra);
          load_pending(2 * kWsChain + c, ra);
        }
        if (3 * kWsChain + c < count) load_raw(3 * kWsChain + c, rb);
      }
      named_bar(kBarPro, 128);  // groups 0 and 1 published
      request_inputs(0);
      load_small(0);
    }

    for (int j = 0; j < count; ++j) {
      Ops &op = sm.ops[j % kWsOpsBufs];
      const WsIn<Q> &in = sm.in[j & 1];
      const float dt = dt_n, a_log_h = alog_n;
      const uint32_t braw_bits = beta_n;
      if (j + 1 < count) {
        request_inputs(j + 1);
        requested = j + 2;
        load_small(j + 1);
      }

      bool ok = mbar_wait_bounded(&sm.infull[j & 1], (uint32_t)((j >> 1) & 1));
      if (named_bar_or(kBarPro, 128, !ok)) {
        if (c == 0) report(p.status, KDA_ERR_TIMEOUT);
        break;
      }
      taken = j + 1;
      ItemMeta it;
      const int4 im0 = reinterpret_cast<const int4 *>(in.meta)[0];
      const int4 im1 = reinterpret_cast<const int4 *>(in.meta)[1];
      it.b = im0.x;
      it.h = im0.y;
      it.slot = im0.z;
      it.rec = im0.w;
      it.n = im1.x;
      it.bslot = im1.y;
      it.m = im1.z;
      it.qb = VARLEN ? im1.w : Q;
      it.l = LAYERS ? im1.w : 0;
      const bool live = it.slot >= 0;

      // (inputs are re-read from the stage where needed: fewer live registers)
      float kk[Q], qq[Q], gam[Q], inv[Q];
      float kr[kMaxQ], dr[kMaxQ];
      // the decay d = exp(lb sigmoid(a (g + dt))) as 2^(lb log2(e) / (1 +
      // 2^(-a log2(e) (g + dt)))), with this channel's constants folded once
      const float al = __expf(a_log_h) * kLog2e;
      const float e1 = -al, e0 = -al * dt, lbl = p.lower_bound * kLog2e;
      auto decay_of = [&](float graw) {
        const float e = exp2f_fast(fmaf(e1, graw, e0));
        return exp2f_fast(lbl * __fdividef(1.f, 1.f + e));
      };
      if (live) {
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          kr[t] = 0.f;
          dr[t] = 1.f;
        }
        if (REPLAY) {
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t) {
            if (t >= it.n) break;
            kr[t] = bf16_bits_to_f32(in.kg[t][c]);
            dr[t] = decay_of(bf16_bits_to_f32(in.kg[t][kDim + c]));
          }
        }
        float g = 1.f;
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          qq[t] = bf16_bits_to_f32(in.tok[0][t][c]);
          kk[t] = bf16_bits_to_f32(in.tok[1][t][c]);
          g *= decay_of(bf16_bits_to_f32(in.tok[2][t][c]));
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
      // lanes 0 .. kWsChain - 1: every kWsChain items, group g = j /
      // kWsChain + 1 resolved (it is first requested an item before its
      // first item); then the pending counts of group g + 1 and the rows of
      // group g + 2 are loaded, each used a whole group later
      if (c < kWsChain && j >= kWsChain && j % kWsChain == 0) {
        const int g = j / kWsChain + 1;
        const int i = g * kWsChain + c;
        if (i < count) publish(i, resolve(i, ra));
        ra = rb;
        if (i + kWsChain < count) load_pending(i + kWsChain, ra);
        if (i + 2 * kWsChain < count) load_raw(i + 2 * kWsChain, rb);
      }

      // ---- the ops buffer of item j - kWsOpsBufs must have been consumed ----
      if (j >= kWsOpsBufs) {
        ok = mbar_wait_bounded(&sm.opempty[j % kWsOpsBufs],
                               (uint32_t)((j / kWsOpsBufs - 1) & 1));
        if (named_bar_or(kBarPro, 128, !ok)) {
          if (c == 0) report(p.status, KDA_ERR_TIMEOUT);
          break;
        }
      }
      if (c == 0) {
        // (the operand buffer's meta words are the input buffer's)
        reinterpret_cast<int4 *>(op.meta)[0] = im0;
        reinterpret_cast<int4 *>(op.meta)[1] = im1;
      }
      if (live) {
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          op.x[t][c] = gam[t] * kk[t];
          op.x[Q + t][c] = gam[t] * qq[t];
          sm.ex[t][c] = kk[t] * inv[t];
        }
        // v rows copied 16 bytes at a time (thread u: 8 values of row u / 16)
        if (c < 16 * Q) {
          const int t = c >> 4, q16 = c & 15;
          *reinterpret_cast<uint4 *>(&op.vv[t][8 * q16]) =
              *reinterpret_cast<const uint4 *>(&in.tok[3][t][8 * q16]);
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
          const int pka = WsKeys::a(pl), pkb = WsKeys::b(pl);
          const int xp = ws_xperm<QV>(pl);
#pragma unroll 1
          for (int chunk = warp; chunk < NCHUNK; chunk += 4) {
            const int half = chunk / (Q / QV);
            const int v0 = (chunk - half * (Q / QV)) * QV;  // first vector of the chunk
            float4 xa[QV], xb[QV];
#pragma unroll
            for (int jj = 0; jj < QV; ++jj) {
              const float *x = op.x[half * Q + v0 + (jj ^ xp)];
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
                      sa = lds4(&sm.ex[srow][pka]);
                      sb = lds4(&sm.ex[srow][pkb]);
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
          op.fin_a[t][s2] =
              s2 < t ? sm.dots_ex[s2][t] * rks * rsqrtf(sm.dots_ex[t][t] + kNormEps) : 0.f;
          op.fin_b[t][s2] = s2 <= t ? sm.dots_ex[s2][Q + t] * rks * op.rsq[t] : 0.f;
          if (s2 == t) op.rsk[t] = rks;
        }
        // New key / gate records: the old ones were read above.
        if (it.rec >= 0) {
          uint16_t *kg = p.kg;
          long long kgs = p.kg_row_stride;
          if constexpr (LAYERS) {
            kg = reinterpret_cast<uint16_t *>(lay.kg[it.l]);
            kgs = lay.kg_stride[it.l];
          }
          // 16 bytes per store: unit u of the 32 Q (part, token, 8-channel
          // chunk) units, part 0 the key row, 1 the raw-gate row
          const long long kbase = (long long)it.rec * kgs + (long long)it.h * p.rq * (2 * kDim);
#pragma unroll
          for (int u = c; u < 32 * Q; u += 128) {
            const int part = u / (16 * Q), t = (u >> 4) % Q, q16 = u & 15;
            if (!VARLEN || t < it.qb)
              *reinterpret_cast<uint4 *>(kg + kbase + t * 2 * kDim + part * kDim + 8 * q16) =
                  *reinterpret_cast<const uint4 *>(&in.tok[1 + part][t][8 * q16]);
          }
        }
      }
      named_bar(kBarPro, 128);  // in[j & 1] read, ops[j & 1] complete
      if (c == 0) mbar_arrive(&sm.opfull[j % kWsOpsBufs]);
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
  warpgroup_reg_alloc<kWsRegsMain>();
  constexpr int NG = ws_vectors<Q>() / 8;
  const int mt = tid - 128;
  const int c = lane & 7, R0 = 16 * (mt >> 5) + 4 * (lane >> 3);
  const bool leader = mt == 0;
  int issued_hi = 0;  // lane 0: one past the last item whose page this warp requested
  int consumed = 0;   // items whose page this warp has read (or skipped, inert)
  if (leader) {
    for (; issued_hi < NS && issued_hi < count; ++issued_hi) issue(issued_hi, item_slot(issued_hi));
  }
  // Every main warp counts its read of item j's stage; the eighth (last)
  // reader requests item j + NS's page into it, so no warp waits for another.
  auto stage_read = [&](int j, int next_slot) {
    __syncwarp();
    if (lane == 0) {
      const uint32_t prior = atom_add_acq_rel_smem(&sm.sreads[j % NS], 1u);
      if ((prior & 7u) == 7u && j + NS < count) {
        issue(j + NS, next_slot);
        issued_hi = j + NS + 1;
      }
    }
  };
  auto warp_arrive = [&](uint64_t *bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  // lane 0: the raw slot of item j + NS + 1, loaded an item before its use
  // (the page that may follow item j into its stage is item j + NS's)
  auto raw_slot = [&](int i) { return p.state_slots[req_of(first + i * stride)]; };
  auto valid_slot = [&](int s) { return (s > p.null_slot && s < p.n_slots) ? s : -1; };
  int raw_ahead = -1;
  if (lane == 0 && NS < count) raw_ahead = raw_slot(NS);
  bool failed = false;
  // NORM: a live item's outputs are normed during the next item (after its
  // replay), so the wait for the other warps' sums of squares overlaps that
  // work: its BF16-rounded outputs, gates, token, destination and barrier.
  bool norm_pending = false;
  float pn_o[4] = {0.f, 0.f, 0.f, 0.f};
  uint2 pn_gate = make_uint2(0, 0);
  int pn_tok = -1, pn_buf = 0;
  uint32_t pn_par = 0;
  uint16_t *pn_dst = nullptr;
  auto norm_finish = [&]() -> bool {  // false: the wait gave up
    if constexpr (!NORM) return true;
    else {
    if (!norm_pending) return true;
    norm_pending = false;
    const bool done = mbar_wait_bounded(&sm.nred[pn_buf], pn_par);
    if (__any_sync(0xffffffffu, !done)) return false;
    if (pn_tok >= 0) {
      // the eight warps' sums in warp order
      const float4 s0 = lds4(&sm.nsq[pn_buf][pn_tok][0]);
      const float4 s1 = lds4(&sm.nsq[pn_buf][pn_tok][4]);
      const float tot = ((((((s0.x + s0.y) + s0.z) + s0.w) + s1.x) + s1.y) + s1.z) + s1.w;
      // sigmoid(g) = (1 + tanh(g / 2)) / 2: half of rstd folded into the weight
      const float hr = 0.5f * rsqrtf(tot * (1.0f / kDim) + p.norm_eps);
      const float4 w4 = lds4(&sm.norm_w[R0]);
      const float g0 = bf16_bits_to_f32(pn_gate.x & 0xffffu);
      const float g1 = bf16_bits_to_f32(pn_gate.x >> 16);
      const float g2 = bf16_bits_to_f32(pn_gate.y & 0xffffu);
      const float g3 = bf16_bits_to_f32(pn_gate.y >> 16);
      *reinterpret_cast<uint2 *>(pn_dst) =
          make_uint2(pack_bf16x2(pn_o[0] * (hr * w4.x) * (1.f + tanhf_fast(0.5f * g0)),
                                 pn_o[1] * (hr * w4.y) * (1.f + tanhf_fast(0.5f * g1))),
                     pack_bf16x2(pn_o[2] * (hr * w4.z) * (1.f + tanhf_fast(0.5f * g2)),
                                 pn_o[3] * (hr * w4.w) * (1.f + tanhf_fast(0.5f * g3))));
    }
    return true;
    }
  };
  for (int j = 0; j < count; ++j) {
    int next_slot = -1;
    if (lane == 0 && j + NS < count) {
      next_slot = valid_slot(raw_ahead);
      if (j + NS + 1 < count) raw_ahead = raw_slot(j + NS + 1);
    }

    bool ok = mbar_wait_bounded(&sm.opfull[j % kWsOpsBufs], (uint32_t)((j / kWsOpsBufs) & 1));
    if (__any_sync(0xffffffffu, !ok)) {
      failed = true;
      break;
    }
    // the previous item's norm (its sums of squares are in by now)
    if (!norm_finish()) {
      failed = true;
      break;
    }
    const Ops &op = sm.ops[j % kWsOpsBufs];
    const int h = op.meta[1], slot = op.meta[2], rec = op.meta[3];
    const int n = op.meta[4], bslot = op.meta[5], m = op.meta[6];
    // the layer's outputs and corrections (the call's own without LAYERS),
    // formed where they are used
    auto out_of = [&]() -> uint16_t * {
      if constexpr (LAYERS) return p.out + op.meta[7] * lay.act_stride;
      else return p.out;
    };
    auto corr_of = [&]() -> float * {
      if constexpr (LAYERS) return reinterpret_cast<float *>(lay.corr[op.meta[7]]);
      else return p.corr;
    };
    auto corr_stride_of = [&]() -> long long {
      if constexpr (LAYERS) return lay.corr_stride[op.meta[7]];
      else return p.corr_row_stride;
    };
    // (the window is re-read from the ops buffer where it is used: fewer
    // registers live across the passes)
    auto window = [&](long long &tok0, int &qb) {
      tok0 = VARLEN ? (long long)op.meta[0] : (long long)op.meta[0] * Q;
      qb = VARLEN ? op.meta[7] : Q;
    };

    // NORM: this lane's output token's gate values, loaded now and used
    // after the solve (token c - Q or 8 + c - Q of the window; none if
    // neither is one)
    uint2 gate_raw = make_uint2(0, 0);
    if constexpr (NORM) {
      if (slot >= 0) {
        const int V = c >= Q ? c : 8 + c;
        if (V >= Q && V < 2 * Q) {
          const long long tok = (long long)op.meta[0] * Q + (V - Q);
          gate_raw = *reinterpret_cast<const uint2 *>(p.gate + (tok * p.H + h) * kDim + R0);
        }
      }
    }

    if (slot < 0) {
      // inert item: zero outputs (lane c: token c of its 4 rows).  Its
      // stage phase is an arrival without a copy, made when the item was
      // issued, i.e. after all eight reads of the stage's previous item.
      // Waiting for it keeps this warp from counting its read before a
      // slower warp has counted that previous item's (a warp can run up to
      // kWsOpsBufs - 1 items ahead), which would mix the two items' counts
      // and issue a page twice or never.
      ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
      if (__any_sync(0xffffffffu, !ok)) {
        failed = true;
        break;
      }
      long long tok0;
      int qb;
      window(tok0, qb);
      if (c < qb)
        *reinterpret_cast<uint2 *>(out_of() + ((tok0 + c) * p.H + h) * kDim + R0) =
            make_uint2(0, 0);
      stage_read(j, next_slot);
      // the norm's barrier phase of this ops buffer completes here too (its
      // phases follow the items), with nothing to exchange
      if constexpr (NORM) {
        if (!norm_finish()) {
          failed = true;
          break;
        }
        warp_arrive(&sm.nred[j % kWsOpsBufs]);
      }
      warp_arrive(&sm.opempty[j % kWsOpsBufs]);
      consumed = j + 1;
      continue;
    }

    ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
    if (__any_sync(0xffffffffu, !ok)) {
      failed = true;
      break;
    }
    consumed = j + 1;
    float4 st[4][4];
    WsTile<ST>::load(sm.stage[j % NS], R0, c, st);
    stage_read(j, next_slot);

    // ---------------- pass A: replay, write-back (n > 0) ----------------
    if constexpr (REPLAY) {
      if (n > 0) {
        float *gpage = reinterpret_cast<float *>(p.state) + (long long)slot * p.slot_stride +
                       (long long)h * (kDim * kDim);
        if constexpr (LAYERS) {
          const int l = op.meta[7];
          gpage = reinterpret_cast<float *>(lay.state[l]) + (long long)slot * lay.slot_stride[l] +
                  (long long)h * (kDim * kDim);
        }
        float *gbnd = nullptr;
        if (BOUNDARY && bslot >= 0)
          gbnd = reinterpret_cast<float *>(p.state) + (long long)bslot * p.slot_stride +
                 (long long)h * (kDim * kDim);
        // n is uniform per item: one predicate-free instance per count
        switch (n) {
          case 1: ws_replay<1, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 2: ws_replay<2, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 3: ws_replay<3, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 4: ws_replay<4, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 5: ws_replay<5, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 6: ws_replay<6, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          case 7: ws_replay<7, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
          default: ws_replay<8, BOUNDARY>(st, op, gpage, gbnd, m, R0, c); break;
        }
      }
    }

    // ---------------- pass B: 2Q dots per row ----------------------------
    float d[NG][4];
    ws_dots<NG>(st, &op.x[0][0], c, d);

    // ---------------- row solve, outputs, corrections --------------------
    long long tok0;
    int qb;
    window(tok0, qb);
    float obf[4] = {0.f, 0.f, 0.f, 0.f};
    int tout = -1;
    ws_solve<Q, NG, VARLEN, NORM>(d, op, p, out_of(), corr_of(), corr_stride_of(), tok0, qb, h,
                                  rec, R0, c, lane, obf, tout);
    if constexpr (NORM) {
      // gated RMSNorm over the 128 value rows of each token (page
      // "...kda.fused", the kernel's end): the warp's 16 rows reduced over
      // its 4 row sets and published; the other warps' sums are read, in
      // warp order (every lane of a token gets the same total), when the
      // next item's replay is done
      float sq = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) sq = fmaf(obf[r], obf[r], sq);
      sq += __shfl_xor_sync(0xffffffffu, sq, 8);
      sq += __shfl_xor_sync(0xffffffffu, sq, 16);
      const int mw = mt >> 5;
      if (lane < 8 && tout >= 0) sm.nsq[j % kWsOpsBufs][tout][mw] = sq;
      warp_arrive(&sm.nred[j % kWsOpsBufs]);
      norm_pending = true;
#pragma unroll
      for (int r = 0; r < 4; ++r) pn_o[r] = obf[r];
      pn_gate = gate_raw;
      pn_tok = tout;
      pn_buf = j % kWsOpsBufs;
      pn_par = (uint32_t)((j / kWsOpsBufs) & 1);
      pn_dst = out_of() + ((tok0 + (tout >= 0 ? tout : 0)) * p.H + h) * kDim + R0;
    }
    warp_arrive(&sm.opempty[j % kWsOpsBufs]);
  }
  if (!failed && !norm_finish()) failed = true;  // the last item's norm
  if (failed && lane == 0) report(p.status, KDA_ERR_TIMEOUT);
  // After a timeout, pages this warp requested but never read may still be in
  // flight: let them land (bounded) before this CTA's shared memory goes.
  if (lane == 0) {
    for (int jj = consumed; jj < issued_hi; ++jj)
      mbar_wait_bounded(&sm.full[jj % NS], (uint32_t)((jj / NS) & 1));
  }
}

}  // namespace kda
