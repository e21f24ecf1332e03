// Standalone closed-form commit of accepted tokens into the checkpoint --
// page "vllm.models.kimi_k3.nvidia.recoverssm.cutedsl.commit" (module
// docstring: S_n = S_0 e^{L_n} + sum_{t<n} u_t (k_t e^{L_n - L_t}), and the
// align boundary state; class KdaCommit: per-layer address tables, source /
// length / destination / boundary arrays, null slot).
//
// Design (one CTA per SM, 384 threads, items (layer, request, head) strided
// over the grid):
//  * two prologue warpgroups (warps 0-3 and 4-7, alternate items; thread c
//    <-> key channel c): thread 0 of each resolves its item chain two items
//    ahead and stages each live item's
//    recorded key / gate rows and corrections with two bulk copies, one item
//    ahead; every thread then builds channel c's replay coefficients
//    (recorded key times the suffix decay product, D_n, the boundary's
//    1 / prod_{m<=s<n} d_s) and the corrections scaled by their key's rsqrt
//    norm into one of two shared "ops" buffers.  The product form of the
//    decays is used instead of the log form (the same quantity; it saves one
//    exp per coefficient).
//  * main warpgroups (warps 8-15): each live item's source page (32 KB BF16
//    or 64 KB FP32) arrives by one bulk copy in a ring of NS stages; thread
//    (main warp w, lane 8 rs + c) reads rows 16 w + 4 rs .. + 3, keys
//    32 i + 4 c .. + 3 into registers, and the last warp to read a stage
//    requests the page NS items ahead into it.  S_n = S_0 D_n +
//    sum_t u_t (k_t P_t)^T is formed in registers and stored to the
//    destination (rounded once for a BF16 pool); the boundary state is the
//    partial sum after m terms times 1 / prod_{m<=s<n} d_s.
//  * every wait is bounded; a timeout is reported in the status word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

// Two prologue warpgroups take alternate items (the per-item prologue is a
// latency chain; two of them keep up with the main warpgroups), then two main
// warpgroups.
constexpr int kCmProWGs = 2;
constexpr int kCommitThreads = 128 * (kCmProWGs + 2);
constexpr int kCmOps = 2 * kCmProWGs;  // operand buffers: two per prologue warpgroup
constexpr int kCmBarPro = 1;           // + warpgroup: named barrier of a prologue warpgroup

struct CommitParams {
  const uint64_t *state_ptrs, *corr_ptrs, *kg_ptrs;
  const int64_t *state_strides, *corr_strides, *kg_strides;
  const float *A_log, *dt_bias;
  const int32_t *sources, *commit_lens, *destinations;
  const int32_t *boundaries, *boundary_lens, *record_rows;
  float lower_bound;
  int null_slot, L, H, B, Q, n_slots, n_rows;
  int32_t *status;
};

// One item's operands, built by the prologue.
struct alignas(16) CmOps {
  float kp[kMaxQ][kDim];  // recorded k_t * prod_{t<s<n} d_s
  float dn[kDim];         // prod_{s<n} d_s
  float ir[kDim];         // 1 / prod_{m<=s<n} d_s (boundary)
  float u[kMaxQ][kDim];   // recorded u_t[row] * rsqrt(|k_t|^2 + eps)
  unsigned long long dst, bnd;  // destination / boundary page (0: none)
  // the source page of the item NS later (0: none or dead), which the last
  // reader of this item's stage requests into it
  unsigned long long next_src;
  int meta[4];                  // live, n, m
};

// One item's records and gate bias, staged by bulk copies, and its resolved
// indices (written by the thread that requests the copies).
struct alignas(16) CmIn {
  uint16_t kg[kMaxQ][2 * kDim];
  float corr[kMaxQ][kDim];
  float dt[kDim];
  unsigned long long dst, bnd;
  float a;       // exp(A_log) of the item's (layer, head)
  int meta[3];   // live, n, m
};

template <typename ST>
struct CommitSmem {
  static constexpr int NS = sizeof(ST) == 2 ? 4 : 2;
  ST stage[NS][kDim * kDim];
  CmOps ops[kCmOps];
  CmIn in[kCmProWGs][2];
  float red[kCmProWGs][4][kMaxQ];
  uint64_t full[NS];
  uint64_t opfull[kCmOps];
  uint64_t opempty[kCmOps];
  uint64_t infull[kCmProWGs][2];
  uint32_t sreads[NS];
};

template <typename ST>
struct CommitLayoutCheck {
  using S = CommitSmem<ST>;
  static_assert(sizeof(CmOps) % 16 == 0 && sizeof(CmIn) % 16 == 0, "buffer strides");
  static_assert(offsetof(S, stage) % 128 == 0 && offsetof(S, ops) % 16 == 0 &&
                offsetof(S, in) % 16 == 0 && offsetof(CmOps, kp) % 16 == 0 &&
                offsetof(CmOps, dn) % 16 == 0 && offsetof(CmOps, ir) % 16 == 0 &&
                offsetof(CmOps, u) % 16 == 0 && offsetof(CmIn, kg) % 16 == 0 &&
                offsetof(CmIn, corr) % 16 == 0 && offsetof(CmIn, dt) % 16 == 0,
                "float4-read members / bulk-copy targets");
  static_assert(offsetof(S, full) % 8 == 0 && offsetof(S, opfull) % 8 == 0 &&
                offsetof(S, opempty) % 8 == 0 && offsetof(S, infull) % 8 == 0, "mbarriers");
  static_assert(sizeof(S) <= 232448, "shared memory per CTA");
  static constexpr bool ok = true;
};
static_assert(CommitLayoutCheck<float>::ok && CommitLayoutCheck<uint16_t>::ok, "layout");

// The per-request / per-layer values an item depends on, loaded without
// branching on them (so the loads can be issued well before they are used).
struct CommitRaw {
  int n, src, dst, row, bs, blen;
  uint64_t sp, cp, kp;
  int64_t ss, cs, ks;
};

__device__ __forceinline__ CommitRaw commit_raw(const CommitParams &p, bool align, int item) {
  CommitRaw r;
  const int b = (item / p.H) % p.B, l = item / (p.H * p.B);
  r.n = p.commit_lens[b];
  r.src = p.sources[b];
  r.dst = p.destinations[b];
  r.row = p.record_rows != nullptr ? p.record_rows[b] : b;
  r.bs = align ? p.boundaries[b] : -1;
  r.blen = align ? p.boundary_lens[b] : 0;
  r.sp = p.state_ptrs[l];
  r.cp = p.corr_ptrs[l];
  r.kp = p.kg_ptrs[l];
  r.ss = p.state_strides[l];
  r.cs = p.corr_strides[l];
  r.ks = p.kg_strides[l];
  return r;
}

struct CommitItem {
  bool live;
  int l, h, n, m;
  unsigned long long src, dst, bnd;  // page addresses
  unsigned long long kg, corr;       // record addresses of the item
};

// Liveness and addresses of an item: live = n > 0, source and destination
// above the null slot, record row >= 0; indices outside their pools or
// misaligned tables make the item dead (and are reported when asked).
template <typename ST>
__device__ __forceinline__ CommitItem commit_resolve(const CommitParams &p, int item,
                                                     const CommitRaw &r, bool report_errors) {
  CommitItem it;
  it.h = item % p.H;
  it.l = item / (p.H * p.B);
  const int n = r.n > p.Q ? p.Q : r.n;
  it.n = n;
  it.m = 0;
  it.src = it.dst = it.bnd = it.kg = it.corr = 0;
  it.live = n > 0 && r.src > p.null_slot && r.dst > p.null_slot && r.row >= 0;
  if (!it.live) return it;
  // a per-layer stride below one slot's / row's extent (or negative) would
  // put this item's pages and records outside the layer's pool
  const bool bad = r.src >= p.n_slots || r.dst >= p.n_slots || r.row >= p.n_rows ||
                   r.ss < (int64_t)p.H * kDim * kDim || r.cs < (int64_t)p.H * p.Q * kDim ||
                   r.ks < (int64_t)p.H * p.Q * 2 * kDim;
  const bool misaligned = ((r.sp | r.cp | r.kp) & 15) != 0 ||
                          ((r.ss * (int64_t)sizeof(ST)) & 15) != 0 || ((r.cs * 4) & 15) != 0 ||
                          ((r.ks * 2) & 15) != 0;
  if (bad || misaligned) {
    if (report_errors) report(p.status, misaligned ? KDA_ERR_ALIGN : KDA_ERR_ARG);
    it.live = false;
    return it;
  }
  const unsigned long long hoff = (unsigned long long)it.h * (kDim * kDim) * sizeof(ST);
  it.src = r.sp + (unsigned long long)(r.src * r.ss) * sizeof(ST) + hoff;
  it.dst = r.sp + (unsigned long long)(r.dst * r.ss) * sizeof(ST) + hoff;
  it.kg = r.kp + ((unsigned long long)r.row * r.ks + (unsigned long long)it.h * p.Q * 2 * kDim) * 2;
  it.corr = r.cp + ((unsigned long long)r.row * r.cs + (unsigned long long)it.h * p.Q * kDim) * 4;
  if (r.bs >= p.n_slots) {
    if (report_errors) report(p.status, KDA_ERR_ARG);
  } else if (r.blen > 0 && r.bs > p.null_slot) {
    const int m = r.blen > p.Q ? p.Q : r.blen;
    it.m = m < n ? m : n;
    it.bnd = r.sp + (unsigned long long)(r.bs * r.ss) * sizeof(ST) + hoff;
  }
  return it;
}

// The thread's 4 x 16 tile of a stage, as FP32.
template <typename ST>
__device__ __forceinline__ void cm_load_tile(const ST *page, int R0, int c, float4 (&s)[4][4]);
template <>
__device__ __forceinline__ void cm_load_tile<float>(const float *page, int R0, int c,
                                                    float4 (&s)[4][4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[r][i] = lds4(page + (R0 + r) * kDim + 32 * i + 4 * c);
}
template <>
__device__ __forceinline__ void cm_load_tile<uint16_t>(const uint16_t *page, int R0, int c,
                                                       float4 (&s)[4][4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 w = *reinterpret_cast<const uint2 *>(page + (R0 + r) * kDim + 32 * i + 4 * c);
      s[r][i] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                            __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    }
}

// Four values of a row to a page (BF16: rounded to nearest even).
template <typename ST>
__device__ __forceinline__ void cm_store4(unsigned long long page, int row, int key, float4 v);
template <>
__device__ __forceinline__ void cm_store4<float>(unsigned long long page, int row, int key,
                                                 float4 v) {
  stg4(reinterpret_cast<float *>(page) + row * kDim + key, v);
}
template <>
__device__ __forceinline__ void cm_store4<uint16_t>(unsigned long long page, int row, int key,
                                                    float4 v) {
  *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(page) + row * kDim + key) =
      make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// The fold for NT tokens on the thread's tile (boundary after m terms).
template <typename ST, int NT, bool ALIGN>
__device__ __forceinline__ void cm_fold(float4 (&s)[4][4], const CmOps &op, unsigned long long dst,
                                        unsigned long long bnd, int m, int R0, int c) {
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
    if constexpr (ALIGN) {
      if (bnd != 0 && t == m - 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 ir4 = lds4(&op.ir[32 * i + 4 * c]);
#pragma unroll
          for (int r = 0; r < 4; ++r) cm_store4<ST>(bnd, R0 + r, 32 * i + 4 * c, fmul4(s[r][i], ir4));
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) cm_store4<ST>(dst, R0 + r, 32 * i + 4 * c, s[r][i]);
}

template <typename ST, bool ALIGN>
__global__ void __launch_bounds__(kCommitThreads, 1)
    kda_commit_ws(const CommitParams p, int n_items) {
  using Smem = CommitSmem<ST>;
  constexpr int NS = Smem::NS;
  constexpr uint32_t kPageBytes = kDim * kDim * sizeof(ST);
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int first = blockIdx.x, stride = gridDim.x;
  const int count = first < n_items ? (n_items - first + stride - 1) / stride : 0;
  auto item_of = [&](int j) { return first + j * stride; };

  // Page of item j into stage j % NS (any one thread).
  auto issue = [&](int j, unsigned long long src) {
    uint64_t *bar = &sm.full[j % NS];
    if (src != 0) {
      mbar_arrive_expect_tx(bar, kPageBytes);
      bulk_g2s(sm.stage[j % NS], reinterpret_cast<const void *>(src), kPageBytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  auto page_of = [&](int j) {
    const int item = item_of(j);
    const CommitItem it = commit_resolve<ST>(p, item, commit_raw(p, ALIGN, item), false);
    return it.live ? it.src : 0ull;
  };

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      sm.sreads[s] = 0;
    }
    for (int b = 0; b < kCmOps; ++b) {
      mbar_init(&sm.opfull[b], 1);
      mbar_init(&sm.opempty[b], 8);  // one arrival per main warp
    }
    for (int w = 0; w < kCmProWGs; ++w) {
      mbar_init(&sm.infull[w][0], 1);
      mbar_init(&sm.infull[w][1], 1);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp < 4 * kCmProWGs) {
    // =====================================================================
    // prologue warpgroup pw: items j = pw, pw + 2, ...; thread c owns key
    // channel c.  Its k-th item is j = pw + 2 k.
    // =====================================================================
    const int pw = warp >> 2, wl = warp & 3;
    const int c = tid - 128 * pw;
    const int bar_id = kCmBarPro + pw;
    const int nk = count > pw ? (count - pw + kCmProWGs - 1) / kCmProWGs : 0;
    auto jof = [&](int k) { return pw + kCmProWGs * k; };
    // thread 0's item chain: raw values of item k + 2, resolved item k + 1
    CommitRaw raw2{};
    CommitItem nxt{};
    auto request = [&](int k, const CommitItem &it) {  // thread 0
      uint64_t *bar = &sm.infull[pw][k & 1];
      CmIn &in = sm.in[pw][k & 1];
      in.meta[0] = it.live ? 1 : 0;
      in.meta[1] = it.n;
      in.meta[2] = it.m;
      in.dst = it.dst;
      in.bnd = it.bnd;
      if (!it.live) {
        mbar_arrive(bar);
        return;
      }
      in.a = __expf(p.A_log[it.l * p.H + it.h]);
      const uint32_t bytes = (uint32_t)it.n * kDim * 4u;  // per record tensor
      mbar_arrive_expect_tx(bar, 2u * bytes + kDim * 4u);
      bulk_g2s(&in.kg[0][0], reinterpret_cast<const void *>(it.kg), bytes, bar);
      bulk_g2s(&in.corr[0][0], reinterpret_cast<const void *>(it.corr), bytes, bar);
      bulk_g2s(&in.dt[0], p.dt_bias + ((long long)it.l * p.H + it.h) * kDim, kDim * 4u, bar);
    };
    auto resolve = [&](int k, const CommitRaw &r) {
      return commit_resolve<ST>(p, item_of(jof(k)), r, true);
    };
    int requested = 0, taken = 0;
    if (c == 0 && nk > 0) {
      request(0, resolve(0, commit_raw(p, ALIGN, item_of(jof(0)))));
      requested = 1;
      if (nk > 1) nxt = resolve(1, commit_raw(p, ALIGN, item_of(jof(1))));
      if (nk > 2) raw2 = commit_raw(p, ALIGN, item_of(jof(2)));
    }
    bool failed = false;
    for (int k = 0; k < nk; ++k) {
      const int j = jof(k);
      CmOps &op = sm.ops[j % kCmOps];
      const CmIn &in = sm.in[pw][k & 1];
      // thread 0: the source page of item j + NS (items j + 2 and j + 4 are
      // this warpgroup's next two), handed to the main warps with this item
      unsigned long long next_src = 0;
      if (c == 0 && k + 1 < nk) {
        const CommitItem it1 = nxt;  // item j + 2
        request(k + 1, it1);
        requested = k + 2;
        if (k + 2 < nk) nxt = resolve(k + 2, raw2);  // item j + 4
        if (k + 3 < nk) raw2 = commit_raw(p, ALIGN, item_of(jof(k + 3)));
        static_assert(NS == 2 || NS == 4, "page ring of 2 or 4 stages");
        if constexpr (NS == 2) {
          next_src = it1.live ? it1.src : 0ull;
        } else {
          next_src = (k + 2 < nk && nxt.live) ? nxt.src : 0ull;
        }
      }
      bool ok = mbar_wait_bounded(&sm.infull[pw][k & 1], (uint32_t)((k >> 1) & 1));
      if (named_bar_or(bar_id, 128, !ok)) {
        failed = true;
        break;
      }
      taken = k + 1;
      struct {
        bool live;
        int n, m;
        unsigned long long dst, bnd;
      } it;
      it.live = in.meta[0] != 0;
      it.n = in.meta[1];
      it.m = in.meta[2];
      it.dst = in.dst;
      it.bnd = in.bnd;
      const float a = in.a, dt = in.dt[c];
      float kr[kMaxQ], dr[kMaxQ];
      if (it.live) {
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          kr[t] = 0.f;
          dr[t] = 1.f;
          if (t < it.n) {
            kr[t] = bf16_bits_to_f32(in.kg[t][c]);
            dr[t] = gate_decay(a, bf16_bits_to_f32(in.kg[t][kDim + c]), dt, p.lower_bound);
          }
        }
        float sq[kMaxQ];
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) sq[t] = kr[t] * kr[t];
        reduce_scatter<kMaxQ, 8>(sq, lane & 7);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 8);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);
        if (lane < kMaxQ) sm.red[pw][wl][lane] = sq[0];
      }
      // the ops buffer of item j - kCmOps must have been consumed
      if (j >= kCmOps) {
        ok = mbar_wait_bounded(&sm.opempty[j % kCmOps], (uint32_t)((j / kCmOps - 1) & 1));
        if (named_bar_or(bar_id, 128, !ok)) {
          failed = true;
          break;
        }
      }
      if (c == 0) {
        op.meta[0] = it.live ? 1 : 0;
        op.meta[1] = it.n;
        op.meta[2] = it.m;
        op.dst = it.dst;
        op.bnd = it.bnd;
        op.next_src = next_src;
      }
      if (it.live) {
        float fd = 1.f;
#pragma unroll
        for (int t = kMaxQ - 1; t >= 0; --t) {
          if (t < it.n) {
            op.kp[t][c] = kr[t] * fd;
            fd *= dr[t];
          }
        }
        op.dn[c] = fd;
        if constexpr (ALIGN) {
          if (it.bnd != 0) {
            float rm = 1.f;  // prod_{m <= s < n} d_s
#pragma unroll
            for (int t = kMaxQ - 1; t >= 0; --t)
              if (t >= it.m && t < it.n) rm *= dr[t];
            op.ir[c] = __fdividef(1.f, rm);
          }
        }
        named_bar(bar_id, 128);  // channel sums written
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) {
          if (t < it.n) {
            const float tot = (sm.red[pw][0][t] + sm.red[pw][2][t]) +
                              (sm.red[pw][1][t] + sm.red[pw][3][t]);
            op.u[t][c] = in.corr[t][c] * rsqrtf(tot + kNormEps);
          }
        }
      }
      named_bar(bar_id, 128);  // in and the sums read, the ops buffer complete
      if (c == 0) mbar_arrive(&sm.opfull[j % kCmOps]);
    }
    if (failed && c == 0) report(p.status, KDA_ERR_TIMEOUT);
    // after a timeout: record copies requested but never waited for land first
    if (c == 0) {
      for (int i = taken; i < requested; ++i)
        mbar_wait_bounded(&sm.infull[pw][i & 1], (uint32_t)((i >> 1) & 1));
    }
    return;
  }

  // =======================================================================
  // main warpgroups
  // =======================================================================
  const int mt = tid - 128 * kCmProWGs;
  const int c = lane & 7, R0 = 16 * (mt >> 5) + 4 * (lane >> 3);
  int issued_hi = 0;  // lane 0: one past the last item whose page this warp requested
  int consumed = 0;   // items whose page this warp has read (or skipped)
  if (mt == 0) {
    for (; issued_hi < NS && issued_hi < count; ++issued_hi) issue(issued_hi, page_of(issued_hi));
  }
  auto stage_read = [&](int j, unsigned long long next_src) {
    __syncwarp();
    if (lane == 0) {
      const uint32_t prior = atom_add_acq_rel_smem(&sm.sreads[j % NS], 1u);
      if ((prior & 7u) == 7u && j + NS < count) {
        issue(j + NS, next_src);
        issued_hi = j + NS + 1;
      }
    }
  };
  bool failed = false;
  for (int j = 0; j < count; ++j) {
    bool ok = mbar_wait_bounded(&sm.opfull[j % kCmOps], (uint32_t)((j / kCmOps) & 1));
    if (__any_sync(0xffffffffu, !ok)) {
      failed = true;
      break;
    }
    const CmOps &op = sm.ops[j % kCmOps];
    const unsigned long long next_src = op.next_src;
    const bool live = op.meta[0] != 0;
    const int n = op.meta[1], m = op.meta[2];
    const unsigned long long dst = op.dst, bnd = op.bnd;
    if (!live) {
      // The stage phase of an item that is not live is an arrival without a
      // copy, made when the item was issued, after all eight reads of the
      // stage's previous item; waiting for it keeps this warp (up to
      // kCmOps - 1 items ahead of the slowest) from counting its read among
      // that previous item's, which would issue a page twice or never.
      ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
      if (__any_sync(0xffffffffu, !ok)) {
        failed = true;
        break;
      }
      stage_read(j, next_src);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.opempty[j % kCmOps]);
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
    cm_load_tile<ST>(sm.stage[j % NS], R0, c, st);
    stage_read(j, next_src);
    switch (n) {
      case 1: cm_fold<ST, 1, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 2: cm_fold<ST, 2, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 3: cm_fold<ST, 3, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 4: cm_fold<ST, 4, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 5: cm_fold<ST, 5, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 6: cm_fold<ST, 6, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      case 7: cm_fold<ST, 7, ALIGN>(st, op, dst, bnd, m, R0, c); break;
      default: cm_fold<ST, 8, ALIGN>(st, op, dst, bnd, m, R0, c); break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.opempty[j % kCmOps]);
  }
  if (failed && lane == 0) report(p.status, KDA_ERR_TIMEOUT);
  if (lane == 0) {
    for (int jj = consumed; jj < issued_hi; ++jj)
      mbar_wait_bounded(&sm.full[jj % NS], (uint32_t)((jj / NS) & 1));
  }
}

std::atomic<uint64_t> g_commit_configured[4];

template <typename ST, bool ALIGN>
int launch_commit_t(const CommitParams &p, int n_items, cudaStream_t stream, int slot) {
  auto kern = kda_commit_ws<ST, ALIGN>;
  const size_t smem = sizeof(CommitSmem<ST>);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(g_commit_configured[slot].load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return KDA_ERR_CUDA;
    g_commit_configured[slot].fetch_or(bit);
  }
  const int grid = n_items < device_sm_count(dev) ? n_items : device_sm_count(dev);
  kern<<<grid, kCommitThreads, smem, stream>>>(p, n_items);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

int launch_commit(const uint64_t *state_ptrs, const uint64_t *corr_ptrs, const uint64_t *kg_ptrs,
                  const int64_t *state_strides, const int64_t *corr_strides,
                  const int64_t *kg_strides, const float *A_log, const float *dt_bias,
                  const int32_t *sources, const int32_t *commit_lens,
                  const int32_t *destinations, const int32_t *boundaries,
                  const int32_t *boundary_lens, const int32_t *record_rows, int state_dtype,
                  float lower_bound, int null_slot, int L, int H, int B, int Q, int n_slots,
                  int n_rows, int32_t *status, cudaStream_t stream) {
  CommitParams p;
  p.state_ptrs = state_ptrs;
  p.corr_ptrs = corr_ptrs;
  p.kg_ptrs = kg_ptrs;
  p.state_strides = state_strides;
  p.corr_strides = corr_strides;
  p.kg_strides = kg_strides;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.sources = sources;
  p.commit_lens = commit_lens;
  p.destinations = destinations;
  p.boundaries = boundaries;
  p.boundary_lens = boundary_lens;
  p.record_rows = record_rows;
  p.lower_bound = lower_bound;
  p.null_slot = null_slot;
  p.L = L;
  p.H = H;
  p.B = B;
  p.Q = Q;
  p.n_slots = n_slots;
  p.n_rows = n_rows;
  p.status = status;
  const long long items = (long long)L * B * H;
  if (items > 0x7fffffffLL) return KDA_ERR_ARG;
  const bool align = boundaries != nullptr;
  if (state_dtype == KDA_STATE_BF16)
    return align ? launch_commit_t<uint16_t, true>(p, (int)items, stream, 0)
                 : launch_commit_t<uint16_t, false>(p, (int)items, stream, 1);
  return align ? launch_commit_t<float, true>(p, (int)items, stream, 2)
               : launch_commit_t<float, false>(p, (int)items, stream, 3);
}

}  // namespace kda
