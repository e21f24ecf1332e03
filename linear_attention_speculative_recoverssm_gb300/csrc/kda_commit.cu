// Standalone closed-form commit of accepted tokens into the checkpoint --
// page "vllm.models.kimi_k3.nvidia.recoverssm.cutedsl.commit" (module
// docstring: S_n = S_0 e^{L_n} + sum_{t<n} u_t (k_t e^{L_n - L_t}), and the
// align boundary state; class KdaCommit: per-layer address tables, source /
// length / destination / boundary arrays, null slot).
//
// Design: persistent CTAs (one per SM) walk the (layer, request, head)
// items; thread 0 streams each live item's source page (32 KB BF16 or 64 KB
// FP32) into a ring of shared-memory stages with one bulk copy per page, NS
// pages ahead.  Threads 0-127 build key channel c's replay coefficients
// (recorded key times the suffix decay product, D_n, and the same for the
// boundary length), threads 128-255 fetch the recorded corrections; then
// every thread folds 2 rows x 32 keys of the page in registers and stores
// the result (and the boundary state) straight to global memory.  The
// product form of the decays is used instead of the log form (the same
// quantity; it saves one exp per coefficient).
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kCommitThreads = 256;

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

template <typename ST>
struct CommitSmem {
  static constexpr int NS = sizeof(ST) == 2 ? 6 : 3;
  ST stage[NS][kDim * kDim];
  float kp[kMaxQ][kDim];
  float dn[kDim];
  float kpb[kMaxQ][kDim];
  float db[kDim];
  float uold[kMaxQ][kDim];
  float red[4][kMaxQ];
  uint64_t full[NS];
};

template <typename ST>
struct CommitLayoutCheck {
  using S = CommitSmem<ST>;
  static_assert(offsetof(S, stage) % 128 == 0 && offsetof(S, kp) % 16 == 0 &&
                offsetof(S, dn) % 16 == 0 && offsetof(S, kpb) % 16 == 0 &&
                offsetof(S, db) % 16 == 0 && offsetof(S, full) % 8 == 0,
                "float4-read members / barrier alignment");
  static constexpr bool ok = true;
};
static_assert(CommitLayoutCheck<float>::ok && CommitLayoutCheck<uint16_t>::ok, "layout");

struct CommitItem {
  int l, b, h;
  bool live;
  int src, dst, row, n, bslot, m;
};

template <typename ST, bool ALIGN>
__device__ __forceinline__ CommitItem commit_item(const CommitParams &p,
                                                  int item, bool report_errors) {
  CommitItem it;
  it.h = item % p.H;
  it.b = (item / p.H) % p.B;
  it.l = item / (p.H * p.B);
  int n = p.commit_lens[it.b];
  n = n > p.Q ? p.Q : n;
  it.n = n;
  it.src = p.sources[it.b];
  it.dst = p.destinations[it.b];
  it.row = p.record_rows != nullptr ? p.record_rows[it.b] : it.b;
  it.live = n > 0 && it.src > p.null_slot && it.dst > p.null_slot && it.row >= 0;
  it.bslot = -1;
  it.m = 0;
  if (!it.live) return it;
  bool bad = it.src >= p.n_slots || it.dst >= p.n_slots || it.row >= p.n_rows;
  const uint64_t sp = p.state_ptrs[it.l], cp = p.corr_ptrs[it.l], kp = p.kg_ptrs[it.l];
  const bool misaligned = ((sp | cp | kp) & 15) != 0 ||
                          ((p.state_strides[it.l] * (int64_t)sizeof(ST)) & 15) != 0 ||
                          ((p.corr_strides[it.l] * 4) & 15) != 0 ||
                          ((p.kg_strides[it.l] * 2) & 15) != 0;
  if (bad || misaligned) {
    if (report_errors) report(p.status, misaligned ? KDA_ERR_ALIGN : KDA_ERR_ARG);
    it.live = false;
    return it;
  }
  if (ALIGN && p.boundaries != nullptr) {
    const int bs = p.boundaries[it.b];
    int m = p.boundary_lens[it.b];
    m = m > p.Q ? p.Q : m;
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
__device__ __forceinline__ ST *commit_page(const CommitParams &p, int l, int slot, int h) {
  return reinterpret_cast<ST *>(p.state_ptrs[l]) + (long long)slot * p.state_strides[l] +
         (long long)h * (kDim * kDim);
}

template <typename ST>
__device__ __forceinline__ float4 load_page4(const ST *page, int row, int key);
template <>
__device__ __forceinline__ float4 load_page4<float>(const float *page, int row, int key) {
  return lds4(page + row * kDim + key);
}
template <>
__device__ __forceinline__ float4 load_page4<uint16_t>(const uint16_t *page, int row, int key) {
  const uint2 w = *reinterpret_cast<const uint2 *>(page + row * kDim + key);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

template <typename ST>
__device__ __forceinline__ void store_page4(ST *page, int row, int key, float4 v);
template <>
__device__ __forceinline__ void store_page4<float>(float *page, int row, int key, float4 v) {
  stg4(page + row * kDim + key, v);
}
template <>
__device__ __forceinline__ void store_page4<uint16_t>(uint16_t *page, int row, int key, float4 v) {
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2 *>(page + row * kDim + key) = w;
}

template <typename ST, bool ALIGN>
__global__ void __launch_bounds__(kCommitThreads, 1)
    kda_commit_persistent(const CommitParams p, int n_items) {
  using Smem = CommitSmem<ST>;
  constexpr int NS = Smem::NS;
  constexpr uint32_t kPageBytes = kDim * kDim * sizeof(ST);
  constexpr int kRotate = sizeof(ST) == 4 ? 1 : 3;
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

  auto issue = [&](int j) {
    const CommitItem it = commit_item<ST, ALIGN>(p, first + j * stride, false);
    uint64_t *bar = &sm.full[j % NS];
    if (it.live) {
      mbar_arrive_expect_tx(bar, kPageBytes);
      bulk_g2s(sm.stage[j % NS], commit_page<ST>(p, it.l, it.src, it.h), kPageBytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  if (tid == 0) {
    for (int j = 0; j < NS && j < count; ++j) issue(j);
  }

  const int g = tid >> 2, l4 = tid & 3;
  const int c = tid & (kDim - 1);
  for (int j = 0; j < count; ++j) {
    const CommitItem it = commit_item<ST, ALIGN>(p, first + j * stride, tid == 0);
    if (!it.live) {
      if (tid == 0 && j + NS < count) issue(j + NS);
      continue;
    }
    // ---- coefficients (threads 0-127) and corrections (128-255) ----
    if (tid < kDim) {
      const float a = __expf(p.A_log[it.l * p.H + it.h]);
      const float dt = p.dt_bias[((long long)it.l * p.H + it.h) * kDim + c];
      const uint16_t *kg = reinterpret_cast<const uint16_t *>(p.kg_ptrs[it.l]) +
                           (long long)it.row * p.kg_strides[it.l] +
                           (long long)it.h * p.Q * (2 * kDim) + c;
      float kr[kMaxQ], dr[kMaxQ];
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t) {
        kr[t] = 0.f;
        dr[t] = 1.f;
        if (t < it.n) {
          kr[t] = bf16_bits_to_f32(kg[t * 2 * kDim]);
          dr[t] = gate_decay(a, bf16_bits_to_f32(kg[t * 2 * kDim + kDim]), dt, p.lower_bound);
        }
      }
      float fd = 1.f;
#pragma unroll
      for (int t = kMaxQ - 1; t >= 0; --t) {
        if (t < it.n) {
          sm.kp[t][c] = kr[t] * fd;
          fd *= dr[t];
        }
      }
      sm.dn[c] = fd;
      if constexpr (ALIGN) {
        if (it.bslot >= 0) {
          float fb = 1.f;
#pragma unroll
          for (int t = kMaxQ - 1; t >= 0; --t) {
            if (t < it.m) {
              sm.kpb[t][c] = kr[t] * fb;
              fb *= dr[t];
            }
          }
          sm.db[c] = fb;
        }
      }
      float sq[kMaxQ];
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t) sq[t] = kr[t] * kr[t];
      reduce_scatter<kMaxQ, 8>(sq, lane & 7);
      sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 8);
      sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);
      if (lane < kMaxQ) sm.red[warp][lane] = sq[0];
    } else {
      const float *corr = reinterpret_cast<const float *>(p.corr_ptrs[it.l]) +
                          (long long)it.row * p.corr_strides[it.l] +
                          (long long)it.h * p.Q * kDim + c;
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t)
        if (t < it.n) sm.uold[t][c] = corr[t * kDim];
    }
    const bool ok = mbar_wait_bounded(&sm.full[j % NS], (uint32_t)((j / NS) & 1));
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        report(p.status, KDA_ERR_TIMEOUT);
        for (int jj = j; jj < j + NS && jj < count; ++jj)
          mbar_wait_bounded(&sm.full[jj % NS], (uint32_t)((jj / NS) & 1));
      }
      __syncthreads();
      return;
    }

    // ---- fold 2 rows x 32 keys per thread ----
    const int v0 = g, v1 = g + 64;
    float u0[kMaxQ], u1[kMaxQ];
#pragma unroll
    for (int t = 0; t < kMaxQ; ++t) {
      u0[t] = u1[t] = 0.f;
      if (t < it.n) {
        const float tot = (sm.red[0][t] + sm.red[2][t]) + (sm.red[1][t] + sm.red[3][t]);
        const float rs = rsqrtf(tot + kNormEps);
        u0[t] = sm.uold[t][v0] * rs;
        u1[t] = sm.uold[t][v1] * rs;
      }
    }
    const ST *page = sm.stage[j % NS];
    ST *dst = commit_page<ST>(p, it.l, it.dst, it.h);
    ST *bnd = (ALIGN && it.bslot >= 0) ? commit_page<ST>(p, it.l, it.bslot, it.h) : nullptr;
#pragma unroll
    for (int cc0 = 0; cc0 < 8; ++cc0) {
      const int cc = cc0 ^ (g & kRotate);
      const int key = 4 * (l4 + 4 * cc);
      const float4 s0 = load_page4<ST>(page, v0, key);
      const float4 s1 = load_page4<ST>(page, v1, key);
      if constexpr (ALIGN) {
        if (bnd != nullptr) {
          const float4 d4 = lds4(&sm.db[key]);
          float4 b0 = make_float4(s0.x * d4.x, s0.y * d4.y, s0.z * d4.z, s0.w * d4.w);
          float4 b1 = make_float4(s1.x * d4.x, s1.y * d4.y, s1.z * d4.z, s1.w * d4.w);
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t) {
            if (t < it.m) {
              const float4 k4 = lds4(&sm.kpb[t][key]);
              b0.x = fmaf(u0[t], k4.x, b0.x); b0.y = fmaf(u0[t], k4.y, b0.y);
              b0.z = fmaf(u0[t], k4.z, b0.z); b0.w = fmaf(u0[t], k4.w, b0.w);
              b1.x = fmaf(u1[t], k4.x, b1.x); b1.y = fmaf(u1[t], k4.y, b1.y);
              b1.z = fmaf(u1[t], k4.z, b1.z); b1.w = fmaf(u1[t], k4.w, b1.w);
            }
          }
          store_page4<ST>(bnd, v0, key, b0);
          store_page4<ST>(bnd, v1, key, b1);
        }
      }
      const float4 d4 = lds4(&sm.dn[key]);
      float4 r0 = make_float4(s0.x * d4.x, s0.y * d4.y, s0.z * d4.z, s0.w * d4.w);
      float4 r1 = make_float4(s1.x * d4.x, s1.y * d4.y, s1.z * d4.z, s1.w * d4.w);
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t) {
        if (t < it.n) {
          const float4 k4 = lds4(&sm.kp[t][key]);
          r0.x = fmaf(u0[t], k4.x, r0.x); r0.y = fmaf(u0[t], k4.y, r0.y);
          r0.z = fmaf(u0[t], k4.z, r0.z); r0.w = fmaf(u0[t], k4.w, r0.w);
          r1.x = fmaf(u1[t], k4.x, r1.x); r1.y = fmaf(u1[t], k4.y, r1.y);
          r1.z = fmaf(u1[t], k4.z, r1.z); r1.w = fmaf(u1[t], k4.w, r1.w);
        }
      }
      store_page4<ST>(dst, v0, key, r0);
      store_page4<ST>(dst, v1, key, r1);
    }
    __syncthreads();  // the stage and the coefficient arrays are free again
    if (tid == 0 && j + NS < count) issue(j + NS);
  }
}

std::atomic<uint64_t> g_commit_configured[4];

template <typename ST, bool ALIGN>
int launch_commit_t(const CommitParams &p, int n_items, cudaStream_t stream, int slot) {
  auto kern = kda_commit_persistent<ST, ALIGN>;
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
