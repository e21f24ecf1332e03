// Cluster-split variant of the fused replay + verify step, for batches too
// small to fill the GPU with whole items -- page "vllm.models.kimi_k3.
// nvidia.specialized_decode.cutedsl.kda.fused", module docstring ("a cluster
// of split CTAs per (request, head) splits the state rows; the rows of the
// chunked form are independent").
//
// A cluster of SPLIT CTAs (2 or 4) serves one (request, head) item; CTA rank
// r owns state rows [r * 128 / SPLIT, (r + 1) * 128 / SPLIT) and streams only
// those (one bulk copy of 32 or 16 KB).  Every CTA builds the per-channel
// vectors it needs for all 128 key channels, but the channel reductions
// (sums of squares of q, k and the recorded keys, and the raw pair products)
// are split: rank r reduces channels [r * 128 / SPLIT, ...), and the partial
// sums are exchanged through distributed shared memory (each CTA stores its
// partial vector into every peer's exchange slot for its rank, then one
// cluster barrier with release / acquire semantics publishes them).  Each
// CTA adds the SPLIT partials in rank order, so all ranks see identical
// totals.  Rank 0 writes the new key / gate records once every CTA of the
// item has passed that barrier, i.e. after every old record was read.
#pragma once

#include <cstddef>

#include "kda_step.cuh"

namespace kda {

template <int Q, int SPLIT, bool BOUNDARY>
struct ClusterSmem {
  static constexpr int kRows = kDim / SPLIT;
  static constexpr int kNX = Red<Q>::kN + kMaxQ;  // token scalars + record sums
  float stage[kRows * kDim];
  float xk[Q][kDim];
  float xq[Q][kDim];
  float dots[2 * Q][kRows];
  float kp[kMaxQ][kDim];
  float dn[kDim];
  float kpb[BOUNDARY ? kMaxQ : 1][kDim];
  float db[kDim];
  float uold[kMaxQ][kRows];
  float vv[Q][kRows];
  float beta[kMaxQ];
  float red_tok[4][Red<Q>::kPad];
  float red_rec[4][kMaxQ];
  float xch[SPLIT][kNX];  // partials pushed by each rank
  float scal[Red<Q>::kN];
  float rsrec[kMaxQ];
  uint64_t full;
};

template <int Q, int SPLIT, bool BOUNDARY>
struct ClusterLayoutCheck {
  using S = ClusterSmem<Q, SPLIT, BOUNDARY>;
  static_assert(offsetof(S, stage) % 128 == 0 && offsetof(S, xk) % 16 == 0 &&
                offsetof(S, xq) % 16 == 0 && offsetof(S, kp) % 16 == 0 &&
                offsetof(S, dn) % 16 == 0 && offsetof(S, kpb) % 16 == 0 &&
                offsetof(S, db) % 16 == 0 && offsetof(S, full) % 8 == 0,
                "float4-read members / barrier alignment");
  static constexpr bool ok = true;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_release_acquire() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store one float into the shared memory of CTA `rank` of this cluster, at
// the address `local` has in this CTA.
__device__ __forceinline__ void st_peer_f32(float *local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// VARLEN: windows from query_start_loc (p.qsl, non-null), each of q_b <= Q
// tokens; otherwise request b's window is tokens b*Q .. b*Q + Q - 1.
template <int Q, int SPLIT, bool BOUNDARY, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    kda_step_cluster(const StepParams p) {
  using Smem = ClusterSmem<Q, SPLIT, BOUNDARY>;
  static_assert(ClusterLayoutCheck<Q, SPLIT, BOUNDARY>::ok, "layout");
  constexpr int ROWS = Smem::kRows;           // state rows of this CTA
  constexpr int L = kThreads / ROWS;          // lanes per row (4 or 8)
  constexpr int NCH = kDim / (4 * L);         // 4-key chunks per lane
  constexpr int ROT = L == 4 ? 1 : 0;         // bank rotation of the chunks
  constexpr int NR = Red<Q>::kN;
  constexpr int NRP = Red<Q>::kPad;
  constexpr int NX = Smem::kNX;
  constexpr int CHW = ROWS / 32;              // warps of this rank's channels
  constexpr uint32_t kBytes = ROWS * kDim * 4;
  constexpr int NDP = round_up(2 * Q, L);     // padded dots per row

  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int row0 = (int)rank * ROWS;
  const int item = blockIdx.y;

  cluster_arrive_relaxed();  // waited before the first store into a peer

  const ItemMeta it = item_meta<true, BOUNDARY, VARLEN>(p, item, Q, tid == 0 && rank == 0);
  const long long tok0 = VARLEN ? (long long)it.tok0 : (long long)it.b * Q;
  const int qb = VARLEN ? it.qb : Q;  // window length (Q without VARLEN)
  if (it.slot < 0) {
    for (int e = tid; e < qb * ROWS; e += kThreads) {
      const int t = e / ROWS, r = e - t * ROWS;
      p.out[((tok0 + t) * p.H + it.h) * kDim + row0 + r] = 0;
    }
    cluster_wait();
    return;
  }

  if (tid == 0) {
    mbar_init(&sm.full, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&sm.full, kBytes);
    bulk_g2s(sm.stage, page_ptr<float>(p, it.slot, it.h) + (long long)row0 * kDim, kBytes,
             &sm.full);
  }

  const bool token_half = tid < kDim;
  const int c = tid & (kDim - 1);
  const bool my_warp = (warp & 3) >= (int)rank * CHW && (warp & 3) < ((int)rank + 1) * CHW;
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
      // tokens past the window count as zero inputs (their results are
      // never written)
      const long long off = ((tok0 + t) * p.H + it.h) * kDim + c;
      uint16_t qbits = 0;
      kbits[t] = gbits[t] = 0;
      if (t < qb) {
        kbits[t] = p.k[off];
        gbits[t] = p.g[off];
        qbits = p.q[off];
      }
      kk[t] = bf16_bits_to_f32(kbits[t]);
      qq[t] = bf16_bits_to_f32(qbits);
      dd[t] = gate_decay(a, bf16_bits_to_f32(gbits[t]), dt, p.lower_bound);
      gam *= dd[t];
      sm.xk[t][c] = gam * kk[t];
      sm.xq[t][c] = gam * qq[t];
      red[t] = kk[t] * kk[t];
      red[Q + t] = qq[t] * qq[t];
    }
    if (my_warp) {
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
      const int wl = warp - (int)rank * CHW;
#pragma unroll
      for (int i = 0; i < NRP / 32; ++i) sm.red_tok[wl][lane * (NRP / 32) + i] = red[i];
    }
  } else {
    if (it.n > 0) {
      const float a = __expf(p.A_log[it.h]);
      const float dt = p.dt_bias[it.h * kDim + c];
      const long long cbase = (long long)it.rec * p.corr_row_stride +
                              (long long)it.h * p.rq * kDim;
      const long long kbase = (long long)it.rec * p.kg_row_stride +
                              (long long)it.h * p.rq * (2 * kDim) + c;
      float kr[kMaxQ], dr[kMaxQ];
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t) {
        kr[t] = 0.f;
        dr[t] = 1.f;
        if (t < it.n) {
          if (c < ROWS) sm.uold[t][c] = p.corr[cbase + t * kDim + row0 + c];
          kr[t] = bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim]);
          dr[t] = gate_decay(a, bf16_bits_to_f32(p.kg[kbase + t * 2 * kDim + kDim]), dt,
                             p.lower_bound);
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
      if constexpr (BOUNDARY) {
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
      if (my_warp) {
        float sq[kMaxQ];
#pragma unroll
        for (int t = 0; t < kMaxQ; ++t) sq[t] = kr[t] * kr[t];
        reduce_scatter<kMaxQ, 8>(sq, lane & 7);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 8);
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 16);
        if (lane < kMaxQ) sm.red_rec[(warp & 3) - (int)rank * CHW][lane] = sq[0];
      }
    }
    const long long voff = (tok0 * p.H + it.h) * kDim + row0 + c;
    if (c < ROWS) {
#pragma unroll
      for (int t = 0; t < Q; ++t)
        sm.vv[t][c] = t < qb ? bf16_bits_to_f32(p.v[voff + (long long)t * p.H * kDim]) : 0.f;
    }
    if (c < Q)
      sm.beta[c] =
          c < qb ? sigmoidf_fast(bf16_bits_to_f32(p.beta[(tok0 + c) * p.H + it.h])) : 0.f;
  }
  __syncthreads();

  // This rank's partial sums (its channel range), pushed to every peer.
  cluster_wait();  // every peer has started: its shared memory is live
  if (tid < NX) {
    float part = 0.f;
    if (tid < NR) {
#pragma unroll
      for (int w = 0; w < CHW; ++w) part += sm.red_tok[w][tid];
    } else if (it.n > 0) {
#pragma unroll
      for (int w = 0; w < CHW; ++w) part += sm.red_rec[w][tid - NR];
    }
#pragma unroll
    for (int r = 0; r < SPLIT; ++r) st_peer_f32(&sm.xch[rank][tid], (uint32_t)r, part);
  }
  cluster_sync_release_acquire();

  // Totals in rank order; final scalars.
  auto tot = [&](int i) {
    float s = sm.xch[0][i];
#pragma unroll
    for (int r = 1; r < SPLIT; ++r) s += sm.xch[r][i];
    return s;
  };
  if (tid < NR) {
    const float x = tot(tid);
    float val;
    if (tid < Q) {
      val = rsqrtf(x + kNormEps);
    } else if (tid < 2 * Q) {
      val = rsqrtf(x + kNormEps) * p.q_scale;
    } else {
      const int pi = tid - 2 * Q;
      const int a = pi / Q, bb = pi - a * Q;
      if (bb <= a) {
        val = x * rsqrtf(tot(bb) + kNormEps) * (rsqrtf(tot(Q + a) + kNormEps) * p.q_scale);
      } else {
        val = x * rsqrtf(tot(a) + kNormEps) * rsqrtf(tot(bb) + kNormEps);
      }
    }
    sm.scal[tid] = val;
  } else if (tid >= 128 && tid < 128 + kMaxQ) {
    const int t = tid - 128;
    sm.rsrec[t] = t < it.n ? rsqrtf(tot(NR + t) + kNormEps) : 0.f;
  }
  // New key / gate records (rank 0): every CTA has read the old ones.
  if (rank == 0 && token_half && it.rec >= 0) {
    const long long kbase = (long long)it.rec * p.kg_row_stride +
                            (long long)it.h * p.rq * (2 * kDim) + c;
#pragma unroll
    for (int t = 0; t < Q; ++t) {
      if (t < qb) {
        p.kg[kbase + t * 2 * kDim] = kbits[t];
        p.kg[kbase + t * 2 * kDim + kDim] = gbits[t];
      }
    }
  }
  const bool ok = mbar_wait_bounded(&sm.full, 0);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) {
      report(p.status, KDA_ERR_TIMEOUT);
      mbar_wait_bounded(&sm.full, 0);
    }
    __syncthreads();
    return;
  }

  // ---------------- main loop: one row per thread group of L lanes ---------
  const int g = tid / L, l = tid % L;
  float u[kMaxQ], ub[kMaxQ];
#pragma unroll
  for (int t = 0; t < kMaxQ; ++t) {
    u[t] = ub[t] = 0.f;
    if (t < it.n) {
      u[t] = sm.uold[t][g] * sm.rsrec[t];
      if (BOUNDARY && t < it.m) ub[t] = u[t];
    }
  }
  float *gout = reinterpret_cast<float *>(p.state) + (long long)it.slot * p.slot_stride +
                (long long)it.h * (kDim * kDim) + (long long)(row0 + g) * kDim;
  float *gbnd = nullptr;
  if (BOUNDARY && it.bslot >= 0)
    gbnd = reinterpret_cast<float *>(p.state) + (long long)it.bslot * p.slot_stride +
           (long long)it.h * (kDim * kDim) + (long long)(row0 + g) * kDim;
  float acc[NDP];
#pragma unroll
  for (int jj = 0; jj < NDP; ++jj) acc[jj] = 0.f;
#pragma unroll
  for (int cc0 = 0; cc0 < NCH; ++cc0) {
    const int cc = cc0 ^ (g & ROT);
    const int key = 4 * (l + L * cc);
    float4 s = lds4(&sm.stage[g * kDim + key]);
    if (it.n > 0) {
      if constexpr (BOUNDARY) {
        if (gbnd != nullptr) {
          const float4 d4 = lds4(&sm.db[key]);
          float4 bq = make_float4(s.x * d4.x, s.y * d4.y, s.z * d4.z, s.w * d4.w);
#pragma unroll
          for (int t = 0; t < kMaxQ; ++t) {
            if (t < it.m) {
              const float4 k4 = lds4(&sm.kpb[t][key]);
              bq.x = fmaf(ub[t], k4.x, bq.x); bq.y = fmaf(ub[t], k4.y, bq.y);
              bq.z = fmaf(ub[t], k4.z, bq.z); bq.w = fmaf(ub[t], k4.w, bq.w);
            }
          }
          stg4(gbnd + key, bq);
        }
      }
      const float4 d4 = lds4(&sm.dn[key]);
      s = make_float4(s.x * d4.x, s.y * d4.y, s.z * d4.z, s.w * d4.w);
#pragma unroll
      for (int t = 0; t < kMaxQ; ++t) {
        if (t < it.n) {
          const float4 k4 = lds4(&sm.kp[t][key]);
          s.x = fmaf(u[t], k4.x, s.x); s.y = fmaf(u[t], k4.y, s.y);
          s.z = fmaf(u[t], k4.z, s.z); s.w = fmaf(u[t], k4.w, s.w);
        }
      }
      stg4(gout + key, s);
    }
#pragma unroll
    for (int jj = 0; jj < Q; ++jj) {
      const float4 x = lds4(&sm.xk[jj][key]);
      acc[jj] = fmaf(s.x, x.x, fmaf(s.y, x.y, fmaf(s.z, x.z, fmaf(s.w, x.w, acc[jj]))));
      const float4 y = lds4(&sm.xq[jj][key]);
      acc[Q + jj] = fmaf(s.x, y.x, fmaf(s.y, y.y, fmaf(s.z, y.z, fmaf(s.w, y.w, acc[Q + jj]))));
    }
  }
  reduce_scatter<NDP, L>(acc, l);
#pragma unroll
  for (int i = 0; i < NDP / L; ++i) {
    const int idx = l * (NDP / L) + i;
    if (idx < 2 * Q) sm.dots[idx][g] = acc[i];
  }
  __syncthreads();

  // ---------------- row solve for this CTA's rows ----------------
  if (tid < ROWS) {
    const int r = tid, row = row0 + tid;
    float uu[Q];
#pragma unroll
    for (int t = 0; t < Q; ++t) {
      float a_t = sm.vv[t][r] - sm.dots[t][r] * sm.scal[t];
#pragma unroll
      for (int s2 = 0; s2 < t; ++s2) a_t = fmaf(-sm.scal[2 * Q + s2 * Q + t], uu[s2], a_t);
      uu[t] = sm.beta[t] * a_t;
    }
#pragma unroll
    for (int t = 0; t < Q; ++t) {
      float o = sm.dots[Q + t][r] * sm.scal[Q + t];
#pragma unroll
      for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sm.scal[2 * Q + t * Q + s2], uu[s2], o);
      if (t < qb) p.out[((tok0 + t) * p.H + it.h) * kDim + row] = f32_to_bf16_bits(o);
    }
    if (it.rec >= 0) {
      const long long cbase = (long long)it.rec * p.corr_row_stride +
                              (long long)it.h * p.rq * kDim + row;
#pragma unroll
      for (int t = 0; t < Q; ++t)
        if (t < qb) p.corr[cbase + t * kDim] = uu[t];
    }
  }
}

}  // namespace kda
