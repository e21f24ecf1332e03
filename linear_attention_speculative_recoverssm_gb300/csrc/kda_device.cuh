// Device building blocks of the KDA RecoverSSM kernels (sm_103a).
//
// Hand-written PTX for the async-proxy bulk copies and mbarriers, bounded
// waits (every spin ends after a fixed time and reports KDA_ERR_TIMEOUT),
// warp reduce-scatter, BF16 bit conversions and the gate decay.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda_recoverssm.h"

namespace kda {

constexpr int kDim = KDA_HEAD_DIM;  // K = V = 128
constexpr int kMaxQ = KDA_MAX_WINDOW;
constexpr float kNormEps = 1e-6f;   // inside the rsqrt of the L2 norms
// Upper bound on any device-side wait (ns of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// status reporting
// ---------------------------------------------------------------------------

__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// BF16 bit patterns
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) {
  return __uint_as_float(bits << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}

// ---------------------------------------------------------------------------
// gate math (KdaFused.decay): exp(lb * sigmoid(exp(A_log) * (raw_g + dt)))
// `a` is exp(A_log) of the head, computed once per item.
// ---------------------------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware's approximate base-2 exponential (ex2.approx.ftz.f32).
__device__ __forceinline__ float exp2f_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh(x) by the hardware's approximation (tanh.approx.f32, relative error
// about 2^-11: for values that round to BF16 afterwards).
__device__ __forceinline__ float tanhf_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float sigmoidf_fast(float z) {
  return __fdividef(1.0f, 1.0f + __expf(-z));
}

// Computed as 2^(lb log2(e) / (1 + 2^(-a log2(e) (raw_g + dt)))): two base-2
// exponentials and one reciprocal, with the products that do not depend on
// raw_g folded (hoisted out of a caller's loop over tokens).
__device__ __forceinline__ float gate_decay(float a, float raw_g, float dt,
                                            float lower_bound) {
  const float al = a * kLog2e;
  const float e = exp2f_fast(fmaf(-al, raw_g, -al * dt));
  return exp2f_fast((lower_bound * kLog2e) * __fdividef(1.f, 1.f + e));
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers and the bulk-copy engine
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Make initialised barriers visible to the async proxy (and the cluster).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `hint_ns` passed, instead of spinning (a spinning
// warp takes issue slots from the warps doing the work).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with the given parity to complete; gives up
// after kWaitLimitNs and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar,
                                                  uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (global_ns() - start > kWaitLimitNs) return false;
  }
}

// One bulk (non-tensor) copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`.  Addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void *smem_dst,
                                              const void *gmem_src,
                                              uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes."
      "L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// One tiled tensor copy (3-D box) global -> this CTA's shared memory through
// the tensor map at `tmap` (a kernel-parameter address), completing its bytes
// on `bar`.  The innermost coordinate x times the element size must be a
// multiple of 16 bytes; the shared destination 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// The same for a 4-D box (coordinates x, y, z, w; x as in tma_load_3d).
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const void *tmap, int x, int y, int z,
                                            int w, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w),
      "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the load/store path
// (not the bulk-copy engine).  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts against the count the barrier was initialised with).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// vector shared / global accesses
// ---------------------------------------------------------------------------

__device__ __forceinline__ float4 lds4(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}

__device__ __forceinline__ void stg4(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}

__device__ __forceinline__ void sts4(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}

// ---------------------------------------------------------------------------
// packed FP32 pairs (the float2 FMA / multiply of sm_100+): one instruction
// for two lanes of FP32 arithmetic, each rounded like the scalar op.
// ---------------------------------------------------------------------------

// (a.x * b.x + c.x, a.y * b.y + c.y), each rounded like the scalar FMA
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// s (4 floats) <- s * d, elementwise, as two packed multiplies
__device__ __forceinline__ float4 fmul4(float4 s, float4 d) {
  const float2 lo = fmul2(make_float2(s.x, s.y), make_float2(d.x, d.y));
  const float2 hi = fmul2(make_float2(s.z, s.w), make_float2(d.z, d.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// s <- u * k + s (u scalar), as two packed FMAs
__device__ __forceinline__ float4 ffma4s(float u, float4 k, float4 s) {
  const float2 uu = make_float2(u, u);
  const float2 lo = ffma2(uu, make_float2(k.x, k.y), make_float2(s.x, s.y));
  const float2 hi = ffma2(uu, make_float2(k.z, k.w), make_float2(s.z, s.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// acc (even-key, odd-key partial sums) += s . x over 4 keys
__device__ __forceinline__ float2 dot4_acc(float4 s, float4 x, float2 acc) {
  acc = ffma2(make_float2(s.x, s.y), make_float2(x.x, x.y), acc);
  return ffma2(make_float2(s.z, s.w), make_float2(x.z, x.w), acc);
}

// ---------------------------------------------------------------------------
// named barriers (a warpgroup's own barrier, not the whole CTA's)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier that also ORs a predicate over the participating threads, so a
// decision taken after a bounded wait is the same for all of them.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: let the next kernel in the stream, launched
// with programmatic stream serialization, start before this grid completes.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grids this one depends on programmatically have completed
// and their memory is visible (returns at once if there are none).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory counter increment with acquire-release ordering at CTA
// scope; returns the prior value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_smem(uint32_t *p, uint32_t v) {
  uint32_t prior;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(prior)
               : "r"(smem_u32(p)), "r"(v)
               : "memory");
  return prior;
}

// Hand registers between warpgroups: every thread of the warpgroup executes
// the same instruction.  The decreases and increases of one CTA must add up
// to at most the registers it was launched with (threads x registers).
template <int N>
__device__ __forceinline__ void warpgroup_reg_dealloc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void warpgroup_reg_alloc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------
// warp reduce-scatter
// ---------------------------------------------------------------------------
//
// `v` holds N partial values per lane; the LANES consecutive lanes of a
// group (LANES a power of two dividing 32, N a multiple of LANES) add them up
// so that afterwards lane l of the group holds the totals of indices
// [l * N / LANES, (l + 1) * N / LANES) in v[0 .. N / LANES).  It takes
// N/2 + N/4 + ... + N/LANES shuffles instead of N * log2(LANES).
template <int N, int LANES>
__device__ __forceinline__ void reduce_scatter(float (&v)[N], int lane) {
  static_assert(N % LANES == 0, "N must be a multiple of the group size");
#pragma unroll
  for (int o = LANES / 2, cnt = N; o >= 1; o >>= 1, cnt >>= 1) {
    const bool upper = (lane & o) != 0;
    const int half = cnt / 2;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[half + i];
      const float keep = upper ? v[half + i] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace kda
