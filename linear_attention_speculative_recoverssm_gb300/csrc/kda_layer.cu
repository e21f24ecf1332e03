// The model layer around the RecoverSSM step (page "vllm.models.kimi_k3.
// nvidia.specialized_decode.cutedsl.kda.fused", KdaFused.kernel: the
// convolution operands, convolution and SiLU, gate projection, the window
// written last; the gated RMSNorm at the kernel's end).  Two kernels bracket
// the step: the prologue turns the layer's packed projections into the
// step's q, k, v (the convolution kernel) and raw gates (the projection
// kernel), and the epilogue normalises its outputs.  The prologue's two
// kernels run at the same time: the projection first, on half the SMs, and
// the convolution as its programmatic dependent on the rest and beside it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kda_recoverssm.h"
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kConvThreads = 128;  // threads of a convolution CTA

struct LayerParams {
  const uint16_t *x;       // [B*Q, 3*D] q | k | v channels before the convolution
  const uint16_t *conv_w;  // [3, 4, D]; tap 3 multiplies the current token
  const uint16_t *conv_b;  // [3*D] or nullptr
  uint16_t *conv_state;    // [slots, 3*D, rq + 2]
  long long conv_slot_stride;
  const uint16_t *f_a;  // [B*Q, 128]
  const uint16_t *f_b;  // [D, 128]
  const int32_t *state_slots, *record_rows, *pending;
  int n_slots, n_rows, rq;
  uint16_t *q, *k, *v, *g;  // [B*Q, H, 128]
  int B, H, null_slot;
  int32_t *status;
};

// CTAs over (request, slice of channels); each thread takes groups of 8
// consecutive channels (one part, one head), so every access is 16 bytes:
// the Q inputs of the group are one uint4 per token, the group's 8 windows
// (8 * (rq + 2) BF16, contiguous) are rq + 2 uint4, the outputs one uint4
// per token.  The slot and pending count are loaded once per CTA.  Channel
// j of a group is convolved over [window[off .. off+2], x_0 .. x_{Q-1}]
// (off = n - 1 after n pending tokens, 0 without), SiLU-ed, rounded to BF16,
// and its window rewritten to [window[off+1], window[off+2], x_0 ..]; the
// windows pass through a thread-private shared-memory block.
// CTAs per request: 16 measured best beside the projection (8: 1% slower on
// the large batch, 6% on a quarter of it; 2 and 4, or 24 and 32, slower)
constexpr int kConvCtas = 16;

// WHOLE (record capacity rq = Q, Q even): the new window is the whole
// window, so each lane builds a channel pair's new windows (2 (Q + 2) BF16,
// 8-byte aligned) in registers and stores them 8 bytes at a time, and reads
// each channel's three taps as two 32-bit words (a lane's block is 8 (Q + 2)
// BF16 from its neighbour's, so a warp's 2-byte accesses hit each bank up to
// 8 times).
template <int Q, bool WHOLE>
__device__ __forceinline__ void conv_request(const LayerParams &p, uint16_t *wins) {
  static_assert(!WHOLE || Q % 2 == 0, "whole-window rewrite: an even window");
  const int b = blockIdx.x;
  const int slot = p.state_slots[b];
  const int rec = p.pending != nullptr ? (p.record_rows != nullptr ? p.record_rows[b] : b) : -1;
  if (slot >= p.n_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(p.status, KDA_ERR_ARG);
    return;
  }
  if (slot <= p.null_slot) return;  // inert: the step writes its zero outputs
  int n = 0;  // pending tokens (their count sets the window offset)
  if (rec >= p.n_rows) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(p.status, KDA_ERR_ARG);
  } else if (rec >= 0) {
    n = p.pending[rec];
    n = n < 0 ? 0 : (n > p.rq ? p.rq : n);
  }
  const int off = n > 0 ? n - 1 : 0;
  const int D = p.H * kDim;
  const int W = p.rq + 2;
  const int groups = 3 * D / 8;
  const long long tok0 = (long long)b * Q;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the warp's 32 window blocks lie back to back, as in HBM, so both copies
  // move 512 contiguous bytes per instruction
  uint16_t *area = wins + warp * 32 * 8 * (kMaxQ + 2);
  uint4 *sw = reinterpret_cast<uint4 *>(area);
  uint16_t *mine = area + lane * 8 * W;
  for (int base = blockIdx.y * kConvThreads + warp * 32; base < groups;
       base += kConvCtas * kConvThreads) {  // warp-uniform trip count
    const int g = base + lane;
    const bool active = g < groups;
    const int nvec = (groups - base < 32 ? groups - base : 32) * W;  // the active lanes' blocks
    // this lane's inputs and weights first: they do not wait for the windows
    const int ch = 8 * (active ? g : base), part = ch / D, hc = ch - part * D;  // hc = h*128 + c0
    uint4 xv[Q];
#pragma unroll
    for (int t = 0; t < Q; ++t)
      xv[t] = *reinterpret_cast<const uint4 *>(p.x + (tok0 + t) * (3LL * D) + ch);
    uint4 wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      wv[i] = *reinterpret_cast<const uint4 *>(p.conv_w + (long long)(part * 4 + i) * D + hc);
    uint4 bv = make_uint4(0, 0, 0, 0);
    if (p.conv_b != nullptr) bv = *reinterpret_cast<const uint4 *>(p.conv_b + ch);
    uint4 *gw = reinterpret_cast<uint4 *>(p.conv_state + (long long)slot * p.conv_slot_stride +
                                          8LL * base * W);
    for (int j = lane; j < nvec; j += 32) sw[j] = gw[j];
    __syncwarp();
    if (active) {
      const uint16_t *xh[Q];
#pragma unroll
      for (int t = 0; t < Q; ++t) xh[t] = reinterpret_cast<const uint16_t *>(&xv[t]);
      const uint16_t *wh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) wh[i] = reinterpret_cast<const uint16_t *>(&wv[i]);
      const uint16_t *bh = reinterpret_cast<const uint16_t *>(&bv);
      uint32_t res[Q][4];
      constexpr int kWords = (Q + 2) / 2;  // a channel's window, in 32-bit words (WHOLE)
      uint32_t nwin[WHOLE ? 2 * kWords : 1];  // the current channel pair's new windows
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint16_t *win = mine + j * W;
        uint16_t t0, t1, t2;
        if constexpr (WHOLE) {
          // the taps off .. off + 2 lie in words off / 2 and off / 2 + 1
          const uint32_t *ww = reinterpret_cast<const uint32_t *>(win);
          const uint32_t wa = ww[off >> 1], wb = ww[(off >> 1) + 1];
          if ((off & 1) == 0) {
            t0 = (uint16_t)(wa & 0xffffu);
            t1 = (uint16_t)(wa >> 16);
            t2 = (uint16_t)(wb & 0xffffu);
          } else {
            t0 = (uint16_t)(wa >> 16);
            t1 = (uint16_t)(wb & 0xffffu);
            t2 = (uint16_t)(wb >> 16);
          }
        } else {
          t0 = win[off];
          t1 = win[off + 1];
          t2 = win[off + 2];
        }
        float seq[Q + 3];
        seq[0] = bf16_bits_to_f32(t0);
        seq[1] = bf16_bits_to_f32(t1);
        seq[2] = bf16_bits_to_f32(t2);
#pragma unroll
        for (int t = 0; t < Q; ++t) seq[3 + t] = bf16_bits_to_f32(xh[t][j]);
        const float bias = bf16_bits_to_f32(bh[j]);
#pragma unroll
        for (int t = 0; t < Q; ++t) {
          float acc = bias;
#pragma unroll
          for (int i = 0; i < 4; ++i) acc = fmaf(seq[t + i], bf16_bits_to_f32(wh[i][j]), acc);
          // (the fast exp and divide are good to ~1e-6 relative; the result
          // is rounded to BF16, 2^-9)
          const uint32_t bits = f32_to_bf16_bits(__fdividef(acc, 1.f + __expf(-acc)));
          if (j & 1) res[t][j >> 1] |= bits << 16;
          else res[t][j >> 1] = bits;
        }
        if constexpr (WHOLE) {
          const int jj = (j & 1) * kWords;
          nwin[jj] = (uint32_t)t1 | ((uint32_t)t2 << 16);
#pragma unroll
          for (int w = 1; w < kWords; ++w)
            nwin[jj + w] = (uint32_t)xh[2 * w - 2][j] | ((uint32_t)xh[2 * w - 1][j] << 16);
          if (j & 1) {  // channels j - 1 and j: 2 (Q + 2) BF16 from element (j - 1) W
            uint2 *pair = reinterpret_cast<uint2 *>(mine + (j - 1) * W);
#pragma unroll
            for (int w = 0; w < kWords; ++w) pair[w] = make_uint2(nwin[2 * w], nwin[2 * w + 1]);
          }
        } else {
          win[0] = t1;  // entries from 2 + Q on (rq > Q) are kept
          win[1] = t2;
#pragma unroll
          for (int t = 0; t < Q; ++t) win[2 + t] = xh[t][j];
        }
      }

      uint16_t *out = part == 0 ? p.q : (part == 1 ? p.k : p.v);
      const int h = hc / kDim, c0 = hc - h * kDim;
#pragma unroll
      for (int t = 0; t < Q; ++t)
        *reinterpret_cast<uint4 *>(out + ((tok0 + t) * p.H + h) * kDim + c0) =
            make_uint4(res[t][0], res[t][1], res[t][2], res[t][3]);
    }
    __syncwarp();
    for (int j = lane; j < nvec; j += 32) gw[j] = sw[j];
    __syncwarp();  // the area is refilled on the next trip
  }
}

template <int Q, bool WHOLE>
__global__ void __launch_bounds__(kConvThreads, 5) kda_layer_conv(const LayerParams p) {
  __shared__ __align__(16) uint16_t wins[kConvThreads * 8 * (kMaxQ + 2)];
  grid_launch_dependents();  // a programmatic dependent may start at once
  conv_request<Q, WHOLE>(p, wins);
  // This kernel runs beside the gate projection, launched as its
  // programmatic dependent (or as the first of the two, the projection then
  // being its dependent).  One CTA, the last, waits for that grid as it
  // exits (at once when there is none), so this grid completes after it and
  // later work in the stream sees both; the others exit at once and free
  // their SM for the next CTAs (a wait in every CTA would hold the first
  // wave's slots until the projection ends).
  if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && threadIdx.x == 0)
    grid_dependency_wait();
}

// ---------------------------------------------------------------------------
// The gate projection on the fifth-generation tensor cores
// ---------------------------------------------------------------------------
// raw_g[t, h, f] = BF16(sum_j f_b[h*128 + f, j] f_a[t, j]) is a [T x 128] by
// [128 x D] product (D = H*128) whose K is only 128.  A unit is one (128
// tokens, head) tile, units u = m * H + h.  A persistent CTA per SM takes a
// contiguous range of units, so consecutive units share their token tile m
// and its f_a rows (A) stay in shared memory while the heads' f_b rows (B)
// stream through a two-stage ring:
//  * warp 4, lane 0 (copies): loads each new token tile's A into one of two
//    A slots and each unit's B into the next B stage, with tensor copies 64
//    K-elements wide in the 128-byte swizzled K-major layout (rows of 128
//    bytes, 8-row groups 1024 bytes apart); it runs ahead of the MMAs as far
//    as the free stages allow;
//  * warp 5, lane 0 (MMA): issues the eight K = 16 steps of one M = N = 128
//    BF16 MMA (tcgen05.mma, FP32 accumulation) per unit into one of four
//    128-column TMEM accumulators, and commits them to "accumulator full",
//    "B stage free" and, after a token tile's last unit, "A slot free";
//  * warps 0-3 (read-back): warp w reads TMEM lanes (tokens) 32 w .. 32 w +
//    31 of the accumulator, 32 columns per load, rounds to BF16 and writes
//    each thread's 256-byte row into the warp's shared staging rows, then
//    marks the accumulator free; the warp then stores two whole rows per
//    instruction (16 lanes x 16 bytes each).  Stores straight from the
//    registers touch 32 rows 16 KB apart per warp instruction, and took
//    about half the kernel's time.  A staged row's 16-byte chunk c sits at
//    position c ^ (row & 7), so both the row writes (eight rows, one chunk)
//    and the row reads (one row, eight chunks) hit distinct banks.  The
//    request's liveness is loaded before the accumulator wait.
// The shared memory (161 KB) leaves room on the SM for three convolution
// CTAs, which run beside this kernel.
// Tokens past the activations (zero rows from the tensor copy) and tokens
// of inert requests are not written.  Every mbarrier wait is bounded; after
// a timeout the copy lane waits (bounded) for the copies it issued and the
// MMA lane for its MMAs, and the TMEM columns are released on every path.

constexpr int kGateTile = 128;   // tokens (M) and features (N) of a unit
constexpr int kGateKBlock = 64;  // BF16 elements per 128-byte swizzled row
constexpr int kGateASlots = 2;   // token tiles (f_a) in shared memory
constexpr int kGateBStages = 2;  // head tiles (f_b) in flight
constexpr int kGateAccs = 4;     // TMEM accumulators
constexpr int kGateThreads = 192;  // read-back warps 0-3, copy warp 4, MMA warp 5
constexpr uint32_t kGateBlockBytes = kGateTile * kGateKBlock * 2;  // 16 KB
constexpr uint32_t kGateTileBytes = 2 * kGateBlockBytes;           // a 128 x 128 operand
constexpr uint32_t kGateOutPitch = kGateTile * 2;  // a staged BF16 row (chunks swizzled)
constexpr uint32_t kGateOutBytes = kGateTile * kGateOutPitch;  // the staging rows
constexpr uint32_t kGateSmem = (kGateASlots + kGateBStages) * kGateTileBytes + kGateOutBytes +
                               1024;  // + alignment slack
static_assert(kGateSmem + 3 * (20 + 1) * 1024 + 1024 <= 228 * 1024,
              "gate projection: room for three convolution CTAs on its SM");
static_assert(2 * kGateSmem > 228 * 1024, "gate projection: one CTA per SM");
// FP32 accumulator columns: 128 per accumulator, all 512 of the SM.  One CTA
// fits on an SM (161 KB of shared memory), so an allocation never waits.
constexpr uint32_t kGateTmemCols = kGateAccs * kGateTile;
static_assert(kGateTmemCols <= 512, "TMEM columns");
// Instruction descriptor of kind::f16: FP32 accumulator (bits 4-5 = 1), A
// and B BF16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3
// at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kGateIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(kGateTile >> 3) << 17) |
                                ((uint32_t)(kGateTile >> 4) << 24);

// Tensor maps of f_a [T, 128] and f_b [D, 128] as 2-D BF16 tensors with a
// (64, 128) box and the 128-byte swizzle.
struct GateMaps {
  CUtensorMap a, b;
};

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: start address >> 4 (bits 0-13), leading byte offset
// (bits 16-29; not used by swizzled K-major operands), stride byte offset
// 1024 >> 4 between 8-row groups (bits 32-45), the fixed 0b001 at bits
// 46-48, swizzle mode 2 = 128 bytes (bits 61-63).  The 1024-byte aligned
// tile base keeps the base-offset field at 0; a K step inside the 128-byte
// row advances the start address by its 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[M x K] . B[N x K]^T for one K = 16 step.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive FP32 columns of this warp's 32 TMEM lanes, one lane per
// thread; waits for the load.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kGateThreads, 1)
    kda_layer_gate(const LayerParams p, const __grid_constant__ GateMaps maps, int Q,
                   int n_tokens, int n_units) {
  extern __shared__ uint8_t gate_raw[];
  // the convolution kernel, launched after this one, may start at once: the
  // two are independent and share the SMs
  grid_launch_dependents();
  __shared__ uint64_t a_full[kGateASlots];     // the slot's token tile landed
  __shared__ uint64_t a_free[kGateASlots];     // the tile's last MMA has read it
  __shared__ uint64_t b_full[kGateBStages];    // the stage's head tile landed
  __shared__ uint64_t b_free[kGateBStages];    // the MMA has read the stage
  __shared__ uint64_t acc_full[kGateAccs];     // the accumulator holds its unit
  __shared__ uint64_t acc_free[kGateAccs];     // the read-back warps are done with it
  __shared__ uint64_t mma_done;                // every MMA of this CTA completed
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's units: a contiguous range
  const int u_begin = (int)((long long)n_units * blockIdx.x / gridDim.x);
  const int n_mine = (int)((long long)n_units * (blockIdx.x + 1) / gridDim.x) - u_begin;
  const int m_first = u_begin / p.H;
  // A slots, B stages and staging rows from a 1024-byte aligned base
  const uint32_t pad = (1024u - (smem_u32(gate_raw) & 1023u)) & 1023u;
  uint8_t *a_tiles = gate_raw + pad;
  uint8_t *b_tiles = a_tiles + kGateASlots * kGateTileBytes;
  uint8_t *staging = b_tiles + kGateBStages * kGateTileBytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGateASlots; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_free[s], 1);
    }
    for (int s = 0; s < kGateBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_free[s], 1);
    }
    for (int s = 0; s < kGateAccs; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_free[s], 4);
    }
    mbar_init(&mma_done, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, kGateTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // unit i of this CTA starts a token tile when its m differs from unit i-1's
  const auto new_tile = [&](int i) {
    return i == 0 || (u_begin + i) / p.H != (u_begin + i - 1) / p.H;
  };
  if (warp == 4) {
    if (lane == 0) {
      bool ok = true;
      int a_last = -1;  // the last token tile loaded (index from m_first)
      int b_issued = 0;
      for (int i = 0; i < n_mine && ok; ++i) {
        const int u = u_begin + i, m = u / p.H, h = u - m * p.H;
        if (new_tile(i)) {
          const int ai = m - m_first, as = ai & 1;
          if (ai >= kGateASlots)
            ok = mbar_wait_bounded(&a_free[as], ((uint32_t)(ai >> 1) & 1u) ^ 1u);
          if (!ok) break;
          uint8_t *dst = a_tiles + as * kGateTileBytes;
          mbar_arrive_expect_tx(&a_full[as], kGateTileBytes);
          tma_load_2d(dst, &maps.a, 0, m * kGateTile, &a_full[as]);
          tma_load_2d(dst + kGateBlockBytes, &maps.a, kGateKBlock, m * kGateTile, &a_full[as]);
          a_last = ai;
        }
        const int bs = i % kGateBStages;
        const uint32_t bu = (uint32_t)(i / kGateBStages);
        if (i >= kGateBStages) ok = mbar_wait_bounded(&b_free[bs], (bu & 1u) ^ 1u);
        if (!ok) break;
        uint8_t *dst = b_tiles + bs * kGateTileBytes;
        mbar_arrive_expect_tx(&b_full[bs], kGateTileBytes);
        tma_load_2d(dst, &maps.b, 0, h * kGateTile, &b_full[bs]);
        tma_load_2d(dst + kGateBlockBytes, &maps.b, kGateKBlock, h * kGateTile, &b_full[bs]);
        b_issued = i + 1;
      }
      if (!ok) {
        // (the read-back warps time out on their own waits) wait for every
        // copy still in flight before the CTA can exit
        report(p.status, KDA_ERR_TIMEOUT);
        for (int i = b_issued - kGateBStages; i < b_issued; ++i)
          if (i >= 0)
            mbar_wait_bounded(&b_full[i % kGateBStages], (uint32_t)(i / kGateBStages) & 1u);
        for (int ai = a_last - 1; ai <= a_last; ++ai)
          if (ai >= 0) mbar_wait_bounded(&a_full[ai & 1], (uint32_t)(ai >> 1) & 1u);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < n_mine; ++i) {
        const int u = u_begin + i, m = u / p.H;
        const int ai = m - m_first, as = ai & 1;
        const int bs = i % kGateBStages, acc = i % kGateAccs;
        if (new_tile(i)) ok = mbar_wait_bounded(&a_full[as], (uint32_t)(ai >> 1) & 1u);
        if (ok) ok = mbar_wait_bounded(&b_full[bs], (uint32_t)(i / kGateBStages) & 1u);
        if (ok && i >= kGateAccs)
          ok = mbar_wait_bounded(&acc_free[acc], ((uint32_t)(i / kGateAccs) & 1u) ^ 1u);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_s = smem_u32(a_tiles + as * kGateTileBytes);
        const uint32_t b_s = smem_u32(b_tiles + bs * kGateTileBytes);
#pragma unroll
        for (int ks = 0; ks < kDim / 16; ++ks) {
          // K step ks: 32 bytes into the 128-byte rows of k-block ks / 4
          const uint32_t off = (uint32_t)(ks >> 2) * kGateBlockBytes + (uint32_t)(ks & 3) * 32u;
          umma_bf16(tmem + (uint32_t)(acc * kGateTile), umma_desc_sw128(a_s + off),
                    umma_desc_sw128(b_s + off), kGateIdesc, ks > 0);
        }
        umma_commit(&acc_full[acc]);
        umma_commit(&b_free[bs]);
        if (i + 1 == n_mine || new_tile(i + 1)) umma_commit(&a_free[as]);
      }
      if (!ok) report(p.status, KDA_ERR_TIMEOUT);
      // every MMA issued has completed before the columns are released
      umma_commit(&mma_done);
      mbar_wait_bounded(&mma_done, 0u);
    }
  } else {
    for (int i = 0; i < n_mine; ++i) {
      const int acc = i % kGateAccs;
      const int u = u_begin + i, m = u / p.H, h = u - m * p.H;
      const int t = m * kGateTile + warp * 32 + lane;
      bool live = t < n_tokens;
      if (live) {
        const int slot = p.state_slots[t / Q];
        live = slot > p.null_slot && slot < p.n_slots;
      }
      const bool ok = __all_sync(
          0xffffffffu, mbar_wait_bounded(&acc_full[acc], (uint32_t)(i / kGateAccs) & 1u));
      if (!ok) {
        if (lane == 0) report(p.status, KDA_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      uint8_t *rows = staging + warp * 32 * kGateOutPitch;  // this warp's 32 rows
      uint8_t *row = rows + lane * kGateOutPitch;
      const int sw = lane & 7;  // this row's chunk swizzle
#pragma unroll
      for (int c = 0; c < kGateTile / 32; ++c) {
        uint32_t r[32];
        tmem_load32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * kGateTile + c * 32),
                    r);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(row + (((c * 4 + j) ^ sw) * 16)) = make_uint4(
              pack_bf16x2(__uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1])),
              pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
              pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
              pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_free[acc]);
      const uint32_t live_rows = __ballot_sync(0xffffffffu, live);
      const long long t0 = (long long)(t - lane);
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int r = 2 * k + (lane >> 4);
        const uint4 v = *reinterpret_cast<const uint4 *>(rows + r * kGateOutPitch +
                                                         (((lane & 15) ^ (r & 7)) * 16));
        if ((live_rows >> r) & 1u)
          *reinterpret_cast<uint4 *>(p.g + ((t0 + r) * p.H + h) * kDim + (lane & 15) * 8) = v;
      }
      __syncwarp();  // the rows are read before the next unit rewrites them
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kGateTmemCols);
  }
  // launched as the convolution's programmatic dependent, it completes only
  // after that grid (no wait without one)
  if (threadIdx.x == 0) grid_dependency_wait();
}

// Half a warp per (token, head) row of 128 outputs, 8 per lane (16-byte
// accesses; two rows per warp):
// out = BF16(o * rsqrt(mean(o^2) + eps) * w * sigmoid(gate)).
__global__ void __launch_bounds__(256) kda_layer_epilogue(const uint16_t *__restrict__ o,
                                                          const uint16_t *__restrict__ gate,
                                                          const float *__restrict__ w, float eps,
                                                          uint16_t *__restrict__ out, long long rows) {
  const int lane = threadIdx.x & 31;
  const long long r = (blockIdx.x * 8LL + (threadIdx.x >> 5)) * 2 + (lane >> 4);
  const bool valid = r < rows;
  const long long base = (valid ? r : 0) * kDim + 8 * (lane & 15);
  const uint4 ob = *reinterpret_cast<const uint4 *>(o + base);
  const uint4 gb = *reinterpret_cast<const uint4 *>(gate + base);
  const float4 wa = *reinterpret_cast<const float4 *>(w + 8 * (lane & 15));
  const float4 wb = *reinterpret_cast<const float4 *>(w + 8 * (lane & 15) + 4);
  const uint32_t op[4] = {ob.x, ob.y, ob.z, ob.w}, gp[4] = {gb.x, gb.y, gb.z, gb.w};
  const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
  float ov[8], gv[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ov[2 * i] = __uint_as_float(op[i] << 16);
    ov[2 * i + 1] = __uint_as_float(op[i] & 0xffff0000u);
    gv[2 * i] = __uint_as_float(gp[i] << 16);
    gv[2 * i + 1] = __uint_as_float(gp[i] & 0xffff0000u);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(ov[i], ov[i], ss);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);  // within the half
  const float rstd = 1.f / sqrtf(ss * (1.f / kDim) + eps);
  // (the fast exp and divide are good to ~1e-6 relative; the result is BF16)
  uint32_t res[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = ov[2 * i] * rstd * wv[2 * i] * __fdividef(1.f, 1.f + __expf(-gv[2 * i]));
    const float c =
        ov[2 * i + 1] * rstd * wv[2 * i + 1] * __fdividef(1.f, 1.f + __expf(-gv[2 * i + 1]));
    res[i] = pack_bf16x2(a, c);
  }
  if (valid) *reinterpret_cast<uint4 *>(out + base) = make_uint4(res[0], res[1], res[2], res[3]);
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 gate_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// f_a [n_tokens, 128] and f_b [H*128, 128] (BF16, 256-byte rows) with a (64,
// 128) box in the 128-byte swizzle; rows past the tensor arrive as zeros.
int encode_gate_maps(const LayerParams &p, int n_tokens, GateMaps &maps) {
  const auto encode = gate_map_encoder();
  if (encode == nullptr) return KDA_ERR_CUDA;
  const cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kGateKBlock, (cuuint32_t)kGateTile};
  const cuuint32_t estride[2] = {1, 1};
  const cuuint64_t dims_a[2] = {(cuuint64_t)kDim, (cuuint64_t)n_tokens};
  const cuuint64_t dims_b[2] = {(cuuint64_t)kDim, (cuuint64_t)p.H * kDim};
  if (encode(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.f_a), dims_a,
             strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KDA_ERR_CUDA;
  if (encode(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.f_b), dims_b,
             strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

// Launch order of the prologue's two kernels (the second overlaps the
// first).  Measured on the large batch (H = 64, B = 512, Q = 8): the gate
// projection first on half the SMs, 162-164 us for both; on all SMs,
// 167-173 us; the convolution first, 178 us; one after the other, 180 us.
// The convolution alone takes 151 us.
constexpr bool kPrologueConvFirst = false;

template <int Q>
int launch_prologue_q(const LayerParams &p, int items, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kda_layer_gate, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGateSmem) != cudaSuccess)
      return KDA_ERR_CUDA;
    configured.fetch_or(bit);
  }
  const int n_tokens = p.B * Q;
  GateMaps maps;
  const int st = encode_gate_maps(p, n_tokens, maps);
  if (st != KDA_OK) return st;
  const long long units = (long long)((n_tokens + kGateTile - 1) / kGateTile) * p.H;
  if (units > 0x7fffffffLL) return KDA_ERR_ARG;
  // the gate projection's persistent CTAs on half the SMs: the convolution
  // runs on the other half (and beside them, three CTAs to an SM)
  const int sms = device_sm_count(dev);
  const int half = sms / 2 > 0 ? sms / 2 : 1;
  const int grid = units < half ? (int)units : half;
  // The two kernels are independent.  The second is launched as the first's
  // programmatic dependent (each kernel lets dependents start as it begins),
  // so it starts while the first is still running and shares the SMs with
  // it; it waits for the first grid only as it exits, so its completion
  // implies both and work after this call stays ordered.
  const auto launch = [&](auto kernel, dim3 grid_dim, dim3 block, uint32_t smem, bool dependent,
                          auto... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid_dim;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
  };
  const auto launch_gate = [&](bool dependent) {
    return launch(kda_layer_gate, dim3(grid), dim3(kGateThreads), kGateSmem, dependent, p, maps, Q,
                  n_tokens, (int)units);
  };
  const auto launch_conv = [&](bool dependent) {
    const dim3 g(p.B, kConvCtas), b(kConvThreads);
    if constexpr (Q % 2 == 0) {
      if (p.rq == Q) return launch(kda_layer_conv<Q, true>, g, b, 0u, dependent, p);
    }
    return launch(kda_layer_conv<Q, false>, g, b, 0u, dependent, p);
  };
  cudaError_t e;
  if (kPrologueConvFirst) {
    e = launch_conv(false);
    if (e == cudaSuccess) e = launch_gate(true);
  } else {
    e = launch_gate(false);
    if (e == cudaSuccess) e = launch_conv(true);
  }
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace
}  // namespace kda

extern "C" {

int kda_layer_prologue(const kda_bf16 *x, const kda_bf16 *conv_weight, const kda_bf16 *conv_bias,
                       kda_bf16 *conv_state, int64_t conv_slot_stride, const kda_bf16 *f_a,
                       const kda_bf16 *f_b, const int32_t *state_slots,
                       const int32_t *record_rows, const int32_t *pending, int n_slots,
                       int n_rows, int rq, kda_bf16 *q, kda_bf16 *k, kda_bf16 *v, kda_bf16 *raw_g,
                       int B, int H, int Q, int null_slot, int32_t *status, void *stream) {
  if (B < 0 || H < 1 || Q < 1 || Q > KDA_MAX_WINDOW || rq < Q || rq > KDA_MAX_WINDOW)
    return KDA_ERR_ARG;
  if (B == 0) return KDA_OK;
  if (!x || !conv_weight || !conv_state || !f_a || !f_b || !state_slots || !q || !k || !v ||
      !raw_g)
    return KDA_ERR_ARG;
  if (n_slots < 1 || n_rows < 0) return KDA_ERR_ARG;
  if (conv_slot_stride < 3LL * H * KDA_HEAD_DIM * (rq + 2)) return KDA_ERR_ARG;
  if ((long long)B * H * 3 > 0x7fffffffLL || (long long)B * Q > 0x7fffffffLL || H > 65535)
    return KDA_ERR_ARG;
  if (!kda::aligned16(x) || !kda::aligned16(conv_weight) ||
      (conv_bias != nullptr && !kda::aligned16(conv_bias)) || !kda::aligned16(f_a) ||
      !kda::aligned16(f_b) || !kda::aligned16(conv_state) || !kda::aligned16(q) ||
      !kda::aligned16(k) || !kda::aligned16(v) || !kda::aligned16(raw_g) ||
      conv_slot_stride % 8 != 0)
    return KDA_ERR_ALIGN;
  kda::LayerParams p;
  p.x = x;
  p.conv_w = conv_weight;
  p.conv_b = conv_bias;
  p.conv_state = conv_state;
  p.conv_slot_stride = conv_slot_stride;
  p.f_a = f_a;
  p.f_b = f_b;
  p.state_slots = state_slots;
  p.record_rows = record_rows;
  p.pending = pending;
  p.n_slots = n_slots;
  p.n_rows = n_rows;
  p.rq = rq;
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = raw_g;
  p.B = B;
  p.H = H;
  p.null_slot = null_slot;
  p.status = status;
  const int items = B * H;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (Q) {
    case 1: return kda::launch_prologue_q<1>(p, items, s);
    case 2: return kda::launch_prologue_q<2>(p, items, s);
    case 3: return kda::launch_prologue_q<3>(p, items, s);
    case 4: return kda::launch_prologue_q<4>(p, items, s);
    case 5: return kda::launch_prologue_q<5>(p, items, s);
    case 6: return kda::launch_prologue_q<6>(p, items, s);
    case 7: return kda::launch_prologue_q<7>(p, items, s);
    default: return kda::launch_prologue_q<8>(p, items, s);
  }
}

int kda_layer_epilogue(const kda_bf16 *o, const kda_bf16 *gate, const float *norm_weight,
                       float eps, kda_bf16 *out, int n_tokens, int H, void *stream) {
  if (n_tokens < 0 || H < 1) return KDA_ERR_ARG;
  if (n_tokens == 0) return KDA_OK;
  if (!o || !gate || !norm_weight || !out) return KDA_ERR_ARG;
  if (!(eps >= 0.f)) return KDA_ERR_ARG;
  if (!kda::aligned16(o) || !kda::aligned16(gate) || !kda::aligned16(norm_weight) ||
      !kda::aligned16(out))
    return KDA_ERR_ALIGN;
  const long long rows = (long long)n_tokens * H;
  const long long blocks = (rows + 15) / 16;  // 16 rows per block of 8 warps
  if (blocks > 0x7fffffffLL) return KDA_ERR_ARG;
  kda::kda_layer_epilogue<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      o, gate, norm_weight, eps, out, rows);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
