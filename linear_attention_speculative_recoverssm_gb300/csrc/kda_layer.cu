// The model layer around the RecoverSSM step (page "vllm.models.kimi_k3.
// nvidia.specialized_decode.cutedsl.kda.fused", KdaFused.kernel: the
// convolution operands, convolution and SiLU, gate projection, the window
// written last; the gated RMSNorm at the kernel's end).  Two kernels bracket
// the step: the prologue turns the layer's packed projections into the
// step's q, k, v (the convolution kernel) and raw gates (the projection
// kernel), and the epilogue normalises its outputs.
#include <cuda_runtime.h>

#include "../../include/kda_recoverssm.h"
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kConvThreads = 128;  // threads of a convolution CTA
constexpr int kGateTokens = 128;   // tokens per gate-projection CTA (8 warps x 16)

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
constexpr int kConvCtas = 8;  // CTAs per request

template <int Q>
__global__ void __launch_bounds__(kConvThreads) kda_layer_conv(const LayerParams p) {
  __shared__ __align__(16) uint16_t wins[kConvThreads * 8 * (kMaxQ + 2)];
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
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint16_t *win = mine + j * W;
        const uint16_t t0 = win[off], t1 = win[off + 1], t2 = win[off + 2];
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
        win[0] = t1;  // entries from 2 + Q on (rq > Q) are kept
        win[1] = t2;
#pragma unroll
        for (int t = 0; t < Q; ++t) win[2 + t] = xh[t][j];
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

// D[16 x 8] += A[16 x 16] . B[16 x 8]: BF16 operands, FP32 accumulation
// (mma.sync m16n8k16, A row-major, B column-major).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The gate projection raw_g[t, h, f] = BF16(sum_j f_b[h*128 + f, j] f_a[t, j])
// on the tensor cores: one CTA per (128 tokens, head).  The head's f_b block
// (128 features x 128 k, BF16) is staged once in shared memory with rows
// padded by 16 bytes, so the 8 rows a B fragment spans fall in distinct
// banks.  Warp w takes tokens 16 w .. 16 w + 15: their f_a rows are the A
// fragments of all 8 k-steps, held in registers; the warp then walks the
// 16 feature tiles of 8.  Tokens of inert requests are not written.
constexpr int kGateRow = kDim + 8;  // padded f_b row in shared memory (BF16)

__global__ void __launch_bounds__(256) kda_layer_gate(const LayerParams p, int Q, int n_tokens) {
  __shared__ __align__(16) uint16_t fbs[kDim * kGateRow];
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(p.f_b + (long long)h * kDim * kDim);
    for (int e = threadIdx.x; e < kDim * kDim / 8; e += 256) {
      const int row = e >> 4, col8 = e & 15;
      *reinterpret_cast<uint4 *>(fbs + row * kGateRow + col8 * 8) = __ldg(src + e);
    }
  }
  __syncthreads();
  const int row0 = blockIdx.x * kGateTokens + warp * 16;
  if (row0 >= n_tokens) return;
  const int ra = row0 + grp, rb = row0 + grp + 8;
  const bool va = ra < n_tokens, vb = rb < n_tokens;
  const uint32_t *fa_a = reinterpret_cast<const uint32_t *>(p.f_a + (long long)(va ? ra : row0) * kDim);
  const uint32_t *fa_b = reinterpret_cast<const uint32_t *>(p.f_a + (long long)(vb ? rb : row0) * kDim);
  uint32_t a[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    a[ks][0] = fa_a[ks * 8 + tig];
    a[ks][1] = fa_b[ks * 8 + tig];
    a[ks][2] = fa_a[ks * 8 + 4 + tig];
    a[ks][3] = fa_b[ks * 8 + 4 + tig];
  }
  const auto live = [&](int row) {
    const int s = p.state_slots[row / Q];
    return s > p.null_slot && s < p.n_slots;
  };
  const bool la = va && live(ra), lb = vb && live(rb);
  uint16_t *ga = p.g + ((long long)ra * p.H + h) * kDim + 2 * tig;
  uint16_t *gb = p.g + ((long long)rb * p.H + h) * kDim + 2 * tig;
#pragma unroll 4
  for (int nt = 0; nt < kDim / 8; ++nt) {
    const uint32_t *fb = reinterpret_cast<const uint32_t *>(fbs + (nt * 8 + grp) * kGateRow);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) mma_bf16_16816(d, a[ks], fb[ks * 8 + tig], fb[ks * 8 + 4 + tig]);
    if (la) *reinterpret_cast<uint32_t *>(ga + nt * 8) = pack_bf16x2(d[0], d[1]);
    if (lb) *reinterpret_cast<uint32_t *>(gb + nt * 8) = pack_bf16x2(d[2], d[3]);
  }
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

template <int Q>
int launch_prologue_q(const LayerParams &p, int items, cudaStream_t stream) {
  kda_layer_conv<Q><<<dim3(p.B, kConvCtas), kConvThreads, 0, stream>>>(p);
  const int n_tokens = p.B * Q;
  const dim3 grid((n_tokens + kGateTokens - 1) / kGateTokens, p.H);
  kda_layer_gate<<<grid, 256, 0, stream>>>(p, Q, n_tokens);
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
      !kda::aligned16(k) || !kda::aligned16(v) || conv_slot_stride % 8 != 0)
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
