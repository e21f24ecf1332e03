// Host-side launch of the step kernels for one window size Q; included by
// the per-Q translation units kda_step_q<Q>.cu so they compile in parallel.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kda_launch.h"
#include "kda_step.cuh"
#include "kda_step_cluster.cuh"
#include "kda_step_ws.cuh"

namespace kda {

// cuTensorMapEncodeTiled from the driver, looked up once.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// The four token-major inputs [n_tokens, H, 128] (BF16) as 3-D tensors (128,
// H, n_tokens) with a (128, 1, Q) box: one item's window rows per copy (rows
// past the activations arrive as zeros).
template <int Q>
int encode_token_maps(const StepParams &p, WsMaps &maps) {
  const auto encode = tensor_map_encoder();
  if (encode == nullptr) return KDA_ERR_CUDA;
  const uint16_t *src[4] = {p.q, p.k, p.g, p.v};
  const cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)p.H, (cuuint64_t)p.n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)p.H * kDim * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kDim, 1, (cuuint32_t)Q};
  const cuuint32_t estride[3] = {1, 1, 1};
  for (int x = 0; x < 4; ++x) {
    if (encode(&maps.tok[x], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<uint16_t *>(src[x]), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

// The stacked inputs of the multi-layer step [L, n_tokens, H, 128] as 4-D
// tensors (128, H, n_tokens, L) with a (128, 1, Q, 1) box.
template <int Q>
int encode_layer_token_maps(const StepParams &p, const LayerBases &lay, WsMaps &maps) {
  const auto encode = tensor_map_encoder();
  if (encode == nullptr) return KDA_ERR_CUDA;
  const uint16_t *src[4] = {p.q, p.k, p.g, p.v};
  const cuuint64_t dims[4] = {(cuuint64_t)kDim, (cuuint64_t)p.H, (cuuint64_t)p.n_tokens,
                              (cuuint64_t)lay.L};
  const cuuint64_t strides[3] = {(cuuint64_t)kDim * 2, (cuuint64_t)p.H * kDim * 2,
                                 (cuuint64_t)lay.act_stride * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kDim, 1, (cuuint32_t)Q, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  for (int x = 0; x < 4; ++x) {
    if (encode(&maps.tok[x], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<uint16_t *>(src[x]), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

template <int Q, typename ST, bool REPLAY, bool BOUNDARY, bool VARLEN, bool LAYERS = false,
          bool NORM = false>
int launch_ws(const StepParams &p, int n_items, cudaStream_t stream,
              const LayerBases *bases = nullptr) {
  auto kern = kda_step_ws<Q, ST, REPLAY, BOUNDARY, VARLEN, LAYERS, NORM>;
  constexpr size_t smem = sizeof(WsSmem<Q, ST, BOUNDARY, NORM>);
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return KDA_ERR_CUDA;
    configured.fetch_or(bit);
  }
  const int sms = device_sm_count(dev);
  const int grid = n_items < sms ? n_items : sms;
  WsMaps maps;
  WsLayers<LAYERS> lay{};
  int st;
  if constexpr (LAYERS) {
    static_cast<LayerBases &>(lay) = *bases;
    st = encode_layer_token_maps<Q>(p, *bases, maps);
  } else {
    (void)bases;
    st = encode_token_maps<Q>(p, maps);
  }
  if (st != KDA_OK) return st;
  kern<<<grid, kWsThreads, smem, stream>>>(p, maps, lay, n_items);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// The multi-layer replay + verify (persistent kernel, uniform windows).
template <int Q>
int launch_step_layers_q(const StepParams &p, const LayerBases &lay, int n_items,
                         cudaStream_t stream) {
  return launch_ws<Q, float, true, false, false, true>(p, n_items, stream, &lay);
}

template <int Q, int SPLIT, bool BOUNDARY, bool VARLEN>
int launch_cluster(const StepParams &p, int n_items, cudaStream_t stream) {
  auto kern = kda_step_cluster<Q, SPLIT, BOUNDARY, VARLEN>;
  constexpr size_t smem = sizeof(ClusterSmem<Q, SPLIT, BOUNDARY>);
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return KDA_ERR_CUDA;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(SPLIT, (unsigned)n_items, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return KDA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// The persistent kernel for one variant: 0 verify (FP32 state), 1 verify
// (BF16 state), 2 replay + verify, 3 replay + verify with boundary states,
// 4 replay + verify with the gated RMSNorm folded in (uniform windows).
template <int Q, bool VARLEN>
int launch_ws_variant(const StepParams &p, int n_items, int variant, cudaStream_t stream) {
  switch (variant) {
    case 0: return launch_ws<Q, float, false, false, VARLEN>(p, n_items, stream);
    case 1: return launch_ws<Q, uint16_t, false, false, VARLEN>(p, n_items, stream);
    case 2: return launch_ws<Q, float, true, false, VARLEN>(p, n_items, stream);
    case 3: return launch_ws<Q, float, true, true, VARLEN>(p, n_items, stream);
    case 4:
      if constexpr (VARLEN) return KDA_ERR_UNSUPPORTED;
      else return launch_ws<Q, float, true, false, false, false, true>(p, n_items, stream);
    default: return KDA_ERR_ARG;
  }
}

// One window kind (VARLEN: windows from query_start_loc; its instances live
// in kda_step_varlen_q<Q>.cu, the uniform ones in kda_step_q<Q>.cu).  Split
// 1 is the persistent kernel; 2 or 4 the cluster split, which serves the
// fused FP32 replay + verify.
template <int Q, bool VARLEN>
int launch_step_q(const StepParams &p, int n_items, int variant, int split,
                  cudaStream_t stream) {
  if (split == 1) return launch_ws_variant<Q, VARLEN>(p, n_items, variant, stream);
  if (variant != 2 && variant != 3) return KDA_ERR_UNSUPPORTED;  // (the norm: split 1 only)
  const bool bnd = variant == 3;
  if (split == 2)
    return bnd ? launch_cluster<Q, 2, true, VARLEN>(p, n_items, stream)
               : launch_cluster<Q, 2, false, VARLEN>(p, n_items, stream);
  if (split == 4)
    return bnd ? launch_cluster<Q, 4, true, VARLEN>(p, n_items, stream)
               : launch_cluster<Q, 4, false, VARLEN>(p, n_items, stream);
  return KDA_ERR_ARG;
}

}  // namespace kda
