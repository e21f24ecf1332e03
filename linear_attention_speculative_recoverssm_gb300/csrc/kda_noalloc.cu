// kda_layer_step_noalloc: the fused layer step for callers that cannot
// allocate device memory when they call it.  A serving runtime that reserves
// all device memory in its own pool at start-up, or a plugin whose host
// framework owns every device allocation, may not call cudaMalloc on the
// decode path (it could fail, stall, or break the framework's accounting).
// kda_layer_step needs a caller workspace for the step's operands; this entry
// point uses a fixed array of device memory that belongs to the library
// instead, so the caller passes inputs and outputs only.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it, whether or not this entry point is called.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/kda_recoverssm.h"

namespace {

// The step's q, k, v and raw_g of one call (kda_layer_step's workspace).
static __device__ __align__(256) unsigned char g_layer_step_scratch[KDA_LAYER_STEP_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
// Device address of the array on each device, 0 until that device's first
// call looks it up.  (In host code the array's name is only a stand-in for
// the symbol, never an address a kernel may use.)
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];

// The array's address on the current device.  The first call on a device
// asks the runtime for it (with that device current); later calls reuse it.
// Two threads racing on the first call store the same value.
int scratch_on_current_device(void **addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layer_step_scratch) != cudaSuccess || p == nullptr)
      return KDA_ERR_CUDA;
    a = reinterpret_cast<uintptr_t>(p);
    g_scratch_addr[dev].store(a, std::memory_order_release);
  }
  *addr = reinterpret_cast<void *>(a);
  return KDA_OK;
}

}  // namespace

extern "C" int kda_layer_step_noalloc(
    const kda_bf16 *x, const kda_bf16 *conv_weight, const kda_bf16 *conv_bias,
    kda_bf16 *conv_state, int64_t conv_slot_stride, const kda_bf16 *f_a, const kda_bf16 *f_b,
    const kda_bf16 *raw_beta, const float *A_log, const float *dt_bias, float lower_bound,
    float q_scale, float *state_pool, int64_t slot_stride, int n_slots,
    const int32_t *state_slots, const int32_t *record_rows, const int32_t *pending, float *corr,
    kda_bf16 *key_gate, int64_t corr_row_stride, int64_t kg_row_stride, int n_rows, int rq,
    const kda_bf16 *gate, const float *norm_weight, float eps, kda_bf16 *out, int B, int H, int Q,
    int null_slot, int32_t *status, void *stream) {
  const int64_t need = kda_layer_step_workspace_bytes(B, H, Q);
  if (need < 0) return KDA_ERR_ARG;
  if (need > KDA_LAYER_STEP_NOALLOC_MAX_BYTES) return KDA_ERR_SCRATCH;
  if (B == 0) return KDA_OK;
  void *scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != KDA_OK) return rc;
  // Nothing in the array needs clearing: the step reads only the operands
  // this call's prologue has just written there.
  return kda_layer_step(x, conv_weight, conv_bias, conv_state, conv_slot_stride, f_a, f_b,
                        raw_beta, A_log, dt_bias, lower_bound, q_scale, state_pool, slot_stride,
                        n_slots, state_slots, record_rows, pending, corr, key_gate,
                        corr_row_stride, kg_row_stride, n_rows, rq, gate, norm_weight, eps, out,
                        scratch, (int64_t)KDA_LAYER_STEP_NOALLOC_MAX_BYTES, B, H, Q, null_slot,
                        status, stream);
}
