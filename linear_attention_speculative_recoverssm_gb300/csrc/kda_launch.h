// Internal launch interface between the C ABI (kda_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

struct StepParams;
struct LayerBases;

// SMs of `dev`, cached after the first query.
int device_sm_count(int dev);

// The replay / verify step for window Q (1..8).
//   variant 0: verify only, FP32 pool      1: verify only, BF16 pool
//           2: replay + verify (FP32)      3: replay + verify + boundary
//           4: replay + verify with the gated RMSNorm folded in (split 1,
//              uniform windows)
//   split   1: persistent CTAs; 2 / 4: cluster of that many CTAs per item.
int launch_step(const StepParams &p, int n_items, int Q, int variant, int split,
                cudaStream_t stream);

// The multi-layer replay + verify for window Q (1..8), persistent CTAs.
int launch_step_layers(const StepParams &p, const LayerBases &lay, int n_items, int Q,
                       cudaStream_t stream);

int launch_commit(const uint64_t *state_ptrs, const uint64_t *corr_ptrs, const uint64_t *kg_ptrs,
                  const int64_t *state_strides, const int64_t *corr_strides,
                  const int64_t *kg_strides, const float *A_log, const float *dt_bias,
                  const int32_t *sources, const int32_t *commit_lens,
                  const int32_t *destinations, const int32_t *boundaries,
                  const int32_t *boundary_lens, const int32_t *record_rows, int state_dtype,
                  float lower_bound, int null_slot, int L, int H, int B, int Q, int n_slots,
                  int n_rows, int32_t *status, cudaStream_t stream);

int launch_defer_commit(const int32_t *state_slots, int32_t *commit_lens,
                        const int32_t *record_rows, int32_t *pending, const uint8_t *eager, int B,
                        int null_slot, int n_rows, int32_t *status, cudaStream_t stream);

int launch_flush_plan(const int32_t *state_slots, const int32_t *record_rows,
                      const int32_t *pending, int32_t *commit_lens, int32_t *final_slots,
                      int32_t *boundary_slots, int32_t *boundary_lens, int B, int Q,
                      int null_slot, int n_rows, int32_t *status, cudaStream_t stream);

int launch_selftest_timeout(int32_t *status, cudaStream_t stream);

}  // namespace kda
