// Deferred RecoverSSM bookkeeping -- page "vllm.models.kimi_k3.nvidia.
// specialized_decode.recoverssm.kernels": _defer_commit_kernel (after
// sampling, move each request's commit length into the pending count of its
// record slot) and _prepare_flush_plan_kernel (the in-place commit plan of
// the pending replays).  One thread per request; integer work only.
#include <cuda_runtime.h>

#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

__global__ void kda_defer_commit_kernel(const int32_t *state_slots, int32_t *commit_lens,
                                        const int32_t *record_rows, int32_t *pending,
                                        const uint8_t *eager, int B, int null_slot, int n_rows,
                                        int32_t *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int rec = record_rows[b];
  const int slot = state_slots[b];
  if (rec < 0 || slot <= null_slot) return;
  if (rec >= n_rows) {
    report(status, KDA_ERR_ARG);
    return;
  }
  if (eager != nullptr && eager[b] != 0) {
    pending[rec] = 0;
  } else {
    pending[rec] = commit_lens[b];
    commit_lens[b] = 0;
  }
}

__global__ void kda_flush_plan_kernel(const int32_t *state_slots, const int32_t *record_rows,
                                      const int32_t *pending, int32_t *commit_lens,
                                      int32_t *final_slots, int32_t *boundary_slots,
                                      int32_t *boundary_lens, int B, int Q, int null_slot,
                                      int n_rows, int32_t *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int slot = state_slots[b];
  const int rec = record_rows[b];
  int len = 0;
  if (rec >= 0) {
    if (rec < n_rows) {
      len = pending[rec];
    } else {
      report(status, KDA_ERR_ARG);
    }
  }
  len = len < 0 ? 0 : (len > Q ? Q : len);
  commit_lens[b] = (slot > null_slot && len > 0) ? len : 0;
  final_slots[b] = slot;
  boundary_slots[b] = null_slot;
  boundary_lens[b] = 0;
}

// Failure-detection self-test: a bounded wait on a barrier whose phase
// nothing completes.  The wait gives up after the library's fixed limit and
// the kernel reports KDA_ERR_TIMEOUT, exactly as the step kernels do when a
// copy or a hand-off never arrives; nothing faults and nothing hangs.
__global__ void kda_selftest_timeout_kernel(int32_t *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0u);
  if (!ok && threadIdx.x == 0) report(status, KDA_ERR_TIMEOUT);
}

constexpr int kBookThreads = 128;

}  // namespace

int launch_defer_commit(const int32_t *state_slots, int32_t *commit_lens,
                        const int32_t *record_rows, int32_t *pending, const uint8_t *eager, int B,
                        int null_slot, int n_rows, int32_t *status, cudaStream_t stream) {
  const int grid = (B + kBookThreads - 1) / kBookThreads;
  kda_defer_commit_kernel<<<grid, kBookThreads, 0, stream>>>(
      state_slots, commit_lens, record_rows, pending, eager, B, null_slot, n_rows, status);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int launch_flush_plan(const int32_t *state_slots, const int32_t *record_rows,
                      const int32_t *pending, int32_t *commit_lens, int32_t *final_slots,
                      int32_t *boundary_slots, int32_t *boundary_lens, int B, int Q,
                      int null_slot, int n_rows, int32_t *status, cudaStream_t stream) {
  const int grid = (B + kBookThreads - 1) / kBookThreads;
  kda_flush_plan_kernel<<<grid, kBookThreads, 0, stream>>>(
      state_slots, record_rows, pending, commit_lens, final_slots, boundary_slots,
      boundary_lens, B, Q, null_slot, n_rows, status);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int launch_selftest_timeout(int32_t *status, cudaStream_t stream) {
  kda_selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
