// Step kernels for windows of at most 7 token(s) given by query_start_loc.
#include "kda_step_launch.cuh"

namespace kda {
int launch_step_varlen_q7(const StepParams &p, int n_items, int variant, int split,
                           cudaStream_t stream) {
  return launch_step_q<7, true>(p, n_items, variant, split, stream);
}
}  // namespace kda
