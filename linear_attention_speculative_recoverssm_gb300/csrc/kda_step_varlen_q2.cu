// Step kernels for windows of at most 2 token(s) given by query_start_loc.
#include "kda_step_launch.cuh"

namespace kda {
int launch_step_varlen_q2(const StepParams &p, int n_items, int variant, int split,
                           cudaStream_t stream) {
  return launch_step_q<2, true>(p, n_items, variant, split, stream);
}
}  // namespace kda
