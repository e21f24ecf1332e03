// Persistent step kernels for windows of at most 7 token(s) given by
// query_start_loc.
#include "kda_step_launch.cuh"

namespace kda {
int launch_step_varlen_q7(const StepParams &p, int n_items, int variant, cudaStream_t stream) {
  return launch_ws_variant<7, true>(p, n_items, variant, stream);
}
}  // namespace kda
