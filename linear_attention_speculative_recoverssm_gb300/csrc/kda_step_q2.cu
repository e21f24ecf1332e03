// Step kernels for a window of 2 token(s).
#include "kda_step_launch.cuh"

namespace kda {
int launch_step_q2(const StepParams &p, int n_items, int variant, int split,
                    cudaStream_t stream) {
  return launch_step_q<2, false>(p, n_items, variant, split, stream);
}
int launch_step_layers_q2(const StepParams &p, const LayerBases &lay, int n_items,
                           cudaStream_t stream) {
  return launch_step_layers_q<2>(p, lay, n_items, stream);
}
}  // namespace kda
