// Step kernels for a window of 4 token(s).
#include "kda_step_launch.cuh"

namespace kda {
int launch_step_q4(const StepParams &p, int n_items, int variant, int split,
                    cudaStream_t stream) {
  return launch_step_q<4, false>(p, n_items, variant, split, stream);
}
int launch_step_layers_q4(const StepParams &p, const LayerBases &lay, int n_items,
                           cudaStream_t stream) {
  return launch_step_layers_q<4>(p, lay, n_items, stream);
}
}  // namespace kda
