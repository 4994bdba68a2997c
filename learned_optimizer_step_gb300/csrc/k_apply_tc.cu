// K2 (tensor-core path): placeholder until the tcgen05 kernel lands.
#include "lopt_internal.cuh"
#include "lopt.h"

namespace lopt {

bool apply_tc_supported(int) { return false; }

cudaError_t launch_apply_tc(const StepArgs&, cudaStream_t) { return cudaErrorNotSupported; }

int w1fold_floats(int hidden, int path) {
  (void)path;
  return (kStats + 1) * hidden;
}

}  // namespace lopt
