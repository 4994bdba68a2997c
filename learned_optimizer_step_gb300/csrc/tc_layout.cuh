// Operand layouts of the tensor-core apply path (placeholder).
#pragma once
#include "lopt_internal.cuh"

namespace lopt {
__device__ inline void fold_w1_tc(int, const float*, const float*, const double*, double, float*) {}
}  // namespace lopt
