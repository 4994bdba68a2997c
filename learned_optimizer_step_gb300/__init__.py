"""GB300-native learned-optimizer step (small_fc_lopt kind).

The compute lives in liblopt.so (C ABI in include/lopt.h, CUDA kernels for
sm_103a); this package holds the in-tree build and the ctypes binding."""
from .lopt import (LearnedOptimizer, LoptError, PreparedList, TensorState,  # noqa: F401
                   load_library, schedule_info, weight_set_size, zeros_state, MLP_FP32, MLP_TC)
