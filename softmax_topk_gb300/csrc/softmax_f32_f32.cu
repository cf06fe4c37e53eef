// Softmax kernels instantiated for input float, output float.
#include "internal.h"
#include "softmax_dispatch.cuh"

OS_DEFINE_SOFTMAX_PAIR(f32_f32, float, float)
