// Softmax kernels instantiated for input __nv_bfloat16, output float.
#include "internal.h"
#include "softmax_dispatch.cuh"

OS_DEFINE_SOFTMAX_PAIR(bf16_f32, __nv_bfloat16, float)
