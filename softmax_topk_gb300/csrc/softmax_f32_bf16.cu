// Softmax kernels instantiated for input float, output __nv_bfloat16.
#include "internal.h"
#include "softmax_dispatch.cuh"

OS_DEFINE_SOFTMAX_PAIR(f32_bf16, float, __nv_bfloat16)
