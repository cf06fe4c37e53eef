// Softmax kernels instantiated for input __nv_bfloat16, output __nv_bfloat16.
#include "internal.h"
#include "softmax_dispatch.cuh"

OS_DEFINE_SOFTMAX_PAIR(bf16_bf16, __nv_bfloat16, __nv_bfloat16)
