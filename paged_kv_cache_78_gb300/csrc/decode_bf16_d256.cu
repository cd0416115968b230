// Decode kernels for bf16 elements, head size 256, query-group sizes 1..8.
#include "decode_inst.cuh"

PA_DEFINE_DECODE_UNIT(__nv_bfloat16, bf16, 256)
