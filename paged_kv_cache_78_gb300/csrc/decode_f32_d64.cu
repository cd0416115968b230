// Decode kernels for f32 elements, head size 64, query-group sizes 1..8.
#include "decode_inst.cuh"

PA_DEFINE_DECODE_UNIT(float, f32, 64)
