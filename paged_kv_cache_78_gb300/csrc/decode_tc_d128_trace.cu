#include "decode_tc_inst.cuh"
PA_DEFINE_TC_UNIT(128, true, launch_tc_d128_trace)
