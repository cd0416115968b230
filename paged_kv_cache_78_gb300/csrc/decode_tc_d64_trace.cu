#include "decode_tc_inst.cuh"
PA_DEFINE_TC_UNIT(64, true, launch_tc_d64_trace)
