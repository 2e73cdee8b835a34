// One-byte tensor-core kernel instances: int8 and fp8 e4m3 state, bf16
// inputs, 64 x 128, rounding to nearest and Philox stochastic rounding.
#include "rsm_instances.h"
#include "rsm_q8tc_kernel.cuh"

template const void* rsm::kernel_for_q8tc<RSM_I8, false>();
template const void* rsm::kernel_for_q8tc<RSM_I8, true>();
template const void* rsm::kernel_for_q8tc<RSM_FP8_E4M3, false>();
template const void* rsm::kernel_for_q8tc<RSM_FP8_E4M3, true>();
