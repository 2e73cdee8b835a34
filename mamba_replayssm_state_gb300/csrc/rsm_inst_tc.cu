// Tensor-core (long-window) kernel instances: bf16 and fp16 state, bf16 inputs, 64 x 128.
#include "rsm_instances.h"
#include "rsm_tc_kernel.cuh"

template const void* rsm::kernel_for_tc<RSM_BF16>();
template const void* rsm::kernel_for_tc<RSM_F16>();
