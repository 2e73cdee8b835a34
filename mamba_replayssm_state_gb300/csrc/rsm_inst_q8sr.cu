// Kernel instances for one-byte state with Philox stochastic rounding.
#include "rsm_instances.h"
#include "rsm_q8_kernel.cuh"

#define RSM_INSTANTIATE(SF, IF, D, N) template const void* rsm::kernel_for_sr<SF, IF, D, N>();
RSM_INSTANCES_Q8(RSM_INSTANTIATE)
