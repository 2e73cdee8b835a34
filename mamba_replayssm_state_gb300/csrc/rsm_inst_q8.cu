// Kernel instances for one-byte state, rounding to nearest (compiled as its own
// translation unit so that the library builds in parallel).
#include "rsm_instances.h"
#include "rsm_q8_kernel.cuh"

#define RSM_INSTANTIATE(SF, IF, D, N) template const void* rsm::kernel_for<SF, IF, D, N>();
RSM_INSTANCES_Q8(RSM_INSTANTIATE)
