// The gated-delta-rule commit kernels (fp32, and the tcgen05 backend),
// compiled in their own translation unit.
#include "gdn_kernel.cuh"
#include "gdn_tc_kernel.cuh"

namespace gdn {
const void* commit_kernel() { return reinterpret_cast<const void*>(&gdn_commit_kernel); }
const void* commit_tc_kernel() { return reinterpret_cast<const void*>(&gdn_commit_tc_kernel); }
}  // namespace gdn
