// The gated-delta-rule commit kernel, compiled in its own translation unit.
#include "gdn_kernel.cuh"

namespace gdn {
const void* commit_kernel() { return reinterpret_cast<const void*>(&gdn_commit_kernel); }
}  // namespace gdn
