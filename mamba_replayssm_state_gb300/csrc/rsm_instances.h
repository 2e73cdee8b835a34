// rsm_instances.h -- the compiled (state dtype, input dtype, dim, dstate)
// combinations.  One-byte state exists for (64, 128) only.
#pragma once

#define RSM_INSTANCES_WIDE(X, SF)                                                          \
  X(SF, RSM_BF16, 16, 16) X(SF, RSM_BF16, 64, 64) X(SF, RSM_BF16, 64, 128)                 \
  X(SF, RSM_F32, 16, 16) X(SF, RSM_F32, 64, 64) X(SF, RSM_F32, 64, 128)

#define RSM_INSTANCES_BYTE(X, SF) X(SF, RSM_BF16, 64, 128) X(SF, RSM_F32, 64, 128)

#define RSM_INSTANCES_F32(X) RSM_INSTANCES_WIDE(X, RSM_F32)
#define RSM_INSTANCES_BF16(X) RSM_INSTANCES_WIDE(X, RSM_BF16)
#define RSM_INSTANCES_F16(X) RSM_INSTANCES_WIDE(X, RSM_F16)
#define RSM_INSTANCES_Q8(X) RSM_INSTANCES_BYTE(X, RSM_I8) RSM_INSTANCES_BYTE(X, RSM_FP8_E4M3)

#define RSM_FOR_EACH_INSTANCE(X) \
  RSM_INSTANCES_F32(X) RSM_INSTANCES_BF16(X) RSM_INSTANCES_F16(X) RSM_INSTANCES_Q8(X)

namespace rsm {
// Defined (explicitly instantiated) in the rsm_inst_*.cu translation units:
// the kernel for philox_rounds == 0 (16-bit and fp32 state: for every call) ...
template <int SF, int IF, int D, int N>
const void* kernel_for();
// ... and, for one-byte state, the stochastic-rounding instance (rsm_inst_q8sr.cu).
template <int SF, int IF, int D, int N>
const void* kernel_for_sr();
// The tensor-core long-window variant (rsm_inst_tc.cu): 16-bit state, bf16 inputs, 64 x 128.
template <int SF>
const void* kernel_for_tc();
// The one-byte tensor-core kernel (rsm_inst_q8tc.cu): int8 / fp8 state, bf16
// inputs, 64 x 128, items of two heads; SR: Philox stochastic rounding.
template <int SF, bool SR>
const void* kernel_for_q8tc();
}  // namespace rsm
