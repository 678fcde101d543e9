// tc_gla.cu -- tcgen05 tensor-core CCQ-GLA forward (bf16 in, fp32 state).
#include "common.cuh"

namespace ccq {

bool tc_gla_supported(const CcqParams &) { return false; }

cudaError_t launch_tc_gla(const CcqParams &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ccq
