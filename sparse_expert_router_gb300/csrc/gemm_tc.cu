// tcgen05 GEMM (placeholder until the tensor-core kernel lands).
#include "common.cuh"
#include "gemm.h"

namespace moe {
bool gemm_tc_supported(const GemmProblem&) { return false; }
cudaError_t gemm_tc(const GemmProblem*, int, void*, cudaStream_t, bool) {
  return cudaErrorNotSupported;
}
}  // namespace moe
