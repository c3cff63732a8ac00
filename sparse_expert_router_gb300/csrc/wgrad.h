// Weight-gradient GEMM over ragged row groups (see gemm_wgrad.cu).
#pragma once

#include <stdint.h>
#include <cuda_runtime.h>

namespace moe {

// For every group g and its rows r in [offsets[g], offsets[g+1]) (clamped to [0, rows)):
//   out[g][m][n] = sum_r a[r][m] * b[r][n],   m < M, n < N.
// a: [rows, M] and b: [rows, N] bf16 row-major; out: [G, M, N] bf16 (fp32 accumulation).
// Groups with no rows get zeros. M must be a multiple of 128 and N of 64.
struct WgradProblem {
  const void* a;
  const void* b;
  int64_t lda = 0, ldb = 0;   // elements between rows of a and b (0: M and N)
  const int32_t* offsets;   // [G + 1], device
  int G = 1;
  int M = 0, N = 0;
  int64_t rows = 0;
  void* out = nullptr;
};

cudaError_t gemm_wgrad(const WgradProblem* probs, int n_probs, void* dev_header,
                       cudaStream_t stream, bool pdl);
bool gemm_wgrad_supported(const WgradProblem& p);

}  // namespace moe
