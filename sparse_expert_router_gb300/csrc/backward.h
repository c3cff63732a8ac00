// Memory-bound kernels of the layer's backward (see backward.cu).
#pragma once

#include "common.cuh"

namespace moe {

// dy_perm[slot_of[t, j]] = gate[t, j] * dc[t] (bf16) and dgate[t, j] = <dc[t], y_perm[slot]>
// (fp32) for every kept assignment; dgate is 0 for dropped ones. dc, y_perm, dy_perm bf16.
cudaError_t combine_backward(const void* dc, const void* y_perm, const int32_t* slot_of,
                             const float* gate, int64_t T, int k, int L, int64_t pool_rows,
                             void* dy_perm, float* dgate, cudaStream_t st, bool pdl);

// dh[t] = sum over kept j of dx_perm[slot_of[t, j]]; with zhat = z rstd (rstd from z's mean
// square and eps): dz = rstd (dh gamma - zhat mean(dh gamma zhat)) as bf16, and
// dhz[t] = dh zhat (fp32, summed over t for the gain's gradient).
cudaError_t rms_backward(const void* dx_perm, const int32_t* slot_of, const float* z,
                         const float* gamma, float eps, int64_t T, int k, int L, int64_t pool_rows,
                         void* dz, float* dhz, cudaStream_t st, bool pdl);

// The selected logits' gradient dl_j = g_j (dgate_j - sum_i g_i dgate_i); dx[t] =
// bf16(dx32[t] + sum_j dl_j wrT[idx_j]) (wrT = W_r^T [E, d] bf16); dl32 / dlbf [T, E] the
// dense logit gradient (zero off the selection) in fp32 and bf16.
cudaError_t router_backward(const int32_t* idx, const float* gate, const float* dgate,
                            const void* wrT, const float* dx32, int64_t T, int k, int E, int d,
                            void* dx, float* dl32, void* dlbf, cudaStream_t st, bool pdl);

// p[0] = a, p[1] = b (device).
cudaError_t write_int2(int32_t* p, int32_t a, int32_t b, cudaStream_t st, bool pdl);

// out[c] = sum over r of m[r * cols + c], fp32, in a fixed order: COLSUM_CHUNKS row chunks are
// summed in parallel into partial [COLSUM_CHUNKS, cols], then the chunks in order.
constexpr int COLSUM_CHUNKS = 128;
cudaError_t column_sum(const float* m, int64_t rows, int cols, float* partial, float* out,
                       cudaStream_t st, bool pdl);

}  // namespace moe
