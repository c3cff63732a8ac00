// The layer backward's memory-bound steps around its GEMMs: the combine's backward (scatter of
// the gate-weighted output gradient to the expert rows and the gates' gradient), the
// un-permute with the RMSNorm backward, the router's softmax backward with its input-gradient
// term, and a column sum for the bias and gain gradients. One block per token (or column
// range); every reduction runs in a fixed order, so results are bitwise reproducible.
#include "backward.h"

namespace moe {
namespace {

constexpr int BT = 128;   // threads per token block

// Sum of v over the block (4 warps) in a fixed order; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* s_red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
  __syncthreads();
  return (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
}

__global__ void __launch_bounds__(BT) combine_backward_kernel(
    const bf16* dc, const bf16* y_perm, const int32_t* slot_of, const float* gate, int64_t T,
    int k, int L, int64_t pool_rows, bf16* dy_perm, float* dgate) {
  pdl_wait();
  __shared__ float s_red[4];
  const int64_t t = blockIdx.x;
  const bf16* dct = dc + t * L;
  for (int j = 0; j < k; ++j) {
    const int32_t s = slot_of[t * k + j];
    if (s < 0 || s >= pool_rows) {           // dropped (or padding): no row, no gate gradient
      if (threadIdx.x == 0) dgate[t * k + j] = 0.0f;
      continue;
    }
    const float g = gate[t * k + j];
    const bf16* yr = y_perm + (int64_t)s * L;
    bf16* dr = dy_perm + (int64_t)s * L;
    float dot = 0.0f;
    for (int i = threadIdx.x * 8; i < L; i += BT * 8) {
      float a[8], b[8], o[8];
      ld8(dct + i, a);
      ld8(yr + i, b);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dot = fmaf(a[q], b[q], dot);
        o[q] = g * a[q];
      }
      st8(dr + i, o);
    }
    dot = block_sum(dot, s_red);
    if (threadIdx.x == 0) dgate[t * k + j] = dot;
  }
}

__global__ void __launch_bounds__(BT) rms_backward_kernel(
    const bf16* dx_perm, const int32_t* slot_of, const float* z, const float* gamma, float eps,
    int64_t T, int k, int L, int64_t pool_rows, bf16* dz, float* dhz) {
  pdl_wait();
  __shared__ float s_red[4];
  const int64_t t = blockIdx.x;
  const float* zt = z + t * L;
  int32_t slots[32];
  int ns = 0;
  for (int j = 0; j < k; ++j) {
    const int32_t s = slot_of[t * k + j];
    if (s >= 0 && s < pool_rows) slots[ns++] = s;
  }
  // rstd from the row's mean square, as in the forward's gather
  float ss = 0.0f;
  for (int i = threadIdx.x * 8; i < L; i += BT * 8) {
    float v[8];
    ld8(zt + i, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
  }
  ss = block_sum(ss, s_red);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)L), eps)));
  // first pass: dot = sum dh gamma zhat
  float dot = 0.0f;
  for (int i = threadIdx.x * 8; i < L; i += BT * 8) {
    float dh[8] = {0, 0, 0, 0, 0, 0, 0, 0}, v[8], g[8];
    for (int j = 0; j < ns; ++j) {
      float r[8];
      ld8(dx_perm + (int64_t)slots[j] * L + i, r);
#pragma unroll
      for (int q = 0; q < 8; ++q) dh[q] += r[q];
    }
    ld8(zt + i, v);
    ld8(gamma + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) dot = fmaf(dh[q] * g[q], v[q] * rstd, dot);
  }
  const float mean = block_sum(dot, s_red) / (float)L;
  // second pass: dz and dh zhat
  for (int i = threadIdx.x * 8; i < L; i += BT * 8) {
    float dh[8] = {0, 0, 0, 0, 0, 0, 0, 0}, v[8], g[8], o[8], p[8];
    for (int j = 0; j < ns; ++j) {
      float r[8];
      ld8(dx_perm + (int64_t)slots[j] * L + i, r);
#pragma unroll
      for (int q = 0; q < 8; ++q) dh[q] += r[q];
    }
    ld8(zt + i, v);
    ld8(gamma + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float zh = v[q] * rstd;
      o[q] = rstd * (dh[q] * g[q] - zh * mean);
      p[q] = dh[q] * zh;
    }
    st8(dz + t * L + i, o);
    st8(dhz + t * L + i, p);
  }
}

__global__ void __launch_bounds__(256) router_backward_kernel(
    const int32_t* idx, const float* gate, const float* dgate, const bf16* wrT, const float* dx32,
    int64_t T, int k, int E, int d, bf16* dx, float* dl32, bf16* dlbf) {
  pdl_wait();
  const int64_t t = blockIdx.x;
  float dl[32];
  int32_t ids[32];
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = fmaf(gate[t * k + j], dgate[t * k + j], s);
  for (int j = 0; j < k; ++j) {
    ids[j] = idx[t * k + j];
    dl[j] = gate[t * k + j] * (dgate[t * k + j] - s);
  }
  for (int i = threadIdx.x * 8; i < d; i += 256 * 8) {
    float acc[8];
    ld8(dx32 + t * d + i, acc);
    for (int j = 0; j < k; ++j) {
      float w[8];
      ld8(wrT + (int64_t)ids[j] * d + i, w);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(dl[j], w[q], acc[q]);
    }
    st8(dx + t * d + i, acc);
  }
  for (int e = threadIdx.x; e < E; e += 256) {
    float v = 0.0f;
    for (int j = 0; j < k; ++j) v = (ids[j] == e) ? dl[j] : v;
    dl32[t * E + e] = v;
    dlbf[t * E + e] = __float2bfloat16_rn(v);
  }
}

// Block (x, y): columns 256x.., rows of chunk y; partial[y][c] = the chunk's column sums.
__global__ void __launch_bounds__(256) column_partial_kernel(const float* m, int64_t rows,
                                                             int cols, float* partial) {
  pdl_wait();
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= cols) return;
  const int64_t per = cdiv(rows, (int64_t)gridDim.y);
  const int64_t r0 = blockIdx.y * per, r1 = imin64(rows, r0 + per);
  float acc = 0.0f;
  for (int64_t r = r0; r < r1; ++r) acc += m[r * cols + c];
  partial[(int64_t)blockIdx.y * cols + c] = acc;
}

__global__ void __launch_bounds__(256) column_final_kernel(const float* partial, int chunks,
                                                           int cols, float* out) {
  pdl_wait();
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= cols) return;
  float acc = 0.0f;
  for (int y = 0; y < chunks; ++y) acc += partial[(int64_t)y * cols + c];
  out[c] = acc;
}

__global__ void write_int2_kernel(int32_t* p, int32_t a, int32_t b) {
  pdl_wait();
  if (threadIdx.x == 0) { p[0] = a; p[1] = b; }
}

}  // namespace

cudaError_t write_int2(int32_t* p, int32_t a, int32_t b, cudaStream_t st, bool pdl) {
  return launch(write_int2_kernel, dim3(1), dim3(32), 0, st, pdl, p, a, b);
}

cudaError_t combine_backward(const void* dc, const void* y_perm, const int32_t* slot_of,
                             const float* gate, int64_t T, int k, int L, int64_t pool_rows,
                             void* dy_perm, float* dgate, cudaStream_t st, bool pdl) {
  return launch(combine_backward_kernel, dim3((unsigned)T), dim3(BT), 0, st, pdl,
                static_cast<const bf16*>(dc), static_cast<const bf16*>(y_perm), slot_of, gate, T,
                k, L, pool_rows, static_cast<bf16*>(dy_perm), dgate);
}

cudaError_t rms_backward(const void* dx_perm, const int32_t* slot_of, const float* z,
                         const float* gamma, float eps, int64_t T, int k, int L, int64_t pool_rows,
                         void* dz, float* dhz, cudaStream_t st, bool pdl) {
  return launch(rms_backward_kernel, dim3((unsigned)T), dim3(BT), 0, st, pdl,
                static_cast<const bf16*>(dx_perm), slot_of, z, gamma, eps, T, k, L, pool_rows,
                static_cast<bf16*>(dz), dhz);
}

cudaError_t router_backward(const int32_t* idx, const float* gate, const float* dgate,
                            const void* wrT, const float* dx32, int64_t T, int k, int E, int d,
                            void* dx, float* dl32, void* dlbf, cudaStream_t st, bool pdl) {
  return launch(router_backward_kernel, dim3((unsigned)T), dim3(256), 0, st, pdl, idx, gate,
                dgate, static_cast<const bf16*>(wrT), dx32, T, k, E, d, static_cast<bf16*>(dx),
                dl32, static_cast<bf16*>(dlbf));
}

cudaError_t column_sum(const float* m, int64_t rows, int cols, float* partial, float* out,
                       cudaStream_t st, bool pdl) {
  const unsigned cx = (unsigned)cdiv(cols, 256);
  cudaError_t e = launch(column_partial_kernel, dim3(cx, COLSUM_CHUNKS), dim3(256), 0, st, pdl,
                         m, rows, cols, partial);
  if (e != cudaSuccess) return e;
  return launch(column_final_kernel, dim3(cx), dim3(256), 0, st, pdl, (const float*)partial,
                COLSUM_CHUNKS, cols, out);
}

}  // namespace moe
