// CUDA-core GEMM for the fp32 configuration and as the bf16 cross-check path.
//
// 64 x 64 output tile per 256-thread block, 4 x 4 outputs per thread, k staged 16 at a time
// through shared memory, the next step's tile loaded into registers while the current one is
// multiplied. Every output is accumulated sequentially over k with fused
// multiply-adds, so its rounding error is bounded by gamma_K * sum_k |a_k w_k| (the router's
// certified top-k relies on this bound).
#include "common.cuh"
#include "gemm.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename T>
__device__ __forceinline__ const T* weight_ptr(const GemmProblem& p, const GemmSeg& s,
                                               const void* base, int g, int k, int c) {
  const T* w = static_cast<const T*>(base);
  if (p.group == GROUP_ROWS) return w + ((int64_t)g * s.K + k) * p.M + c;
  if (p.group == GROUP_COLS) return w + ((int64_t)(c / p.Mg) * s.K + k) * p.Mg + (c % p.Mg);
  return w + (int64_t)k * p.M + c;
}

// Up to three independent problems per launch (the front GEMMs: router, down-projection,
// shared gate/up), problem blockIdx.z; blocks past a problem's tiles leave at once.
constexpr int SIMT_MAX_PROBS = 3;
struct SimtLaunch {
  GemmProblem p[SIMT_MAX_PROBS];
};

__host__ __device__ __forceinline__ int64_t simt_row_tiles(const GemmProblem& p) {
  return cdiv(p.rows, BM) + (p.group == GROUP_ROWS ? p.G : 0);
}

template <typename T>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(const __grid_constant__ SimtLaunch L) {
  const GemmProblem& p = L.p[blockIdx.z];
  if ((int64_t)blockIdx.x >= simt_row_tiles(p) || (int64_t)blockIdx.y * BN >= p.M) return;
  pdl_wait();
  __shared__ float sA[BK][BM + 4];
  __shared__ float sW[BK][BN];
  __shared__ float sW3[BK][BN];
  __shared__ int s_g, s_r0, s_r1;

  const int tid = threadIdx.x;
  const int c0 = blockIdx.y * BN;
  if (tid == 0) {
    int g = 0, r0 = 0, r1 = 0;
    if (p.group == GROUP_ROWS) {
      // map the linear tile index onto (group, row tile) with clamped, monotone offsets
      int64_t want = blockIdx.x, prev = 0;
      g = -1;
      for (int gg = 0; gg < p.G; ++gg) {
        int64_t lo = imin64(imax64((int64_t)p.offsets[gg], prev), p.rows);
        int64_t hi = imin64(imax64((int64_t)p.offsets[gg + 1], lo), p.rows);
        prev = hi;
        int64_t nt = (hi - lo + BM - 1) / BM;
        if (want < nt) { g = gg; r0 = (int)(lo + want * BM); r1 = (int)imin64(hi, (int64_t)r0 + BM); break; }
        want -= nt;
      }
    } else {
      r0 = blockIdx.x * BM;
      r1 = (int)imin64(p.rows, (int64_t)r0 + BM);
    }
    s_g = g; s_r0 = r0; s_r1 = r1;
  }
  __syncthreads();
  const int g = s_g, r0 = s_r0, r1 = s_r1;
  if (g < 0 || r0 >= r1) return;

  const bool glu = (p.epi == EPI_SWIGLU);
  const int tx = tid % 16, ty = tid / 16;   // thread owns rows ty*4.., cols tx*4..
  float acc[4][4] = {}, acc3[4][4] = {};

  // The k steps of all segments in order. Each step's tile is loaded into registers one step
  // ahead (all of a thread's loads issued together, then stored to shared memory), so the loads
  // of step s+1 are in flight while step s is multiplied; the accumulation order over k is that
  // of the segments' k.
  constexpr int A_PER = BM * BK / NT, W_PER = BK * BN / NT;
  int n_steps = 0;
  for (int si = 0; si < p.n_seg; ++si) n_steps += (p.seg[si].K + BK - 1) / BK;
  float ra[A_PER], rw[W_PER], rw3[W_PER];
  auto load_step = [&](int step) {
    int si = 0, k0 = step * BK;   // segment si, k offset k0 within it
    while (k0 >= ((p.seg[si].K + BK - 1) / BK) * BK) {
      k0 -= ((p.seg[si].K + BK - 1) / BK) * BK;
      ++si;
    }
    const GemmSeg& sg = p.seg[si];
    const T* act = static_cast<const T*>(sg.act);
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      const int idx = tid + i * NT, rr = idx / BK, kk = idx % BK;
      const int r = r0 + rr, k = k0 + kk;
      ra[i] = (r < r1 && k < sg.K) ? ld_f(act, (int64_t)r * sg.K + k) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < W_PER; ++i) {
      const int idx = tid + i * NT, kk = idx / BN, cc = idx % BN;
      const int k = k0 + kk, c = c0 + cc;
      const bool ok = (k < sg.K && c < p.M);
      rw[i] = ok ? ld_f(weight_ptr<T>(p, sg, sg.w, g, k, c), 0) : 0.0f;
      rw3[i] = (ok && glu) ? ld_f(weight_ptr<T>(p, sg, sg.w3, g, k, c), 0) : 0.0f;
    }
  };
  if (n_steps > 0) load_step(0);
  for (int step = 0; step < n_steps; ++step) {
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      const int idx = tid + i * NT;
      sA[idx % BK][idx / BK] = ra[i];
    }
#pragma unroll
    for (int i = 0; i < W_PER; ++i) {
      const int idx = tid + i * NT;
      sW[idx / BN][idx % BN] = rw[i];
      sW3[idx / BN][idx % BN] = rw3[i];
    }
    __syncthreads();
    if (step + 1 < n_steps) load_step(step + 1);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], w[4], w3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) { w[j] = sW[kk][tx * 4 + j]; w3[j] = glu ? sW3[kk][tx * 4 + j] : 0.0f; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
          if (glu) acc3[i][j] = fmaf(a[i], w3[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int r = r0 + ty * 4 + i;
    if (r >= r1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int c = c0 + tx * 4 + j;
      if (c >= p.M) continue;
      int64_t o = (int64_t)r * p.ld_out + p.out_col0 + c;
      if (p.epi == EPI_F32) {
        float v = acc[i][j];
        if (p.bias) v = __fadd_rn(v, p.bias[c]);
        static_cast<float*>(p.out)[o] = v;
      } else if (p.epi == EPI_SWIGLU) {
        st_f(static_cast<T*>(p.out), o,
             sizeof(T) == 4 ? swiglu_ieee(acc[i][j], acc3[i][j]) : swiglu(acc[i][j], acc3[i][j]));
      } else {
        st_f(static_cast<T*>(p.out), o, acc[i][j]);
      }
    }
  }
}

}  // namespace

cudaError_t gemm_simt(const GemmProblem* probs, int n, cudaStream_t stream, bool pdl) {
  SimtLaunch L{};
  int m = 0;
  int64_t gx = 0, gy = 0;
  auto flush = [&]() -> cudaError_t {
    if (m == 0) return cudaSuccess;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)m);
    const bool bf = L.p[0].dtype == DT_BF16;
    cudaError_t e = bf ? launch(simt_gemm_kernel<bf16>, grid, dim3(NT), 0, stream, pdl, L)
                       : launch(simt_gemm_kernel<float>, grid, dim3(NT), 0, stream, pdl, L);
    m = 0;
    gx = gy = 0;
    return e;
  };
  for (int i = 0; i < n; ++i) {
    const GemmProblem& p = probs[i];
    // fp8, transposed weights and the backward epilogues run on tensor cores only
    if (p.w_fp8 || p.out_fp8 || p.a_kmajor || p.epi > EPI_SWIGLU) return cudaErrorNotSupported;
    for (int s = 0; s < p.n_seg; ++s)
      if (p.seg[s].ld && p.seg[s].ld != p.seg[s].K) return cudaErrorNotSupported;
    if (p.rows <= 0 || p.M <= 0) continue;
    if (m == SIMT_MAX_PROBS || (m > 0 && p.dtype != L.p[0].dtype)) {
      cudaError_t e = flush();
      if (e != cudaSuccess) return e;
    }
    L.p[m++] = p;
    gx = imax64(gx, simt_row_tiles(p));
    gy = imax64(gy, cdiv(p.M, BN));
  }
  return flush();
}

}  // namespace moe
