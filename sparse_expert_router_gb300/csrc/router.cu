// Router top-k selection with an exactness guarantee, and the renormalised softmax gates.
//
// The router (teardown "Marin 535B-A23B: the half of a training run nobody usually shows
// you", sections "What is actually being trained" and "The one knob nobody pinned") picks the
// top_k experts of every token. Its section "What I'd take from it" reports that computing the
// router in more accurate arithmetic changed the top-8 of ~9% of tokens, so here the selection
// is defined on the exact real-valued logits of the stored inputs (ties to the lowest expert
// index) and computed in three stages:
//
//  1. fp32 logits from the router GEMM, each with a rigorous error bound
//       |l~ - l| <= c * gamma_d * ||x_t||_2 ||w_e||_2 + 2u |l~|,   gamma_d = d u / (1 - d u),
//     (Cauchy-Schwarz bounds sum_i |x_i w_ie|; c = 1 for the sequential FMA accumulation of the
//     CUDA-core GEMM, a safety factor c > 1 for the tensor-core accumulation). An expert is
//     surely selected when its lower bound exceeds the (k+1)-th largest upper bound, surely
//     not when its upper bound is below the k-th largest lower bound. A token whose k experts
//     are all sure is done.
//  2. Otherwise the undecided experts get a compensated dot product (Ogita, Rump and Oishi,
//     "Accurate sum and dot product", SIAM J. Sci. Comput. 26(6), 2005: error-free TwoSum
//     accumulation, plus error-free TwoProduct for fp32 inputs), whose error is at most
//     2u|res| + 2 gamma_n^2 sum|x_i w_ie|, and the token is re-classified.
//  3. Tokens still undecided get exact logits: every product of two bf16/fp32 numbers is an
//     integer times a power of two, accumulated exactly in 32-bit-limb integer bins.
// Gates are the softmax over the k selected fp32 logits (the full softmax renormalised over
// the selection); indices are written in ascending expert order.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "router.h"

namespace moe {
namespace {

constexpr int RT_WARPS = 8;
constexpr float U32 = 5.9604644775390625e-08f;  // 2^-24
constexpr int NB = 20;                           // exact accumulator: 20 x 32-bit limbs
constexpr int EXP_BIAS = 298;                    // -(smallest product exponent)

// ---- warp helpers ----------------------------------------------------------------------

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}

// k-th largest (k >= 1) element of vals[0..E) counted with multiplicity; -inf if k > E.
// work is E floats of per-warp scratch. Experts are owned by lane e % 32.
__device__ float warp_kth_largest(const float* vals, float* work, int E, int k, int lane) {
  for (int e = lane; e < E; e += 32) work[e] = vals[e];
  __syncwarp();
  float v = -INFINITY;
  for (int it = 0; it < k; ++it) {
    float best = -INFINITY;
    int bi = INT_MAX;
    for (int e = lane; e < E; e += 32) {
      float w = work[e];
      if (w > best) { best = w; bi = e; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float ob = __shfl_xor_sync(~0u, best, o);
      int oi = __shfl_xor_sync(~0u, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    v = best;
    if (bi != INT_MAX && (bi & 31) == lane) work[bi] = -INFINITY;
    __syncwarp();
  }
  return v;
}

// Classify every expert from its interval [lo, hi]: 1 = surely in the top-k, 0 = surely out,
// 2 = undecided. Returns the number of sure experts.
__device__ int warp_classify(const float* lo, const float* hi, float* work, uint8_t* sel, int E,
                             int k, int lane) {
  float Lk = warp_kth_largest(lo, work, E, k, lane);
  float Uk1 = (k < E) ? warp_kth_largest(hi, work, E, k + 1, lane) : -INFINITY;
  int n_in = 0;
  for (int e = lane; e < E; e += 32) {
    uint8_t s = 2;
    if (lo[e] > Uk1) { s = 1; ++n_in; }
    else if (hi[e] < Lk) s = 0;
    sel[e] = s;
  }
  __syncwarp();
  return warp_sum_i(n_in);
}

// Write the k experts with sel[e] == 1 in ascending order and their softmax gates.
__device__ void warp_write_selection(const float* lg, const uint8_t* sel, int E, int k, int lane,
                                     int32_t* idx_out, float* gate_out) {
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32)
    if (sel[e] == 1) m = fmaxf(m, lg[e]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(~0u, m, o));
  float s = 0.0f;
  for (int e = lane; e < E; e += 32)
    if (sel[e] == 1) s += expf(lg[e] - m);
  s = warp_sum_f(s);
  int base = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    int e = e0 + lane;
    bool on = (e < E) && sel[e] == 1;
    unsigned b = __ballot_sync(~0u, on);
    if (on) {
      int pos = base + __popc(b & ((1u << lane) - 1u));
      if (pos < k) {
        idx_out[pos] = e;
        gate_out[pos] = __fdiv_rn(expf(lg[e] - m), s);
      }
    }
    base += __popc(b);
  }
}

// Load a token's logits and stage-1 intervals into per-warp shared arrays.
// Loops over a token's experts take EU experts per lane per trip and issue all their global
// loads before any shared-memory store, so that a trip costs one memory latency, not EU.
constexpr int EU = 4;

__device__ void warp_stage1(const float* logits_t, const float* wnorm, float xn, float cgam,
                            int E, int lane, float* lg, float* lo, float* hi) {
  const float cx = __fmul_ru(cgam, xn);
  for (int e0 = lane; e0 < E; e0 += 32 * EU) {
    float l[EU], wn[EU];
#pragma unroll
    for (int u = 0; u < EU; ++u) {
      const int e = e0 + 32 * u;
      l[u] = e < E ? logits_t[e] : 0.0f;
      wn[u] = e < E ? wnorm[e] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < EU; ++u) {
      const int e = e0 + 32 * u;
      if (e < E) {
        float b = __fadd_ru(__fmul_ru(cx, wn[u]), __fmul_ru(2.0f * U32, fabsf(l[u])));
        b = __fadd_ru(b, 1e-30f);
        lg[e] = l[u];
        lo[e] = __fsub_rd(l[u], b);
        hi[e] = __fadd_ru(l[u], b);
      }
    }
  }
  __syncwarp();
}

// 8 elements as loaded (16 B of bf16 or 32 B of fp32), converted to fp32 on use.
template <typename T>
struct Raw8;
template <>
struct Raw8<bf16> {
  uint4 u;
  __device__ __forceinline__ void load(const bf16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ bf16 raw(int q) const {   // element q
    const uint32_t wd = q < 2 ? u.x : q < 4 ? u.y : q < 6 ? u.z : u.w;
    return __ushort_as_bfloat16((unsigned short)((q & 1) ? (wd >> 16) : (wd & 0xFFFFu)));
  }
  __device__ __forceinline__ void get(float v[8]) const {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ float raw(int q) const {   // element q
    const float4& h = q < 4 ? a : b;
    const int r = q & 3;
    return r == 0 ? h.x : r == 1 ? h.y : r == 2 ? h.z : h.w;
  }
  __device__ __forceinline__ void get(float v[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// Upper bound of ||x||_2 for a row of d elements (d a multiple of 8).
// Each lane issues the loads of XU groups of 8 elements (128 bytes) before it adds any of them
// (the sum keeps its order).
template <typename T>
__device__ float warp_norm_ub(const T* x, int d, float gam_d, int lane) {
  constexpr int XU = sizeof(T) == 4 ? 4 : 8;
  float s = 0.0f;
  for (int i0 = lane * 8; i0 < d; i0 += 256 * XU) {
    Raw8<T> r[XU];
#pragma unroll
    for (int u = 0; u < XU; ++u)
      if (i0 + 256 * u < d) r[u].load(x + i0 + 256 * u);
#pragma unroll
    for (int u = 0; u < XU; ++u) {
      if (i0 + 256 * u >= d) break;
      float v[8];
      r[u].get(v);
#pragma unroll
      for (int j = 0; j < 8; ++j) s = fmaf(v[j], v[j], s);
    }
  }
  s = warp_sum_f(s);
  // s~ >= (1 - gamma_d) s, so s <= s~ (1 + 2 gamma_d) for gamma_d <= 1/2
  return __fmul_ru(__fsqrt_ru(__fmul_ru(s, 1.0f + 2.0f * gam_d)), 1.0f + 4.0f * U32);
}

// ---- stage 2: compensated dot product ---------------------------------------------------

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

constexpr int MC = 4;   // candidates evaluated together (their loads overlap)

// x . w_j + bias_j for up to MC candidate rows w_j of W_r^T, each with a bound on its error;
// lane 0 returns the values. Error-free TwoSum accumulation (plus TwoProduct for fp32) per
// lane, the lanes' (sum, compensation) pairs combined with TwoSum.
template <typename T, int NMC = MC>
__device__ void warp_dot2_multi(const T* x, const T* wrT, const int* cand, int nc, int d,
                                const float* bias, float g2, int lane, float* res, float* eb) {
  constexpr int MC = NMC;
  const bool f32 = sizeof(T) == 4;
  float s[MC], c[MC], sa[MC];
  const T* wp[MC];
#pragma unroll
  for (int j = 0; j < MC; ++j) {
    const int e = cand[j < nc ? j : nc - 1];
    const float b = (bias && lane == 0 && j < nc) ? bias[e] : 0.0f;
    s[j] = b;
    c[j] = 0.0f;
    sa[j] = fabsf(b);
    wp[j] = wrT + (int64_t)e * d;
  }
  // U consecutive 256-element steps per trip: all their loads are issued before any of their
  // products, so U * (MC + 1) loads per lane are in flight (the sums keep their order)
  constexpr int U = f32 ? 2 : 4;
  for (int i0 = lane * 8; i0 < d; i0 += 256 * U) {
    Raw8<T> xr[U], wr[U][MC];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + 256 * u;
      if (i < d) {
        xr[u].load(x + i);
#pragma unroll
        for (int j = 0; j < MC; ++j) wr[u][j].load(wp[j] + i);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + 256 * u >= d) break;
      float xv[8];
      xr[u].get(xv);
#pragma unroll
      for (int j = 0; j < MC; ++j) {
        float wv[8];
        wr[u][j].get(wv);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float p = __fmul_rn(xv[q], wv[q]);
          float ep = f32 ? fmaf(xv[q], wv[q], -p) : 0.0f;   // TwoProduct (exact when bf16)
          float t, e;
          two_sum(s[j], p, t, e);
          s[j] = t;
          c[j] = __fadd_rn(c[j], __fadd_rn(e, ep));
          sa[j] = __fadd_rn(sa[j], fabsf(p));
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < MC; ++j) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float s2 = __shfl_xor_sync(~0u, s[j], o);
      float c2 = __shfl_xor_sync(~0u, c[j], o);
      float a2 = __shfl_xor_sync(~0u, sa[j], o);
      float t, e;
      two_sum(s[j], s2, t, e);
      s[j] = t;
      c[j] = __fadd_rn(__fadd_rn(c[j], c2), e);
      sa[j] = __fadd_rn(sa[j], a2);
    }
    const float r = __fadd_rn(s[j], c[j]);
    // sum|p| is computed with relative error <= gamma_n: inflate it, then apply the bound
    const float sa_ub = __fmul_ru(sa[j], 1.0f + sqrtf(g2) * 2.0f);
    float b = __fadd_ru(__fmul_ru(2.0f * U32, fabsf(r)), __fmul_ru(2.0f * g2, sa_ub));
    if (j < nc) { res[j] = r; eb[j] = __fadd_ru(b, 1e-30f); }
  }
}

// ---- stage 3: exact logits --------------------------------------------------------------

template <typename T>
__device__ __forceinline__ bool decompose(T v, uint32_t& M, int& q, uint32_t& sign);

template <>
__device__ __forceinline__ bool decompose<float>(float v, uint32_t& M, int& q, uint32_t& sign) {
  uint32_t b = __float_as_uint(v);
  sign = b >> 31;
  uint32_t e = (b >> 23) & 0xFF, m = b & 0x7FFFFF;
  if (e == 0xFF) return false;
  if (e == 0) { M = m; q = -149; } else { M = m | 0x800000u; q = (int)e - 150; }
  return true;
}
template <>
__device__ __forceinline__ bool decompose<bf16>(bf16 v, uint32_t& M, int& q, uint32_t& sign) {
  uint32_t b = (uint32_t)__bfloat16_as_ushort(v);
  sign = b >> 15;
  uint32_t e = (b >> 7) & 0xFF, m = b & 0x7F;
  if (e == 0xFF) return false;
  if (e == 0) { M = m; q = -133; } else { M = m | 0x80u; q = (int)e - 134; }
  return true;
}

// a[u] for a runtime u < N without dynamic indexing (the array stays in registers)
template <typename R, int N>
__device__ __forceinline__ R pick(const R (&a)[N], int u) {
  R r = a[0];
#pragma unroll
  for (int i = 1; i < N; ++i)
    if (u == i) r = a[i];
  return r;
}

// Block-wide exact x . w + bias (blockDim = RT_WARPS * 32) into canonical form `out`. Every
// thread accumulates its products in 20 register limbs (updated with predicated adds, so the
// limbs stay in registers); warps add their limbs with shuffles, warp 0 adds the warps' limbs
// (from `red`, RT_WARPS * NB int64 of shared memory), one limb per lane, and lane 0 propagates
// the carries. Requires d % 8 == 0 and 16-byte aligned rows.
template <typename T>
__device__ bool block_exact(const T* x, const T* w, int d, float bias,
                            long long* red, unsigned long long* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long bins[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) bins[i] = 0;
  bool ok = true;
  auto add = [&](uint64_t M, int q, uint32_t neg) {
    if (M == 0) return;
    const int p = q + EXP_BIAS;
    const int bi = p >> 5, sh = p & 31;
    const uint64_t lo = (M & 0xFFFFFFFFull) << sh;
    const uint64_t hi = (M >> 32) << sh;
    long long c0 = (long long)(lo & 0xFFFFFFFFull);
    long long c1 = (long long)((lo >> 32) + (hi & 0xFFFFFFFFull));
    long long c2 = (long long)(hi >> 32);
    if (neg) { c0 = -c0; c1 = -c1; c2 = -c2; }
#pragma unroll
    for (int i = 0; i < NB; ++i)
      bins[i] += (i == bi) ? c0 : (i == bi + 1) ? c1 : (i == bi + 2) ? c2 : 0ll;
  };
  // XB groups of 8 elements per thread per trip, all their loads issued before any product;
  // the limb sums are exact, so how elements are assigned to threads does not change them
  constexpr int XB = 4;
  const int nv = d >> 3;
  for (int v0 = tid; v0 < nv; v0 += RT_WARPS * 32 * XB) {
    Raw8<T> xr[XB], wr[XB];
#pragma unroll
    for (int u = 0; u < XB; ++u) {
      const int v = v0 + RT_WARPS * 32 * u;
      if (v < nv) {
        xr[u].load(x + 8 * v);
        wr[u].load(w + 8 * v);
      }
    }
    // one compact loop over the loaded elements: the kernel runs once per step, from a cold
    // instruction cache, so its code size matters more than its instruction count
    const int nu = min(XB, (nv - v0 + RT_WARPS * 32 - 1) / (RT_WARPS * 32));
#pragma unroll 1
    for (int uq = 0; uq < nu * 8; ++uq) {
      const int u = uq >> 3, q = uq & 7;
      uint32_t Mx = 0, Mw = 0, sx = 0, sw = 0;
      int qx = 0, qw = 0;
      const bool fx = decompose<T>(pick(xr, u).raw(q), Mx, qx, sx);
      const bool fw = decompose<T>(pick(wr, u).raw(q), Mw, qw, sw);
      ok &= fx && fw;
      if (fx && fw) add((uint64_t)Mx * (uint64_t)Mw, qx + qw, sx ^ sw);
    }
  }
  if (tid == 0) {
    uint32_t Mb = 0, sb = 0;
    int qb = 0;
    bool fb = decompose<float>(bias, Mb, qb, sb);   // the bias is Mb 2^qb, qb >= -149
    ok &= fb;
    if (fb) add((uint64_t)Mb, qb, sb);
  }
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    long long v = bins[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    if (lane == 0) red[warp * NB + i] = v;
  }
  ok = __syncthreads_and(ok);
  // lane i of warp 0 adds limb i over the warps, then lane 0 propagates the carries
  if (warp == 0) {
    long long v = 0;
    if (lane < NB) {
#pragma unroll
      for (int wv = 0; wv < RT_WARPS; ++wv) v += red[wv * NB + lane];
    }
    __syncwarp();
    if (lane < NB) red[lane] = v;
    __syncwarp();
    if (lane == 0) {
      long long carry = 0;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const long long t = carry + red[i];
        if (i < NB - 1) {
          out[i] = (unsigned long long)(t & 0xFFFFFFFFll);
          carry = t >> 32;   // arithmetic shift: floor division
        } else {
          out[i] = (unsigned long long)t;
        }
      }
    }
  }
  __syncthreads();
  return ok;
}

// -1, 0, +1 as a < b, a == b, a > b for canonical exact values.
__device__ int exact_cmp(const unsigned long long* a, const unsigned long long* b) {
  int64_t ta = (int64_t)a[NB - 1], tb = (int64_t)b[NB - 1];
  if (ta != tb) return ta < tb ? -1 : 1;
  for (int i = NB - 2; i >= 0; --i)
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  return 0;
}

// ---- kernels ----------------------------------------------------------------------------

template <typename T>
__global__ void wr_transpose_kernel(const T* __restrict__ w, T* __restrict__ wt, int d, int E) {
  pdl_wait();
  __shared__ T tile[32][33];
  int i0 = blockIdx.y * 32, e0 = blockIdx.x * 32;
  for (int r = threadIdx.y; r < 32; r += 8) {
    int i = i0 + r, e = e0 + threadIdx.x;
    if (i < d && e < E) tile[r][threadIdx.x] = w[(int64_t)i * E + e];
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    int e = e0 + r, i = i0 + threadIdx.x;
    if (i < d && e < E) wt[(int64_t)e * d + i] = tile[threadIdx.x][r];
  }
}

template <typename T>
__global__ void wr_norm_kernel(const T* __restrict__ wt, float* __restrict__ wnorm, int d, int E,
                               float gam_d) {
  pdl_wait();
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= E) return;
  float n = warp_norm_ub(wt + (int64_t)warp * d, d, gam_d, lane);
  if (lane == 0) wnorm[warp] = n;
}

struct WarpArrays {
  float *lg, *lo, *hi, *work;
  uint8_t *sel, *refined;
};
__device__ __forceinline__ WarpArrays warp_arrays(unsigned char* base, int E, int warp) {
  size_t per = (size_t)E * 18;
  per = (per + 15) & ~(size_t)15;
  unsigned char* p = base + per * warp;
  WarpArrays a;
  a.lg = reinterpret_cast<float*>(p);
  a.lo = a.lg + E;
  a.hi = a.lo + E;
  a.work = a.hi + E;
  a.sel = reinterpret_cast<uint8_t*>(a.work + E);
  a.refined = a.sel + E;
  return a;
}

// Stage 1 for every token. Every expert's logit gets the same, token-wide error bound beta
// (the largest of the per-expert bounds), so one extraction of the k+1 largest fp32 logits
// decides. Tokens with an undecided expert go to the refine list.
template <typename T>
__global__ void __launch_bounds__(RT_WARPS * 32, 5)
router_select_kernel(RouterArgs a) {
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * RT_WARPS + warp;
  if (t >= a.T) return;
  float* work = reinterpret_cast<float*>(smem) + (size_t)warp * a.E;   // this warp's logits
  const T* x = static_cast<const T*>(a.x) + t * a.d;
  const float xn = warp_norm_ub(x, a.d, a.gam_d, lane);
  if (lane == 0) a.xnorm[t] = xn;
  const float* lt = a.logits + t * a.E;
  float wmax = 0.0f, amax = 0.0f;
  for (int e0 = lane; e0 < a.E; e0 += 32 * EU) {
    float l[EU], wn[EU];
#pragma unroll
    for (int u = 0; u < EU; ++u) {
      const int e = e0 + 32 * u;
      l[u] = e < a.E ? lt[e] : 0.0f;
      wn[u] = e < a.E ? a.wnorm[e] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < EU; ++u) {
      const int e = e0 + 32 * u;
      if (e < a.E) {
        work[e] = l[u];
        wmax = fmaxf(wmax, wn[u]);
        amax = fmaxf(amax, fabsf(l[u]));
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    wmax = fmaxf(wmax, __shfl_xor_sync(~0u, wmax, o));
    amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
  }
  float beta = __fadd_ru(__fmul_ru(__fmul_ru(a.cgam, xn), wmax), __fmul_ru(2.0f * U32, amax));
  beta = __fadd_ru(beta, 1e-30f);
  __syncwarp();
  // the k+1 largest fp32 logits (with multiplicity, ties to the lower index), lane j keeping
  // the j-th of them
  float lk = -INFINITY, lk1 = -INFINITY, my_v = -INFINITY;
  int my_i = INT_MAX;
  const int kk = min(a.k + 1, a.E);
  for (int it = 0; it < kk; ++it) {
    float best = -INFINITY;
    int bi = INT_MAX;
    for (int e = lane; e < a.E; e += 32) {
      const float v = work[e];
      if (v > best) { best = v; bi = e; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(~0u, best, o);
      const int oi = __shfl_xor_sync(~0u, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    if (lane == it && it < a.k) { my_v = best; my_i = bi; }
    if (it == a.k - 1) lk = best;
    if (it == a.k) lk1 = best;
    if (bi != INT_MAX && (bi & 31) == lane) work[bi] = -INFINITY;
    __syncwarp();
  }
  // An expert is surely in when l_e - beta > l_(k+1) + beta and surely out when
  // l_e + beta < l_(k) - beta. Every expert above l_(k+1) is one of the k largest, so the
  // token is decided exactly when the k-th largest is surely in; its top-k is then the k
  // logits found above.
  const float in_thr = __fadd_ru(__fadd_ru(lk1, beta), beta);
  if (lk > in_thr) {
    const float m = __shfl_sync(~0u, my_v, 0);            // the largest logit
    const float ex = lane < a.k ? expf(my_v - m) : 0.0f;
    const float sum = warp_sum_f(ex);
    int pos = 0;                                          // rank by expert index
    for (int j = 0; j < a.k; ++j) pos += (__shfl_sync(~0u, my_i, j) < my_i) ? 1 : 0;
    if (lane < a.k) {
      a.idx[t * a.k + pos] = my_i;
      a.gate[t * a.k + pos] = __fdiv_rn(ex, sum);
    }
  } else if (lane == 0) {
    int pos = atomicAdd(&a.hdr->n_refine, 1);
    a.refine_list[pos] = (int32_t)t;
  }
}

// Stage-3 work of the tokens whose classification the refine stage saved (the first n_saved of
// the exact list) is spread over EXACT_PARTS blocks per token: each takes every EXACT_PARTS-th
// undecided expert and publishes its exact value; the last block to arrive ranks them all.
constexpr int EXACT_PARTS = 8;

// The saved state of exact-list slot `it` inside RouterArgs::saved: the refine stage's final
// classification of the token, and the exact values the exact stage's blocks publish.
struct SavedSlot {
  uint8_t* sel;                // [E]: 1 surely in, 0 surely out, 2 undecided after stage 2
  int32_t* n_in;               // experts surely in
  unsigned long long* forms;   // [E, NB]: exact values of the undecided experts
  int32_t* arrived;            // blocks of this token done with their experts
};
__host__ __device__ __forceinline__ size_t al256z(size_t b) { return (b + 255) & ~(size_t)255; }
__device__ __forceinline__ SavedSlot saved_slot(const RouterArgs& a, int it) {
  unsigned char* base = static_cast<unsigned char*>(a.saved);
  const size_t ns = al256z((size_t)a.n_saved * a.E);
  const size_t nn = al256z((size_t)a.n_saved * 4);
  const size_t nf = al256z((size_t)a.n_saved * a.E * NB * 8);
  SavedSlot v;
  v.sel = base + (size_t)it * a.E;
  v.n_in = reinterpret_cast<int32_t*>(base + ns) + it;
  v.forms = reinterpret_cast<unsigned long long*>(base + ns + nn) + (size_t)it * a.E * NB;
  v.arrived = reinterpret_cast<int32_t*>(base + ns + nn + nf) + it;
  return v;
}

template <typename T>
__global__ void __launch_bounds__(RT_WARPS * 32)
router_refine_kernel(RouterArgs a) {
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpArrays w = warp_arrays(smem, a.E, warp);
  const int n = min(a.hdr->n_refine, (int)a.T);
  // consecutive list entries go to consecutive blocks (one per SM), so that a short list still
  // spreads over every SM
  for (int it = warp * gridDim.x + blockIdx.x; it < n; it += gridDim.x * RT_WARPS) {
    const int64_t t = a.refine_list[it];
    const T* x = static_cast<const T*>(a.x) + t * a.d;
    warp_stage1(a.logits + t * a.E, a.wnorm, a.xnorm[t], a.cgam, a.E, lane, w.lg, w.lo, w.hi);
    int n_in = warp_classify(w.lo, w.hi, w.work, w.sel, a.E, a.k, lane);
    // Refine undecided experts MC at a time (highest fp32 logit first among those left) and
    // re-classify after every batch; stop once the top-k is decided or nothing is left.
    for (int e = lane; e < a.E; e += 32) w.refined[e] = 0;
    __syncwarp();
    while (n_in < a.k) {
      int cand[MC];
      int nc = 0;
      for (int j = 0; j < MC; ++j) {
        float best = -INFINITY;
        int bi = INT_MAX;
        for (int e = lane; e < a.E; e += 32)
          if (w.sel[e] == 2 && !w.refined[e] && (w.lg[e] > best || (w.lg[e] == best && e < bi))) {
            best = w.lg[e];
            bi = e;
          }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          float ob = __shfl_xor_sync(~0u, best, o);
          int oi = __shfl_xor_sync(~0u, bi, o);
          if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
        }
        if (bi == INT_MAX) break;
        cand[nc++] = bi;
        if ((bi & 31) == lane) w.refined[bi] = 1;
        __syncwarp();
      }
      if (nc == 0) break;
      float res[MC], eb[MC];
      warp_dot2_multi(x, static_cast<const T*>(a.wrT), cand, nc, a.d, a.bias, a.g2, lane, res,
                      eb);
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < MC; ++j) {
          if (j < nc) {
            const int ee = cand[j];
            w.lo[ee] = fmaxf(w.lo[ee], __fsub_rd(res[j], eb[j]));
            w.hi[ee] = fminf(w.hi[ee], __fadd_ru(res[j], eb[j]));
          }
        }
      }
      __syncwarp();
      n_in = warp_classify(w.lo, w.hi, w.work, w.sel, a.E, a.k, lane);
    }
    if (n_in == a.k) {
      warp_write_selection(w.lg, w.sel, a.E, a.k, lane, a.idx + t * a.k, a.gate + t * a.k);
    } else {
      int pos = 0;
      if (lane == 0) {
        pos = atomicAdd(&a.hdr->n_exact, 1);
        a.exact_list[pos] = (int32_t)t;
      }
      pos = __shfl_sync(~0u, pos, 0);
      // its classification goes with it, so that the exact stage starts from it
      if (a.saved && pos < a.n_saved) {
        const SavedSlot sv = saved_slot(a, pos);
        for (int e = lane; e < a.E; e += 32) sv.sel[e] = w.sel[e];
        if (lane == 0) {
          *sv.n_in = n_in;
          *sv.arrived = 0;
        }
      }
    }
  }
}

// Tokens still undecided after stage 2. Warp 0 builds the candidate list: from the
// classification the refine stage saved for the token (EXACT_PARTS blocks per token, see
// above) or, past the saved slots, from stage 1 and the compensated dot product of every
// stage-1 candidate on the block's 8 warps (one block per token). Only experts still
// undecided then get exact logits, each computed by a whole block; the remaining top-k slots
// go to the largest exact values, ties to the lower index.
template <typename T>
__global__ void __launch_bounds__(RT_WARPS * 32)
router_exact_kernel(RouterArgs a) {
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpArrays w = warp_arrays(smem, a.E, 0);
  size_t per = ((size_t)a.E * 18 + 15) & ~(size_t)15;
  unsigned long long* forms = reinterpret_cast<unsigned long long*>(smem + per);   // [E][NB]
  long long* red = reinterpret_cast<long long*>(forms + (size_t)a.E * NB);      // [RT_WARPS][NB]
  int32_t* cand = reinterpret_cast<int32_t*>(red + RT_WARPS * NB);             // [E]
  float* cres = reinterpret_cast<float*>(cand + a.E);                           // [E]
  float* ceb = cres + a.E;                                                      // [E]
  __shared__ int s_ncand, s_nin, s_ok, s_last;
  const int n = min(a.hdr->n_exact, (int)a.T);
  const int ns = a.saved ? min(n, a.n_saved) : 0;
  const int n_items = ns * EXACT_PARTS + (n - ns);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const bool split = item < ns * EXACT_PARTS;
    const int it = split ? item / EXACT_PARTS : ns + (item - ns * EXACT_PARTS);
    const int part = split ? item % EXACT_PARTS : 0;
    const int64_t t = a.exact_list[it];
    const T* x = static_cast<const T*>(a.x) + t * a.d;
    SavedSlot sv{};
    if (split) sv = saved_slot(a, it);
    if (warp == 0) {
      int n_in0;
      if (split) {
        // the refine stage's classification of the token
        for (int e0 = lane; e0 < a.E; e0 += 32 * EU) {
          uint8_t c[EU];
#pragma unroll
          for (int u = 0; u < EU; ++u) c[u] = (e0 + 32 * u < a.E) ? sv.sel[e0 + 32 * u] : 0;
#pragma unroll
          for (int u = 0; u < EU; ++u)
            if (e0 + 32 * u < a.E) w.sel[e0 + 32 * u] = c[u];
        }
        n_in0 = *sv.n_in;
        __syncwarp();
      } else {
        warp_stage1(a.logits + t * a.E, a.wnorm, a.xnorm[t], a.cgam, a.E, lane, w.lg, w.lo, w.hi);
        n_in0 = warp_classify(w.lo, w.hi, w.work, w.sel, a.E, a.k, lane);
      }
      int base = 0;
      for (int e0 = 0; e0 < a.E; e0 += 32) {
        int e = e0 + lane;
        bool on = e < a.E && w.sel[e] == 2;
        unsigned b = __ballot_sync(~0u, on);
        if (on) cand[base + __popc(b & ((1u << lane) - 1u))] = e;
        base += __popc(b);
      }
      if (lane == 0) { s_ncand = base; s_ok = 1; s_nin = n_in0; }
    }
    __syncthreads();
    if (!split) {
      // stage 2 for every candidate, one warp per candidate
      const int nc = s_ncand;
      for (int ci = warp; ci < nc; ci += RT_WARPS) {
        float res[1], eb[1];
        warp_dot2_multi<T, 1>(x, static_cast<const T*>(a.wrT), cand + ci, 1, a.d, a.bias, a.g2,
                              lane, res, eb);
        if (lane == 0) { cres[ci] = res[0]; ceb[ci] = eb[0]; }
      }
      __syncthreads();
      if (warp == 0) {
        for (int ci = lane; ci < nc; ci += 32) {
          const int e = cand[ci];
          w.lo[e] = fmaxf(w.lo[e], __fsub_rd(cres[ci], ceb[ci]));
          w.hi[e] = fminf(w.hi[e], __fadd_ru(cres[ci], ceb[ci]));
        }
        __syncwarp();
        int n_in = warp_classify(w.lo, w.hi, w.work, w.sel, a.E, a.k, lane);
        int base = 0;
        for (int e0 = 0; e0 < a.E; e0 += 32) {
          int e = e0 + lane;
          bool on = e < a.E && w.sel[e] == 2;
          unsigned b = __ballot_sync(~0u, on);
          if (on) cand[base + __popc(b & ((1u << lane) - 1u))] = e;
          base += __popc(b);
        }
        if (lane == 0) { s_ncand = base; s_nin = n_in; }
      }
      __syncthreads();
    }
    // stage 3: exact values of the experts still undecided, one block-wide sum each
    const int nc2 = s_ncand;
    const int step = split ? EXACT_PARTS : 1;
    for (int ci = part; ci < nc2; ci += step) {
      const int e = cand[ci];
      bool ok = block_exact(x, static_cast<const T*>(a.wrT) + (int64_t)e * a.d, a.d,
                            a.bias ? a.bias[e] : 0.0f, red, forms + (size_t)ci * NB);
      if (!ok && threadIdx.x == 0) s_ok = 0;
      if (split && threadIdx.x < NB)
        sv.forms[(size_t)e * NB + threadIdx.x] = forms[(size_t)ci * NB + threadIdx.x];
    }
    if (split) {
      // publish this block's values; the last of the token's blocks reads everyone's and ranks
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) s_last = (atomicAdd(sv.arrived, 1) == EXACT_PARTS - 1);
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int q = threadIdx.x; q < nc2 * NB; q += blockDim.x) {
          const int ci = q / NB, i = q - ci * NB;
          forms[q] = __ldcg(sv.forms + (size_t)cand[ci] * NB + i);
        }
      }
      __syncthreads();
    }
    if (warp == 0) {
      if (!s_ok && lane == 0) report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t);
      if (!split || s_last) {
        if (split) {
          const float* lt = a.logits + t * a.E;
          for (int e = lane; e < a.E; e += 32) w.lg[e] = lt[e];
          __syncwarp();
        }
        const int need = a.k - s_nin;
        // rank each candidate among the candidates: larger exact value first, then lower index
        for (int ci = lane; ci < nc2; ci += 32) {
          int r = 0;
          for (int cj = 0; cj < nc2; ++cj) {
            if (cj == ci) continue;
            int c = exact_cmp(forms + (size_t)cj * NB, forms + (size_t)ci * NB);
            if (c > 0 || (c == 0 && cand[cj] < cand[ci])) ++r;
          }
          w.sel[cand[ci]] = (r < need) ? 1 : 0;
        }
        __syncwarp();
        warp_write_selection(w.lg, w.sel, a.E, a.k, lane, a.idx + t * a.k, a.gate + t * a.k);
      }
    }
    __syncthreads();
  }
}

size_t warp_smem(int E) { return ((size_t)E * 18 + 15) & ~(size_t)15; }

}  // namespace

size_t router_saved_bytes(int E, int n_saved) {
  // the layout of saved_slot: classifications, sure-in counts, exact values and arrival
  // counters, the first three rounded up to 256 B
  return al256z((size_t)n_saved * E) + al256z((size_t)n_saved * 4) +
         al256z((size_t)n_saved * E * NB * 8) + (size_t)n_saved * 4;
}

cudaError_t router_prepare(const RouterArgs& a, int dtype, cudaStream_t st, bool pdl) {
  dim3 tg(cdiv(a.E, 32), cdiv(a.d, 32)), tb(32, 8);
  cudaError_t err;
  if (dtype == DT_BF16)
    err = launch(wr_transpose_kernel<bf16>, tg, tb, 0, st, pdl, (const bf16*)a.w_router,
                 (bf16*)a.wrT, a.d, a.E);
  else
    err = launch(wr_transpose_kernel<float>, tg, tb, 0, st, pdl, (const float*)a.w_router,
                 (float*)a.wrT, a.d, a.E);
  if (err != cudaSuccess) return err;
  dim3 ng(cdiv((int64_t)a.E * 32, 256));
  if (dtype == DT_BF16)
    return launch(wr_norm_kernel<bf16>, ng, dim3(256), 0, st, pdl, (const bf16*)a.wrT,
                  a.wnorm, a.d, a.E, a.gam_d);
  return launch(wr_norm_kernel<float>, ng, dim3(256), 0, st, pdl, (const float*)a.wrT, a.wnorm,
                a.d, a.E, a.gam_d);
}

cudaError_t router_select(const RouterArgs& a, int dtype, int num_sms, cudaStream_t st, bool pdl) {
  const size_t sm_sel = (size_t)a.E * 4 * RT_WARPS;
  const size_t sm_ref = warp_smem(a.E) * RT_WARPS;
  size_t sm_exact = warp_smem(a.E) + (size_t)a.E * NB * 8 + (size_t)RT_WARPS * NB * 8 +
                    (size_t)a.E * 12;
  cudaError_t err;
  auto sel = (dtype == DT_BF16) ? router_select_kernel<bf16> : router_select_kernel<float>;
  auto ref = (dtype == DT_BF16) ? router_refine_kernel<bf16> : router_refine_kernel<float>;
  auto ex = (dtype == DT_BF16) ? router_exact_kernel<bf16> : router_exact_kernel<float>;
  cudaFuncSetAttribute(sel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_sel);
  cudaFuncSetAttribute(ref, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_ref);
  cudaFuncSetAttribute(ex, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_exact);
  err = launch(sel, dim3((unsigned)cdiv(a.T, RT_WARPS)), dim3(RT_WARPS * 32), sm_sel, st, pdl, a);
  if (err != cudaSuccess) return err;
  err = launch(ref, dim3(num_sms), dim3(RT_WARPS * 32), sm_ref, st, pdl, a);
  if (err != cudaSuccess) return err;
  return launch(ex, dim3(num_sms), dim3(RT_WARPS * 32), sm_exact, st, pdl, a);
}

}  // namespace moe
