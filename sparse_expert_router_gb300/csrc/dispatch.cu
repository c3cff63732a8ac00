// Dispatch and combine: expert histogram, capacity clamp and exclusive scan (group offsets),
// stable token permutation, RMSNorm-and-scatter of the latent rows, and the gate-weighted
// ordered gather that combines expert outputs.
//
// The layer sends each token, projected down and normalised, to its experts and combines
// their outputs with the gates ("Marin 535B-A23B: the half of a training run nobody usually
// shows you", section "What is actually being trained"). Rows reach the expert GEMMs grouped
// by expert, in token order within an expert (section "21% to 27% MFU without stopping the
// run"); assignments past an expert's capacity are dropped and the token skips that expert
// ("Marin Begins Open Training of a 535B-Parameter MoE Model", section 2). The combine is an
// ordered gather rather than an atomic scatter-add, so repeated runs are bitwise identical
// (weekly summary of 2026-09-14, post-training epic, #9144).
#include "common.cuh"
#include <type_traits>

#include "dispatch.h"

namespace moe {
namespace {

constexpr int CH = 128;   // tokens per dispatch chunk (one thread per token)

__global__ void header_reset_kernel(DeviceHeader* h, int clear_status, int amax_mask) {
  pdl_wait();
  if (threadIdx.x == 0) {
    if (clear_status) { h->status = 0; h->detail = 0; }
    h->n_refine = 0;
    h->n_exact = 0;
    if (amax_mask & 1) h->amax_x = 0;
    if (amax_mask & 2) h->amax_h = 0;
  }
}

// An assignment (t, j) is valid when its expert id is in range and the token's ids ascend.
__device__ __forceinline__ bool valid_assignment(const int32_t* row, int j, int E) {
  int e = row[j];
  return e >= 0 && e < E && (j == 0 || row[j - 1] < e);
}

__global__ void __launch_bounds__(CH) hist_kernel(DispatchArgs a) {
  pdl_wait();
  extern __shared__ int s_cnt[];
  for (int e = threadIdx.x; e < a.E; e += CH) s_cnt[e] = 0;
  __syncthreads();
  int64_t t = (int64_t)blockIdx.x * CH + threadIdx.x;
  if (t < a.T && (!a.mask || a.mask[t])) {   // padding tokens are not dispatched
    const int32_t* row = a.idx + t * a.k;
    for (int j = 0; j < a.k; ++j) {
      if (valid_assignment(row, j, a.E)) atomicAdd(&s_cnt[row[j]], 1);
      else report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += CH)
    a.chunk_hist[(int64_t)blockIdx.x * a.E + e] = s_cnt[e];
}

// One block per expert: exclusive scan of the expert's per-chunk counts (the base of each
// chunk's ranks) and the expert's total count.
__global__ void __launch_bounds__(256) scan_chunks_kernel(DispatchArgs a) {
  pdl_wait();
  __shared__ int s_warp[8];
  __shared__ int s_carry;
  const int e = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int64_t c0 = 0; c0 < a.n_chunks; c0 += 256) {
    const int64_t c = c0 + threadIdx.x;
    const int v = (c < a.n_chunks) ? a.chunk_hist[c * a.E + e] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(~0u, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = (lane < 8) ? s_warp[lane] : 0;
      int iw = w;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        int u = __shfl_up_sync(~0u, iw, o);
        if (lane >= o) iw += u;
      }
      if (lane < 8) s_warp[lane] = iw - w;   // exclusive prefix of warp totals
    }
    __syncthreads();
    const int carry = s_carry;
    const int excl = carry + s_warp[warp] + incl - v;
    if (c < a.n_chunks) a.chunk_base[c * a.E + e] = excl;
    __syncthreads();
    if (threadIdx.x == 255) s_carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) a.counts[e] = s_carry;
}

// One block: capacity clamp, exclusive scan of the kept counts into the group offsets, drops.
__global__ void __launch_bounds__(1024) scan_offsets_kernel(DispatchArgs a) {
  pdl_wait();
  __shared__ int s_warp[32];
  __shared__ int s_drop[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int cnt = (e < a.E) ? a.counts[e] : 0;
  int kept = (a.cap >= 0) ? min(cnt, a.cap) : cnt;
  int drop = cnt - kept;
  int incl = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += v;
  }
  int wdrop = drop;
#pragma unroll
  for (int o = 16; o; o >>= 1) wdrop += __shfl_xor_sync(~0u, wdrop, o);
  if (lane == 31) s_warp[warp] = incl;
  if (lane == 0) s_drop[warp] = wdrop;
  __syncthreads();
  if (warp == 0) {
    int v = s_warp[lane], dv = s_drop[lane];
    int iv = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(~0u, iv, o);
      if (lane >= o) iv += u;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) dv += __shfl_xor_sync(~0u, dv, o);
    s_warp[lane] = iv - v;   // exclusive prefix of warp totals
    if (lane == 0) s_drop[0] = dv;
  }
  __syncthreads();
  int excl = s_warp[warp] + incl - kept;
  if (e < a.E) a.offsets[e] = excl;
  if (e == a.E - 1) a.offsets[a.E] = excl + kept;
  if (e == 0 && a.n_dropped) *a.n_dropped = s_drop[0];
}

// Slots: stable rank of each token among the tokens of its chunk that chose the same expert
// (bitmask per expert and popcount), plus the chunk's base.
__global__ void __launch_bounds__(CH) rank_kernel(DispatchArgs a) {
  pdl_wait();
  extern __shared__ uint32_t s_mask[];   // [E][CH / 32]
  constexpr int W = CH / 32;
  for (int i = threadIdx.x; i < a.E * W; i += CH) s_mask[i] = 0u;
  __syncthreads();
  const int tl = threadIdx.x;
  const int64_t t = (int64_t)blockIdx.x * CH + tl;
  const int32_t* row = a.idx + t * a.k;
  const bool real = t < a.T && (!a.mask || a.mask[t]);
  if (real)
    for (int j = 0; j < a.k; ++j)
      if (valid_assignment(row, j, a.E)) atomicOr(&s_mask[row[j] * W + (tl >> 5)], 1u << (tl & 31));
  __syncthreads();
  if (t >= a.T) return;
  for (int j = 0; j < a.k; ++j) {
    int32_t slot = -1;
    if (real && valid_assignment(row, j, a.E)) {
      const int e = row[j];
      int r = __popc(s_mask[e * W + (tl >> 5)] & ((1u << (tl & 31)) - 1u));
      for (int w = 0; w < (tl >> 5); ++w) r += __popc(s_mask[e * W + w]);
      r += a.chunk_base[(int64_t)blockIdx.x * a.E + e];
      if (a.cap < 0 || r < a.cap) {
        slot = a.offsets[e] + r;
        if (slot >= a.pool_rows) { report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t); slot = -1; }
        else a.perm[slot] = (int32_t)(t * a.k + j);
      }
    }
    a.slot_of[t * a.k + j] = slot;
  }
}

// h = z * rsqrt(mean(z^2) + eps) * gamma written to every kept slot of the token. With E4M3
// output the rows hold the codes of h * x_scale (round to nearest even, saturating) and the
// block's max |h| joins the layer's amax when the token has a kept slot.
template <typename T>
__global__ void __launch_bounds__(128) gather_kernel(DispatchArgs a) {
  constexpr bool kFp8 = std::is_same<T, e4m3>::value;
  pdl_wait();
  __shared__ float s_red[4];
  const int64_t t = blockIdx.x;
  const float* z = a.z + t * a.L;
  float ss = 0.0f;
  for (int i = threadIdx.x * 8; i < a.L; i += 1024) {
    float v[8];
    ld8(z + i, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(~0u, ss, o);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  ss = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)a.L), a.eps)));
  int32_t slots[32];
  int ns = 0;
  for (int j = 0; j < a.k; ++j) {
    int32_t s = a.slot_of[t * a.k + j];
    if (s >= 0 && s < a.pool_rows) slots[ns++] = s;
  }
  T* xp = static_cast<T*>(a.x_perm);
  const float qs = kFp8 ? *a.x_scale : 1.0f;
  float amax = 0.0f;
  for (int i = threadIdx.x * 8; i < a.L; i += 1024) {
    float v[8], g[8];
    ld8(z + i, v);
    ld8(a.gamma + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = v[q] * rstd * g[q];
    if (kFp8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        amax = fmaxf(amax, fabsf(v[q]));
        v[q] = v[q] * qs;
      }
    }
    for (int j = 0; j < ns; ++j) st8(xp + (int64_t)slots[j] * a.L + i, v);
  }
  if (kFp8 && ns > 0) {
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
    if ((threadIdx.x & 31) == 0) amax_update(&a.hdr->amax_x, amax);
  }
}

// c[t] = sum_j gate[t, j] * y_perm[slot_of[t, j]] over kept j, in order j = 0..k-1.
template <typename T>
// One block per `tpb` consecutive tokens (several when k is small, so that a block moves enough
// bytes). Each token's kept rows are summed in the fixed order j = 0..k-1; the loads of up to four
// rows are issued together before their products are accumulated in that order.
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a, int tpb) {
  pdl_wait();
  const T* yp = static_cast<const T*>(a.y_perm);
  T* out = static_cast<T*>(a.out);
  const int64_t t_end = imin64(a.T, ((int64_t)blockIdx.x + 1) * tpb);
  for (int64_t t = (int64_t)blockIdx.x * tpb; t < t_end; ++t) {
    int32_t slots[32];
    float gates[32];
    int ns = 0;
    for (int j = 0; j < a.k; ++j) {
      int32_t s = a.slot_of[t * a.k + j];
      if (s >= a.pool_rows || s < -1) {
        if (threadIdx.x == 0) report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t);
        continue;
      }
      if (s >= 0) { slots[ns] = s; gates[ns] = a.gate[t * a.k + j]; ++ns; }
    }
    for (int i = threadIdx.x * 8; i < a.L; i += 1024) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      int j = 0;
      for (; j + 4 <= ns; j += 4) {
        float v[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) ld8(yp + (int64_t)slots[j + u] * a.L + i, v[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(gates[j + u], v[u][q], acc[q]);
        }
      }
      for (; j < ns; ++j) {
        float v[8];
        ld8(yp + (int64_t)slots[j] * a.L + i, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(gates[j], v[q], acc[q]);
      }
      st8(out + t * a.ld_out + i, acc);
    }
  }
}

__global__ void validate_offsets_kernel(const int32_t* off, int G, int64_t rows, DeviceHeader* h) {
  pdl_wait();
  for (int g = threadIdx.x; g <= G; g += blockDim.x) {
    int v = off[g];
    bool bad = v < 0 || v > rows || (g > 0 && off[g - 1] > v);
    if (bad) report_error(h, MOE_ERR_BAD_ROUTING, g);
  }
}

}  // namespace

cudaError_t header_reset(DeviceHeader* h, bool clear_status, cudaStream_t st, bool pdl,
                         int amax_mask) {
  return launch(header_reset_kernel, dim3(1), dim3(32), 0, st, pdl, h, clear_status ? 1 : 0,
                amax_mask);
}

int64_t dispatch_chunks(int64_t T) { return cdiv(T, CH); }

cudaError_t dispatch_run(const DispatchArgs& a, int dtype, cudaStream_t st, bool pdl) {
  cudaError_t err;
  const unsigned nch = (unsigned)a.n_chunks;
  err = launch(hist_kernel, dim3(nch), dim3(CH), (size_t)a.E * 4, st, pdl, a);
  if (err != cudaSuccess) return err;
  err = launch(scan_chunks_kernel, dim3(a.E), dim3(256), 0, st, pdl, a);
  if (err != cudaSuccess) return err;
  err = launch(scan_offsets_kernel, dim3(1), dim3(1024), 0, st, pdl, a);
  if (err != cudaSuccess) return err;
  err = launch(rank_kernel, dim3(nch), dim3(CH), (size_t)a.E * (CH / 32) * 4, st, pdl, a);
  if (err != cudaSuccess) return err;
  if (a.x_perm == nullptr) return cudaSuccess;
  if (a.xperm_fp8)
    return launch(gather_kernel<e4m3>, dim3((unsigned)a.T), dim3(128), 0, st, pdl, a);
  if (dtype == DT_BF16) return launch(gather_kernel<bf16>, dim3((unsigned)a.T), dim3(128), 0, st, pdl, a);
  return launch(gather_kernel<float>, dim3((unsigned)a.T), dim3(128), 0, st, pdl, a);
}

cudaError_t combine_run(const CombineArgs& a, int dtype, cudaStream_t st, bool pdl) {
  // tokens per block: at least ~4 rows of input per block
  const int tpb = a.k >= 4 ? 1 : (a.k == 1 ? 4 : 2);
  const dim3 grid((unsigned)cdiv(a.T, tpb));
  if (dtype == DT_BF16) return launch(combine_kernel<bf16>, grid, dim3(128), 0, st, pdl, a, tpb);
  return launch(combine_kernel<float>, grid, dim3(128), 0, st, pdl, a, tpb);
}

cudaError_t validate_offsets(const int32_t* off, int G, int64_t rows, DeviceHeader* h,
                             cudaStream_t st, bool pdl) {
  return launch(validate_offsets_kernel, dim3(1), dim3(256), 0, st, pdl, off, G, rows, h);
}

}  // namespace moe
