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

// Tokens per dispatch chunk: one warp lane per token. A token's slot for expert e is
// offsets[e] + (tokens of earlier chunks that chose e: the chunk base) + (earlier tokens of its
// own chunk that chose e: a 32-bit mask and a popcount), so slots are stable in token order and
// need no atomics.
constexpr int CH = 32;
constexpr int HIST_WARPS = 4;   // chunks per histogram block

__global__ void header_reset_kernel(DeviceHeader* h, int clear_status, int amax_mask,
                                    uint32_t* zero, int n_zero) {
  pdl_wait();
  if (threadIdx.x == 0) {
    if (clear_status) { h->status = 0; h->detail = 0; }
    h->n_refine = 0;
    h->n_exact = 0;
    if (amax_mask & 1) h->amax_x = 0;
    if (amax_mask & 2) h->amax_h = 0;
  }
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero[i] = 0u;
}

// An assignment (t, j) is valid when its expert id is in range and the token's ids ascend.
__device__ __forceinline__ bool valid_assignment(const int32_t* row, int j, int E) {
  int e = row[j];
  return e >= 0 && e < E && (j == 0 || row[j - 1] < e);
}

// Per-chunk expert counts: each warp counts one 32-token chunk in shared memory. Also zeroes the
// ticket of the scan that follows.
__global__ void __launch_bounds__(32 * HIST_WARPS) hist_kernel(DispatchArgs a) {
  pdl_wait();
  extern __shared__ int s_cnt[];   // [HIST_WARPS][E]
  if (blockIdx.x == 0 && threadIdx.x == 0) a.hdr->dispatch_ticket = 0u;
  for (int i = threadIdx.x; i < HIST_WARPS * a.E; i += 32 * HIST_WARPS) s_cnt[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * HIST_WARPS + warp;
  const int64_t t = c * CH + lane;
  int* cnt = s_cnt + warp * a.E;
  if (t < a.T && (!a.mask || a.mask[t])) {   // padding tokens are not dispatched
    const int32_t* row = a.idx + t * a.k;
    for (int j = 0; j < a.k; ++j) {
      if (valid_assignment(row, j, a.E)) atomicAdd(&cnt[row[j]], 1);
      else report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t);
    }
  }
  __syncwarp();
  if (c < a.n_chunks)
    for (int e = lane; e < a.E; e += 32) a.chunk_hist[c * a.E + e] = cnt[e];
}

// One block per expert: exclusive scan of the expert's per-chunk counts (the base of each
// chunk's ranks) and the expert's total count. The last block to finish (a ticket in the device
// report) then clamps every expert to the capacity, scans the kept counts into the group
// offsets and counts the drops.
__global__ void __launch_bounds__(256) scan_kernel(DispatchArgs a) {
  pdl_wait();
  __shared__ int s_warp[8];
  __shared__ int s_carry;
  __shared__ int s_last;
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
  if (threadIdx.x == 0) {
    a.counts[e] = s_carry;
    __threadfence();                       // the count is visible before the ticket is taken
    s_last = atomicAdd(&a.hdr->dispatch_ticket, 1u) == (unsigned)(a.E - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the last block: capacity clamp and exclusive scan of the kept counts, E <= 1024 experts as
  // four consecutive experts per thread
  constexpr int PER = 4;
  int kept[PER], sum = 0, drop = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int ee = threadIdx.x * PER + i;
    const int cnt = (ee < a.E) ? __ldcg(a.counts + ee) : 0;
    kept[i] = (a.cap >= 0) ? min(cnt, a.cap) : cnt;
    drop += cnt - kept[i];
    sum += kept[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += u;
  }
  int wdrop = drop;
#pragma unroll
  for (int o = 16; o; o >>= 1) wdrop += __shfl_xor_sync(~0u, wdrop, o);
  __shared__ int s_wsum[8], s_wdrop[8];
  if (lane == 31) s_wsum[warp] = incl;
  if (lane == 0) s_wdrop[warp] = wdrop;
  __syncthreads();
  int wbase = 0, dtot = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) wbase += s_wsum[w];
    dtot += s_wdrop[w];
  }
  int run = wbase + incl - sum;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int ee = threadIdx.x * PER + i;
    if (ee < a.E) a.offsets[ee] = run;
    run += kept[i];
    if (ee == a.E - 1) a.offsets[a.E] = run;
  }
  if (threadIdx.x == 0 && a.n_dropped) *a.n_dropped = dtot;
}

// One block per token. Warp 0 first gives the token its slots: the chunk's 32 tokens mark, per
// expert, a 32-bit mask of the tokens that chose it; the token's rank among them is the popcount
// below its lane, plus the chunk base. Slots past the expert's capacity are -1 (dropped). Then
// h = z * rsqrt(mean(z^2) + eps) * gamma is written to every kept slot of the token. With E4M3
// output the rows hold the codes of h * x_scale (round to nearest even, saturating) and the
// block's max |h| joins the layer's amax when the token has a kept slot.
template <typename T>
__global__ void __launch_bounds__(128) gather_kernel(DispatchArgs a) {
  constexpr bool kFp8 = std::is_same<T, e4m3>::value;
  pdl_wait();
  __shared__ float s_red[4];
  __shared__ uint32_t s_mask[1024];          // E <= 1024
  __shared__ int32_t s_slot[32];             // k <= 32
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    for (int e = lane; e < a.E; e += 32) s_mask[e] = 0u;
    __syncwarp();
    const int64_t c = t / CH;
    const int tl = (int)(t % CH);
    const int64_t tt = c * CH + lane;           // this lane's token of the chunk
    if (tt < a.T && (!a.mask || a.mask[tt])) {
      const int32_t* rowl = a.idx + tt * a.k;
      for (int j = 0; j < a.k; ++j)
        if (valid_assignment(rowl, j, a.E)) atomicOr(&s_mask[rowl[j]], 1u << lane);
    }
    __syncwarp();
    if (lane < a.k) {                           // lane j: the token's assignment j
      const int j = lane;
      const int32_t* row = a.idx + t * a.k;
      int32_t slot = -1;
      if ((!a.mask || a.mask[t]) && valid_assignment(row, j, a.E)) {
        const int e = row[j];
        const int r = __popc(s_mask[e] & ((1u << tl) - 1u)) + a.chunk_base[c * a.E + e];
        if (a.cap < 0 || r < a.cap) {
          slot = a.offsets[e] + r;
          if (slot < 0 || slot >= a.pool_rows) {
            report_error(a.hdr, MOE_ERR_BAD_ROUTING, (int)t);
            slot = -1;
          } else {
            a.perm[slot] = (int32_t)(t * a.k + j);
          }
        }
      }
      a.slot_of[t * a.k + j] = slot;
      s_slot[j] = slot;
    }
  }
  // Rows of up to ZC * 1024 features stay in registers between the two passes (all of a
  // thread's loads in flight at once); longer rows are read again. Either way each thread sums
  // its squares in the same order.
  constexpr int ZC = 4;
  const bool cached = a.L <= ZC * 1024;
  const float* z = a.z + t * a.L;
  float zc[ZC][8];
  float ss = 0.0f;
  if (cached) {
#pragma unroll
    for (int u = 0; u < ZC; ++u) {
      const int i = threadIdx.x * 8 + u * 1024;
      if (i < a.L) ld8(z + i, zc[u]);
    }
#pragma unroll
    for (int u = 0; u < ZC; ++u) {
      if (threadIdx.x * 8 + u * 1024 < a.L) {
#pragma unroll
        for (int q = 0; q < 8; ++q) ss = fmaf(zc[u][q], zc[u][q], ss);
      }
    }
  } else {
    for (int i = threadIdx.x * 8; i < a.L; i += 1024) {
      float v[8];
      ld8(z + i, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(~0u, ss, o);
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  if (a.x_perm == nullptr) return;
  ss = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)a.L), a.eps)));
  int ns = 0;
  for (int j = 0; j < a.k; ++j) ns += s_slot[j] >= 0;
  T* xp = static_cast<T*>(a.x_perm);
  const float qs = kFp8 ? *a.x_scale : 1.0f;
  float amax = 0.0f;
  auto emit = [&](int i, float v[8]) {
    float g[8];
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
    for (int j = 0; j < a.k; ++j) {
      const int32_t sl = s_slot[j];
      if (sl >= 0) st8(xp + (int64_t)sl * a.L + i, v);
    }
  };
  if (cached) {
#pragma unroll
    for (int u = 0; u < ZC; ++u) {
      const int i = threadIdx.x * 8 + u * 1024;
      if (i < a.L) emit(i, zc[u]);
    }
  } else {
    for (int i = threadIdx.x * 8; i < a.L; i += 1024) {
      float v[8];
      ld8(z + i, v);
      emit(i, v);
    }
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
                         int amax_mask, uint32_t* zero, int n_zero) {
  return launch(header_reset_kernel, dim3(1), dim3(256), 0, st, pdl, h, clear_status ? 1 : 0,
                amax_mask, zero, n_zero);
}

int64_t dispatch_chunks(int64_t T) { return cdiv(T, CH); }

cudaError_t dispatch_run(const DispatchArgs& a, int dtype, cudaStream_t st, bool pdl) {
  if (a.E > 1024 || a.k > 32) return cudaErrorInvalidValue;
  cudaError_t err;
  const unsigned nhb = (unsigned)cdiv(a.n_chunks, HIST_WARPS);
  err = launch(hist_kernel, dim3(nhb), dim3(32 * HIST_WARPS), (size_t)HIST_WARPS * a.E * 4, st,
               pdl, a);
  if (err != cudaSuccess) return err;
  err = launch(scan_kernel, dim3(a.E), dim3(256), 0, st, pdl, a);
  if (err != cudaSuccess) return err;
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
