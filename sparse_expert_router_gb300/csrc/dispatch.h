// Dispatch / combine kernels (see dispatch.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct DispatchArgs {
  const int32_t* idx;     // [T, k] ascending expert ids
  const uint8_t* mask;    // [T] or NULL: 0 = attention-mask padding, not dispatched
  int64_t T;
  int k, E, L;
  int cap;                // capacity, -1 = none
  int64_t n_chunks;
  int32_t* chunk_hist;    // [n_chunks, E] workspace
  int32_t* chunk_base;    // [n_chunks, E] workspace
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E + 1]
  int32_t* n_dropped;     // [1] or NULL
  int32_t* slot_of;       // [T, k]
  int32_t* perm;          // [pool_rows]
  int64_t pool_rows;
  const float* z;         // [T, L] fp32 latent before the norm
  const float* gamma;     // [L]
  float eps;
  void* x_perm;           // [pool_rows, L] or NULL (no scatter)
  // fp8 experts: x_perm holds E4M3 codes of h * x_scale[0]; max |h| over the quantized rows
  // goes to hdr->amax_x
  int xperm_fp8;
  const float* x_scale;
  DeviceHeader* hdr;
};

struct CombineArgs {
  const void* y_perm;     // [pool_rows, L]
  const int32_t* slot_of; // [T, k]
  const float* gate;      // [T, k]
  int64_t T;
  int k, L;
  int64_t pool_rows;
  void* out;              // [T, ld_out] (first L columns written)
  int64_t ld_out;
  DeviceHeader* hdr;
};

// Zeroes the router counters, and the status (clear_status) and the amax fields named by
// amax_mask (bit 0: amax_x, bit 1: amax_h), and n_zero words at `zero`.
cudaError_t header_reset(DeviceHeader* h, bool clear_status, cudaStream_t st, bool pdl,
                         int amax_mask = 0, uint32_t* zero = nullptr, int n_zero = 0);
int64_t dispatch_chunks(int64_t T);
cudaError_t dispatch_run(const DispatchArgs& a, int dtype, cudaStream_t st, bool pdl);
cudaError_t combine_run(const CombineArgs& a, int dtype, cudaStream_t st, bool pdl);
cudaError_t validate_offsets(const int32_t* off, int G, int64_t rows, DeviceHeader* h,
                             cudaStream_t st, bool pdl);

}  // namespace moe
