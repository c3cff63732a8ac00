// Router selection kernels (see router.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct RouterArgs {
  const void* x;          // [T, d]
  const void* w_router;   // [d, E]
  const float* bias;      // [E] or NULL
  const float* logits;    // [T, E] fp32 logits (bias included) from the router GEMM
  void* wrT;              // [E, d] workspace: W_r transposed
  float* wnorm;           // [E] workspace: upper bounds of ||W_r[:, e]||_2
  float* xnorm;           // [T] workspace: upper bounds of ||x_t||_2
  int64_t T;
  int d, E, k;
  float gam_d;            // gamma_d = d u / (1 - d u), u = 2^-24, rounded up
  float cgam;             // c * gamma_d: the logit GEMM's accumulation error factor
  float g2;               // gamma_n^2 of the compensated dot product, rounded up
  int32_t* idx;           // [T, k] out
  float* gate;            // [T, k] out
  int32_t* refine_list;   // [T] workspace
  int32_t* exact_list;    // [T] workspace
  DeviceHeader* hdr;
  // router_saved_bytes(E, n_saved) of workspace, or NULL: the final classification of the
  // first n_saved tokens of the exact list (written by the refine stage), which lets the exact
  // stage skip stages 1 and 2 and split stage 3 over several blocks per token
  void* saved;
  int n_saved;
};

size_t router_saved_bytes(int E, int n_saved);

// W_r^T and the column-norm bounds (needed before router_select).
cudaError_t router_prepare(const RouterArgs& a, int dtype, cudaStream_t st, bool pdl);
// Stage 1 (all tokens), stage 2 (undecided tokens) and stage 3 (still undecided tokens).
// hdr->n_refine and hdr->n_exact must be zero before the call.
cudaError_t router_select(const RouterArgs& a, int dtype, int num_sms, cudaStream_t st, bool pdl);

}  // namespace moe
