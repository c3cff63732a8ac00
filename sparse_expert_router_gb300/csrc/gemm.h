// GEMM problem description shared by the CUDA-core and the tcgen05 GEMM kernels.
//
// One problem computes, for every row r and output column c in [0, M):
//   acc(r, c) = sum over segments s of  sum_k act_s[r, k] * W_s[group][k, col]
// and writes an epilogue of acc to out[r, out_col0 + c]. Row grouping follows the expert
// layout of the layer: GROUP_ROWS takes the rows of group g from offsets[g]..offsets[g+1]
// and uses expert g's weights (the grouped expert GEMM over ragged groups); GROUP_COLS uses
// one weight matrix per block of Mg output columns for every row (the shared experts, stacked
// [S, d, F_s]); GROUP_NONE is a plain dense GEMM.
#pragma once

#include <stdint.h>
#include <cuda_runtime.h>

namespace moe {

// EPI_SWIGLU_SAVE: as EPI_SWIGLU, and also stores both pre-activations (out2 = x W, out3 = x W3).
// EPI_SWIGLU_BWD: acc = dA (the hidden's gradient); with G, U of the same rows read from aux_g,
// aux_u: out = dA * U * silu'(G), out2 = dA * silu(G).
enum Epi { EPI_F32 = 0, EPI_STORE = 1, EPI_SWIGLU = 2, EPI_SWIGLU_SAVE = 3, EPI_SWIGLU_BWD = 4 };
enum GroupMode { GROUP_NONE = 0, GROUP_ROWS = 1, GROUP_COLS = 2 };

constexpr int GEMM_MAX_SEG = 6;

struct GemmSeg {
  const void* act;   // [rows, K] row-major (leading dimension ld, or K when ld is 0)
  // NONE: [K, M]; ROWS: [G, K, M]; COLS: [M / Mg, K, Mg]. With a_kmajor the bank holds the
  // transposed matrices, [M, K] per weight group (a stored [d_in, d_out] weight used as W^T).
  const void* w;
  const void* w3;    // EPI_SWIGLU: the up-projection weights, same layout as w
  int K;
  int64_t ld = 0;    // tcgen05 only: elements between rows of act (0: K)
};

struct GemmProblem {
  int epi = EPI_STORE;
  int group = GROUP_NONE;
  int M = 0;                 // output columns
  int Mg = 0;                // GROUP_COLS: columns per weight matrix
  int n_seg = 1;
  GemmSeg seg[GEMM_MAX_SEG] = {};
  const int32_t* offsets = nullptr;  // GROUP_ROWS: [G + 1], device
  int G = 1;
  int64_t rows = 0;          // rows of act and out (GROUP_ROWS: physical rows; offsets clamp to it)
  void* out = nullptr;
  int64_t ld_out = 0;        // elements per output row
  int out_col0 = 0;
  const float* bias = nullptr;  // EPI_F32: [M] or NULL
  int dtype = 0;             // DT_BF16 / DT_F32: act, weights and EPI_STORE/EPI_SWIGLU output
  // tcgen05 only, EPI_F32 dense single-segment problems: the accumulator is restarted every
  // kchunk k-blocks of 64 and the chunk results are summed in fp32 by the epilogue (a tighter
  // rounding-error bound for the router's certified top-k). 0 = one accumulation over K.
  int kchunk = 0;
  // tcgen05 only: weights (w, w3) and activations are E4M3 codes (MMA kind::f8f6f4). The
  // epilogue multiplies each output feature's accumulator by fp32(1 / act_scale[0]) times the
  // feature's weight scale ([G, M] fp32: w_scale for w, w3_scale for w3) before the epilogue
  // function.
  int w_fp8 = 0;
  const float* w_scale = nullptr;
  const float* w3_scale = nullptr;
  const float* act_scale = nullptr;
  // EPI_SWIGLU with E4M3 output: out receives the codes of value * out_scale[0]; the largest
  // |value| is max-reduced into *amax (fp32 bits).
  int out_fp8 = 0;
  const float* out_scale = nullptr;
  uint32_t* amax = nullptr;
  // tcgen05 only, bf16: the weight operand is K-major ([M, K] per group, see GemmSeg::w)
  int a_kmajor = 0;
  // EPI_SWIGLU_SAVE / EPI_SWIGLU_BWD extra outputs and inputs ([rows, M] bf16, leading
  // dimension ld_out for outputs and ld_aux for inputs)
  void* out2 = nullptr;
  void* out3 = nullptr;
  const void* aux_g = nullptr;
  const void* aux_u = nullptr;
  int64_t ld_aux = 0;
  // tcgen05 only, one dense bf16 problem per launch: segment cmb_seg's activations (bf16
  // [rows, K]) are the gate-weighted combine c[t] = sum over kept j, in order, of
  // gate[t, j] * y_perm[slot_of[t, j]], computed in the same launch by the epilogue warps before
  // they drain any accumulator. A token tile of that segment is loaded only after
  // cmb_ready[tile] (zeroed before the launch, [ceil(rows / 128)]) counts all of its rows.
  int cmb_seg = -1;
  const void* cmb_y_perm = nullptr;
  const int32_t* cmb_slot = nullptr;
  const float* cmb_gate = nullptr;
  int cmb_k = 0;
  int64_t cmb_pool_rows = 0;
  uint32_t* cmb_ready = nullptr;
};

// CUDA-core GEMM (fp32 FMA, sequential accumulation over k for every output). The n problems
// must be independent; up to three share one launch.
cudaError_t gemm_simt(const GemmProblem* probs, int n, cudaStream_t stream, bool pdl);

// tcgen05 GEMM (bf16 operands, fp32 accumulation in tensor memory). Up to 3 problems share
// one persistent launch. Returns cudaErrorNotSupported when a problem does not fit its rules.
cudaError_t gemm_tc(const GemmProblem* probs, int n_probs, void* dev_header, cudaStream_t stream,
                    bool pdl);
bool gemm_tc_supported(const GemmProblem& p);
// Whether gemm_tc would run these problems, launched together, as CTA pairs.
bool gemm_tc_pairs(const GemmProblem* probs, int n_probs);

// Self-test of the kernels' bounded mbarrier wait (a barrier nothing arrives at).
cudaError_t bounded_wait_selftest(void* dev_header, uint64_t limit_ns, cudaStream_t stream);

}  // namespace moe
