/*
 * moe_gb300.h -- C ABI of the routed mixture-of-experts forward layer for NVIDIA GB300 (sm_103a).
 *
 * The layer (pages: "Marin 535B-A23B: the half of a training run nobody usually shows you",
 * section "What is actually being trained"; "Marin Begins Open Training of a 535B-Parameter
 * MoE Model", section 2): a router picks top_k of n_experts routed experts per token; the
 * token is projected from d_model down to a d_latent-wide latent and RMS-normalised; each
 * chosen expert (a SwiGLU MLP of width d_ff in the latent) processes it; the expert outputs
 * are combined with the router's gates, projected back up to d_model and added to the output
 * of n_shared shared SwiGLU experts (width d_ff_shared) that read every token.
 *
 *   logits = x W_r + b_r                      router, [T, E]
 *   idx, gate = top_k(logits), softmax over the selected logits
 *   z = x W_down;  h = z / sqrt(mean(z^2) + eps) * gamma
 *   o_{t,j} = (silu(h_t W1_e) * (h_t W3_e)) W2_e,  e = idx[t, j]
 *   c_t = sum_j gate[t, j] o_{t,j}            (ascending expert order, dropped terms skipped)
 *   y = c W_up + sum_s (silu(x W1_s[s]) * (x W3_s[s])) W2_s[s]
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every buffer (device memory unless stated) and the workspace.
 *     The library allocates no device memory, keeps no pointer after a call returns and frees
 *     nothing.
 *   - Streams: `stream` is a cudaStream_t (NULL = legacy default stream). Every call only
 *     enqueues work on it and returns; nothing synchronises the host except
 *     moe_get_device_status().
 *   - Layouts: all matrices are row-major and densely packed. Activations and weights have
 *     the element type cfg->dtype (bf16 or fp32); b_router, rms_gamma and gates are fp32;
 *     indices, counts, offsets and slots are int32.
 *   - Alignment: every pointer must be 16-byte aligned; d_model, d_latent, d_ff and d_ff_shared
 *     must be multiples of 8, and so must n_experts for the bf16 router (moe_route,
 *     moe_forward); MOE_ERR_ALIGNMENT otherwise.
 *   - Workspace: caller-owned device memory of moe_workspace_size() bytes, 256-byte aligned. Its
 *     first 256 bytes hold the device report; clear them once after allocating the workspace
 *     (moe_clear_device_status, or zero-filled memory). moe_forward clears the report itself;
 *     the split calls accumulate into it.
 *   - Errors: argument errors return before anything is enqueued. A failed launch returns
 *     MOE_ERR_CUDA. Errors found on the device (an out-of-range expert id or slot, offsets that
 *     are not monotone, a device wait that timed out) are recorded in a status word inside the
 *     workspace and read by moe_get_device_status(); the kernels then skip the offending item
 *     instead of touching memory out of range. No call aborts the process.
 *   - Determinism: outputs are bitwise identical for identical inputs and configuration (the
 *     combine sums each token's terms in a fixed order, as the ordered-gather combine of the
 *     Marin summary for the week of 2026-09-14, post-training epic (#9144), does).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* a NULL required pointer, a non-positive size, top_k > n_experts */
  MOE_ERR_UNSUPPORTED = 2,    /* a size beyond the limits below */
  MOE_ERR_WORKSPACE = 3,      /* ws_bytes smaller than moe_workspace_size() */
  MOE_ERR_ALIGNMENT = 4,      /* a pointer not 16-byte aligned, or a bf16 width not a multiple of 8 */
  MOE_ERR_CUDA = 5,           /* a CUDA launch or runtime call failed */
  MOE_ERR_BAD_ROUTING = 6,    /* device: an expert id, slot or offset out of range or unordered */
  MOE_ERR_DEVICE_TIMEOUT = 7  /* device: a bounded wait inside a kernel gave up */
} moe_status_t;

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype_t;

/* cfg->flags */
#define MOE_FLAG_PDL  (1u << 0)  /* launch dependent kernels with programmatic dependent launch */
#define MOE_FLAG_SIMT (1u << 1)  /* bf16: run every GEMM on CUDA cores (fp32 FMA) instead of tcgen05 */
/* bf16 layers on the tensor-core path: the routed expert MLP runs as fp8 ragged dots (the Marin
 * summary of the week of 2026-07-06, B200 training MFU epic, #6880 / #7079: E4M3 in the forward
 * pass, delayed scaling). Both operands of both expert GEMMs are FP8 E4M3 (OCP: 1 sign, 4
 * exponent bits with bias 7, 3 fraction bits, largest finite 448): the banks w1, w3, w2 with
 * one fp32 scale per expert output column, the grouped rows x_perm and the SwiGLU hidden with
 * one fp32 quantization multiplier each (moe_fp8_t). Router, latent projection, shared experts,
 * combine and up-projection stay bf16. Requires d_latent and d_ff to be multiples of 128. */
#define MOE_FLAG_FP8_EXPERTS (1u << 2)

/* Operands and state of the fp8 expert MLP (MOE_FLAG_FP8_EXPERTS). All pointers are device
 * memory owned by the caller.
 * A tensor v is quantized with its multiplier S to codes q = e4m3(fp32(v * S)), round to nearest
 * even, magnitudes beyond 448 saturated; it is dequantized as q * fp32(1 / S). x_scale and
 * h_scale are the delayed-scaling state (set from the amax of earlier steps by the caller);
 * x_amax and h_amax receive this call's max |v| of the tensors quantized (before
 * quantization), for the caller's next scales. */
typedef struct {
  const float* w1_scale;  /* [E, F] expert weight = E4M3 value * its column's scale */
  const float* w3_scale;  /* [E, F] */
  const float* w2_scale;  /* [E, L] */
  const float* x_scale;   /* [1] S_x: multiplier of the grouped rows h (x_perm) */
  const float* h_scale;   /* [1] S_h: multiplier of the hidden silu(x W1) * (x W3) */
  float*       x_amax;    /* [1] or NULL: max |h| over the rows written to x_perm */
  float*       h_amax;    /* [1] or NULL: max |hidden| over the active rows */
} moe_fp8_t;

/* Limits: 1 <= top_k <= 32, top_k <= n_experts <= 1024, T * top_k < 2^31. The tensor-core
 * GEMMs (bf16 layers without MOE_FLAG_SIMT, and every fp8-expert layer) also need n_experts,
 * d_model, d_latent and d_ff of at least 64, and d_ff_shared a multiple of 128 when n_shared > 0;
 * other sizes return MOE_ERR_UNSUPPORTED before any launch (MOE_FLAG_SIMT runs them). */

typedef struct {
  int64_t  T;            /* tokens */
  int32_t  d_model;      /* d */
  int32_t  d_latent;     /* L */
  int32_t  n_experts;    /* E */
  int32_t  top_k;        /* k */
  int32_t  d_ff;         /* F, routed expert SwiGLU width */
  int32_t  n_shared;     /* S, shared experts (0 allowed) */
  int32_t  d_ff_shared;  /* F_s */
  /* Per-expert capacity C = ceil(capacity_num * T * top_k / (capacity_den * n_experts)),
   * computed in integers; capacity_num <= 0 means no capacity (nothing is dropped). The
   * capacity factors 1.10 / 1.15 and the drop of assignments past a fixed buffer are those of
   * the open-training page, section 2; a dropped assignment contributes nothing and the other
   * gates are not renormalised ("the token skips that expert", teardown section "21% to 27%
   * MFU without stopping the run"). */
  int32_t  capacity_num;
  int32_t  capacity_den;
  float    rms_eps;      /* RMSNorm epsilon */
  int32_t  dtype;        /* moe_dtype_t */
  uint32_t flags;        /* MOE_FLAG_* */
  /* Physical rows of the expert-grouped buffers x_perm / y_perm passed to moe_expert_ffn and
   * moe_combine; 0 means T * top_k. Rows past expert_offsets[E] are padding that no kernel
   * reads or writes (the "mask-free" ragged expert MLP with physical vs active group sizes,
   * teardown section "21% to 27% MFU without stopping the run"). */
  int64_t  pool_rows;
} moe_config_t;

/* Weights of one layer. Expert banks are stacked [experts, d_in, d_out] (teardown section
 * "A sphere for every matrix"). */
typedef struct {
  const void*  w_router;   /* [d, E] */
  const float* b_router;   /* [E] fp32, may be NULL (zero bias) */
  const void*  w_down;     /* [d, L] */
  const float* rms_gamma;  /* [L] fp32 */
  const void*  w1;         /* [E, L, F] gate projection */
  const void*  w3;         /* [E, L, F] up projection */
  const void*  w2;         /* [E, F, L] down projection */
  const void*  w1_s;       /* [S, d, F_s] */
  const void*  w3_s;       /* [S, d, F_s] */
  const void*  w2_s;       /* [S, F_s, d] */
  const void*  w_up;       /* [L, d] */
  const moe_fp8_t* fp8;    /* MOE_FLAG_FP8_EXPERTS: required (w1, w3, w2 are E4M3); else ignored */
} moe_weights_t;

/* Optional extras of moe_forward; every pointer may be NULL. Device buffers receive copies of
 * the routing results. stage_events, when not NULL, holds MOE_FORWARD_STAGES + 1 cudaEvent_t
 * handles created by the caller; event i is recorded on `stream` before stage i and the last
 * one after the final stage, so that the caller can time stages without a profiler. Under
 * stream capture they are recorded as external event nodes: every replay of the graph records
 * them, and the caller can synchronize on them and time them as usual.
 * moe_forward may be captured in a CUDA graph (its kernels, their programmatic-dependent-launch
 * edges and these events) and replayed; the graph keeps the buffers it was captured with. */
#define MOE_FORWARD_STAGES 8   /* prep, front GEMM, router select, dispatch, expert GEMM 1,
                                  expert GEMM 2, combine, back GEMM */
typedef struct {
  int32_t* topk_idx;        /* [T, k] */
  float*   topk_gate;       /* [T, k] */
  int32_t* expert_counts;   /* [E] assignments per expert before the capacity clamp */
  int32_t* expert_offsets;  /* [E + 1] */
  int32_t* slot_of;         /* [T, k] */
  int32_t* n_dropped;       /* [1] */
  void* const* stage_events;
  /* Input, [T] bytes or NULL (every token real): 0 marks attention-mask padding, which is
   * routed but not dispatched (the weekly summary of 2026-09-14, hero-run epic, #9159, excludes
   * attention-mask padding from MoE dispatch). A padding token's assignments are not counted,
   * take no capacity, are not drops and get slot -1; its routed output is zero, so y[t] is the
   * shared experts' output alone. */
  const uint8_t* token_mask;
} moe_forward_aux_t;

/* Diagnostics recorded on the device by the last calls (see moe_get_device_status). */
typedef struct {
  int32_t status;          /* moe_status_t of the first device-detected error, MOE_OK if none */
  int32_t detail;          /* error-specific detail (e.g. the offending token or expert) */
  int32_t n_refined;       /* tokens whose top-k needed the compensated re-evaluation */
  int32_t n_exact;         /* tokens whose top-k needed exact (integer) logits */
} moe_device_report_t;

MOE_API int32_t     moe_abi_version(void);
MOE_API const char* moe_status_string(moe_status_t status);

/* The cudaError_t behind the calling thread's most recent MOE_ERR_CUDA (cudaSuccess if none), and
 * its name in *name (static storage) when name is not NULL. */
MOE_API int32_t moe_last_cuda_error(const char** name);

/* Bytes of workspace every call below needs for this configuration (one size fits all calls).
 * The workspace must be 256-byte aligned device memory owned by the caller. */
MOE_API moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Byte offsets, from the start of the workspace, of the intermediates that moe_forward leaves
 * there after its call (stream-ordered): the fp32 latent z [T, L] before the RMSNorm, the
 * expert-grouped rows x_perm [pool_rows, L] (bf16, fp32 for an fp32 layer, or E4M3 codes with
 * MOE_FLAG_FP8_EXPERTS), the routed SwiGLU hidden [pool_rows, F] (same type), the routed experts'
 * outputs y_perm [pool_rows, L], the shared experts' hidden a_shared [T, S*F_s], the combine
 * c [T, L] (16-bit or fp32 like the layer), perm [pool_rows] int32 and the group offsets
 * [E + 1] int32. Rows of x_perm, hidden and y_perm at or past expert_offsets[E] are padding that
 * no kernel writes. For inspection and testing; the regions are overwritten by the next call that
 * uses the workspace. Returns MOE_ERR_INVALID_ARG for a NULL argument and the configuration
 * errors of moe_workspace_size. */
typedef struct {
  size_t z, x_perm, hidden, y_perm, a_shared, combined, perm, expert_offsets;
} moe_workspace_regions_t;
MOE_API moe_status_t moe_workspace_regions(const moe_config_t* cfg, moe_workspace_regions_t* out);

/* Router: logits = x W_r + b_r, then per token the top_k experts by the exact real value of
 * the logit (ties to the lowest index), written in ascending expert order to topk_idx [T, k],
 * and gates topk_gate [T, k] = softmax over the selected logits. The router weight and bias
 * are those of the teardown's section "The one knob nobody pinned". The selection is exact:
 * fp32 logits decide a token when their rigorous error bounds separate the k-th from the
 * (k+1)-th expert; otherwise the candidates are re-evaluated with a compensated dot product
 * and, if still too close, with exact integer arithmetic (the teardown's section "What I'd
 * take from it" reports that router arithmetic alone changed the top-8 of ~9% of tokens). */
MOE_API moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* b_router, int32_t* topk_idx, float* topk_gate,
                       void* ws, size_t ws_bytes, void* stream);

/* Dispatch: z = x W_down, h = RMSNorm(z) * gamma; expert_counts [E] (before capacity);
 * expert_offsets [E+1] = exclusive prefix sum of min(counts, C); slot_of [T, k] = the row of
 * assignment (t, j) in the expert-grouped buffer (rows of one expert in ascending token order,
 * as the ragged transport delivers them), -1 if dropped; perm [T*k] = t*k + j at each used
 * row (entries past expert_offsets[E] are left untouched); n_dropped [1];
 * x_perm [pool_rows, L] receives h at every used row. topk_idx must hold ascending, distinct
 * expert ids (as moe_route writes them). Under MOE_FLAG_FP8_EXPERTS x_perm receives the E4M3
 * codes of h (one byte each) under fp8->x_scale, and fp8->x_amax (if not NULL) max |h| over the
 * rows written; fp8 is ignored (may be NULL) otherwise. token_mask ([T] bytes or NULL) marks
 * attention-mask padding with 0: those tokens are not dispatched (see moe_forward_aux_t). */
MOE_API moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const void* w_down,
                         const float* rms_gamma, const int32_t* topk_idx,
                         const uint8_t* token_mask,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                         int32_t* slot_of, int32_t* n_dropped, void* x_perm,
                         const moe_fp8_t* fp8, void* ws, size_t ws_bytes, void* stream);

/* Experts: for every expert e and every row r in [expert_offsets[e], expert_offsets[e+1]):
 * y_perm[r] = (silu(x_perm[r] W1_e) * (x_perm[r] W3_e)) W2_e. Rows past expert_offsets[E]
 * (pool padding) are neither read nor written; an expert with no rows loads no weights.
 * The grouped GEMM reads expert_offsets only after the kernel that wrote them has completed
 * (the hang of the weekly summary of 2026-09-14, hero-run epic, came from warps that read
 * the group boundaries early under programmatic dependent launch).
 * Under MOE_FLAG_FP8_EXPERTS, x_perm and w1/w3/w2 are E4M3 codes (x_perm as moe_permute
 * writes it), fp8 supplies their scales, the hidden is quantized with fp8->h_scale before the
 * second GEMM, fp8->h_amax (if not NULL) receives max |hidden|; y_perm is bf16 either way.
 * fp8 is ignored (may be NULL) without the flag.
 * When x is not NULL, also the shared experts' hidden activations
 * a_shared [T, S*F_s] = concat_s silu(x W1_s[s]) * (x W3_s[s]). */
MOE_API moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_perm,
                                    const int32_t* expert_offsets, const void* w1, const void* w3,
                                    const void* w2, const moe_fp8_t* fp8, void* y_perm,
                                    const void* x, const void* w1_s, const void* w3_s,
                                    void* a_shared, void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace moe_expert_ffn_backward needs (256-byte aligned device memory owned by the
 * caller, zero-filled before its first use like the forward's; it starts with the same device
 * report, read with moe_get_device_status). */
MOE_API moe_status_t moe_backward_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Backward of moe_expert_ffn's routed experts, given dy_perm = dL/dy_perm [pool_rows, L]: with
 * G = x W1_e, U = x W3_e and A = silu(G) * U for the rows of expert e (recomputed here),
 *   dA = dy W2_e^T, dG = dA * U * silu'(G), dU = dA * silu(G),
 *   dx_perm = dG W1_e^T + dU W3_e^T            [pool_rows, L] (rows past expert_offsets[E] untouched),
 *   dw1[e] = x^T dG, dw3[e] = x^T dU            [E, L, F], dw2[e] = A^T dy  [E, F, L]
 * (experts with no rows get zero gradients). This is the custom VJP of the ragged dot in the
 * Marin summary of the week of 2026-07-06 (#5330): the input gradient is a grouped GEMM against
 * the transposed expert weights, the weight gradients contract over each expert's ragged rows.
 * bf16 layers on the tensor-core path only (else MOE_ERR_UNSUPPORTED); d_latent and d_ff must
 * be multiples of 128 (else MOE_ERR_ALIGNMENT). All outputs bf16 with fp32 accumulation. */
MOE_API moe_status_t moe_expert_ffn_backward(const moe_config_t* cfg, const void* x_perm,
                                             const int32_t* expert_offsets, const void* w1,
                                             const void* w3, const void* w2, const void* dy_perm,
                                             void* dx_perm, void* dw1, void* dw3, void* dw2,
                                             void* ws, size_t ws_bytes, void* stream);

/* Gradients of one layer's weights (device memory owned by the caller; layouts as in
 * moe_weights_t, bf16 unless stated). */
typedef struct {
  void*  dw_router;   /* [d, E] */
  float* db_router;   /* [E] fp32, or NULL (not computed) */
  void*  dw_down;     /* [d, L] */
  float* drms_gamma;  /* [L] fp32, or NULL (not computed) */
  void*  dw1;         /* [E, L, F] */
  void*  dw3;         /* [E, L, F] */
  void*  dw2;         /* [E, F, L] */
  void*  dw1_s;       /* [S, d, F_s] (NULL when S = 0) */
  void*  dw3_s;       /* [S, d, F_s] */
  void*  dw2_s;       /* [S, F_s, d] */
  void*  dw_up;       /* [L, d] */
} moe_grads_t;

/* Bytes of workspace moe_backward needs (256-byte aligned, zero-filled before first use). */
MOE_API moe_status_t moe_layer_backward_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Backward of moe_forward: given dy = dL/dy [T, d], writes dx = dL/dx [T, d] and every weight
 * gradient into g. fwd_ws is the workspace of a moe_forward call with the same cfg, weights and
 * x, left untouched since: the backward reads the routing, gates, slots, group offsets, the
 * latent z, the grouped rows, the experts' outputs, the combine c and the shared hidden from
 * it. Top-k selection has no gradient; the router's logits get the softmax-over-selection
 * gradient G_j (dG_j - sum_i G_i dG_i) of their gates. The routed experts run
 * moe_expert_ffn_backward's kernels; everything else is bf16 GEMMs on tensor cores (K-major
 * weight tiles for the input gradients, row-contracting kernels for the weight gradients) and
 * per-token kernels for the combine, RMSNorm and router backward. Padding tokens (token_mask)
 * and dropped assignments contribute nothing to the routed part. bf16 layers on the
 * tensor-core path only, without fp8 experts (else MOE_ERR_UNSUPPORTED); d, d_latent, d_ff and
 * n_shared * d_ff_shared multiples of 128, n_experts and d_ff_shared of 64, n_shared <= 2. */
MOE_API moe_status_t moe_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                                  const void* dy, void* dx, const moe_grads_t* g,
                                  const void* fwd_ws, size_t fwd_ws_bytes, void* ws,
                                  size_t ws_bytes, void* stream);

/* Combine: c[t] = sum over j with slot_of[t, j] >= 0, in order j = 0..k-1, of
 * topk_gate[t, j] * y_perm[slot_of[t, j]] (fp32 accumulation). When w_up is NULL, out [T, L]
 * receives c (the gate-weighted un-permute back to arrival order, e.g. of one expert-parallel
 * rank's slice with k = 1); otherwise out [T, d] receives y = c W_up + a_shared W2_s
 * (a_shared / w2_s may be NULL when n_shared == 0). */
MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* slot_of,
                         const float* topk_gate, const void* a_shared, const void* w_up,
                         const void* w2_s, void* out, void* ws, size_t ws_bytes, void* stream);

/* The whole layer: y [T, d] from x [T, d], all stages enqueued on `stream` with no host
 * synchronisation. aux may be NULL. */
MOE_API moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, void* y,
                         void* ws, size_t ws_bytes, void* stream, const moe_forward_aux_t* aux);

/* Serving over host memory: moe_forward on n_batches batches, batch i reading x_host[i] and
 * writing y_host[i] ([T, d] each in the layer dtype; pinned host memory makes the copies
 * asynchronous). Batch i + 1's input is copied in on h2d_stream and batch i - 1's output copied
 * out on d2h_stream while batch i runs on `stream`; x_stage and y_stage are device staging
 * buffers of 2 * T * d elements each (two slots), ws as for moe_forward. The three streams must
 * be distinct. Returns once everything is enqueued; `stream` completes after the last output
 * copy. */
MOE_API moe_status_t moe_forward_pipelined(const moe_config_t* cfg, const moe_weights_t* w,
                                           int32_t n_batches, const void* const* x_host,
                                           void* const* y_host, void* x_stage, void* y_stage,
                                           void* ws, size_t ws_bytes, void* stream,
                                           void* h2d_stream, void* d2h_stream);

/* Waits for `stream`, then copies the device report out of the workspace into *out (host
 * memory). Returns MOE_ERR_CUDA if the wait or the copy fails. */
MOE_API moe_status_t moe_get_device_status(const void* ws, size_t ws_bytes, void* stream,
                                   moe_device_report_t* out);

/* Enqueues a reset of the device report (status, detail and counters) to zero. */
MOE_API moe_status_t moe_clear_device_status(void* ws, size_t ws_bytes, void* stream);

/* Self-test of failure detection: enqueues a kernel whose single thread waits, with the bounded
 * mbarrier wait every tensor-core kernel of this library uses, on a barrier that nothing ever
 * arrives at. After limit_ms (1..10000) the wait gives up and records MOE_ERR_DEVICE_TIMEOUT
 * (detail 99) in the workspace's device report; the kernel then returns normally and the CUDA
 * context stays usable. Read the result with moe_get_device_status. */
MOE_API moe_status_t moe_selftest_device_timeout(void* ws, size_t ws_bytes, uint32_t limit_ms,
                                                 void* stream);

/* Routing for callers that cannot allocate device memory. Some callers of this library run
 * where no allocation may happen: inside an allocator-free runtime or plugin that is handed only
 * its input and output buffers, or code that must not call cudaMalloc (which can synchronise
 * the device) while other work is in flight. For them this entry point computes exactly what
 * moe_route computes (same kernels, same results) but takes no workspace: its scratch is a
 * fixed array of 32 MiB inside the library, present on every GPU that loads the library until
 * the process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Sizes: the routing scratch (256 B + T*E*4 + E*d*elem + E*4 + 3*T*4 bytes, plus
 *     64*(E*161 + 8) bytes of exact-stage state, each region rounded up to 256 B) must fit in
 *     32 MiB, else MOE_ERR_WORKSPACE and nothing is enqueued; the 535B-shaped router
 *     (T = 8192, E = 384, d = 6144, bf16) needs 21.4 MB.
 *   - Set-up: every call looks up the array's device address in the current device's context.
 *     The array's memory is committed when the library's device code is first loaded on a
 *     device (with lazy module loading, the default, that is the first call into the library on
 *     that device), and that load can synchronise the device. Callers that cannot accept this
 *     mid-run make one library call on each device during their set-up, before any stream
 *     capture, e.g. one moe_route_noalloc on a small input.
 *   - Sharing: every call on a device uses the same array and leaves its contents behind; each
 *     call clears what must start at zero. Calls whose GPU work overlaps (other streams, other
 *     host threads) race on the array: serialise them.
 *   - device_report: NULL, or 4 int32 of device memory that receive, stream-ordered, the status,
 *     detail, refined-token and exact-token counts of moe_device_report_t for this call.
 * The pages describe no counterpart of this entry point. */
MOE_API moe_status_t moe_route_noalloc(const moe_config_t* cfg, const void* x, const void* w_router,
                                       const float* b_router, int32_t* topk_idx, float* topk_gate,
                                       int32_t* device_report, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
