// The C ABI: argument validation, workspace layout and the stage sequence of the layer.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "backward.h"
#include "common.cuh"
#include "dispatch.h"
#include "gemm.h"
#include "router.h"
#include "wgrad.h"

using namespace moe;

namespace {

// Factor on the worst-case fp32 accumulation error bound gamma_d * sum|x w| of the tensor-core
// router logits: 2 covers an accumulation that truncates (rounds toward zero) at fp32
// precision at every step; the CUDA-core GEMM accumulates sequentially with round-to-nearest
// FMA and uses 1. Certification needs only a valid bound; a looser bound sends more tokens to
// the compensated stage. tests/test_parity_gpu.py checks the bound on real logits.
constexpr float TC_BOUND_FACTOR = 2.0f;
// The tensor-core router GEMM restarts its accumulator every ROUTER_KCHUNK k-blocks of 64 and
// sums the chunk results in fp32 (error bound c*gamma_256 per chunk plus gamma_nchunks over the
// chunk sums, instead of c*gamma_d).
constexpr int ROUTER_KCHUNK = 4;
// Tokens of the exact stage whose classification the refine stage hands over (the rest, if ever
// more, recompute it, one block per token).
constexpr int ROUTER_SAVED = 64;

int64_t pool_rows_of(const moe_config_t& c) {
  return c.pool_rows > 0 ? c.pool_rows : c.T * (int64_t)c.top_k;
}

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

// Token tiles of the back GEMM (at least 128 rows each) whose combined rows a fused combine counts.
int64_t ready_tiles(int64_t T) { return (T + 127) / 128; }

// Whether the forward's front GEMMs split into a router launch (single-CTA, K-chunked) and a
// CTA-pair launch of the down-projection and shared experts. The pair kernel reads each token tile
// once for two weight tiles, which pays once the front GEMMs are large: the 535B layer's took
// 0.998 -> 0.977 ms at T=8192 (1.6 TFLOP) and 9.80 -> 8.57 ms at T=65536, while on the small bf16
// layer (T=4096, d=2048: 0.16 TFLOP) the router launch running alone cost more than the pairs
// saved (0.121 -> 0.127 ms). So the split is taken from 0.5 TFLOP of front GEMMs up;
// MOE_FRONT_SPLIT in the environment forces it on ("1") or off ("0").
bool front_split_enabled(const moe_config_t& c) {
  static const int mode = [] {
    const char* e = getenv("MOE_FRONT_SPLIT");
    return !e ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (mode >= 0) return mode == 1;
  const double cols = (double)c.n_experts + c.d_latent + 2.0 * c.n_shared * c.d_ff_shared;
  return 2.0 * c.T * (double)c.d_model * cols >= 0.5e12;
}

// Whether the combine runs inside the back GEMM's launch (the shared experts' K segment first,
// while the launch's epilogue warps combine). There the combine is latency-bound: twelve warps per
// SM gather y_perm. It pays only while y_perm, just written by expert GEMM 2, is still in L2 (the
// small bf16 layer, 67 MB of rows: 0.091 -> 0.079 ms for combine and up-projection); with rows
// from HBM the separate combine kernel, spread over one block per token, is faster (the 535B layer
// at T=8192, 403 MB: 0.735 -> 0.826 ms). MOE_FUSED_COMBINE in the environment forces it on ("1")
// or off ("0").
bool fused_combine_enabled(const moe_config_t& c) {
  static const int mode = [] {
    const char* e = getenv("MOE_FUSED_COMBINE");
    return !e ? -1 : (e[0] == '0' ? 0 : 1);
  }();
  if (mode >= 0) return mode == 1;
  const int64_t es = (c.dtype == MOE_BF16) ? 2 : 4;
  return pool_rows_of(c) * (int64_t)c.d_latent * es <= ((int64_t)96 << 20);
}

struct Layout {
  size_t hdr, logits, wrT, wnorm, xnorm, rlist, elist, rsaved, idx, gate, z, chist, cbase, counts,
      offsets, ndrop, slot_of, perm, x_perm, hid, y_perm, a_s, c, cready, total;
};

Layout make_layout(const moe_config_t& c) {
  Layout L{};
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    size_t o = off;
    off = al256(off + (size_t)bytes);
    return o;
  };
  const int64_t es = (c.dtype == MOE_BF16) ? 2 : 4;
  const int64_t T = c.T, E = c.n_experts, k = c.top_k, d = c.d_model, Lt = c.d_latent,
                F = c.d_ff, SF = (int64_t)c.n_shared * c.d_ff_shared, P = pool_rows_of(c),
                nch = dispatch_chunks(T);
  L.hdr = take(sizeof(DeviceHeader));
  L.logits = take(T * E * 4);
  L.wrT = take(E * d * es);
  L.wnorm = take(E * 4);
  L.xnorm = take(T * 4);
  L.rlist = take(T * 4);
  L.elist = take(T * 4);
  L.rsaved = take((int64_t)router_saved_bytes(E, ROUTER_SAVED));
  L.idx = take(T * k * 4);
  L.gate = take(T * k * 4);
  L.z = take(T * Lt * 4);
  L.chist = take(nch * E * 4);
  L.cbase = take(nch * E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.ndrop = take(4);
  L.slot_of = take(T * k * 4);
  L.perm = take(P * 4);
  L.x_perm = take(P * Lt * es);
  L.hid = take(P * F * es);
  L.y_perm = take(P * Lt * es);
  L.a_s = take(T * (SF > 0 ? SF : 1) * es);
  L.c = take(T * Lt * es);
  L.cready = take(ready_tiles(T) * 4);
  L.total = off;
  return L;
}

// Workspace of moe_expert_ffn_backward: the device report, then the recomputed G = X W1,
// U = X W3 and A = silu(G) U and the gradients dG, dU, each [pool_rows, F] bf16.
struct BwdLayout {
  size_t hdr, g, u, a, dg, du, total;
};

BwdLayout make_bwd_layout(const moe_config_t& c) {
  BwdLayout L{};
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    size_t o = off;
    off = al256(off + (size_t)bytes);
    return o;
  };
  const int64_t PF = pool_rows_of(c) * (int64_t)c.d_ff * 2;
  L.hdr = take(sizeof(DeviceHeader));
  L.g = take(PF);
  L.u = take(PF);
  L.a = take(PF);
  L.dg = take(PF);
  L.du = take(PF);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->d_model < 1 || c->d_latent < 1 || c->n_experts < 1 || c->top_k < 1 ||
      c->d_ff < 1 || c->n_shared < 0 || (c->n_shared > 0 && c->d_ff_shared < 1))
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->capacity_num > 0 && c->capacity_den < 1) return MOE_ERR_INVALID_ARG;
  if (c->pool_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.0f) || !isfinite(c->rms_eps)) return MOE_ERR_INVALID_ARG;
  if (c->top_k > 32 || c->n_experts > 1024) return MOE_ERR_UNSUPPORTED;
  if (c->T * (int64_t)c->top_k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (pool_rows_of(*c) >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if ((c->d_model % 8) || (c->d_latent % 8) || (c->d_ff % 8) ||
      (c->n_shared > 0 && (c->d_ff_shared % 8)))
    return MOE_ERR_ALIGNMENT;
  if (c->flags & MOE_FLAG_FP8_EXPERTS) {
    if (c->dtype != MOE_BF16 || (c->flags & MOE_FLAG_SIMT)) return MOE_ERR_UNSUPPORTED;
    if ((c->d_latent % 128) || (c->d_ff % 128)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

bool fp8_experts(const moe_config_t& c) { return (c.flags & MOE_FLAG_FP8_EXPERTS) != 0; }

// The fp8 operands a call reads must be present (and 16-byte aligned where they are arrays).
moe_status_t check_fp8(const moe_config_t& c, const moe_fp8_t* f, bool rows, bool mlp) {
  if (!fp8_experts(c)) return MOE_OK;
  if (!f) return MOE_ERR_INVALID_ARG;
  if (rows && !f->x_scale) return MOE_ERR_INVALID_ARG;
  if (mlp && (!f->w1_scale || !f->w3_scale || !f->w2_scale || !f->x_scale || !f->h_scale))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The router weight [d, E] is read by TMA in the bf16 tensor-core path: 16-byte row pitch.
moe_status_t check_router_width(const moe_config_t* c) {
  return (c->dtype == MOE_BF16 && (c->n_experts % 8)) ? MOE_ERR_ALIGNMENT : MOE_OK;
}

moe_status_t check_ptrs(std::initializer_list<const void*> req,
                        std::initializer_list<const void*> opt) {
  for (const void* p : req) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  for (const void* p : opt)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

moe_status_t check_ws(const moe_config_t& c, const void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((uintptr_t)ws & 255u) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < make_layout(c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int capacity_of(const moe_config_t& c) {
  if (c.capacity_num <= 0) return -1;
  int64_t num = (int64_t)c.capacity_num * c.T * c.top_k;
  int64_t den = (int64_t)c.capacity_den * c.n_experts;
  int64_t C = (num + den - 1) / den;
  return (int)(C > (int64_t)INT32_MAX ? INT32_MAX : C);
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

float round_up_f(double v) {
  float f = (float)v;
  if ((double)f < v) f = nextafterf(f, INFINITY);
  return f;
}

// One call's resolved state.
struct Call {
  moe_config_t c;
  cudaStream_t st;
  bool pdl, tc;
  unsigned char* ws;
  Layout L;
  template <typename P> P* at(size_t off) const { return reinterpret_cast<P*>(ws + off); }
  DeviceHeader* hdr() const { return at<DeviceHeader>(L.hdr); }
};

Call make_call(const moe_config_t* cfg, void* ws, void* stream) {
  Call k;
  k.c = *cfg;
  k.st = static_cast<cudaStream_t>(stream);
  k.pdl = (cfg->flags & MOE_FLAG_PDL) != 0;
  k.tc = cfg->dtype == MOE_BF16 && !(cfg->flags & MOE_FLAG_SIMT);
  k.ws = static_cast<unsigned char*>(ws);
  k.L = make_layout(*cfg);
  return k;
}

// The CUDA error behind the calling thread's last MOE_ERR_CUDA (moe_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = e;
  return MOE_ERR_CUDA;
}

#define MOE_TRY_CUDA(expr)                         \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return cuda_status(e_); \
  } while (0)

cudaError_t run_gemms(const Call& k, GemmProblem* probs, int n) {
  if (n == 0) return cudaSuccess;
  if (k.tc) return gemm_tc(probs, n, k.hdr(), k.st, k.pdl);
  return gemm_simt(probs, n, k.st, k.pdl);   // independent problems, one launch per three
}

moe_status_t check_tc(const Call& k, const GemmProblem* probs, int n) {
  if (!k.tc) return MOE_OK;
  for (int i = 0; i < n; ++i)
    if (!gemm_tc_supported(probs[i])) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

RouterArgs router_args(const Call& k, const void* x, const void* w_router, const float* b,
                       int32_t* idx, float* gate) {
  const moe_config_t& c = k.c;
  RouterArgs a{};
  a.x = x;
  a.w_router = w_router;
  a.bias = b;
  a.logits = k.at<float>(k.L.logits);
  a.wrT = k.at<void>(k.L.wrT);
  a.wnorm = k.at<float>(k.L.wnorm);
  a.xnorm = k.at<float>(k.L.xnorm);
  a.T = c.T;
  a.d = c.d_model;
  a.E = c.n_experts;
  a.k = c.top_k;
  const double u = ldexp(1.0, -24);
  const double gd = c.d_model * u / (1.0 - c.d_model * u);
  a.gam_d = round_up_f(gd);
  if (k.tc) {
    // chunked accumulation: |err| <= (c g_kc + g_nch (1 + c g_kc)) sum|x w| + 2u|l|
    const double kc = 64.0 * ROUTER_KCHUNK;
    const double nch = ceil(c.d_model / kc);
    const double g_kc = kc * u / (1.0 - kc * u), g_n = nch * u / (1.0 - nch * u);
    const double cf = TC_BOUND_FACTOR;
    a.cgam = round_up_f(cf * g_kc + g_n * (1.0 + cf * g_kc));
  } else {
    a.cgam = round_up_f(gd);
  }
  const double n2 = (c.dtype == MOE_F32 ? 2.0 : 1.0) * (c.d_model + 1) + 64.0;
  const double gn = n2 * u / (1.0 - n2 * u);
  a.g2 = round_up_f(gn * gn);
  a.idx = idx;
  a.gate = gate;
  a.refine_list = k.at<int32_t>(k.L.rlist);
  a.exact_list = k.at<int32_t>(k.L.elist);
  a.saved = k.at<unsigned char>(k.L.rsaved);
  a.n_saved = ROUTER_SAVED;
  a.hdr = k.hdr();
  return a;
}

GemmProblem router_problem(const Call& k, const void* x, const void* w_router, const float* b) {
  GemmProblem p;
  p.epi = EPI_F32;
  p.group = GROUP_NONE;
  p.M = k.c.n_experts;
  p.seg[0] = {x, w_router, nullptr, k.c.d_model};
  p.rows = k.c.T;
  p.out = k.at<void>(k.L.logits);
  p.ld_out = k.c.n_experts;
  p.bias = b;
  p.dtype = k.c.dtype;
  p.kchunk = k.tc ? ROUTER_KCHUNK : 0;
  return p;
}

GemmProblem down_problem(const Call& k, const void* x, const void* w_down) {
  GemmProblem p;
  p.epi = EPI_F32;
  p.group = GROUP_NONE;
  p.M = k.c.d_latent;
  p.seg[0] = {x, w_down, nullptr, k.c.d_model};
  p.rows = k.c.T;
  p.out = k.at<void>(k.L.z);
  p.ld_out = k.c.d_latent;
  p.dtype = k.c.dtype;
  return p;
}

GemmProblem shared_problem(const Call& k, const void* x, const void* w1_s, const void* w3_s,
                           void* a_s) {
  GemmProblem p;
  p.epi = EPI_SWIGLU;
  p.group = GROUP_COLS;
  p.M = k.c.n_shared * k.c.d_ff_shared;
  p.Mg = k.c.d_ff_shared;
  p.seg[0] = {x, w1_s, w3_s, k.c.d_model};
  p.rows = k.c.T;
  p.out = a_s;
  p.ld_out = p.M;
  p.dtype = k.c.dtype;
  return p;
}

GemmProblem expert_up_problem(const Call& k, const void* x_perm, const int32_t* offsets,
                              const void* w1, const void* w3, const moe_fp8_t* f8) {
  GemmProblem p;
  if (fp8_experts(k.c)) {        // E4M3 rows and weights in, E4M3 hidden out
    p.w_fp8 = 1;
    p.w_scale = f8->w1_scale;
    p.w3_scale = f8->w3_scale;
    p.act_scale = f8->x_scale;
    p.out_fp8 = 1;
    p.out_scale = f8->h_scale;
    p.amax = &k.hdr()->amax_h;
  }
  p.epi = EPI_SWIGLU;
  p.group = GROUP_ROWS;
  p.M = k.c.d_ff;
  p.seg[0] = {x_perm, w1, w3, k.c.d_latent};
  p.offsets = offsets;
  p.G = k.c.n_experts;
  p.rows = pool_rows_of(k.c);
  p.out = k.at<void>(k.L.hid);
  p.ld_out = k.c.d_ff;
  p.dtype = k.c.dtype;
  return p;
}

GemmProblem expert_down_problem(const Call& k, const int32_t* offsets, const void* w2,
                                void* y_perm, const moe_fp8_t* f8) {
  GemmProblem p;
  if (fp8_experts(k.c)) {        // E4M3 hidden and weights in, bf16 out
    p.w_fp8 = 1;
    p.w_scale = f8->w2_scale;
    p.act_scale = f8->h_scale;
  }
  p.epi = EPI_STORE;
  p.group = GROUP_ROWS;
  p.M = k.c.d_latent;
  p.seg[0] = {k.at<void>(k.L.hid), w2, nullptr, k.c.d_ff};
  p.offsets = offsets;
  p.G = k.c.n_experts;
  p.rows = pool_rows_of(k.c);
  p.out = y_perm;
  p.ld_out = k.c.d_latent;
  p.dtype = k.c.dtype;
  return p;
}

// The back GEMM with the combine inside its launch: the shared experts' segment first, then
// the combine's, whose rows the launch's epilogue warps write into c_buf before they drain any
// accumulator (the tensor cores run the first segment meanwhile).
GemmProblem back_problem_fused(const Call& k, void* c_buf, const void* w_up, const void* a_s,
                               const void* w2_s, void* y, const void* y_perm,
                               const int32_t* slot_of, const float* gate, uint32_t* ready) {
  GemmProblem p;
  p.epi = EPI_STORE;
  p.group = GROUP_NONE;
  p.M = k.c.d_model;
  p.seg[0] = {a_s, w2_s, nullptr, k.c.n_shared * k.c.d_ff_shared};
  p.seg[1] = {c_buf, w_up, nullptr, k.c.d_latent};
  p.n_seg = 2;
  p.rows = k.c.T;
  p.out = y;
  p.ld_out = k.c.d_model;
  p.dtype = k.c.dtype;
  p.cmb_seg = 1;
  p.cmb_y_perm = y_perm;
  p.cmb_slot = slot_of;
  p.cmb_gate = gate;
  p.cmb_k = k.c.top_k;
  p.cmb_pool_rows = pool_rows_of(k.c);
  p.cmb_ready = ready;
  return p;
}

GemmProblem back_problem(const Call& k, const void* c_buf, const void* w_up, const void* a_s,
                         const void* w2_s, void* y) {
  GemmProblem p;
  p.epi = EPI_STORE;
  p.group = GROUP_NONE;
  p.M = k.c.d_model;
  p.seg[0] = {c_buf, w_up, nullptr, k.c.d_latent};
  p.n_seg = 1;
  if (k.c.n_shared > 0 && a_s && w2_s) {
    p.seg[1] = {a_s, w2_s, nullptr, k.c.n_shared * k.c.d_ff_shared};
    p.n_seg = 2;
  }
  p.rows = k.c.T;
  p.out = y;
  p.ld_out = k.c.d_model;
  p.dtype = k.c.dtype;
  return p;
}

DispatchArgs dispatch_args(const Call& k, const int32_t* idx, const uint8_t* mask,
                           const float* gamma,
                           int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* slot_of,
                           int32_t* n_dropped, void* x_perm, const moe_fp8_t* f8) {
  const moe_config_t& c = k.c;
  DispatchArgs a{};
  a.idx = idx;
  a.mask = mask;
  a.T = c.T;
  a.k = c.top_k;
  a.E = c.n_experts;
  a.L = c.d_latent;
  a.cap = capacity_of(c);
  a.n_chunks = dispatch_chunks(c.T);
  a.chunk_hist = k.at<int32_t>(k.L.chist);
  a.chunk_base = k.at<int32_t>(k.L.cbase);
  a.counts = counts;
  a.offsets = offsets;
  a.n_dropped = n_dropped;
  a.slot_of = slot_of;
  a.perm = perm;
  a.pool_rows = pool_rows_of(c);
  a.z = k.at<float>(k.L.z);
  a.gamma = gamma;
  a.eps = c.rms_eps;
  a.x_perm = x_perm;
  a.xperm_fp8 = fp8_experts(c) ? 1 : 0;
  a.x_scale = a.xperm_fp8 ? f8->x_scale : nullptr;
  a.hdr = k.hdr();
  return a;
}

CombineArgs combine_args(const Call& k, const void* y_perm, const int32_t* slot_of,
                         const float* gate, void* out) {
  CombineArgs a{};
  a.y_perm = y_perm;
  a.slot_of = slot_of;
  a.gate = gate;
  a.T = k.c.T;
  a.k = k.c.top_k;
  a.L = k.c.d_latent;
  a.pool_rows = pool_rows_of(k.c);
  a.out = out;
  a.ld_out = k.c.d_latent;
  a.hdr = k.hdr();
  return a;
}

// Stage event i on st. Under stream capture the record becomes an external event node of the
// graph, so that the caller can still synchronize on and time the events of each replay.
void record(const moe_forward_aux_t* aux, int i, cudaStream_t st) {
  if (!aux || !aux->stage_events || !aux->stage_events[i]) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(aux->stage_events[i]), st,
                           cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                               : cudaEventRecordDefault);
}

// ---- routing without caller-allocated scratch -------------------------------------------
// Scratch of moe_route_noalloc: one fixed array per GPU that loads this library, kept until the
// process exits. Its size caps the routing problems that entry point accepts.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_route_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_route_scratch in the current device's context (in host code the array's
// name is only a host-side stand-in). Looked up on every call: the lookup allocates nothing, is
// safe from several host threads at once, and stays right after a context is torn down and
// re-created. On failure returns the CUDA error and leaves *addr NULL.
cudaError_t noalloc_scratch_address(void** addr) {
  *addr = nullptr;
  return cudaGetSymbolAddress(addr, g_route_scratch);
}

// Layout of the routing scratch inside the fixed array (the same regions moe_route uses).
struct NoallocLayout {
  size_t hdr, logits, wrT, wnorm, xnorm, rlist, elist, rsaved, total;
};
NoallocLayout noalloc_layout(const moe_config_t& c) {
  NoallocLayout L{};
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    size_t o = off;
    off = al256(off + (size_t)bytes);
    return o;
  };
  const int64_t es = (c.dtype == MOE_BF16) ? 2 : 4;
  L.hdr = take(sizeof(DeviceHeader));
  L.logits = take(c.T * c.n_experts * 4);
  L.wrT = take((int64_t)c.n_experts * c.d_model * es);
  L.wnorm = take((int64_t)c.n_experts * 4);
  L.xnorm = take(c.T * 4);
  L.rlist = take(c.T * 4);
  L.elist = take(c.T * 4);
  L.rsaved = take((int64_t)router_saved_bytes(c.n_experts, ROUTER_SAVED));
  L.total = off;
  return L;
}

__global__ void noalloc_report_kernel(const DeviceHeader* h, int32_t* out) {
  if (threadIdx.x == 0) {
    out[0] = h->status;
    out[1] = h->detail;
    out[2] = h->n_refine;
    out[3] = h->n_exact;
  }
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer or width";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_ROUTING: return "bad routing data on the device";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int32_t moe_last_cuda_error(const char** name) {
  if (name) *name = cudaGetErrorName(g_last_cuda_error);
  return (int32_t)g_last_cuda_error;
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_workspace_regions(const moe_config_t* cfg, moe_workspace_regions_t* out) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!out) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*cfg);
  out->z = L.z;
  out->x_perm = L.x_perm;
  out->hidden = L.hid;
  out->y_perm = L.y_perm;
  out->a_shared = L.a_s;
  out->combined = L.c;
  out->perm = L.perm;
  out->expert_offsets = L.offsets;
  return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* b_router, int32_t* topk_idx, float* topk_gate, void* ws,
                       size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_router_width(cfg)) != MOE_OK) return s;
  if ((s = check_ptrs({x, w_router, topk_idx, topk_gate}, {b_router})) != MOE_OK) return s;
  if ((s = check_ws(*cfg, ws, ws_bytes)) != MOE_OK) return s;
  Call k = make_call(cfg, ws, stream);
  GemmProblem p = router_problem(k, x, w_router, b_router);
  if ((s = check_tc(k, &p, 1)) != MOE_OK) return s;
  RouterArgs ra = router_args(k, x, w_router, b_router, topk_idx, topk_gate);
  MOE_TRY_CUDA(header_reset(k.hdr(), false, k.st, false));
  MOE_TRY_CUDA(router_prepare(ra, cfg->dtype, k.st, k.pdl));
  MOE_TRY_CUDA(run_gemms(k, &p, 1));
  MOE_TRY_CUDA(router_select(ra, cfg->dtype, num_sms(), k.st, k.pdl));
  return MOE_OK;
}

// Copies an amax the kernels max-reduced into the workspace header to the caller's buffer.
cudaError_t copy_amax(float* dst, const uint32_t* src, cudaStream_t st) {
  if (!dst) return cudaSuccess;
  return cudaMemcpyAsync(dst, src, sizeof(float), cudaMemcpyDeviceToDevice, st);
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const void* w_down,
                         const float* rms_gamma, const int32_t* topk_idx,
                         const uint8_t* token_mask, int32_t* expert_counts,
                         int32_t* expert_offsets, int32_t* perm, int32_t* slot_of,
                         int32_t* n_dropped, void* x_perm, const moe_fp8_t* fp8, void* ws,
                         size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_ptrs({x, w_down, rms_gamma, topk_idx, expert_counts, expert_offsets, perm,
                       slot_of, x_perm},
                      {n_dropped})) != MOE_OK)
    return s;
  if ((s = check_fp8(*cfg, fp8, true, false)) != MOE_OK) return s;
  if ((s = check_ws(*cfg, ws, ws_bytes)) != MOE_OK) return s;
  Call k = make_call(cfg, ws, stream);
  const bool f8 = fp8_experts(*cfg);
  GemmProblem p = down_problem(k, x, w_down);
  if ((s = check_tc(k, &p, 1)) != MOE_OK) return s;
  if (f8) MOE_TRY_CUDA(header_reset(k.hdr(), false, k.st, false, 1));
  MOE_TRY_CUDA(run_gemms(k, &p, 1));
  DispatchArgs da = dispatch_args(k, topk_idx, token_mask, rms_gamma, expert_counts,
                                  expert_offsets, perm, slot_of, n_dropped, x_perm, fp8);
  MOE_TRY_CUDA(dispatch_run(da, cfg->dtype, k.st, k.pdl));
  if (f8) MOE_TRY_CUDA(copy_amax(fp8->x_amax, &k.hdr()->amax_x, k.st));
  return MOE_OK;
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_perm,
                            const int32_t* expert_offsets, const void* w1, const void* w3,
                            const void* w2, const moe_fp8_t* fp8, void* y_perm, const void* x,
                            const void* w1_s, const void* w3_s, void* a_shared, void* ws,
                            size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_ptrs({x_perm, expert_offsets, w1, w3, w2, y_perm},
                      {x, w1_s, w3_s, a_shared})) != MOE_OK)
    return s;
  if ((s = check_fp8(*cfg, fp8, true, true)) != MOE_OK) return s;
  const bool shared = x && cfg->n_shared > 0;
  if (shared && (!w1_s || !w3_s || !a_shared)) return MOE_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes)) != MOE_OK) return s;
  Call k = make_call(cfg, ws, stream);
  const bool f8 = fp8_experts(*cfg);
  GemmProblem up = expert_up_problem(k, x_perm, expert_offsets, w1, w3, fp8);
  GemmProblem sh;
  if (shared) sh = shared_problem(k, x, w1_s, w3_s, a_shared);
  GemmProblem down = expert_down_problem(k, expert_offsets, w2, y_perm, fp8);
  if ((s = check_tc(k, &up, 1)) != MOE_OK) return s;
  if (shared && (s = check_tc(k, &sh, 1)) != MOE_OK) return s;
  if ((s = check_tc(k, &down, 1)) != MOE_OK) return s;
  if (f8) MOE_TRY_CUDA(header_reset(k.hdr(), false, k.st, false, 2));
  MOE_TRY_CUDA(validate_offsets(expert_offsets, cfg->n_experts, pool_rows_of(*cfg), k.hdr(), k.st,
                                false));
  if (shared && !f8) {
    GemmProblem both[2] = {up, sh};          // one launch: the grouped and the shared GEMM
    MOE_TRY_CUDA(run_gemms(k, both, 2));
  } else {                                   // an fp8 launch holds fp8 problems only
    MOE_TRY_CUDA(run_gemms(k, &up, 1));
    if (shared) MOE_TRY_CUDA(run_gemms(k, &sh, 1));
  }
  MOE_TRY_CUDA(run_gemms(k, &down, 1));
  if (f8) MOE_TRY_CUDA(copy_amax(fp8->h_amax, &k.hdr()->amax_h, k.st));
  return MOE_OK;
}

moe_status_t moe_backward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_bwd_layout(*cfg).total;
  return MOE_OK;
}

// The routed experts' backward on the grouped rows: recompute G, U, A; dA with the SwiGLU
// backward; dX; the weight gradients. Scratch buffers G, U, A, dG, dU ([pool_rows, F] bf16).
struct ExpertBwdScratch {
  void *g, *u, *a, *dg, *du;
};

moe_status_t expert_backward_launches(const Call& k, const void* x_perm, const int32_t* offsets,
                                      const void* w1, const void* w3, const void* w2,
                                      const void* dy_perm, void* dx_perm, void* dw1, void* dw3,
                                      void* dw2, const ExpertBwdScratch& B) {
  const moe_config_t& c = k.c;
  const int64_t P = pool_rows_of(c);
  const int E = c.n_experts, L = c.d_latent, F = c.d_ff;
  // 1. recompute G, U and A = silu(G) U over the grouped rows
  GemmProblem rec;
  rec.epi = EPI_SWIGLU_SAVE;
  rec.group = GROUP_ROWS;
  rec.M = F;
  rec.seg[0] = {x_perm, w1, w3, L};
  rec.offsets = offsets;
  rec.G = E;
  rec.rows = P;
  rec.out = B.a;
  rec.out2 = B.g;
  rec.out3 = B.u;
  rec.ld_out = F;
  rec.dtype = DT_BF16;
  // 2. dA = dY W2^T, then dG = dA U silu'(G), dU = dA silu(G) in the epilogue
  GemmProblem da;
  da.epi = EPI_SWIGLU_BWD;
  da.group = GROUP_ROWS;
  da.M = F;
  da.seg[0] = {dy_perm, w2, nullptr, L};
  da.a_kmajor = 1;
  da.offsets = offsets;
  da.G = E;
  da.rows = P;
  da.out = B.dg;
  da.out2 = B.du;
  da.ld_out = F;
  da.aux_g = B.g;
  da.aux_u = B.u;
  da.ld_aux = F;
  da.dtype = DT_BF16;
  // 3. dX = dG W1^T + dU W3^T
  GemmProblem dx;
  dx.epi = EPI_STORE;
  dx.group = GROUP_ROWS;
  dx.M = L;
  dx.n_seg = 2;
  dx.seg[0] = {B.dg, w1, nullptr, F};
  dx.seg[1] = {B.du, w3, nullptr, F};
  dx.a_kmajor = 1;
  dx.offsets = offsets;
  dx.G = E;
  dx.rows = P;
  dx.out = dx_perm;
  dx.ld_out = L;
  dx.dtype = DT_BF16;
  // 4. dW2 = A^T dY; dW1 = X^T dG, dW3 = X^T dU, contracting over each expert's rows
  WgradProblem w2g;
  w2g.a = B.a;
  w2g.b = dy_perm;
  w2g.offsets = offsets;
  w2g.G = E;
  w2g.M = F;
  w2g.N = L;
  w2g.rows = P;
  w2g.out = dw2;
  WgradProblem w13[2];
  w13[0].a = x_perm;
  w13[0].b = B.dg;
  w13[0].offsets = offsets;
  w13[0].G = E;
  w13[0].M = L;
  w13[0].N = F;
  w13[0].rows = P;
  w13[0].out = dw1;
  w13[1] = w13[0];
  w13[1].b = B.du;
  w13[1].out = dw3;
  if (!gemm_tc_supported(rec) || !gemm_tc_supported(da) || !gemm_tc_supported(dx) ||
      !gemm_wgrad_supported(w2g) || !gemm_wgrad_supported(w13[0]))
    return MOE_ERR_UNSUPPORTED;
  MOE_TRY_CUDA(validate_offsets(offsets, E, P, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_tc(&rec, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_tc(&da, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_tc(&dx, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_wgrad(&w2g, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_wgrad(w13, 2, k.hdr(), k.st, k.pdl));
  return MOE_OK;
}

// Conditions of the tensor-core backward: bf16, no fp8 experts, widths the tiles divide.
moe_status_t check_backward_cfg(const moe_config_t& c) {
  if (c.dtype != MOE_BF16 || (c.flags & (MOE_FLAG_SIMT | MOE_FLAG_FP8_EXPERTS)))
    return MOE_ERR_UNSUPPORTED;
  if ((c.d_latent % 128) || (c.d_ff % 128)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

moe_status_t moe_expert_ffn_backward(const moe_config_t* cfg, const void* x_perm,
                                     const int32_t* expert_offsets, const void* w1,
                                     const void* w3, const void* w2, const void* dy_perm,
                                     void* dx_perm, void* dw1, void* dw3, void* dw2, void* ws,
                                     size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_ptrs({x_perm, expert_offsets, w1, w3, w2, dy_perm, dx_perm, dw1, dw3, dw2},
                      {})) != MOE_OK)
    return s;
  if ((s = check_backward_cfg(*cfg)) != MOE_OK) return s;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((uintptr_t)ws & 255u) return MOE_ERR_ALIGNMENT;
  const BwdLayout B = make_bwd_layout(*cfg);
  if (ws_bytes < B.total) return MOE_ERR_WORKSPACE;
  Call k = make_call(cfg, ws, stream);
  k.L.hdr = B.hdr;                                   // the report sits at the same place
  auto at = [&](size_t off) { return static_cast<void*>(k.ws + off); };
  MOE_TRY_CUDA(header_reset(k.hdr(), false, k.st, false));
  return expert_backward_launches(k, x_perm, expert_offsets, w1, w3, w2, dy_perm, dx_perm, dw1,
                                  dw3, dw2, {at(B.g), at(B.u), at(B.a), at(B.dg), at(B.du)});
}

// Workspace of moe_backward: the experts' backward scratch, then the rest of the layer's
// intermediates (sizes from the configuration).
struct LayerBwdLayout {
  BwdLayout e;
  size_t dc, gs, us, as2, dgs, dus, dy_perm, dgate, dx_perm, dz, dhz, dx32, dl32, dlbf, off01,
      colsum, total;
};

LayerBwdLayout make_layer_bwd_layout(const moe_config_t& c) {
  LayerBwdLayout L{};
  L.e = make_bwd_layout(c);
  size_t off = L.e.total;
  auto take = [&](int64_t bytes) {
    size_t o = off;
    off = al256(off + (size_t)bytes);
    return o;
  };
  const int64_t T = c.T, k = c.top_k, d = c.d_model, Lt = c.d_latent, E = c.n_experts,
                SF = (int64_t)c.n_shared * c.d_ff_shared, P = pool_rows_of(c);
  const int64_t sf = SF > 0 ? SF : 1;
  L.dc = take(T * Lt * 2);
  L.gs = take(T * sf * 2);
  L.us = take(T * sf * 2);
  L.as2 = take(T * sf * 2);
  L.dgs = take(T * sf * 2);
  L.dus = take(T * sf * 2);
  L.dy_perm = take(P * Lt * 2);
  L.dgate = take(T * k * 4);
  L.dx_perm = take(P * Lt * 2);
  L.dz = take(T * Lt * 2);
  L.dhz = take(T * Lt * 4);
  L.dx32 = take(T * d * 4);
  L.dl32 = take(T * E * 4);
  L.dlbf = take(T * E * 2);
  L.off01 = take(2 * 4);
  L.colsum = take((int64_t)COLSUM_CHUNKS * (Lt > E ? Lt : E) * 4);
  L.total = off;
  return L;
}

moe_status_t moe_layer_backward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layer_bwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                          const void* dy, void* dx, const moe_grads_t* g, const void* fwd_ws,
                          size_t fwd_ws_bytes, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!w || !g) return MOE_ERR_INVALID_ARG;
  if ((s = check_ptrs({x, dy, dx, w->w_router, w->w_down, w->rms_gamma, w->w1, w->w3, w->w2,
                       w->w_up, g->dw_router, g->dw_down, g->dw1, g->dw3, g->dw2, g->dw_up},
                      {g->db_router, g->drms_gamma})) != MOE_OK)
    return s;
  const int S = cfg->n_shared, Fs = cfg->d_ff_shared;
  if (S > 0 && (s = check_ptrs({w->w1_s, w->w3_s, w->w2_s, g->dw1_s, g->dw3_s, g->dw2_s}, {})) !=
                   MOE_OK)
    return s;
  if ((s = check_backward_cfg(*cfg)) != MOE_OK) return s;
  const int64_t T = cfg->T, P = pool_rows_of(*cfg), SF = (int64_t)S * Fs;
  const int d = cfg->d_model, L = cfg->d_latent, E = cfg->n_experts, kk = cfg->top_k;
  // tile divisibility of the dense gradients (output rows of 128, columns of 64) and at most
  // two shared experts (the input gradient's GEMM sums at most six K segments)
  if ((d % 128) || (E % 64) || (S > 0 && ((SF % 128) || (Fs % 64))) || S > 2)
    return MOE_ERR_UNSUPPORTED;
  if (!fwd_ws || fwd_ws_bytes < make_layout(*cfg).total) return MOE_ERR_WORKSPACE;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 255u) || ((uintptr_t)fwd_ws & 255u)) return MOE_ERR_ALIGNMENT;
  const LayerBwdLayout B = make_layer_bwd_layout(*cfg);
  if (ws_bytes < B.total) return MOE_ERR_WORKSPACE;
  Call k = make_call(cfg, ws, stream);
  k.L.hdr = B.e.hdr;
  auto at = [&](size_t off) { return static_cast<void*>(k.ws + off); };
  const Layout FL = make_layout(*cfg);
  const unsigned char* fw = static_cast<const unsigned char*>(fwd_ws);
  auto fat = [&](size_t off) { return static_cast<const void*>(fw + off); };
  const int32_t* idx = static_cast<const int32_t*>(fat(FL.idx));
  const float* gate = static_cast<const float*>(fat(FL.gate));
  const int32_t* slot_of = static_cast<const int32_t*>(fat(FL.slot_of));
  const int32_t* offsets = static_cast<const int32_t*>(fat(FL.offsets));
  int32_t* off01 = static_cast<int32_t*>(at(B.off01));

  // 1. the shared experts' pre-activations (recomputed)
  GemmProblem shr;
  if (S > 0) {
    shr = shared_problem(k, x, w->w1_s, w->w3_s, at(B.as2));
    shr.epi = EPI_SWIGLU_SAVE;
    shr.out2 = at(B.gs);
    shr.out3 = at(B.us);
  }
  // 2. dc = dy W_up^T and the shared experts' dA = dy W2s^T with their SwiGLU backward, in two
  // launches: dc's 256-feature items fill tensor memory with one accumulator buffer, and in a
  // shared launch the SwiGLU-backward items would lose the second buffer that hides their
  // epilogue's loads of G and U behind the next item's main loop
  GemmProblem d1[2];
  d1[0].epi = EPI_STORE;
  d1[0].M = L;
  d1[0].seg[0] = {dy, w->w_up, nullptr, d};
  d1[0].a_kmajor = 1;
  d1[0].rows = T;
  d1[0].out = at(B.dc);
  d1[0].ld_out = L;
  d1[0].dtype = DT_BF16;
  if (S > 0) {
    d1[1].epi = EPI_SWIGLU_BWD;
    d1[1].M = (int)SF;
    d1[1].seg[0] = {dy, w->w2_s, nullptr, d};
    d1[1].a_kmajor = 1;
    d1[1].rows = T;
    d1[1].out = at(B.dgs);
    d1[1].out2 = at(B.dus);
    d1[1].ld_out = SF;
    d1[1].aux_g = at(B.gs);
    d1[1].aux_u = at(B.us);
    d1[1].ld_aux = SF;
    d1[1].dtype = DT_BF16;
  }
  // 3. dW_up = c^T dy and dW2s = a_s^T dy (one group of T rows)
  WgradProblem w1g[2];
  w1g[0].a = fat(FL.c);
  w1g[0].b = dy;
  w1g[0].offsets = off01;
  w1g[0].M = L;
  w1g[0].N = d;
  w1g[0].rows = T;
  w1g[0].out = g->dw_up;
  if (S > 0) {
    w1g[1] = w1g[0];
    w1g[1].a = fat(FL.a_s);
    w1g[1].M = (int)SF;
    w1g[1].out = g->dw2_s;
  }
  // 8. dx32 = dz W_down^T + sum_s dG_s W1_s[s]^T + dU_s W3_s[s]^T
  GemmProblem dxp;
  dxp.epi = EPI_F32;
  dxp.M = d;
  dxp.seg[0] = {at(B.dz), w->w_down, nullptr, L};
  dxp.n_seg = 1;
  for (int e = 0; e < S; ++e) {
    const int64_t wo = (int64_t)e * d * Fs * 2;      // bytes to shared expert e's [d, F_s]
    GemmSeg g1, g3;
    g1.act = static_cast<const unsigned char*>(at(B.dgs)) + (int64_t)e * Fs * 2;
    g1.w = static_cast<const unsigned char*>(w->w1_s) + wo;
    g1.w3 = nullptr;
    g1.K = Fs;
    g1.ld = SF;
    g3 = g1;
    g3.act = static_cast<const unsigned char*>(at(B.dus)) + (int64_t)e * Fs * 2;
    g3.w = static_cast<const unsigned char*>(w->w3_s) + wo;
    dxp.seg[dxp.n_seg++] = g1;
    dxp.seg[dxp.n_seg++] = g3;
  }
  dxp.a_kmajor = 1;
  dxp.rows = T;
  dxp.out = at(B.dx32);
  dxp.ld_out = d;
  dxp.dtype = DT_BF16;
  // 11. dW_down = x^T dz; dW1_s[s] = x^T dG_s, dW3_s[s] = x^T dU_s; dW_r = x^T dl
  WgradProblem w2g[6];
  int n_w2 = 0;
  WgradProblem base;
  base.a = x;
  base.offsets = off01;
  base.M = d;
  base.rows = T;
  w2g[n_w2] = base;
  w2g[n_w2].b = at(B.dz);
  w2g[n_w2].N = L;
  w2g[n_w2++].out = g->dw_down;
  for (int e = 0; e < S; ++e) {
    const int64_t wo = (int64_t)e * d * Fs * 2;
    w2g[n_w2] = base;
    w2g[n_w2].b = static_cast<const unsigned char*>(at(B.dgs)) + (int64_t)e * Fs * 2;
    w2g[n_w2].ldb = SF;
    w2g[n_w2].N = Fs;
    w2g[n_w2++].out = static_cast<unsigned char*>(g->dw1_s) + wo;
    w2g[n_w2] = w2g[n_w2 - 1];
    w2g[n_w2].b = static_cast<const unsigned char*>(at(B.dus)) + (int64_t)e * Fs * 2;
    w2g[n_w2++].out = static_cast<unsigned char*>(g->dw3_s) + wo;
  }
  w2g[n_w2] = base;
  w2g[n_w2].b = at(B.dlbf);
  w2g[n_w2].N = E;
  w2g[n_w2++].out = g->dw_router;

  if ((S > 0 && !gemm_tc_supported(shr)) || !gemm_tc_supported(d1[0]) ||
      (S > 0 && !gemm_tc_supported(d1[1])) || !gemm_tc_supported(dxp))
    return MOE_ERR_UNSUPPORTED;
  for (int i = 0; i < (S > 0 ? 2 : 1); ++i)
    if (!gemm_wgrad_supported(w1g[i])) return MOE_ERR_UNSUPPORTED;
  for (int i = 0; i < n_w2; ++i)
    if (!gemm_wgrad_supported(w2g[i])) return MOE_ERR_UNSUPPORTED;

  MOE_TRY_CUDA(header_reset(k.hdr(), false, k.st, false));
  MOE_TRY_CUDA(write_int2(off01, 0, (int32_t)T, k.st, k.pdl));
  if (S > 0) MOE_TRY_CUDA(gemm_tc(&shr, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_tc(&d1[0], 1, k.hdr(), k.st, k.pdl));
  if (S > 0) MOE_TRY_CUDA(gemm_tc(&d1[1], 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(gemm_wgrad(w1g, S > 0 ? 2 : 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(combine_backward(at(B.dc), fat(FL.y_perm), slot_of, gate, T, kk, L, P,
                                at(B.dy_perm), static_cast<float*>(at(B.dgate)), k.st, k.pdl));
  moe_status_t es = expert_backward_launches(
      k, fat(FL.x_perm), offsets, w->w1, w->w3, w->w2, at(B.dy_perm), at(B.dx_perm), g->dw1,
      g->dw3, g->dw2, {at(B.e.g), at(B.e.u), at(B.e.a), at(B.e.dg), at(B.e.du)});
  if (es != MOE_OK) return es;
  MOE_TRY_CUDA(rms_backward(at(B.dx_perm), slot_of, static_cast<const float*>(fat(FL.z)),
                            w->rms_gamma, cfg->rms_eps, T, kk, L, P, at(B.dz),
                            static_cast<float*>(at(B.dhz)), k.st, k.pdl));
  if (g->drms_gamma)
    MOE_TRY_CUDA(column_sum(static_cast<const float*>(at(B.dhz)), T, L,
                            static_cast<float*>(at(B.colsum)), g->drms_gamma, k.st, k.pdl));
  MOE_TRY_CUDA(gemm_tc(&dxp, 1, k.hdr(), k.st, k.pdl));
  MOE_TRY_CUDA(router_backward(idx, gate, static_cast<const float*>(at(B.dgate)), fat(FL.wrT),
                               static_cast<const float*>(at(B.dx32)), T, kk, E, d, dx,
                               static_cast<float*>(at(B.dl32)), at(B.dlbf), k.st, k.pdl));
  if (g->db_router)
    MOE_TRY_CUDA(column_sum(static_cast<const float*>(at(B.dl32)), T, E,
                            static_cast<float*>(at(B.colsum)), g->db_router, k.st, k.pdl));
  MOE_TRY_CUDA(gemm_wgrad(w2g, n_w2, k.hdr(), k.st, k.pdl));
  return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* slot_of,
                         const float* topk_gate, const void* a_shared, const void* w_up,
                         const void* w2_s, void* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_ptrs({y_perm, slot_of, topk_gate, out}, {a_shared, w_up, w2_s})) != MOE_OK)
    return s;
  if ((s = check_ws(*cfg, ws, ws_bytes)) != MOE_OK) return s;
  Call k = make_call(cfg, ws, stream);
  if (!w_up) {
    CombineArgs ca = combine_args(k, y_perm, slot_of, topk_gate, out);
    MOE_TRY_CUDA(combine_run(ca, cfg->dtype, k.st, k.pdl));
    return MOE_OK;
  }
  if (cfg->n_shared > 0 && (!a_shared || !w2_s)) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && k.tc && fused_combine_enabled(*cfg)) {
    // the combine inside the up-projection's launch
    uint32_t* ready = k.at<uint32_t>(k.L.cready);
    GemmProblem p = back_problem_fused(k, k.at<void>(k.L.c), w_up, a_shared, w2_s, out, y_perm,
                                       slot_of, topk_gate, ready);
    if ((s = check_tc(k, &p, 1)) != MOE_OK) return s;
    MOE_TRY_CUDA(cudaMemsetAsync(ready, 0, (size_t)ready_tiles(cfg->T) * 4, k.st));
    MOE_TRY_CUDA(run_gemms(k, &p, 1));
    return MOE_OK;
  }
  GemmProblem p = back_problem(k, k.at<void>(k.L.c), w_up, a_shared, w2_s, out);
  if ((s = check_tc(k, &p, 1)) != MOE_OK) return s;
  CombineArgs ca = combine_args(k, y_perm, slot_of, topk_gate, k.at<void>(k.L.c));
  MOE_TRY_CUDA(combine_run(ca, cfg->dtype, k.st, k.pdl));
  MOE_TRY_CUDA(run_gemms(k, &p, 1));
  return MOE_OK;
}

moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, void* y,
                         void* ws, size_t ws_bytes, void* stream, const moe_forward_aux_t* aux) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!w) return MOE_ERR_INVALID_ARG;
  if ((s = check_router_width(cfg)) != MOE_OK) return s;
  if ((s = check_ptrs({x, y, w->w_router, w->w_down, w->rms_gamma, w->w1, w->w3, w->w2, w->w_up},
                      {w->b_router})) != MOE_OK)
    return s;
  if ((s = check_fp8(*cfg, w->fp8, true, true)) != MOE_OK) return s;
  if (cfg->n_shared > 0 && (s = check_ptrs({w->w1_s, w->w3_s, w->w2_s}, {})) != MOE_OK) return s;
  if (cfg->pool_rows != 0 && cfg->pool_rows < cfg->T * (int64_t)cfg->top_k)
    return MOE_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes)) != MOE_OK) return s;
  if (aux) {
    if ((s = check_ptrs({}, {aux->topk_idx, aux->topk_gate, aux->expert_counts,
                             aux->expert_offsets, aux->slot_of, aux->n_dropped})) != MOE_OK)
      return s;
  }
  Call k = make_call(cfg, ws, stream);
  const Layout& L = k.L;
  const bool shared = cfg->n_shared > 0;
  void* a_s = k.at<void>(L.a_s);
  int32_t* idx = k.at<int32_t>(L.idx);
  float* gate = k.at<float>(L.gate);
  int32_t* offsets = k.at<int32_t>(L.offsets);
  int32_t* slot_of = k.at<int32_t>(L.slot_of);

  GemmProblem front[3] = {router_problem(k, x, w->w_router, w->b_router),
                          down_problem(k, x, w->w_down)};
  int n_front = 2;
  if (shared) front[n_front++] = shared_problem(k, x, w->w1_s, w->w3_s, a_s);
  GemmProblem up = expert_up_problem(k, k.at<void>(L.x_perm), offsets, w->w1, w->w3, w->fp8);
  GemmProblem down = expert_down_problem(k, offsets, w->w2, k.at<void>(L.y_perm), w->fp8);
  // the combine inside the back GEMM's launch (tensor-core layers with shared experts)
  const bool fuse = shared && k.tc && fused_combine_enabled(*cfg);
  uint32_t* ready = k.at<uint32_t>(L.cready);
  GemmProblem back = fuse ? back_problem_fused(k, k.at<void>(L.c), w->w_up, a_s, w->w2_s, y,
                                               k.at<void>(L.y_perm), slot_of, gate, ready)
                          : back_problem(k, k.at<void>(L.c), w->w_up, shared ? a_s : nullptr,
                                         shared ? w->w2_s : nullptr, y);
  if ((s = check_tc(k, front, n_front)) != MOE_OK) return s;
  if ((s = check_tc(k, &up, 1)) != MOE_OK) return s;
  if ((s = check_tc(k, &down, 1)) != MOE_OK) return s;
  if ((s = check_tc(k, &back, 1)) != MOE_OK) return s;

  RouterArgs ra = router_args(k, x, w->w_router, w->b_router, idx, gate);
  DispatchArgs da = dispatch_args(k, idx, aux ? aux->token_mask : nullptr, w->rms_gamma,
                                  k.at<int32_t>(L.counts), offsets,
                                  k.at<int32_t>(L.perm), slot_of, k.at<int32_t>(L.ndrop),
                                  k.at<void>(L.x_perm), w->fp8);
  CombineArgs ca = combine_args(k, k.at<void>(L.y_perm), slot_of, gate, k.at<void>(L.c));

  record(aux, 0, k.st);
  const bool f8 = fp8_experts(*cfg);
  MOE_TRY_CUDA(header_reset(k.hdr(), true, k.st, false, f8 ? 3 : 0, fuse ? ready : nullptr,
                            fuse ? (int)ready_tiles(cfg->T) : 0));
  MOE_TRY_CUDA(router_prepare(ra, cfg->dtype, k.st, k.pdl));
  record(aux, 1, k.st);
  // The router's k-chunked fp32 problem runs on single CTAs. When the down-projection and the
  // shared experts can run as CTA pairs, they get a launch of their own.
  if (k.tc && front_split_enabled(*cfg) && gemm_tc_pairs(front + 1, n_front - 1)) {
    MOE_TRY_CUDA(run_gemms(k, front, 1));
    MOE_TRY_CUDA(run_gemms(k, front + 1, n_front - 1));
  } else {
    MOE_TRY_CUDA(run_gemms(k, front, n_front));
  }
  record(aux, 2, k.st);
  MOE_TRY_CUDA(router_select(ra, cfg->dtype, num_sms(), k.st, k.pdl));
  record(aux, 3, k.st);
  MOE_TRY_CUDA(dispatch_run(da, cfg->dtype, k.st, k.pdl));
  record(aux, 4, k.st);
  MOE_TRY_CUDA(run_gemms(k, &up, 1));
  record(aux, 5, k.st);
  MOE_TRY_CUDA(run_gemms(k, &down, 1));
  record(aux, 6, k.st);
  if (!fuse) MOE_TRY_CUDA(combine_run(ca, cfg->dtype, k.st, k.pdl));
  record(aux, 7, k.st);
  MOE_TRY_CUDA(run_gemms(k, &back, 1));
  record(aux, 8, k.st);

  if (aux) {
    const int64_t Tk = cfg->T * (int64_t)cfg->top_k;
    auto cp = [&](void* dst, size_t off, size_t bytes) -> cudaError_t {
      if (!dst) return cudaSuccess;
      return cudaMemcpyAsync(dst, k.ws + off, bytes, cudaMemcpyDeviceToDevice, k.st);
    };
    MOE_TRY_CUDA(cp(aux->topk_idx, L.idx, Tk * 4));
    MOE_TRY_CUDA(cp(aux->topk_gate, L.gate, Tk * 4));
    MOE_TRY_CUDA(cp(aux->expert_counts, L.counts, (size_t)cfg->n_experts * 4));
    MOE_TRY_CUDA(cp(aux->expert_offsets, L.offsets, ((size_t)cfg->n_experts + 1) * 4));
    MOE_TRY_CUDA(cp(aux->slot_of, L.slot_of, Tk * 4));
    MOE_TRY_CUDA(cp(aux->n_dropped, L.ndrop, 4));
  }
  if (f8) {
    MOE_TRY_CUDA(copy_amax(w->fp8->x_amax, &k.hdr()->amax_x, k.st));
    MOE_TRY_CUDA(copy_amax(w->fp8->h_amax, &k.hdr()->amax_h, k.st));
  }
  return MOE_OK;
}

moe_status_t moe_forward_pipelined(const moe_config_t* cfg, const moe_weights_t* w,
                                   int32_t n_batches, const void* const* x_host,
                                   void* const* y_host, void* x_stage, void* y_stage, void* ws,
                                   size_t ws_bytes, void* stream, void* h2d_stream,
                                   void* d2h_stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (n_batches < 1 || !x_host || !y_host || !w) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_batches; ++i)
    if (!x_host[i] || !y_host[i]) return MOE_ERR_INVALID_ARG;
  if ((s = check_ptrs({x_stage, y_stage}, {})) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t up = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t dn = static_cast<cudaStream_t>(d2h_stream);
  if (up == st || dn == st || up == dn) return MOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)cfg->T * cfg->d_model * (cfg->dtype == MOE_BF16 ? 2 : 4);
  unsigned char* xs = static_cast<unsigned char*>(x_stage);
  unsigned char* ys = static_cast<unsigned char*>(y_stage);
  // events: input copied in, forward done, output copied out (per batch)
  const int n = n_batches;
  cudaEvent_t* ev = new cudaEvent_t[3 * (size_t)n]();
  auto cleanup = [&]() {
    for (int i = 0; i < 3 * n; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);   // released once the recorded work completes
    delete[] ev;
  };
  for (int i = 0; i < 3 * n; ++i)
    if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
      ev[i] = nullptr;
      cleanup();
      return MOE_ERR_CUDA;
    }
  cudaEvent_t* in = ev;
  cudaEvent_t* done = ev + n;
  cudaEvent_t* out = ev + 2 * n;
  moe_status_t rs = MOE_OK;
  for (int i = 0; i < n && rs == MOE_OK; ++i) {
    const size_t o = (size_t)(i & 1) * bytes;
    auto step = [&]() -> moe_status_t {
      // batch i's input into staging slot i % 2, once batch i - 2's forward has read it
      if (i >= 2) MOE_TRY_CUDA(cudaStreamWaitEvent(up, done[i - 2], 0));
      MOE_TRY_CUDA(cudaMemcpyAsync(xs + o, x_host[i], bytes, cudaMemcpyHostToDevice, up));
      MOE_TRY_CUDA(cudaEventRecord(in[i], up));
      // the forward, once its input has landed and batch i - 2's output has been copied out
      MOE_TRY_CUDA(cudaStreamWaitEvent(st, in[i], 0));
      if (i >= 2) MOE_TRY_CUDA(cudaStreamWaitEvent(st, out[i - 2], 0));
      moe_status_t f = moe_forward(cfg, w, xs + o, ys + o, ws, ws_bytes, stream, nullptr);
      if (f != MOE_OK) return f;
      MOE_TRY_CUDA(cudaEventRecord(done[i], st));
      // batch i's output back to the host
      MOE_TRY_CUDA(cudaStreamWaitEvent(dn, done[i], 0));
      MOE_TRY_CUDA(cudaMemcpyAsync(y_host[i], ys + o, bytes, cudaMemcpyDeviceToHost, dn));
      MOE_TRY_CUDA(cudaEventRecord(out[i], dn));
      return MOE_OK;
    };
    rs = step();
  }
  // the caller's stream completes after the last output copy
  if (rs == MOE_OK && cudaStreamWaitEvent(st, out[n - 1], 0) != cudaSuccess) rs = MOE_ERR_CUDA;
  cleanup();
  return rs;
}

moe_status_t moe_get_device_status(const void* ws, size_t ws_bytes, void* stream,
                                   moe_device_report_t* out) {
  if (!ws || !out || ws_bytes < sizeof(DeviceHeader)) return MOE_ERR_INVALID_ARG;
  DeviceHeader h;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY_CUDA(cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st));
  MOE_TRY_CUDA(cudaStreamSynchronize(st));
  out->status = h.status;
  out->detail = h.detail;
  out->n_refined = h.n_refine;
  out->n_exact = h.n_exact;
  return MOE_OK;
}

moe_status_t moe_selftest_device_timeout(void* ws, size_t ws_bytes, uint32_t limit_ms,
                                         void* stream) {
  if (!ws || ws_bytes < sizeof(DeviceHeader)) return MOE_ERR_INVALID_ARG;
  if ((uintptr_t)ws & 255u) return MOE_ERR_ALIGNMENT;
  if (limit_ms < 1 || limit_ms > 10000) return MOE_ERR_INVALID_ARG;
  return cuda_status(bounded_wait_selftest(ws, (uint64_t)limit_ms * 1000000ull,
                                           static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_clear_device_status(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(DeviceHeader)) return MOE_ERR_INVALID_ARG;
  return cuda_status(header_reset(static_cast<DeviceHeader*>(ws), true,
                                  static_cast<cudaStream_t>(stream), false));
}

moe_status_t moe_route_noalloc(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* b_router, int32_t* topk_idx, float* topk_gate,
                               int32_t* device_report, void* stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_router_width(cfg)) != MOE_OK) return s;
  if ((s = check_ptrs({x, w_router, topk_idx, topk_gate}, {b_router, device_report})) != MOE_OK)
    return s;
  const NoallocLayout NL = noalloc_layout(*cfg);
  if (NL.total > NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* scratch_addr = nullptr;
  MOE_TRY_CUDA(noalloc_scratch_address(&scratch_addr));
  unsigned char* scratch = static_cast<unsigned char*>(scratch_addr);
  // The routing stages index the workspace through a Layout; point the regions they use into
  // the fixed array (the other regions are not touched by routing).
  Call k = make_call(cfg, scratch, stream);
  k.L.hdr = NL.hdr;
  k.L.logits = NL.logits;
  k.L.wrT = NL.wrT;
  k.L.wnorm = NL.wnorm;
  k.L.xnorm = NL.xnorm;
  k.L.rlist = NL.rlist;
  k.L.elist = NL.elist;
  k.L.rsaved = NL.rsaved;
  GemmProblem p = router_problem(k, x, w_router, b_router);
  if ((s = check_tc(k, &p, 1)) != MOE_OK) return s;
  RouterArgs ra = router_args(k, x, w_router, b_router, topk_idx, topk_gate);
  // the report and the refinement counters start from zero on every call
  MOE_TRY_CUDA(header_reset(k.hdr(), true, k.st, false));
  MOE_TRY_CUDA(router_prepare(ra, cfg->dtype, k.st, k.pdl));
  MOE_TRY_CUDA(run_gemms(k, &p, 1));
  MOE_TRY_CUDA(router_select(ra, cfg->dtype, num_sms(), k.st, k.pdl));
  if (device_report) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(1);
    lc.blockDim = dim3(32);
    lc.stream = k.st;
    MOE_TRY_CUDA(cudaLaunchKernelEx(&lc, noalloc_report_kernel,
                                    static_cast<const DeviceHeader*>(k.hdr()), device_report));
  }
  return MOE_OK;
}

}  // extern "C"
