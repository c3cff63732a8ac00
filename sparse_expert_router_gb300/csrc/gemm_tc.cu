// tcgen05 / TMEM / TMA GEMM for sm_103a: the grouped expert GEMMs over ragged expert groups
// and the dense GEMMs of the layer.
//
// Orientation ("swap AB"): the MMA's A operand is a 128-feature tile of a weight matrix
// (weights are stored [d_in, d_out], so the tile is MN-major) and its B operand is a tile of
// up to 256 token rows of the activations (K-major). The accumulator in tensor memory holds
// features in its 128 lanes and tokens in its columns, so a ragged expert group of ~171 rows
// is one N = 176 tile instead of two 128-row tiles, and every weight tile is streamed from HBM
// once per token tile. The grouped GEMM reads the expert group boundaries (the pages' cu_seqlens)
// only after every thread of the kernel has executed griddepcontrol.wait: the Marin summary
// of the week of 2026-09-14 (hero-run epic, #9183) traces a hang to MMA and epilogue warps
// that decoded their tiles from group boundaries before the producing kernel had written them.
//
// Roles of the warps of a CTA (one CTA per SM, persistent over work items):
//   warp 0: TMA producer (one thread) filling a ring of shared-memory stages;
//   warp 1: TMEM allocator and MMA issuer (one thread issues tcgen05.mma, commits to barriers);
//   warps 2..: epilogue, tcgen05.ld from tensor memory, fused epilogue, global stores.
// fp8 problems (the fp8 ragged dot of the expert MLP in the Marin summary of the week of
// 2026-07-06, #6880 / #7079) take E4M3 weights and E4M3 activations straight into
// tcgen05.mma kind::f8f6f4: a stage then carries 128 k per 128-byte swizzle row instead of 64,
// and the epilogue applies the per-tensor activation scale and the per-feature weight scales.
// Every wait on an mbarrier is bounded: after a few seconds the kernel records
// MOE_ERR_DEVICE_TIMEOUT, stops issuing work, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

#ifndef MOE_TC_BN
#define MOE_TC_BN 256
#endif
#ifndef MOE_TC_SMEM_BUDGET
#define MOE_TC_SMEM_BUDGET (220 * 1024)   // dynamic shared memory per CTA, bytes
#endif
// Pair launches: a sixth stage of 32 KB fits next to the epilogue tiles within the 227 KB a CTA
// may use (static shared memory included), so that as many weight bytes are in flight per SM as
// with three 64 KB stages.
constexpr int PAIR_SMEM_BUDGET = 225 * 1024;
constexpr int BM = 128;        // features per tile (MMA M, tensor-memory lanes)
constexpr int BN = MOE_TC_BN;  // max token rows per tile (MMA N)
constexpr int BN_CHUNKED = 128;   // token rows per tile of a k-chunked problem beside others
constexpr int BN_CHUNKED_MAX = 192;   // ... and at most, in a launch of k-chunked problems only
constexpr int64_t DENSE_BAND_BYTES = (int64_t)32 << 20;   // activation rows per band of dense tiles
constexpr int BK = 64;         // k per stage (one 128-byte swizzle row of bf16)
constexpr int BK8 = 128;       // k per stage of an fp8 problem (one 128-byte row of E4M3)
#ifndef MOE_TC_EPI_WARPS
#define MOE_TC_EPI_WARPS 12
#endif
// Kernel instances: KC runs k-chunked fp32 problems (the router) with 8 epilogue warps; the
// others (bf16 or FP8 operands, and BWD: the backward's transposed weights and its SwiGLU
// epilogues) take MOE_TC_EPI_WARPS. The warps of one tensor-memory lane
// quadrant take alternate 16-token chunks. Keeping the instances apart keeps each one's
// registers within what its warp count allows (three or four warps share one sub-partition's
// 16K registers).
template <bool FP8, bool KC, bool BWD> struct Inst {
  static constexpr int EW = KC ? 8 : MOE_TC_EPI_WARPS;
};
constexpr int EPI_TILE_MAX = 16 * 32 * 4;   // transpose tile of one warp: 16 tokens x 32 fp32
constexpr int MAX_PROBS = 3;
constexpr int MAX_GROUPS = 1024;
constexpr int A_HALF = 64 * BK * 2;          // one 64-feature TMA box: 8 KB
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
#ifndef MOE_TC_BBOX
#define MOE_TC_BBOX 32
#endif
constexpr int B_BOX_ROWS = MOE_TC_BBOX;
constexpr int B_BOX_BYTES = B_BOX_ROWS * BK * 2;   // 4 KB
static_assert(BN % B_BOX_ROWS == 0 && BN % 16 == 0 && BN <= 256, "token tile");
static_assert(MOE_TC_EPI_WARPS % 4 == 0 && MOE_TC_EPI_WARPS <= 12, "epilogue warps");

struct TcSeg {
  CUtensorMap a1, a3, b;
  int kblocks;
};

struct TcProblem {
  TcSeg seg[GEMM_MAX_SEG];
  int n_seg;
  int epi, group, M, Mg, m_tiles;
  int n_fastest;               // dense problems: token tiles vary fastest
  int dual;                    // item = 256 features as two 128-feature tiles sharing the token tile
  int kchunk;                  // k-blocks per accumulation chunk (0 = whole K)
  int bn;                      // token rows per tile
  int band;                    // dense problems: token tiles per band (0: all of them)
  const float* w_scale;        // fp8: per-feature weight scales [G, M] of w (and of w3)
  const float* w3_scale;
  const float* act_scale;      // fp8: quantization multiplier of the activations ([1])
  int out_fp8;                 // fp8 SwiGLU output: E4M3 codes of value * out_scale[0]
  const float* out_scale;
  uint32_t* amax;              // fp8 output: running max |value| (fp32 bits)
  int a_kmajor;                // weight tiles K-major ([M, K] per group)
  void* out2;                  // EPI_SWIGLU_SAVE / EPI_SWIGLU_BWD second and third outputs
  void* out3;
  const void* aux_g;           // EPI_SWIGLU_BWD: G and U of the same rows, [rows, M] bf16
  const void* aux_u;
  int64_t ld_aux;
  int64_t rows;
  void* out;
  int64_t ld_out;
  int out_col0;
  const float* bias;
  const int32_t* offsets;
  int G;
  int64_t item_base;           // first item of this problem (grouped: filled on device)
  int64_t n_items;             // dense: m_tiles * n_tiles (grouped: filled on device)
};

// The combine computed inside a dense launch (GemmProblem::cmb_*).
struct TcCombine {
  int active;
  int seg;                     // segment of problem 0 whose activations are c
  const bf16* y_perm;          // [pool_rows, L]
  const int32_t* slot;         // [T, k]
  const float* gate;           // [T, k]
  bf16* c;                     // [T, L]
  int64_t T;
  int k, L;
  int64_t pool_rows;
  uint32_t* ready;             // rows of c written, per token tile
  int bn;                      // token rows per tile of the launch
};

struct TcParams {
  TcProblem p[MAX_PROBS];
  TcCombine cmb;
  int n_probs;
  int grouped;                 // index of the grouped problem (always the last) or -1
  int glu;                     // any problem uses two A tiles per stage (SwiGLU or dual)
  int stages;
  int fp8;                     // E4M3 weights and activations (kind::f8f6f4)
  uint32_t* amax;              // running max |value| of the launch's fp8 output, or NULL
  int nacc;                    // accumulator buffers in tensor memory (1 or 2)
  int acc2_off;                // column offset of the second accumulator of a two-A item
  int b_bytes;                 // bytes of the token tile slot of a stage
  int epi_tile;                // bytes of each epilogue warp's transpose tile (widest output)
  DeviceHeader* hdr;
};

// Instruction descriptor: fp32 accumulator (bits 4..5 = 1), A and B formats at bits 7..9 and
// 10..12 (kind::f16: 1 = bf16; kind::f8f6f4: 0 = E4M3), A MN-major (transposed, bit 15),
// B K-major, N >> 3 at bits 17..22, M >> 4 at bits 24..28.
__device__ __forceinline__ uint32_t make_idesc(int n, bool fp8, bool a_kmajor = false,
                                               int m = BM) {
  const uint32_t ab = fp8 ? 0u : 1u;
  const uint32_t ta = a_kmajor ? 0u : 1u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (ta << 15) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// Problems whose items carry two weight tiles (gate and up) and two accumulators.
__host__ __device__ __forceinline__ bool is_glu(int epi) {
  return epi == EPI_SWIGLU || epi == EPI_SWIGLU_SAVE;
}

// ---- work decomposition -----------------------------------------------------------------

struct Item {
  int p;           // problem
  int wg;          // weight group (expert for grouped problems, shared expert for GROUP_COLS)
  int m_w;         // first feature within the weight group's matrix
  int m0;          // first output column (relative to the problem's M)
  int64_t row0;
  int nrows;
};

// Schedule of the grouped problem, in dynamic shared memory after the stages:
// clamped group bounds and the exclusive prefix of the groups' work items.
struct Sched {
  int32_t* glo;     // [G]
  int32_t* ghi;     // [G]
  int32_t* gitem;   // [G + 1]
};

// Token and feature tile of item `local` of a dense problem. Token tiles vary fastest within
// bands of q.band of them, the bands one after another: the items in flight on the persistent
// grid share the band's activation rows in L2 while every weight tile passes over them.
__device__ __forceinline__ void dense_tile(const TcProblem& q, int64_t local, int64_t n_tiles,
                                           int& n_t, int& m_t) {
  const int64_t band = (q.band > 0 && q.band < n_tiles) ? q.band : n_tiles;
  const int64_t per_band = band * q.m_tiles;
  const int64_t b = local / per_band;
  const int64_t within = local - b * per_band;
  const int64_t bt = imin64(band, n_tiles - b * band);   // token tiles of this band
  n_t = (int)(b * band + within % bt);
  m_t = (int)(within / bt);
}

__device__ __forceinline__ Item decode(const TcParams& P, const Sched& S, int64_t w) {
  Item it;
  int p = 0;
  while (p + 1 < P.n_probs && w >= P.p[p + 1].item_base) ++p;
  const TcProblem& q = P.p[p];
  int64_t local = w - (p == P.grouped ? (int64_t)S.gitem[0] : q.item_base);
  it.p = p;
  if (q.group == GROUP_ROWS) {
    int lo = 0, hi = q.G;   // largest g with gitem[g] <= local
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if ((int64_t)S.gitem[mid] - S.gitem[0] <= local) lo = mid; else hi = mid;
    }
    int g = lo;
    int64_t within = local - ((int64_t)S.gitem[g] - S.gitem[0]);
    const int n_t = (int)(within / q.m_tiles), m_t = (int)(within % q.m_tiles);
    it.wg = g;
    it.m0 = m_t * BM * (q.dual ? 2 : 1);
    it.m_w = it.m0;
    it.row0 = S.glo[g] + (int64_t)n_t * q.bn;
    it.nrows = (int)imin64(q.bn, (int64_t)S.ghi[g] - it.row0);
  } else {
    int64_t n_tiles = cdiv(q.rows, q.bn);
    int n_t, m_t;
    if (q.n_fastest) dense_tile(q, local, n_tiles, n_t, m_t);
    else { n_t = (int)(local / q.m_tiles); m_t = (int)(local % q.m_tiles); }
    it.m0 = m_t * BM * (q.dual ? 2 : 1);
    if (q.group == GROUP_COLS) { it.wg = it.m0 / q.Mg; it.m_w = it.m0 % q.Mg; }
    else { it.wg = 0; it.m_w = it.m0; }
    it.row0 = (int64_t)n_t * q.bn;
    it.nrows = (int)imin64(q.bn, q.rows - it.row0);
  }
  return it;
}

// ---- the combine of a dense launch -------------------------------------------------------

// c rows of this CTA's share of the tokens: each of the launch's epilogue warps takes one token
// at a time. Every element is sum over the token's kept assignments, in order j = 0..k-1, of
// fmaf(gate, y_perm value, acc) in fp32, rounded once to bf16, with the loads of up to four rows
// in flight: the same arithmetic as the separate combine kernel, so c is bitwise the same. After
// a token's row is written, lane 0 counts it in its tile's ready counter (release).
__device__ void combine_rows(const TcCombine& C, int w, int n_w, int lane, DeviceHeader* hdr) {
  const int64_t per = cdiv(C.T, (int64_t)gridDim.x);
  const int64_t t0 = (int64_t)blockIdx.x * per, t1 = imin64(C.T, t0 + per);
  for (int64_t t = t0 + w; t < t1; t += n_w) {
    int32_t s = -1;
    float g = 0.0f;
    if (lane < C.k) {
      s = C.slot[t * C.k + lane];
      g = C.gate[t * C.k + lane];
      if (s >= C.pool_rows || s < -1) {
        report_error(hdr, MOE_ERR_BAD_ROUTING, (int)t);
        s = -1;
      }
    }
    const unsigned kept = __ballot_sync(~0u, s >= 0);
    // every lane runs every iteration (the shuffles below take the whole warp); lanes past the
    // row's end only skip their loads and stores
    for (int i0 = 0; i0 < C.L; i0 += 256) {
      const int i = i0 + lane * 8;
      const bool on = i < C.L;
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      unsigned m = kept;
      while (m) {
        int js[4];
        int nn = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (m) {
            js[u] = __ffs(m) - 1;
            m &= m - 1;
            ++nn;
          }
        }
        float v[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u < nn) {
            const int32_t sj = __shfl_sync(~0u, s, js[u]);
            if (on) ld8(C.y_perm + (int64_t)sj * C.L + i, v[u]);
            else
#pragma unroll
              for (int q = 0; q < 8; ++q) v[u][q] = 0.0f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u < nn) {
            const float gj = __shfl_sync(~0u, g, js[u]);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(gj, v[u][q], acc[q]);
          }
        }
      }
      if (on) st8(C.c + t * C.L + i, acc);
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(C.ready + t / C.bn, 1u);
    }
  }
}

// Waits (bounded) until the combine has written all `rows` rows of token tile `tile`; then orders
// the TMA loads that follow after those writes. False when the kernel is aborting.
__device__ bool wait_combined(const TcCombine& C, int64_t tile, int rows, volatile int* abort_flag,
                              DeviceHeader* hdr) {
  const uint32_t* p = C.ready + tile;
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= (uint32_t)rows) break;
    if (*abort_flag) return false;
    __nanosleep(64);
    if ((i & 63u) == 63u) {
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > TIMEOUT_NS) {
        report_error(hdr, MOE_ERR_DEVICE_TIMEOUT, 7);
        *abort_flag = 1;
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ---- the kernel ---------------------------------------------------------------------------

// Two instances: FP8 = false (bf16 operands, k-chunked fp32 problems) and FP8 = true (E4M3
// operands, scales and the E4M3 SwiGLU output), so that neither carries the other's registers:
// with 10 warps per CTA three warps share one sub-partition's 16K registers, 168 per thread.
// Two instances: FP8 = false (bf16 operands, k-chunked fp32 problems) and FP8 = true (E4M3
// operands, scales and the E4M3 SwiGLU output), so that neither carries the other's registers:
// with 10 warps per CTA three warps share one sub-partition's 16K registers, 168 per thread.
// CMB: the launch's epilogue warps first compute the combine that one segment's activations are
// (TcCombine), and the producer loads a token tile of that segment once its rows are written;
// an instance of its own, so that the other launches carry none of that code.
template <bool FP8, bool KC, bool BWD, bool CMB = false>
__global__ void __launch_bounds__(64 + 32 * Inst<FP8, KC, BWD>::EW, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams P) {
  constexpr int EPI_WARPS = Inst<FP8, KC, BWD>::EW;
  static_assert(!CMB || (!FP8 && !KC && !BWD), "combine launches: bf16 dense problems");
  const int EPI_STAGE_BYTES = P.epi_tile;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * 8 + 4];
  __shared__ int64_t s_total;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = P.stages;
  const bool glu = P.glu != 0;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = (glu ? 2 * A_BYTES : A_BYTES) + P.b_bytes;
  auto sA1 = [&](int s) { return base + s * stage_bytes; };
  auto sA3 = [&](int s) { return base + s * stage_bytes + A_BYTES; };
  auto sB = [&](int s) { return base + s * stage_bytes + (glu ? 2 * A_BYTES : A_BYTES); };
  constexpr bool fp8 = FP8;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[8]);
  // Accumulators in tensor memory (512 columns): buffer b starts at column b*BN. A launch keeps
  // two buffers, so that the epilogue of one tile overlaps the main loop of the next, unless a
  // two-A item (SwiGLU gate+up or a dual 256-feature item) with more than 128 token columns needs
  // both halves; two-A items of at most 128 token columns put their second accumulator at
  // column +128 of their buffer.
  const int nacc = P.nacc;
  const uint32_t acc2 = (uint32_t)P.acc2_off;
  auto tmem_full = [&](int b) { return smem_u32(&bars[16 + b]); };
  auto tmem_empty = [&](int b) { return smem_u32(&bars[18 + b]); };
  Sched S;
  unsigned char* epi_stage = base + (size_t)stages * stage_bytes;   // [EPI_WARPS][EPI_STAGE_BYTES]
  {
    int32_t* sp = reinterpret_cast<int32_t*>(epi_stage + EPI_WARPS * EPI_STAGE_BYTES);
    const int G = (P.grouped >= 0) ? P.p[P.grouped].G : 0;
    S.glo = sp;
    S.ghi = sp + G;
    S.gitem = sp + 2 * G;
  }
  auto full = [&](int s) { return full0 + 8u * s; };
  auto empty = [&](int s) { return empty0 + 8u * s; };

  // set-up that reads nothing a preceding kernel writes
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), 32 * EPI_WARPS);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int p = 0; p < P.n_probs; ++p)
      for (int s = 0; s < P.p[p].n_seg; ++s) {
        prefetch_map(&P.p[p].seg[s].a1);
        prefetch_map(&P.p[p].seg[s].b);
        if (glu) prefetch_map(&P.p[p].seg[s].a3);
      }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // Every thread waits for the preceding kernel before it reads the group offsets.
  pdl_wait();

  // schedule of the grouped problem: clamped group bounds and the prefix of its items
  if (P.grouped >= 0) {
    const TcProblem& q = P.p[P.grouped];
    if (warp == 0) {
      const int G = q.G;
      const int per = (G + 31) / 32;
      int64_t sum = 0;
      for (int i = 0; i < per; ++i) {
        int g = lane * per + i;
        if (g < G) {
          int64_t lo = imin64(imax64(q.offsets[g], 0), q.rows);
          int64_t hi = imin64(imax64(q.offsets[g + 1], lo), q.rows);
          S.glo[g] = (int32_t)lo;
          S.ghi[g] = (int32_t)hi;
          sum += cdiv(hi - lo, q.bn) * q.m_tiles;
        }
      }
      int64_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t v = __shfl_up_sync(~0u, incl, o);
        if (lane >= o) incl += v;
      }
      int64_t run = incl - sum + q.item_base;
      for (int i = 0; i < per; ++i) {
        int g = lane * per + i;
        if (g < G) {
          S.gitem[g] = (int32_t)run;
          run += cdiv((int64_t)S.ghi[g] - S.glo[g], q.bn) * q.m_tiles;
        }
      }
      if (lane == 31) { S.gitem[G] = (int32_t)run; s_total = run; }
    }
  } else if (threadIdx.x == 0) {
    const TcProblem& q = P.p[P.n_probs - 1];
    s_total = q.item_base + q.n_items;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int64_t total = s_total;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int bk = fp8 ? BK8 : BK;
    for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      Item it = decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      const int nb = (it.nrows + B_BOX_ROWS - 1) / B_BOX_ROWS;
      const bool two_a = is_glu(q.epi) || q.dual;
      const uint32_t bytes = (two_a ? 2 * A_BYTES : A_BYTES) + nb * B_BOX_BYTES;
      for (int s = 0; s < q.n_seg && ok; ++s) {
        const TcSeg& sg = q.seg[s];
        if constexpr (CMB) {
          if (s == P.cmb.seg &&
              !wait_combined(P.cmb, it.row0 / P.cmb.bn, it.nrows, &s_abort, P.hdr)) {
            ok = false;
            break;
          }
        }
        for (int kb = 0; kb < sg.kblocks; ++kb) {
          const int k0 = kb * bk;
          if (!mbar_wait(empty(stage), phase ^ 1u, &s_abort, P.hdr, 1)) { ok = false; break; }
          mbar_expect_tx(full(stage), bytes);
          if constexpr (FP8) {
            // one [128 k][128 features] box of E4M3 per A tile
            tma_load_3d(smem_u32(sA1(stage)), &sg.a1, full(stage), it.m_w, k0, it.wg);
            if (is_glu(q.epi))
              tma_load_3d(smem_u32(sA3(stage)), &sg.a3, full(stage), it.m_w, k0, it.wg);
            else if (q.dual)
              tma_load_3d(smem_u32(sA3(stage)), &sg.a1, full(stage), it.m_w + BM, k0, it.wg);
          } else if (BWD && q.a_kmajor) {
            // one [128 features][64 k] box per A tile (K-major)
            tma_load_3d(smem_u32(sA1(stage)), &sg.a1, full(stage), k0, it.m_w, it.wg);
            if (is_glu(q.epi))
              tma_load_3d(smem_u32(sA3(stage)), &sg.a3, full(stage), k0, it.m_w, it.wg);
            else if (q.dual)
              tma_load_3d(smem_u32(sA3(stage)), &sg.a1, full(stage), k0, it.m_w + BM, it.wg);
          } else {
            tma_load_3d(smem_u32(sA1(stage)), &sg.a1, full(stage), it.m_w, k0, it.wg);
            tma_load_3d(smem_u32(sA1(stage)) + A_HALF, &sg.a1, full(stage), it.m_w + 64, k0, it.wg);
            if (is_glu(q.epi)) {
              tma_load_3d(smem_u32(sA3(stage)), &sg.a3, full(stage), it.m_w, k0, it.wg);
              tma_load_3d(smem_u32(sA3(stage)) + A_HALF, &sg.a3, full(stage), it.m_w + 64, k0, it.wg);
            } else if (q.dual) {
              tma_load_3d(smem_u32(sA3(stage)), &sg.a1, full(stage), it.m_w + BM, k0, it.wg);
              tma_load_3d(smem_u32(sA3(stage)) + A_HALF, &sg.a1, full(stage), it.m_w + BM + 64, k0,
                          it.wg);
            }
          }
          for (int b = 0; b < nb; ++b)
            tma_load_2d(smem_u32(sB(stage)) + b * B_BOX_BYTES, &sg.b, full(stage), k0,
                        (int)(it.row0 + b * B_BOX_ROWS));
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int ev = 0;      // accumulator events of this CTA: one per item, or one per k-chunk
    for (int64_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      Item it = decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      const bool sw = is_glu(q.epi) || q.dual;   // second A tile -> second accumulator
      const int n = ((it.nrows + 15) / 16) * 16;
      const bool akm = BWD && q.a_kmajor;
      const uint32_t idesc = make_idesc(n, fp8, akm);
      int kb_total = 0;
      for (int s2 = 0; s2 < q.n_seg; ++s2) kb_total += q.seg[s2].kblocks;
      const int per_ev = q.kchunk ? q.kchunk : kb_total;
      for (int kb0 = 0; kb0 < kb_total && ok; kb0 += per_ev, ++ev) {
        const int buf = ev % nacc;
        const uint32_t acc_phase = (uint32_t)(ev / nacc) & 1u;
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        if (!mbar_wait(tmem_empty(buf), acc_phase ^ 1u, &s_abort, P.hdr, 2)) { ok = false; break; }
        tc_fence_after();
        uint32_t accumulate = 0;
        const int kb_end = min(kb0 + per_ev, kb_total);
        for (int kk = kb0; kk < kb_end; ++kk) {
          if (!mbar_wait(full(stage), phase, &s_abort, P.hdr, 3)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a1 = smem_u32(sA1(stage)), a3 = smem_u32(sA3(stage)), b = smem_u32(sB(stage));
          // MN-major A: LBO = stride between 128-byte feature atoms (two 64-feature halves for
          // bf16; one atom holds all 128 E4M3 features), SBO = stride between 8-row k groups;
          // K-major B: SBO = stride between 8-row groups, LBO unused. Every MMA consumes 32
          // bytes of each 128-byte row: 16 k of bf16 or 32 k of E4M3.
          const uint32_t albo = (uint32_t)A_HALF, asbo = 1024u;
          if constexpr (FP8) {
#pragma unroll
            for (int k32 = 0; k32 < BK8 / 32; ++k32) {
              const uint64_t bd = smem_desc(b + k32 * 32, 16, 1024);
              mma_e4m3(d_tmem, smem_desc(a1 + k32 * 4096, albo, asbo), bd, idesc, accumulate);
              if (sw)
                mma_e4m3(d_tmem + acc2, smem_desc(a3 + k32 * 4096, albo, asbo), bd, idesc,
                         accumulate);
              accumulate = 1;
            }
          } else {
            // K-major A tiles advance 32 bytes per k16 like B; MN-major ones 16 rows (2 KB)
            const uint32_t astep = akm ? 32u : 2048u;
            const uint32_t alb = akm ? 16u : albo;
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t bd = smem_desc(b + k16 * 32, 16, 1024);
              mma_bf16(d_tmem, smem_desc(a1 + k16 * astep, alb, asbo), bd, idesc, accumulate);
              if (sw)
                mma_bf16(d_tmem + acc2, smem_desc(a3 + k16 * astep, alb, asbo), bd, idesc,
                         accumulate);
              accumulate = 1;
            }
          }
          mma_commit(empty(stage));
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        mma_commit(tmem_full(buf));
      }
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // Warp w reads tensor-memory lanes 32*(w%4).. (its quadrant); with 8 epilogue warps the two
    // warps of a quadrant take alternate 16-token chunks. Each chunk (32 features x 16 tokens)
    // is transposed through a per-warp shared-memory tile so that every lane then writes whole
    // 16-byte pieces of output rows.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;                    // 0, or 1 for the second warp of a quadrant
    unsigned char* stg = epi_stage + (warp - 2) * EPI_STAGE_BYTES;
    float* stg_f = reinterpret_cast<float*>(stg);
    bf16* stg_h = reinterpret_cast<bf16*>(stg);
    // Writes the transpose tile's 16 token rows x 32 E4M3 codes (byte j * 32 + lane = token j,
    // feature lane) to out: lane -> (row lane / 2, 16-byte half lane % 2).
    auto store_e4m3_tile = [&](void* out, int64_t ld, int col0, const Item& it, int c0, int f0,
                               int M) {
      const int rows_here = min(16, it.nrows - c0);
      const int row = lane >> 1, part = lane & 1;
      if (f0 + part * 16 < M && row < rows_here) {
        const uint4 val = *reinterpret_cast<const uint4*>(stg + row * 32 + part * 16);
        const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 16;
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + o) = val;
      }
    };
    // Writes the transpose tile's 16 token rows x 32 bf16 values (element j * 32 + lane = token
    // j, feature lane) to out: lane -> (rows lane / 4 and lane / 4 + 8, 16-byte part lane % 4).
    auto store_bf16_tile = [&](void* out, int64_t ld, int col0, const Item& it, int c0, int f0,
                               int M) {
      const int rows_here = min(16, it.nrows - c0);
      const int part = lane & 3;
      const bool ok = f0 + part * 8 < M;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = (lane >> 2) + 8 * r;
        if (ok && row < rows_here) {
          const uint4 val = *reinterpret_cast<const uint4*>(stg_h + row * 32 + part * 8);
          const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 8;
          *reinterpret_cast<uint4*>(static_cast<bf16*>(out) + o) = val;
        }
      }
    };
    // Writes one 16-token x 32-feature chunk of this warp (values final: lane = feature,
    // v[j] = token c0 + j) to out[row][col0 + feature] through the transpose tile, so that every
    // lane stores whole 16-byte pieces of output rows. kind: 0 fp32, 1 bf16.
    auto store_rows = [&](void* out, int64_t ld, int col0, int kind, const Item& it, int c0,
                          int f0, int M, const float* v) {
      if (kind == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) stg_f[j * 32 + lane] = v[j];
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) stg_h[j * 32 + lane] = __float2bfloat16_rn(v[j]);
      }
      __syncwarp();
      const int rows_here = min(16, it.nrows - c0);
      if (kind == 0) {
        const int part = lane & 7;
        const bool ok = f0 + part * 4 < M;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int row = (lane >> 3) + 4 * r;
          if (ok && row < rows_here) {
            const float4 val = *reinterpret_cast<const float4*>(stg_f + row * 32 + part * 4);
            const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 4;
            *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = val;
          }
        }
      } else {
        store_bf16_tile(out, ld, col0, it, c0, f0, M);
      }
      __syncwarp();
    };
    int ev = 0;
    float amax = 0.0f;                                   // fp8 output: this thread's max |value|
    if constexpr (CMB) combine_rows(P.cmb, warp - 2, EPI_WARPS, lane, P.hdr);
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
      Item it = decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      if (KC && q.kchunk) {
        // k-chunked fp32 problem: sum the chunk accumulators in registers, in chunk order.
        // This warp owns columns half*16 + 32*i (i < KCW) of the <= BN_CHUNKED_MAX-token tile.
        constexpr int KCW = BN_CHUNKED_MAX / 32;
        static_assert(!KC || EPI_WARPS == 8, "k-chunked epilogue layout");
        int kb_total = q.seg[0].kblocks;
        const int f0 = it.m0 + quad * 32;
        float acc[KCW][16];
#pragma unroll
        for (int i = 0; i < KCW; ++i)
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[i][j] = 0.0f;
        bool ok = true;
        for (int kb0 = 0; kb0 < kb_total; kb0 += q.kchunk, ++ev) {
          const int buf = ev % nacc;
          const uint32_t acc_phase = (uint32_t)(ev / nacc) & 1u;
          if (!mbar_wait(tmem_full(buf), acc_phase, &s_abort, P.hdr, 4)) { ok = false; break; }
          tc_fence_after();
          const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN);
#pragma unroll
          for (int i = 0; i < KCW; ++i) {
            const int c0 = half * 16 + 32 * i;
            if (c0 < it.nrows) {
              float v[16];
              tmem_ld16(lane_addr + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[i][j] = __fadd_rn(acc[i][j], v[j]);
            }
          }
          tc_fence_before();
          mbar_arrive(tmem_empty(buf));
        }
        if (!ok) break;
        const float bias = (q.bias && f0 + lane < q.M) ? q.bias[f0 + lane] : 0.0f;
#pragma unroll
        for (int i = 0; i < KCW; ++i) {
          const int c0 = half * 16 + 32 * i;
          if (c0 < it.nrows) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fadd_rn(acc[i][j], bias);
            store_rows(q.out, q.ld_out, q.out_col0, 0, it, c0, f0, q.M, v);
          }
        }
        continue;
      }
      if constexpr (BWD) {
        if (q.epi == EPI_SWIGLU_BWD) {
          // G and U of this item (nrows x 128 or, dual, 256 features, 128-byte lines) head for
          // L2 while the main loop runs, so that the epilogue's loads of them hit L2
          const int lpr = q.dual ? 4 : 2;         // lines of 128 bytes per row and tensor
          const int nl = it.nrows * 2 * lpr;
          for (int i = threadIdx.x - 64; i < nl; i += 32 * EPI_WARPS) {
            const int r = i / (2 * lpr), t2 = (i / lpr) & 1, line = i % lpr;
            const bf16* base_p = static_cast<const bf16*>(t2 ? q.aux_u : q.aux_g);
            const bf16* ptr = base_p + (it.row0 + r) * q.ld_aux + it.m0 + line * 64;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
          }
        }
      }
      const int buf = ev % nacc;
      const uint32_t acc_phase = (uint32_t)(ev / nacc) & 1u;
      ++ev;
      // fp8: dequantization factor of each accumulator, fp32(1 / activation scale) times the
      // feature's weight scale in this expert (w, and w3 for the up projection). Loaded before
      // the wait for the accumulator, so that their latency hides behind the main loop.
      float sc1s[2] = {1.0f, 1.0f}, sc3s[2] = {1.0f, 1.0f}, osc = 1.0f;
      if constexpr (FP8) {
        const float da = __fdiv_rn(1.0f, *q.act_scale);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int f0 = it.m0 + sub * BM + quad * 32;
          const bool fok = (sub == 0 || q.dual) && f0 + lane < q.M;
          const int64_t fs = (int64_t)it.wg * q.M + f0 + lane;
          sc1s[sub] = fok ? __fmul_rn(da, q.w_scale[fs]) : 0.0f;
          sc3s[sub] = (fok && q.w3_scale) ? __fmul_rn(da, q.w3_scale[fs]) : 0.0f;
        }
        if (q.out_fp8) osc = *q.out_scale;
      }
      if (!mbar_wait(tmem_full(buf), acc_phase, &s_abort, P.hdr, 4)) break;
      tc_fence_after();
      if constexpr (FP8) {
        if (q.out_fp8 && is_glu(q.epi)) {
          // E4M3 hidden: the SwiGLU of every chunk of this warp is computed and packed into
          // registers first, then the accumulators are released, so that the next item's MMAs
          // run while this warp writes its codes out
          constexpr int CPW = (BN / 16 + EPI_WARPS / 4 - 1) / (EPI_WARPS / 4);   // chunks per warp
          const int f0 = it.m0 + quad * 32;
          const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                     (uint32_t)(buf * BN);
          const bool fok = f0 + lane < q.M;
          const float sc1 = sc1s[0], sc3 = sc3s[0];
          uint32_t pk[CPW][4];
#pragma unroll
          for (int i = 0; i < CPW; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
              float v[16], v3[16];
              tmem_ld16(lane_addr + c0, v);
              tmem_ld16(lane_addr + acc2 + c0, v3);
              tmem_wait_ld();
              const int valid = min(16, it.nrows - c0);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float h = swiglu(__fmul_rn(v[j], sc1), __fmul_rn(v3[j], sc3));
                if (fok && j < valid) amax = fmaxf(amax, fabsf(h));
                v[j] = __fmul_rn(h, osc);
              }
#pragma unroll
              for (int j = 0; j < 16; j += 4)
                pk[i][j / 4] = e4m3x2(v[j + 1], v[j]) | (e4m3x2(v[j + 3], v[j + 2]) << 16);
            }
          }
          tc_fence_before();
          mbar_arrive(tmem_empty(buf));
          uint8_t* stg_b = reinterpret_cast<uint8_t*>(stg);
#pragma unroll
          for (int i = 0; i < CPW; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                stg_b[j * 32 + lane] = (uint8_t)((pk[i][j / 4] >> (8 * (j % 4))) & 0xFFu);
              __syncwarp();
              store_e4m3_tile(q.out, q.ld_out, q.out_col0, it, c0, f0, q.M);
              __syncwarp();
            }
          }
          continue;
        }
      }
      if constexpr (!FP8 && !KC && !BWD) {
        if (q.epi == EPI_SWIGLU) {
          // bf16 hidden: as for E4M3 above, the SwiGLU of a warp's first CPR chunks is packed
          // into registers before the accumulators are released; chunks past those (tiles of
          // more than 192 tokens) are written out first, in place
          constexpr int CPW = (BN / 16 + EPI_WARPS / 4 - 1) / (EPI_WARPS / 4);   // chunks per warp
          constexpr int CPR = CPW < 4 ? CPW : 4;
          const int f0 = it.m0 + quad * 32;
          const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                     (uint32_t)(buf * BN);
          for (int i = CPR; i < CPW; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
              float v[16], v3[16];
              tmem_ld16(lane_addr + c0, v);
              tmem_ld16(lane_addr + acc2 + c0, v3);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = swiglu(v[j], v3[j]);
              store_rows(q.out, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v);
            }
          }
          uint32_t pk[CPR][8];
#pragma unroll
          for (int i = 0; i < CPR; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
              float v[16], v3[16];
              tmem_ld16(lane_addr + c0, v);
              tmem_ld16(lane_addr + acc2 + c0, v3);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(swiglu(v[j], v3[j]),
                                                                swiglu(v[j + 1], v3[j + 1]));
                pk[i][j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
              }
            }
          }
          tc_fence_before();
          mbar_arrive(tmem_empty(buf));
#pragma unroll
          for (int i = 0; i < CPR; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                stg_h[j * 32 + lane] = __ushort_as_bfloat16((unsigned short)(pk[i][j / 2] & 0xFFFFu));
                stg_h[(j + 1) * 32 + lane] = __ushort_as_bfloat16((unsigned short)(pk[i][j / 2] >> 16));
              }
              __syncwarp();
              store_bf16_tile(q.out, q.ld_out, q.out_col0, it, c0, f0, q.M);
              __syncwarp();
            }
          }
          continue;
        }
      }
      for (int sub = 0; sub < (q.dual ? 2 : 1); ++sub) {
      const int f0 = it.m0 + sub * BM + quad * 32;       // first feature of this warp
      const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                 (uint32_t)(buf * BN) + (uint32_t)sub * acc2;
      const bool f32out = (q.epi == EPI_F32);
      const bool fok = f0 + lane < q.M;
      const float bias = (f32out && q.bias && fok) ? q.bias[f0 + lane] : 0.0f;
      const float sc1 = sub ? sc1s[1] : sc1s[0], sc3 = sub ? sc3s[1] : sc3s[0];
      for (int c0 = half * 16; c0 < it.nrows; c0 += 16 * (EPI_WARPS / 4)) {
        float v[16], v3[16];
        tmem_ld16(lane_addr + c0, v);
        if (is_glu(q.epi)) tmem_ld16(lane_addr + acc2 + c0, v3);
        tmem_wait_ld();
        if (f32out) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __fadd_rn(v[j], bias);
        }
        if constexpr (FP8) {
#pragma unroll
          for (int j = 0; j < 16; ++j) { v[j] = __fmul_rn(v[j], sc1); v3[j] = __fmul_rn(v3[j], sc3); }
        }
        if constexpr (BWD) {
          if (q.epi == EPI_SWIGLU_SAVE) {
            // the pre-activations of the backward's recompute, then the hidden below
            store_rows(q.out2, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v);
            store_rows(q.out3, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v3);
          } else if (q.epi == EPI_SWIGLU_BWD) {
            // v = dA; G and U of the same (row, feature): dG = dA U silu'(G), dU = dA silu(G)
            const bf16* gp = static_cast<const bf16*>(q.aux_g);
            const bf16* up = static_cast<const bf16*>(q.aux_u);
            const int valid = min(16, it.nrows - c0);
            // all 32 loads first (packed in pairs), so that they are in flight together
            __nv_bfloat162 gg[8], uu[8];
            const bf16 zero = __float2bfloat16_rn(0.0f);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              bf16 g0 = zero, g1 = zero, u0 = zero, u1 = zero;
              const int64_t o = (it.row0 + c0 + j) * q.ld_aux + f0 + lane;
              if (fok && j < valid) { g0 = gp[o]; u0 = up[o]; }
              if (fok && j + 1 < valid) { g1 = gp[o + q.ld_aux]; u1 = up[o + q.ld_aux]; }
              gg[j / 2] = __halves2bfloat162(g0, g1);
              uu[j / 2] = __halves2bfloat162(u0, u1);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float g = (j & 1) ? __high2float(gg[j / 2]) : __low2float(gg[j / 2]);
              const float u = (j & 1) ? __high2float(uu[j / 2]) : __low2float(uu[j / 2]);
              const float sg = sigmoid_bf16(g);                      // sigmoid(G)
              v3[j] = v[j] * u * (sg * (1.0f + g * (1.0f - sg)));
              v[j] = v[j] * (g * sg);
            }
            store_rows(q.out, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v3);
            store_rows(q.out2, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v);
            continue;
          }
        }
        if (is_glu(q.epi)) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = swiglu(v[j], v3[j]);
        }
        store_rows(q.out, q.ld_out, q.out_col0, f32out ? 0 : 1, it, c0, f0, q.M, v);
      }
      }
      tc_fence_before();
      mbar_arrive(tmem_empty(buf));
    }
    if (FP8 && P.amax) {
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
      if (lane == 0 && amax > 0.0f) amax_update(P.amax, amax);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base)
                 : "memory");
  }
}

// ---- the CTA-pair kernel ------------------------------------------------------------------
//
// A cluster of two CTAs runs each item with tcgen05.mma.cta_group::2: an MMA of M = 256 takes
// 128 weight rows from each CTA and the token tile from both, each CTA loading half of it (N / 2
// rows); each CTA's tensor memory receives its own 128 rows of the accumulator over all N
// columns. Every item keeps two weight tiles per CTA, as in tc_gemm_kernel, so a pair item spans
// twice the features of a single-CTA item: a SwiGLU item 256 output features (each CTA the gate
// and up tiles of its 128), a dual item 512 (each CTA two 128-feature tiles). The token tile is
// loaded once per pair instead of once per CTA: 46 KB per k-block and SM instead of 60 KB for the
// same MMAs, where L2-to-SM ingest is what bounds the dense GEMMs.
// Forward problems (EPI_SWIGLU, EPI_STORE, EPI_F32), bf16 or E4M3 operands; no combine.

// Item w of a pair launch: SwiGLU items of 256 features, dual items of 512.
__device__ __forceinline__ Item pair_decode(const TcParams& P, const Sched& S, int64_t w) {
  Item it;
  int p = 0;
  while (p + 1 < P.n_probs && w >= P.p[p + 1].item_base) ++p;
  const TcProblem& q = P.p[p];
  const int pw = q.dual ? 4 * BM : 2 * BM;             // features of a pair item
  int64_t local = w - (p == P.grouped ? (int64_t)S.gitem[0] : q.item_base);
  it.p = p;
  if (q.group == GROUP_ROWS) {
    int lo = 0, hi = q.G;
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if ((int64_t)S.gitem[mid] - S.gitem[0] <= local) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int64_t within = local - ((int64_t)S.gitem[g] - S.gitem[0]);
    const int n_t = (int)(within / q.m_tiles), m_t = (int)(within % q.m_tiles);
    it.wg = g;
    it.m0 = m_t * pw;
    it.m_w = it.m0;
    it.row0 = S.glo[g] + (int64_t)n_t * q.bn;
    it.nrows = (int)imin64(q.bn, (int64_t)S.ghi[g] - it.row0);
  } else {
    const int64_t n_tiles = cdiv(q.rows, q.bn);
    int n_t, m_t;
    dense_tile(q, local, n_tiles, n_t, m_t);
    it.m0 = m_t * pw;
    if (q.group == GROUP_COLS) { it.wg = it.m0 / q.Mg; it.m_w = it.m0 % q.Mg; }
    else { it.wg = 0; it.m_w = it.m0; }
    it.row0 = (int64_t)n_t * q.bn;
    it.nrows = (int)imin64(q.bn, q.rows - it.row0);
  }
  return it;
}

// FP8: E4M3 weights and activations (kind::f8f6f4), a stage carrying 128 k in the same bytes;
// the epilogue applies the activation and per-feature weight scales and, for a SwiGLU GEMM,
// writes an E4M3 hidden and keeps its running max |value|.
template <bool FP8>
__global__ void __launch_bounds__(64 + 32 * MOE_TC_EPI_WARPS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcParams P) {
  constexpr int EPI_WARPS = MOE_TC_EPI_WARPS;
  const int EPI_STAGE_BYTES = P.epi_tile;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * 8 + 4];
  __shared__ int64_t s_total;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = P.stages;
  const uint32_t rank = cluster_ctarank();                 // this CTA in its pair
  const int64_t unit = blockIdx.x >> 1, n_units = gridDim.x >> 1;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = 2 * A_BYTES + P.b_bytes;         // two weight tiles, half a token tile
  auto sA1 = [&](int s) { return base + s * stage_bytes; };
  auto sA3 = [&](int s) { return base + s * stage_bytes + A_BYTES; };
  auto sB = [&](int s) { return base + s * stage_bytes + 2 * A_BYTES; };
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[8]);
  auto full = [&](int s) { return full0 + 8u * s; };
  auto empty = [&](int s) { return empty0 + 8u * s; };
  auto tmem_full = [&](int b) { return smem_u32(&bars[16 + b]); };
  auto tmem_empty = [&](int b) { return smem_u32(&bars[18 + b]); };
  const int nacc = P.nacc;
  const uint32_t acc2 = (uint32_t)P.acc2_off;
  unsigned char* epi_stage = base + (size_t)stages * stage_bytes;   // [EPI_WARPS][EPI_STAGE_BYTES]
  Sched S;
  {
    int32_t* sp = reinterpret_cast<int32_t*>(epi_stage + EPI_WARPS * EPI_STAGE_BYTES);
    const int G = (P.grouped >= 0) ? P.p[P.grouped].G : 0;
    S.glo = sp;
    S.ghi = sp + G;
    S.gitem = sp + 2 * G;
  }

  // set-up that reads nothing a preceding kernel writes
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), 2 * 32 * EPI_WARPS);      // rank 0's: both CTAs' epilogues
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int p = 0; p < P.n_probs; ++p)
      for (int s = 0; s < P.p[p].n_seg; ++s) {
        prefetch_map(&P.p[p].seg[s].a1);
        prefetch_map(&P.p[p].seg[s].b);
        if (is_glu(P.p[p].epi)) prefetch_map(&P.p[p].seg[s].a3);
      }
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, collectively, the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }

  // Every thread waits for the preceding kernel before it reads the group offsets.
  pdl_wait();

  // schedule of the grouped problem (as in tc_gemm_kernel)
  if (P.grouped >= 0) {
    const TcProblem& q = P.p[P.grouped];
    if (warp == 0) {
      const int G = q.G;
      const int per = (G + 31) / 32;
      int64_t sum = 0;
      for (int i = 0; i < per; ++i) {
        int g = lane * per + i;
        if (g < G) {
          int64_t lo = imin64(imax64(q.offsets[g], 0), q.rows);
          int64_t hi = imin64(imax64(q.offsets[g + 1], lo), q.rows);
          S.glo[g] = (int32_t)lo;
          S.ghi[g] = (int32_t)hi;
          sum += cdiv(hi - lo, q.bn) * q.m_tiles;
        }
      }
      int64_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t v = __shfl_up_sync(~0u, incl, o);
        if (lane >= o) incl += v;
      }
      int64_t run = incl - sum + q.item_base;
      for (int i = 0; i < per; ++i) {
        int g = lane * per + i;
        if (g < G) {
          S.gitem[g] = (int32_t)run;
          run += cdiv((int64_t)S.ghi[g] - S.glo[g], q.bn) * q.m_tiles;
        }
      }
      if (lane == 31) { S.gitem[G] = (int32_t)run; s_total = run; }
    }
  } else if (threadIdx.x == 0) {
    const TcProblem& q = P.p[P.n_probs - 1];
    s_total = q.item_base + q.n_items;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int64_t total = s_total;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    // This CTA's two 128-row weight tiles and its half (N / 2 rows) of the token tile; the bytes
    // of both CTAs complete on rank 0's full barrier, which rank 0 arms with their sum.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t w = unit; w < total && ok; w += n_units) {
      Item it = pair_decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      const int half_rows = ((it.nrows + 15) / 16) * 8;
      const int nb = (half_rows + B_BOX_ROWS - 1) / B_BOX_ROWS;
      const uint32_t bytes = 2u * (uint32_t)(2 * A_BYTES + nb * B_BOX_BYTES);
      const int64_t my_row0 = it.row0 + (int64_t)rank * half_rows;
      const bool gl = is_glu(q.epi);
      // SwiGLU: gate (W1) and up (W3) tiles of features m_w + 128 rank ..; dual: features
      // m_w + 256 rank .. and .. + 128 of the one weight matrix
      const int mx1 = it.m_w + (gl ? BM : 2 * BM) * (int)rank;
      const int mx3 = gl ? mx1 : mx1 + BM;
      for (int s = 0; s < q.n_seg && ok; ++s) {
        const TcSeg& sg = q.seg[s];
        const CUtensorMap* m3 = gl ? &sg.a3 : &sg.a1;
        for (int kb = 0; kb < sg.kblocks; ++kb) {
          const int k0 = kb * (FP8 ? BK8 : BK);
          if (!mbar_wait(empty(stage), phase ^ 1u, &s_abort, P.hdr, 1)) { ok = false; break; }
          const uint32_t fb = mapa_shared(full(stage), 0);
          if (rank == 0) mbar_expect_tx(full(stage), bytes);
          if constexpr (FP8) {
            // one [128 k][128 features] box of E4M3 per weight tile
            tma_load_3d_pair(smem_u32(sA1(stage)), &sg.a1, fb, mx1, k0, it.wg);
            tma_load_3d_pair(smem_u32(sA3(stage)), m3, fb, mx3, k0, it.wg);
          } else {
            tma_load_3d_pair(smem_u32(sA1(stage)), &sg.a1, fb, mx1, k0, it.wg);
            tma_load_3d_pair(smem_u32(sA1(stage)) + A_HALF, &sg.a1, fb, mx1 + 64, k0, it.wg);
            tma_load_3d_pair(smem_u32(sA3(stage)), m3, fb, mx3, k0, it.wg);
            tma_load_3d_pair(smem_u32(sA3(stage)) + A_HALF, m3, fb, mx3 + 64, k0, it.wg);
          }
          for (int b = 0; b < nb; ++b)
            tma_load_2d_pair(smem_u32(sB(stage)) + b * B_BOX_BYTES, &sg.b, fb, k0,
                             (int)(my_row0 + b * B_BOX_ROWS));
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer: rank 0 issues for both CTAs ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int ev = 0;      // accumulator events: one per item
    for (int64_t w = unit; w < total && ok; w += n_units) {
      Item it = pair_decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      const int n = ((it.nrows + 15) / 16) * 16;
      const uint32_t idesc = make_idesc(n, FP8, false, 2 * BM);
      int kb_total = 0;
      for (int s2 = 0; s2 < q.n_seg; ++s2) kb_total += q.seg[s2].kblocks;
      const int buf = ev % nacc;
      const uint32_t acc_phase = (uint32_t)(ev / nacc) & 1u;
      ++ev;
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
      if (!mbar_wait_cluster(tmem_empty(buf), acc_phase ^ 1u, &s_abort, P.hdr, 2)) break;
      tc_fence_after();
      uint32_t accumulate = 0;
      for (int kk = 0; kk < kb_total; ++kk) {
        if (!mbar_wait(full(stage), phase, &s_abort, P.hdr, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a1 = smem_u32(sA1(stage)), a3 = smem_u32(sA3(stage)),
                       b = smem_u32(sB(stage));
        // MN-major A (LBO: the two 64-feature atoms of bf16, SBO: 8-row k groups), K-major B;
        // every MMA consumes 32 bytes of each 128-byte row: 16 k of bf16 or 32 k of E4M3
        if constexpr (FP8) {
#pragma unroll
          for (int k32 = 0; k32 < BK8 / 32; ++k32) {
            const uint64_t bd = smem_desc(b + k32 * 32, 16, 1024);
            mma_e4m3_pair(d_tmem, smem_desc(a1 + k32 * 4096u, (uint32_t)A_HALF, 1024u), bd,
                          idesc, accumulate);
            mma_e4m3_pair(d_tmem + acc2, smem_desc(a3 + k32 * 4096u, (uint32_t)A_HALF, 1024u),
                          bd, idesc, accumulate);
            accumulate = 1;
          }
        } else {
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            const uint64_t bd = smem_desc(b + k16 * 32, 16, 1024);
            mma_bf16_pair(d_tmem, smem_desc(a1 + k16 * 2048u, (uint32_t)A_HALF, 1024u), bd,
                          idesc, accumulate);
            mma_bf16_pair(d_tmem + acc2, smem_desc(a3 + k16 * 2048u, (uint32_t)A_HALF, 1024u), bd,
                          idesc, accumulate);
            accumulate = 1;
          }
        }
        mma_commit_pair(empty(stage), 3);         // frees the stage in both CTAs
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      mma_commit_pair(tmem_full(buf), 3);
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // As in tc_gemm_kernel: warp w reads tensor-memory lanes 32*(w%4).. (its quadrant), the
    // warps of a quadrant take alternate 16-token chunks, transposed through a per-warp
    // shared-memory tile so that every lane writes whole 16-byte pieces of output rows.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    unsigned char* stg = epi_stage + (warp - 2) * EPI_STAGE_BYTES;
    float* stg_f = reinterpret_cast<float*>(stg);
    bf16* stg_h = reinterpret_cast<bf16*>(stg);
    // 16 token rows x 32 E4M3 codes of the transpose tile (byte j * 32 + lane = token j,
    // feature lane): lane -> (row lane / 2, 16-byte half lane % 2)
    auto store_e4m3_tile = [&](void* out, int64_t ld, int col0, const Item& it, int c0, int f0,
                               int M) {
      const int rows_here = min(16, it.nrows - c0);
      const int row = lane >> 1, part = lane & 1;
      if (f0 + part * 16 < M && row < rows_here) {
        const uint4 val = *reinterpret_cast<const uint4*>(stg + row * 32 + part * 16);
        const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 16;
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + o) = val;
      }
    };
    auto store_bf16_tile = [&](void* out, int64_t ld, int col0, const Item& it, int c0, int f0,
                               int M) {
      const int rows_here = min(16, it.nrows - c0);
      const int part = lane & 3;
      const bool ok = f0 + part * 8 < M;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = (lane >> 2) + 8 * r;
        if (ok && row < rows_here) {
          const uint4 val = *reinterpret_cast<const uint4*>(stg_h + row * 32 + part * 8);
          const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 8;
          *reinterpret_cast<uint4*>(static_cast<bf16*>(out) + o) = val;
        }
      }
    };
    // one 16-token x 32-feature chunk (lane = feature, v[j] = token c0 + j); kind 0 fp32, 1 bf16
    auto store_rows = [&](void* out, int64_t ld, int col0, int kind, const Item& it, int c0,
                          int f0, int M, const float* v) {
      if (kind == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) stg_f[j * 32 + lane] = v[j];
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) stg_h[j * 32 + lane] = __float2bfloat16_rn(v[j]);
      }
      __syncwarp();
      const int rows_here = min(16, it.nrows - c0);
      if (kind == 0) {
        const int part = lane & 7;
        const bool ok = f0 + part * 4 < M;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int row = (lane >> 3) + 4 * r;
          if (ok && row < rows_here) {
            const float4 val = *reinterpret_cast<const float4*>(stg_f + row * 32 + part * 4);
            const int64_t o = (it.row0 + c0 + row) * ld + col0 + f0 + part * 4;
            *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = val;
          }
        }
      } else {
        store_bf16_tile(out, ld, col0, it, c0, f0, M);
      }
      __syncwarp();
    };
    // releases rank 0's accumulator buffer (a remote arrive from rank 1)
    auto release = [&](int b) {
      tc_fence_before();
      mbar_arrive_cluster(mapa_shared(tmem_empty(b), 0));
    };
    int ev = 0;
    float amax = 0.0f;                                   // fp8 hidden: this thread's max |value|
    for (int64_t w = unit; w < total; w += n_units) {
      Item it = pair_decode(P, S, w);
      const TcProblem& q = P.p[it.p];
      const int buf = ev % nacc;
      const uint32_t acc_phase = (uint32_t)(ev / nacc) & 1u;
      ++ev;
      // fp8: dequantization factor of each accumulator of this CTA's features, fp32(1 /
      // activation scale) times the feature's weight scale in this expert (w, and w3 for the up
      // projection), loaded before the wait for the accumulator
      float sc1s[2] = {1.0f, 1.0f}, sc3s[2] = {1.0f, 1.0f}, osc = 1.0f;
      if constexpr (FP8) {
        const float da = __fdiv_rn(1.0f, *q.act_scale);
        const bool gl = is_glu(q.epi);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int f = (gl ? it.m0 + (int)rank * BM : it.m0 + (int)rank * 2 * BM + sub * BM) +
                        quad * 32 + lane;
          const bool fok = (sub == 0 || !gl) && f < q.M;
          const int64_t fs = (int64_t)it.wg * q.M + f;
          sc1s[sub] = fok ? __fmul_rn(da, q.w_scale[fs]) : 0.0f;
          sc3s[sub] = (fok && q.w3_scale) ? __fmul_rn(da, q.w3_scale[fs]) : 0.0f;
        }
        if (q.out_fp8) osc = *q.out_scale;
      }
      if (!mbar_wait(tmem_full(buf), acc_phase, &s_abort, P.hdr, 4)) break;
      tc_fence_after();
      const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN);
      if constexpr (FP8) {
        if (is_glu(q.epi)) {
          // E4M3 hidden of this CTA's 128 features: the SwiGLU of every chunk of this warp is
          // packed into registers, the accumulators released, then the codes written out
          constexpr int CPW = (BN / 16 + EPI_WARPS / 4 - 1) / (EPI_WARPS / 4);   // chunks per warp
          const int f0 = it.m0 + (int)rank * BM + quad * 32;
          const bool fok = f0 + lane < q.M;
          const float sc1 = sc1s[0], sc3 = sc3s[0];
          uint32_t pk[CPW][4];
#pragma unroll
          for (int i = 0; i < CPW; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
              float v[16], v3[16];
              tmem_ld16(lane_addr + c0, v);
              tmem_ld16(lane_addr + acc2 + c0, v3);
              tmem_wait_ld();
              const int valid = min(16, it.nrows - c0);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float h = swiglu(__fmul_rn(v[j], sc1), __fmul_rn(v3[j], sc3));
                if (fok && j < valid) amax = fmaxf(amax, fabsf(h));
                v[j] = __fmul_rn(h, osc);
              }
#pragma unroll
              for (int j = 0; j < 16; j += 4)
                pk[i][j / 4] = e4m3x2(v[j + 1], v[j]) | (e4m3x2(v[j + 3], v[j + 2]) << 16);
            }
          }
          release(buf);
          uint8_t* stg_b = reinterpret_cast<uint8_t*>(stg);
#pragma unroll
          for (int i = 0; i < CPW; ++i) {
            const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
            if (c0 < it.nrows) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                stg_b[j * 32 + lane] = (uint8_t)((pk[i][j / 4] >> (8 * (j % 4))) & 0xFFu);
              __syncwarp();
              store_e4m3_tile(q.out, q.ld_out, q.out_col0, it, c0, f0, q.M);
              __syncwarp();
            }
          }
          continue;
        }
      }
      if (is_glu(q.epi)) {
        // bf16 hidden of this CTA's 128 features: the SwiGLU of a warp's first CPR chunks is
        // packed into registers before the accumulators are released; chunks past those (tiles
        // of more than 192 tokens) are written out first, in place
        constexpr int CPW = (BN / 16 + EPI_WARPS / 4 - 1) / (EPI_WARPS / 4);   // chunks per warp
        constexpr int CPR = CPW < 4 ? CPW : 4;
        const int f0 = it.m0 + (int)rank * BM + quad * 32;
        for (int i = CPR; i < CPW; ++i) {
          const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
          if (c0 < it.nrows) {
            float v[16], v3[16];
            tmem_ld16(lane_addr + c0, v);
            tmem_ld16(lane_addr + acc2 + c0, v3);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = swiglu(v[j], v3[j]);
            store_rows(q.out, q.ld_out, q.out_col0, 1, it, c0, f0, q.M, v);
          }
        }
        uint32_t pk[CPR][8];
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
          const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
          if (c0 < it.nrows) {
            float v[16], v3[16];
            tmem_ld16(lane_addr + c0, v);
            tmem_ld16(lane_addr + acc2 + c0, v3);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(swiglu(v[j], v3[j]),
                                                              swiglu(v[j + 1], v3[j + 1]));
              pk[i][j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
          }
        }
        release(buf);
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
          const int c0 = half * 16 + i * 16 * (EPI_WARPS / 4);
          if (c0 < it.nrows) {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              stg_h[j * 32 + lane] = __ushort_as_bfloat16((unsigned short)(pk[i][j / 2] & 0xFFFFu));
              stg_h[(j + 1) * 32 + lane] = __ushort_as_bfloat16((unsigned short)(pk[i][j / 2] >> 16));
            }
            __syncwarp();
            store_bf16_tile(q.out, q.ld_out, q.out_col0, it, c0, f0, q.M);
            __syncwarp();
          }
        }
        continue;
      }
      // a dual item: this CTA holds features m0 + 256 rank .. (first accumulator) and .. + 128
      // (second)
      const bool f32out = (q.epi == EPI_F32);
      for (int sub = 0; sub < 2; ++sub) {
        const int f0 = it.m0 + (int)rank * 2 * BM + sub * BM + quad * 32;
        const uint32_t la = lane_addr + (uint32_t)sub * acc2;
        const float bias = (f32out && q.bias && f0 + lane < q.M) ? q.bias[f0 + lane] : 0.0f;
        const float sc = sub ? sc1s[1] : sc1s[0];
        for (int c0 = half * 16; c0 < it.nrows; c0 += 16 * (EPI_WARPS / 4)) {
          float v[16];
          tmem_ld16(la + c0, v);
          tmem_wait_ld();
          if (f32out) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fadd_rn(v[j], bias);
          }
          if constexpr (FP8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], sc);
          }
          store_rows(q.out, q.ld_out, q.out_col0, f32out ? 0 : 1, it, c0, f0, q.M, v);
        }
      }
      release(buf);
    }
    if (FP8 && P.amax) {
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
      if (lane == 0 && amax > 0.0f) amax_update(P.amax, amax);
    }
  }

  tc_fence_before();
  __syncthreads();
  // After a timeout, copies and MMAs either CTA issued may still be in flight: give them 20 ms
  // (they take microseconds) before either CTA frees its shared or tensor memory. Then neither
  // CTA leaves while the other can still signal its barriers.
  if (s_abort) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 20000000ull) __nanosleep(1000);
  }
  cluster_sync();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem_base)
                 : "memory");
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing arrives at, with
// the same routine the GEMM's roles use; it gives up after limit_ns and records
// MOE_ERR_DEVICE_TIMEOUT (detail 99) in the device report.
__global__ void bounded_wait_selftest_kernel(DeviceHeader* hdr, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(smem_u32(&bar), 0, &s_abort, hdr, 99, limit_ns);
  }
}

// ---- host side ----------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Weights [G, K, Mw] (Mw contiguous): 3-D map with a 64 x 64 x 1 box, 128-byte swizzle.
bool map_weights(CUtensorMap* m, const void* ptr, int64_t Mw, int64_t K, int64_t G) {
  cuuint64_t dims[3] = {(cuuint64_t)Mw, (cuuint64_t)K, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)(Mw * 2), (cuuint64_t)(Mw * K * 2)};
  cuuint32_t box[3] = {64, BK, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 weights [G, K, Mw] (Mw contiguous bytes): 3-D map with a 128 x 128 x 1 box (one 128-byte
// swizzle row of 128 features per k), 128-byte swizzle.
bool map_weights_fp8(CUtensorMap* m, const void* ptr, int64_t Mw, int64_t K, int64_t G) {
  cuuint64_t dims[3] = {(cuuint64_t)Mw, (cuuint64_t)K, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)Mw, (cuuint64_t)(Mw * K)};
  cuuint32_t box[3] = {128, BK8, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Transposed weights [G, Mw, K] (K contiguous): 3-D map with a 64 x 128 x 1 box, 128-byte swizzle
// (one K-major tile of 128 features by 64 k).
bool map_weights_kmajor(CUtensorMap* m, const void* ptr, int64_t Mw, int64_t K, int64_t G) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Mw, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)(K * 2), (cuuint64_t)(Mw * K * 2)};
  cuuint32_t box[3] = {BK, BM, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations [rows, K] (K contiguous): 2-D map with a box of one 128-byte swizzle row (64 bf16
// or 128 E4M3) by 32 rows, 128-byte swizzle.
bool map_act(CUtensorMap* m, const void* ptr, int64_t K, int64_t rows, bool fp8, int64_t ld = 0) {
  const int64_t es_bytes = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)((ld ? ld : K) * es_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)(fp8 ? BK8 : BK), B_BOX_ROWS};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_tc() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// Which launches use CTA pairs: by default every launch whose items all have two weight tiles
// (SwiGLU or dual) of bf16 forward problems, where pairs measured faster at every size on GB300
// (the 535B layer at T=8192: GEMM 1 2.31 -> 2.24 ms, GEMM 2 1.26 -> 1.18 ms, the back GEMM 0.60
// -> 0.50 ms). MOE_TC_PAIR in the environment selects none ("0"), launches with dual items only
// ("dual"), launches with SwiGLU items only ("glu") or all of them ("1", the default); no launch
// uses them once a query finds that no pair fits on the GPU.
enum PairMode { PAIR_NONE = 0, PAIR_ALL = 1, PAIR_DUAL = 2, PAIR_GLU = 3 };
std::atomic<int> g_pair_mode{-1};
int pair_mode() {
  int m = g_pair_mode.load(std::memory_order_relaxed);
  if (m < 0) {
    const char* e = getenv("MOE_TC_PAIR");
    m = PAIR_ALL;
    if (e && !strcmp(e, "0")) m = PAIR_NONE;
    else if (e && !strcmp(e, "dual")) m = PAIR_DUAL;
    else if (e && !strcmp(e, "glu")) m = PAIR_GLU;
    g_pair_mode.store(m, std::memory_order_relaxed);
  }
  return m;
}
void pair_disable() { g_pair_mode.store(PAIR_NONE, std::memory_order_relaxed); }

cudaLaunchConfig_t pair_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 2;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cfg;
}

// Pairs (clusters of two CTAs, one CTA per SM) of the pair kernel that fit on the GPU at once,
// cached per device: the persistent grid of a pair launch.
int max_pairs(void (*kern)(TcParams), dim3 block) {
  static std::mutex mu;
  static std::map<std::pair<int, void*>, int> cache;   // (device, kernel instance)
  int dev = 0;
  cudaGetDevice(&dev);
  const std::pair<int, void*> key(dev, reinterpret_cast<void*>(kern));
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR_SMEM_BUDGET) ==
      cudaSuccess) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(dim3(2), block, PAIR_SMEM_BUDGET, nullptr, false, attr);
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();   // a failed query leaves no error behind
  cache[key] = n;
  return n;
}

cudaError_t launch_pair(void (*kern)(TcParams), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t stream, bool pdl, const TcParams& P) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(grid, block, smem, stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

bool gemm_tc_supported(const GemmProblem& p) {
  if (p.dtype != DT_BF16) return false;
  const int Mw = (p.group == GROUP_COLS) ? p.Mg : p.M;
  if (Mw < 64 || (Mw % 8)) return false;
  if (p.group == GROUP_COLS && (p.Mg % BM || p.M % p.Mg)) return false;
  if (p.group == GROUP_ROWS && (p.G < 1 || p.G > MAX_GROUPS)) return false;
  if (p.n_seg < 1 || p.n_seg > GEMM_MAX_SEG) return false;
  for (int s = 0; s < p.n_seg; ++s)   // an activation row stride: 16-byte aligned, >= K
    if (p.seg[s].ld && (p.seg[s].ld < p.seg[s].K || (p.seg[s].ld % 8) || p.w_fp8)) return false;
  for (int s = 0; s < p.n_seg; ++s)
    if (p.seg[s].K < 8 || (p.seg[s].K % 8)) return false;
  if (p.epi < EPI_F32 || p.epi > EPI_SWIGLU_BWD) return false;
  if (p.epi == EPI_SWIGLU_SAVE || p.epi == EPI_SWIGLU_BWD) {
    if (p.w_fp8 || p.kchunk || !p.out2 || (p.epi == EPI_SWIGLU_SAVE && !p.out3)) return false;
    if (p.epi == EPI_SWIGLU_BWD && (!p.aux_g || !p.aux_u || p.ld_aux < p.M)) return false;
  }
  if (p.a_kmajor && (p.w_fp8 || p.kchunk || p.group == GROUP_COLS)) return false;
  // the epilogue writes 16-byte pieces of output rows
  if ((p.M % 8) || (p.ld_out % 8) || (p.out_col0 % 8)) return false;
  if (p.kchunk < 0) return false;
  if (p.kchunk > 0 && (p.epi != EPI_F32 || p.group != GROUP_NONE || p.n_seg != 1))
    return false;
  if (p.w_fp8) {
    const int Mw8 = (p.group == GROUP_COLS) ? p.Mg : p.M;
    if (Mw8 % BM || p.n_seg != 1 || p.kchunk || p.epi == EPI_F32 || !p.w_scale ||
        !p.act_scale || (p.epi == EPI_SWIGLU && !p.w3_scale) || (p.seg[0].K % 16))
      return false;
  }
  if (p.out_fp8 && (!p.w_fp8 || p.epi != EPI_SWIGLU || !p.out_scale || (p.M % 16) ||
                    (p.ld_out % 16) || (p.out_col0 % 16)))
    return false;
  if (p.cmb_seg >= 0) {   // a combine inside the launch: dense bf16, c written in place of act
    if (p.cmb_seg >= p.n_seg || p.group != GROUP_NONE || p.w_fp8 || p.a_kmajor || p.kchunk ||
        !p.cmb_y_perm || !p.cmb_slot || !p.cmb_gate || !p.cmb_ready || p.cmb_k < 1 ||
        p.cmb_k > 32 || p.seg[p.cmb_seg].ld || (p.seg[p.cmb_seg].K % 8))
      return false;
  }
  return true;
}

bool gemm_tc_pairs(const GemmProblem* probs, int n_probs) {
  const int pmode = pair_mode();
  if (pmode == PAIR_NONE || n_probs < 1 || n_probs > MAX_PROBS) return false;
  for (int j = 0; j < n_probs; ++j) {
    const GemmProblem& g = probs[j];
    if (!gemm_tc_supported(g) || g.w_fp8 || g.kchunk || g.a_kmajor || g.cmb_seg >= 0) return false;
    const int Mw = (g.group == GROUP_COLS) ? g.Mg : g.M;
    if (is_glu(g.epi)) {
      if (g.epi != EPI_SWIGLU || Mw % (2 * BM) || g.M % (2 * BM) || pmode == PAIR_DUAL) return false;
    } else {   // a dual item, as gemm_tc forms them
      if (g.group == GROUP_COLS || (g.epi != EPI_STORE && g.epi != EPI_F32) ||
          g.M % (4 * BM) || pmode == PAIR_GLU)
        return false;
    }
  }
  return true;
}

cudaError_t gemm_tc(const GemmProblem* probs, int n_probs, void* dev_header, cudaStream_t stream,
                    bool pdl) {
  if (n_probs < 1 || n_probs > MAX_PROBS) return cudaErrorInvalidValue;
  if (!encode_fn()) return cudaErrorNotSupported;
  static TcParams P;   // large; filled on the host for each launch (launches copy it)
  memset(&P, 0, sizeof(P));
  P.hdr = static_cast<DeviceHeader*>(dev_header);
  P.grouped = -1;
  // dense problems first, the (single) grouped problem last
  int order[MAX_PROBS], n = 0;
  for (int i = 0; i < n_probs; ++i) if (probs[i].group != GROUP_ROWS) order[n++] = i;
  for (int i = 0; i < n_probs; ++i) if (probs[i].group == GROUP_ROWS) order[n++] = i;
  int64_t base = 0;
  for (int j = 0; j < n_probs; ++j) {
    const GemmProblem& g = probs[order[j]];
    if (!gemm_tc_supported(g)) return cudaErrorNotSupported;
    if (g.group == GROUP_ROWS && j != n_probs - 1) return cudaErrorNotSupported;
    TcProblem& q = P.p[j];
    q.n_seg = g.n_seg;
    q.epi = g.epi;
    q.group = g.group;
    q.M = g.M;
    q.Mg = g.Mg;
    q.m_tiles = (int)cdiv(g.M, BM);
    q.n_fastest = (g.group != GROUP_ROWS);
    // two 128-feature tiles per item share one token tile: half the token-tile traffic and
    // twice the weight bytes in flight per stage
    q.kchunk = g.kchunk;
    q.bn = g.kchunk ? BN_CHUNKED : BN;
    // (for the backward's SwiGLU epilogue only on dense problems: on the grouped expert dA, which
    // streams its weights from HBM, its global loads of G and U are better hidden behind the next
    // item's main loop, which double-buffered accumulators allow; a dense dA is bound by the
    // operand ingest of single 128-feature items instead)
    q.dual = (!g.kchunk && !is_glu(g.epi) && g.group != GROUP_COLS && g.M % (2 * BM) == 0 &&
              (g.epi != EPI_SWIGLU_BWD || g.group == GROUP_NONE))
                 ? 1 : 0;
    if (q.dual) q.m_tiles = (int)(g.M / (2 * BM));
    q.rows = g.rows;
    q.out = g.out;
    q.ld_out = g.ld_out;
    q.out_col0 = g.out_col0;
    q.bias = g.bias;
    q.offsets = g.offsets;
    q.G = g.G;
    const int64_t Mw = (g.group == GROUP_COLS) ? g.Mg : g.M;
    const int64_t Gw = (g.group == GROUP_ROWS) ? g.G : (g.group == GROUP_COLS ? g.M / g.Mg : 1);
    q.w_scale = g.w_scale;
    q.w3_scale = g.w3_scale;
    q.act_scale = g.act_scale;
    q.a_kmajor = g.a_kmajor;
    q.out2 = g.out2;
    q.out3 = g.out3;
    q.aux_g = g.aux_g;
    q.aux_u = g.aux_u;
    q.ld_aux = g.ld_aux;
    q.out_fp8 = g.out_fp8;
    q.out_scale = g.out_scale;
    if (g.out_fp8) {
      if (P.amax && P.amax != g.amax) return cudaErrorNotSupported;   // one amax per launch
      P.amax = g.amax;
    }
    if (j == 0) P.fp8 = g.w_fp8 ? 1 : 0;
    if ((g.w_fp8 ? 1 : 0) != P.fp8) return cudaErrorNotSupported;   // all or none per launch
    for (int s = 0; s < g.n_seg; ++s) {
      const GemmSeg& sg = g.seg[s];
      TcSeg& ts = q.seg[s];
      ts.kblocks = (int)cdiv(sg.K, g.w_fp8 ? BK8 : BK);
      auto mapw = [&](CUtensorMap* m, const void* w) {
        if (g.w_fp8) return map_weights_fp8(m, w, Mw, sg.K, Gw);
        return g.a_kmajor ? map_weights_kmajor(m, w, Mw, sg.K, Gw) : map_weights(m, w, Mw, sg.K, Gw);
      };
      if (!mapw(&ts.a1, sg.w)) return cudaErrorInvalidValue;
      if (is_glu(g.epi) && !mapw(&ts.a3, sg.w3)) return cudaErrorInvalidValue;
      if (!map_act(&ts.b, sg.act, sg.K, g.rows, g.w_fp8 != 0, sg.ld)) return cudaErrorInvalidValue;
    }
    q.item_base = base;
    if (g.group == GROUP_ROWS) {
      P.grouped = j;
      q.n_items = 0;
    } else {
      q.n_items = q.m_tiles * cdiv(g.rows, q.bn);
      base += q.n_items;
    }
    if (is_glu(g.epi) || q.dual) P.glu = 1;
  }
  P.n_probs = n_probs;
  bool any_cmb = false;
  for (int j = 0; j < n_probs; ++j) any_cmb = any_cmb || probs[j].cmb_seg >= 0;
  if (any_cmb) {
    if (n_probs != 1) return cudaErrorNotSupported;   // the combine needs the launch to itself
    const GemmProblem& g = probs[0];
    P.cmb.active = 1;
    P.cmb.seg = g.cmb_seg;
    P.cmb.y_perm = static_cast<const bf16*>(g.cmb_y_perm);
    P.cmb.slot = g.cmb_slot;
    P.cmb.gate = g.cmb_gate;
    P.cmb.c = static_cast<bf16*>(const_cast<void*>(g.seg[g.cmb_seg].act));
    P.cmb.T = g.rows;
    P.cmb.k = g.cmb_k;
    P.cmb.L = g.seg[g.cmb_seg].K;
    P.cmb.pool_rows = g.cmb_pool_rows;
    P.cmb.ready = g.cmb_ready;
  }
  bool kc = false, bwd = false;
  for (int j = 0; j < n_probs; ++j) {
    kc = kc || P.p[j].kchunk > 0;
    bwd = bwd || P.p[j].a_kmajor || P.p[j].epi == EPI_SWIGLU_SAVE || P.p[j].epi == EPI_SWIGLU_BWD;
  }
  if (kc && bwd) return cudaErrorNotSupported;
  // CTA pairs (cta_group::2) for launches whose every item has two weight tiles: bf16, or E4M3
  // with an E4M3 hidden out of the SwiGLU GEMM and a bf16 output of the dual one
  const int pmode = pair_mode();
  bool pair = pmode != PAIR_NONE && !kc && !bwd && !P.cmb.active;
  for (int j = 0; j < n_probs; ++j) {
    const TcProblem& q = P.p[j];
    const int Mw = (q.group == GROUP_COLS) ? q.Mg : q.M;
    pair = pair && (P.fp8 ? (is_glu(q.epi) ? q.out_fp8 != 0 : q.out_fp8 == 0) : q.out_fp8 == 0);
    // a pair item spans 256 (SwiGLU) or 512 (dual) features, within one weight group
    pair = pair && (is_glu(q.epi) || q.dual) &&
           (q.epi == EPI_SWIGLU || q.epi == EPI_STORE || q.epi == EPI_F32) &&
           (is_glu(q.epi) ? (Mw % (2 * BM) == 0 && q.M % (2 * BM) == 0) : q.M % (4 * BM) == 0) &&
           !(pmode == PAIR_DUAL && is_glu(q.epi)) && !(pmode == PAIR_GLU && q.dual);
  }
  const dim3 block(64 + 32 * (P.fp8 ? Inst<true, false, false>::EW
                                    : (kc ? Inst<false, true, false>::EW
                                          : (bwd ? Inst<false, false, true>::EW
                                                 : Inst<false, false, false>::EW))));
  const int n_pairs =
      pair ? max_pairs(P.fp8 ? tc_gemm_pair_kernel<true> : tc_gemm_pair_kernel<false>, block) : 0;
  if (pair && n_pairs < 1) {   // no CTA pair fits: this and later launches run without pairs
    pair_disable();
    pair = false;
  }
  if (pair) {   // items of the pair width, and the dense problems' item ranges again
    int64_t pbase = 0;
    for (int j = 0; j < n_probs; ++j) {
      TcProblem& q = P.p[j];
      q.m_tiles = (int)(q.M / (q.dual ? 4 * BM : 2 * BM));
      q.item_base = pbase;
      if (q.group != GROUP_ROWS) {
        q.n_items = q.m_tiles * cdiv(q.rows, q.bn);
        pbase += q.n_items;
      }
    }
    base = pbase;
  }
  // Dense launches without fp32 k-chunked problems: choose the token tile height so that the
  // items fill whole waves of the persistent grid, by the estimate (waves rounded up) x height.
  // The back GEMM's 24 x 32 tiles of 256 rows are 5.05 waves on 152 SMs; 224-row tiles make
  // 888 items, 5.84 waves, for 12% less estimated time. A pair of SMs runs one item at a time.
  if (P.grouped < 0 && !kc) {
    const int64_t sms = pair ? n_pairs : num_sms_tc();
    int best_bn = BN;
    int64_t best_cost = -1;
    // heights in whole 32-row TMA boxes: the B slot of a stage holds max_bn rows
    for (int bn = BN; bn >= 160; bn -= B_BOX_ROWS) {
      int64_t items = 0;
      for (int j = 0; j < n_probs; ++j) items += (int64_t)P.p[j].m_tiles * cdiv(P.p[j].rows, bn);
      const int64_t cost = cdiv(items, sms) * bn;
      if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_bn = bn; }
    }
    base = 0;
    for (int j = 0; j < n_probs; ++j) {
      TcProblem& q = P.p[j];
      q.bn = best_bn;
      q.item_base = base;
      q.n_items = q.m_tiles * cdiv(q.rows, q.bn);
      base += q.n_items;
    }
  }
  // A launch of k-chunked problems only (the router's logits): the token tile height that
  // fills whole waves, by the same estimate, from 128 to BN_CHUNKED_MAX rows. The router of the
  // 535B layer at T=8192 has 3 x 64 items of 128 rows (1.26 waves on 152 SMs), or 3 x 43 of 192
  // (one wave), each item reading its whole K of both operands.
  bool kc_only = kc;
  for (int j = 0; j < n_probs; ++j) kc_only = kc_only && P.p[j].kchunk > 0;
  if (kc_only) {
    const int64_t sms = num_sms_tc();
    int best_bn = BN_CHUNKED;
    int64_t best_cost = -1;
    for (int bn = BN_CHUNKED; bn <= BN_CHUNKED_MAX; bn += B_BOX_ROWS) {
      int64_t items = 0;
      for (int j = 0; j < n_probs; ++j) items += (int64_t)P.p[j].m_tiles * cdiv(P.p[j].rows, bn);
      const int64_t cost = cdiv(items, sms) * bn;
      if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_bn = bn; }
    }
    base = 0;
    for (int j = 0; j < n_probs; ++j) {
      TcProblem& q = P.p[j];
      q.bn = best_bn;
      q.item_base = base;
      q.n_items = q.m_tiles * cdiv(q.rows, q.bn);
      base += q.n_items;
    }
  }
  // Dense problems walk their token tiles in bands of about DENSE_BAND_BYTES of activation rows
  // (all K segments), which stay in L2 while the band's weight tiles stream past them.
  for (int j = 0; j < n_probs; ++j) {
    TcProblem& q = P.p[j];
    q.band = 0;
    if (q.group == GROUP_ROWS || q.kchunk || !q.n_fastest) continue;
    int64_t row_bytes = 0;
    for (int s = 0; s < q.n_seg; ++s)
      row_bytes += (int64_t)q.seg[s].kblocks * (P.fp8 ? BK8 : 2 * BK);
    q.band = (int)imax64(1, DENSE_BAND_BYTES / ((int64_t)q.bn * row_bytes));
  }
  if (P.cmb.active) P.cmb.bn = P.p[0].bn;
  int max_bn = 0, max_two_a_bn = 0;
  for (int j = 0; j < n_probs; ++j) {
    max_bn = max(max_bn, P.p[j].bn);
    if (is_glu(P.p[j].epi) || P.p[j].dual) max_two_a_bn = max(max_two_a_bn, P.p[j].bn);
  }
  P.nacc = (max_two_a_bn > 128) ? 1 : 2;
  P.acc2_off = (max_two_a_bn > 128) ? BN : 128;
  // token rows of a stage's B slot (a pair CTA loads half of the 16-rounded tile), whole boxes
  const int64_t b_rows = pair ? cdiv(max_bn, 16) * 8 : max_bn;
  P.b_bytes = (int)cdiv(b_rows, B_BOX_ROWS) * B_BOX_BYTES;
  const int stage_bytes = (P.glu ? 2 * A_BYTES : A_BYTES) + P.b_bytes;
  // transpose tiles sized for the widest output of the launch
  P.epi_tile = 16 * 32 * 2;
  for (int j = 0; j < n_probs; ++j)
    if (P.p[j].epi == EPI_F32) P.epi_tile = EPI_TILE_MAX;
  const int ew = P.fp8 ? Inst<true, false, false>::EW
                       : (kc ? Inst<false, true, false>::EW
                             : (bwd ? Inst<false, false, true>::EW : Inst<false, false, false>::EW));
  const size_t epi_bytes = (size_t)ew * P.epi_tile;
  // as many stages as fit next to the epilogue tiles and the schedule (at most 8)
  {
    const size_t fixed = 1024 + epi_bytes +
                         (size_t)(3 * ((P.grouped >= 0) ? P.p[P.grouped].G : 0) + 1) * 4;
    const size_t budget = pair ? (size_t)PAIR_SMEM_BUDGET : (size_t)MOE_TC_SMEM_BUDGET;
    int st = (int)((budget - fixed) / (size_t)stage_bytes);
    P.stages = st < 2 ? 2 : (st > 8 ? 8 : st);
  }
  const int G = (P.grouped >= 0) ? P.p[P.grouped].G : 0;
  const size_t smem = (size_t)P.stages * stage_bytes + 1024 +
                      epi_bytes + (size_t)(3 * G + 1) * 4;
  auto kern = pair ? (P.fp8 ? tc_gemm_pair_kernel<true> : tc_gemm_pair_kernel<false>)
             : P.cmb.active ? tc_gemm_kernel<false, false, false, true>
             : P.fp8 ? tc_gemm_kernel<true, false, false>
                     : (kc ? tc_gemm_kernel<false, true, false>
                           : (bwd ? tc_gemm_kernel<false, false, true>
                                  : tc_gemm_kernel<false, false, false>));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (pair) {
    int units = n_pairs;
    if (P.grouped < 0) units = (int)imin64(units, base);
    if (units < 1) return cudaSuccess;
    return launch_pair(kern, dim3(2 * units), block, smem, stream, pdl, P);
  }
  int grid = num_sms_tc();
  if (P.grouped < 0) grid = (int)imin64(grid, base);
  if (grid < 1) return cudaSuccess;
  return launch(kern, dim3(grid), block, smem, stream, pdl, P);
}

cudaError_t bounded_wait_selftest(void* dev_header, uint64_t limit_ns, cudaStream_t stream) {
  return launch(bounded_wait_selftest_kernel, dim3(1), dim3(32), 0, stream, false,
                static_cast<DeviceHeader*>(dev_header), limit_ns);
}

}  // namespace moe
