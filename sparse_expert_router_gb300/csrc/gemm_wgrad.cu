// tcgen05 weight-gradient GEMM over ragged row groups, for the backward of the grouped expert
// MLP: dW_e = X_e^T dY_e, where the contraction runs over the rows of expert e. The Marin
// summary of the week of 2026-07-06 (#5330) describes this as the ragged-contracting-dimension
// kernel of the ragged dot's custom VJP.
//
// Both operands are MN-major in shared memory: the contraction index is their row index, so a
// k step holds 64 rows of a (two 64-feature boxes, 128 features) and of b (four 64-column boxes,
// 256 columns). A group's rows start anywhere; its last k step may run past the group's end, so
// the MMA warp zeroes the rows past the end in both tiles before it issues that step's MMAs.
//
// Work units are (problem, group, 256-column n tile, chunk of mc 128-row m tiles). The b tile of
// a unit is the same for all its m tiles: when the group has at most WB_SLOTS * 64 rows it is
// loaded once into the b slots and stays there for the whole unit, and only the a tiles stream
// through their own ring (for an expert of 171 rows and mc = 24 this is 52 KB of operands per
// 64 KB of output instead of 144 KB). Larger groups stream b through the same slots, one load per
// m tile and k step. A launch whose problems are all single groups (the dense weight gradients)
// streams both tiles as one stage: a stage s and b slot s filled under one barrier.
//
// Roles of the warps of a CTA (one CTA per SM, persistent over units, n tiles fastest so the
// units of one group run together and share its rows in L2):
//   warp 0: TMA producer (one thread); warp 1: TMEM allocator and MMA issuer (the whole warp
//   zeroes tail rows, one thread issues MMAs); warps 2..9: epilogue, the two warps of a lane
//   quadrant each taking half of the 256 columns, 64 per tensor-memory load, and each thread
//   writing its row's 64 values into a 128-byte-swizzled shared tile that one TMA bulk tensor
//   store then copies out (whole 128-byte lines, no scattered stores). Accumulators are
//   double-buffered (2 x 256 tensor-memory columns), one per m tile. Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "wgrad.h"

namespace moe {
namespace {

using namespace tc;

constexpr int WM = 128;              // output rows (features of a) per m tile: MMA M, TMEM lanes
constexpr int WN = 256;              // output columns per unit: MMA N
constexpr int WK = 64;               // contraction rows per k step
constexpr int W_EPI = 8;             // epilogue warps
constexpr int W_THREADS = 64 + 32 * W_EPI;
constexpr int WA_HALF = 64 * WK * 2; // one [64 rows][64 features] box: 8 KB
constexpr int WA_BYTES = 2 * WA_HALF;
constexpr int WB_ATOM = 64 * WK * 2; // one [64 rows][64 columns] box: 8 KB
constexpr int WB_BYTES = 4 * WB_ATOM;
constexpr int WA_STAGES = 4;         // a ring
constexpr int WB_SLOTS = 4;          // b slots: groups of at most 256 rows keep b resident
constexpr int W_MAX_PROBS = 6;
constexpr int W_OUT_TILE = 32 * 64 * 2;   // one warp's store tile: 32 rows x 64 bf16 columns
constexpr int W_SMEM = WB_SLOTS * WB_BYTES + WA_STAGES * WA_BYTES + W_EPI * W_OUT_TILE;
static_assert(WA_STAGES == WB_SLOTS, "one-ring launches pair a stage s with b slot s");

struct WgProb {
  CUtensorMap a, b, o;
  const int32_t* offsets;
  int G, M, N, m_tiles, n_tiles;
  int mc, m_chunks;                  // m tiles per unit, units per (group, n tile)
  int64_t rows;
  bf16* out;
  int64_t item_base;
};

struct WgParams {
  WgProb p[W_MAX_PROBS];
  int n_probs;
  // every problem is one group: no unit keeps b resident, and each k step's a and b tiles share
  // one stage (a stage s, b slot s) and one barrier, as in a plain streamed GEMM
  int one_ring;
  int64_t total;
  DeviceHeader* hdr;
};

struct WUnit {
  int p, g, n0, mt0, nmt;
  int64_t lo, hi;   // the group's rows
};

__device__ __forceinline__ WUnit wdecode(const WgParams& P, int64_t w) {
  WUnit u;
  int p = 0;
  while (p + 1 < P.n_probs && w >= P.p[p + 1].item_base) ++p;
  const WgProb& q = P.p[p];
  const int64_t local = w - q.item_base;
  const int per_group = q.n_tiles * q.m_chunks;
  u.p = p;
  u.g = (int)(local / per_group);
  const int rem = (int)(local % per_group);
  u.n0 = (rem % q.n_tiles) * WN;
  u.mt0 = (rem / q.n_tiles) * q.mc;
  u.nmt = q.mc;
  const int64_t lo = imin64(imax64(q.offsets[u.g], 0), q.rows);
  u.lo = lo;
  u.hi = imin64(imax64(q.offsets[u.g + 1], lo), q.rows);
  return u;
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, both MN-major (transposed), N, M=128.
__device__ __forceinline__ uint32_t wg_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
         ((uint32_t)(WN >> 3) << 17) | ((uint32_t)(WM >> 4) << 24);
}

__global__ void __launch_bounds__(W_THREADS, 1) wgrad_kernel(const __grid_constant__ WgParams P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * WA_STAGES + 2 * WB_SLOTS + 4];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // a stage s and b slot s side by side (48 KB per pair): measured faster than two separate
  // regions, for both the resident and the streamed schedule
  auto sA = [&](int s) { return base + s * (WA_BYTES + WB_BYTES); };
  auto sB = [&](int s) { return base + s * (WA_BYTES + WB_BYTES) + WA_BYTES; };
  auto a_full = [&](int s) { return smem_u32(&bars[s]); };
  auto a_empty = [&](int s) { return smem_u32(&bars[WA_STAGES + s]); };
  auto b_full = [&](int s) { return smem_u32(&bars[2 * WA_STAGES + s]); };
  auto b_empty = [&](int s) { return smem_u32(&bars[2 * WA_STAGES + WB_SLOTS + s]); };
  auto tmem_full = [&](int b) { return smem_u32(&bars[2 * WA_STAGES + 2 * WB_SLOTS + b]); };
  auto tmem_empty = [&](int b) { return smem_u32(&bars[2 * WA_STAGES + 2 * WB_SLOTS + 2 + b]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < WA_STAGES; ++s) { mbar_init(a_full(s), 1); mbar_init(a_empty(s), 1); }
    for (int s = 0; s < WB_SLOTS; ++s) { mbar_init(b_full(s), 1); mbar_init(b_empty(s), 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(tmem_full(b), 1); mbar_init(tmem_empty(b), 32 * W_EPI); }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int p = 0; p < P.n_probs; ++p) { prefetch_map(&P.p[p].a); prefetch_map(&P.p[p].b); }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // every thread waits for the kernel that wrote the group offsets and the operands
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int as = 0;
    uint32_t aph = 0;
    uint32_t bl = 0;         // b loads issued: slot bl % WB_SLOTS, phase (bl / WB_SLOTS) & 1
    bool ok = true;
    auto load_b = [&](const WgProb& q, int n0, int64_t r0) {
      const int slot = (int)(bl % WB_SLOTS);
      const uint32_t ph = (bl / WB_SLOTS) & 1u;
      ++bl;
      if (!mbar_wait(b_empty(slot), ph ^ 1u, &s_abort, P.hdr, 15)) return false;
      mbar_expect_tx(b_full(slot), (uint32_t)WB_BYTES);
      const uint32_t b = smem_u32(sB(slot));
#pragma unroll
      for (int i = 0; i < 4; ++i)
        tma_load_2d(b + i * WB_ATOM, &q.b, b_full(slot), n0 + 64 * i, (int)r0);
      return true;
    };
    for (int64_t w = blockIdx.x; w < P.total && ok; w += gridDim.x) {
      const WUnit u = wdecode(P, w);
      if (u.hi <= u.lo) continue;
      const WgProb& q = P.p[u.p];
      if (P.one_ring) {
        // a stage s and b slot s filled together under one barrier
        for (int j = 0; j < u.nmt && ok; ++j) {
          const int m0 = (u.mt0 + j) * WM;
          for (int64_t r0 = u.lo; r0 < u.hi; r0 += WK) {
            if (!mbar_wait(a_empty(as), aph ^ 1u, &s_abort, P.hdr, 11)) { ok = false; break; }
            mbar_expect_tx(a_full(as), (uint32_t)(WA_BYTES + WB_BYTES));
            const uint32_t a = smem_u32(sA(as)), b = smem_u32(sB(as));
            tma_load_2d(a, &q.a, a_full(as), m0, (int)r0);
            tma_load_2d(a + WA_HALF, &q.a, a_full(as), m0 + 64, (int)r0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              tma_load_2d(b + i * WB_ATOM, &q.b, a_full(as), u.n0 + 64 * i, (int)r0);
            if (++as == WA_STAGES) { as = 0; aph ^= 1u; }
          }
        }
        continue;
      }
      const int nk = (int)((u.hi - u.lo + WK - 1) / WK);
      const bool resident = nk <= WB_SLOTS;
      if (resident)
        for (int k = 0; k < nk && ok; ++k) ok = load_b(q, u.n0, u.lo + (int64_t)k * WK);
      for (int j = 0; j < u.nmt && ok; ++j) {
        const int m0 = (u.mt0 + j) * WM;
        for (int k = 0; k < nk; ++k) {
          const int64_t r0 = u.lo + (int64_t)k * WK;
          if (!resident && !(ok = load_b(q, u.n0, r0))) break;
          if (!mbar_wait(a_empty(as), aph ^ 1u, &s_abort, P.hdr, 11)) { ok = false; break; }
          mbar_expect_tx(a_full(as), (uint32_t)WA_BYTES);
          const uint32_t a = smem_u32(sA(as));
          tma_load_2d(a, &q.a, a_full(as), m0, (int)r0);
          tma_load_2d(a + WA_HALF, &q.a, a_full(as), m0 + 64, (int)r0);
          if (++as == WA_STAGES) { as = 0; aph ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp: tail zeroing) ----------------
    const uint32_t idesc = wg_idesc();
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    // Rows of the group in a k step: MMAs only for the 16-row slices holding some of them. Rows
    // past the group's end belong to the next group (or are padding); the ones inside the last
    // slice are zeroed in the a tile and, when it was just loaded, the b tile. A row is one
    // 128-byte line per 64-wide box (swizzling permutes 16-byte pieces within the line only).
    auto zero_tail = [&](unsigned char* ta, unsigned char* tb, int valid, int zr) {
      ta += valid * 128;
      for (int i = lane; i < zr * 16; i += 32)     // zr rows x 2 boxes x 8 pieces
        *reinterpret_cast<uint4*>(ta + ((i >> 3) & 1) * WA_HALF + (i >> 4) * 128 + (i & 7) * 16) = z;
      if (tb) {
        tb += valid * 128;
        for (int i = lane; i < zr * 32; i += 32)   // zr rows x 4 boxes x 8 pieces
          *reinterpret_cast<uint4*>(tb + ((i >> 3) & 3) * WB_ATOM + (i >> 5) * 128 + (i & 7) * 16) = z;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    };
    auto issue = [&](uint32_t d_tmem, uint32_t a, uint32_t b, int nk16, uint32_t& accumulate) {
#pragma unroll
      for (int k16 = 0; k16 < WK / 16; ++k16) {
        if (k16 < nk16) {
          mma_bf16(d_tmem, smem_desc(a + k16 * 2048, WA_HALF, 1024),
                   smem_desc(b + k16 * 2048, WB_ATOM, 1024), idesc, accumulate);
          accumulate = 1;
        }
      }
    };
    int as = 0;
    uint32_t aph = 0;
    int ev = 0;
    bool ok = true;
    if (P.one_ring) {
      // single-group problems: a stage s and b slot s under one barrier
      for (int64_t w = blockIdx.x; w < P.total && ok; w += gridDim.x) {
        const WUnit u = wdecode(P, w);
        if (u.hi <= u.lo) continue;
        for (int j = 0; j < u.nmt && ok; ++j) {
          const int buf = ev & 1;
          const uint32_t acc_phase = (uint32_t)(ev >> 1) & 1u;
          ++ev;
          ok = mbar_wait(tmem_empty(buf), acc_phase ^ 1u, &s_abort, P.hdr, 12);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * WN);
          uint32_t accumulate = 0;
          for (int64_t r0 = u.lo; r0 < u.hi; r0 += WK) {
            ok = mbar_wait(a_full(as), aph, &s_abort, P.hdr, 13);
            if (!__all_sync(~0u, ok)) { ok = false; break; }
            tc_fence_after();
            const int valid = (int)imin64(WK, u.hi - r0);
            const int nk16 = (valid + 15) >> 4;
            const int zr = (nk16 << 4) - valid;
            if (zr > 0) zero_tail(sA(as), sB(as), valid, zr);
            if (lane == 0) {
              issue(d_tmem, smem_u32(sA(as)), smem_u32(sB(as)), nk16, accumulate);
              mma_commit(a_empty(as));
            }
            __syncwarp();
            if (++as == WA_STAGES) { as = 0; aph ^= 1u; }
          }
          if (!ok) break;
          if (lane == 0) mma_commit(tmem_full(buf));
          __syncwarp();
        }
      }
    } else {
      uint32_t bl = 0;
      for (int64_t w = blockIdx.x; w < P.total && ok; w += gridDim.x) {
        const WUnit u = wdecode(P, w);
        if (u.hi <= u.lo) continue;                     // empty group: the epilogue writes zeros
        const int nk = (int)((u.hi - u.lo + WK - 1) / WK);
        const bool resident = nk <= WB_SLOTS;
        const uint32_t b0 = bl;
        for (int j = 0; j < u.nmt && ok; ++j) {
          const int buf = ev & 1;
          const uint32_t acc_phase = (uint32_t)(ev >> 1) & 1u;
          ++ev;
          ok = mbar_wait(tmem_empty(buf), acc_phase ^ 1u, &s_abort, P.hdr, 12);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * WN);
          uint32_t accumulate = 0;
          for (int k = 0; k < nk; ++k) {
            const uint32_t bidx = resident ? b0 + (uint32_t)k : bl++;
            const int slot = (int)(bidx % WB_SLOTS);
            const bool fresh = !resident || j == 0;      // b slot loaded for this use
            const bool last_use = !resident || j == u.nmt - 1;
            ok = mbar_wait(b_full(slot), (bidx / WB_SLOTS) & 1u, &s_abort, P.hdr, 16);
            if (ok) ok = mbar_wait(a_full(as), aph, &s_abort, P.hdr, 13);
            if (!__all_sync(~0u, ok)) { ok = false; break; }
            tc_fence_after();
            const int valid = (int)imin64(WK, u.hi - (u.lo + (int64_t)k * WK));
            const int nk16 = (valid + 15) >> 4;
            const int zr = (nk16 << 4) - valid;
            if (zr > 0) zero_tail(sA(as), fresh ? sB(slot) : nullptr, valid, zr);
            if (lane == 0) {
              issue(d_tmem, smem_u32(sA(as)), smem_u32(sB(slot)), nk16, accumulate);
              mma_commit(a_empty(as));
              if (last_use) mma_commit(b_empty(slot));
            }
            __syncwarp();
            if (++as == WA_STAGES) { as = 0; aph ^= 1u; }
          }
          if (!ok) break;
          if (lane == 0) mma_commit(tmem_full(buf));
          __syncwarp();
        }
        if (resident) bl = b0 + (uint32_t)nk;
      }
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // Warp w reads tensor-memory lanes 32*(w%4).. (its quadrant); the two warps of a quadrant
    // take the two halves of the columns.
    const int quad = warp & 3, half = (warp - 2) >> 2;
    unsigned char* otile = base + WB_SLOTS * WB_BYTES + WA_STAGES * WA_BYTES +
                           (warp - 2) * W_OUT_TILE;
    int ev = 0;
    bool ok = true;
    for (int64_t w = blockIdx.x; w < P.total && ok; w += gridDim.x) {
      const WUnit u = wdecode(P, w);
      const WgProb& q = P.p[u.p];
      for (int j = 0; j < u.nmt; ++j) {
        const int m0 = (u.mt0 + j) * WM;
        const int m = m0 + quad * 32 + lane;
        bf16* orow = q.out + ((int64_t)u.g * q.M + m) * q.N;
        const bool mok = m < q.M;
        if (u.hi <= u.lo) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int c0 = half * (WN / 2); c0 < (half + 1) * (WN / 2); c0 += 64) {
            const int n = u.n0 + c0;
            if (mok && n < q.N) {
#pragma unroll
              for (int p8 = 0; p8 < 8; ++p8) *reinterpret_cast<uint4*>(orow + n + 8 * p8) = z;
            }
          }
          continue;
        }
        const int buf = ev & 1;
        const uint32_t acc_phase = (uint32_t)(ev >> 1) & 1u;
        ++ev;
        if (!mbar_wait(tmem_full(buf), acc_phase, &s_abort, P.hdr, 14)) { ok = false; break; }
        tc_fence_after();
        const uint32_t lane_addr =
            tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * WN);
        // this warp's half of the columns, 64 at a time: one tensor-memory load and one wait per
        // 64 columns; each thread puts its row's 128 bytes into the shared tile in the 128-byte
        // swizzle (16-byte piece p of row r at piece p ^ (r % 8)), then one bulk tensor store
        for (int c0 = half * (WN / 2); c0 < (half + 1) * (WN / 2); c0 += 64) {
          float v[64];
          tmem_ld64(lane_addr + c0, v);
          tmem_wait_ld();
          const int n = u.n0 + c0;
          if (n < q.N) {
            if (lane == 0) bulk_wait_read0();       // the tile's previous store has read it
            __syncwarp();
#pragma unroll
            for (int p8 = 0; p8 < 8; ++p8) {
              uint4 pk;
              __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                h[i] = __floats2bfloat162_rn(v[8 * p8 + 2 * i], v[8 * p8 + 2 * i + 1]);
              *reinterpret_cast<uint4*>(otile + lane * 128 + ((p8 ^ (lane & 7)) << 4)) = pk;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tma_store_2d(&q.o, smem_u32(otile), n, u.g * q.M + m0 + quad * 32);
          }
        }
        tc_fence_before();
        mbar_arrive(tmem_empty(buf));
      }
    }
    if (lane == 0) bulk_wait0();                 // every store of this warp has completed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base)
                 : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 wg_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult qr;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, cols] bf16 row-major as an MN-major operand: 64 columns (one 128-byte swizzle row) by
// 64 rows per box.
bool map_mn(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, int64_t ld) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)((ld ? ld : cols) * 2)};
  cuuint32_t box[2] = {64, WK};
  cuuint32_t es[2] = {1, 1};
  return wg_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output [G * M rows, N] bf16 for bulk tensor stores: 64 columns by 32 rows per box,
// 128-byte swizzle (the layout the epilogue writes its shared tile in).
bool map_out(CUtensorMap* m, void* ptr, int64_t cols, int64_t rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t es[2] = {1, 1};
  return wg_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_wgrad_supported(const WgradProblem& p) {
  return p.a && p.b && p.offsets && p.out && p.G >= 1 && p.M >= WM && p.M % WM == 0 &&
         p.N >= 64 && p.N % 64 == 0 && p.rows >= 0 && p.rows < (1ll << 31) &&
         (p.lda == 0 || (p.lda >= p.M && p.lda % 8 == 0)) &&
         (p.ldb == 0 || (p.ldb >= p.N && p.ldb % 8 == 0));
}

cudaError_t gemm_wgrad(const WgradProblem* probs, int n_probs, void* dev_header,
                       cudaStream_t stream, bool pdl) {
  if (n_probs < 1 || n_probs > W_MAX_PROBS) return cudaErrorInvalidValue;
  if (!wg_encode_fn()) return cudaErrorNotSupported;
  static WgParams P;
  memset(&P, 0, sizeof(P));
  P.hdr = static_cast<DeviceHeader*>(dev_header);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  int64_t base = 0;
  for (int j = 0; j < n_probs; ++j) {
    const WgradProblem& g = probs[j];
    if (!gemm_wgrad_supported(g)) return cudaErrorNotSupported;
    WgProb& q = P.p[j];
    const int64_t rows = g.rows > 0 ? g.rows : 1;
    if (!map_mn(&q.a, g.a, g.M, rows, g.lda) || !map_mn(&q.b, g.b, g.N, rows, g.ldb) ||
        !map_out(&q.o, g.out, g.N, (int64_t)g.G * g.M))
      return cudaErrorInvalidValue;
    q.offsets = g.offsets;
    q.G = g.G;
    q.M = g.M;
    q.N = g.N;
    q.m_tiles = g.M / WM;
    q.n_tiles = (int)cdiv(g.N, WN);
    // m tiles per unit: as many as keep at least 8 units per SM (a resident b tile then serves
    // them all), one when even that leaves fewer units
    q.mc = 1;
    for (int mc = q.m_tiles; mc > 1; --mc)
      if (q.m_tiles % mc == 0 && (int64_t)g.G * q.n_tiles * (q.m_tiles / mc) >= 8ll * sms) {
        q.mc = mc;
        break;
      }
    q.m_chunks = q.m_tiles / q.mc;
    q.rows = g.rows;
    q.out = static_cast<bf16*>(g.out);
    q.item_base = base;
    base += (int64_t)g.G * q.n_tiles * q.m_chunks;
  }
  P.n_probs = n_probs;
  P.total = base;
  P.one_ring = 1;
  for (int j = 0; j < n_probs; ++j) P.one_ring &= (probs[j].G == 1) ? 1 : 0;
  const size_t smem = (size_t)W_SMEM + 1024;
  cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)imin64(sms, base);
  if (grid < 1) return cudaSuccess;
  return launch(wgrad_kernel, dim3(grid), dim3(W_THREADS), smem, stream, pdl, P);
}

}  // namespace moe
