// Shared device/host helpers of the GB300 routed-MoE library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// The device report lives at the start of every workspace (256 bytes).
struct DeviceHeader {
  int32_t status;      // first device-detected moe_status_t
  int32_t detail;
  int32_t n_refine;    // ambiguous-token list length (router stage 2)
  int32_t n_exact;     // exact-token list length (router stage 3)
  uint32_t amax_x;     // fp8 experts: bits of max |row| quantized by the gather (fp32, >= 0)
  uint32_t amax_h;     // fp8 experts: bits of max |hidden| quantized by expert GEMM 1
  uint32_t dispatch_ticket;   // blocks of the dispatch scan that have finished (reset per call)
  int32_t reserved[57];
};
static_assert(sizeof(DeviceHeader) == 256, "header is 256 bytes");

__device__ __forceinline__ void report_error(DeviceHeader* h, int code, int detail) {
  if (atomicCAS(&h->status, 0, code) == 0) atomicExch(&h->detail, detail);
}

// ---- element access ------------------------------------------------------------------
__device__ __forceinline__ float ld_f(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const bf16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_f(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_f(bf16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// 8 consecutive elements <-> floats (16-byte bf16 or 2 x 16-byte fp32 accesses).
__device__ __forceinline__ void ld8(const bf16* p, float v[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(b[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void ld8(const float* p, float v[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(bf16* p, const float v[8]) {
  uint4 u;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
// An FP8 E4M3 code (sign, 4 exponent bits with bias 7, 3 fraction bits; largest finite 448).
struct e4m3 {
  uint8_t bits;
};
// Two fp32 values to two E4M3 codes, round to nearest even, saturating at +-448; `hi` goes to
// the upper byte.
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Eight values (already multiplied by their quantization scale) to eight codes, one 8-byte store.
__device__ __forceinline__ void st8(e4m3* p, const float v[8]) {
  uint2 u;
  u.x = e4m3x2(v[1], v[0]) | (e4m3x2(v[3], v[2]) << 16);
  u.y = e4m3x2(v[5], v[4]) | (e4m3x2(v[7], v[6]) << 16);
  *reinterpret_cast<uint2*>(p) = u;
}
// Running maximum of non-negative fp32 values kept as their bit patterns (monotone for >= 0).
__device__ __forceinline__ void amax_update(uint32_t* dst, float m) {
  atomicMax(dst, __float_as_uint(m));
}
__device__ __forceinline__ void st8(float* p, const float v[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// silu(u) * v for a hidden stored in bf16 or E4M3. The exponential and the division are the
// hardware approximations __expf (at most 2 + floor(1.173 |u|) ulp) and __fdividef (2 ulp),
// about 2e-6 relative for |u| <= 10: three orders of magnitude below the 2^-9 rounding of the
// bf16 hidden. The approximate fused SwiGLU of the Marin summary for the week of 2026-07-06
// (#7024) caused a ~2.6% output mismatch, an error at the scale of the stored precision.
__device__ __forceinline__ float swiglu(float u, float v) {
  return __fdividef(u, 1.0f + __expf(-u)) * v;
}
// The same for an fp32 hidden (the fp32 layer): accurate exponential and IEEE division.
__device__ __forceinline__ float swiglu_ieee(float u, float v) {
  return __fdiv_rn(u, 1.0f + expf(-u)) * v;
}
// sigmoid(g) for the SwiGLU backward of a bf16 hidden, with the same approximations as swiglu.
__device__ __forceinline__ float sigmoid_bf16(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// ---- programmatic dependent launch ----------------------------------------------------
// Every thread of a consumer kernel executes pdl_wait() before it reads anything a preceding
// kernel wrote (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

// Element type tag for host dispatch.
enum DType { DT_BF16 = 0, DT_F32 = 1 };

// ---- host-side launch helper ----------------------------------------------------------
// Launches `kernel` with optional programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
