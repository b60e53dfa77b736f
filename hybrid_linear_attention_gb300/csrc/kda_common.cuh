// kda_common.cuh -- small device helpers shared by the KDA kernels (sm_103a only).
#pragma once

#include "kda_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace kda {

typedef __nv_bfloat16 bf16;

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), looked up once through the
// runtime; nullptr when the driver does not provide it.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// Sticky device error bits (written by kernels whose bounded waits ran out).
// device error flag bits (ERR_*): kda_internal.h

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ bf16 from_f<bf16>(float x) {
  return __float2bfloat16_rn(x);
}

// Four consecutive elements <-> float4 (16-byte fp32 or 8-byte bf16 accesses).
__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void store4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// The same four-element accesses with streaming cache hints (evict-first loads, streaming
// stores): for data touched once, such as a state streamed through once per step, so that it
// does not push out of L2 what is still to be read (the next units' prefetched state).
__device__ __forceinline__ float4 load4_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4_stream(const bf16* p) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4_stream(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}
__device__ __forceinline__ void store4_stream(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  __stcs(reinterpret_cast<uint2*>(p), u);
}

// Two consecutive elements <-> float2.
__device__ __forceinline__ float2 load2(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float2 load2(const bf16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void store2(float* p, float2 v) {
  *reinterpret_cast<float2*>(p) = v;
}
__device__ __forceinline__ void store2(bf16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x * sigmoidf_(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Dynamic FP8 quantisation of one output group (the d_v values of one token and head, which
// meet one 128-row block of o_proj's block-FP8 weight): with a = max(amax, 1e-10), the fp32
// scale o_proj multiplies back is a / 448, and code = E4M3 of x * (448 / a), rounded to
// nearest even and saturated at +-448.  The divisions (once per group) and the product are
// IEEE round-to-nearest, so the codes are a function of the fp32 values alone.
constexpr float FP8_MAX = 448.f, FP8_EPS = 1e-10f;
__device__ __forceinline__ float fp8_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, FP8_EPS), FP8_MAX);
}
__device__ __forceinline__ float fp8_inv_scale(float amax) {
  return __fdiv_rn(FP8_MAX, fmaxf(amax, FP8_EPS));
}
__device__ __forceinline__ uint8_t fp8_code(float x, float inv_scale) {
  return (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(x, inv_scale), __NV_SATFINITE, __NV_E4M3);
}

// Sequence containing packed token t: the largest n with cu[n] <= t (empty sequences
// share their offset with the next one, so this lands on the non-empty owner).
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int n_seqs, int64_t t) {
  int lo = 0, hi = n_seqs;  // answer in [0, n_seqs)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace kda
