// Device helpers shared by the CSA kernels: storage-dtype conversion, vector
// loads, RoPE angles, block reductions.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

// ---------------------------------------------------------------- dtype
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// value of x once stored in T (round to nearest even)
template <typename T> __device__ __forceinline__ float rnd(float x) { return to_f(from_f<T>(x)); }

// 8 consecutive elements -> fp32 (16-byte aligned source)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* o) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8_nc(const __nv_bfloat16* p, float* o) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_nc(const float* p, float* o) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// copy 8 elements (16 B for bf16, 32 B for f32)
template <typename T> __device__ __forceinline__ void copy8(T* dst, const T* src);
template <> __device__ __forceinline__ void copy8<__nv_bfloat16>(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}
template <> __device__ __forceinline__ void copy8<float>(float* dst, const float* src) {
  reinterpret_cast<float4*>(dst)[0] = reinterpret_cast<const float4*>(src)[0];
  reinterpret_cast<float4*>(dst)[1] = reinterpret_cast<const float4*>(src)[1];
}
template <typename T> __device__ __forceinline__ void zero8(T* dst);
template <> __device__ __forceinline__ void zero8<__nv_bfloat16>(__nv_bfloat16* dst) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
}
template <> __device__ __forceinline__ void zero8<float>(float* dst) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  reinterpret_cast<float4*>(dst)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------- packed variable-length batches
// The tokens (queries) of B sequences packed back to back: sequence b owns rows [cu[b], cu[b+1]) of every packed
// tensor (cu: [B + 1] device int32, cu[0] = 0, non-decreasing, cu[B] = N).  The sequence of row q is the last b
// with cu[b] <= q (an empty sequence is passed over); the result is always in [0, B).
__device__ __forceinline__ int varlen_seq(const int32_t* __restrict__ cu, int nseq, int q) {
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- RoPE
// theta_i = (float)p * inv_freq[i], one fp32 multiply; accurate sincosf
// (the library is built without fast-math: angles reach ~2.7e5 rad).
__device__ __forceinline__ void rope_cs(int p, const float* inv_freq, int i, float* c, float* s) {
  float th = __fmul_rn((float)p, __ldg(inv_freq + i));
  sincosf(th, s, c);
}

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel is launched with programmatic stream serialization: it lets the
// next kernel in the stream start its prologue early (trigger), and itself
// touches no global memory written or read by its predecessor before the
// predecessor has completed (wait).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- reductions
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
// deterministic block sum (fixed tree); `red` holds >= 32 floats; all threads get the result
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// order-preserving map of fp32 to uint32 (larger float -> larger uint); -0 == +0
__device__ __forceinline__ uint32_t ord_key(float f) {
  uint32_t u = (f == 0.0f) ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa
