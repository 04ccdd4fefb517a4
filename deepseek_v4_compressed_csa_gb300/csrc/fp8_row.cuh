// Rotated E4M3 rows of 128 values: the index keys and index queries of a layer whose index pool holds fp8 rows.
//
// The indexer of the mlx-lm DeepSeek-V4 port (mlx-lm#1189, the indexer thread) rotates the index operands by a
// Hadamard matrix and simulates low-precision activations; the rotation cancels in the dot product, since
// (H q) . (H k) = 128 q . k for the unnormalised 128-point transform.  The row format here is this library's:
// the transform in fp32 with butterflies of span 1, 2, 4, .., 64 in that order, scale = amax / 448, codes =
// E4M3(rotated / scale) rounded to nearest even and saturating, an all-zero row has scale 0 and zero codes.
#pragma once
#include <cuda_fp8.h>
#include <stdint.h>

namespace csa {

constexpr int kFp8RowBytes = 144;  // 128 codes, the fp32 scale at byte 128, 12 zero bytes

// One warp, one row: lane l holds values 4l .. 4l+3 in u[] (every lane of the warp takes part).  Returns this
// lane's four codes packed little-endian (value 4l in the low byte) and the row's scale in *scale.
__device__ __forceinline__ uint32_t fp8_rotate_quantize(float u[4], int lane, float* scale) {
  // spans 1 and 2 inside the lane, then spans 4 .. 64 with lane partner l ^ (span / 4); (a, b) -> (a + b, a - b),
  // a the value whose span bit is clear
  {
    const float a0 = u[0], a1 = u[1], a2 = u[2], a3 = u[3];
    u[0] = __fadd_rn(a0, a1); u[1] = __fsub_rn(a0, a1); u[2] = __fadd_rn(a2, a3); u[3] = __fsub_rn(a2, a3);
    const float b0 = u[0], b1 = u[1], b2 = u[2], b3 = u[3];
    u[0] = __fadd_rn(b0, b2); u[2] = __fsub_rn(b0, b2); u[1] = __fadd_rn(b1, b3); u[3] = __fsub_rn(b1, b3);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, u[e], m);
      u[e] = upper ? __fsub_rn(o, u[e]) : __fadd_rn(u[e], o);
    }
  }
  float amax = fmaxf(fmaxf(fabsf(u[0]), fabsf(u[1])), fmaxf(fabsf(u[2]), fabsf(u[3])));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float sc = __fdiv_rn(amax, 448.f);
  uint32_t packed = 0;
  if (amax != 0.f) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      packed |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(u[e], sc), __NV_SATFINITE, __NV_E4M3) << (8 * e);
  }
  *scale = amax != 0.f ? sc : 0.f;
  return packed;
}

// Store one warp's row at dst (a 16-byte aligned kFp8RowBytes row): codes, scale, zero padding.
__device__ __forceinline__ void fp8_row_store(uint8_t* dst, int lane, uint32_t packed, float scale) {
  *reinterpret_cast<uint32_t*>(dst + 4 * lane) = packed;
  if (lane == 0) *reinterpret_cast<uint4*>(dst + 128) = make_uint4(__float_as_uint(scale), 0u, 0u, 0u);
}

}  // namespace csa
