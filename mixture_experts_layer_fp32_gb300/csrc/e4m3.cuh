// E4M3 helpers shared by the quantisation kernels: the power-of-two scale of
// the FP8 recipe, bf16 unpacking and the 16-value conversion.
//
// Recipe: the scale of a row (or channel) is 2^e with e the smallest integer
// such that amax * 2^-e <= 448, the largest finite E4M3 value; amax below
// 2^-100 or not finite gives e = 0.  Codes are round-to-nearest-even with
// saturation (cvt ... satfinite through the cuda_fp8.h conversion).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {
namespace e4m3 {

// e from the bits of amax (>= 0): amax = m * 2^E with m in [0.5, 1);
// 448 = 0.875 * 2^9, so e = E - 9 when m <= 0.875 (mantissa field <=
// 0x600000) and E - 8 otherwise.
__device__ __forceinline__ int scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int field = static_cast<int>((b >> 23) & 0xffu);
  if (!(amax >= 0x1p-100f) || field == 0xff) return 0;
  const int E = field - 126;
  return (b & 0x7fffffu) <= 0x600000u ? E - 9 : E - 8;
}

// 2^e as a float, for e in [-126, 127]
__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float amax_bf16x8(const uint4& u, float m) {
  float f[8];
  bf16x8_to_float(u, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// 16 floats (already scaled) -> 16 E4M3 codes in a uint4
__device__ __forceinline__ uint4 to_codes16(const float (&v)[16]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i], v[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i + 2], v[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
    w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// two 16-byte vectors of 8 bf16 each, times inv -> 16 codes
__device__ __forceinline__ uint4 quantize16(const uint4& a, const uint4& b, float inv) {
  float v[16], f[8];
  bf16x8_to_float(a, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = f[i] * inv;
  bf16x8_to_float(b, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[8 + i] = f[i] * inv;
  return to_codes16(v);
}

}  // namespace e4m3
}  // namespace moe
