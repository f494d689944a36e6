// E4M3 quantisation for the FP8 expert MLP (the FP8 GEMMs the Megatron Core
// report names as its most effective single optimisation; the pages print no
// scaling recipe).  Recipe: E4M3 codes with one power-of-two scale 2^e per
// token row of the activations (and per row of the SwiGLU output) and per
// output channel of each weight matrix, e the smallest integer with
// amax * 2^-e <= 448 (amax below 2^-100 or not finite: e = 0).  The codes
// are round-to-nearest-even with saturation at 448 (cvt.rn.satfinite).
//
// Kernels:
//   quantize_rows_kernel   one CTA per row: the row's largest magnitude, its
//                          scale, then 16 codes per thread step (two 16-byte
//                          bf16 loads, one 16-byte store)
//   col_scale_kernel       one thread per weight column (output channel):
//                          the largest magnitude over K -> the channel scale
//   quantize_cols_kernel   64 (K) x 64 (N) tiles through shared memory:
//                          codes written K-major ([E][N][K]), 16 per thread
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// e of the recipe from the bits of amax (>= 0): amax = m * 2^E with m in
// [0.5, 1); 448 = 0.875 * 2^9, so e = E - 9 when m <= 0.875 (mantissa field
// <= 0x600000) and E - 8 otherwise.
__device__ __forceinline__ int fp8_scale_exp(float amax) {
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

// 16 floats (already scaled) -> 16 E4M3 codes in a uint4
__device__ __forceinline__ uint4 to_e4m3x16(const float (&v)[16]) {
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

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is reused row after row
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < (kQThreads / 32) ? red[lane] : 0.f;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return __shfl_sync(0xffffffffu, v, 0);
}

// in [rows, cols] bf16 -> codes [rows, cols], scales [rows]; with row_count
// (device) only rows < *row_count are written.  cols % 16 == 0.
__global__ void __launch_bounds__(kQThreads)
    quantize_rows_kernel(int64_t rows, int cols, const __nv_bfloat16* __restrict__ in,
                         uint8_t* __restrict__ codes, float* __restrict__ scales,
                         const int32_t* __restrict__ row_count) {
  __shared__ float red[kQThreads / 32];
  const int64_t n = row_count ? min(rows, static_cast<int64_t>(*row_count)) : rows;
  const int groups = cols / 16;
  for (int64_t r = blockIdx.x; r < n; r += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * cols);
    float m = 0.f;
    for (int g = threadIdx.x; g < groups; g += kQThreads) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float f[8];
        bf16x8_to_float(src[2 * g + h], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
      }
    }
    m = block_max(m, red);
    const int e = fp8_scale_exp(m);
    if (threadIdx.x == 0) scales[r] = pow2f(e);
    const float inv = pow2f(-e);
    uint4* dst = reinterpret_cast<uint4*>(codes + r * cols);
    for (int g = threadIdx.x; g < groups; g += kQThreads) {
      float v[16], f[8];
      bf16x8_to_float(src[2 * g], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = f[i] * inv;
      bf16x8_to_float(src[2 * g + 1], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 + i] = f[i] * inv;
      dst[g] = to_e4m3x16(v);
    }
  }
}

// W [E][K][N] bf16 -> scales [E][N]: one thread per column n of expert e.
__global__ void __launch_bounds__(kQThreads)
    col_scale_kernel(int K, int N, const __nv_bfloat16* __restrict__ W, float* __restrict__ scales) {
  const int e = blockIdx.y;
  const int n = blockIdx.x * kQThreads + threadIdx.x;
  if (n >= N) return;
  const __nv_bfloat16* w = W + static_cast<int64_t>(e) * K * N + n;
  float m = 0.f;
  for (int k = 0; k < K; ++k) m = fmaxf(m, fabsf(__bfloat162float(w[static_cast<int64_t>(k) * N])));
  scales[static_cast<int64_t>(e) * N + n] = pow2f(fp8_scale_exp(m));
}

// W [E][K][N] bf16 -> codes [E][N][K] with the channel scales of
// col_scale_kernel; tile 64 (K) x 64 (N) per CTA, K % 64 == N % 64 == 0.
__global__ void __launch_bounds__(kQThreads)
    quantize_cols_kernel(int K, int N, const __nv_bfloat16* __restrict__ W,
                         const float* __restrict__ scales, uint8_t* __restrict__ codes) {
  __shared__ float tile[64][65];  // [k][n], padded against bank conflicts on the column reads
  const int e = blockIdx.z;
  const int n0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  const __nv_bfloat16* w = W + static_cast<int64_t>(e) * K * N;
  for (int i = threadIdx.x; i < 64 * 8; i += kQThreads) {  // 64 rows x 8 vectors of 8 bf16
    const int kk = i >> 3, v = i & 7;
    float f[8];
    bf16x8_to_float(*reinterpret_cast<const uint4*>(w + static_cast<int64_t>(k0 + kk) * N + n0 + 8 * v), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) tile[kk][8 * v + j] = f[j];
  }
  __syncthreads();
  const int nn = threadIdx.x >> 2, g = threadIdx.x & 3;  // column nn, K values 16g .. 16g+15
  const float s = scales[static_cast<int64_t>(e) * N + n0 + nn];
  const float inv = pow2f(127 - static_cast<int>((__float_as_uint(s) >> 23) & 0xffu));  // 2^-e
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = tile[16 * g + j][nn] * inv;
  *reinterpret_cast<uint4*>(codes + (static_cast<int64_t>(e) * N + n0 + nn) * K + k0 + 16 * g) =
      to_e4m3x16(v);
}

}  // namespace

cudaError_t launch_quantize_rows(int64_t rows, int cols, const void* in, uint8_t* codes,
                                 float* scales, const int32_t* row_count, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * 8;
  if (grid > rows) grid = rows;
  quantize_rows_kernel<<<static_cast<unsigned>(grid), kQThreads, 0, s>>>(
      rows, cols, static_cast<const __nv_bfloat16*>(in), codes, scales, row_count);
  return cudaGetLastError();
}

cudaError_t launch_quantize_cols(int E, int K, int N, const void* W, uint8_t* codes,
                                 float* scales, cudaStream_t s) {
  if (E == 0) return cudaSuccess;
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(W);
  col_scale_kernel<<<dim3((N + kQThreads - 1) / kQThreads, E), kQThreads, 0, s>>>(K, N, w, scales);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  quantize_cols_kernel<<<dim3(N / 64, K / 64, E), kQThreads, 0, s>>>(K, N, w, scales, codes);
  return cudaGetLastError();
}

}  // namespace moe
