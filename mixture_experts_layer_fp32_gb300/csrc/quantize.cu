// E4M3 quantisation for the FP8 expert MLP (the FP8 GEMMs the Megatron Core
// report names as its most effective single optimisation; the pages print no
// scaling recipe).  Recipe: E4M3 codes with one power-of-two scale 2^e per
// token row of the activations (and per row of the SwiGLU output) and per
// output channel of each weight matrix, e the smallest integer with
// amax * 2^-e <= 448 (amax below 2^-100 or not finite: e = 0).  The codes
// are round-to-nearest-even with saturation at 448 (cvt.rn.satfinite).
//
// Kernels:
//   quantize_rows_kernel   a warp (rows up to 2048) or a CTA (up to 32768)
//                          per row, the row held in registers: its largest
//                          magnitude, its scale, 16 codes per 16-byte store
//   col_scale_kernel       one thread per weight column (output channel):
//                          the largest magnitude over K -> the channel scale
//   quantize_cols_kernel   64 (K) x 64 (N) tiles through shared memory:
//                          codes written K-major ([E][N][K]), 16 per thread
#include "common.cuh"
#include "e4m3.cuh"

namespace moe {
namespace {

using e4m3::pow2f;
using e4m3::scale_exp;

constexpr int kQThreads = 256;

// in [rows, cols] bf16 -> codes [rows, cols], scales [rows]; with row_count
// (device) only rows < *row_count are written; cols % 16 == 0.
// A team of TPR threads (32 to 256, the smallest that covers the row with
// G groups of 16 values per thread) takes a row; each thread keeps its
// groups in registers, so the row is read from memory once: largest
// magnitude (shuffles, plus shared memory across the team's warps), scale,
// codes.  Rows wider than 256 * 16 * G take the fallback below, which reads
// the row twice.
template <int TPR, int G>
__global__ void __launch_bounds__(kQThreads)
    quantize_rows_kernel(int64_t rows, int cols, const __nv_bfloat16* __restrict__ in,
                         uint8_t* __restrict__ codes, float* __restrict__ scales,
                         const int32_t* __restrict__ row_count) {
  constexpr int TEAMS = kQThreads / TPR;
  __shared__ float red[kQThreads / 32];
  const int64_t n = row_count ? min(rows, static_cast<int64_t>(*row_count)) : rows;
  const int t = threadIdx.x % TPR, lane = threadIdx.x & 31;
  const int groups = cols / 16;
  // every thread runs the same number of row iterations (the CTA-wide
  // reduction below needs all of them)
  for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * TEAMS; r0 < n;
       r0 += static_cast<int64_t>(gridDim.x) * TEAMS) {
    const int64_t r = r0 + threadIdx.x / TPR;
    const bool live = r < n;
    const uint4* src = reinterpret_cast<const uint4*>(in + (live ? r : 0) * cols);
    uint4 v[2 * G];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int g = t + i * TPR;
      if (live && g < groups) {
        v[2 * i] = src[2 * g];
        v[2 * i + 1] = src[2 * g + 1];
        m = e4m3::amax_bf16x8(v[2 * i + 1], e4m3::amax_bf16x8(v[2 * i], m));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (TPR > 32) {
      constexpr int W = TPR / 32;  // warps per team
      if (lane == 0) red[threadIdx.x >> 5] = m;
      __syncthreads();
      const int w0 = (threadIdx.x / TPR) * W;
      m = red[w0];
#pragma unroll
      for (int w = 1; w < W; ++w) m = fmaxf(m, red[w0 + w]);
      __syncthreads();  // red is rewritten for the next row
    }
    if (!live) continue;
    const int e = scale_exp(m);
    if (t == 0) scales[r] = pow2f(e);
    const float inv = pow2f(-e);
    uint4* dst = reinterpret_cast<uint4*>(codes + r * cols);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int g = t + i * TPR;
      if (g < groups) dst[g] = e4m3::quantize16(v[2 * i], v[2 * i + 1], inv);
    }
  }
}

// Fallback for rows wider than 32768: one warp per row, read twice.
__global__ void __launch_bounds__(kQThreads)
    quantize_wide_rows_kernel(int64_t rows, int cols, const __nv_bfloat16* __restrict__ in,
                              uint8_t* __restrict__ codes, float* __restrict__ scales,
                              const int32_t* __restrict__ row_count) {
  const int64_t n = row_count ? min(rows, static_cast<int64_t>(*row_count)) : rows;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQThreads / 32);
  const int groups = cols / 16;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (kQThreads / 32) + (threadIdx.x >> 5); r < n;
       r += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * cols);
    float m = 0.f;
    for (int g = lane; g < groups; g += 32)
      m = e4m3::amax_bf16x8(src[2 * g + 1], e4m3::amax_bf16x8(src[2 * g], m));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = scale_exp(m);
    if (lane == 0) scales[r] = pow2f(e);
    const float inv = pow2f(-e);
    uint4* dst = reinterpret_cast<uint4*>(codes + r * cols);
    for (int g = lane; g < groups; g += 32)
      dst[g] = e4m3::quantize16(src[2 * g], src[2 * g + 1], inv);
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
  scales[static_cast<int64_t>(e) * N + n] = pow2f(scale_exp(m));
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
    e4m3::bf16x8_to_float(
        *reinterpret_cast<const uint4*>(w + static_cast<int64_t>(k0 + kk) * N + n0 + 8 * v), f);
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
      e4m3::to_codes16(v);
}

}  // namespace

cudaError_t launch_quantize_rows(int64_t rows, int cols, const void* in, uint8_t* codes,
                                 float* scales, const int32_t* row_count, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(in);
  const int groups = cols / 16;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  auto grid = [&](int rows_per_cta) {
    const int64_t need = (rows + rows_per_cta - 1) / rows_per_cta;
    return static_cast<unsigned>(need < cap ? need : cap);
  };
  // team size: the smallest power of two >= 32 with 4 groups per thread
  if (groups <= 32 * 4)
    quantize_rows_kernel<32, 4><<<grid(8), kQThreads, 0, s>>>(rows, cols, x, codes, scales,
                                                               row_count);
  else if (groups <= 64 * 4)
    quantize_rows_kernel<64, 4><<<grid(4), kQThreads, 0, s>>>(rows, cols, x, codes, scales,
                                                               row_count);
  else if (groups <= 128 * 4)
    quantize_rows_kernel<128, 4><<<grid(2), kQThreads, 0, s>>>(rows, cols, x, codes, scales,
                                                                row_count);
  else if (groups <= 256 * 4)
    quantize_rows_kernel<256, 4><<<grid(1), kQThreads, 0, s>>>(rows, cols, x, codes, scales,
                                                                row_count);
  else if (groups <= 256 * 8)
    quantize_rows_kernel<256, 8><<<grid(1), kQThreads, 0, s>>>(rows, cols, x, codes, scales,
                                                                row_count);
  else
    quantize_wide_rows_kernel<<<grid(kQThreads / 32), kQThreads, 0, s>>>(rows, cols, x, codes,
                                                                       scales, row_count);
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
