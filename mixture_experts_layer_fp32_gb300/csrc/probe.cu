// Measurement probe (not a step of the MoE method): the FP32 FMA rate of the
// GPU, the denominator of the router's roofline where the router is bound by
// the FMA pipe (the fp32 logits GEMM with E >= 64).  Every thread runs 8
// independent chains of dependent fmaf(v, a, b); 4 CTAs of 256 threads per
// SM keep 8 warps per scheduler with 8-way instruction-level parallelism,
// enough to cover the FMA latency.  The result is never stored unless it is
// NaN (it cannot be), which keeps the compiler from removing the chains.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;
constexpr int kProbeUnroll = 16;

__global__ void __launch_bounds__(kProbeThreads)
    fp32_fma_probe_kernel(int64_t iters, float a, float b, float* out) {
  float v[kProbeChains];
#pragma unroll
  for (int i = 0; i < kProbeChains; ++i) v[i] = 1e-3f * threadIdx.x + i;
  for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u)
#pragma unroll
      for (int i = 0; i < kProbeChains; ++i) v[i] = fmaf(v[i], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kProbeChains; ++i) s += v[i];
  if (s != s) out[blockIdx.x] = s;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_probe_fp32_fma(int64_t iters, float* out, double* flops,
                                         moe_stream_t stream) {
  if (iters <= 0 || out == nullptr || flops == nullptr) return MOE_ERR_INVALID_ARG;
  const int grid = 4 * moe::device_sm_count();
  *flops = 2.0 * grid * moe::kProbeThreads * static_cast<double>(iters) * moe::kProbeUnroll *
           moe::kProbeChains;
  moe::fp32_fma_probe_kernel<<<grid, moe::kProbeThreads, 0, stream>>>(iters, 0.9999999f, 1e-7f,
                                                                      out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
