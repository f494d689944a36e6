// fp32 grouped expert MLP (SIMT FMA), the path of the fp32 workload.
//
// Grouped expert MLP of §10 of "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
// (r00kie-liu.github.io): every local expert's GEMMs in one launch over the
// expert-major rows.  SwiGLU: fc1 computes silu(X.W1[e]) * (X.W3[e]); fc2
// computes H.W2[e].  The tensor cores have no fp32 mode that keeps fp32
// accuracy (TF32 rounds operands to 10 mantissa bits), so fp32 stays on the
// FMA units.  CTA tile 64 rows x 64 columns, K in chunks of 16, 256 threads
// with a 4x4 micro-tile each; a CTA belongs to one expert's row block,
// found from the expert offsets.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SBM = 64, SBN = 64, SBK = 16, SThreads = 256;

template <bool SWIGLU>
__global__ void __launch_bounds__(SThreads)
    simt_grouped_kernel(int E, int K, int N, int64_t max_rows, const float* __restrict__ A,
                        const int32_t* __restrict__ offsets, const float* __restrict__ B0,
                        const float* __restrict__ B1, float* __restrict__ C,
                        int* __restrict__ err) {
  __shared__ int off[MOE_MAX_EXPERTS + 1];
  __shared__ int tstart[MOE_MAX_EXPERTS + 1];
  __shared__ __align__(16) float As[SBK][SBM];
  __shared__ __align__(16) float Bs0[SBK][SBN];
  __shared__ __align__(16) float Bs1[SWIGLU ? SBK : 1][SWIGLU ? SBN : 4];

  // no offsets array: one dense group (E = 1) over rows [0, max_rows)
  for (int e = threadIdx.x; e <= E; e += blockDim.x)
    off[e] = offsets ? offsets[e] : (e == 0 ? 0 : static_cast<int>(max_rows));
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = off[0] == 0;
    int s = 0;
    for (int e = 0; e < E; ++e) {
      ok = ok && off[e + 1] >= off[e];
      tstart[e] = s;
      s += (off[e + 1] - off[e] + SBM - 1) / SBM;
    }
    ok = ok && off[E] <= max_rows;
    if (!ok) {
      report_error(err, DEV_ERR_INDEX, -1);
      s = 0;
      for (int e = 0; e <= E; ++e) tstart[e] = 0;
    }
    tstart[E] = s;
  }
  __syncthreads();
  const int tile = blockIdx.x;
  if (tile >= tstart[E]) return;
  int e = 0;
  while (e + 1 < E && tstart[e + 1] <= tile) ++e;
  const int m0 = off[e] + (tile - tstart[e]) * SBM;
  const int mend = off[e + 1];
  const int n0 = blockIdx.y * SBN;
  const float* b0 = B0 + (int64_t)e * K * N;
  const float* b1 = SWIGLU ? B1 + (int64_t)e * K * N : nullptr;

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 16 threads
  float acc0[4][4] = {}, acc1[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SBK) {
    for (int i = threadIdx.x; i < SBM * SBK; i += SThreads) {
      const int r = i / SBK, kk = i % SBK;
      const int row = m0 + r;
      As[kk][r] = (row < mend && k0 + kk < K) ? A[(int64_t)row * K + k0 + kk] : 0.f;
    }
    for (int i = threadIdx.x; i < SBK * SBN; i += SThreads) {
      const int kk = i / SBN, c = i % SBN;
      const bool ok = (k0 + kk < K) && (n0 + c < N);
      Bs0[kk][c] = ok ? b0[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
      if (SWIGLU) Bs1[kk][c] = ok ? b1[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      float a[4], b[4], g[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bs0[kk][tx * 4 + j];
        if (SWIGLU) g[j] = Bs1[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(a[i], b[j], acc0[i][j]);
          if (SWIGLU) acc1[i][j] = fmaf(a[i], g[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row >= mend) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= N) continue;
      float v = acc0[i][j];
      if (SWIGLU) v = v / (1.f + expf(-v)) * acc1[i][j];
      C[(int64_t)row * N + c] = v;
    }
  }
}

dim3 simt_grid(int E, int N, int64_t max_rows) {
  const int64_t mt = (max_rows + SBM - 1) / SBM + E;
  return dim3(static_cast<unsigned>(mt), static_cast<unsigned>((N + SBN - 1) / SBN));
}

}  // namespace

cudaError_t launch_simt_fc1(int E, int h, int f, int64_t max_rows, const float* x_perm,
                            const int32_t* offsets, const float* W1, const float* W3,
                            float* h_mid, int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  simt_grouped_kernel<true><<<simt_grid(E, f, max_rows), SThreads, 0, s>>>(
      E, h, f, max_rows, x_perm, offsets, W1, W3, h_mid, err);
  return cudaGetLastError();
}

cudaError_t launch_simt_fc2(int E, int h, int f, int64_t max_rows, const float* h_mid,
                            const int32_t* offsets, const float* W2, float* y_perm, int* err,
                            cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  simt_grouped_kernel<false><<<simt_grid(E, h, max_rows), SThreads, 0, s>>>(
      E, f, h, max_rows, h_mid, offsets, W2, nullptr, y_perm, err);
  return cudaGetLastError();
}

}  // namespace moe
