// fp32 grouped expert MLP (SIMT FMA), the path of the fp32 workload.
//
// Grouped expert MLP of §10 of "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
// (r00kie-liu.github.io): every local expert's GEMMs in one launch over the
// expert-major rows.  SwiGLU: fc1 computes silu(X.W1[e]) * (X.W3[e]); fc2
// computes H.W2[e].  The tensor cores have no fp32 mode that keeps fp32
// accuracy (TF32 rounds operands to 10 mantissa bits), so fp32 stays on the
// FMA units.  CTA tile 32 rows x 32 columns, K in chunks of 64, 256 threads
// with a 2x2 micro-tile each; a CTA belongs to one expert's row block,
// found from the expert offsets.  The fp32 workloads are small (latency
// bound): small tiles give many CTAs and wide K chunks few memory round
// trips per CTA, each thread's loads of a chunk issued before its stores.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SBM = 32, SBN = 32, SBK = 64, SThreads = 256;
constexpr int SPA = SBM * SBK / SThreads;  // A values per thread per chunk (8)
constexpr int SPB = SBK * SBN / SThreads;  // B values per thread per chunk (8)

template <bool SWIGLU>
__global__ void __launch_bounds__(SThreads)
    simt_grouped_kernel(int E, int K, int N, int64_t max_rows, const float* __restrict__ A,
                        const int32_t* __restrict__ offsets, const float* __restrict__ B0,
                        const float* __restrict__ B1, float* __restrict__ C,
                        int* __restrict__ err) {
  __shared__ int off[MOE_MAX_EXPERTS + 1];
  __shared__ int tstart[MOE_MAX_EXPERTS + 1];
  __shared__ __align__(16) float As[SBK][SBM + 1];  // +1: the transposing stores spread over the banks
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
  float acc0[2][2] = {}, acc1[2][2] = {};
  for (int k0 = 0; k0 < K; k0 += SBK) {
    float ra[SPA], rb0[SPB], rb1[SWIGLU ? SPB : 1];
#pragma unroll
    for (int u = 0; u < SPA; ++u) {
      const int i = threadIdx.x + u * SThreads;
      const int r = i / SBK, kk = i % SBK;
      const int row = m0 + r;
      ra[u] = (row < mend && k0 + kk < K) ? A[(int64_t)row * K + k0 + kk] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < SPB; ++u) {
      const int i = threadIdx.x + u * SThreads;
      const int kk = i / SBN, c = i % SBN;
      const bool ok = (k0 + kk < K) && (n0 + c < N);
      rb0[u] = ok ? b0[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
      if (SWIGLU) rb1[u] = ok ? b1[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < SPA; ++u) {
      const int i = threadIdx.x + u * SThreads;
      As[i % SBK][i / SBK] = ra[u];
    }
#pragma unroll
    for (int u = 0; u < SPB; ++u) {
      const int i = threadIdx.x + u * SThreads;
      Bs0[i / SBN][i % SBN] = rb0[u];
      if (SWIGLU) Bs1[i / SBN][i % SBN] = rb1[u];
    }
    __syncthreads();
#pragma unroll 16
    for (int kk = 0; kk < SBK; ++kk) {
      float a[2], b[2], g[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) a[i] = As[kk][ty * 2 + i];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        b[j] = Bs0[kk][tx * 2 + j];
        if (SWIGLU) g[j] = Bs1[kk][tx * 2 + j];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc0[i][j] = fmaf(a[i], b[j], acc0[i][j]);
          if (SWIGLU) acc1[i][j] = fmaf(a[i], g[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = m0 + ty * 2 + i;
    if (row >= mend) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = n0 + tx * 2 + j;
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
