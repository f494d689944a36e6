// fp32 grouped expert MLP (SIMT FMA), the path of the fp32 workload.
//
// Grouped expert MLP of §10 of "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
// (r00kie-liu.github.io): every local expert's GEMMs in one launch over the
// expert-major rows.  SwiGLU: fc1 computes silu(X.W1[e]) * (X.W3[e]); fc2
// computes H.W2[e].  The layer backward's GEMMs (the chain rule on that
// forward) run here for the fp32 dtype too:
//   FC1_BWD  fc1's two products again, a = X.W1[e] and g = X.W3[e], with the
//            SwiGLU backward in the epilogue: reads dH, writes [da | dg]
//   DGRAD    C = A . B^T with B a weight read in place (its rows are C's
//            columns), K split between two weights (fc1's [W1 ; W3]^T)
//   simt_wgrad_kernel  dW[e] = A_e^T . B_e, the sum over expert e's rows
// With no offsets array a launch is one dense group (E = 1) over rows
// [0, max_rows) (the shared expert).
// The tensor cores have no fp32 mode that keeps fp32 accuracy (TF32 rounds
// operands to 10 mantissa bits), so fp32 stays on the FMA units.  CTA tile 32 rows x 32 columns, K in chunks of 64, 256 threads
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

enum { S_FC1 = 0, S_FC2 = 1, S_FC1_BWD = 2, S_DGRAD = 3 };

struct SimtArgs {
  int E, K, N;
  int64_t max_rows;
  const float* A;          // [rows, K]
  const int32_t* offsets;  // [E+1] or NULL (one dense group)
  const float* B0;         // FC1/FC2/FC1_BWD: [E][K][N]; DGRAD: [E][N][kb_split]
  const float* B1;         // FC1/FC1_BWD: [E][K][N]; DGRAD: [E][N][K - kb_split]
  int kb_split;            // DGRAD: columns of A taken against B0
  float* C;                // [rows, N] ([rows, 2N] for FC1_BWD: da then dg)
  const float* aux;        // FC1_BWD: dH [rows, N]
  int accumulate;          // FC2 / DGRAD: C += result
  int* err;
};

template <int MODE>
__global__ void __launch_bounds__(SThreads) simt_grouped_kernel(SimtArgs args) {
  constexpr bool TWO = MODE == S_FC1 || MODE == S_FC1_BWD;  // two products per output
  const int E = args.E, K = args.K, N = args.N;
  const int64_t max_rows = args.max_rows;
  const float* __restrict__ A = args.A;
  const int32_t* __restrict__ offsets = args.offsets;
  int* __restrict__ err = args.err;
  __shared__ int off[MOE_MAX_EXPERTS + 1];
  __shared__ int tstart[MOE_MAX_EXPERTS + 1];
  __shared__ __align__(16) float As[SBK][SBM + 1];  // +1: the transposing stores spread over the banks
  __shared__ __align__(16) float Bs0[SBK][SBN + 1];
  __shared__ __align__(16) float Bs1[TWO ? SBK : 1][TWO ? SBN + 1 : 4];

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
  const int K0 = MODE == S_DGRAD ? args.kb_split : K;  // K columns against B0
  const float* b0 = args.B0 + (int64_t)e * K0 * N;
  const float* b1 = TWO ? args.B1 + (int64_t)e * K * N
                  : MODE == S_DGRAD ? args.B1 + (int64_t)e * (K - K0) * N : nullptr;

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 16 threads
  float acc0[2][2] = {}, acc1[2][2] = {};
  for (int k0 = 0; k0 < K; k0 += SBK) {
    float ra[SPA], rb0[SPB], rb1[TWO ? SPB : 1];
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
      if (MODE == S_DGRAD) {  // weight rows are output columns: contiguous along K
        const int kk = i % SBK, c = i / SBK;
        const int k = k0 + kk;
        const bool ok = (k < K) && (n0 + c < N);
        rb0[u] = !ok ? 0.f
               : k < K0 ? b0[(int64_t)(n0 + c) * K0 + k]
                        : b1[(int64_t)(n0 + c) * (K - K0) + (k - K0)];
      } else {
        const int kk = i / SBN, c = i % SBN;
        const bool ok = (k0 + kk < K) && (n0 + c < N);
        rb0[u] = ok ? b0[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
        if (TWO) rb1[u] = ok ? b1[(int64_t)(k0 + kk) * N + n0 + c] : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < SPA; ++u) {
      const int i = threadIdx.x + u * SThreads;
      As[i % SBK][i / SBK] = ra[u];
    }
#pragma unroll
    for (int u = 0; u < SPB; ++u) {
      const int i = threadIdx.x + u * SThreads;
      if (MODE == S_DGRAD) {
        Bs0[i % SBK][i / SBK] = rb0[u];
      } else {
        Bs0[i / SBN][i % SBN] = rb0[u];
        if (TWO) Bs1[i / SBN][i % SBN] = rb1[u];
      }
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
        if (TWO) g[j] = Bs1[kk][tx * 2 + j];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc0[i][j] = fmaf(a[i], b[j], acc0[i][j]);
          if (TWO) acc1[i][j] = fmaf(a[i], g[j], acc1[i][j]);
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
      const float a = acc0[i][j];
      if (MODE == S_FC1) {
        args.C[(int64_t)row * N + c] = a / (1.f + expf(-a)) * acc1[i][j];
      } else if (MODE == S_FC1_BWD) {
        // h = silu(a) g: dh/da = g sig (1 + a (1 - sig)), dh/dg = a sig
        const float g = acc1[i][j];
        const float dh = args.aux[(int64_t)row * N + c];
        const float sg = 1.f / (1.f + expf(-a));
        args.C[(int64_t)row * 2 * N + c] = dh * g * (sg * (1.f + a * (1.f - sg)));
        args.C[(int64_t)row * 2 * N + N + c] = dh * (a * sg);
      } else {
        float* dst = args.C + (int64_t)row * N + c;
        *dst = args.accumulate ? *dst + a : a;
      }
    }
  }
}

// dW[e] [M, N] = A_e^T . B_e, the sum over expert e's rows (A [rows, lda],
// B [rows, ldb]): a CTA per (32 x 32 tile of dW, expert), the rows in chunks
// of 64 through shared memory, a 2 x 2 micro-tile per thread; an expert
// without rows gets zeros.
__global__ void __launch_bounds__(SThreads)
    simt_wgrad_kernel(int E, int M, int N, int64_t max_rows, const float* __restrict__ A,
                      int lda, const float* __restrict__ B, int ldb,
                      const int32_t* __restrict__ offsets, float* __restrict__ dW,
                      int* __restrict__ err) {
  __shared__ __align__(16) float As[SBK][SBM + 1];
  __shared__ __align__(16) float Bs[SBK][SBN + 1];
  const int e = blockIdx.y;
  const int nb = (N + SBN - 1) / SBN;
  const int m0 = (blockIdx.x / nb) * SBM, n0 = (blockIdx.x % nb) * SBN;
  int r_begin = 0, r_end = static_cast<int>(max_rows);
  if (offsets) {
    r_begin = offsets[e];
    r_end = offsets[e + 1];
    if (r_begin < 0 || r_end < r_begin || r_end > max_rows) {
      if (threadIdx.x == 0) report_error(err, DEV_ERR_INDEX, e);
      r_begin = r_end = 0;
    }
  }
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[2][2] = {};
  for (int r0 = r_begin; r0 < r_end; r0 += SBK) {
    float ra[SPA], rb[SPB];
#pragma unroll
    for (int u = 0; u < SPA; ++u) {  // 64 rows x 32 columns of A and of B
      const int i = threadIdx.x + u * SThreads;
      const int rr = i / SBM, c = i % SBM;
      const int r = r0 + rr;
      ra[u] = (r < r_end && m0 + c < M) ? A[(int64_t)r * lda + m0 + c] : 0.f;
      rb[u] = (r < r_end && n0 + c < N) ? B[(int64_t)r * ldb + n0 + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < SPA; ++u) {
      const int i = threadIdx.x + u * SThreads;
      As[i / SBM][i % SBM] = ra[u];
      Bs[i / SBM][i % SBM] = rb[u];
    }
    __syncthreads();
#pragma unroll 16
    for (int rr = 0; rr < SBK; ++rr) {
      const float a0 = As[rr][ty * 2], a1 = As[rr][ty * 2 + 1];
      const float b0 = Bs[rr][tx * 2], b1 = Bs[rr][tx * 2 + 1];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
    __syncthreads();
  }
  float* out = dW + (int64_t)e * M * N;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int m = m0 + ty * 2 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = n0 + tx * 2 + j;
      if (n < N) out[(int64_t)m * N + n] = acc[i][j];
    }
  }
}

dim3 simt_grid(int E, int N, int64_t max_rows) {
  const int64_t mt = (max_rows + SBM - 1) / SBM + E;
  return dim3(static_cast<unsigned>(mt), static_cast<unsigned>((N + SBN - 1) / SBN));
}

cudaError_t launch_simt(int mode, const SimtArgs& a, cudaStream_t s) {
  if (a.max_rows == 0) return cudaSuccess;
  const dim3 grid = simt_grid(a.E, a.N, a.max_rows);
  switch (mode) {
    case S_FC1: simt_grouped_kernel<S_FC1><<<grid, SThreads, 0, s>>>(a); break;
    case S_FC2: simt_grouped_kernel<S_FC2><<<grid, SThreads, 0, s>>>(a); break;
    case S_FC1_BWD: simt_grouped_kernel<S_FC1_BWD><<<grid, SThreads, 0, s>>>(a); break;
    default: simt_grouped_kernel<S_DGRAD><<<grid, SThreads, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fc1(int E, int h, int f, int64_t max_rows, const float* x_perm,
                            const int32_t* offsets, const float* W1, const float* W3,
                            float* h_mid, int* err, cudaStream_t s) {
  return launch_simt(S_FC1, SimtArgs{E, h, f, max_rows, x_perm, offsets, W1, W3, 0, h_mid,
                                     nullptr, 0, err}, s);
}

cudaError_t launch_simt_fc2(int E, int h, int f, int64_t max_rows, const float* h_mid,
                            const int32_t* offsets, const float* W2, float* y_perm, int* err,
                            cudaStream_t s) {
  return launch_simt(S_FC2, SimtArgs{E, f, h, max_rows, h_mid, offsets, W2, nullptr, 0, y_perm,
                                     nullptr, 0, err}, s);
}

cudaError_t launch_simt_dgrad_fc2(int E, int h, int f, int64_t max_rows, const float* dY,
                                  const int32_t* offsets, const float* W2, float* dH, int* err,
                                  cudaStream_t s) {
  // dH [rows, f] = dY [rows, h] . W2[e]^T, W2[e] [f, h]: its rows are dH's columns
  return launch_simt(S_DGRAD, SimtArgs{E, h, f, max_rows, dY, offsets, W2, W2, h, dH, nullptr, 0,
                                       err}, s);
}

cudaError_t launch_simt_fc1_bwd(int E, int h, int f, int64_t max_rows, const float* x_perm,
                                const int32_t* offsets, const float* W1, const float* W3,
                                const float* dH, float* dA, int* err, cudaStream_t s) {
  return launch_simt(S_FC1_BWD, SimtArgs{E, h, f, max_rows, x_perm, offsets, W1, W3, 0, dA, dH,
                                         0, err}, s);
}

cudaError_t launch_simt_dgrad_fc1(int E, int h, int f, int64_t max_rows, const float* dA,
                                  const int32_t* offsets, const float* W1, const float* W3,
                                  float* dx, int* err, cudaStream_t s, bool accumulate) {
  // dx [rows, h] = [da | dg] [rows, 2f] . [W1[e] ; W3[e]]^T, W1[e], W3[e] [h, f]
  return launch_simt(S_DGRAD, SimtArgs{E, 2 * f, h, max_rows, dA, offsets, W1, W3, f, dx,
                                       nullptr, accumulate ? 1 : 0, err}, s);
}

cudaError_t launch_simt_wgrad(int E, int M, int N, int64_t max_rows, const float* A, int lda,
                              const float* B, int ldb, const int32_t* offsets, float* dW,
                              int* err, cudaStream_t s) {
  const int tiles = ((M + SBM - 1) / SBM) * ((N + SBN - 1) / SBN);
  if (tiles == 0 || E == 0) return cudaSuccess;
  simt_wgrad_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(E)), SThreads, 0,
                      s>>>(E, M, N, max_rows, A, lda, B, ldb, offsets, dW, err);
  return cudaGetLastError();
}

}  // namespace moe
