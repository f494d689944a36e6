// Backward of the MoE layer around the expert GEMMs: the gradient of
// L = sum(dy * y) for fixed routing decisions (the chain rule on the forward
// of the Megatron Core page: combine of §2, score functions of §5, gating of
// §3).  The expert GEMMs' backward lives in gemm_tc.cu / gemm_wgrad.cu.
//
// Kernels:
//   combine_bwd_kernel  per token: for each kept slot j, dY_perm[row] =
//                       p[t,j] dy[t] (bf16) and dp[t,j] = <dy[t], y_perm[row]>
//   router_bwd_kernel   one warp per token: dlogits from dp through the score
//                       function (softmax after / before top-k, sigmoid,
//                       sqrtsoftplus with renormalisation), fp32
//   dwg_kernel          dWg [h,E] = x^T dlogits: 64 x 64 output tiles, the
//                       tokens split across CTAs (partial sums added in
//                       split order by dwg_reduce_kernel) and streamed
//                       through shared memory
//   dwg_small_kernel    the same for E <= 32: a thread owns two rows of dWg
//                       and all E columns, x streamed straight from memory
//   dgb_kernel          dgate_bias[e] = sum_t dlogits[t,e], one CTA per expert
//   dx_router_kernel    dx_router [T,h] = dlogits . Wg^T: 64 x 64 tiles
//   dx_router_small_kernel  the same for E <= 16: a thread owns four columns
//                       of h with their Wg rows in registers (write-bound)
//   split3_kernel       fp32 -> bf16 hi/lo triples for the tensor-core path
//                       (E % 64 == 0): dWg and dx_router as tcgen05 GEMMs
//   fold_halves_kernel  dWg = the hi and lo halves of that GEMM's output
// The token gradient dx = sum_j dx_perm[row(t,j)] + dx_router[t] is the
// combine kernel with unit weights and dx_router as its addend.
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBwdThreads = 128;

// 8 consecutive activations (bf16 or fp32) of a row as floats: vector v
// covers elements 8v .. 8v+7
template <typename AT>
struct Act8;
template <>
struct Act8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* row, int v, float (&d)[8]) {
    const uint4 u = reinterpret_cast<const uint4*>(row)[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      d[2 * i] = __uint_as_float(w[i] << 16);
      d[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* row, int v, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(row)[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Act8<float> {
  __device__ static void load(const float* row, int v, float (&d)[8]) {
    const float4 a = reinterpret_cast<const float4*>(row)[2 * v];
    const float4 b = reinterpret_cast<const float4*>(row)[2 * v + 1];
    d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
    d[4] = b.x; d[5] = b.y; d[6] = b.z; d[7] = b.w;
  }
  __device__ static void store(float* row, int v, const float (&o)[8]) {
    reinterpret_cast<float4*>(row)[2 * v] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(row)[2 * v + 1] = make_float4(o[4], o[5], o[6], o[7]);
  }
};

// dy [T,h] (AT), y_perm [rows,h] fp32 -> dY_perm [rows,h] (AT), dp [T,k] fp32
template <typename AT>
__global__ void __launch_bounds__(kBwdThreads)
    combine_bwd_kernel(int T, int h, int k, const AT* __restrict__ dy,
                       const int32_t* __restrict__ row_map, const float* __restrict__ topk_prob,
                       const float* __restrict__ y_perm, AT* __restrict__ dY_perm,
                       float* __restrict__ dp) {
  __shared__ float red[kBwdThreads / 32][MOE_MAX_TOPK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h8 = h / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int rows[MOE_MAX_TOPK];
    float p[MOE_MAX_TOPK], dot[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      rows[j] = j < k ? row_map[(int64_t)t * k + j] : -1;
      p[j] = rows[j] >= 0 ? topk_prob[(int64_t)t * k + j] : 0.f;
      dot[j] = 0.f;
    }
    for (int v = threadIdx.x; v < h8; v += kBwdThreads) {
      float d[8];
      Act8<AT>::load(dy + (int64_t)t * h, v, d);
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (rows[j] < 0) continue;
        const float4* yp = reinterpret_cast<const float4*>(y_perm + (int64_t)rows[j] * h) + 2 * v;
        const float4 y0 = yp[0], y1 = yp[1];
        dot[j] += d[0] * y0.x + d[1] * y0.y + d[2] * y0.z + d[3] * y0.w + d[4] * y1.x +
                  d[5] * y1.y + d[6] * y1.z + d[7] * y1.w;
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = p[j] * d[i];
        Act8<AT>::store(dY_perm + (int64_t)rows[j] * h, v, o);
      }
    }
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      float v = dot[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][j] = v;
    }
    __syncthreads();
    if (threadIdx.x < k) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kBwdThreads / 32; ++w) v += red[w][threadIdx.x];
      dp[(int64_t)t * k + threadIdx.x] = rows[threadIdx.x] >= 0 ? v : 0.f;
    }
    __syncthreads();
  }
}

constexpr int kPerLane = MOE_MAX_EXPERTS / 32;

// logits: nsplit partial sums [S,T,E] (added in split order) + gate bias.
__global__ void __launch_bounds__(256)
    router_bwd_kernel(int T, int E, int k, int score, const float* __restrict__ logits, int nsplit,
                      const float* __restrict__ gate_bias, const int32_t* __restrict__ topk_idx,
                      const float* __restrict__ dp, float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int t = blockIdx.x * nwarps + (threadIdx.x >> 5); t < T; t += gridDim.x * nwarps) {
    float l[kPerLane], s[kPerLane], dl[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      dl[i] = 0.f;
      if (e < E) {
        float v = logits[(int64_t)t * E + e];
        for (int sp = 1; sp < nsplit; ++sp) v += logits[((int64_t)sp * T + t) * E + e];
        l[i] = gate_bias ? v + gate_bias[e] : v;
      } else {
        l[i] = -FLT_MAX;
      }
      s[i] = l[i];
    }
    // the chosen experts, their scores and dp (lane j holds slot j)
    int my_e = -1;
    float my_dp = 0.f;
    if (lane < k) {
      my_e = topk_idx[(int64_t)t * k + lane];
      my_dp = dp[(int64_t)t * k + lane];
    }
    if (score == MOE_SCORE_SOFTMAX_PRE) {
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) m = fmaxf(m, s[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        s[i] = (lane + 32 * i < E) ? expf(s[i] - m) : 0.f;
        z += s[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) s[i] /= z;
    } else if (score == MOE_SCORE_SIGMOID || score == MOE_SCORE_SQRTSOFTPLUS) {
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        if (lane + 32 * i >= E) {
          s[i] = 0.f;
          continue;
        }
        s[i] = score == MOE_SCORE_SIGMOID
                   ? 1.f / (1.f + expf(-l[i]))
                   : sqrtf(fmaxf(l[i], 0.f) + log1pf(expf(-fabsf(l[i]))));
      }
    }
    // score of each chosen expert, gathered to its slot's lane
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, my_e, j);
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i)
        if (lane + 32 * i == e) v = s[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == j) my_s = v;
    }
    float add = 0.f;  // this lane's slot's contribution to dlogits[my_e]
    if (score == MOE_SCORE_SOFTMAX_POST) {
      float m = lane < k ? my_s : -FLT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float ex = lane < k ? expf(my_s - m) : 0.f;
      float z = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float p = ex / z;
      float sdp = p * my_dp;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sdp += __shfl_xor_sync(0xffffffffu, sdp, o);
      add = lane < k ? p * (my_dp - sdp) : 0.f;
    } else if (score == MOE_SCORE_SOFTMAX_PRE) {
      // ds = dp at the chosen experts; dl = s (ds - <ds, s>)
      float sds = lane < k ? my_dp * my_s : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sds += __shfl_xor_sync(0xffffffffu, sds, o);
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) dl[i] = -s[i] * sds;
      add = lane < k ? my_s * my_dp : 0.f;
    } else {
      float z = lane < k ? my_s : 0.f, spd = lane < k ? my_dp * my_s : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        z += __shfl_xor_sync(0xffffffffu, z, o);
        spd += __shfl_xor_sync(0xffffffffu, spd, o);
      }
      z += 1e-20f;
      const float ds = my_dp / z - spd / (z * z);
      float lv = 0.f;  // the chosen expert's logit
      for (int j = 0; j < k; ++j) {
        const int e = __shfl_sync(0xffffffffu, my_e, j);
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
          if (lane + 32 * i == e) v = l[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == j) lv = v;
      }
      const float deriv = score == MOE_SCORE_SIGMOID ? my_s * (1.f - my_s)
                                                    : (1.f / (1.f + expf(-lv))) / (2.f * my_s);
      add = lane < k ? ds * deriv : 0.f;
    }
    // scatter the k slot contributions onto their experts (distinct experts)
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, my_e, j);
      const float a = __shfl_sync(0xffffffffu, add, j);
#pragma unroll
      for (int i = 0; i < kPerLane; ++i)
        if (lane + 32 * i == e) dl[i] += a;
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E) dlogits[(int64_t)t * E + e] = dl[i];
    }
  }
}

// dWg [h,E] = x^T dl: tile 64 (h) x 64 (E), tokens streamed 32 at a time;
// 256 threads, 4 x 4 outputs each.  gridDim.z splits the tokens: split z
// covers tokens [z * tps, (z+1) * tps) and writes its own partial sums
// (out + z * h * E), which dwg_reduce_kernel adds in split order.
template <typename XT>
__global__ void __launch_bounds__(256)
    dwg_kernel(int T, int h, int E, int tps, const XT* __restrict__ x,
               const float* __restrict__ dl, float* __restrict__ out) {
  __shared__ float xs[32][64 + 4];
  __shared__ float ls[32][64 + 4];
  const int i0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
  const int tbeg = blockIdx.z * tps, tend = min(T, tbeg + tps);
  float* dWg = out + static_cast<int64_t>(blockIdx.z) * h * E;
  float acc[4][4] = {};
  for (int t0 = tbeg; t0 < tend; t0 += 32) {
    for (int v = threadIdx.x; v < 32 * 64; v += 256) {
      const int tt = v >> 6, c = v & 63;
      const int t = t0 + tt;
      xs[tt][c] = (t < tend && i0 + c < h) ? static_cast<float>(x[(int64_t)t * h + i0 + c]) : 0.f;
      ls[tt][c] = (t < tend && e0 + c < E) ? dl[(int64_t)t * E + e0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int tt = 0; tt < 32; ++tt) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = xs[tt][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = ls[tt][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + ty * 4 + r, e = e0 + tx * 4 + c;
      if (i < h && e < E) dWg[(int64_t)i * E + e] = acc[r][c];
    }
}

// dWg [h,E] = x^T dl for E <= EC (EC = 8, 16 or 32): thread j of the grid
// owns rows i = 2j, 2j+1 of dWg and their EC columns (packed fp32x2 FMAs on
// the two rows); tokens of split z are [z * tps, (z+1) * tps), their dl rows
// staged 64 at a time in shared memory.  Each split writes its partial sums
// to out + z * h * E (added in split order by dwg_reduce_kernel).
// x as pairs of consecutive features: bf16x2 or float2, widened to float2
template <typename XT>
struct XPair;
template <>
struct XPair<__nv_bfloat16> {
  using P = __nv_bfloat162;
  __device__ static float2 get(P v) { return __bfloat1622float2(v); }
};
template <>
struct XPair<float> {
  using P = float2;
  __device__ static float2 get(P v) { return v; }
};

template <int EC, typename XT>
__global__ void __launch_bounds__(256)
    dwg_small_kernel(int T, int h, int E, int tps, const XT* __restrict__ x,
                     const float* __restrict__ dl, float* __restrict__ out) {
  using P = typename XPair<XT>::P;
  constexpr int TCH = 64;
  __shared__ __align__(16) float ls[TCH][EC];
  const int i = (blockIdx.x * 256 + threadIdx.x) * 2;
  const int tbeg = blockIdx.z * tps, tend = min(T, tbeg + tps);
  float2 acc[EC];
#pragma unroll
  for (int e = 0; e < EC; ++e) acc[e] = make_float2(0.f, 0.f);
  const P* xr = reinterpret_cast<const P*>(x + i);
  const int64_t step = h / 2;  // pairs per token row
  for (int t0 = tbeg; t0 < tend; t0 += TCH) {
    const int n = min(TCH, tend - t0);
    for (int v = threadIdx.x; v < TCH * EC; v += 256) {
      const int tt = v / EC, e = v - tt * EC;
      ls[tt][e] = (tt < n && e < E) ? dl[static_cast<int64_t>(t0 + tt) * E + e] : 0.f;
    }
    __syncthreads();
    if (i < h) {
      const P* xp = xr + static_cast<int64_t>(t0) * step;
      int tt = 0;
      for (; tt + 8 <= n; tt += 8) {
        float2 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) xv[u] = XPair<XT>::get(xp[static_cast<int64_t>(tt + u) * step]);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4* lr = reinterpret_cast<const float4*>(ls[tt + u]);
#pragma unroll
          for (int e4 = 0; e4 < EC / 4; ++e4) {
            const float4 l = lr[e4];
            acc[4 * e4] = __ffma2_rn(xv[u], make_float2(l.x, l.x), acc[4 * e4]);
            acc[4 * e4 + 1] = __ffma2_rn(xv[u], make_float2(l.y, l.y), acc[4 * e4 + 1]);
            acc[4 * e4 + 2] = __ffma2_rn(xv[u], make_float2(l.z, l.z), acc[4 * e4 + 2]);
            acc[4 * e4 + 3] = __ffma2_rn(xv[u], make_float2(l.w, l.w), acc[4 * e4 + 3]);
          }
        }
      }
      for (; tt < n; ++tt) {
        const float2 xv = XPair<XT>::get(xp[static_cast<int64_t>(tt) * step]);
#pragma unroll
        for (int e = 0; e < EC; ++e) acc[e] = __ffma2_rn(xv, make_float2(ls[tt][e], ls[tt][e]), acc[e]);
      }
    }
    __syncthreads();
  }
  if (i < h) {
    float* o = out + static_cast<int64_t>(blockIdx.z) * h * E + static_cast<int64_t>(i) * E;
#pragma unroll
    for (int e = 0; e < EC; ++e)
      if (e < E) {
        o[e] = acc[e].x;
        o[E + e] = acc[e].y;
      }
  }
}

// dWg = the S partial sums of dwg_kernel: 8 threads per output (lanes 8j..
// 8j+7 of a warp hold output j of 4), thread q summing splits q, q+8, ...
// in order, then the 8 sums added in a fixed tree: a deterministic order
// with S/8 loads per thread in flight instead of S in a row.
__global__ void __launch_bounds__(256)
    dwg_reduce_kernel(int64_t n, int S, const float* __restrict__ part, float* __restrict__ dWg) {
  const int q = threadIdx.x & 7;
  const unsigned group = 0xffu << (threadIdx.x & 24);  // the 8 lanes sharing an output
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) >> 3; i < n;
       i += static_cast<int64_t>(gridDim.x) * 32) {
    float v = 0.f;
    for (int z = q; z < S; z += 8) v += part[z * n + i];
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) v += __shfl_xor_sync(group, v, o);
    if (q == 0) dWg[i] = v;
  }
}

// dgate_bias[e] = sum over tokens of dl[t,e] (fixed order: strided partial
// sums, then a tree over the block)
__global__ void __launch_bounds__(256)
    dgb_kernel(int T, int E, const float* __restrict__ dl, float* __restrict__ dgb) {
  __shared__ float red[256];
  const int e = blockIdx.x;
  float v = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) v += dl[(int64_t)t * E + e];
  red[threadIdx.x] = v;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) dgb[e] = red[0];
}

// dx_router [T,h] = dl [T,E] . Wg^T (Wg [h,E]): tile 64 tokens x 64 of h,
// E in chunks of 32 through shared memory; 4 x 4 outputs per thread.
__global__ void __launch_bounds__(256)
    dx_router_kernel(int T, int h, int E, const float* __restrict__ dl,
                     const float* __restrict__ Wg, float* __restrict__ out) {
  __shared__ float ls[32][64 + 4];  // [e][t]
  __shared__ float ws[32][64 + 4];  // [e][i]
  const int t0 = blockIdx.x * 64, i0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int e0 = 0; e0 < E; e0 += 32) {
    for (int v = threadIdx.x; v < 32 * 64; v += 256) {
      const int rr = v >> 5, ee = v & 31;  // row of the tile, expert in the chunk
      const int e = e0 + ee;
      ls[ee][rr] = (t0 + rr < T && e < E) ? dl[(int64_t)(t0 + rr) * E + e] : 0.f;
      ws[ee][rr] = (i0 + rr < h && e < E) ? Wg[(int64_t)(i0 + rr) * E + e] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int ee = 0; ee < 32; ++ee) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = ls[ee][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = ws[ee][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int t = t0 + ty * 4 + r, i = i0 + tx * 4 + c;
      if (t < T && i < h) out[(int64_t)t * h + i] = acc[r][c];
    }
}

// dx_router [T,h] = dl . Wg^T for E <= EC (EC = 8 or 16): a block covers 256
// columns of h (64 threads x 4) and 64 tokens (4 thread rows x 16); a thread
// keeps Wg's rows for its 4 columns in registers and reads each token's dl
// row from shared memory (a broadcast), writing 16 bytes per token.
template <int EC>
__global__ void __launch_bounds__(256)
    dx_router_small_kernel(int T, int h, int E, const float* __restrict__ dl,
                           const float* __restrict__ Wg, float* __restrict__ out) {
  __shared__ __align__(16) float ls[64][EC];
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const int i = (blockIdx.y * 64 + tx) * 4, t0 = blockIdx.x * 64;
  for (int v = threadIdx.x; v < 64 * EC; v += 256) {
    const int tt = v / EC, e = v - tt * EC;
    ls[tt][e] = (t0 + tt < T && e < E) ? dl[static_cast<int64_t>(t0 + tt) * E + e] : 0.f;
  }
  float w[4][EC];
  if (E == EC && (reinterpret_cast<uintptr_t>(Wg) & 15) == 0) {  // whole, aligned rows: 16-byte loads
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e4 = 0; e4 < EC / 4; ++e4) {
        const float4 v = i + c < h ? *reinterpret_cast<const float4*>(
                                         Wg + static_cast<int64_t>(i + c) * E + 4 * e4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        w[c][4 * e4] = v.x;
        w[c][4 * e4 + 1] = v.y;
        w[c][4 * e4 + 2] = v.z;
        w[c][4 * e4 + 3] = v.w;
      }
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < EC; ++e)
        w[c][e] = (i + c < h && e < E) ? Wg[static_cast<int64_t>(i + c) * E + e] : 0.f;
  }
  __syncthreads();
  if (i >= h) return;
#pragma unroll 4
  for (int tt = ty; tt < 64; tt += 4) {
    const int t = t0 + tt;
    if (t >= T) break;
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
    const float4* lr = reinterpret_cast<const float4*>(ls[tt]);
#pragma unroll
    for (int e4 = 0; e4 < EC / 4; ++e4) {
      const float4 l = lr[e4];
      const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 4 * e4 + u;
        a01 = __ffma2_rn(make_float2(w[0][e], w[1][e]), make_float2(lv[u], lv[u]), a01);
        a23 = __ffma2_rn(make_float2(w[2][e], w[3][e]), make_float2(lv[u], lv[u]), a23);
      }
    }
    *reinterpret_cast<float4*>(out + static_cast<int64_t>(t) * h + i) =
        make_float4(a01.x, a01.y, a23.x, a23.y);
  }
}

// v [rows, E] fp32 -> dst [rows, 3E] bf16: hi = bf16(v), lo = bf16(v - hi)
// (v - hi is exact in fp32), written as [hi | lo | hi] (lo_last == 0) or
// [hi | hi | lo] (lo_last == 1).
__global__ void __launch_bounds__(256)
    split3_kernel(int64_t rows, int E, int lo_last, const float* __restrict__ v,
                  __nv_bfloat16* __restrict__ dst) {
  const int64_t n = rows * E;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t r = i / E;
    const int e = static_cast<int>(i - r * E);
    const float x = v[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    __nv_bfloat16* d = dst + r * 3 * E + e;
    d[0] = hi;
    d[E] = lo_last ? hi : lo;
    d[2 * E] = lo_last ? lo : hi;
  }
}

// dWg [h, E] = out [h, 2E]: columns e and E + e added
__global__ void __launch_bounds__(256)
    fold_halves_kernel(int64_t n, int E, const float* __restrict__ two, float* __restrict__ dWg) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t r = i / E;
    const int e = static_cast<int>(i - r * E);
    dWg[i] = two[r * 2 * E + e] + two[r * 2 * E + E + e];
  }
}

}  // namespace

cudaError_t launch_combine_bwd(int T, int h, int k, int dtype, const void* dy,
                               const int32_t* row_map, const float* topk_prob,
                               const float* y_perm, void* dY_perm, float* dp, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int cap = device_sm_count() * 16;
  const int grid = T < cap ? T : cap;
  if (dtype == MOE_F32)
    combine_bwd_kernel<float><<<grid, kBwdThreads, 0, s>>>(
        T, h, k, static_cast<const float*>(dy), row_map, topk_prob, y_perm,
        static_cast<float*>(dY_perm), dp);
  else
    combine_bwd_kernel<__nv_bfloat16><<<grid, kBwdThreads, 0, s>>>(
        T, h, k, static_cast<const __nv_bfloat16*>(dy), row_map, topk_prob, y_perm,
        static_cast<__nv_bfloat16*>(dY_perm), dp);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(int T, int E, int k, int score, const float* logits, int nsplit,
                              const float* gate_bias, const int32_t* topk_idx, const float* dp,
                              float* dlogits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int blocks = (T + 7) / 8;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  router_bwd_kernel<<<blocks, 256, 0, s>>>(T, E, k, score, logits, nsplit, gate_bias, topk_idx,
                                           dp, dlogits);
  return cudaGetLastError();
}

int dwg_splits(int T, int h, int E) {
  // about four CTAs per SM over (blocks of dWg) x splits; E <= 32: blocks of
  // 512 rows, each split at least 64 tokens, at most 128 splits; else 64 x 64
  // tiles, each split at least 256 tokens, at most 32 splits
  const bool small = E <= 32;
  const int64_t tiles = small ? (h + 511) / 512
                              : static_cast<int64_t>((h + 63) / 64) * ((E + 63) / 64);
  int64_t S = (4LL * device_sm_count() + tiles - 1) / tiles;
  const int64_t by_tokens = small ? (T + 63) / 64 : (T + 255) / 256;
  if (S > by_tokens) S = by_tokens;
  if (S > (small ? 128 : 32)) S = small ? 128 : 32;
  return S < 1 ? 1 : static_cast<int>(S);
}

template <typename XT>
void launch_dwg(int T, int h, int E, int S, int tps, const XT* x, const float* dl, float* dst,
                cudaStream_t s) {
  const dim3 small_grid((h + 511) / 512, 1, S);
  if (E <= 8)
    dwg_small_kernel<8, XT><<<small_grid, 256, 0, s>>>(T, h, E, tps, x, dl, dst);
  else if (E <= 16)
    dwg_small_kernel<16, XT><<<small_grid, 256, 0, s>>>(T, h, E, tps, x, dl, dst);
  else if (E <= 32)
    dwg_small_kernel<32, XT><<<small_grid, 256, 0, s>>>(T, h, E, tps, x, dl, dst);
  else
    dwg_kernel<XT><<<dim3((h + 63) / 64, (E + 63) / 64, S), 256, 0, s>>>(T, h, E, tps, x, dl, dst);
}

cudaError_t launch_router_param_grads(int T, int h, int E, int dtype, const void* x,
                                      const float* dl, float* dWg, float* part, float* dgb,
                                      cudaStream_t s) {
  const int S = dwg_splits(T, h, E);
  const int tps = S > 1 ? (T + S - 1) / S : (T > 0 ? T : 1);
  float* dst = S > 1 ? part : dWg;
  if (dtype == MOE_F32)
    launch_dwg(T, h, E, S, tps, static_cast<const float*>(x), dl, dst, s);
  else
    launch_dwg(T, h, E, S, tps, static_cast<const __nv_bfloat16*>(x), dl, dst, s);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  if (S > 1) {
    const int64_t n = static_cast<int64_t>(h) * E;
    int64_t grid = (n + 31) / 32;  // 32 outputs per CTA
    if (grid > 8LL * device_sm_count()) grid = 8LL * device_sm_count();
    dwg_reduce_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(n, S, part, dWg);
    st = cudaGetLastError();
  }
  if (st != cudaSuccess || dgb == nullptr) return st;
  dgb_kernel<<<E, 256, 0, s>>>(T, E, dl, dgb);
  return cudaGetLastError();
}

cudaError_t launch_dx_router(int T, int h, int E, const float* dl, const float* Wg, float* out,
                             cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 small_grid((T + 63) / 64, (h + 255) / 256);
  if (E <= 8)
    dx_router_small_kernel<8><<<small_grid, 256, 0, s>>>(T, h, E, dl, Wg, out);
  else if (E <= 16)
    dx_router_small_kernel<16><<<small_grid, 256, 0, s>>>(T, h, E, dl, Wg, out);
  else
    dx_router_kernel<<<dim3((T + 63) / 64, (h + 63) / 64), 256, 0, s>>>(T, h, E, dl, Wg, out);
  return cudaGetLastError();
}

bool router_grads_on_tc(int E) { return E >= 64 && E % 64 == 0; }

cudaError_t launch_router_grads_tc(int T, int h, int E, const void* x, const float* dl,
                                   const float* Wg, void* dl3, void* wg3, float* dwg2, float* dWg,
                                   float* dgb, float* dx_router, int* err, cudaStream_t s) {
  if (!router_grads_on_tc(E)) return cudaErrorInvalidValue;
  const int cap = 8 * device_sm_count();
  auto blocks = [&](int64_t n) {
    const int64_t b = (n + 255) / 256;
    return static_cast<unsigned>(b < cap ? (b > 0 ? b : 1) : cap);
  };
  __nv_bfloat16* d3 = static_cast<__nv_bfloat16*>(dl3);
  __nv_bfloat16* w3 = static_cast<__nv_bfloat16*>(wg3);
  split3_kernel<<<blocks(static_cast<int64_t>(T) * E), 256, 0, s>>>(T, E, 0, dl, d3);
  split3_kernel<<<blocks(static_cast<int64_t>(h) * E), 256, 0, s>>>(h, E, 1, Wg, w3);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  // dWg: one dense group over the T tokens, M = h, N = 2E ([hi | lo] of dl3)
  st = launch_tc_wgrad(1, h, 2 * E, T, x, h, d3, 3 * E, nullptr, dwg2, err, s);
  if (st != cudaSuccess) return st;
  fold_halves_kernel<<<blocks(static_cast<int64_t>(h) * E), 256, 0, s>>>(
      static_cast<int64_t>(h) * E, E, dwg2, dWg);
  st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  if (dgb != nullptr) {
    dgb_kernel<<<E, 256, 0, s>>>(T, E, dl, dgb);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  return launch_tc_dense_nt_f32(T, 3 * E, h, d3, w3, dx_router, h, err, s);
}

}  // namespace moe
