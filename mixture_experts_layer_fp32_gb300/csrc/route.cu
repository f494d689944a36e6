// Router of the MoE layer forward, following the page "MoE我们喜欢你（三）：
// Megatron Core MoE 源码路径解析" (r00kie-liu.github.io):
//   §3 Gating            logits = x . Wg (+ bias) with the router math in fp32
//   §4-§5 Score function softmax before/after top-k, or sigmoid with a
//                        choice-only expert bias and renormalisation
//   §8 Token dropping    per-expert capacity, policy "probs" or "position"
//
// Kernels:
//   router_logits_kernel  fp32 SIMT GEMM, CTA tile BT tokens x ET experts,
//                         K staged through shared memory in BK chunks
//                         (double-buffered), each thread a TT x TE micro-tile.
//   router_topk_kernel    one warp per token: scores, top-k by k rounds of a
//                         warp arg-max (ties -> lower expert id), weights,
//                         per-expert counts via a block histogram.
//   drop_select_kernel    one CTA per expert: if over capacity, a radix
//                         select over 64-bit keys (prob bits, then ~token)
//                         finds the capacity-th best pair; worse pairs drop.
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;

template <typename XT>
struct XVec;  // 16-byte vector of x elements
template <>
struct XVec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
};
template <>
struct XVec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(b[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};

// logits[t, e] = sum_i x[t, i] * Wg[i, e] + gate_bias[e], fp32 FMA.
template <int BT, int ET, int TT, int TE, int BK, typename XT>
__global__ void __launch_bounds__(kRouteThreads)
    router_logits_kernel(int T, int h, int E, const XT* __restrict__ x,
                         const float* __restrict__ Wg, const float* __restrict__ gate_bias,
                         float* __restrict__ logits) {
  constexpr int NTE = ET / TE;
  constexpr int NTT = BT / TT;
  static_assert(NTE * NTT == kRouteThreads, "thread layout");
  constexpr int V = XVec<XT>::N;                 // elements per 16-byte vector
  constexpr int XVECS = BT * BK / V;             // vectors per x tile
  constexpr int XPT = (XVECS + kRouteThreads - 1) / kRouteThreads;
  constexpr int WPT = (BK * ET + kRouteThreads - 1) / kRouteThreads;
  constexpr int XS = BT + 4;                     // padded row of the transposed x tile

  __shared__ __align__(16) float xs[2][BK][XS];
  __shared__ __align__(16) float wsm[2][BK][ET];

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * BT;
  const int e0 = blockIdx.y * ET;
  const int te = tid % NTE;
  const int tt = tid / NTE;

  float xr[XPT][V];
  float wr[WPT];

  auto load_tiles = [&](int k0) {
#pragma unroll
    for (int r = 0; r < XPT; ++r) {
      const int v = tid + r * kRouteThreads;
      const int row = v / (BK / V);
      const int kk = (v % (BK / V)) * V;
      const bool ok = v < XVECS && (t0 + row) < T && (k0 + kk) < h;
      if (ok) {
        XVec<XT>::load(x + (int64_t)(t0 + row) * h + k0 + kk, xr[r]);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) xr[r][i] = 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < WPT; ++r) {
      const int v = tid + r * kRouteThreads;
      const int kk = v / ET;
      const int ee = v % ET;
      wr[r] = (v < BK * ET && (k0 + kk) < h && (e0 + ee) < E) ? Wg[(int64_t)(k0 + kk) * E + e0 + ee]
                                                              : 0.f;
    }
  };
  auto store_tiles = [&](int buf) {
#pragma unroll
    for (int r = 0; r < XPT; ++r) {
      const int v = tid + r * kRouteThreads;
      if (v < XVECS) {
        const int row = v / (BK / V);
        const int kk = (v % (BK / V)) * V;
#pragma unroll
        for (int i = 0; i < V; ++i) xs[buf][kk + i][row] = xr[r][i];
      }
    }
#pragma unroll
    for (int r = 0; r < WPT; ++r) {
      const int v = tid + r * kRouteThreads;
      if (v < BK * ET) wsm[buf][v / ET][v % ET] = wr[r];
    }
  };

  float acc[TT][TE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.f;

  const int nk = (h + BK - 1) / BK;
  load_tiles(0);
  store_tiles(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    if (kt + 1 < nk) load_tiles((kt + 1) * BK);
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[TT], b[TE];
#pragma unroll
      for (int i = 0; i < TT; ++i) a[i] = xs[cur][kk][tt * TT + i];
#pragma unroll
      for (int j = 0; j < TE; ++j) b[j] = wsm[cur][kk][te * TE + j];
#pragma unroll
      for (int i = 0; i < TT; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < nk) store_tiles(cur ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const int t = t0 + tt * TT + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TE; ++j) {
      const int e = e0 + te * TE + j;
      if (e < E) logits[(int64_t)t * E + e] = acc[i][j] + (gate_bias ? gate_bias[e] : 0.f);
    }
  }
}

template <typename XT, int ET, int TE, int TT, int BK>
cudaError_t launch_logits_variant(int T, int h, int E, const XT* x, const float* Wg,
                                  const float* gb, float* logits, cudaStream_t s) {
  constexpr int NTE = ET / TE;
  constexpr int NTT = kRouteThreads / NTE;
  constexpr int BT = NTT * TT;
  dim3 grid((T + BT - 1) / BT, (E + ET - 1) / ET);
  router_logits_kernel<BT, ET, TT, TE, BK, XT><<<grid, kRouteThreads, 0, s>>>(T, h, E, x, Wg, gb,
                                                                              logits);
  return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_logits_typed(int T, int h, int E, const XT* x, const float* Wg,
                                const float* gb, float* logits, cudaStream_t s) {
  if (E <= 8) return launch_logits_variant<XT, 8, 1, 1, 64>(T, h, E, x, Wg, gb, logits, s);
  if (E <= 16) return launch_logits_variant<XT, 16, 2, 1, 64>(T, h, E, x, Wg, gb, logits, s);
  if (E <= 32) return launch_logits_variant<XT, 32, 4, 1, 64>(T, h, E, x, Wg, gb, logits, s);
  return launch_logits_variant<XT, 64, 4, 4, 32>(T, h, E, x, Wg, gb, logits, s);
}

// ------------------------------------------------------------------ top-k
constexpr int kMaxPerLane = MOE_MAX_EXPERTS / 32;  // 8

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(256)
    router_topk_kernel(int T, int E, int k, int score, const float* __restrict__ logits,
                       const float* __restrict__ expert_bias, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_prob, uint8_t* __restrict__ keep,
                       uint8_t* __restrict__ routing_map, int32_t* __restrict__ counts,
                       int* __restrict__ err) {
  __shared__ int hist[MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  for (int t = blockIdx.x * nwarps + warp; t < T; t += gridDim.x * nwarps) {
    const float* lrow = logits + (int64_t)t * E;
    float s[kMaxPerLane], sel[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      s[i] = (e < E) ? lrow[e] : -FLT_MAX;
    }
    if (score == MOE_SCORE_SOFTMAX_PRE) {
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) m = fmaxf(m, s[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        s[i] = (e < E) ? expf(s[i] - m) : 0.f;
        z += s[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        s[i] = (e < E) ? s[i] / z : 0.f;
        sel[i] = (e < E) ? s[i] : -FLT_MAX;
      }
    } else if (score == MOE_SCORE_SIGMOID) {
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          s[i] = 1.f / (1.f + expf(-s[i]));
          sel[i] = expert_bias ? s[i] + expert_bias[e] : s[i];
        } else {
          s[i] = 0.f;
          sel[i] = -FLT_MAX;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) sel[i] = s[i];
    }

    // k rounds of a warp-wide arg-max over the not-yet-taken experts
    uint32_t taken = 0;
    int my_idx = -1;   // lane j < k keeps slot j
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !(taken >> i & 1u) && better(sel[i], e, bv, bi)) {
          bv = sel[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi < 0 || bi >= E) {  // only on NaN logits
        if (lane == 0) report_error(err, DEV_ERR_INDEX, t);
        bi = 0;
      }
      const int owner = bi & 31;
      float sv = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (lane == owner && (bi >> 5) == i) {
          taken |= 1u << i;
          sv = s[i];
        }
      sv = __shfl_sync(0xffffffffu, sv, owner);
      if (lane == j) {
        my_idx = bi;
        my_s = sv;
      }
    }

    // combine weights
    float p = 0.f;
    if (score == MOE_SCORE_SOFTMAX_POST) {
      const float m = __shfl_sync(0xffffffffu, my_s, 0);
      const float ex = (lane < k) ? expf(my_s - m) : 0.f;
      float z = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      p = ex / z;
    } else if (score == MOE_SCORE_SOFTMAX_PRE) {
      p = my_s;
    } else {
      float z = (lane < k) ? my_s : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      p = my_s / (z + 1e-20f);
    }
    if (lane < k) {
      topk_idx[(int64_t)t * k + lane] = my_idx;
      topk_prob[(int64_t)t * k + lane] = p;
      keep[(int64_t)t * k + lane] = 1;
      atomicAdd(&hist[my_idx], 1);
    }
    if (routing_map) {
      int chosen[MOE_MAX_TOPK];
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) chosen[j] = __shfl_sync(0xffffffffu, my_idx, j);
      for (int e = lane; e < E; e += 32) {
        bool hit = false;
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) hit |= (j < k && chosen[j] == e);
        routing_map[(int64_t)t * E + e] = hit ? 1 : 0;
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// ------------------------------------------------------------------ drop
__global__ void __launch_bounds__(1024)
    drop_select_kernel(int k, int E, int64_t capacity, int policy,
                       const int32_t* __restrict__ cand_offsets,
                       const int32_t* __restrict__ cand_pair, float* __restrict__ topk_prob,
                       uint8_t* __restrict__ keep, uint8_t* __restrict__ routing_map,
                       int32_t* __restrict__ kept_per_expert) {
  const int e = blockIdx.x;
  const int begin = cand_offsets[e];
  const int n = cand_offsets[e + 1] - begin;
  if (capacity < 0 || n <= capacity) {
    if (threadIdx.x == 0) kept_per_expert[e] = n;
    return;
  }
  const int cap = static_cast<int>(capacity);
  __shared__ int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_remaining;

  auto key_of = [&](int r) -> unsigned long long {
    const int pair = cand_pair[begin + r];
    const uint32_t pb = __float_as_uint(topk_prob[pair]);  // probabilities are >= 0
    const uint32_t tok = static_cast<uint32_t>(pair / k);
    return (static_cast<unsigned long long>(pb) << 32) | (0xFFFFFFFFu - tok);
  };

  unsigned long long thr = 0;
  if (policy == MOE_DROP_PROBS) {
    if (threadIdx.x == 0) {
      s_prefix = 0ull;
      s_remaining = cap;  // rank (1-based, from the top) of the threshold key
    }
    unsigned long long mask = 0ull;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      const unsigned long long prefix = s_prefix;
      for (int r = threadIdx.x; r < n; r += blockDim.x) {
        const unsigned long long key = key_of(r);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int cum = 0, rem = s_remaining;
        for (int b = 255; b >= 0; --b) {
          if (cum + hist[b] >= rem) {
            s_remaining = rem - cum;
            s_prefix = prefix | (static_cast<unsigned long long>(b) << shift);
            break;
          }
          cum += hist[b];
        }
      }
      mask |= 255ull << shift;
      __syncthreads();
    }
    thr = s_prefix;  // keys are unique: exactly `cap` keys are >= thr
  }
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const bool kept = (policy == MOE_DROP_PROBS) ? (key_of(r) >= thr) : (r < cap);
    if (!kept) {
      const int pair = cand_pair[begin + r];
      keep[pair] = 0;
      topk_prob[pair] = 0.f;
      if (routing_map) routing_map[static_cast<int64_t>(pair / k) * E + e] = 0;
    }
  }
  if (threadIdx.x == 0) kept_per_expert[e] = cap;
}

}  // namespace

cudaError_t launch_router_logits(int T, int h, int E, int dtype, const void* x, const float* Wg,
                                 const float* gate_bias, float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (dtype == MOE_F32)
    return launch_logits_typed<float>(T, h, E, static_cast<const float*>(x), Wg, gate_bias,
                                      logits, s);
  return launch_logits_typed<__nv_bfloat16>(T, h, E, static_cast<const __nv_bfloat16*>(x), Wg,
                                            gate_bias, logits, s);
}

cudaError_t launch_router_topk(int T, int E, int k, int score, const float* logits,
                               const float* expert_bias, int32_t* topk_idx, float* topk_prob,
                               uint8_t* keep, uint8_t* routing_map, int32_t* counts, int* err,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = 8;
  int blocks = (T + warps_per_block - 1) / warps_per_block;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  router_topk_kernel<<<blocks, 32 * warps_per_block, 0, s>>>(
      T, E, k, score, logits, expert_bias, topk_idx, topk_prob, keep, routing_map, counts, err);
  return cudaGetLastError();
}

cudaError_t launch_drop_select(int T, int E, int k, int64_t capacity, int policy,
                               const int32_t* cand_offsets, const int32_t* cand_pair,
                               float* topk_prob, uint8_t* keep, uint8_t* routing_map,
                               int32_t* kept_per_expert, cudaStream_t s) {
  (void)T;
  drop_select_kernel<<<E, 1024, 0, s>>>(k, E, capacity, policy, cand_offsets, cand_pair,
                                        topk_prob, keep, routing_map, kept_per_expert);
  return cudaGetLastError();
}

}  // namespace moe
