// Router of the MoE layer forward, following the page "MoE我们喜欢你（三）：
// Megatron Core MoE 源码路径解析" (r00kie-liu.github.io):
//   §3 Gating            logits = x . Wg (+ bias) with the router math in fp32
//   §4-§5 Score function softmax before/after top-k, or sigmoid / sqrtsoftplus
//                        with a choice-only expert bias and renormalisation;
//                        optionally group-limited (compute_topk's num_groups,
//                        group_topk: the best group_topk groups by the sum of
//                        their k/group_topk best scores, top-k inside them)
//   §8 Token dropping    per-expert capacity, policy "probs" or "position"
//
// Kernels:
//   router_fused_small_e_kernel  E <= 8: logits and top-k in one pass over x,
//                         the gate matrix staged in shared memory.
//   router_sgemm_kernel   E >= 64 (E % 4 == 0): register-blocked fp32 GEMM
//                         (8 x 8 micro-tiles, paired FMAs), operands through a
//                         4-stage cp.async ring, K split S ways into partial sums.
//   router_logits_kernel  other shapes: fp32 SIMT GEMM, CTA tile BT tokens x
//                         ET experts, K staged through shared memory in BK
//                         chunks (double-buffered), a TT x TE micro-tile each.
//   router_split3_kernel  the opt-in tensor-core logits: Wg as three exact
//                         bf16 pieces, transposed (the GEMM is gemm_tc.cu's).
//   router_topk_kernel    one warp per token: scores, (group scores and the
//                         kept groups), top-k by k rounds of a warp arg-max
//                         (ties -> lower expert / group id), weights,
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

// partial logits[t, e] = sum_i x[t, i] * Wg[i, e], fp32 FMA (the gate bias is
// added by the top-k kernel).
template <int BT, int ET, int TT, int TE, int BK, typename XT>
__global__ void __launch_bounds__(kRouteThreads)
    router_logits_kernel(int T, int h, int E, const XT* __restrict__ x,
                         const float* __restrict__ Wg, float* __restrict__ logits) {
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
      if (e < E) logits[(int64_t)t * E + e] = acc[i][j];
    }
  }
}

template <typename XT, int ET, int TE, int TT, int BK>
cudaError_t launch_logits_variant(int T, int h, int E, const XT* x, const float* Wg,
                                  float* logits, cudaStream_t s) {
  constexpr int NTE = ET / TE;
  constexpr int NTT = kRouteThreads / NTE;
  constexpr int BT = NTT * TT;
  dim3 grid((T + BT - 1) / BT, (E + ET - 1) / ET);
  router_logits_kernel<BT, ET, TT, TE, BK, XT><<<grid, kRouteThreads, 0, s>>>(T, h, E, x, Wg,
                                                                              logits);
  return cudaGetLastError();
}

// Small-E logits (E <= 8): the gate rows of one slice of h, padded to 8
// experts, sit in shared memory; each warp takes 4 tokens at a time, lane l
// streams the 16-byte x vectors l, l+32, ... of that slice of those 4 rows
// (kept packed in registers, several loads in flight per lane) and
// accumulates 4 x 8 partial dot products; a 5-step shuffle reduce-scatter
// then leaves the total of (token l/8, expert l%8) in lane l.  gridDim.y
// splits h into slices (two CTAs fit per SM); each slice writes its own
// partial sums.
constexpr int kSmallE = 8;
constexpr int kSmallTok = 4;
constexpr int kSmallUnroll = 4;

// Gate row r (8 fp32) is two 16-byte chunks, 2r and 2r+1.  Lanes read rows
// 8 apart, i.e. chunks 256 bytes apart: all in one bank group.  XOR-ing the
// chunk's position inside its 128-byte line with (chunk / 16) % 8 spreads a
// quarter-warp over the 8 bank groups.
__device__ __forceinline__ int swz_chunk(int i) { return (i & ~7) | ((i & 7) ^ ((i >> 4) & 7)); }

template <typename XT>
struct Packed;  // element c of a 16-byte vector kept as raw bits
template <>
struct Packed<float> {
  __device__ static float at(const uint4& q, int c) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    return __uint_as_float(w[c]);
  }
};
template <>
struct Packed<__nv_bfloat16> {
  __device__ static float at(const uint4& q, int c) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const uint32_t b = (c & 1) ? (w[c >> 1] & 0xFFFF0000u) : (w[c >> 1] << 16);
    return __uint_as_float(b);
  }
};

// Gate rows [hb, hb + hn) of Wg [h, E], padded to 8 experts, into shared
// memory in the chunk swizzle (by the whole CTA; the caller synchronises).
__device__ __forceinline__ void stage_gate_rows(const float* __restrict__ Wg, int E, int hb,
                                                int hn, float* wsm) {
  if (E == kSmallE && (reinterpret_cast<uintptr_t>(Wg) & 15) == 0) {
    // 16-byte copies, 8 loads in flight per thread before their stores
    const float4* src = reinterpret_cast<const float4*>(Wg + (int64_t)hb * kSmallE);
    float4* dst = reinterpret_cast<float4*>(wsm);
    const int n4 = hn * kSmallE / 4;
    for (int i0 = threadIdx.x; i0 < n4; i0 += blockDim.x * 8) {
      float4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * (int)blockDim.x < n4) r[u] = src[i0 + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * (int)blockDim.x < n4) dst[swz_chunk(i0 + u * blockDim.x)] = r[u];
    }
  } else {
    for (int i0 = threadIdx.x; i0 < hn * kSmallE; i0 += blockDim.x * 8) {
      float r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * blockDim.x;
        const int row = i / kSmallE, e = i % kSmallE;
        r[u] = (i < hn * kSmallE && e < E) ? Wg[(int64_t)(hb + row) * E + e] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < hn * kSmallE) wsm[swz_chunk(i >> 2) * 4 + (i & 3)] = r[u];
      }
    }
  }
}

// Dot products of the 4 tokens t0 .. t0+3 with the 8 staged gate columns over
// features [hb, hb + hn) (hb, hn multiples of the vector width), by one
// warp: lane l returns the sum for token t0 + l/8, expert l%8 (0 past T).
template <typename XT>
__device__ __forceinline__ float small_e_group_logits(const XT* __restrict__ x, int T, int h,
                                                      int hb, int hn, const float* wsm, int t0,
                                                      int lane) {
  constexpr int V = XVec<XT>::N;
  const int nvec = hn / V;
  const uint4* xq = reinterpret_cast<const uint4*>(x);
  const int row_vecs = h / V;
  const int vb = hb / V;
  float acc[kSmallTok * kSmallE];
#pragma unroll
  for (int i = 0; i < kSmallTok * kSmallE; ++i) acc[i] = 0.f;
  for (int v0 = lane; v0 < nvec; v0 += 32 * kSmallUnroll) {
    uint4 xr[kSmallUnroll][kSmallTok];
#pragma unroll
    for (int u = 0; u < kSmallUnroll; ++u) {
      const int v = v0 + 32 * u;
#pragma unroll
      for (int tk = 0; tk < kSmallTok; ++tk)
        xr[u][tk] = (v < nvec && t0 + tk < T) ? xq[(int64_t)(t0 + tk) * row_vecs + vb + v]
                                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kSmallUnroll; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const float4* wr = reinterpret_cast<const float4*>(wsm);
        const int chunk = 2 * (v * V + c);
        const float4 w0 = wr[swz_chunk(chunk)], w1 = wr[swz_chunk(chunk + 1)];
        const float w[kSmallE] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int tk = 0; tk < kSmallTok; ++tk) {
          const float xe = Packed<XT>::at(xr[u][tk], c);
#pragma unroll
          for (int e = 0; e < kSmallE; ++e)
            acc[tk * kSmallE + e] = fmaf(xe, w[e], acc[tk * kSmallE + e]);
        }
      }
    }
  }
  // reduce-scatter: after the step with offset o, a lane keeps the half of
  // its values selected by (lane & o); at the end lane l holds index l.
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float keep = upper ? acc[j + n / 2] : acc[j];
      const float send = upper ? acc[j] : acc[j + n / 2];
      acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return acc[0];
}

template <typename XT>
__global__ void __launch_bounds__(kRouteThreads, 2)
    router_logits_small_e_kernel(int T, int h, int E, int hslice, const XT* __restrict__ x,
                                 const float* __restrict__ Wg, float* __restrict__ partials) {
  extern __shared__ __align__(16) float wsm_small[];  // [hslice][8], chunk-swizzled
  const int hb = blockIdx.y * hslice;                  // first feature of this slice
  const int hn = min(hslice, h - hb);                  // features in this slice
  float* logits = partials + (int64_t)blockIdx.y * T * E;
  stage_gate_rows(Wg, E, hb, hn, wsm_small);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int groups = (T + kSmallTok - 1) / kSmallTok;
  for (int g = blockIdx.x * (kRouteThreads / 32) + warp; g < groups;
       g += gridDim.x * (kRouteThreads / 32)) {
    const int t0 = g * kSmallTok;
    const float v = small_e_group_logits<XT>(x, T, h, hb, hn, wsm_small, t0, lane);
    const int t = t0 + lane / kSmallE;
    const int e = lane % kSmallE;
    if (t < T && e < E) logits[(int64_t)t * E + e] = v;
  }
}

constexpr int kSmallESliceMax = 3072;  // 3072 x 8 x 4 B = 96 KB: two CTAs per SM
constexpr int kSmallEMaxHidden = 6 * kSmallESliceMax;

template <typename XT>
cudaError_t launch_logits_small_e(int T, int h, int E, const XT* x, const float* Wg,
                                  float* partials, int* nsplit, cudaStream_t s) {
  // slices of whole 16-byte vectors, at most kSmallESliceMax features each
  constexpr int V = XVec<XT>::N;
  int slices = (h + kSmallESliceMax - 1) / kSmallESliceMax;
  if (slices < 2 && h >= 1024) slices = 2;
  int hslice = (h / V + slices - 1) / slices * V;
  slices = (h + hslice - 1) / hslice;
  *nsplit = slices;
  const int smem = hslice * kSmallE * static_cast<int>(sizeof(float));
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 64 && !configured[dev]) {
    st = cudaFuncSetAttribute(router_logits_small_e_kernel<XT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmallESliceMax * kSmallE * static_cast<int>(sizeof(float)));
    if (st != cudaSuccess) return st;
    configured[dev] = true;
  }
  const int groups = (T + kSmallTok - 1) / kSmallTok;
  int gx = (groups + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
  const int cap = (2 * device_sm_count() + slices - 1) / slices;
  if (gx > cap) gx = cap;
  router_logits_small_e_kernel<XT><<<dim3(gx, slices), kRouteThreads, smem, s>>>(
      T, h, E, hslice, x, Wg, partials);
  return cudaGetLastError();
}

// Large-E logits: a register-blocked SGEMM.  CTA tile 128 tokens x BN
// experts, K in chunks of 16 (double-buffered through shared memory), each
// thread an 8 x 8 micro-tile made of two 4-wide halves (rows ty*4 and
// 64+ty*4, columns tx*4 and BN/2+tx*4) so that a quarter-warp's 16-byte
// shared loads are contiguous.  The micro-tile's FMAs are packed in pairs
// of columns (fp32x2 FMA, each lane a fused multiply-add rounded once, the
// same arithmetic as fmaf): the kernel is bound by instruction issue, and
// the pairs halve the FMA instructions.  Measured on GB300 (2070 MHz):
// DeepSeek-V3 route stage 349 us against 411 us with scalar FMAs, Qwen3
// 434 against 483; two CTAs per SM (128 registers, a few spilled) beat one
// CTA per SM without spills (427 / 513 us).  gridDim.z splits K; each split writes its own
// partial sums, which the top-k kernel adds in split order.  Operands move by
// cp.async through a 4-stage ring (raw x and gate rows, 3 K tiles ahead),
// and each K tile's x is converted to fp32 into a transposed double buffer
// one tile ahead of its use.
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 16;
constexpr int kMaxSplits = kRouterMaxSplits;

// 16-byte asynchronous global -> shared copy (cp.async, cached in L2 only);
// src_bytes 0 fills the 16 bytes with zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stages of the SGEMM's copy ring: a K tile's raw x rows and gate rows are
// copied kStages - 2 tiles ahead of their conversion and kStages - 1 ahead of
// their use, with no registers held for them.
constexpr int kSgemmStages = 4;

template <int BN, typename XT>
constexpr int sgemm_smem_bytes() {
  return kSgemmStages * (kGemmBM * kGemmBK * static_cast<int>(sizeof(XT)) + kGemmBK * BN * 4) +
         2 * kGemmBK * kGemmBM * 4;
}

template <int BN, typename XT>
__global__ void __launch_bounds__(BN * 2, 256 / BN)
    router_sgemm_kernel(int T, int h, int E, int k_per_split, const XT* __restrict__ x,
                        const float* __restrict__ Wg, float* __restrict__ partials) {
  constexpr int TX = BN / 8;          // threads along experts
  constexpr int NT = TX * 16;         // threads
  constexpr int V = XVec<XT>::N;
  constexpr int AV = kGemmBM * kGemmBK / V;      // x vectors (16 bytes) per tile
  constexpr int APT = (AV + NT - 1) / NT;
  constexpr int BV = kGemmBK * BN / 4;           // Wg float4 per tile
  constexpr int BPT = BV / NT;
  static_assert(AV % NT == 0 && BV % NT == 0, "copy split");
  // dynamic shared memory: Araw[kSgemmStages][BM][BK] (x as stored), then
  // Bs[kSgemmStages][BK][BN], then As[2][BK][BM] (x in fp32, transposed)
  extern __shared__ __align__(16) uint8_t sgemm_smem[];
  XT* Araw = reinterpret_cast<XT*>(sgemm_smem);
  float* Bs = reinterpret_cast<float*>(sgemm_smem + kSgemmStages * kGemmBM * kGemmBK * sizeof(XT));
  float* As = Bs + kSgemmStages * kGemmBK * BN;

  const int tid = threadIdx.x;
  const int tx = tid % TX, ty = tid / TX;
  const int t0 = blockIdx.x * kGemmBM;
  const int e0 = blockIdx.y * BN;
  const int kbeg = blockIdx.z * k_per_split;
  const int kend = min(h, kbeg + k_per_split);
  float* out = partials + (int64_t)blockIdx.z * T * E;

  // copies of K tile kt into ring stage kt % kSgemmStages (zeros past T, E or
  // the split's end), one commit group per tile (empty past the last)
  const int nk = (kend - kbeg + kGemmBK - 1) / kGemmBK;
  auto issue = [&](int kt) {
    if (kt < nk) {
      const int k0 = kbeg + kt * kGemmBK;
      const int st = kt % kSgemmStages;
#pragma unroll
      for (int r = 0; r < APT; ++r) {
        const int v = tid + r * NT;
        const int row = v / (kGemmBK / V), kk = (v % (kGemmBK / V)) * V;
        const bool ok = t0 + row < T && k0 + kk < kend;
        cp_async16(Araw + ((int64_t)st * kGemmBM + row) * kGemmBK + kk,
                   ok ? static_cast<const void*>(x + (int64_t)(t0 + row) * h + k0 + kk) : x,
                   ok ? 16 : 0);
      }
#pragma unroll
      for (int r = 0; r < BPT; ++r) {
        const int v = tid + r * NT;
        const int kk = v / (BN / 4), cc = (v % (BN / 4)) * 4;
        const bool ok = k0 + kk < kend && e0 + cc < E;
        cp_async16(Bs + ((int64_t)st * kGemmBK + kk) * BN + cc,
                   ok ? static_cast<const void*>(Wg + (int64_t)(k0 + kk) * E + e0 + cc) : Wg,
                   ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  // x of K tile kt, from its ring stage to fp32 in As[buf] (transposed: [k][row])
  auto convert = [&](int kt, int buf) {
    const int st = kt % kSgemmStages;
#pragma unroll
    for (int r = 0; r < APT; ++r) {
      const int v = tid + r * NT;
      const int row = v / (kGemmBK / V), kk = (v % (kGemmBK / V)) * V;
      float f[V];
      XVec<XT>::load(Araw + ((int64_t)st * kGemmBM + row) * kGemmBK + kk, f);
#pragma unroll
      for (int c2 = 0; c2 < V; ++c2) As[(buf * kGemmBK + kk + c2) * kGemmBM + row] = f[c2];
    }
  };

  // acc[i][jj]: micro-tile row i, columns 2jj and 2jj+1 (packed: one
  // fp32x2 FMA instruction updates both, halving the FMA instructions)
  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

#pragma unroll
  for (int kt = 0; kt < kSgemmStages - 1; ++kt) issue(kt);
  if (nk > 0) {
    cp_async_wait<kSgemmStages - 2>();  // tile 0 has landed (this thread's copies)
    __syncthreads();
    convert(0, 0);
  }
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    // tiles <= kt + 1 have landed; the barrier also publishes As[cur] and
    // frees the ring stage and As buffer that iteration kt - 1 read
    cp_async_wait<kSgemmStages - 3>();
    __syncthreads();
    if (kt + 1 < nk) convert(kt + 1, cur ^ 1);
    issue(kt + kSgemmStages - 1);
    const float* Ac = As + cur * kGemmBK * kGemmBM;
    const float* Bc = Bs + (kt % kSgemmStages) * kGemmBK * BN;
#pragma unroll
    for (int kk = 0; kk < kGemmBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(Ac + kk * kGemmBM + ty * 4);
      const float4 a1 = *reinterpret_cast<const float4*>(Ac + kk * kGemmBM + 64 + ty * 4);
      const float4 b0 = *reinterpret_cast<const float4*>(Bc + kk * BN + tx * 4);
      const float4 b1 = *reinterpret_cast<const float4*>(Bc + kk * BN + BN / 2 + tx * 4);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                           make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
      }
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (t >= T) continue;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int e = e0 + half * (BN / 2) + tx * 4;
      if (e < E)  // E % 4 == 0 on this path: the 4 columns are all valid
        *reinterpret_cast<float4*>(out + (int64_t)t * E + e) =
            make_float4(acc[i][half * 2].x, acc[i][half * 2].y, acc[i][half * 2 + 1].x,
                        acc[i][half * 2 + 1].y);
    }
  }
}

template <int BN, typename XT>
cudaError_t launch_sgemm(int T, int h, int E, const XT* x, const float* Wg, float* partials,
                         int max_splits, int* nsplit, cudaStream_t s) {
  // choose the split count that minimises the most CTAs any SM runs, per
  // unit of split work: ceil(tiles * S / SMs) / S (plus a small cost per
  // split for the partial sums), with at least 16 K chunks per split
  const int tiles = ((T + kGemmBM - 1) / kGemmBM) * ((E + BN - 1) / BN);
  const int sms = device_sm_count();
  int splits = 1;
  double best = 1e30;
  for (int S = 1; S <= max_splits && S <= h / 256; ++S) {
    const double cost = double((int64_t(tiles) * S + sms - 1) / sms) / S + 0.002 * S;
    if (cost < best - 1e-9) {
      best = cost;
      splits = S;
    }
  }
  int kps = (h + splits - 1) / splits;
  kps = (kps + kGemmBK - 1) / kGemmBK * kGemmBK;
  splits = (h + kps - 1) / kps;
  *nsplit = splits;
  dim3 grid((T + kGemmBM - 1) / kGemmBM, (E + BN - 1) / BN, splits);
  constexpr int smem = sgemm_smem_bytes<BN, XT>();
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    st = cudaFuncSetAttribute(router_sgemm_kernel<BN, XT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (st != cudaSuccess) return st;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  router_sgemm_kernel<BN, XT><<<grid, BN * 2, smem, s>>>(T, h, E, kps, x, Wg, partials);
  return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_logits_typed(int T, int h, int E, const XT* x, const float* Wg,
                                float* partials, int max_splits, int* nsplit, cudaStream_t s) {
  *nsplit = 1;
  const bool wg16 = (reinterpret_cast<uintptr_t>(Wg) & 15) == 0;  // 16-byte gate loads
  if (E <= kSmallE && h <= kSmallEMaxHidden)
    return launch_logits_small_e<XT>(T, h, E, x, Wg, partials, nsplit, s);
  if (wg16 && E % 4 == 0 && E >= 64) {
    if (E % 128 == 0)
      return launch_sgemm<128, XT>(T, h, E, x, Wg, partials, max_splits, nsplit, s);
    return launch_sgemm<64, XT>(T, h, E, x, Wg, partials, max_splits, nsplit, s);
  }
  if (E <= 8) return launch_logits_variant<XT, 8, 1, 1, 64>(T, h, E, x, Wg, partials, s);
  if (E <= 16) return launch_logits_variant<XT, 16, 2, 1, 64>(T, h, E, x, Wg, partials, s);
  if (E <= 32) return launch_logits_variant<XT, 32, 4, 1, 64>(T, h, E, x, Wg, partials, s);
  return launch_logits_variant<XT, 64, 4, 4, 32>(T, h, E, x, Wg, partials, s);
}

// ------------------------------------------------------------------ top-k
constexpr int kMaxPerLane = MOE_MAX_EXPERTS / 32;  // 8
constexpr int kTopkWarps = 8;                       // warps (tokens in flight) per CTA

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// PL: experts per lane (E <= 32 * PL): the per-lane loops cover no more
// entries than E needs.
template <int PL>
__global__ void __launch_bounds__(256)
    router_topk_kernel(int T, int E, int k, int score, int num_groups, int group_topk,
                       const float* __restrict__ logits,
                       int nsplit, const float* __restrict__ gate_bias,
                       const float* __restrict__ expert_bias, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_prob, uint8_t* __restrict__ keep,
                       uint8_t* __restrict__ routing_map, int32_t* __restrict__ counts,
                       int* __restrict__ err) {
  __shared__ int hist[MOE_MAX_EXPERTS];
  __shared__ float gsel[kTopkWarps][MOE_MAX_EXPERTS];  // per warp: a token's selection scores
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int per_group = num_groups > 1 ? E / num_groups : E;
  for (int t = blockIdx.x * nwarps + warp; t < T; t += gridDim.x * nwarps) {
    // logits = (partial sums in split order) + gate bias; the partial sums
    // are loaded SB splits at a time before they are added, so the loads
    // overlap instead of waiting on one another (SB = 2 at 8 experts per
    // lane keeps the batch in registers)
    constexpr int SB = PL >= 8 ? 2 : 4;
    float s[PL], sel[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      s[i] = e < E ? logits[(int64_t)t * E + e] : 0.f;
    }
    for (int sp = 1; sp < nsplit; sp += SB) {
      float v[SB][PL];
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int i = 0; i < PL; ++i) {
          const int e = lane + 32 * i;
          v[j][i] = (sp + j < nsplit && e < E) ? logits[((int64_t)(sp + j) * T + t) * E + e] : 0.f;
        }
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int i = 0; i < PL; ++i)
          if (sp + j < nsplit) s[i] += v[j][i];
    }
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      s[i] = e < E ? (gate_bias ? s[i] + gate_bias[e] : s[i]) : -FLT_MAX;
    }
    if (score == MOE_SCORE_SOFTMAX_PRE) {
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < PL; ++i) m = fmaxf(m, s[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        s[i] = (e < E) ? expf(s[i] - m) : 0.f;
        z += s[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        s[i] = (e < E) ? s[i] / z : 0.f;
        sel[i] = (e < E) ? s[i] : -FLT_MAX;
      }
    } else if (score == MOE_SCORE_SIGMOID || score == MOE_SCORE_SQRTSOFTPLUS) {
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          if (score == MOE_SCORE_SIGMOID) {
            s[i] = 1.f / (1.f + expf(-s[i]));
          } else {
            // softplus(l) = log(1 + e^l) = max(l, 0) + log1p(e^-|l|): no overflow
            s[i] = sqrtf(fmaxf(s[i], 0.f) + log1pf(expf(-fabsf(s[i]))));
          }
          sel[i] = expert_bias ? s[i] + expert_bias[e] : s[i];
        } else {
          s[i] = 0.f;
          sel[i] = -FLT_MAX;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < PL; ++i) sel[i] = s[i];
    }

    // group-limited top-k: lane g < num_groups scores group g (the sum of its
    // k/group_topk best selection scores, largest first), then group_topk
    // rounds of a warp arg-max keep the best groups; the other groups'
    // experts are marked taken so that the expert rounds skip them
    uint32_t taken = 0;
    if (num_groups > 1) {
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) gsel[warp][e] = sel[i];
      }
      __syncwarp();
      float gs = -INFINITY;
      if (lane < num_groups) {
        const float* g = gsel[warp] + lane * per_group;
        const int m = k / group_topk;
        uint32_t used[MOE_MAX_EXPERTS / 32] = {0, 0, 0, 0, 0, 0, 0, 0};
        gs = 0.f;
        for (int r = 0; r < m; ++r) {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          for (int c = 0; c < per_group; ++c)
            if (!(used[c >> 5] >> (c & 31) & 1u) && better(g[c], c, bv, bi)) {
              bv = g[c];
              bi = c;
            }
          if (bi >= per_group) break;  // only on NaN scores (reported by the expert rounds)
          used[bi >> 5] |= 1u << (bi & 31);
          gs += bv;
        }
      }
      __syncwarp();  // gsel is rewritten for the next token
      uint32_t kept = 0;
      for (int r = 0; r < group_topk; ++r) {
        float bv = (lane < num_groups && !(kept >> lane & 1u)) ? gs : -INFINITY;
        int bi = (lane < num_groups && !(kept >> lane & 1u)) ? lane : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (bi < num_groups) kept |= 1u << bi;
      }
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !(kept >> (e / per_group) & 1u)) taken |= 1u << i;
      }
    }

    // k rounds of a warp-wide arg-max over the not-yet-taken experts
    int my_idx = -1;   // lane j < k keeps slot j
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
      // this lane's best candidate as an ordered key (a larger score, a larger
      // key; -0 as +0; 0 = none, NaN scores never count), the lower expert on
      // ties (i rises with e); then the warp's largest key and, among the
      // lanes holding it, the lowest expert: two warp reductions
      uint32_t bk = 0;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !(taken >> i & 1u) && !isnan(sel[i])) {
          uint32_t u = __float_as_uint(sel[i]);
          if (u == 0x80000000u) u = 0u;
          const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
          if (key > bk) {
            bk = key;
            bi = e;
          }
        }
      }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
      bi = static_cast<int>(
          __reduce_min_sync(0xffffffffu, (mk != 0u && bk == mk) ? static_cast<uint32_t>(bi)
                                                                : 0x7fffffffu));
      if (mk == 0u || bi >= E) {  // only on NaN logits
        if (lane == 0) report_error(err, DEV_ERR_INDEX, t);
        bi = 0;
      }
      const int owner = bi & 31;
      float sv = 0.f;
#pragma unroll
      for (int i = 0; i < PL; ++i)
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

// ------------------------------------------------------------------ fused small-E router
// E <= 8 without expert groups: logits and top-k in one kernel (one pass over
// x, no logits buffer, one launch instead of two).  The whole gate matrix,
// padded to 8 experts, sits in shared memory (one CTA per SM).  A warp forms
// the logits of 4 tokens the way the small-E logits kernel does, over all of
// h; afterwards lane 8q + e holds expert e of token t0 + q, so each 8-lane
// segment is one token.  The segment then applies the gate bias, the score
// function, k rounds of an arg-max (ties to the lower expert) and the
// combine weights, with the formulas of the warp-per-token top-k kernel.
constexpr int kFusedThreads = 512;
constexpr int kFusedMaxHidden = 6144;  // 6144 x 8 x 4 B = 192 KB of gate rows

template <typename XT>
__global__ void __launch_bounds__(kFusedThreads, 1)
    router_fused_small_e_kernel(int T, int h, int E, int k, int score, const XT* __restrict__ x,
                                const float* __restrict__ Wg, const float* __restrict__ gate_bias,
                                const float* __restrict__ expert_bias,
                                int32_t* __restrict__ topk_idx, float* __restrict__ topk_prob,
                                uint8_t* __restrict__ keep, uint8_t* __restrict__ routing_map,
                                int32_t* __restrict__ counts, int* __restrict__ err) {
  extern __shared__ __align__(16) float wsm_fused[];  // [h][8] chunk-swizzled, then hist[8]
  int* hist = reinterpret_cast<int*>(wsm_fused + static_cast<size_t>(h) * kSmallE);
  if (threadIdx.x < kSmallE) hist[threadIdx.x] = 0;
  stage_gate_rows(Wg, E, 0, h, wsm_fused);
  __syncthreads();
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int e = lane & (kSmallE - 1);  // this lane's expert in its segment
  const int seg0 = lane & ~(kSmallE - 1);
  const bool ev = e < E;
  const int groups = (T + kSmallTok - 1) / kSmallTok;
  // groups dealt round-robin over the CTAs first (group = warp * grid + CTA),
  // so that every SM gets work when there are fewer groups than warps
  for (int g = warp * gridDim.x + blockIdx.x; g < groups; g += gridDim.x * (kFusedThreads / 32)) {
    const int t = g * kSmallTok + lane / kSmallE;  // this segment's token
    const float l = small_e_group_logits<XT>(x, T, h, 0, h, wsm_fused, g * kSmallTok, lane);
    float sv = ev ? (gate_bias ? l + gate_bias[e] : l) : -FLT_MAX;
    float sel;
    if (score == MOE_SCORE_SOFTMAX_PRE) {
      float m = sv;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kAll, m, o));
      sv = ev ? expf(sv - m) : 0.f;
      float z = sv;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) z += __shfl_xor_sync(kAll, z, o);
      sv = ev ? sv / z : 0.f;
      sel = ev ? sv : -FLT_MAX;
    } else if (score == MOE_SCORE_SIGMOID || score == MOE_SCORE_SQRTSOFTPLUS) {
      if (ev) {
        if (score == MOE_SCORE_SIGMOID)
          sv = 1.f / (1.f + expf(-sv));
        else  // softplus(l) = max(l, 0) + log1p(e^-|l|): no overflow
          sv = sqrtf(fmaxf(sv, 0.f) + log1pf(expf(-fabsf(sv))));
        sel = expert_bias ? sv + expert_bias[e] : sv;
      } else {
        sv = 0.f;
        sel = -FLT_MAX;
      }
    } else {
      sel = sv;
    }

    // k rounds of an arg-max over the segment's not-yet-taken experts; the
    // lane of expert j (j < k) keeps slot j
    bool taken = false;
    int my_idx = -1;
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
      const bool cand = ev && !taken && better(sel, e, -INFINITY, 0x7fffffff);
      float bv = cand ? sel : -INFINITY;
      int bi = cand ? e : 0x7fffffff;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kAll, bv, o);
        const int oi = __shfl_xor_sync(kAll, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi < 0 || bi >= E) {  // only on NaN logits
        if (e == 0 && t < T) report_error(err, DEV_ERR_INDEX, t);
        bi = 0;
      }
      if (e == bi) taken = true;
      const float chosen = __shfl_sync(kAll, sv, seg0 + bi);
      if (e == j) {
        my_idx = bi;
        my_s = chosen;
      }
    }

    // combine weights
    float p = 0.f;
    if (score == MOE_SCORE_SOFTMAX_POST) {
      const float m = __shfl_sync(kAll, my_s, seg0);  // slot 0 holds the largest
      const float ex = (e < k) ? expf(my_s - m) : 0.f;
      float z = ex;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) z += __shfl_xor_sync(kAll, z, o);
      p = ex / z;
    } else if (score == MOE_SCORE_SOFTMAX_PRE) {
      p = my_s;
    } else {
      float z = (e < k) ? my_s : 0.f;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) z += __shfl_xor_sync(kAll, z, o);
      p = my_s / (z + 1e-20f);
    }
    if (t < T) {
      if (e < k) {
        topk_idx[(int64_t)t * k + e] = my_idx;
        topk_prob[(int64_t)t * k + e] = p;
        keep[(int64_t)t * k + e] = 1;
        atomicAdd(&hist[my_idx], 1);
      }
      if (routing_map && ev) routing_map[(int64_t)t * E + e] = taken ? 1 : 0;
    }
  }
  __syncthreads();
  if (threadIdx.x < E && hist[threadIdx.x]) atomicAdd(&counts[threadIdx.x], hist[threadIdx.x]);
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
  constexpr int kCache = 4096;  // candidates whose keys stay in shared memory (32 KB)
  __shared__ unsigned long long skey[kCache];
  __shared__ int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_remaining;
  const int lane = threadIdx.x & 31;

  auto key_of = [&](int r) -> unsigned long long {
    const int pair = cand_pair[begin + r];
    const uint32_t pb = __float_as_uint(topk_prob[pair]);  // probabilities are >= 0
    const uint32_t tok = static_cast<uint32_t>(pair / k);
    return (static_cast<unsigned long long>(pb) << 32) | (0xFFFFFFFFu - tok);
  };
  // keys read from memory once (two dependent loads each), not once per pass
  const bool cached = policy == MOE_DROP_PROBS && n <= kCache;
  if (cached)
    for (int r = threadIdx.x; r < n; r += blockDim.x) skey[r] = key_of(r);
  auto key_at = [&](int r) -> unsigned long long { return cached ? skey[r] : key_of(r); };

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
        const unsigned long long key = key_at(r);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // the bin holding the rem-th largest key: lane l owns bins 255-8l ..
        // 248-8l (descending), a warp prefix sum over the lanes' totals, the
        // first lane whose running total reaches rem walks its 8 bins
        const int rem = s_remaining;
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - (lane * 8 + j)];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, incl >= rem);
        if (hit && lane == __ffs(hit) - 1) {
          int cum = incl - sum;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (cum + c[j] >= rem) {
              s_remaining = rem - cum;
              s_prefix = prefix | (static_cast<unsigned long long>(255 - (lane * 8 + j)) << shift);
              break;
            }
            cum += c[j];
          }
        }
      }
      mask |= 255ull << shift;
      __syncthreads();
    }
    thr = s_prefix;  // keys are unique: exactly `cap` keys are >= thr
  }
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const bool kept = (policy == MOE_DROP_PROBS) ? (key_at(r) >= thr) : (r < cap);
    if (!kept) {
      const int pair = cand_pair[begin + r];
      keep[pair] = 0;
      topk_prob[pair] = 0.f;
      if (routing_map) routing_map[static_cast<int64_t>(pair / k) * E + e] = 0;
    }
  }
  if (threadIdx.x == 0) kept_per_expert[e] = cap;
}

// Gate weights for the tensor-core logits: Wg [h, E] fp32 -> Wk [3E, h] bf16
// (transposed: K contiguous), row p*E + e holding piece p of column e, where
// v = p0 + p1 + p2 + r with p0 = bf16(v), p1 = bf16(v - p0), p2 =
// bf16(v - p0 - p1): each difference is exact in fp32 (it keeps the bits
// below the piece just taken), so the pieces hold v's 24 significant bits and
// |r| <= 2^-27 |v| (normal range).  A non-finite weight goes whole into piece
// 0.  32 x 32 tiles through shared memory, coalesced on both sides.
__global__ void __launch_bounds__(256)
    router_split3_kernel(int h, int E, const float* __restrict__ Wg,
                         __nv_bfloat16* __restrict__ Wk) {
  __shared__ float tile[32][33];
  const int e0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int k = k0 + ty + 8 * i, e = e0 + tx;
    tile[ty + 8 * i][tx] = (k < h && e < E) ? Wg[static_cast<int64_t>(k) * E + e] : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = e0 + ty + 8 * i, k = k0 + tx;
    if (e >= E || k >= h) continue;
    const float v = tile[tx][ty + 8 * i];
    __nv_bfloat16 p0 = __float2bfloat16_rn(v), p1 = __float2bfloat16_rn(0.f), p2 = p1;
    if (isfinite(v)) {
      const float r1 = v - __bfloat162float(p0);
      p1 = __float2bfloat16_rn(r1);
      p2 = __float2bfloat16_rn(r1 - __bfloat162float(p1));
    }
    Wk[static_cast<int64_t>(e) * h + k] = p0;
    Wk[static_cast<int64_t>(E + e) * h + k] = p1;
    Wk[static_cast<int64_t>(2 * E + e) * h + k] = p2;
  }
}

}  // namespace

cudaError_t launch_router_split3(int h, int E, const float* Wg, void* Wk, cudaStream_t s) {
  if (h == 0 || E == 0) return cudaSuccess;
  dim3 grid((E + 31) / 32, (h + 31) / 32);
  router_split3_kernel<<<grid, 256, 0, s>>>(h, E, Wg, static_cast<__nv_bfloat16*>(Wk));
  return cudaGetLastError();
}

cudaError_t launch_router_logits(int T, int h, int E, int dtype, const void* x, const float* Wg,
                                 float* partials, int* nsplit, cudaStream_t s) {
  *nsplit = 1;
  if (T == 0) return cudaSuccess;
  if (dtype == MOE_F32)
    return launch_logits_typed<float>(T, h, E, static_cast<const float*>(x), Wg, partials,
                                      kMaxSplits, nsplit, s);
  return launch_logits_typed<__nv_bfloat16>(T, h, E, static_cast<const __nv_bfloat16*>(x), Wg,
                                            partials, kMaxSplits, nsplit, s);
}

cudaError_t launch_router_topk(int T, int E, int k, int score, int num_groups, int group_topk,
                               const float* logits, int nsplit,
                               const float* gate_bias, const float* expert_bias,
                               int32_t* topk_idx, float* topk_prob,
                               uint8_t* keep, uint8_t* routing_map, int32_t* counts, int* err,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = kTopkWarps;
  int blocks = (T + warps_per_block - 1) / warps_per_block;
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  auto kern = E <= 32 ? router_topk_kernel<1> : E <= 64 ? router_topk_kernel<2>
             : E <= 128 ? router_topk_kernel<4> : router_topk_kernel<kMaxPerLane>;
  kern<<<blocks, 32 * warps_per_block, 0, s>>>(T, E, k, score, num_groups, group_topk, logits,
                                               nsplit, gate_bias, expert_bias, topk_idx, topk_prob,
                                               keep, routing_map, counts, err);
  return cudaGetLastError();
}

bool router_fused_ok(int h, int E, int k, int num_groups) {
  return E >= 1 && E <= kSmallE && k >= 1 && k <= E && num_groups <= 1 && h >= 1 &&
         h <= kFusedMaxHidden;
}

cudaError_t launch_router_fused(int T, int h, int E, int k, int dtype, int score, const void* x,
                                const float* Wg, const float* gate_bias,
                                const float* expert_bias, int32_t* topk_idx, float* topk_prob,
                                uint8_t* keep, uint8_t* routing_map, int32_t* counts, int* err,
                                cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (!router_fused_ok(h, E, k, 0)) return cudaErrorInvalidValue;
  const int smem = h * kSmallE * static_cast<int>(sizeof(float)) + kSmallE * 4;
  static bool configured[2][64] = {{false}};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  const int ti = dtype == MOE_F32 ? 0 : 1;
  if (dev < 64 && !configured[ti][dev]) {
    const int max_smem = kFusedMaxHidden * kSmallE * static_cast<int>(sizeof(float)) + kSmallE * 4;
    st = ti == 0 ? cudaFuncSetAttribute(router_fused_small_e_kernel<float>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)
                 : cudaFuncSetAttribute(router_fused_small_e_kernel<__nv_bfloat16>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (st != cudaSuccess) return st;
    configured[ti][dev] = true;
  }
  const int groups = (T + kSmallTok - 1) / kSmallTok;
  int grid = groups;  // one CTA per SM, as many SMs as there are 4-token groups
  if (grid > device_sm_count()) grid = device_sm_count();
  if (ti == 0)
    router_fused_small_e_kernel<float><<<grid, kFusedThreads, smem, s>>>(
        T, h, E, k, score, static_cast<const float*>(x), Wg, gate_bias, expert_bias, topk_idx,
        topk_prob, keep, routing_map, counts, err);
  else
    router_fused_small_e_kernel<__nv_bfloat16><<<grid, kFusedThreads, smem, s>>>(
        T, h, E, k, score, static_cast<const __nv_bfloat16*>(x), Wg, gate_bias, expert_bias,
        topk_idx, topk_prob, keep, routing_map, counts, err);
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
