// Local permutation (dispatch_preprocess) and combine of the MoE layer forward.
//
// Permutation, after the page "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
// (r00kie-liu.github.io) §9 (sequence-major -> expert-major) and step 4 of
// §8 "The All-to-All path" of "MoE Internals: DeepSpeed-Megatron Expert
// Parallel Implementation" (duoan.github.io).  Rows are expert-major and,
// inside an expert, in ascending token order (a stable counting sort of the
// T*k (token, slot) pairs keyed by expert):
//   perm_hist_kernel  per tile of 2048 pairs: kept-pair count per expert
//   perm_scan_kernel  one CTA: per-expert prefix over tiles, expert offsets
//   perm_rank_kernel  per tile: stable rank of each pair inside its tile
//                     (warp match_any + per-warp counts) -> row_map
//   perm_scan_rank_kernel  scan and rank in one launch for up to 128 tiles:
//                     each tile's CTA sums the per-tile counts itself (all
//                     tiles, and those before it), scans the totals into the
//                     expert offsets and ranks its tile
//   perm_copy_kernel  per token: read the x row once (16-byte vectors),
//                     write it to each of its kept rows
//   perm_copy_e4m3_kernel  the same for E4M3 rows: the token's row is
//                     quantised once (power-of-two scale) on the way
// Permutation by a [T,E] routing map (the padded map of pad_to_capacity, §8:
// the dispatcher permutes by the map, so an expert's rows are the tokens of
// its column in ascending order, padding tokens among them):
//   map_hist_kernel   per tile of 128 tokens: the map's ones per expert
//   map_scan_kernel   one CTA: first row of each (tile, expert), the offsets
//   map_rank_kernel   per tile: a thread per expert walks the tile's tokens
//                     in order -> row_src of each row, row_map of the kept
//                     pairs (-1 for the other slots)
//   perm_gather_kernel  per row: x_perm[r] = x[row_src[r]]
//   pad_fill_kernel   per (256-token chunk, expert): the lowest-index tokens
//                     not routed to the expert fill its column up to the quota
//
// Combine, after §2 (combine) of the Megatron Core page and step 8 of §8 of
// the DeepSpeed page (unpermute, weight by the router probabilities):
//   combine_kernel    per token: gather its k rows, fp32 weighted sum in
//                     slot order, plus the shared expert's row when there is
//                     one, one rounding to the output dtype
#include "common.cuh"
#include "e4m3.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(kPermThreads)
    perm_hist_kernel(int64_t npairs, int E, const int32_t* __restrict__ topk_idx,
                     const uint8_t* __restrict__ keep, int32_t* __restrict__ tile_counts,
                     int* __restrict__ err) {
  constexpr int kPer = kPermTile / kPermThreads;
  pdl_trigger();  // the scan+rank kernel may launch (it waits for these counts)
  __shared__ int hist[MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  // every load of this thread's pairs issued before the first atomic (one
  // round trip to memory, not one per pair)
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPermTile + threadIdx.x;
  int ev[kPer];
  uint8_t kv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int64_t p = base + u * kPermThreads;
    ev[u] = p < npairs ? topk_idx[p] : 0;
    kv[u] = p < npairs ? (keep ? keep[p] : 1) : 0;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (!kv[u]) continue;
    if (ev[u] >= 0 && ev[u] < E)
      atomicAdd(&hist[ev[u]], 1);
    else
      report_error(err, DEV_ERR_INDEX, static_cast<int>(base + u * kPermThreads));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    tile_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// tile_counts [ntiles][E]: counts in, first row of each (tile, expert) out.
__global__ void __launch_bounds__(1024)
    perm_scan_kernel(int64_t ntiles, int E, int32_t* __restrict__ tile_counts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ tokens_per_expert) {
  __shared__ int total[MOE_MAX_EXPERTS];
  __shared__ int start[MOE_MAX_EXPERTS + 1];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int64_t t = 0; t < ntiles; ++t) {
      const int c = tile_counts[t * E + e];
      tile_counts[t * E + e] = s;
      s += c;
    }
    total[e] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // exclusive scan of E <= 256 totals by one warp
    const int lane = threadIdx.x;
    int v[MOE_MAX_EXPERTS / 32];
    int run = 0;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) {
      const int e = lane * (MOE_MAX_EXPERTS / 32) + i;
      v[i] = (e < E) ? total[e] : 0;
      run += v[i];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int excl = incl - run;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) {
      const int e = lane * (MOE_MAX_EXPERTS / 32) + i;
      if (e <= E) start[e] = excl;
      excl += v[i];
    }
    if (lane == 31 && E == MOE_MAX_EXPERTS) start[E] = excl;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = start[e];
  if (tokens_per_expert)
    for (int e = threadIdx.x; e < E; e += blockDim.x) tokens_per_expert[e] = total[e];
  for (int64_t i = threadIdx.x; i < ntiles * E; i += blockDim.x)
    tile_counts[i] += start[i % E];
}

constexpr int kWarps = kPermThreads / 32;
constexpr int kChunks = kPermTile / kPermThreads;  // 32-pair chunks per warp

__global__ void __launch_bounds__(kPermThreads)
    perm_rank_kernel(int64_t npairs, int E, const int32_t* __restrict__ topk_idx,
                     const uint8_t* __restrict__ keep, const int32_t* __restrict__ tile_base,
                     int32_t* __restrict__ row_map, int32_t* __restrict__ row_src) {
  __shared__ int cnt[kWarps][MOE_MAX_EXPERTS];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * MOE_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
  __syncthreads();

  // warp w owns pairs [base + w*256, base + w*256 + 256), processed in
  // chunks of 32 consecutive pairs; the tile order is (warp, chunk, lane),
  // which is the pair order.
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPermTile + warp * (kChunks * 32);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int key[kChunks], rank[kChunks];
  // all of this lane's loads first (one round trip), then the ranking
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int64_t p = base + c * 32 + lane;
    int e = -1;
    if (p < npairs) {
      e = topk_idx[p];
      if (keep && !keep[p]) e = -1;
      if (e < 0 || e >= E) e = -1;  // flagged by perm_hist_kernel
    }
    key[c] = e;
  }
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int e = key[c];
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int before = 0;
    if (e >= 0) before = cnt[warp][e];
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp][e] = before + __popc(peers);
    __syncwarp();
    rank[c] = before + __popc(peers & lt_mask);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int v = cnt[w][e];
      cnt[w][e] = s;
      s += v;
    }
  }
  __syncthreads();
  const int32_t* tb = tile_base + static_cast<int64_t>(blockIdx.x) * E;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int64_t p = base + c * 32 + lane;
    if (p >= npairs) continue;
    const int e = key[c];
    if (e >= 0) {
      const int row = tb[e] + cnt[warp][e] + rank[c];
      row_map[p] = row;
      if (row_src) row_src[row] = static_cast<int32_t>(p);
    } else {
      row_map[p] = -1;
    }
  }
}

// Scan and rank in one launch (after perm_hist_kernel) when there are at
// most kFusedMaxTiles tiles: each tile's CTA sums the per-tile counts itself
// (all tiles for the totals, the earlier ones for its base), scans the
// totals into the expert offsets and ranks its tile; CTA 0 writes the
// offsets and tokens_per_expert.  The same order as perm_scan + perm_rank.
constexpr int64_t kFusedMaxTiles = 128;

__global__ void __launch_bounds__(kPermThreads)
    perm_scan_rank_kernel(int64_t npairs, int E, const int32_t* __restrict__ topk_idx,
                          const uint8_t* __restrict__ keep, const int32_t* tile_counts,
                          int32_t* __restrict__ row_map, int32_t* __restrict__ row_src,
                          int32_t* __restrict__ offsets, int32_t* __restrict__ tokens_per_expert) {
  __shared__ int before[MOE_MAX_EXPERTS], total[MOE_MAX_EXPERTS], start[MOE_MAX_EXPERTS + 1];
  __shared__ int cnt[kWarps][MOE_MAX_EXPERTS];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t ntiles = gridDim.x;  // one CTA per tile
  const int64_t tile = blockIdx.x;
  for (int i = threadIdx.x; i < kWarps * MOE_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
  // this tile's pairs: every load issued before the ranking
  const int64_t base = tile * kPermTile + warp * (kChunks * 32);
  int key[kChunks], rank[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int64_t p = base + c * 32 + lane;
    int e = -1;
    if (p < npairs) {
      e = topk_idx[p];
      if (keep && !keep[p]) e = -1;
      if (e < 0 || e >= E) e = -1;  // flagged by perm_hist_kernel
    }
    key[c] = e;
  }
  pdl_trigger();  // the copy may launch (it waits for row_map)
  pdl_wait();     // the per-tile counts of perm_hist_kernel
  // the totals and this tile's base, one expert per thread
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int all = 0, bef = 0;
#pragma unroll 8
    for (int64_t t = 0; t < ntiles; ++t) {
      const int c = __ldcg(tile_counts + t * E + e);  // written by perm_hist_kernel
      all += c;
      bef += t < tile ? c : 0;
    }
    total[e] = all;
    before[e] = bef;
  }
  __syncthreads();
  if (warp == 0) {  // expert offsets: exclusive scan of the totals (E <= 256)
    int v[MOE_MAX_EXPERTS / 32];
    int run = 0;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) {
      const int e = lane * (MOE_MAX_EXPERTS / 32) + i;
      v[i] = (e < E) ? total[e] : 0;
      run += v[i];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int excl = incl - run;
#pragma unroll
    for (int i = 0; i < MOE_MAX_EXPERTS / 32; ++i) {
      const int e = lane * (MOE_MAX_EXPERTS / 32) + i;
      if (e <= E) start[e] = excl;
      excl += v[i];
    }
    if (lane == 31 && E == MOE_MAX_EXPERTS) start[E] = excl;
  }
  // stable rank inside the tile, as perm_rank_kernel
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int e = key[c];
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int bef = 0;
    if (e >= 0) bef = cnt[warp][e];
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp][e] = bef + __popc(peers);
    __syncwarp();
    rank[c] = bef + __popc(peers & lt_mask);
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = start[e];
    if (tokens_per_expert)
      for (int e = threadIdx.x; e < E; e += blockDim.x) tokens_per_expert[e] = total[e];
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int sum = start[e] + before[e];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int v = cnt[w][e];
      cnt[w][e] = sum;
      sum += v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int64_t p = base + c * 32 + lane;
    if (p >= npairs) continue;
    const int e = key[c];
    if (e >= 0) {
      const int row = cnt[warp][e] + rank[c];
      row_map[p] = row;
      if (row_src) row_src[row] = static_cast<int32_t>(p);
    } else {
      row_map[p] = -1;
    }
  }
}

constexpr int kCopyThreads = 128;
constexpr int kCopyUnroll = 4;

// x_perm[row_map[t, j]] = x[t] for every kept slot j; 16-byte vectors.  A
// CTA moves 2^tpi_log2 tokens per round with kCopyThreads >> tpi_log2
// threads each, chosen so that short rows still give every thread
// kCopyUnroll loads in flight (one token per round for rows of >= 512
// vectors).
template <int TPI_LOG2>
__global__ void __launch_bounds__(kCopyThreads)
    perm_copy_kernel(int T, int row_vecs, int k, const uint4* __restrict__ x,
                     const int32_t* row_map, uint4* __restrict__ x_perm) {
  // row_map comes from the kernel before this one, which may still be running
  // until pdl_wait: it is read after the wait with coherent loads (no
  // read-only assumption a restrict qualifier would allow)
  constexpr int tpt = kCopyThreads >> TPI_LOG2;  // threads per token
  const int sub = threadIdx.x / tpt, lt = threadIdx.x % tpt;
  constexpr int64_t tpi = int64_t{1} << TPI_LOG2;
  bool waited = false;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * tpi; t0 < T; t0 += gridDim.x * tpi) {
    const int64_t t = t0 + sub;
    if (t >= T) continue;  // no barriers in this kernel
    const uint4* src = x + t * row_vecs;
    int rows[MOE_MAX_TOPK];
    for (int v0 = lt; v0 < row_vecs; v0 += tpt * kCopyUnroll) {
      uint4 buf[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int v = v0 + u * tpt;
        if (v < row_vecs) buf[u] = __ldcs(src + v);
      }
      if (v0 == lt) {  // the token's first vectors are in flight: now its rows
        if (!waited) {
          pdl_wait();  // row_map from the rank kernel
          waited = true;
        }
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) rows[j] = (j < k) ? __ldcg(row_map + t * k + j) : -1;
      }
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (rows[j] < 0) continue;
        uint4* dst = x_perm + (int64_t)rows[j] * row_vecs;
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const int v = v0 + u * tpt;
          if (v < row_vecs) dst[v] = buf[u];
        }
      }
    }
  }
}

// log2 of the tokens a CTA handles per round: the largest power of two
// (<= 2^max_log2) that does not exceed threads * per_thread / vecs_per_row.
int tokens_per_round_log2(int vecs_per_row, int threads, int per_thread, int max_log2) {
  int l = 0;
  while (l < max_log2 && (int64_t{2} << l) * vecs_per_row <= int64_t{threads} * per_thread) ++l;
  return l;
}

// E4M3 rows (FP8 experts): the token's bf16 row is reduced to its largest
// magnitude, converted once to E4M3 with the row's power-of-two scale, and
// the codes go to each kept row together with the scale.  h % 16 == 0.
__global__ void __launch_bounds__(kCopyThreads)
    perm_copy_e4m3_kernel(int T, int h, int k, const uint4* __restrict__ x,
                          const int32_t* __restrict__ row_map, uint8_t* __restrict__ x_perm_q,
                          float* __restrict__ row_scale) {
  __shared__ float red[kCopyThreads / 32];
  const int groups = h / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int rows[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) rows[j] = (j < k) ? row_map[(int64_t)t * k + j] : -1;
    const uint4* src = x + (int64_t)t * (h / 8);
    float m = 0.f;
    for (int g = threadIdx.x; g < groups; g += kCopyThreads)
      m = e4m3::amax_bf16x8(src[2 * g + 1], e4m3::amax_bf16x8(src[2 * g], m));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kCopyThreads / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();  // red is rewritten for the next token
    const int e = e4m3::scale_exp(m);
    const float inv = e4m3::pow2f(-e);
    if (threadIdx.x < k && rows[threadIdx.x] >= 0) row_scale[rows[threadIdx.x]] = e4m3::pow2f(e);
    for (int g = threadIdx.x; g < groups; g += kCopyThreads) {
      const uint4 c = e4m3::quantize16(src[2 * g], src[2 * g + 1], inv);
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j)
        if (rows[j] >= 0)
          *reinterpret_cast<uint4*>(x_perm_q + (int64_t)rows[j] * h + 16 * g) = c;
    }
  }
}

template <typename OT>
struct Out4;
template <>
struct Out4<float> {
  __device__ static void store(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }
};
template <>
struct Out4<__nv_bfloat16> {
  __device__ static void store(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    __stcs(reinterpret_cast<uint2*>(p), u);
  }
};

constexpr int kCombineThreads = 256;

// A CTA combines 2^TPI_LOG2 tokens per round, kCombineThreads >> TPI_LOG2
// threads each (several tokens per round when rows are short).  K1: top-1
// (one row per token), four vectors per thread in flight.
template <typename OT, int TPI_LOG2, bool K1, int U>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(int T, int h, int k, int64_t max_rows, const float* __restrict__ y_perm,
                   const int32_t* __restrict__ row_map, const float* __restrict__ topk_prob,
                   const float* __restrict__ y_shared, OT* __restrict__ y) {
  const int h4 = h >> 2;
  constexpr int tpt = kCombineThreads >> TPI_LOG2;  // threads per token
  const int sub = threadIdx.x / tpt, lt = threadIdx.x % tpt;
  constexpr int tpi = 1 << TPI_LOG2;
  for (int t0 = blockIdx.x * tpi; t0 < T; t0 += gridDim.x * tpi) {
    const int t = t0 + sub;
    if (t >= T) continue;  // no barriers in this kernel
    int rows[MOE_MAX_TOPK];
    float p[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      rows[j] = (j < k) ? row_map[(int64_t)t * k + j] : -1;
      if (rows[j] >= max_rows) rows[j] = -1;  // a row outside y_perm is treated as dropped
      // no weights (the backward's unpermute-sum of dx rows): weight 1
      p[j] = (rows[j] >= 0) ? (topk_prob ? topk_prob[(int64_t)t * k + j] : 1.f) : 0.f;
    }
    if constexpr (K1) {
      const int64_t r = rows[0];
      for (int v0 = lt; v0 < h4; v0 += 4 * tpt) {
        float4 a[4], b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * tpt;
          a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (v < h4 && r >= 0) a[u] = __ldcs(reinterpret_cast<const float4*>(y_perm + r * h) + v);
          if (v < h4 && y_shared)
            b[u] = __ldcs(reinterpret_cast<const float4*>(y_shared + (int64_t)t * h) + v);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * tpt;
          if (v >= h4) continue;
          // the same operations as below: fma with the weight, then the shared row
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r >= 0) {
            acc.x = fmaf(p[0], a[u].x, acc.x);
            acc.y = fmaf(p[0], a[u].y, acc.y);
            acc.z = fmaf(p[0], a[u].z, acc.z);
            acc.w = fmaf(p[0], a[u].w, acc.w);
          }
          if (y_shared) {
            acc.x += b[u].x;
            acc.y += b[u].y;
            acc.z += b[u].z;
            acc.w += b[u].w;
          }
          Out4<OT>::store(y + (int64_t)t * h + 4 * v, acc);
        }
      }
    } else {
      // U vectors of the row per thread at a time: each slot's U loads are
      // issued together (k x U in flight; U = 4 for k <= 2, where k loads
      // alone leave the HBM idle, 1 for more slots, where the registers of
      // more would cost occupancy), the fp32 sum still in slot order
      for (int v0 = lt; v0 < h4; v0 += U * tpt) {
        float4 acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) {
          if (rows[j] < 0) continue;
          const float4* src = reinterpret_cast<const float4*>(y_perm + (int64_t)rows[j] * h);
          float4 a[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = v0 + u * tpt;
            a[u] = v < h4 ? __ldcs(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            acc[u].x = fmaf(p[j], a[u].x, acc[u].x);
            acc[u].y = fmaf(p[j], a[u].y, acc[u].y);
            acc[u].z = fmaf(p[j], a[u].z, acc[u].z);
            acc[u].w = fmaf(p[j], a[u].w, acc[u].w);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * tpt;
          if (v >= h4) continue;
          if (y_shared) {  // the shared expert's output, added after the routed sum
            const float4 b = __ldcs(reinterpret_cast<const float4*>(y_shared + (int64_t)t * h) + v);
            acc[u].x += b.x;
            acc[u].y += b.y;
            acc[u].z += b.z;
            acc[u].w += b.w;
          }
          Out4<OT>::store(y + (int64_t)t * h + 4 * v, acc[u]);
        }
      }
    }
  }
}

// ------------------------------------------------ permutation by a routing map
constexpr int kMapTile = 128;  // tokens per tile

// The tile's rows of the routing map [t0, t1) x E into shared memory (16-byte
// copies when the map and E allow them); the caller synchronises.
__device__ __forceinline__ void stage_map_tile(const uint8_t* __restrict__ map, int64_t t0,
                                               int64_t t1, int E, uint8_t* tile) {
  const int64_t n = (t1 - t0) * E;
  const uint8_t* src = map + t0 * E;
  if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (n & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(tile);
    for (int64_t i = threadIdx.x; i < n / 16; i += blockDim.x) d4[i] = s4[i];
  } else {
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) tile[i] = src[i];
  }
}

// per tile: the map's ones of each expert (thread e counts column e)
__global__ void __launch_bounds__(kPermThreads)
    map_hist_kernel(int T, int E, const uint8_t* __restrict__ map,
                    int32_t* __restrict__ tile_counts) {
  __shared__ __align__(16) uint8_t tile[kMapTile * MOE_MAX_EXPERTS];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kMapTile;
  const int64_t t1 = min(static_cast<int64_t>(T), t0 + kMapTile);
  stage_map_tile(map, t0, t1, E, tile);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int64_t t = 0; t < t1 - t0; ++t) c += tile[t * E + e] != 0;
    tile_counts[static_cast<int64_t>(blockIdx.x) * E + e] = c;
  }
}

// tile_counts [ntiles][E]: counts in, first row of each (tile, expert) out;
// offsets [E+1] out.  The map has many short tiles, so each expert's tiles
// are split over G = 1024/E threads: chunk sums, an exclusive scan of the
// chunks per expert and of the expert totals, then each thread rewrites its
// chunk from its base (loads of a batch issued before its stores).
constexpr int kMapScanThreads = 1024;
constexpr int kMapScanBatch = 16;
__global__ void __launch_bounds__(kMapScanThreads)
    map_scan_kernel(int64_t ntiles, int E, int32_t* __restrict__ tile_counts,
                    int32_t* __restrict__ offsets) {
  __shared__ int part[kMapScanThreads];
  __shared__ int start[MOE_MAX_EXPERTS + 1];
  const int G = kMapScanThreads / E;
  const int e = threadIdx.x % E, g = threadIdx.x / E;
  const int64_t per = (ntiles + G - 1) / G;
  const int64_t a = min(ntiles, static_cast<int64_t>(g) * per), b = min(ntiles, a + per);
  const bool active = g < G;
  int sum = 0;
  if (active)
    for (int64_t t = a; t < b; ++t) sum += tile_counts[t * E + e];
  if (active) part[g * E + e] = sum;
  __syncthreads();
  if (threadIdx.x < E) {  // exclusive prefix of expert e's chunk sums
    int run = 0;
    for (int q = 0; q < G; ++q) {
      const int v = part[q * E + threadIdx.x];
      part[q * E + threadIdx.x] = run;
      run += v;
    }
    start[threadIdx.x] = run;  // the total, scanned below
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // exclusive scan of E <= 256 totals
    int run = 0;
    for (int x = 0; x < E; ++x) {
      const int v = start[x];
      start[x] = run;
      run += v;
    }
    start[E] = run;
  }
  __syncthreads();
  for (int x = threadIdx.x; x <= E; x += blockDim.x) offsets[x] = start[x];
  if (!active) return;
  int base = start[e] + part[g * E + e];
  for (int64_t t = a; t < b; t += kMapScanBatch) {
    int c[kMapScanBatch];
#pragma unroll
    for (int u = 0; u < kMapScanBatch; ++u) c[u] = (t + u < b) ? tile_counts[(t + u) * E + e] : 0;
#pragma unroll
    for (int u = 0; u < kMapScanBatch; ++u)
      if (t + u < b) {
        tile_counts[(t + u) * E + e] = base;
        base += c[u];
      }
  }
}

// Per tile: the map, topk_idx and keep of its tokens in shared memory.  Each
// expert column is split over Q = blockDim/E threads (Q token ranges): every
// thread counts its range, adds the counts of the ranges before it to the
// tile's first row of the expert and walks its range in token order.  Rows
// past max_rows (a map with more ones than the permuted buffers hold) are
// reported and not written.
__global__ void __launch_bounds__(kPermThreads)
    map_rank_kernel(int T, int E, int k, int64_t max_rows, const uint8_t* __restrict__ map,
                    const int32_t* __restrict__ topk_idx, const uint8_t* __restrict__ keep,
                    const int32_t* __restrict__ tile_base, int32_t* __restrict__ row_map,
                    int32_t* __restrict__ row_src, int* __restrict__ err) {
  __shared__ __align__(16) uint8_t tile[kMapTile * MOE_MAX_EXPERTS];
  __shared__ int32_t sidx[kMapTile * MOE_MAX_TOPK];
  __shared__ uint8_t skeep[kMapTile * MOE_MAX_TOPK];
  __shared__ int cnt[kPermThreads];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kMapTile;
  const int64_t t1 = min(static_cast<int64_t>(T), t0 + kMapTile);
  stage_map_tile(map, t0, t1, E, tile);
  const int64_t np = (t1 - t0) * k;
  for (int64_t i = threadIdx.x; i < np; i += blockDim.x) {
    sidx[i] = topk_idx[t0 * k + i];
    skeep[i] = keep ? keep[t0 * k + i] : 1;
    row_map[t0 * k + i] = -1;  // the kept pairs are overwritten below
  }
  __syncthreads();
  const int Q = blockDim.x / E;  // >= 1 (E <= 256)
  const int e = threadIdx.x % E, q = threadIdx.x / E;
  const int n = static_cast<int>(t1 - t0);
  const int len = (n + Q - 1) / Q;
  const int u0 = min(n, q * len), u1 = min(n, u0 + len);
  int c = 0;
  if (q < Q)
    for (int u = u0; u < u1; ++u) c += tile[u * E + e] != 0;
  cnt[threadIdx.x] = c;
  __syncthreads();
  if (q >= Q) return;
  int64_t row = tile_base[static_cast<int64_t>(blockIdx.x) * E + e];
  for (int qq = 0; qq < q; ++qq) row += cnt[qq * E + e];
  for (int u = u0; u < u1; ++u) {
    if (!tile[u * E + e]) continue;
    if (row >= max_rows) {
      report_error(err, DEV_ERR_INDEX, static_cast<int>(t0 + u));
      return;
    }
    row_src[row] = static_cast<int32_t>(t0 + u);
    for (int j = 0; j < k; ++j)  // a token routes to an expert through one slot at most
      if (sidx[u * k + j] == e && skeep[u * k + j])
        row_map[(t0 + u) * k + j] = static_cast<int32_t>(row);
    ++row;
  }
}

// One warp per row (grid-stride): rows [0, min(offsets[E], max_rows)).
__global__ void __launch_bounds__(kCopyThreads)
    perm_gather_kernel(int64_t max_rows, int row_vecs, const int32_t* __restrict__ total_rows,
                       const int32_t* __restrict__ row_src, const uint4* __restrict__ x,
                       uint4* __restrict__ x_perm) {
  const int64_t R = min(static_cast<int64_t>(*total_rows), max_rows);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < R;
       r += nwarps) {
    const uint4* src = x + static_cast<int64_t>(row_src[r]) * row_vecs;
    uint4* dst = x_perm + r * row_vecs;
    for (int v = lane; v < row_vecs; v += 32) dst[v] = src[v];
  }
}

constexpr int kPadChunk = 256;

// First index i in [0, m) with cand_pair[begin + i] / k >= bound, by one warp:
// each round the 32 lanes test 32 evenly spaced pivots, shrinking the range
// 32-fold (a handful of dependent loads instead of log2(m)).
__device__ __forceinline__ int warp_lower_bound(const int32_t* __restrict__ cand_pair, int begin,
                                                int m, int k, int bound, int lane) {
  int lo = 0, hi = m;  // the answer lies in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int pos = lo + lane * step;
    const bool below = pos < hi && cand_pair[begin + pos] / k < bound;
    const int c = __popc(__ballot_sync(0xffffffffu, below));  // pivots below: lanes 0 .. c-1
    const int nlo = c == 0 ? lo : lo + (c - 1) * step + 1;
    hi = min(hi, lo + c * step);
    lo = nlo;
  }
  const int pos = lo + lane;
  const bool below = pos < hi && cand_pair[begin + pos] / k < bound;
  return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// dst[r] = src[row_src[r]] for rows [0, min(offsets[E], max_rows)): the
// E4M3 rows' scales after a permutation by the map
__global__ void __launch_bounds__(256)
    perm_gather_scale_kernel(int64_t max_rows, const int32_t* __restrict__ total_rows,
                             const int32_t* __restrict__ row_src, const float* __restrict__ src,
                             float* __restrict__ dst) {
  const int64_t R = min(static_cast<int64_t>(*total_rows), max_rows);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < R;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[r] = src[row_src[r]];
}

// Expert blockIdx.y's column of the routing map, tokens [t0, t0 + 256): an
// expert under capacity kept all of its m routed pairs (the candidate pairs
// cand_pair[cand_off[e] ..], ascending), so it needs quota - m padding
// tokens, the lowest-index tokens not routed to it.  A token's rank among
// the free tokens is (t0 - the routed tokens below t0) plus the free tokens
// before it in the chunk (a block scan).  Without candidate lists (capacity
// >= T: nothing dropped) every token is taken.  tokens_per_expert becomes the
// quota (the column sums of the padded map).
__global__ void __launch_bounds__(kPadChunk)
    pad_fill_kernel(int T, int E, int k, int quota, const int32_t* __restrict__ cand_off,
                    const int32_t* __restrict__ cand_pair, int32_t* __restrict__ tokens_per_expert,
                    uint8_t* __restrict__ map) {
  __shared__ int s_lo, s_hi;
  __shared__ uint8_t routed[kPadChunk];
  __shared__ int warp_free[kPadChunk / 32];
  const int e = blockIdx.y;
  const int t0 = blockIdx.x * kPadChunk;
  const int begin = cand_off ? cand_off[e] : 0;
  const int m = cand_off ? cand_off[e + 1] - begin : 0;
  const int need = quota - m;  // <= 0: at or over capacity, nothing to add
  if (blockIdx.x == 0 && threadIdx.x == 0) tokens_per_expert[e] = quota;
  if (need <= 0) return;
  routed[threadIdx.x] = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < 2) {  // routed tokens below t0 (warp 0) and below t0 + 256 (warp 1)
    const int v = warp_lower_bound(cand_pair, begin, m, k, t0 + warp * kPadChunk, lane);
    if (lane == 0) {
      if (warp) s_hi = v; else s_lo = v;
    }
  }
  __syncthreads();
  for (int i = s_lo + threadIdx.x; i < s_hi; i += blockDim.x)
    routed[cand_pair[begin + i] / k - t0] = 1;
  __syncthreads();
  const int t = t0 + threadIdx.x;
  const bool free_tok = t < T && !routed[threadIdx.x];
  const unsigned ballot = __ballot_sync(0xffffffffu, free_tok);
  if (lane == 0) warp_free[warp] = __popc(ballot);
  __syncthreads();
  int before = __popc(ballot & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) before += warp_free[w];
  if (free_tok && (t0 - s_lo) + before < need) map[static_cast<int64_t>(t) * E + e] = 1;
}

template <typename OT, bool K1, int U>
void launch_combine_t(int l, int grid, cudaStream_t s, int T, int h, int k, int64_t max_rows,
                      const float* y_perm, const int32_t* row_map, const float* topk_prob,
                      const float* y_shared, OT* y) {
  switch (l) {
    case 0: combine_kernel<OT, 0, K1, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, y_perm, row_map, topk_prob, y_shared, y); break;
    case 1: combine_kernel<OT, 1, K1, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, y_perm, row_map, topk_prob, y_shared, y); break;
    case 2: combine_kernel<OT, 2, K1, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, y_perm, row_map, topk_prob, y_shared, y); break;
    default: combine_kernel<OT, 3, K1, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, y_perm, row_map, topk_prob, y_shared, y); break;
  }
}

int grid_for_tokens(int T, int per_sm) {
  const int cap = device_sm_count() * per_sm;
  return T < cap ? T : cap;
}

}  // namespace

cudaError_t launch_perm_hist(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                             int32_t* tile_counts, int* err, cudaStream_t s) {
  const int64_t nt = perm_tiles(npairs);
  if (nt == 0) return cudaSuccess;
  perm_hist_kernel<<<static_cast<unsigned>(nt), kPermThreads, 0, s>>>(npairs, E, topk_idx, keep,
                                                                       tile_counts, err);
  return cudaGetLastError();
}

cudaError_t launch_perm_scan(int64_t ntiles, int E, int32_t* tile_counts, int32_t* offsets,
                             int32_t* tokens_per_expert, cudaStream_t s) {
  perm_scan_kernel<<<1, 1024, 0, s>>>(ntiles, E, tile_counts, offsets, tokens_per_expert);
  return cudaGetLastError();
}

cudaError_t launch_perm_rank(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                             const int32_t* tile_base, int32_t* row_map, int32_t* row_src,
                             cudaStream_t s) {
  const int64_t nt = perm_tiles(npairs);
  if (nt == 0) return cudaSuccess;
  perm_rank_kernel<<<static_cast<unsigned>(nt), kPermThreads, 0, s>>>(npairs, E, topk_idx, keep,
                                                                       tile_base, row_map, row_src);
  return cudaGetLastError();
}

cudaError_t launch_perm_index(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                              int32_t* tile_counts, int32_t* row_map, int32_t* row_src,
                              int32_t* offsets, int32_t* tokens_per_expert, int* err,
                              cudaStream_t s) {
  const int64_t nt = perm_tiles(npairs);
  cudaError_t st = launch_perm_hist(npairs, E, topk_idx, keep, tile_counts, err, s);
  if (st != cudaSuccess) return st;
  if (nt == 0 || nt > kFusedMaxTiles) {
    st = launch_perm_scan(nt, E, tile_counts, offsets, tokens_per_expert, s);
    if (st == cudaSuccess)
      st = launch_perm_rank(npairs, E, topk_idx, keep, tile_counts, row_map, row_src, s);
    return st;
  }
  return launch_dependent(perm_scan_rank_kernel, dim3(static_cast<unsigned>(nt)),
                          dim3(kPermThreads), 0, s, npairs, E, topk_idx, keep,
                          static_cast<const int32_t*>(tile_counts), row_map, row_src, offsets,
                          tokens_per_expert);
}

cudaError_t launch_perm_copy(int T, int h, int k, int dtype, const void* x, const int32_t* row_map,
                             void* x_perm, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int row_vecs = h * (dtype == MOE_F32 ? 4 : 2) / 16;
  const int l = tokens_per_round_log2(row_vecs, kCopyThreads, kCopyUnroll, 5);
  const int grid = grid_for_tokens((T + (1 << l) - 1) >> l, 16);
  const uint4* src = static_cast<const uint4*>(x);
  uint4* dst = static_cast<uint4*>(x_perm);
  // launched as a dependent of the rank kernel: the x loads start early
  void (*kern)(int, int, int, const uint4*, const int32_t*, uint4*) =
      l == 0 ? perm_copy_kernel<0> : l == 1 ? perm_copy_kernel<1> : l == 2 ? perm_copy_kernel<2>
      : l == 3 ? perm_copy_kernel<3> : l == 4 ? perm_copy_kernel<4> : perm_copy_kernel<5>;
  return launch_dependent(kern, dim3(grid), dim3(kCopyThreads), 0, s, T, row_vecs, k, src,
                          row_map, dst);
}

int64_t map_tiles(int T) { return (static_cast<int64_t>(T) + kMapTile - 1) / kMapTile; }

cudaError_t launch_perm_by_map(int T, int row_bytes, int E, int k, int64_t max_rows,
                               const void* x, const uint8_t* map, const int32_t* topk_idx,
                               const uint8_t* keep, int32_t* tile_counts, int32_t* row_src,
                               void* x_perm, int32_t* row_map, int32_t* offsets, int* err,
                               cudaStream_t s) {
  const int64_t nt = map_tiles(T);
  if (nt > 0) {
    map_hist_kernel<<<static_cast<unsigned>(nt), kPermThreads, 0, s>>>(T, E, map, tile_counts);
    cudaError_t st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  map_scan_kernel<<<1, kMapScanThreads, 0, s>>>(nt, E, tile_counts, offsets);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess || nt == 0) return st;
  map_rank_kernel<<<static_cast<unsigned>(nt), kPermThreads, 0, s>>>(
      T, E, k, max_rows, map, topk_idx, keep, tile_counts, row_map, row_src, err);
  st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  const int row_vecs = row_bytes / 16;
  perm_gather_kernel<<<device_sm_count() * 8, kCopyThreads, 0, s>>>(
      max_rows, row_vecs, offsets + E, row_src, static_cast<const uint4*>(x),
      static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_gather_scales(int64_t max_rows, const int32_t* total_rows,
                                 const int32_t* row_src, const float* src, float* dst,
                                 cudaStream_t s) {
  int64_t grid = (max_rows + 255) / 256;
  if (grid > 8LL * device_sm_count()) grid = 8LL * device_sm_count();
  if (grid < 1) return cudaSuccess;
  perm_gather_scale_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(max_rows, total_rows,
                                                                        row_src, src, dst);
  return cudaGetLastError();
}

cudaError_t launch_pad_fill(int T, int E, int k, int quota, const int32_t* cand_off,
                            const int32_t* cand_pair, int32_t* tokens_per_expert, uint8_t* map,
                            cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((T + kPadChunk - 1) / kPadChunk > 0
                                            ? (T + kPadChunk - 1) / kPadChunk : 1),
                  static_cast<unsigned>(E));
  pad_fill_kernel<<<grid, kPadChunk, 0, s>>>(T, E, k, quota, cand_off, cand_pair,
                                             tokens_per_expert, map);
  return cudaGetLastError();
}

cudaError_t launch_perm_copy_e4m3(int T, int h, int k, const void* x, const int32_t* row_map,
                                  uint8_t* x_perm_q, float* row_scale, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  perm_copy_e4m3_kernel<<<grid_for_tokens(T, 16), kCopyThreads, 0, s>>>(
      T, h, k, static_cast<const uint4*>(x), row_map, x_perm_q, row_scale);
  return cudaGetLastError();
}

// Combine over a y_perm stored as fp16 with one power-of-two scale per 32
// columns (value = fp16 * 2^exp, exact in fp32): per token the kept slots'
// values in slot order, fp32 FMA with the weights, one rounding to bf16 --
// the combine kernel's arithmetic on the decoded values.  A thread takes 8
// columns (16 bytes of fp16 and the chunk's exponent byte) of U vectors at a
// time; the loads of every slot (at most KMAX) are issued before the sum, so
// KMAX * U * 16 bytes per thread are in flight.
template <int TPI_LOG2, int KMAX, int U>
__global__ void __launch_bounds__(kCombineThreads)
    combine_f16s_kernel(int T, int h, int k, int64_t max_rows, const uint4* __restrict__ y16,
                        const int8_t* __restrict__ y16_exp, const int32_t* __restrict__ row_map,
                        const float* __restrict__ topk_prob, const float4* __restrict__ y_shared,
                        uint4* __restrict__ y) {
  const int h8 = h >> 3;    // 16-byte vectors per row
  const int nch = h >> 5;   // exponent bytes per row
  constexpr int tpt = kCombineThreads >> TPI_LOG2;
  const int sub = threadIdx.x / tpt, lt = threadIdx.x % tpt;
  constexpr int tpi = 1 << TPI_LOG2;
  for (int t0 = blockIdx.x * tpi; t0 < T; t0 += gridDim.x * tpi) {
    const int t = t0 + sub;
    if (t >= T) continue;  // no barriers in this kernel
    int rows[KMAX];
    float p[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = (j < k) ? row_map[(int64_t)t * k + j] : -1;
      if (rows[j] >= max_rows) rows[j] = -1;  // a row outside y_perm is treated as dropped
      p[j] = (rows[j] >= 0) ? topk_prob[(int64_t)t * k + j] : 0.f;
    }
    for (int v0 = lt; v0 < h8; v0 += U * tpt) {
      uint4 a[KMAX][U];
      int ex[KMAX][U];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * tpt;
          const bool ld = rows[j] >= 0 && v < h8;
          a[j][u] = ld ? __ldcs(y16 + (int64_t)rows[j] * h8 + v) : make_uint4(0u, 0u, 0u, 0u);
          ex[j][u] = ld ? y16_exp[(int64_t)rows[j] * nch + (v >> 2)] : 0;
        }
      // one vector at a time: its slots in order, then its store (8 sums live)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * tpt;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (rows[j] < 0) continue;
          const float up = __uint_as_float(static_cast<uint32_t>(127 + ex[j][u]) << 23);  // 2^e
          const uint32_t w4[4] = {a[j][u].x, a[j][u].y, a[j][u].z, a[j][u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
            acc[2 * q] = fmaf(p[j], f.x * up, acc[2 * q]);
            acc[2 * q + 1] = fmaf(p[j], f.y * up, acc[2 * q + 1]);
          }
        }
        if (v >= h8) continue;
        if (y_shared) {  // the shared expert's output, added after the routed sum
          const float4 s0 = __ldcs(y_shared + ((int64_t)t * h8 + v) * 2);
          const float4 s1 = __ldcs(y_shared + ((int64_t)t * h8 + v) * 2 + 1);
          acc[0] += s0.x;
          acc[1] += s0.y;
          acc[2] += s0.z;
          acc[3] += s0.w;
          acc[4] += s1.x;
          acc[5] += s1.y;
          acc[6] += s1.z;
          acc[7] += s1.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
          o[q] = *reinterpret_cast<uint32_t*>(&b);
        }
        __stcs(y + (int64_t)t * h8 + v, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

template <int KMAX, int U>
void launch_combine_f16s_t(int l, int grid, cudaStream_t s, int T, int h, int k, int64_t max_rows,
                           const uint4* src, const int8_t* ex, const int32_t* row_map,
                           const float* topk_prob, const float4* ys, uint4* dst) {
  switch (l) {
    case 0: combine_f16s_kernel<0, KMAX, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, src, ex, row_map, topk_prob, ys, dst); break;
    case 1: combine_f16s_kernel<1, KMAX, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, src, ex, row_map, topk_prob, ys, dst); break;
    case 2: combine_f16s_kernel<2, KMAX, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, src, ex, row_map, topk_prob, ys, dst); break;
    default: combine_f16s_kernel<3, KMAX, U><<<grid, kCombineThreads, 0, s>>>(T, h, k, max_rows, src, ex, row_map, topk_prob, ys, dst); break;
  }
}

cudaError_t launch_combine_f16s(int T, int h, int k, const void* y16, const int8_t* y16_exp,
                                const int32_t* row_map, const float* topk_prob,
                                const float* y_shared, void* y, cudaStream_t s,
                                int64_t max_rows) {
  if (T == 0) return cudaSuccess;
  const uint4* src = static_cast<const uint4*>(y16);
  const float4* ys = reinterpret_cast<const float4*>(y_shared);
  uint4* dst = static_cast<uint4*>(y);
  // 128 bytes of loads per thread in flight: 2 slots x 4 vectors, 4 x 2 or 8 x 1
  const int U = k <= 2 ? 4 : k <= 4 ? 2 : 1;
  const int l = tokens_per_round_log2(h / 8, kCombineThreads, U, 3);
  const int grid = grid_for_tokens((T + (1 << l) - 1) >> l, 8);
  if (k <= 2)
    launch_combine_f16s_t<2, 4>(l, grid, s, T, h, k, max_rows, src, y16_exp, row_map, topk_prob, ys,
                                dst);
  else if (k <= 4)
    launch_combine_f16s_t<4, 2>(l, grid, s, T, h, k, max_rows, src, y16_exp, row_map, topk_prob, ys,
                                dst);
  else
    launch_combine_f16s_t<MOE_MAX_TOPK, 1>(l, grid, s, T, h, k, max_rows, src, y16_exp, row_map,
                                           topk_prob, ys, dst);
  return cudaGetLastError();
}

// Top-1 layers whose combine runs in fc2's epilogue: each row's token and
// combine weight (row_map inverted: a top-1 token owns at most one row), and
// zeros for the output rows of tokens whose pair was dropped -- what the
// combine kernel writes for them.  A warp per token, grid-stride.
__global__ void __launch_bounds__(256)
    top1_rows_kernel(int T, int row_vecs, int64_t max_rows, const int32_t* __restrict__ row_map,
                     const float* __restrict__ topk_prob, int32_t* __restrict__ row_token,
                     float* __restrict__ row_weight, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    const int r = row_map[t];
    if (r >= 0 && r < max_rows) {
      if (lane == 0) {
        row_token[r] = t;
        row_weight[r] = topk_prob[t];
      }
    } else {
      uint4* dst = y + static_cast<int64_t>(t) * row_vecs;
      for (int v = lane; v < row_vecs; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

cudaError_t launch_top1_rows(int T, int h, int dtype, int64_t max_rows, const int32_t* row_map,
                             const float* topk_prob, int32_t* row_token, float* row_weight,
                             void* y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int row_vecs = h * (dtype == MOE_F32 ? 4 : 2) / 16;
  top1_rows_kernel<<<grid_for_tokens((T + 7) / 8, 8), 256, 0, s>>>(
      T, row_vecs, max_rows, row_map, topk_prob, row_token, row_weight, static_cast<uint4*>(y));
  return cudaGetLastError();
}

cudaError_t launch_combine(int T, int h, int k, int dtype, const float* y_perm,
                           const int32_t* row_map, const float* topk_prob, const float* y_shared,
                           void* y, cudaStream_t s, int64_t max_rows) {
  if (T == 0) return cudaSuccess;
  if (max_rows < 0) max_rows = static_cast<int64_t>(T) * k;
  const int l = tokens_per_round_log2(h / 4, kCombineThreads, 4, 3);
  const int grid = grid_for_tokens((T + (1 << l) - 1) >> l, 8);
  if (dtype == MOE_F32) {
    float* o = static_cast<float*>(y);
    if (k == 1)
      launch_combine_t<float, true, 1>(l, grid, s, T, h, k, max_rows, y_perm, row_map, topk_prob,
                                       y_shared, o);
    else if (k == 2)
      launch_combine_t<float, false, 4>(l, grid, s, T, h, k, max_rows, y_perm, row_map,
                                        topk_prob, y_shared, o);
    else
      launch_combine_t<float, false, 1>(l, grid, s, T, h, k, max_rows, y_perm, row_map,
                                        topk_prob, y_shared, o);
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(y);
    if (k == 1)
      launch_combine_t<__nv_bfloat16, true, 1>(l, grid, s, T, h, k, max_rows, y_perm, row_map,
                                               topk_prob, y_shared, o);
    else if (k == 2)
      launch_combine_t<__nv_bfloat16, false, 4>(l, grid, s, T, h, k, max_rows, y_perm, row_map,
                                                topk_prob, y_shared, o);
    else
      launch_combine_t<__nv_bfloat16, false, 1>(l, grid, s, T, h, k, max_rows, y_perm, row_map,
                                                topk_prob, y_shared, o);
  }
  return cudaGetLastError();
}

}  // namespace moe
