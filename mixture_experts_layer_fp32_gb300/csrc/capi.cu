// C ABI of the MoE layer forward: argument validation, workspace carve-up and
// the launch sequence of each stage.  No device memory is allocated here;
// nothing synchronises the host except moe_check().
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace moe {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev >= 64) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }
  if (cache[dev] == 0) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace moe

namespace {

using namespace moe;

thread_local char g_last_cuda_error[256] = "";

struct Layout {
  size_t err, logits, assigned, tiles, cand_rowmap, cand_src, cand_off, cand_tiles;
  size_t topk_idx, topk_prob, keep, tpe, offsets, row_map, x_perm, h_mid, y_perm;
  size_t map, map_tiles, row_src, top1_token, top1_weight, router_wk, total;
};

size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int64_t capacity_of(const moe_config& c) {
  if (c.capacity_factor <= 0.f) return -1;
  const double v = ceil((static_cast<double>(c.num_tokens) * c.topk / c.num_experts) *
                        static_cast<double>(c.capacity_factor));
  int64_t cap = static_cast<int64_t>(v);
  if (cap < c.min_capacity) cap = c.min_capacity;
  return cap;
}

// Rows of the permuted buffers: T*k, or with pad_to_capacity E * min(cap, T)
// when that is more (every expert padded to its capacity).
int64_t rows_of(const moe_config& c) {
  const int64_t np = static_cast<int64_t>(c.num_tokens) * c.topk;
  if (!c.pad_to_capacity) return np;
  int64_t q = capacity_of(c);
  if (q < 0 || q > c.num_tokens) q = c.num_tokens;
  const int64_t padded = q * c.num_experts;
  return padded > np ? padded : np;
}

// bf16 layers whose router GEMM can run on the tensor cores (over the gate
// weights split into three bf16 pieces): every expert count past the fused
// small-E kernel's, E % 4 == 0.
bool router_tc_capable(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.num_experts % 4 == 0 && c.hidden % 64 == 0 &&
         !router_fused_ok(c.hidden, c.num_experts, c.topk, c.num_groups);
}
// The layer's router runs on the CUDA cores (fp32 FMA) unless
// MOE_ROUTER_TC=1 is set in the environment: an opt-in outside the layer's
// specification, which keeps the tensor cores to the expert GEMMs.
bool router_on_tc(const moe_config& c) {
  const char* opt = getenv("MOE_ROUTER_TC");
  return router_tc_capable(c) && opt && opt[0] == '1';
}

// Router logits into `partials` (*nsplit partial sums [nsplit, T, E] that the
// top-k and the router backward add in order); wk: 3 E h bf16 of scratch for
// the split gate weights when router_tc_capable.
cudaError_t router_logits(const moe_config& c, const void* x, const float* Wg, void* wk,
                          float* partials, int* nsplit, int* err, cudaStream_t s) {
  if (!router_on_tc(c))
    return launch_router_logits(c.num_tokens, c.hidden, c.num_experts, c.dtype, x, Wg, partials,
                                nsplit, s);
  cudaError_t st = launch_router_split3(c.hidden, c.num_experts, Wg, wk, s);
  if (st != cudaSuccess) return st;
  return launch_tc_router_logits(c.num_tokens, c.hidden, c.num_experts, x, wk, partials, nsplit,
                                 err, s);
}

Layout make_layout(const moe_config& c) {
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = align_up(o + bytes);
    return r;
  };
  const size_t T = c.num_tokens, k = c.topk, E = c.num_experts, h = c.hidden, f = c.ffn_hidden;
  const size_t np = T * k;
  const size_t nt = static_cast<size_t>(perm_tiles(static_cast<int64_t>(np)));
  const size_t el = c.dtype == MOE_F32 ? 4 : 2;
  L.err = take(kErrBytes);
  L.logits = take(T * E * 4 * kRouterMaxSplits);
  L.assigned = take(E * 4);
  L.tiles = take(nt * E * 4);
  L.cand_rowmap = take(np * 4);
  L.cand_src = take(np * 4);
  L.cand_off = take((E + 1) * 4);
  L.cand_tiles = take(nt * E * 4);
  L.topk_idx = take(np * 4);
  L.topk_prob = take(np * 4);
  L.keep = take(np);
  L.tpe = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.row_map = take(np * 4);
  const size_t rows = static_cast<size_t>(rows_of(c));
  L.x_perm = take(rows * h * el);
  L.h_mid = take(rows * f * el);
  L.y_perm = take(rows * h * 4);
  // the permutation by a routing map (moe_permute_map, and the padded forward)
  L.map = take(c.pad_to_capacity ? T * E : 0);
  L.map_tiles = take(static_cast<size_t>(map_tiles(static_cast<int>(T))) * E * 4);
  L.row_src = take(rows * 4);
  // top-1 layers whose combine runs in fc2's epilogue: each row's token and weight
  L.top1_token = take(k == 1 ? rows * 4 : 0);
  L.top1_weight = take(k == 1 ? rows * 4 : 0);
  L.router_wk = take(router_tc_capable(c) ? 3 * E * h * 2 : 0);
  L.total = o;
  return L;
}

moe_status validate(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->num_tokens < 0 || c->hidden <= 0 || c->num_experts <= 0 || c->topk <= 0 ||
      c->ffn_hidden <= 0 || c->min_capacity < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->score < MOE_SCORE_SOFTMAX_POST || c->score > MOE_SCORE_SQRTSOFTPLUS)
    return MOE_ERR_INVALID_ARG;
  if (c->num_groups < 0 || c->group_topk < 0) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->drop_policy != MOE_DROP_PROBS && c->drop_policy != MOE_DROP_POSITION)
    return MOE_ERR_INVALID_ARG;
  if (isnan(c->capacity_factor) || isinf(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (c->pad_to_capacity != 0 && c->pad_to_capacity != 1) return MOE_ERR_INVALID_ARG;
  if (c->pad_to_capacity && c->capacity_factor <= 0.f) return MOE_ERR_INVALID_ARG;
  if (c->num_experts > MOE_MAX_EXPERTS || c->topk > MOE_MAX_TOPK || c->topk > c->num_experts)
    return MOE_ERR_UNSUPPORTED;
  if (c->hidden % 8 != 0 || c->ffn_hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16 && (c->hidden % 256 != 0 || c->ffn_hidden % 128 != 0))
    return MOE_ERR_UNSUPPORTED;
  if (c->num_groups > 1) {
    const int G = c->num_groups;
    if (G > 32 || c->num_experts % G != 0 || c->group_topk < 1 || c->group_topk > G ||
        c->group_topk > c->topk || c->topk > c->group_topk * (c->num_experts / G))
      return MOE_ERR_UNSUPPORTED;
  }
  const int64_t np = static_cast<int64_t>(c->num_tokens) * c->topk;
  if (np > (int64_t{1} << 30) || rows_of(*c) > (int64_t{1} << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// A device tensor argument: nullptr allowed only when it has no elements.
moe_status need(const void* p, size_t nelem, size_t align) {
  if (nelem == 0) return MOE_OK;
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(p) % align != 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
moe_status optional(const void* p, size_t align) {
  if (p != nullptr && reinterpret_cast<uintptr_t>(p) % align != 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

#define MOE_TRY(expr)                          \
  do {                                         \
    const moe_status st_ = (expr);             \
    if (st_ != MOE_OK) return st_;             \
  } while (0)

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s", cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

moe_status check_ws(const moe_config& c, const void* ws, size_t ws_bytes, size_t need_bytes = 0) {
  if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < (need_bytes ? need_bytes : make_layout(c).total)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// The shared expert's width: positive, and a multiple of the GEMM's column
// granularity (8 for the fp32 path, 128 for the tensor-core path).
moe_status validate_fs(const moe_config& c, int32_t fs) {
  if (fs <= 0) return MOE_ERR_INVALID_ARG;
  if (fs % 8 != 0 || (c.dtype == MOE_BF16 && fs % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// moe_forward_shared's workspace: the routed layout, then h_mid_s [T,fs]
// (dtype) and y_shared [T,h] fp32.
struct SharedLayout {
  size_t h_mid_s, y_shared, total;
};
SharedLayout make_shared_layout(const moe_config& c, int32_t fs) {
  SharedLayout S;
  const size_t T = c.num_tokens, el = c.dtype == MOE_F32 ? 4 : 2;
  S.h_mid_s = make_layout(c).total;
  S.y_shared = align_up(S.h_mid_s + T * static_cast<size_t>(fs) * el);
  S.total = align_up(S.y_shared + T * static_cast<size_t>(c.hidden) * 4);
  return S;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}


// ---- stage bodies (arguments already validated) ----

moe_status do_route(const moe_config& c, const void* x, const float* Wg, const float* gb,
                    const float* eb, int32_t* topk_idx, float* topk_prob, uint8_t* keep,
                    int32_t* tpe, uint8_t* routing_map, void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  const int T = c.num_tokens, E = c.num_experts, k = c.topk;
  int* err = at<int>(ws, L.err);
  const int64_t cap = capacity_of(c);
  const bool drops = cap >= 0 && cap < T;
  MOE_CUDA(cudaMemsetAsync(tpe, 0, E * sizeof(int32_t), s));
  if (T == 0) return MOE_OK;
  // logits then top-k, or both in one kernel for E <= 8; the per-expert
  // counts go to tokens_per_expert, or (with drops) to the assigned counts
  auto route_topk = [&](int32_t* counts) -> cudaError_t {
    if (router_fused_ok(c.hidden, E, k, c.num_groups))
      return launch_router_fused(T, c.hidden, E, k, c.dtype, c.score, x, Wg, gb, eb, topk_idx,
                                 topk_prob, keep, routing_map, counts, err, s);
    float* logits = at<float>(ws, L.logits);
    int nsplit = 1;
    cudaError_t st = router_logits(c, x, Wg, at<void>(ws, L.router_wk), logits, &nsplit, err, s);
    if (st != cudaSuccess) return st;
    return launch_router_topk(T, E, k, c.score, c.num_groups, c.group_topk, logits, nsplit, gb,
                              eb, topk_idx, topk_prob, keep, routing_map, counts, err, s);
  };
  if (!drops) {
    MOE_CUDA(route_topk(tpe));
    if (c.pad_to_capacity)  // capacity >= T: every token to every expert
      MOE_CUDA(launch_pad_fill(T, E, k, T, nullptr, nullptr, tpe, routing_map, s));
    return MOE_OK;
  }
  int32_t* assigned = at<int32_t>(ws, L.assigned);
  MOE_CUDA(cudaMemsetAsync(assigned, 0, E * sizeof(int32_t), s));
  MOE_CUDA(route_topk(assigned));
  // candidate lists: every routed pair, expert-major, ascending token order
  const int64_t np = static_cast<int64_t>(T) * k;
  int32_t* ctiles = at<int32_t>(ws, L.cand_tiles);
  int32_t* coff = at<int32_t>(ws, L.cand_off);
  MOE_CUDA(launch_perm_index(np, E, topk_idx, nullptr, ctiles, at<int32_t>(ws, L.cand_rowmap),
                             at<int32_t>(ws, L.cand_src), coff, nullptr, err, s));
  MOE_CUDA(launch_drop_select(T, E, k, cap, c.drop_policy, coff, at<int32_t>(ws, L.cand_src),
                              topk_prob, keep, routing_map, tpe, s));
  if (c.pad_to_capacity)  // fill the experts under capacity with the lowest free tokens
    MOE_CUDA(launch_pad_fill(T, E, k, static_cast<int>(cap), coff, at<int32_t>(ws, L.cand_src),
                             tpe, routing_map, s));
  return MOE_OK;
}

// Permutation by a [T,E] routing map: an expert's rows are the tokens of its
// column in ascending order; row_map holds the rows of the kept pairs.
moe_status do_permute_map(const moe_config& c, const void* x, const uint8_t* map,
                          const int32_t* topk_idx, const uint8_t* keep, void* x_perm,
                          int32_t* row_map, int32_t* offsets, void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  const int row_bytes = c.hidden * (c.dtype == MOE_F32 ? 4 : 2);
  MOE_CUDA(launch_perm_by_map(c.num_tokens, row_bytes, c.num_experts, c.topk, rows_of(c),
                              x, map, topk_idx, keep, at<int32_t>(ws, L.map_tiles),
                              at<int32_t>(ws, L.row_src), x_perm, row_map, offsets,
                              at<int>(ws, L.err), s));
  return MOE_OK;
}

moe_status do_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                      const uint8_t* keep, void* x_perm, int32_t* row_map, int32_t* offsets,
                      void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  const int T = c.num_tokens, E = c.num_experts, k = c.topk;
  int* err = at<int>(ws, L.err);
  const int64_t np = static_cast<int64_t>(T) * k;
  if (np == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s));
    return MOE_OK;
  }
  int32_t* tiles = at<int32_t>(ws, L.tiles);
  MOE_CUDA(launch_perm_index(np, E, topk_idx, keep, tiles, row_map, nullptr, offsets, nullptr,
                             err, s));
  MOE_CUDA(launch_perm_copy(T, c.hidden, k, c.dtype, x, row_map, x_perm, s));
  return MOE_OK;
}

moe_status do_fc1(const moe_config& c, const void* x_perm, const int32_t* offsets, const void* W1,
                  const void* W3, void* h_mid, void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  int* err = at<int>(ws, L.err);
  const int64_t rows = rows_of(c);
  if (c.dtype == MOE_F32)
    MOE_CUDA(launch_simt_fc1(c.num_experts, c.hidden, c.ffn_hidden, rows,
                             static_cast<const float*>(x_perm), offsets,
                             static_cast<const float*>(W1), static_cast<const float*>(W3),
                             static_cast<float*>(h_mid), err, s));
  else
    MOE_CUDA(launch_tc_fc1(c.num_experts, c.hidden, c.ffn_hidden, rows, x_perm, offsets, W1, W3,
                           h_mid, err, s));
  return MOE_OK;
}

moe_status do_fc2(const moe_config& c, const void* h_mid, const int32_t* offsets, const void* W2,
                  float* y_perm, void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  int* err = at<int>(ws, L.err);
  const int64_t rows = rows_of(c);
  if (c.dtype == MOE_F32)
    MOE_CUDA(launch_simt_fc2(c.num_experts, c.hidden, c.ffn_hidden, rows,
                             static_cast<const float*>(h_mid), offsets,
                             static_cast<const float*>(W2), y_perm, err, s));
  else
    MOE_CUDA(launch_tc_fc2(c.num_experts, c.hidden, c.ffn_hidden, rows, h_mid, offsets, W2, y_perm,
                           err, s));
  return MOE_OK;
}

// fc2 and the combine in one call (layers without pad_to_capacity).  bf16
// top-1: the combine runs in fc2's epilogue (each row, weighted, straight into
// its token's output row; the bits of fc2 + combine).  bf16 top-k (k >= 2):
// fc2 writes y_perm as fp16 with one power-of-two scale per 32 columns into
// the workspace and the combine reads that.  fp32: fc2 into the workspace's
// y_perm, then the combine kernel.
bool fc2_combine_ok(const moe_config& c) { return !c.pad_to_capacity; }
bool fc2_combine_fused(const moe_config& c) {
  return c.topk == 1 && !c.pad_to_capacity && c.dtype == MOE_BF16;
}
bool fc2_combine_f16s(const moe_config& c) {
  return c.topk > 1 && !c.pad_to_capacity && c.dtype == MOE_BF16;
}
// The fp16 y_perm inside the workspace's y_perm region: [R, h] fp16, then
// [R, h/32] exponent bytes (2 + 1/32 bytes per value, within the region's 4).
void* ws_y16(void* ws, const Layout& L) { return at<void>(ws, L.y_perm); }
int8_t* ws_y16_exp(const moe_config& c, void* ws, const Layout& L) {
  const size_t bytes16 = static_cast<size_t>(rows_of(c)) * c.hidden * 2;
  return at<int8_t>(ws, L.y_perm + align_up(bytes16));
}

moe_status do_fc2_combine(const moe_config& c, const void* h_mid, const int32_t* offsets,
                          const void* W2, const int32_t* row_map, const float* topk_prob, void* y,
                          void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  int* err = at<int>(ws, L.err);
  const int64_t rows = rows_of(c);
  if (fc2_combine_f16s(c)) {
    void* y16 = ws_y16(ws, L);
    int8_t* y16e = ws_y16_exp(c, ws, L);
    MOE_CUDA(launch_tc_fc2_f16s(c.num_experts, c.hidden, c.ffn_hidden, rows, h_mid, offsets, W2,
                                y16, y16e, err, s));
    MOE_CUDA(launch_combine_f16s(c.num_tokens, c.hidden, c.topk, y16, y16e, row_map, topk_prob,
                                 nullptr, y, s, rows));
    return MOE_OK;
  }
  if (!fc2_combine_fused(c)) {
    float* y_perm = at<float>(ws, L.y_perm);
    MOE_TRY(do_fc2(c, h_mid, offsets, W2, y_perm, ws, s));
    MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype, y_perm, row_map, topk_prob,
                            nullptr, y, s, rows));
    return MOE_OK;
  }
  int32_t* tok = at<int32_t>(ws, L.top1_token);
  float* wgt = at<float>(ws, L.top1_weight);
  MOE_CUDA(launch_top1_rows(c.num_tokens, c.hidden, c.dtype, rows, row_map, topk_prob, tok, wgt,
                            y, s));
  MOE_CUDA(launch_tc_fc2_top1(c.num_experts, c.hidden, c.ffn_hidden, rows, h_mid, offsets, W2,
                              tok, wgt, y, err, s));
  return MOE_OK;
}

// Shared expert: the grouped MLP kernels as one dense group of all T rows of x.
moe_status do_shared(const moe_config& c, int32_t fs, const void* x, const void* W1s,
                     const void* W3s, const void* W2s, void* h_mid_s, float* y_shared, int* err,
                     cudaStream_t s) {
  const int64_t T = c.num_tokens;
  if (c.dtype == MOE_F32) {
    MOE_CUDA(launch_simt_fc1(1, c.hidden, fs, T, static_cast<const float*>(x), nullptr,
                             static_cast<const float*>(W1s), static_cast<const float*>(W3s),
                             static_cast<float*>(h_mid_s), err, s));
    MOE_CUDA(launch_simt_fc2(1, c.hidden, fs, T, static_cast<const float*>(h_mid_s), nullptr,
                             static_cast<const float*>(W2s), y_shared, err, s));
  } else {
    MOE_CUDA(launch_tc_fc1(1, c.hidden, fs, T, x, nullptr, W1s, W3s, h_mid_s, err, s));
    MOE_CUDA(launch_tc_fc2(1, c.hidden, fs, T, h_mid_s, nullptr, W2s, y_shared, err, s));
  }
  return MOE_OK;
}

// Buffers of the routed path inside the workspace (or the caller's).
struct Routed {
  int32_t* idx;
  float* prob;
  int32_t* tpe;
  int32_t* row_map;
  float* y_perm;
};

// route -> drop -> permute -> fc1 -> fc2 of moe_forward, on `stream`.
moe_status routed_path(const moe_config& c, const void* x, const float* Wg,
                       const float* gate_bias, const float* expert_bias, const void* W1,
                       const void* W3, const void* W2, int32_t* topk_idx, float* topk_prob,
                       int32_t* tokens_per_expert, void* ws, cudaStream_t stream, Routed* out,
                       bool skip_fc2 = false) {
  const Layout L = make_layout(c);
  int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.topk_idx);
  float* prob = topk_prob ? topk_prob : at<float>(ws, L.topk_prob);
  int32_t* tpe = tokens_per_expert ? tokens_per_expert : at<int32_t>(ws, L.tpe);
  uint8_t* keep = at<uint8_t>(ws, L.keep);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_map = at<int32_t>(ws, L.row_map);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h_mid = at<void>(ws, L.h_mid);
  float* y_perm = at<float>(ws, L.y_perm);
  // pad_to_capacity: the padded routing map (workspace) drives the permutation
  uint8_t* map = c.pad_to_capacity ? at<uint8_t>(ws, L.map) : nullptr;
  MOE_TRY(do_route(c, x, Wg, gate_bias, expert_bias, idx, prob, keep, tpe, map, ws, stream));
  if (map)
    MOE_TRY(do_permute_map(c, x, map, idx, keep, x_perm, row_map, offsets, ws, stream));
  else
    MOE_TRY(do_permute(c, x, idx, keep, x_perm, row_map, offsets, ws, stream));
  MOE_TRY(do_fc1(c, x_perm, offsets, W1, W3, h_mid, ws, stream));
  if (!skip_fc2) MOE_TRY(do_fc2(c, h_mid, offsets, W2, y_perm, ws, stream));
  *out = Routed{idx, prob, tpe, row_map, y_perm};
  return MOE_OK;
}

// The library's second stream per device (for the shared expert) and the
// fork / join events; created on first use, kept until exit.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

moe_status side_stream(SideStream** out) {
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  SideStream& ss = g_side[dev];
  if (ss.stream == nullptr) {
    MOE_CUDA(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming));
    MOE_CUDA(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming));
    MOE_CUDA(cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking));
  }
  *out = &ss;
  return MOE_OK;
}

// FP8 (E4M3) workspace: the routed layout (its h_mid holds the bf16 SwiGLU
// output), then the permuted codes [T*k,h] and their row scales [T*k], the
// SwiGLU codes [T*k,f] and scales.
struct E4m3Layout {
  size_t xperm_q, xperm_s, hq, hs, xq_tok, xs_tok, total;
};
E4m3Layout make_e4m3_layout(const moe_config& c) {
  E4m3Layout Q;
  const size_t T = c.num_tokens, np = static_cast<size_t>(rows_of(c)), h = c.hidden,
               f = c.ffn_hidden;
  size_t o = make_layout(c).total;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = align_up(o + bytes);
    return r;
  };
  Q.xperm_q = take(np * h);
  Q.xperm_s = take(np * 4);
  Q.hq = take(np * f);
  Q.hs = take(np * 4);
  // pad_to_capacity: x quantised once per token, then gathered by the map
  Q.xq_tok = take(c.pad_to_capacity ? T * h : 0);
  Q.xs_tok = take(c.pad_to_capacity ? T * 4 : 0);
  Q.total = o;
  return Q;
}

moe_status validate_e4m3(const moe_config& c) {
  return c.dtype == MOE_BF16 ? MOE_OK : MOE_ERR_UNSUPPORTED;  // bf16 in/out, E4M3 experts
}

// E4M3 permute: quantise x per token, rank the pairs, copy code rows and scales.
moe_status do_permute_e4m3(const moe_config& c, const void* x, const int32_t* topk_idx,
                           const uint8_t* keep, uint8_t* xperm_q, float* xperm_s,
                           int32_t* row_map, int32_t* offsets, void* ws, cudaStream_t s) {
  const Layout L = make_layout(c);
  const int T = c.num_tokens, E = c.num_experts, k = c.topk;
  int* err = at<int>(ws, L.err);
  const int64_t np = static_cast<int64_t>(T) * k;
  if (np == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s));
    return MOE_OK;
  }
  int32_t* tiles = at<int32_t>(ws, L.tiles);
  MOE_CUDA(launch_perm_index(np, E, topk_idx, keep, tiles, row_map, nullptr, offsets, nullptr,
                             err, s));
  MOE_CUDA(launch_perm_copy_e4m3(T, c.hidden, k, x, row_map, xperm_q, xperm_s, s));
  return MOE_OK;
}

// E4M3 permutation by a routing map (pad_to_capacity): every token's row
// quantised once, the code rows gathered by the map, their scales after them.
moe_status do_permute_map_e4m3(const moe_config& c, const void* x, const uint8_t* map,
                               const int32_t* topk_idx, const uint8_t* keep, uint8_t* xperm_q,
                               float* xperm_s, int32_t* row_map, int32_t* offsets, void* ws,
                               cudaStream_t s) {
  const Layout L = make_layout(c);
  const E4m3Layout Q = make_e4m3_layout(c);
  uint8_t* xq_tok = at<uint8_t>(ws, Q.xq_tok);
  float* xs_tok = at<float>(ws, Q.xs_tok);
  int32_t* row_src = at<int32_t>(ws, L.row_src);
  const int64_t rows = rows_of(c);
  MOE_CUDA(launch_quantize_rows(c.num_tokens, c.hidden, x, xq_tok, xs_tok, nullptr, s));
  MOE_CUDA(launch_perm_by_map(c.num_tokens, c.hidden, c.num_experts, c.topk, rows, xq_tok, map,
                              topk_idx, keep, at<int32_t>(ws, L.map_tiles), row_src, xperm_q,
                              row_map, offsets, at<int>(ws, L.err), s));
  MOE_CUDA(launch_gather_scales(rows, offsets + c.num_experts, row_src, xs_tok, xperm_s, s));
  return MOE_OK;
}

// E4M3 experts: fc1 (scaled, SwiGLU, bf16 h_mid), per-row quantisation of the
// rows that exist (expert_offsets[E] on the device), fc2 (scaled) into the
// fp32 y_perm, or, with y16, into the fp16 y_perm with a scale per 32 columns.
moe_status do_mlp_e4m3(const moe_config& c, const uint8_t* xperm_q, const float* xperm_s,
                       const int32_t* offsets, const uint8_t* W1q, const float* s1,
                       const uint8_t* W3q, const float* s3, const uint8_t* W2q, const float* s2,
                       void* h_mid, uint8_t* hq, float* hs, float* y_perm, void* ws,
                       cudaStream_t s, void* y16 = nullptr, int8_t* y16_exp = nullptr) {
  const Layout L = make_layout(c);
  int* err = at<int>(ws, L.err);
  const int64_t rows = rows_of(c);
  const int E = c.num_experts, h = c.hidden, f = c.ffn_hidden;
  MOE_CUDA(launch_tc_fc1_e4m3(E, h, f, rows, xperm_q, xperm_s, nullptr, offsets, W1q, s1, W3q,
                              s3, h_mid, err, s));
  MOE_CUDA(launch_quantize_rows(rows, f, h_mid, hq, hs, offsets + E, s));
  if (y16)
    MOE_CUDA(launch_tc_fc2_e4m3_f16s(E, h, f, rows, hq, hs, offsets, W2q, s2, y16, y16_exp, err,
                                     s));
  else
    MOE_CUDA(launch_tc_fc2_e4m3(E, h, f, rows, hq, hs, offsets, W2q, s2, y_perm, err, s));
  return MOE_OK;
}

// Backward workspace: error word, router partial logits [S,T,E], dp [T,k],
// dlogits [T,E], dWg partial sums, dx_router [T,h] fp32, dY_perm [T*k,h] bf16, dH [T*k,f] bf16,
// dA = [da | dg] [T*k,2f] bf16, dx_perm [T*k,h] fp32.
// moe_backward's workspace; with a shared expert of width fs (> 0), its dH_s
// [T,fs] and dA_s [T,2fs] (bf16) follow.
// The router's gradients on the tensor cores (hi/lo bf16 splits) for bf16
// layers with E % 64 == 0; otherwise (and for fp32) on the FMA units.
bool bwd_router_on_tc(const moe_config& c) {
  return c.dtype == MOE_BF16 && router_grads_on_tc(c.num_experts);
}

// The backward's expert GEMMs for the configuration's dtype: the tcgen05
// kernels for bf16, the SIMT kernels for fp32 (offsets NULL: one dense group).
cudaError_t bwd_dgrad_fc2(const moe_config& c, int E, int f, int64_t rows, const void* dY,
                          const int32_t* off, const void* W2, void* dH, int* err, cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_simt_dgrad_fc2(E, c.hidden, f, rows, static_cast<const float*>(dY), off,
                                 static_cast<const float*>(W2), static_cast<float*>(dH), err, s);
  return launch_tc_dgrad_fc2(E, c.hidden, f, rows, dY, off, W2, dH, err, s);
}
cudaError_t bwd_fc1_recompute(const moe_config& c, int E, int f, int64_t rows, const void* x,
                              const int32_t* off, const void* W1, const void* W3, const void* dH,
                              void* dA, int* err, cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_simt_fc1_bwd(E, c.hidden, f, rows, static_cast<const float*>(x), off,
                               static_cast<const float*>(W1), static_cast<const float*>(W3),
                               static_cast<const float*>(dH), static_cast<float*>(dA), err, s);
  return launch_tc_fc1_bwd(E, c.hidden, f, rows, x, off, W1, W3, dH, dA, err, s);
}
cudaError_t bwd_dgrad_fc1(const moe_config& c, int E, int f, int64_t rows, const void* dA,
                          const int32_t* off, const void* W1, const void* W3, float* dx, int* err,
                          cudaStream_t s, bool accumulate = false) {
  if (c.dtype == MOE_F32)
    return launch_simt_dgrad_fc1(E, c.hidden, f, rows, static_cast<const float*>(dA), off,
                                 static_cast<const float*>(W1), static_cast<const float*>(W3), dx,
                                 err, s, accumulate);
  return launch_tc_dgrad_fc1(E, c.hidden, f, rows, dA, off, W1, W3, dx, err, s, accumulate);
}
// dW [E, M, N] fp32 = A_e^T . B_e; lda / ldb in elements, B may start at a
// column offset (dA's dg half)
cudaError_t bwd_wgrad(const moe_config& c, int E, int M, int N, int64_t rows, const void* A,
                      int lda, const void* B, int ldb, const int32_t* off, float* dW, int* err,
                      cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_simt_wgrad(E, M, N, rows, static_cast<const float*>(A), lda,
                             static_cast<const float*>(B), ldb, off, dW, err, s);
  return launch_tc_wgrad(E, M, N, rows, A, lda, B, ldb, off, dW, err, s);
}
// element `i` of an activation buffer of the configuration's dtype
const void* act_at(const moe_config& c, const void* p, size_t i) {
  return static_cast<const char*>(p) + i * (c.dtype == MOE_F32 ? 4 : 2);
}

struct BwdLayout {
  size_t err, logits, dp, dl, dwg_part, dl3, wg3, dwg2, router_wk, dx_router, dY_perm, dH, dA, dx_perm;
  size_t dH_s, dA_s, total;
};
BwdLayout make_bwd_layout(const moe_config& c, int32_t fs = 0) {
  BwdLayout B;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = align_up(o + bytes);
    return r;
  };
  const size_t T = c.num_tokens, E = c.num_experts, h = c.hidden, f = c.ffn_hidden;
  const size_t R = static_cast<size_t>(rows_of(c));  // padded rows with pad_to_capacity
  const size_t el = c.dtype == MOE_F32 ? 4 : 2;  // the activation gradients' element
  B.err = take(kErrBytes);
  B.logits = take(T * E * 4 * kRouterMaxSplits);
  B.dp = take(T * c.topk * 4);
  B.dl = take(T * E * 4);
  const bool tc = bwd_router_on_tc(c);
  B.dwg_part = take(tc ? 0 : static_cast<size_t>(dwg_splits(c.num_tokens, c.hidden, c.num_experts)) * h * E * 4);
  B.dl3 = take(tc ? T * 3 * E * 2 : 0);
  B.wg3 = take(tc ? h * 3 * E * 2 : 0);
  B.dwg2 = take(tc ? h * 2 * E * 4 : 0);
  B.router_wk = take(router_tc_capable(c) ? 3 * E * h * 2 : 0);
  B.dx_router = take(T * h * 4);
  B.dY_perm = take(R * h * el);
  B.dH = take(R * f * el);
  B.dA = take(R * 2 * f * el);
  B.dx_perm = take(R * h * 4);
  const size_t F = fs > 0 ? static_cast<size_t>(fs) : 0;
  B.dH_s = take(T * F * el);
  B.dA_s = take(T * 2 * F * el);
  B.total = o;
  return B;
}

// The library's host-I/O streams per device for moe_forward_host: one for
// host->device copies, one for device->host copies, and the events that
// order them against the compute stream (per staging slot: input ready,
// input free, output ready, output free; plus the entry fork and the two
// final joins).  Created on first use, kept until exit.
struct CopyStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t x_ready[2] = {}, x_free[2] = {}, y_ready[2] = {}, y_free[2] = {};
  cudaEvent_t fork = nullptr, h2d_done = nullptr, d2h_done = nullptr;
};
std::mutex g_copy_mu;
CopyStreams g_copy[64];

moe_status copy_streams(CopyStreams** out) {
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  CopyStreams& cs = g_copy[dev];
  if (cs.h2d == nullptr) {
    cudaEvent_t* evs[] = {&cs.x_ready[0], &cs.x_ready[1], &cs.x_free[0], &cs.x_free[1],
                          &cs.y_ready[0], &cs.y_ready[1], &cs.y_free[0], &cs.y_free[1],
                          &cs.fork,       &cs.h2d_done,   &cs.d2h_done};
    for (cudaEvent_t* e : evs) MOE_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    MOE_CUDA(cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking));
    MOE_CUDA(cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking));
  }
  *out = &cs;
  return MOE_OK;
}

// moe_forward_host's workspace: the routed layout, then two input staging
// buffers [T,h] (dtype) and two output staging buffers [T,h] (dtype).
struct HostLayout {
  size_t x_stage[2], y_stage[2], total;
};
// Staging for the host-I/O forward: two input and two output slots of [T,h]
// after the forward's own workspace (`base` bytes: the routed, shared or
// E4M3 layout).
HostLayout make_host_layout(const moe_config& c, size_t base) {
  HostLayout H;
  const size_t row = static_cast<size_t>(c.num_tokens) * c.hidden * (c.dtype == MOE_F32 ? 4 : 2);
  size_t o = base;
  for (int i = 0; i < 2; ++i) {
    H.x_stage[i] = o;
    o = align_up(o + row);
  }
  for (int i = 0; i < 2; ++i) {
    H.y_stage[i] = o;
    o = align_up(o + row);
  }
  H.total = o;
  return H;
}

// The shared expert's backward (dense, over all T tokens, weight 1): the
// dgrad chain with its dx added to dx_acc (fp32 [T,h]), then its weight
// gradients.  The first half runs before the routed token-gradient combine,
// the second after it (see do_backward).
struct SharedBwd {
  int32_t fs;
  const void *W1s, *W3s, *W2s, *h_mid_s;
  float *dW1s, *dW3s, *dW2s;
};
moe_status shared_bwd_dgrad(const moe_config& c, const SharedBwd& sh, const void* x,
                            const void* dy, float* dx_acc, void* dH_s, void* dA_s, int* err,
                            cudaStream_t s) {
  const int T = c.num_tokens, fs = sh.fs;
  MOE_CUDA(bwd_dgrad_fc2(c, 1, fs, T, dy, nullptr, sh.W2s, dH_s, err, s));
  MOE_CUDA(bwd_fc1_recompute(c, 1, fs, T, x, nullptr, sh.W1s, sh.W3s, dH_s, dA_s, err, s));
  MOE_CUDA(bwd_dgrad_fc1(c, 1, fs, T, dA_s, nullptr, sh.W1s, sh.W3s, dx_acc, err, s,
                         /*accumulate=*/true));
  return MOE_OK;
}
moe_status shared_bwd_wgrad(const moe_config& c, const SharedBwd& sh, const void* x,
                            const void* dy, const void* dA_s, int* err, cudaStream_t s) {
  const int T = c.num_tokens, h = c.hidden, fs = sh.fs;
  MOE_CUDA(bwd_wgrad(c, 1, fs, h, T, sh.h_mid_s, fs, dy, h, nullptr, sh.dW2s, err, s));
  MOE_CUDA(bwd_wgrad(c, 1, h, fs, T, x, h, dA_s, 2 * fs, nullptr, sh.dW1s, err, s));
  MOE_CUDA(bwd_wgrad(c, 1, h, fs, T, x, h, act_at(c, dA_s, fs), 2 * fs, nullptr, sh.dW3s, err,
                     s));
  return MOE_OK;
}

moe_status check_shared_bwd(const moe_config& c, const SharedBwd& sh) {
  MOE_TRY(validate_fs(c, sh.fs));
  const size_t T = c.num_tokens, h = c.hidden, fs = sh.fs;
  MOE_TRY(need(sh.W1s, h * fs, 16));
  MOE_TRY(need(sh.W3s, h * fs, 16));
  MOE_TRY(need(sh.W2s, h * fs, 16));
  MOE_TRY(need(sh.h_mid_s, T * fs, 16));
  MOE_TRY(need(sh.dW1s, h * fs, 16));
  MOE_TRY(need(sh.dW3s, h * fs, 16));
  MOE_TRY(need(sh.dW2s, h * fs, 16));
  return MOE_OK;
}

moe_status do_backward(const moe_config* cfg, const void* x, const float* Wg,
                       const float* gate_bias, const void* W1, const void* W3, const void* W2,
                       const int32_t* topk_idx, const float* topk_prob, const int32_t* row_map,
                       const int32_t* expert_offsets, const void* x_perm, const void* h_mid,
                       const float* y_perm, const void* dy, void* dx, float* dWg,
                       float* dgate_bias, float* dW1, float* dW3, float* dW2,
                       const SharedBwd* sh, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (sh) MOE_TRY(check_shared_bwd(c, *sh));
  const size_t T = c.num_tokens, E = c.num_experts, k = c.topk, h = c.hidden, f = c.ffn_hidden;
  const size_t R = static_cast<size_t>(rows_of(c)), wsz = E * h * f;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(need(x_perm, R * h, 16));
  MOE_TRY(need(h_mid, R * f, 16));
  MOE_TRY(need(y_perm, R * h, 16));
  MOE_TRY(need(dy, T * h, 16));
  MOE_TRY(need(dx, T * h, 16));
  MOE_TRY(need(dWg, h * E, 4));
  MOE_TRY(optional(dgate_bias, 4));
  MOE_TRY(need(dW1, wsz, 16));
  MOE_TRY(need(dW3, wsz, 16));
  MOE_TRY(need(dW2, wsz, 16));
  const BwdLayout B = make_bwd_layout(c, sh ? sh->fs : 0);
  MOE_TRY(check_ws(c, ws, ws_bytes, B.total));
  int* err = at<int>(ws, B.err);
  const int Ti = c.num_tokens, Ei = c.num_experts, ki = c.topk, hi = c.hidden, fi = c.ffn_hidden;
  const int64_t rows = static_cast<int64_t>(R);
  float* logits = at<float>(ws, B.logits);
  float* dp = at<float>(ws, B.dp);
  float* dl = at<float>(ws, B.dl);
  float* dx_router = at<float>(ws, B.dx_router);
  void* dY_perm = at<void>(ws, B.dY_perm);
  void* dH = at<void>(ws, B.dH);
  void* dA = at<void>(ws, B.dA);
  float* dx_perm = at<float>(ws, B.dx_perm);
  // pad_to_capacity: the padding rows have no slot, so the combine backward
  // writes no dY row for them; zeros make every gradient they reach zero
  if (c.pad_to_capacity)
    MOE_CUDA(cudaMemsetAsync(dY_perm, 0, R * h * (c.dtype == MOE_F32 ? 4 : 2), stream));
  // router: logits again (the forward does not keep them), then its gradients
  int nsplit = 1;
  MOE_CUDA(router_logits(c, x, Wg, at<void>(ws, B.router_wk), logits, &nsplit, err, stream));
  MOE_CUDA(launch_combine_bwd(Ti, hi, ki, c.dtype, dy, row_map, topk_prob, y_perm, dY_perm, dp,
                              stream));
  MOE_CUDA(launch_router_bwd(Ti, Ei, ki, c.score, logits, nsplit, gate_bias, topk_idx, dp, dl,
                             stream));
  if (bwd_router_on_tc(c)) {
    MOE_CUDA(launch_router_grads_tc(Ti, hi, Ei, x, dl, Wg, at<void>(ws, B.dl3), at<void>(ws, B.wg3),
                                    at<float>(ws, B.dwg2), dWg, dgate_bias, dx_router, err,
                                    stream));
  } else {
    MOE_CUDA(launch_router_param_grads(Ti, hi, Ei, c.dtype, x, dl, dWg, at<float>(ws, B.dwg_part),
                                       dgate_bias, stream));
    MOE_CUDA(launch_dx_router(Ti, hi, Ei, dl, Wg, dx_router, stream));
  }
  // experts: dgrad chain, then the token gradient, then the weight gradients
  MOE_CUDA(bwd_dgrad_fc2(c, Ei, fi, rows, dY_perm, expert_offsets, W2, dH, err, stream));
  MOE_CUDA(bwd_fc1_recompute(c, Ei, fi, rows, x_perm, expert_offsets, W1, W3, dH, dA, err,
                             stream));
  MOE_CUDA(bwd_dgrad_fc1(c, Ei, fi, rows, dA, expert_offsets, W1, W3, dx_perm, err, stream));
  if (sh)  // the shared expert's dx joins dx_router before the one rounding
    MOE_TRY(shared_bwd_dgrad(c, *sh, x, dy, dx_router, at<void>(ws, B.dH_s), at<void>(ws, B.dA_s),
                             err, stream));
  MOE_CUDA(launch_combine(Ti, hi, ki, c.dtype, dx_perm, row_map, nullptr, dx_router, dx, stream,
                          rows));
  MOE_CUDA(bwd_wgrad(c, Ei, fi, hi, rows, h_mid, fi, dY_perm, hi, expert_offsets, dW2, err,
                     stream));
  MOE_CUDA(bwd_wgrad(c, Ei, hi, fi, rows, x_perm, hi, dA, 2 * fi, expert_offsets, dW1, err,
                     stream));
  MOE_CUDA(bwd_wgrad(c, Ei, hi, fi, rows, x_perm, hi, act_at(c, dA, fi), 2 * fi, expert_offsets,
                     dW3, err, stream));
  if (sh) MOE_TRY(shared_bwd_wgrad(c, *sh, x, dy, at<void>(ws, B.dA_s), err, stream));
  return MOE_OK;
}

// moe_forward_shared after its argument checks (also one batch of
// moe_forward_host_shared): the shared expert forked onto the side stream,
// the routed path on `stream`, joined before the combine.
moe_status shared_forward_body(const moe_config& c, int32_t fs, const void* x, const float* Wg,
                               const float* gate_bias, const float* expert_bias, const void* W1,
                               const void* W3, const void* W2, const void* W1s, const void* W3s,
                               const void* W2s, void* y, int32_t* topk_idx, float* topk_prob,
                               int32_t* tokens_per_expert, void* ws, cudaStream_t stream) {
  const SharedLayout S = make_shared_layout(c, fs);
  void* h_mid_s = at<void>(ws, S.h_mid_s);
  float* y_shared = at<float>(ws, S.y_shared);
  int* err = at<int>(ws, make_layout(c).err);

  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* side = nullptr;
  MOE_TRY(side_stream(&side));
  // fork: the shared expert on the side stream, after everything already on `stream`
  MOE_CUDA(cudaEventRecord(side->fork, stream));
  MOE_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
  const moe_status st_side = do_shared(c, fs, x, W1s, W3s, W2s, h_mid_s, y_shared, err,
                                       side->stream);
  const cudaError_t rec = cudaEventRecord(side->join, side->stream);
  Routed r{};
  // bf16 without padding: fc2 into the fp16 y_perm (a scale per 32 columns)
  const bool f16s = c.dtype == MOE_BF16 && !c.pad_to_capacity;
  const Layout L = make_layout(c);
  moe_status st = routed_path(c, x, Wg, gate_bias, expert_bias, W1, W3, W2, topk_idx, topk_prob,
                              tokens_per_expert, ws, stream, &r, f16s);
  if (st == MOE_OK && f16s &&
      launch_tc_fc2_f16s(c.num_experts, c.hidden, c.ffn_hidden, rows_of(c), at<void>(ws, L.h_mid),
                         at<int32_t>(ws, L.offsets), W2, ws_y16(ws, L), ws_y16_exp(c, ws, L), err,
                         stream) != cudaSuccess)
    st = MOE_ERR_CUDA;
  // join even after a failure, so that `stream` never stays forked (a capture
  // in progress would be invalidated)
  const cudaError_t wait = rec == cudaSuccess ? cudaStreamWaitEvent(stream, side->join, 0) : rec;
  MOE_TRY(st_side);
  MOE_TRY(st);
  MOE_CUDA(wait);
  if (f16s)
    MOE_CUDA(launch_combine_f16s(c.num_tokens, c.hidden, c.topk, ws_y16(ws, L),
                                 ws_y16_exp(c, ws, L), r.row_map, r.prob, y_shared, y, stream,
                                 rows_of(c)));
  else
    MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype, r.y_perm, r.row_map, r.prob,
                            y_shared, y, stream, rows_of(c)));
  return MOE_OK;
}

// moe_forward_e4m3 after its argument checks (also one batch of
// moe_forward_host_e4m3).
moe_status e4m3_forward_body(const moe_config& c, const void* x, const float* Wg,
                             const float* gate_bias, const float* expert_bias, const uint8_t* W1q,
                             const float* s1, const uint8_t* W3q, const float* s3,
                             const uint8_t* W2q, const float* s2, void* y, int32_t* topk_idx,
                             float* topk_prob, int32_t* tokens_per_expert, void* ws,
                             cudaStream_t stream) {
  const E4m3Layout Q = make_e4m3_layout(c);
  const Layout L = make_layout(c);
  int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.topk_idx);
  float* prob = topk_prob ? topk_prob : at<float>(ws, L.topk_prob);
  int32_t* tpe = tokens_per_expert ? tokens_per_expert : at<int32_t>(ws, L.tpe);
  uint8_t* keep = at<uint8_t>(ws, L.keep);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_map = at<int32_t>(ws, L.row_map);
  uint8_t* xperm_q = at<uint8_t>(ws, Q.xperm_q);
  float* xperm_s = at<float>(ws, Q.xperm_s);
  uint8_t* map = c.pad_to_capacity ? at<uint8_t>(ws, L.map) : nullptr;
  MOE_TRY(do_route(c, x, Wg, gate_bias, expert_bias, idx, prob, keep, tpe, map, ws, stream));
  if (map)
    MOE_TRY(do_permute_map_e4m3(c, x, map, idx, keep, xperm_q, xperm_s, row_map, offsets, ws,
                                stream));
  else
    MOE_TRY(do_permute_e4m3(c, x, idx, keep, xperm_q, xperm_s, row_map, offsets, ws, stream));
  // y_perm as fp16 with one power-of-two scale per 32 columns (the compact
  // y_perm of the bf16 forward), in the workspace's y_perm region
  void* y16 = ws_y16(ws, L);
  int8_t* y16e = ws_y16_exp(c, ws, L);
  MOE_TRY(do_mlp_e4m3(c, xperm_q, xperm_s, offsets, W1q, s1, W3q, s3, W2q, s2,
                      at<void>(ws, L.h_mid), at<uint8_t>(ws, Q.hq), at<float>(ws, Q.hs), nullptr,
                      ws, stream, y16, y16e));
  MOE_CUDA(launch_combine_f16s(c.num_tokens, c.hidden, c.topk, y16, y16e, row_map, prob, nullptr,
                               y, stream, rows_of(c)));
  return MOE_OK;
}

// The host-I/O loop of the moe_forward_host family: batch b's input is
// copied from the pinned host buffer into staging slot b & 1 on the h2d copy
// stream, forward(x_stage, y_stage) enqueues the forward on `stream`, and the
// output is copied back on the d2h stream, so that neighbouring batches'
// copies overlap the current batch's compute.  Per slot, events order input
// ready / input free / output ready / output free.
template <typename F>
moe_status host_pipeline(const moe_config& c, int32_t num_batches, const void* x_host,
                         size_t x_batch_stride, void* y_host, size_t y_batch_stride,
                         size_t row_bytes, const HostLayout& H, void* ws, cudaStream_t stream,
                         F&& forward) {
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStreams* cs = nullptr;
  MOE_TRY(copy_streams(&cs));
  // both copy streams start after everything already enqueued on `stream`
  MOE_CUDA(cudaEventRecord(cs->fork, stream));
  MOE_CUDA(cudaStreamWaitEvent(cs->h2d, cs->fork, 0));
  MOE_CUDA(cudaStreamWaitEvent(cs->d2h, cs->fork, 0));
  moe_status st = MOE_OK;
  for (int32_t b = 0; b < num_batches && st == MOE_OK; ++b) {
    const int slot = b & 1;
    void* xs = at<void>(ws, H.x_stage[slot]);
    void* ys = at<void>(ws, H.y_stage[slot]);
    const char* xb = static_cast<const char*>(x_host) + static_cast<size_t>(b) * x_batch_stride;
    char* yb = static_cast<char*>(y_host) + static_cast<size_t>(b) * y_batch_stride;
    // input copy: after the forward that last read this staging slot
    st = cuda_status(cudaStreamWaitEvent(cs->h2d, cs->x_free[slot], 0));
    if (st == MOE_OK && row_bytes)
      st = cuda_status(cudaMemcpyAsync(xs, xb, row_bytes, cudaMemcpyHostToDevice, cs->h2d));
    if (st == MOE_OK) st = cuda_status(cudaEventRecord(cs->x_ready[slot], cs->h2d));
    // forward: after its input landed and the output slot was copied out
    if (st == MOE_OK) st = cuda_status(cudaStreamWaitEvent(stream, cs->x_ready[slot], 0));
    if (st == MOE_OK) st = cuda_status(cudaStreamWaitEvent(stream, cs->y_free[slot], 0));
    if (st == MOE_OK) st = forward(xs, ys);
    if (st == MOE_OK) st = cuda_status(cudaEventRecord(cs->x_free[slot], stream));
    if (st == MOE_OK) st = cuda_status(cudaEventRecord(cs->y_ready[slot], stream));
    // output copy: after the forward wrote it
    if (st == MOE_OK) st = cuda_status(cudaStreamWaitEvent(cs->d2h, cs->y_ready[slot], 0));
    if (st == MOE_OK && row_bytes)
      st = cuda_status(cudaMemcpyAsync(yb, ys, row_bytes, cudaMemcpyDeviceToHost, cs->d2h));
    if (st == MOE_OK) st = cuda_status(cudaEventRecord(cs->y_free[slot], cs->d2h));
  }
  // join: `stream` completes only after every copy (also after a failure, so
  // that no copy stream is left running ahead of the caller's stream)
  const cudaError_t j1 = cudaEventRecord(cs->h2d_done, cs->h2d);
  const cudaError_t j2 = cudaEventRecord(cs->d2h_done, cs->d2h);
  const cudaError_t w1 = j1 == cudaSuccess ? cudaStreamWaitEvent(stream, cs->h2d_done, 0) : j1;
  const cudaError_t w2 = j2 == cudaSuccess ? cudaStreamWaitEvent(stream, cs->d2h_done, 0) : j2;
  MOE_TRY(st);
  MOE_CUDA(w1);
  MOE_CUDA(w2);
  return MOE_OK;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_cuda_error(void) { return g_last_cuda_error; }

moe_status moe_capacity(const moe_config* cfg, int64_t* capacity) {
  MOE_TRY(validate(cfg));
  if (capacity == nullptr) return MOE_ERR_INVALID_ARG;
  *capacity = capacity_of(*cfg);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_max_rows(const moe_config* cfg, int64_t* rows) {
  MOE_TRY(validate(cfg));
  if (rows == nullptr) return MOE_ERR_INVALID_ARG;
  *rows = rows_of(*cfg);
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* Wg,
                     const float* gate_bias, const float* expert_bias, int32_t* topk_idx,
                     float* topk_prob, uint8_t* keep, int32_t* tokens_per_expert,
                     uint8_t* routing_map, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t T = c.num_tokens, E = c.num_experts, k = c.topk;
  MOE_TRY(need(x, T * c.hidden, 16));
  MOE_TRY(need(Wg, c.hidden * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(need(keep, T * k, 1));
  MOE_TRY(need(tokens_per_expert, E, 4));
  if (c.pad_to_capacity)  // the padded map is the output the padded permutation needs
    MOE_TRY(need(routing_map, T * E, 1));
  else
    MOE_TRY(optional(routing_map, 1));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_route(c, x, Wg, gate_bias, expert_bias, topk_idx, topk_prob, keep, tokens_per_expert,
                  routing_map, ws, stream);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       const uint8_t* keep, void* x_perm, int32_t* row_map,
                       int32_t* expert_offsets, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (c.pad_to_capacity) return MOE_ERR_INVALID_ARG;  // padding rows come from the map
  const size_t T = c.num_tokens, k = c.topk;
  MOE_TRY(need(x, T * c.hidden, 16));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(optional(keep, 1));
  MOE_TRY(need(x_perm, T * k * c.hidden, 16));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_permute(c, x, topk_idx, keep, x_perm, row_map, expert_offsets, ws, stream);
}

moe_status moe_permute_map(const moe_config* cfg, const void* x, const uint8_t* routing_map,
                           const int32_t* topk_idx, const uint8_t* keep, void* x_perm,
                           int32_t* row_map, int32_t* expert_offsets, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t T = c.num_tokens, k = c.topk, E = c.num_experts;
  MOE_TRY(need(x, T * c.hidden, 16));
  MOE_TRY(need(routing_map, T * E, 1));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(optional(keep, 1));
  MOE_TRY(need(x_perm, static_cast<size_t>(rows_of(c)) * c.hidden, 16));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_permute_map(c, x, routing_map, topk_idx, keep, x_perm, row_map, expert_offsets, ws,
                        stream);
}

moe_status moe_grouped_fc1(const moe_config* cfg, const void* x_perm,
                           const int32_t* expert_offsets, const void* W1, const void* W3,
                           void* h_mid, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t R = static_cast<size_t>(rows_of(c));
  const size_t wsz = static_cast<size_t>(c.num_experts) * c.hidden * c.ffn_hidden;
  MOE_TRY(need(x_perm, R * c.hidden, 16));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(h_mid, R * c.ffn_hidden, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_fc1(c, x_perm, expert_offsets, W1, W3, h_mid, ws, stream);
}

moe_status moe_grouped_fc2(const moe_config* cfg, const void* h_mid,
                           const int32_t* expert_offsets, const void* W2, float* y_perm,
                           void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t R = static_cast<size_t>(rows_of(c));
  const size_t wsz = static_cast<size_t>(c.num_experts) * c.hidden * c.ffn_hidden;
  MOE_TRY(need(h_mid, R * c.ffn_hidden, 16));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(y_perm, R * c.hidden, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_fc2(c, h_mid, expert_offsets, W2, y_perm, ws, stream);
}

moe_status moe_grouped_mlp(const moe_config* cfg, const void* x_perm,
                           const int32_t* expert_offsets, const void* W1, const void* W3,
                           const void* W2, void* h_mid, float* y_perm, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(moe_grouped_fc1(cfg, x_perm, expert_offsets, W1, W3, h_mid, ws, ws_bytes, stream));
  return moe_grouped_fc2(cfg, h_mid, expert_offsets, W2, y_perm, ws, ws_bytes, stream);
}

moe_status moe_grouped_fc2_f16s(const moe_config* cfg, const void* h_mid,
                                const int32_t* expert_offsets, const void* W2, void* y16,
                                int8_t* y16_exp, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const size_t R = static_cast<size_t>(rows_of(c));
  const size_t wsz = static_cast<size_t>(c.num_experts) * c.hidden * c.ffn_hidden;
  MOE_TRY(need(h_mid, R * c.ffn_hidden, 16));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(y16, R * c.hidden, 16));
  MOE_TRY(need(y16_exp, R * (c.hidden / 32), 8));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = make_layout(c);
  MOE_CUDA(launch_tc_fc2_f16s(c.num_experts, c.hidden, c.ffn_hidden, rows_of(c), h_mid,
                              expert_offsets, W2, y16, y16_exp, at<int>(ws, L.err), stream));
  return MOE_OK;
}

moe_status moe_combine_f16s(const moe_config* cfg, const void* y16, const int8_t* y16_exp,
                            const int32_t* row_map, const float* topk_prob,
                            const float* y_shared, void* y, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const size_t T = c.num_tokens, k = c.topk;
  const size_t R = static_cast<size_t>(rows_of(c));
  MOE_TRY(need(y16, R * c.hidden, 16));
  MOE_TRY(need(y16_exp, R * (c.hidden / 32), 8));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(optional(y_shared, 16));
  MOE_TRY(need(y, T * c.hidden, 16));
  MOE_CUDA(launch_combine_f16s(c.num_tokens, c.hidden, c.topk, y16, y16_exp, row_map, topk_prob,
                               y_shared, y, stream, rows_of(c)));
  return MOE_OK;
}

moe_status moe_grouped_fc2_combine(const moe_config* cfg, const void* h_mid,
                                   const int32_t* expert_offsets, const void* W2,
                                   const int32_t* row_map, const float* topk_prob, void* y,
                                   void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (!fc2_combine_ok(c)) return MOE_ERR_UNSUPPORTED;
  const size_t T = c.num_tokens, k = c.topk;
  const size_t R = static_cast<size_t>(rows_of(c));
  const size_t wsz = static_cast<size_t>(c.num_experts) * c.hidden * c.ffn_hidden;
  MOE_TRY(need(h_mid, R * c.ffn_hidden, 16));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(need(y, T * c.hidden, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_fc2_combine(c, h_mid, expert_offsets, W2, row_map, topk_prob, y, ws, stream);
}

moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* row_map,
                       const float* topk_prob, void* y, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t T = c.num_tokens, k = c.topk;
  MOE_TRY(need(y_perm, static_cast<size_t>(rows_of(c)) * c.hidden, 16));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(need(y, T * c.hidden, 16));
  MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype, y_perm, row_map, topk_prob,
                          nullptr, y, stream, rows_of(c)));
  return MOE_OK;
}

moe_status moe_combine_shared(const moe_config* cfg, const float* y_perm, const int32_t* row_map,
                              const float* topk_prob, const float* y_shared, void* y,
                              moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t T = c.num_tokens, k = c.topk;
  MOE_TRY(need(y_perm, static_cast<size_t>(rows_of(c)) * c.hidden, 16));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(topk_prob, T * k, 4));
  MOE_TRY(optional(y_shared, 16));
  MOE_TRY(need(y, T * c.hidden, 16));
  MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype, y_perm, row_map, topk_prob,
                          y_shared, y, stream, rows_of(c)));
  return MOE_OK;
}

moe_status moe_shared_expert(const moe_config* cfg, int32_t fs, const void* x, const void* W1s,
                             const void* W3s, const void* W2s, void* h_mid_s, float* y_shared,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_fs(c, fs));
  const size_t T = c.num_tokens, h = c.hidden;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(W1s, h * fs, 16));
  MOE_TRY(need(W3s, h * fs, 16));
  MOE_TRY(need(W2s, h * fs, 16));
  MOE_TRY(need(h_mid_s, T * fs, 16));
  MOE_TRY(need(y_shared, T * h, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_shared(c, fs, x, W1s, W3s, W2s, h_mid_s, y_shared,
                   at<int>(ws, make_layout(c).err), stream);
}

moe_status moe_workspace_size_shared(const moe_config* cfg, int32_t fs, size_t* bytes) {
  MOE_TRY(validate(cfg));
  MOE_TRY(validate_fs(*cfg, fs));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_shared_layout(*cfg, fs).total;
  return MOE_OK;
}

moe_status moe_forward_shared(const moe_config* cfg, int32_t fs, const void* x, const float* Wg,
                              const float* gate_bias, const float* expert_bias, const void* W1,
                              const void* W3, const void* W2, const void* W1s, const void* W3s,
                              const void* W2s, void* y, int32_t* topk_idx, float* topk_prob,
                              int32_t* tokens_per_expert, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_fs(c, fs));
  const size_t T = c.num_tokens, E = c.num_experts, h = c.hidden;
  const size_t wsz = E * h * c.ffn_hidden;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(W1s, h * fs, 16));
  MOE_TRY(need(W3s, h * fs, 16));
  MOE_TRY(need(W2s, h * fs, 16));
  MOE_TRY(need(y, T * h, 16));
  MOE_TRY(optional(topk_idx, 4));
  MOE_TRY(optional(topk_prob, 4));
  MOE_TRY(optional(tokens_per_expert, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes, make_shared_layout(c, fs).total));
  return shared_forward_body(c, fs, x, Wg, gate_bias, expert_bias, W1, W3, W2, W1s, W3s, W2s, y,
                             topk_idx, topk_prob, tokens_per_expert, ws, stream);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const float* Wg,
                       const float* gate_bias, const float* expert_bias, const void* W1,
                       const void* W3, const void* W2, void* y, int32_t* topk_idx,
                       float* topk_prob, int32_t* tokens_per_expert, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const size_t T = c.num_tokens, E = c.num_experts, h = c.hidden;
  const size_t wsz = E * h * c.ffn_hidden;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(y, T * h, 16));
  MOE_TRY(optional(topk_idx, 4));
  MOE_TRY(optional(topk_prob, 4));
  MOE_TRY(optional(tokens_per_expert, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  Routed r;
  // non-padded layers: fc2 and the combine through do_fc2_combine (top-1 fused,
  // top-k over the fp16 y_perm)
  const bool fuse = fc2_combine_ok(c);
  MOE_TRY(routed_path(c, x, Wg, gate_bias, expert_bias, W1, W3, W2, topk_idx, topk_prob,
                      tokens_per_expert, ws, stream, &r, fuse));
  if (fuse) {
    const Layout L = make_layout(c);
    return do_fc2_combine(c, at<void>(ws, L.h_mid), at<int32_t>(ws, L.offsets), W2, r.row_map,
                          r.prob, y, ws, stream);
  }
  MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype, r.y_perm, r.row_map, r.prob,
                          nullptr, y, stream, rows_of(c)));
  return MOE_OK;
}

moe_status moe_quantize_rows_e4m3(int64_t rows, int32_t cols, const void* in, uint8_t* codes,
                                  float* scales, moe_stream_t stream) {
  if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (cols % 16 != 0) return MOE_ERR_UNSUPPORTED;
  const size_t n = static_cast<size_t>(rows) * cols;
  MOE_TRY(need(in, n, 16));
  MOE_TRY(need(codes, n, 16));
  MOE_TRY(need(scales, static_cast<size_t>(rows), 4));
  MOE_CUDA(launch_quantize_rows(rows, cols, in, codes, scales, nullptr, stream));
  return MOE_OK;
}

moe_status moe_quantize_experts_e4m3(const moe_config* cfg, const void* W1, const void* W3,
                                     const void* W2, uint8_t* W1q, uint8_t* W3q, uint8_t* W2q,
                                     float* s1, float* s3, float* s2, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t E = c.num_experts, h = c.hidden, f = c.ffn_hidden, wsz = E * h * f;
  for (const void* p : {W1, W3, W2}) MOE_TRY(need(p, wsz, 16));
  for (const void* p : {static_cast<const void*>(W1q), static_cast<const void*>(W3q),
                        static_cast<const void*>(W2q)})
    MOE_TRY(need(p, wsz, 16));
  MOE_TRY(need(s1, E * f, 16));
  MOE_TRY(need(s3, E * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  MOE_CUDA(launch_quantize_cols(c.num_experts, c.hidden, c.ffn_hidden, W1, W1q, s1, stream));
  MOE_CUDA(launch_quantize_cols(c.num_experts, c.hidden, c.ffn_hidden, W3, W3q, s3, stream));
  MOE_CUDA(launch_quantize_cols(c.num_experts, c.ffn_hidden, c.hidden, W2, W2q, s2, stream));
  return MOE_OK;
}

moe_status moe_workspace_size_e4m3(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  MOE_TRY(validate_e4m3(*cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_e4m3_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_permute_e4m3(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                            const uint8_t* keep, uint8_t* x_perm_q, float* x_perm_scale,
                            int32_t* row_map, int32_t* expert_offsets, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  if (c.pad_to_capacity) return MOE_ERR_INVALID_ARG;  // padding rows come from the map
  const size_t T = c.num_tokens, k = c.topk;
  MOE_TRY(need(x, T * c.hidden, 16));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(optional(keep, 1));
  MOE_TRY(need(x_perm_q, T * k * c.hidden, 16));
  MOE_TRY(need(x_perm_scale, T * k, 4));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(expert_offsets, c.num_experts + 1, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes, make_e4m3_layout(c).total));
  return do_permute_e4m3(c, x, topk_idx, keep, x_perm_q, x_perm_scale, row_map, expert_offsets,
                         ws, stream);
}

moe_status moe_permute_map_e4m3(const moe_config* cfg, const void* x, const uint8_t* routing_map,
                                const int32_t* topk_idx, const uint8_t* keep, uint8_t* x_perm_q,
                                float* x_perm_scale, int32_t* row_map, int32_t* expert_offsets,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  if (!c.pad_to_capacity) return MOE_ERR_INVALID_ARG;  // its token scratch is the padded layout's
  const size_t T = c.num_tokens, k = c.topk, E = c.num_experts;
  const size_t R = static_cast<size_t>(rows_of(c));
  MOE_TRY(need(x, T * c.hidden, 16));
  MOE_TRY(need(routing_map, T * E, 1));
  MOE_TRY(need(topk_idx, T * k, 4));
  MOE_TRY(optional(keep, 1));
  MOE_TRY(need(x_perm_q, R * c.hidden, 16));
  MOE_TRY(need(x_perm_scale, R, 4));
  MOE_TRY(need(row_map, T * k, 4));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes, make_e4m3_layout(c).total));
  return do_permute_map_e4m3(c, x, routing_map, topk_idx, keep, x_perm_q, x_perm_scale, row_map,
                             expert_offsets, ws, stream);
}

moe_status moe_grouped_mlp_e4m3(const moe_config* cfg, const uint8_t* x_perm_q,
                                const float* x_perm_scale, const int32_t* expert_offsets,
                                const uint8_t* W1q, const float* s1, const uint8_t* W3q,
                                const float* s3, const uint8_t* W2q, const float* s2,
                                void* h_mid, uint8_t* h_q, float* h_scale, float* y_perm,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t R = static_cast<size_t>(rows_of(c)), E = c.num_experts;
  const size_t h = c.hidden, f = c.ffn_hidden, wsz = E * h * f;
  MOE_TRY(need(x_perm_q, R * h, 16));
  MOE_TRY(need(x_perm_scale, R, 4));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(need(W1q, wsz, 16));
  MOE_TRY(need(W3q, wsz, 16));
  MOE_TRY(need(W2q, wsz, 16));
  MOE_TRY(need(s1, E * f, 16));
  MOE_TRY(need(s3, E * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  MOE_TRY(need(h_mid, R * f, 16));
  MOE_TRY(need(h_q, R * f, 16));
  MOE_TRY(need(h_scale, R, 4));
  MOE_TRY(need(y_perm, R * h, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return do_mlp_e4m3(c, x_perm_q, x_perm_scale, expert_offsets, W1q, s1, W3q, s3, W2q, s2, h_mid,
                     h_q, h_scale, y_perm, ws, stream);
}

moe_status moe_grouped_fc1_e4m3(const moe_config* cfg, const uint8_t* x_perm_q,
                                const float* x_perm_scale, const int32_t* expert_offsets,
                                const uint8_t* W1q, const float* s1, const uint8_t* W3q,
                                const float* s3, void* h_mid, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t R = static_cast<size_t>(rows_of(c)), E = c.num_experts;
  const size_t h = c.hidden, f = c.ffn_hidden, wsz = E * h * f;
  MOE_TRY(need(x_perm_q, R * h, 16));
  MOE_TRY(need(x_perm_scale, R, 4));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(need(W1q, wsz, 16));
  MOE_TRY(need(W3q, wsz, 16));
  MOE_TRY(need(s1, E * f, 16));
  MOE_TRY(need(s3, E * f, 16));
  MOE_TRY(need(h_mid, R * f, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  int* err = at<int>(ws, make_layout(c).err);
  MOE_CUDA(launch_tc_fc1_e4m3(c.num_experts, c.hidden, c.ffn_hidden, static_cast<int64_t>(R),
                              x_perm_q, x_perm_scale, nullptr, expert_offsets, W1q, s1, W3q, s3,
                              h_mid, err, stream));
  return MOE_OK;
}

moe_status moe_grouped_fc2_e4m3(const moe_config* cfg, const void* h_mid,
                                const int32_t* expert_offsets, const uint8_t* W2q,
                                const float* s2, uint8_t* h_q, float* h_scale, float* y_perm,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t R = static_cast<size_t>(rows_of(c)), E = c.num_experts;
  const size_t h = c.hidden, f = c.ffn_hidden;
  MOE_TRY(need(h_mid, R * f, 16));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(need(W2q, E * h * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  MOE_TRY(need(h_q, R * f, 16));
  MOE_TRY(need(h_scale, R, 4));
  MOE_TRY(need(y_perm, R * h, 16));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  int* err = at<int>(ws, make_layout(c).err);
  MOE_CUDA(launch_quantize_rows(static_cast<int64_t>(R), c.ffn_hidden, h_mid, h_q, h_scale,
                                expert_offsets + c.num_experts, stream));
  MOE_CUDA(launch_tc_fc2_e4m3(c.num_experts, c.hidden, c.ffn_hidden, static_cast<int64_t>(R), h_q,
                              h_scale, expert_offsets, W2q, s2, y_perm, err, stream));
  return MOE_OK;
}

moe_status moe_grouped_fc2_e4m3_f16s(const moe_config* cfg, const void* h_mid,
                                     const int32_t* expert_offsets, const uint8_t* W2q,
                                     const float* s2, uint8_t* h_q, float* h_scale, void* y16,
                                     int8_t* y16_exp, void* ws, size_t ws_bytes,
                                     moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t R = static_cast<size_t>(rows_of(c)), E = c.num_experts;
  const size_t h = c.hidden, f = c.ffn_hidden;
  MOE_TRY(need(h_mid, R * f, 16));
  MOE_TRY(need(expert_offsets, E + 1, 4));
  MOE_TRY(need(W2q, E * h * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  MOE_TRY(need(h_q, R * f, 16));
  MOE_TRY(need(h_scale, R, 4));
  MOE_TRY(need(y16, R * h, 16));
  MOE_TRY(need(y16_exp, R * (h / 32), 8));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  int* err = at<int>(ws, make_layout(c).err);
  MOE_CUDA(launch_quantize_rows(static_cast<int64_t>(R), c.ffn_hidden, h_mid, h_q, h_scale,
                                expert_offsets + c.num_experts, stream));
  MOE_CUDA(launch_tc_fc2_e4m3_f16s(c.num_experts, c.hidden, c.ffn_hidden, static_cast<int64_t>(R),
                                   h_q, h_scale, expert_offsets, W2q, s2, y16, y16_exp, err,
                                   stream));
  return MOE_OK;
}

moe_status moe_forward_e4m3(const moe_config* cfg, const void* x, const float* Wg,
                            const float* gate_bias, const float* expert_bias, const uint8_t* W1q,
                            const float* s1, const uint8_t* W3q, const float* s3,
                            const uint8_t* W2q, const float* s2, void* y, int32_t* topk_idx,
                            float* topk_prob, int32_t* tokens_per_expert, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  const size_t T = c.num_tokens, E = c.num_experts, h = c.hidden, f = c.ffn_hidden;
  const size_t wsz = E * h * f;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1q, wsz, 16));
  MOE_TRY(need(W3q, wsz, 16));
  MOE_TRY(need(W2q, wsz, 16));
  MOE_TRY(need(s1, E * f, 16));
  MOE_TRY(need(s3, E * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  MOE_TRY(need(y, T * h, 16));
  MOE_TRY(optional(topk_idx, 4));
  MOE_TRY(optional(topk_prob, 4));
  MOE_TRY(optional(tokens_per_expert, 4));
  MOE_TRY(check_ws(c, ws, ws_bytes, make_e4m3_layout(c).total));
  return e4m3_forward_body(c, x, Wg, gate_bias, expert_bias, W1q, s1, W3q, s3, W2q, s2, y,
                           topk_idx, topk_prob, tokens_per_expert, ws, stream);
}

moe_status moe_workspace_size_backward(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_bwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const float* Wg,
                        const float* gate_bias, const void* W1, const void* W3, const void* W2,
                        const int32_t* topk_idx, const float* topk_prob, const int32_t* row_map,
                        const int32_t* expert_offsets, const void* x_perm, const void* h_mid,
                        const float* y_perm, const void* dy, void* dx, float* dWg,
                        float* dgate_bias, float* dW1, float* dW3, float* dW2, void* ws,
                        size_t ws_bytes, moe_stream_t stream) {
  return do_backward(cfg, x, Wg, gate_bias, W1, W3, W2, topk_idx, topk_prob, row_map,
                     expert_offsets, x_perm, h_mid, y_perm, dy, dx, dWg, dgate_bias, dW1, dW3, dW2,
                     nullptr, ws, ws_bytes, stream);
}

moe_status moe_workspace_size_backward_shared(const moe_config* cfg, int32_t fs, size_t* bytes) {
  MOE_TRY(validate(cfg));
  MOE_TRY(validate_fs(*cfg, fs));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_bwd_layout(*cfg, fs).total;
  return MOE_OK;
}

moe_status moe_backward_shared(const moe_config* cfg, int32_t fs, const void* x, const float* Wg,
                               const float* gate_bias, const void* W1, const void* W3,
                               const void* W2, const void* W1s, const void* W3s, const void* W2s,
                               const int32_t* topk_idx, const float* topk_prob,
                               const int32_t* row_map, const int32_t* expert_offsets,
                               const void* x_perm, const void* h_mid, const float* y_perm,
                               const void* h_mid_s, const void* dy, void* dx, float* dWg,
                               float* dgate_bias, float* dW1, float* dW3, float* dW2, float* dW1s,
                               float* dW3s, float* dW2s, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  const SharedBwd sh{fs, W1s, W3s, W2s, h_mid_s, dW1s, dW3s, dW2s};
  return do_backward(cfg, x, Wg, gate_bias, W1, W3, W2, topk_idx, topk_prob, row_map,
                     expert_offsets, x_perm, h_mid, y_perm, dy, dx, dWg, dgate_bias, dW1, dW3, dW2,
                     &sh, ws, ws_bytes, stream);
}

moe_status moe_shared_expert_backward(const moe_config* cfg, int32_t fs, const void* x,
                                      const void* W1s, const void* W3s, const void* W2s,
                                      const void* h_mid_s, const void* dy, float* dx_acc,
                                      float* dW1s, float* dW3s, float* dW2s, void* ws,
                                      size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  const SharedBwd sh{fs, W1s, W3s, W2s, h_mid_s, dW1s, dW3s, dW2s};
  MOE_TRY(check_shared_bwd(c, sh));
  const size_t T = c.num_tokens, h = c.hidden;
  MOE_TRY(need(x, T * h, 16));
  MOE_TRY(need(dy, T * h, 16));
  MOE_TRY(need(dx_acc, T * h, 16));
  const BwdLayout B = make_bwd_layout(c, fs);
  MOE_TRY(check_ws(c, ws, ws_bytes, B.total));
  int* err = at<int>(ws, B.err);
  MOE_TRY(shared_bwd_dgrad(c, sh, x, dy, dx_acc, at<void>(ws, B.dH_s), at<void>(ws, B.dA_s), err,
                           stream));
  return shared_bwd_wgrad(c, sh, x, dy, at<void>(ws, B.dA_s), err, stream);
}

moe_status moe_workspace_size_host(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_host_layout(*cfg, make_layout(*cfg).total).total;
  return MOE_OK;
}

moe_status moe_forward_host(const moe_config* cfg, int32_t num_batches, const void* x_host,
                            size_t x_batch_stride, void* y_host, size_t y_batch_stride,
                            const float* Wg, const float* gate_bias, const float* expert_bias,
                            const void* W1, const void* W3, const void* W2, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  if (num_batches < 0) return MOE_ERR_INVALID_ARG;
  const size_t T = c.num_tokens, E = c.num_experts, h = c.hidden;
  const size_t row_bytes = T * h * (c.dtype == MOE_F32 ? 4 : 2);
  const size_t wsz = E * h * c.ffn_hidden;
  if (num_batches > 0 && row_bytes > 0 && (x_host == nullptr || y_host == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (num_batches > 1 && y_batch_stride != 0 && y_batch_stride < row_bytes)
    return MOE_ERR_INVALID_ARG;  // output batches would overlap
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(W2, wsz, 16));
  const HostLayout H = make_host_layout(c, make_layout(c).total);
  MOE_TRY(check_ws(c, ws, ws_bytes, H.total));
  if (num_batches == 0) return MOE_OK;

  return host_pipeline(c, num_batches, x_host, x_batch_stride, y_host, y_batch_stride, row_bytes,
                       H, ws, stream, [&](void* xs, void* ys) {
                         Routed r{};
                         const bool fuse = fc2_combine_ok(c);
                         MOE_TRY(routed_path(c, xs, Wg, gate_bias, expert_bias, W1, W3, W2,
                                             nullptr, nullptr, nullptr, ws, stream, &r, fuse));
                         if (fuse) {
                           const Layout L = make_layout(c);
                           return do_fc2_combine(c, at<void>(ws, L.h_mid),
                                                 at<int32_t>(ws, L.offsets), W2, r.row_map,
                                                 r.prob, ys, ws, stream);
                         }
                         MOE_CUDA(launch_combine(c.num_tokens, c.hidden, c.topk, c.dtype,
                                                 r.y_perm, r.row_map, r.prob, nullptr, ys,
                                                 stream, rows_of(c)));
                         return MOE_OK;
                       });
}

// Host-buffer argument checks shared by the moe_forward_host family.
static moe_status check_host_io(const moe_config& c, int32_t num_batches, const void* x_host,
                                void* y_host, size_t y_batch_stride, size_t* row_bytes) {
  if (num_batches < 0) return MOE_ERR_INVALID_ARG;
  *row_bytes = static_cast<size_t>(c.num_tokens) * c.hidden * (c.dtype == MOE_F32 ? 4 : 2);
  if (num_batches > 0 && *row_bytes > 0 && (x_host == nullptr || y_host == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (num_batches > 1 && y_batch_stride != 0 && y_batch_stride < *row_bytes)
    return MOE_ERR_INVALID_ARG;  // output batches would overlap
  return MOE_OK;
}

moe_status moe_workspace_size_host_shared(const moe_config* cfg, int32_t fs, size_t* bytes) {
  MOE_TRY(validate(cfg));
  MOE_TRY(validate_fs(*cfg, fs));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_host_layout(*cfg, make_shared_layout(*cfg, fs).total).total;
  return MOE_OK;
}

moe_status moe_forward_host_shared(const moe_config* cfg, int32_t fs, int32_t num_batches,
                                   const void* x_host, size_t x_batch_stride, void* y_host,
                                   size_t y_batch_stride, const float* Wg, const float* gate_bias,
                                   const float* expert_bias, const void* W1, const void* W3,
                                   const void* W2, const void* W1s, const void* W3s,
                                   const void* W2s, void* ws, size_t ws_bytes,
                                   moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_fs(c, fs));
  size_t row_bytes = 0;
  MOE_TRY(check_host_io(c, num_batches, x_host, y_host, y_batch_stride, &row_bytes));
  const size_t E = c.num_experts, h = c.hidden, wsz = E * h * c.ffn_hidden;
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1, wsz, 16));
  MOE_TRY(need(W3, wsz, 16));
  MOE_TRY(need(W2, wsz, 16));
  MOE_TRY(need(W1s, h * fs, 16));
  MOE_TRY(need(W3s, h * fs, 16));
  MOE_TRY(need(W2s, h * fs, 16));
  const HostLayout H = make_host_layout(c, make_shared_layout(c, fs).total);
  MOE_TRY(check_ws(c, ws, ws_bytes, H.total));
  if (num_batches == 0) return MOE_OK;
  return host_pipeline(c, num_batches, x_host, x_batch_stride, y_host, y_batch_stride, row_bytes,
                       H, ws, stream, [&](void* xs, void* ys) {
                         return shared_forward_body(c, fs, xs, Wg, gate_bias, expert_bias, W1, W3,
                                                    W2, W1s, W3s, W2s, ys, nullptr, nullptr,
                                                    nullptr, ws, stream);
                       });
}

moe_status moe_workspace_size_host_e4m3(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  MOE_TRY(validate_e4m3(*cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_host_layout(*cfg, make_e4m3_layout(*cfg).total).total;
  return MOE_OK;
}

moe_status moe_forward_host_e4m3(const moe_config* cfg, int32_t num_batches, const void* x_host,
                                 size_t x_batch_stride, void* y_host, size_t y_batch_stride,
                                 const float* Wg, const float* gate_bias,
                                 const float* expert_bias, const uint8_t* W1q, const float* s1,
                                 const uint8_t* W3q, const float* s3, const uint8_t* W2q,
                                 const float* s2, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(validate_e4m3(c));
  size_t row_bytes = 0;
  MOE_TRY(check_host_io(c, num_batches, x_host, y_host, y_batch_stride, &row_bytes));
  const size_t E = c.num_experts, h = c.hidden, f = c.ffn_hidden, wsz = E * h * f;
  MOE_TRY(need(Wg, h * E, 4));
  MOE_TRY(optional(gate_bias, 4));
  MOE_TRY(optional(expert_bias, 4));
  MOE_TRY(need(W1q, wsz, 16));
  MOE_TRY(need(W3q, wsz, 16));
  MOE_TRY(need(W2q, wsz, 16));
  MOE_TRY(need(s1, E * f, 16));
  MOE_TRY(need(s3, E * f, 16));
  MOE_TRY(need(s2, E * h, 16));
  const HostLayout H = make_host_layout(c, make_e4m3_layout(c).total);
  MOE_TRY(check_ws(c, ws, ws_bytes, H.total));
  if (num_batches == 0) return MOE_OK;
  return host_pipeline(c, num_batches, x_host, x_batch_stride, y_host, y_batch_stride, row_bytes,
                       H, ws, stream, [&](void* xs, void* ys) {
                         return e4m3_forward_body(c, xs, Wg, gate_bias, expert_bias, W1q, s1, W3q,
                                                  s3, W2q, s2, ys, nullptr, nullptr, nullptr, ws,
                                                  stream);
                       });
}

moe_status moe_check(void* ws, moe_stream_t stream, int32_t* info) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaStreamSynchronize(stream));
  int32_t w[2] = {0, 0};
  MOE_CUDA(cudaMemcpyAsync(w, ws, sizeof(w), cudaMemcpyDeviceToHost, stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  if (info) *info = w[1];
  if (w[0] == DEV_ERR_NONE) return MOE_OK;
  MOE_CUDA(cudaMemsetAsync(ws, 0, sizeof(w), stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  return w[0] == DEV_ERR_TIMEOUT ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

}  // extern "C"
