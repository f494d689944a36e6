// Internal declarations shared by the kernels and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Device error word: the first 256 bytes of every workspace.
//   word[0] = code (0 none, DEV_ERR_INDEX, DEV_ERR_TIMEOUT), word[1] = info.
enum : int { DEV_ERR_NONE = 0, DEV_ERR_INDEX = 1, DEV_ERR_TIMEOUT = 2 };
constexpr size_t kErrBytes = 256;

// Programmatic dependent launch: a kernel launched with launch_dependent may
// start while the kernel before it on the stream is still running; it calls
// pdl_wait() before its first read of that kernel's output (the wait returns
// once that kernel has completed and its writes are visible; it returns at
// once when the kernel was launched normally).  pdl_trigger() lets the next
// dependent kernel launch before this one finishes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void report_error(int* err, int code, int info) {
  if (err == nullptr) return;
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, info);
}

// Pairs handled by one permutation tile (256 threads x 8 pairs).
constexpr int kPermTile = 2048;
constexpr int kPermThreads = 256;

inline int64_t perm_tiles(int64_t npairs) { return (npairs + kPermTile - 1) / kPermTile; }

// ---- router ----
// Router logits without the gate bias, as nsplit partial sums [nsplit][T][E]
// (nsplit <= kRouterMaxSplits) that the top-k kernel adds in order.
constexpr int kRouterMaxSplits = 16;
cudaError_t launch_router_logits(int T, int h, int E, int dtype, const void* x, const float* Wg,
                                 float* partials, int* nsplit, cudaStream_t s);
// num_groups > 1: group-limited top-k (group_topk groups kept per token)
cudaError_t launch_router_topk(int T, int E, int k, int score, int num_groups, int group_topk,
                               const float* logits, int nsplit,
                               const float* gate_bias, const float* expert_bias,
                               int32_t* topk_idx, float* topk_prob,
                               uint8_t* keep, uint8_t* routing_map, int32_t* counts, int* err,
                               cudaStream_t s);
// Permutation by a [T,E] routing map (pad_to_capacity): x rows of row_bytes
// (a multiple of 16) each; tile_counts holds map_tiles(T) x E ints, row_src
// max_rows ints; offsets [E+1] out; rows past max_rows are reported in err
// and not written.
int64_t map_tiles(int T);
cudaError_t launch_perm_by_map(int T, int row_bytes, int E, int k, int64_t max_rows,
                               const void* x, const uint8_t* map, const int32_t* topk_idx,
                               const uint8_t* keep, int32_t* tile_counts, int32_t* row_src,
                               void* x_perm, int32_t* row_map, int32_t* offsets, int* err,
                               cudaStream_t s);
// dst[r] = src[row_src[r]] for the rows of a map permutation (E4M3 scales)
cudaError_t launch_gather_scales(int64_t max_rows, const int32_t* total_rows,
                                 const int32_t* row_src, const float* src, float* dst,
                                 cudaStream_t s);
// pad_to_capacity: fill each expert's column of the routing map up to quota
// ones with the lowest-index tokens not routed to it (cand_off / cand_pair:
// the drop candidate lists; NULL when nothing is dropped: every token);
// tokens_per_expert holds the kept counts in and the quota out.
cudaError_t launch_pad_fill(int T, int E, int k, int quota, const int32_t* cand_off,
                            const int32_t* cand_pair, int32_t* tokens_per_expert, uint8_t* map,
                            cudaStream_t s);
// E <= 8 without groups (and h small enough for the whole gate matrix in
// shared memory): logits and top-k fused in one kernel
bool router_fused_ok(int h, int E, int k, int num_groups);
cudaError_t launch_router_fused(int T, int h, int E, int k, int dtype, int score, const void* x,
                                const float* Wg, const float* gate_bias,
                                const float* expert_bias, int32_t* topk_idx, float* topk_prob,
                                uint8_t* keep, uint8_t* routing_map, int32_t* counts, int* err,
                                cudaStream_t s);
cudaError_t launch_drop_select(int T, int E, int k, int64_t capacity, int policy,
                               const int32_t* cand_offsets, const int32_t* cand_pair,
                               float* topk_prob, uint8_t* keep, uint8_t* routing_map,
                               int32_t* kept_per_expert, cudaStream_t s);

// ---- permutation / combine ----
// The stable expert-major order of the T*k (token, slot) pairs: expert
// offsets [E+1], row_map [T*k] (-1 for dropped pairs), optionally row_src
// (pair of each row) and tokens_per_expert.  hist, then scan + rank in one
// launch (up to 128 tiles of 2048 pairs) or in two; tile_counts is
// perm_tiles(npairs) * E ints of scratch.
cudaError_t launch_perm_index(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                              int32_t* tile_counts, int32_t* row_map, int32_t* row_src,
                              int32_t* offsets, int32_t* tokens_per_expert, int* err,
                              cudaStream_t s);
cudaError_t launch_perm_hist(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                             int32_t* tile_counts, int* err, cudaStream_t s);
cudaError_t launch_perm_scan(int64_t ntiles, int E, int32_t* tile_counts, int32_t* offsets,
                             int32_t* tokens_per_expert, cudaStream_t s);
cudaError_t launch_perm_rank(int64_t npairs, int E, const int32_t* topk_idx, const uint8_t* keep,
                             const int32_t* tile_base, int32_t* row_map, int32_t* row_src,
                             cudaStream_t s);
cudaError_t launch_perm_copy(int T, int h, int k, int dtype, const void* x, const int32_t* row_map,
                             void* x_perm, cudaStream_t s);
// E4M3 rows: x bf16 [T,h] quantised per token on the way; codes and the
// token's scale go to each kept row
cudaError_t launch_perm_copy_e4m3(int T, int h, int k, const void* x, const int32_t* row_map,
                                  uint8_t* x_perm_q, float* row_scale, cudaStream_t s);
// y_shared [T, h] fp32 (nullable): the shared expert's output, added last;
// topk_prob nullable: unit weights (the backward's sum of dx rows)
// rows of y_perm at or past max_rows (default T*k) count as dropped pairs
cudaError_t launch_combine(int T, int h, int k, int dtype, const float* y_perm,
                           const int32_t* row_map, const float* topk_prob, const float* y_shared,
                           void* y, cudaStream_t s, int64_t max_rows = -1);
// Top-1 layers with the combine in fc2's epilogue: row -> (token, weight)
// and zero output rows for dropped tokens.
cudaError_t launch_top1_rows(int T, int h, int dtype, int64_t max_rows, const int32_t* row_map,
                             const float* topk_prob, int32_t* row_token, float* row_weight,
                             void* y, cudaStream_t s);

// ---- grouped GEMMs ----
// offsets == nullptr: one dense group (E must be 1) over rows [0, max_rows)
// fp32 SIMT path (dtype MOE_F32)
cudaError_t launch_simt_fc1(int E, int h, int f, int64_t max_rows, const float* x_perm,
                            const int32_t* offsets, const float* W1, const float* W3,
                            float* h_mid, int* err, cudaStream_t s);
cudaError_t launch_simt_fc2(int E, int h, int f, int64_t max_rows, const float* h_mid,
                            const int32_t* offsets, const float* W2, float* y_perm, int* err,
                            cudaStream_t s);
// the layer backward on the FMA units (fp32): dH = dY . W2[e]^T; the fc1
// recompute with the SwiGLU backward ([da | dg] [rows, 2f] from dH);
// dx = [da | dg] . [W1[e] ; W3[e]]^T (added to dx when accumulate);
// dW[e] [M, N] = A_e^T . B_e over expert e's rows (offsets NULL: one dense
// group of max_rows rows)
cudaError_t launch_simt_dgrad_fc2(int E, int h, int f, int64_t max_rows, const float* dY,
                                  const int32_t* offsets, const float* W2, float* dH, int* err,
                                  cudaStream_t s);
cudaError_t launch_simt_fc1_bwd(int E, int h, int f, int64_t max_rows, const float* x_perm,
                                const int32_t* offsets, const float* W1, const float* W3,
                                const float* dH, float* dA, int* err, cudaStream_t s);
cudaError_t launch_simt_dgrad_fc1(int E, int h, int f, int64_t max_rows, const float* dA,
                                  const int32_t* offsets, const float* W1, const float* W3,
                                  float* dx, int* err, cudaStream_t s, bool accumulate = false);
cudaError_t launch_simt_wgrad(int E, int M, int N, int64_t max_rows, const float* A, int lda,
                              const float* B, int ldb, const int32_t* offsets, float* dW,
                              int* err, cudaStream_t s);
// tcgen05 path (dtype MOE_BF16)
cudaError_t launch_tc_fc1(int E, int h, int f, int64_t max_rows, const void* x_perm,
                          const int32_t* offsets, const void* W1, const void* W3, void* h_mid,
                          int* err, cudaStream_t s);
cudaError_t launch_tc_fc2(int E, int h, int f, int64_t max_rows, const void* h_mid,
                          const int32_t* offsets, const void* W2, float* y_perm, int* err,
                          cudaStream_t s);
// fc2 with y_perm as fp16 and one power-of-two scale per 32 columns:
// y16 [rows, h] fp16, y16_exp [rows, h/32] int8, value = fp16 * 2^exp
cudaError_t launch_tc_fc2_f16s(int E, int h, int f, int64_t max_rows, const void* h_mid,
                               const int32_t* offsets, const void* W2, void* y16, int8_t* y16_exp,
                               int* err, cudaStream_t s);
// The combine reading that y_perm (bf16 output): the same slot-order fp32 sum
// of p * value, then the shared expert's fp32 row if given, one rounding.
cudaError_t launch_combine_f16s(int T, int h, int k, const void* y16, const int8_t* y16_exp,
                                const int32_t* row_map, const float* topk_prob,
                                const float* y_shared, void* y, cudaStream_t s,
                                int64_t max_rows);
// fc2 of a top-1 layer with the combine in the epilogue: y[row_token[r]] =
// bf16(row_weight[r] * (h_mid[r] . W2[e]))
cudaError_t launch_tc_fc2_top1(int E, int h, int f, int64_t max_rows, const void* h_mid,
                               const int32_t* offsets, const void* W2, const int32_t* row_token,
                               const float* row_weight, void* y, int* err, cudaStream_t s);

// E4M3 operands (kind::f8f6f4): xq / hq [rows, K] codes with per-row scales
// (x's through row_src: row r uses x_scale[row_src[r]]), K-major weights
// W1q/W3q [E,f,h], W2q [E,h,f] with per-channel scales s1/s3 [E,f], s2 [E,h]
cudaError_t launch_tc_fc1_e4m3(int E, int h, int f, int64_t max_rows, const uint8_t* xq,
                               const float* x_scale, const int32_t* row_src,
                               const int32_t* offsets, const uint8_t* W1q, const float* s1,
                               const uint8_t* W3q, const float* s3, void* h_mid, int* err,
                               cudaStream_t s);
// E4M3 fc2 with the fp16 y_perm (one power-of-two scale per 32 columns)
cudaError_t launch_tc_fc2_e4m3_f16s(int E, int h, int f, int64_t max_rows, const uint8_t* hq,
                                    const float* h_scale, const int32_t* offsets,
                                    const uint8_t* W2q, const float* s2, void* y16,
                                    int8_t* y16_exp, int* err, cudaStream_t s);
cudaError_t launch_tc_fc2_e4m3(int E, int h, int f, int64_t max_rows, const uint8_t* hq,
                               const float* h_scale, const int32_t* offsets, const uint8_t* W2q,
                               const float* s2, float* y_perm, int* err, cudaStream_t s);

// backward (bf16): fc2 dgrad dH [rows,f] = dY [rows,h] . W2[e]^T; fc1 recompute
// with the SwiGLU backward dA [rows,2f] = [da | dg] from dH; fc1 dgrad
// dX [rows,h] fp32 = dA . [W1[e] ; W3[e]]^T (added to dX when accumulate).
// With no offsets each runs as one dense group over rows [0, max_rows) (E = 1).
cudaError_t launch_tc_dgrad_fc2(int E, int h, int f, int64_t max_rows, const void* dY,
                                const int32_t* offsets, const void* W2, void* dH, int* err,
                                cudaStream_t s);
cudaError_t launch_tc_fc1_bwd(int E, int h, int f, int64_t max_rows, const void* x_perm,
                              const int32_t* offsets, const void* W1, const void* W3,
                              const void* dH, void* dA, int* err, cudaStream_t s);
cudaError_t launch_tc_dgrad_fc1(int E, int h, int f, int64_t max_rows, const void* dA,
                                const int32_t* offsets, const void* W1, const void* W3,
                                float* dX, int* err, cudaStream_t s, bool accumulate = false);

// wgrad: dW [E, M, N] fp32 = per expert X_e^T . Y_e over the expert's rows
// (X [rows, M] with row stride ldx, Y [rows, N] with row stride ldy, bf16);
// M % 128 == 0, N % 128 == 0; an expert without rows gets zeros
cudaError_t launch_tc_wgrad(int E, int M, int N, int64_t max_rows, const void* X, int ldx,
                            const void* Y, int ldy, const int32_t* offsets, float* dW, int* err,
                            cudaStream_t s);

// C [rows, N] fp32 (row stride ldc) = A [rows, K] . Bk [N, K]^T, bf16, one
// dense group; K % 64 == 0, N % 256 == 0
cudaError_t launch_tc_dense_nt_f32(int64_t rows, int K, int N, const void* A, const void* Bk,
                                   float* C, int ldc, int* err, cudaStream_t s);

// Router logits of a bf16 layer on the tensor cores: the fp32 gate weights
// split exactly into three bf16 pieces (launch_router_split3: Wk [3E, h],
// row p*E + e = piece p of Wg[:, e], K contiguous), then, with h cut into S
// splits of at most kRouterChainK (S <= kRouterMaxSplits / 3),
// partials[p*S + q][t][e] = x[t, split q] . piece p of Wg[split q, e] (bf16
// products, exact in fp32, accumulated in fp32 on the tensor cores): *nsplit
// = 3S partial sums that the top-k kernel adds in order.  h % 64 == 0,
// E % 4 == 0.
constexpr int kRouterChainK = 1024;
int router_ksplit(int h);
cudaError_t launch_router_split3(int h, int E, const float* Wg, void* Wk, cudaStream_t s);
cudaError_t launch_tc_router_logits(int T, int h, int E, const void* x, const void* Wk,
                                    float* partials, int* nsplit, int* err, cudaStream_t s);

// ---- backward around the GEMMs (backward.cu)
cudaError_t launch_combine_bwd(int T, int h, int k, int dtype, const void* dy,
                               const int32_t* row_map, const float* topk_prob,
                               const float* y_perm, void* dY_perm, float* dp, cudaStream_t s);
cudaError_t launch_router_bwd(int T, int E, int k, int score, const float* logits, int nsplit,
                              const float* gate_bias, const int32_t* topk_idx, const float* dp,
                              float* dlogits, cudaStream_t s);
// dWg partial sums need dwg_splits(T, h, E) * h * E floats at `part`
int dwg_splits(int T, int h, int E);
cudaError_t launch_router_param_grads(int T, int h, int E, int dtype, const void* x,
                                      const float* dl, float* dWg, float* part, float* dgb,
                                      cudaStream_t s);
cudaError_t launch_dx_router(int T, int h, int E, const float* dl, const float* Wg, float* out,
                             cudaStream_t s);
// The router's gradients on the tensor cores when E % 64 == 0: fp32 dl and
// Wg split into bf16 hi + lo (hi = bf16(v), lo = bf16(v - hi)), staged as
// dl3 [T, 3E] = [dl_hi | dl_lo | dl_hi] and wg3 [h, 3E] = [Wg_hi | Wg_hi |
// Wg_lo]; dWg = x^T [dl_hi | dl_lo] with the halves added (via dwg2 [h, 2E]),
// dx_router = dl3 . wg3^T (the lo . lo term, ~2^-16 relative, is dropped);
// dgate_bias (if given) as on the CUDA-core path
bool router_grads_on_tc(int E);
cudaError_t launch_router_grads_tc(int T, int h, int E, const void* x, const float* dl,
                                   const float* Wg, void* dl3, void* wg3, float* dwg2, float* dWg,
                                   float* dgb, float* dx_router, int* err, cudaStream_t s);

// ---- E4M3 quantisation (FP8 experts) ----
// rows of bf16 [rows, cols] -> codes + per-row power-of-two scales (rows >=
// *row_count skipped when row_count is given); cols % 16 == 0
cudaError_t launch_quantize_rows(int64_t rows, int cols, const void* in, uint8_t* codes,
                                 float* scales, const int32_t* row_count, cudaStream_t s);
// W [E][K][N] bf16 -> codes [E][N][K] + per-channel scales [E][N]; K, N % 64 == 0
cudaError_t launch_quantize_cols(int E, int K, int N, const void* W, uint8_t* codes,
                                 float* scales, cudaStream_t s);

int device_sm_count();

}  // namespace moe
