/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE layer forward.
 *
 * One MoE layer forward on one GPU: route -> (capacity drop) -> permute ->
 * grouped SwiGLU experts -> combine.  The operation is the one described on
 * the page "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
 * (r00kie-liu.github.io), §2 "MoE layer 主路径: route -> dispatch -> experts
 * -> combine", with the router of §3-§5, token dropping of §8, the
 * dispatcher's local permutation of §9 and the grouped experts of §10; and
 * on "MoE Internals: DeepSpeed-Megatron Expert Parallel Implementation"
 * (duoan.github.io), §8 "The All-to-All path" steps 2-4 and 6-8 (the
 * all-to-all exchanges are absent: one GPU, no collectives).
 *
 * Conventions (all entry points):
 *  - Pointers are DEVICE pointers owned by the caller, unless stated.  The
 *    library never allocates device memory; scratch comes from `ws`.
 *  - Every tensor is row-major and contiguous.  Device pointers must be
 *    16-byte aligned (MOE_ERR_INVALID_ARG otherwise).
 *  - Calls are asynchronous on `stream` and never synchronise the host.
 *    Per-expert counts stay on the device.
 *  - Argument errors are reported before anything is enqueued.  A failed
 *    launch returns MOE_ERR_CUDA.  Device-side checks (an expert id out of
 *    range, a bounded wait that ran out) set a sticky error word inside
 *    `ws`; moe_check() reads and clears it.
 *  - `ws` must be zero-filled once before its first use (the error word
 *    lives at its start); it is carved internally and may be reused by any
 *    call with the same configuration.  Its size is given by
 *    moe_workspace_size().
 *  - dtype: MOE_BF16 (x, W1/W3/W2, h_mid and y in bf16; tensor-core GEMMs
 *    with fp32 accumulation) or MOE_F32 (everything fp32; SIMT fp32 GEMMs).
 *    The router (Wg, biases, logits, probabilities) is always fp32, as the
 *    router dtype of §3 of the Megatron Core page.
 *  - Shape limits: 1 <= E <= 256, 1 <= k <= min(E, 8), T >= 0, h and f
 *    multiples of 8.  The bf16 path further needs h % 256 == 0 and
 *    f % 128 == 0 (MOE_ERR_UNSUPPORTED otherwise).
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 8

typedef struct CUstream_st* moe_stream_t; /* == cudaStream_t; NULL = legacy default stream */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,   /* shape outside the limits above */
  MOE_ERR_WORKSPACE = 3,     /* ws too small */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_CHECK = 5,  /* a kernel found an invalid index (moe_check) */
  MOE_ERR_TIMEOUT = 6        /* a bounded device wait ran out (moe_check) */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Score functions of §5 of the Megatron Core page (topk_routing_with_score_function). */
typedef enum moe_score {
  MOE_SCORE_SOFTMAX_POST = 0, /* top-k on logits, softmax over the k ("renormalised") */
  MOE_SCORE_SOFTMAX_PRE = 1,  /* softmax over all E, then top-k, no renormalisation */
  MOE_SCORE_SIGMOID = 2,      /* sigmoid; expert_bias only chooses; p = s/(sum s + 1e-20) */
  MOE_SCORE_SQRTSOFTPLUS = 3  /* s = sqrt(softplus(l)); bias and weights as for sigmoid */
} moe_score;

/* Drop policies of §8 of the Megatron Core page (apply_router_token_dropping). */
typedef enum moe_drop_policy {
  MOE_DROP_PROBS = 0,    /* keep the `capacity` highest-probability tokens of an expert */
  MOE_DROP_POSITION = 1  /* keep the first `capacity` tokens in token order */
} moe_drop_policy;

typedef struct moe_config {
  int32_t num_tokens;     /* T */
  int32_t hidden;         /* h */
  int32_t num_experts;    /* E */
  int32_t topk;           /* k */
  int32_t ffn_hidden;     /* f, the expert's intermediate size */
  int32_t score;          /* moe_score */
  int32_t dtype;          /* moe_dtype */
  int32_t drop_policy;    /* moe_drop_policy (used only when capacity_factor > 0) */
  float capacity_factor;  /* <= 0: dropless */
  int32_t min_capacity;   /* capacity is raised to at least this (default 0) */
  /* Group-limited top-k (compute_topk(scores, topk, num_groups, group_topk) of
   * §5; the page does not print its body).  num_groups <= 1: off.  Otherwise
   * the experts form num_groups contiguous groups of E/num_groups; a group's
   * score is the sum of its k/group_topk largest selection scores; each token
   * keeps the group_topk best groups (equal scores: lower group first) and
   * takes its top-k among their experts.  Needs E % num_groups == 0,
   * num_groups <= 32, 1 <= group_topk <= min(num_groups, k) and
   * k <= group_topk * E/num_groups (MOE_ERR_UNSUPPORTED otherwise). */
  int32_t num_groups;
  int32_t group_topk;
  /* pad_to_capacity of apply_router_token_dropping (§8 of the Megatron Core
   * page; moe_pad_expert_input_to_capacity): 1 needs capacity_factor > 0
   * (MOE_ERR_INVALID_ARG otherwise).  The routing map becomes the page's
   * capacity_mask: each expert's column holds exactly min(capacity, T)
   * tokens, its kept pairs and then, for an expert under capacity, the
   * lowest-index tokens not routed to it (the page leaves the order of those
   * equal zero probabilities open; lower token index first is the reading,
   * as for every tie here).  Padding tokens carry no combine weight, so the
   * layer output equals the unpadded one; the permuted buffers hold
   * E * min(capacity, T) rows (moe_max_rows).  0: off.  The E4M3 layer
   * permutes with moe_permute_map_e4m3 (moe_permute_e4m3 returns
   * MOE_ERR_INVALID_ARG); the backward gives the padding rows zero
   * gradients (they carry no combine weight). */
  int32_t pad_to_capacity;
} moe_config;

/* ABI version of the loaded library (MOE_ABI_VERSION). */
int32_t moe_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Text of the last CUDA runtime error behind an MOE_ERR_CUDA returned on the
 * calling host thread ("" if none). */
const char* moe_last_cuda_error(void);

/* Per-expert capacity of §8 of the Megatron Core page: get_capacity(T*k, E, cf),
 * read as ceil((T*k/E)*cf) raised to min_capacity.  *capacity = -1 when
 * dropless (capacity_factor <= 0).  Host-only. */
moe_status moe_capacity(const moe_config* cfg, int64_t* capacity);

/* Bytes of workspace needed by every entry point for this configuration
 * (the forward's need, which covers each stage).  Host-only. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Row capacity of the permuted buffers (x_perm, h_mid, y_perm): T*k (every
 * pair kept), or with pad_to_capacity max(T*k, E * min(capacity, T)). */
moe_status moe_max_rows(const moe_config* cfg, int64_t* rows);

/*
 * Router: §3 gating (logits = x.Wg + gate_bias in fp32), §4-§5 scoring and
 * top-k, and §8 token dropping when capacity_factor > 0.
 *   x            [T,h]  dtype
 *   Wg           [h,E]  fp32 (row i = the E gate weights of input feature i)
 *   gate_bias    [E]    fp32 or NULL: added to the logits (a skew of the router)
 *   expert_bias  [E]    fp32 or NULL: sigmoid / sqrtsoftplus scores only;
 *                       changes the choice, never the weights
 *   topk_idx     [T,k]  int32 out: experts, by selection score descending
 *                       (equal scores: lower expert index first)
 *   topk_prob    [T,k]  fp32 out: combine weights; 0 for dropped pairs
 *   keep         [T,k]  uint8 out: 1 kept, 0 dropped (all 1 when dropless)
 *   tokens_per_expert [E] int32 out: kept pairs per expert (pad_to_capacity:
 *                       the padded count min(capacity, T) of every expert)
 *   routing_map  [T,E]  uint8 out or NULL: 1 where (t,e) is a kept pair; with
 *                       pad_to_capacity it is required and also holds the
 *                       padding tokens (the input of moe_permute_map)
 * The logits are fp32 fused multiply-adds on the CUDA cores.  With
 * MOE_ROUTER_TC=1 in the environment (an opt-in), bf16 layers with E > 8 and
 * E % 4 == 0 form them on the tensor cores instead: Wg split exactly into
 * three bf16 pieces, bf16 products (exact in fp32) accumulated in fp32 chains
 * of at most 1024 products; the result differs from the default only by fp32
 * rounding.  The same applies to moe_forward and the backward's logits.
 */
moe_status moe_route(const moe_config* cfg, const void* x, const float* Wg,
                     const float* gate_bias, const float* expert_bias, int32_t* topk_idx,
                     float* topk_prob, uint8_t* keep, int32_t* tokens_per_expert,
                     uint8_t* routing_map, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Local permutation of §9 (dispatch_preprocess; sequence-major ->
 * expert-major): kept pair (t,j) with expert e goes to row
 * expert_offsets[e] + #{t' < t with a kept pair to e} (stable).
 *   x              [T,h]       dtype
 *   topk_idx, keep [T,k]       as produced by moe_route (keep may be NULL = all kept)
 *   x_perm         [T*k,h]     dtype out: rows [0, R) filled, R = expert_offsets[E]
 *   row_map        [T,k]       int32 out: row of each pair, -1 if dropped
 *   expert_offsets [E+1]       int32 out: exclusive prefix of kept counts
 * An expert id outside [0,E) is skipped and flagged (MOE_ERR_DEVICE_CHECK).
 * With pad_to_capacity the rows come from the padded routing map:
 * MOE_ERR_INVALID_ARG (use moe_permute_map).
 */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       const uint8_t* keep, void* x_perm, int32_t* row_map,
                       int32_t* expert_offsets, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * The permutation of §9 driven by a routing map, as the dispatcher does with
 * the map: expert e's rows are the tokens t with routing_map[t,e] = 1 in
 * ascending order, so padding tokens sit among the kept ones.
 *   x              [T,h]       dtype
 *   routing_map    [T,E]       uint8 (any nonzero byte counts as 1)
 *   topk_idx, keep [T,k]       (keep may be NULL = all kept); a kept pair's
 *                              expert column must be set in the map
 *   x_perm         [moe_max_rows,h] dtype out: rows [0, R) filled, R = the
 *                              map's ones (expert_offsets[E])
 *   row_map        [T,k]       int32 out: row of each kept pair, -1 otherwise
 *   expert_offsets [E+1]       int32 out: exclusive prefix of the column sums
 * A map with more ones than moe_max_rows rows: the rows past it are not
 * written and moe_check reports MOE_ERR_DEVICE_CHECK.  Any configuration;
 * with the routing map of moe_route and no padding it gives moe_permute's
 * result.
 */
moe_status moe_permute_map(const moe_config* cfg, const void* x, const uint8_t* routing_map,
                           const int32_t* topk_idx, const uint8_t* keep, void* x_perm,
                           int32_t* row_map, int32_t* expert_offsets, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/*
 * Grouped expert MLP of §10 (TEGroupedMLP: every local expert in one call),
 * SwiGLU: for the rows [expert_offsets[e], expert_offsets[e+1]) of expert e,
 *   h_mid = silu(x_perm . W1[e]) * (x_perm . W3[e]),  y_perm = h_mid . W2[e].
 *   x_perm [R_max,h] dtype, W1/W3 [E,h,f] dtype, W2 [E,f,h] dtype,
 *   h_mid [R_max,f] dtype out, y_perm [R_max,h] fp32 out (rows >= R untouched),
 *   R_max = moe_max_rows (T*k unless pad_to_capacity).
 * moe_grouped_fc1 / moe_grouped_fc2 are the two halves.
 */
moe_status moe_grouped_mlp(const moe_config* cfg, const void* x_perm,
                           const int32_t* expert_offsets, const void* W1, const void* W3,
                           const void* W2, void* h_mid, float* y_perm, void* ws,
                           size_t ws_bytes, moe_stream_t stream);
moe_status moe_grouped_fc1(const moe_config* cfg, const void* x_perm,
                           const int32_t* expert_offsets, const void* W1, const void* W3,
                           void* h_mid, void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_grouped_fc2(const moe_config* cfg, const void* h_mid,
                           const int32_t* expert_offsets, const void* W2, float* y_perm,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Combine (§2 combine / the unpermute-and-weight step 8 of the DeepSpeed
 * page): y[t] = sum over kept slots j, in slot order, of
 * topk_prob[t,j] * y_perm[row_map[t,j]], accumulated in fp32 and rounded
 * once to dtype.  A token with no kept pair gets 0.
 *   y_perm [R_max,h] fp32, row_map [T,k] int32, topk_prob [T,k] fp32, y [T,h] dtype out.
 */
moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* row_map,
                       const float* topk_prob, void* y, moe_stream_t stream);

/*
 * fc2 and the combine over a compact y_perm (bf16 layers): y_perm stored as
 * fp16 with one power-of-two scale per 32 columns, 2 + 1/32 bytes per value
 * instead of 4.  Row r's columns 32c .. 32c+31 hold
 *   y16[r, 32c + i] = fp16(y_perm[r, 32c + i] * 2^-y16_exp[r, c]),
 * the exponent chosen so that the chunk's largest magnitude lands in
 * [2^14, 2^15) (clamped to [-126, 113]; 0 for a non-finite chunk): a relative
 * error of at most 2^-11 per value, against bf16's 2^-8, which measured too
 * coarse for the layer's bf16 output bar (the output's error beyond its own
 * rounding must stay under 2e-2 of its RMS).  moe_combine_f16s is
 * moe_combine over the decoded values (fp16 * 2^exp, exact in fp32): the
 * same slot-order fp32 sum and one rounding; y_shared (nullable, fp32
 * [T,h]) is the shared expert's output, added after the routed sum as in
 * moe_combine_shared.  moe_forward uses this pair for bf16 layers with k >= 2
 * and no pad_to_capacity, moe_forward_shared for bf16 layers without
 * pad_to_capacity, and moe_forward_e4m3 (with moe_grouped_fc2_e4m3_f16s).
 * Megatron Core walkthrough §10 (experts) and §2 (combine).
 *   y16 [R_max,h] fp16, y16_exp [R_max,h/32] int8 (8-byte aligned); other arguments as
 *   moe_grouped_fc2 / moe_combine.  MOE_ERR_UNSUPPORTED for fp32 layers.
 */
moe_status moe_grouped_fc2_f16s(const moe_config* cfg, const void* h_mid,
                                const int32_t* expert_offsets, const void* W2, void* y16,
                                int8_t* y16_exp, void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_combine_f16s(const moe_config* cfg, const void* y16, const int8_t* y16_exp,
                            const int32_t* row_map, const float* topk_prob,
                            const float* y_shared, void* y, moe_stream_t stream);

/*
 * fc2 and the combine in one call (layers without pad_to_capacity), as
 * moe_forward runs them.  bf16 top-1 layers: the combine runs in fc2's
 * epilogue -- each row goes, weighted, straight into its token's output row
 * (no y_perm; the rows of dropped tokens are zeroed) -- with the bits of
 * moe_grouped_fc2 followed by moe_combine.  bf16 layers with k >= 2:
 * moe_grouped_fc2_f16s then moe_combine_f16s over the workspace.  fp32
 * layers: moe_grouped_fc2 into the workspace, then moe_combine.
 * Megatron Core walkthrough §10 (experts) and §2 (combine).
 *   h_mid [R_max,f] dtype, expert_offsets [E+1], W2 [E,f,h] dtype,
 *   row_map [T,k] int32, topk_prob [T,k] fp32, y [T,h] dtype out.
 * MOE_ERR_UNSUPPORTED with pad_to_capacity (padding rows have no slot);
 * ws: moe_workspace_size bytes (holds y_perm and the rows' tokens and
 * weights).  Calls that share a workspace must not overlap on the GPU.
 */
moe_status moe_grouped_fc2_combine(const moe_config* cfg, const void* h_mid,
                                   const int32_t* expert_offsets, const void* W2,
                                   const int32_t* row_map, const float* topk_prob, void* y,
                                   void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * The whole layer forward (route -> drop -> permute -> experts -> combine),
 * enqueued on `stream` without a host synchronisation.  Intermediates live in
 * `ws`.  topk_idx / topk_prob / tokens_per_expert may be NULL (kept in ws)
 * or caller buffers of the shapes given for moe_route.
 */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* Wg,
                       const float* gate_bias, const float* expert_bias, const void* W1,
                       const void* W3, const void* W2, void* y, int32_t* topk_idx,
                       float* topk_prob, int32_t* tokens_per_expert, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/*
 * Shared expert (§11 of the Megatron Core page, and the layer forward of its
 * §2: hidden = shared_expert(hidden_in) + routed output): one dense SwiGLU MLP
 * of width fs that every token goes through, chosen by no router, its output
 * added to the routed experts' combined output.
 *
 * moe_shared_expert: y_shared = (silu(x . W1s) * (x . W3s)) . W2s for all T
 * tokens (the grouped MLP kernels run as one dense group of T rows).
 *   fs: the shared expert's hidden width, > 0, a multiple of 8 (MOE_F32) or
 *       of 128 (MOE_BF16), else MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED.
 *   x [T,h] dtype, W1s/W3s [h,fs] dtype, W2s [fs,h] dtype,
 *   h_mid_s [T,fs] dtype out (scratch the caller owns), y_shared [T,h] fp32 out.
 *   ws / ws_bytes: a workspace of moe_workspace_size(cfg) bytes or more
 *   (only its error word is used).
 *
 * moe_combine_shared: moe_combine with the shared row added after the routed
 * slots, still in fp32 and rounded once: y[t] = sum_j p[t,j] * y_perm[..] +
 * y_shared[t].  y_shared may be NULL (then it is moe_combine).
 *
 * moe_workspace_size_shared: bytes of the workspace moe_forward_shared needs
 * (moe_workspace_size plus room for h_mid_s and y_shared).
 *
 * moe_forward_shared: moe_forward plus the shared expert.  The shared path
 * does not depend on the routing, so it is enqueued on a second stream of
 * the library's (forked from `stream` by an event and joined back before the
 * combine; capturable in a CUDA graph like the rest).  Same arguments as
 * moe_forward plus fs and the shared weights; ws is moe_workspace_size_shared
 * bytes.
 */
moe_status moe_shared_expert(const moe_config* cfg, int32_t fs, const void* x, const void* W1s,
                             const void* W3s, const void* W2s, void* h_mid_s, float* y_shared,
                             void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_combine_shared(const moe_config* cfg, const float* y_perm, const int32_t* row_map,
                              const float* topk_prob, const float* y_shared, void* y,
                              moe_stream_t stream);
moe_status moe_workspace_size_shared(const moe_config* cfg, int32_t fs, size_t* bytes);
moe_status moe_forward_shared(const moe_config* cfg, int32_t fs, const void* x, const float* Wg,
                              const float* gate_bias, const float* expert_bias, const void* W1,
                              const void* W3, const void* W2, const void* W1s, const void* W3s,
                              const void* W2s, void* y, int32_t* topk_idx, float* topk_prob,
                              int32_t* tokens_per_expert, void* ws, size_t ws_bytes,
                              moe_stream_t stream);

/*
 * FP8 experts.  The Megatron Core report on GB300 names FP8 GEMMs as its
 * most effective single optimisation but prints no scaling recipe; the one
 * used here: E4M3 codes (OCP 8-bit float, round-to-nearest-even, saturating
 * at 448) with one power-of-two scale 2^e per token row of x (and per row of
 * the SwiGLU output) and per output channel of every weight matrix, e the
 * smallest integer with amax * 2^-e <= 448 (amax below 2^-100 or not
 * finite: e = 0).  The grouped GEMMs run on E4M3 tensor-core MMAs
 * (kind::f8f6f4) with fp32 accumulation; scales are applied in the
 * epilogues; the SwiGLU output is rounded to bf16, quantised per row, and
 * the down projection runs on E4M3 as well.  Routing, permutation and the
 * combine are those of the bf16 path.  Needs dtype MOE_BF16 (x and y bf16;
 * MOE_ERR_UNSUPPORTED otherwise).
 *
 * moe_quantize_rows_e4m3: in [rows, cols] bf16 -> codes [rows, cols] uint8
 *   and scales [rows] fp32 (2^e).  cols % 16 == 0.
 * moe_quantize_experts_e4m3: the expert weights in E4M3, once, K-major
 *   (one row of codes per output channel): W1/W3 [E,h,f] bf16 -> W1q/W3q
 *   [E,f,h] codes and s1/s3 [E,f] scales; W2 [E,f,h] -> W2q [E,h,f] and
 *   s2 [E,h].  Scale arrays 16-byte aligned.
 * moe_workspace_size_e4m3: workspace bytes of the E4M3 entry points.
 * moe_permute_e4m3: moe_permute on E4M3 rows: x quantised per token, the
 *   kept pairs' code rows x_perm_q [T*k,h] and their scales x_perm_scale
 *   [T*k] in expert-major order; row_map and expert_offsets as moe_permute.
 * moe_grouped_mlp_e4m3: the E4M3 SwiGLU experts: h_mid [R_max,f] bf16,
 *   h_q [R_max,f] codes and h_scale [R_max] (the quantised SwiGLU output), and
 *   y_perm [R_max,h] fp32 out; rows >= expert_offsets[E] untouched (R_max =
 *   moe_max_rows: T*k unless pad_to_capacity).
 *   moe_grouped_fc1_e4m3 / moe_grouped_fc2_e4m3 are its two halves: fc1
 *   writes h_mid; fc2 quantises h_mid's rows (h_q, h_scale) and writes y_perm.
 * moe_forward_e4m3: the whole layer with E4M3 experts (arguments of
 *   moe_forward, with the quantised weights and their scales).
 */
moe_status moe_quantize_rows_e4m3(int64_t rows, int32_t cols, const void* in, uint8_t* codes,
                                  float* scales, moe_stream_t stream);
moe_status moe_quantize_experts_e4m3(const moe_config* cfg, const void* W1, const void* W3,
                                     const void* W2, uint8_t* W1q, uint8_t* W3q, uint8_t* W2q,
                                     float* s1, float* s3, float* s2, moe_stream_t stream);
moe_status moe_workspace_size_e4m3(const moe_config* cfg, size_t* bytes);
moe_status moe_permute_e4m3(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                            const uint8_t* keep, uint8_t* x_perm_q, float* x_perm_scale,
                            int32_t* row_map, int32_t* expert_offsets, void* ws,
                            size_t ws_bytes, moe_stream_t stream);
/* The E4M3 permutation by the padded routing map of pad_to_capacity (needs
 * it set; MOE_ERR_INVALID_ARG otherwise): every token's row quantised once,
 * the code rows and their scales placed as moe_permute_map places rows;
 * x_perm_q [moe_max_rows,h], x_perm_scale [moe_max_rows]. */
moe_status moe_permute_map_e4m3(const moe_config* cfg, const void* x, const uint8_t* routing_map,
                                const int32_t* topk_idx, const uint8_t* keep, uint8_t* x_perm_q,
                                float* x_perm_scale, int32_t* row_map, int32_t* expert_offsets,
                                void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_grouped_mlp_e4m3(const moe_config* cfg, const uint8_t* x_perm_q,
                                const float* x_perm_scale, const int32_t* expert_offsets,
                                const uint8_t* W1q, const float* s1, const uint8_t* W3q,
                                const float* s3, const uint8_t* W2q, const float* s2,
                                void* h_mid, uint8_t* h_q, float* h_scale, float* y_perm,
                                void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_grouped_fc1_e4m3(const moe_config* cfg, const uint8_t* x_perm_q,
                                const float* x_perm_scale, const int32_t* expert_offsets,
                                const uint8_t* W1q, const float* s1, const uint8_t* W3q,
                                const float* s3, void* h_mid, void* ws, size_t ws_bytes,
                                moe_stream_t stream);
moe_status moe_grouped_fc2_e4m3(const moe_config* cfg, const void* h_mid,
                                const int32_t* expert_offsets, const uint8_t* W2q,
                                const float* s2, uint8_t* h_q, float* h_scale, float* y_perm,
                                void* ws, size_t ws_bytes, moe_stream_t stream);
/* moe_grouped_fc2_e4m3 with y_perm stored as fp16 and one power-of-two scale
 * per 32 columns (y16, y16_exp: the layout of moe_grouped_fc2_f16s), for
 * moe_combine_f16s.  moe_forward_e4m3 runs this pair. */
moe_status moe_grouped_fc2_e4m3_f16s(const moe_config* cfg, const void* h_mid,
                                     const int32_t* expert_offsets, const uint8_t* W2q,
                                     const float* s2, uint8_t* h_q, float* h_scale, void* y16,
                                     int8_t* y16_exp, void* ws, size_t ws_bytes,
                                     moe_stream_t stream);
moe_status moe_forward_e4m3(const moe_config* cfg, const void* x, const float* Wg,
                            const float* gate_bias, const float* expert_bias, const uint8_t* W1q,
                            const float* s1, const uint8_t* W3q, const float* s3,
                            const uint8_t* W2q, const float* s2, void* y, int32_t* topk_idx,
                            float* topk_prob, int32_t* tokens_per_expert, void* ws,
                            size_t ws_bytes, moe_stream_t stream);

/*
 * Backward of the layer (the training step every page's training system
 * runs; the pages print no backward, so it is the chain rule on the
 * forward's definitions): gradients of L = sum(dy * y) for the routing
 * decisions the forward took.  The top-k choice and the capacity drop carry
 * no gradient; the expert bias only chooses and gets none.  Per kept pair:
 * dY = p dy, dp = <dy, Y>, dH = dY W2^T, SwiGLU backward (a and g
 * recomputed by fc1), dX = [da|dg] [W1;W3]^T, dW2 = H^T dY, dW1 = X^T da,
 * dW3 = X^T dg; the router gets dlogits from dp through the score function,
 * dWg = x^T dlogits, dgate_bias = sum_t dlogits, and dx gains dlogits Wg^T.
 * bf16: the expert GEMMs run on the tensor cores (dgrad with the weights
 * read in place, wgrad reducing over each expert's rows); dY, dH, da and dg
 * are rounded to bf16 as GEMM operands; accumulation is fp32.  MOE_F32: the
 * same GEMMs on the FMA units, every intermediate fp32.  pad_to_capacity:
 * the saved buffers hold the padded rows (moe_max_rows); their dY rows are
 * zero, so they add nothing to any gradient.
 *   Saved from the forward (the staged calls' outputs): topk_idx and
 *   topk_prob [T,k] (moe_route), row_map [T,k], expert_offsets [E+1] and
 *   x_perm [R_max,h] (moe_permute), h_mid [R_max,f] and y_perm [R_max,h] fp32
 *   (moe_grouped_mlp).  Parameters as in moe_forward.
 *   dy [T,h] dtype in; dx [T,h] dtype out; dWg [h,E], dgate_bias [E]
 *   (nullable), dW1/dW3 [E,h,f], dW2 [E,f,h] fp32 out (overwritten).
 *   ws: moe_workspace_size_backward bytes (zero-filled once).
 */
moe_status moe_workspace_size_backward(const moe_config* cfg, size_t* bytes);
moe_status moe_backward(const moe_config* cfg, const void* x, const float* Wg,
                        const float* gate_bias, const void* W1, const void* W3, const void* W2,
                        const int32_t* topk_idx, const float* topk_prob, const int32_t* row_map,
                        const int32_t* expert_offsets, const void* x_perm, const void* h_mid,
                        const float* y_perm, const void* dy, void* dx, float* dWg,
                        float* dgate_bias, float* dW1, float* dW3, float* dW2, void* ws,
                        size_t ws_bytes, moe_stream_t stream);

/*
 * Backward with the shared expert (the shared path of §11 of the Megatron
 * Core page, y = routed output + SwiGLU_s(x), no gate): moe_backward's
 * gradients plus the shared expert's, dx including the shared path's
 * dx_s = [da_s | dg_s] [W1s ; W3s]^T before its one rounding.  The shared
 * expert is the routed formula for one expert of weight 1 over every token:
 * dH_s = dy W2s^T, a_s and g_s recomputed, dW2s = H_s^T dy, dW1s = x^T da_s,
 * dW3s = x^T dg_s.  bf16 or fp32 as moe_backward; fs as in moe_shared_expert.
 *   Extra inputs: W1s, W3s [h,fs], W2s [fs,h] dtype and h_mid_s [T,fs] (saved by
 *   moe_shared_expert).  Extra outputs: dW1s, dW3s [h,fs], dW2s [fs,h] fp32
 *   (overwritten).
 *   ws: moe_workspace_size_backward_shared bytes.
 */
moe_status moe_workspace_size_backward_shared(const moe_config* cfg, int32_t fs, size_t* bytes);
moe_status moe_backward_shared(const moe_config* cfg, int32_t fs, const void* x, const float* Wg,
                               const float* gate_bias, const void* W1, const void* W3,
                               const void* W2, const void* W1s, const void* W3s, const void* W2s,
                               const int32_t* topk_idx, const float* topk_prob,
                               const int32_t* row_map, const int32_t* expert_offsets,
                               const void* x_perm, const void* h_mid, const float* y_perm,
                               const void* h_mid_s, const void* dy, void* dx, float* dWg,
                               float* dgate_bias, float* dW1, float* dW3, float* dW2, float* dW1s,
                               float* dW3s, float* dW2s, void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/*
 * The shared expert's backward alone (the counterpart of moe_shared_expert):
 * its token gradient is ADDED to dx_acc [T,h] fp32 (the caller's running
 * sum), its weight gradients dW1s, dW3s [h,fs], dW2s [fs,h] fp32 overwritten.
 * Inputs as moe_backward_shared; ws: moe_workspace_size_backward_shared bytes.
 */
moe_status moe_shared_expert_backward(const moe_config* cfg, int32_t fs, const void* x,
                                      const void* W1s, const void* W3s, const void* W2s,
                                      const void* h_mid_s, const void* dy, float* dx_acc,
                                      float* dW1s, float* dW3s, float* dW2s, void* ws,
                                      size_t ws_bytes, moe_stream_t stream);

/*
 * The layer forward over a sequence of batches held in HOST memory (not a
 * step of the method: the serving loop around moe_forward).  For each batch
 * b in [0, num_batches): its input x_host + b*x_batch_stride ([T,h] dtype)
 * is copied to the device, the forward of moe_forward runs on `stream`, and
 * its output [T,h] dtype is copied to y_host + b*y_batch_stride.  A stride of
 * 0 reuses one host buffer for every batch (each batch still copies it).
 * The copies run on the library's two copy streams, double-buffered in the
 * workspace, so batch b+1's input and batch b-1's output move while batch b
 * computes.  Everything is enqueued asynchronously: the outputs are on the
 * host once `stream` is synchronised (the copy streams are joined to it).
 * Host buffers should be page-locked (cudaHostAlloc / pinned); pageable
 * memory works but the copies then serialise with the host.
 *   ws: moe_workspace_size_host bytes (moe_workspace_size + 4 staging
 *   buffers of T*h elements).  Router outputs stay in the workspace.
 * Errors as moe_forward; MOE_ERR_INVALID_ARG for num_batches < 0, a missing
 * host buffer, or 0 < y_batch_stride < T*h*elt with num_batches > 1.
 * The first call on a device creates the copy streams; make it before any
 * stream capture.
 */
moe_status moe_workspace_size_host(const moe_config* cfg, size_t* bytes);
moe_status moe_forward_host(const moe_config* cfg, int32_t num_batches, const void* x_host,
                            size_t x_batch_stride, void* y_host, size_t y_batch_stride,
                            const float* Wg, const float* gate_bias, const float* expert_bias,
                            const void* W1, const void* W3, const void* W2, void* ws,
                            size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute without a workspace argument.  This entry point is not a step
 * of the MoE method (the pages have no counterpart); it exists for callers
 * that cannot give the library any device memory beyond their inputs and
 * outputs -- a fixed memory budget reserved at start-up, a host framework
 * that forbids allocating outside its own pools, a latency-critical path
 * that must not call cudaMalloc/cudaFree (they may synchronise the device).
 * Its scratch is a fixed array of MOE_PERMUTE_NOALLOC_MAX_COUNTERS int32
 * counters (256 KB) inside the library, held by every GPU that loads the
 * library until exit.  It allocates nothing.
 *   Arguments, outputs and results are those of moe_permute.
 *   Limit: ceil(T*k/2048) * E <= MOE_PERMUTE_NOALLOC_MAX_COUNTERS, otherwise
 *   MOE_ERR_UNSUPPORTED is returned before anything is enqueued.
 *   All calls share the array: calls whose kernels overlap on the GPU race
 *   and corrupt each other; order them (one stream, or events).
 *   Every call looks the array's address up on the current device and keeps
 *   no copy, so calls stay valid after a cudaDeviceReset.  The first call on
 *   a device may load the library's device code there: make it before any
 *   stream capture.
 *   Expert ids outside [0,E) are skipped (row_map -1) without a device
 *   error report.
 */
#define MOE_PERMUTE_NOALLOC_MAX_COUNTERS 65536
moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               const uint8_t* keep, void* x_perm, int32_t* row_map,
                               int32_t* expert_offsets, moe_stream_t stream);

/*
 * moe_forward_host for the layer with a shared expert (the forward of
 * moe_forward_shared per batch) and for E4M3 experts (moe_forward_e4m3 per
 * batch): the same host-buffer contract, staging and copy pipelining.
 *   ws: moe_workspace_size_host_shared / moe_workspace_size_host_e4m3 bytes.
 */
moe_status moe_workspace_size_host_shared(const moe_config* cfg, int32_t fs, size_t* bytes);
moe_status moe_forward_host_shared(const moe_config* cfg, int32_t fs, int32_t num_batches,
                                   const void* x_host, size_t x_batch_stride, void* y_host,
                                   size_t y_batch_stride, const float* Wg, const float* gate_bias,
                                   const float* expert_bias, const void* W1, const void* W3,
                                   const void* W2, const void* W1s, const void* W3s,
                                   const void* W2s, void* ws, size_t ws_bytes,
                                   moe_stream_t stream);
moe_status moe_workspace_size_host_e4m3(const moe_config* cfg, size_t* bytes);
moe_status moe_forward_host_e4m3(const moe_config* cfg, int32_t num_batches, const void* x_host,
                                 size_t x_batch_stride, void* y_host, size_t y_batch_stride,
                                 const float* Wg, const float* gate_bias,
                                 const float* expert_bias, const uint8_t* W1q, const float* s1,
                                 const uint8_t* W3q, const float* s3, const uint8_t* W2q,
                                 const float* s2, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Reads and clears the device error word in `ws` (synchronises `stream`):
 * MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT.  *info (nullable) gets
 * the first failing index or wait site. */
moe_status moe_check(void* ws, moe_stream_t stream, int32_t* info);

/* Failure-detection self-test (not a step of the method): enqueues one
 * thread that waits, through the same bounded-wait routine the grouped GEMM
 * uses for its pipeline barriers, on a barrier that nothing ever signals.
 * After `limit_cycles` SM clock cycles (> 0) the wait gives up, MOE_ERR_TIMEOUT
 * is recorded in the error word of `ws` (at least 256 bytes, 16-byte
 * aligned) and the kernel returns normally; moe_check(ws) then reports
 * MOE_ERR_TIMEOUT and the CUDA context remains usable. */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles,
                                     moe_stream_t stream);

/* Measurement probe (not a step of the method): enqueues a kernel of pure
 * fp32 FMA chains (4 CTAs of 256 threads per SM; per thread `iters` > 0
 * rounds of 128 FMAs in 8 independent chains) and returns in *flops (host) the
 * floating-point operations it performs; the caller times it with events on
 * `stream`.  `out` is a device buffer of 4 * SM-count floats that is written
 * only if the chains produce NaN (never, for these constants).  It gives the
 * FP32 FMA-pipe rate that bounds the fp32 router GEMM. */
moe_status moe_probe_fp32_fma(int64_t iters, float* out, double* flops, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H_ */
