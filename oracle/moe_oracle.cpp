// CPU oracle for the single-GPU MoE layer forward.  TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may
// load this library.  The product path (the CUDA library and its Python
// binding) never calls it and shares no code with it.
//
// Every step is the plain definition written out in double precision over
// the exact input values (bf16 inputs are widened exactly), one loop per
// sum, summed in index order, no blocking, no fusion.  Threads only split
// independent tokens / rows.  Sources, all from the pages on the subject:
//   [MC]  "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析" (r00kie-liu.github.io)
//         §2 main path, §3 Gating, §4 TopKRouter, §5 Score function,
//         §8 Token dropping, §9 Token dispatcher, §10 Experts.
//   [DS]  "MoE Internals: DeepSpeed-Megatron Expert Parallel Implementation"
//         (duoan.github.io) §6 Inside DeepSpeed MoELayer, §8 The All-to-All path.
// Readings where the pages are silent (tie order, the capacity formula's
// body, SwiGLU, the combine order) are stated next to the code.
//
// Parity status: every function below is pinned by the CPU tests
// (tests/test_oracle_pins.py, tests/test_golden.py).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

enum { DT_F32 = 0, DT_BF16 = 1 };
enum { SCORE_SOFTMAX_POST = 0, SCORE_SOFTMAX_PRE = 1, SCORE_SIGMOID = 2, SCORE_SQRTSOFTPLUS = 3 };
enum { DROP_PROBS = 0, DROP_POSITION = 1 };

// Exact value of element i of a tensor stored as fp32 or as bf16 bits.
inline double value_at(const void* p, int dtype, int64_t i) {
  if (dtype == DT_F32) return (double)((const float*)p)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

template <class Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
  if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (n < 2 || nthreads == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  nthreads = (int)std::min<int64_t>(nthreads, n);
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w) {
    pool.emplace_back([=]() {
      for (int64_t i = w; i < n; i += nthreads) fn(i);
    });
  }
  for (auto& t : pool) t.join();
}

// Indices of the k largest values of v[0..n), largest first.  Equal values:
// the lower index comes first (the pages leave torch.topk's tie order open;
// this is the reading used everywhere in this project).
void topk_desc(const float* v, int n, int k, int32_t* out_idx) {
  std::vector<char> taken(n, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
      if (taken[e]) continue;
      if (best < 0 || v[e] > v[best]) best = e;
    }
    taken[best] = 1;
    out_idx[j] = best;
  }
}

// ------------------------------------------------------------ FP8 (E4M3)
// The 8-bit float E4M3 of the OCP 8-bit floating point specification: sign
// bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities; S.1111.111
// is NaN; largest finite value 448 = 1.75 * 2^8; smallest normal 2^-6;
// subnormals m/8 * 2^-6.  Codes 0..126 are the non-negative finite values in
// increasing order.
double e4m3_value(uint8_t c) {
  const int ex = (c >> 3) & 15, m = c & 7;
  if (ex == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double v = ex == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, ex - 7);
  return (c & 0x80) ? -v : v;
}

// The nearest finite E4M3 value to v (ties: the even code, i.e. mantissa
// bit 0 clear); magnitudes at or beyond 448 give 448 (saturation); NaN gives
// the NaN code 0x7F.
uint8_t e4m3_code(double v) {
  static const std::vector<double> table = [] {
    std::vector<double> t(127);
    for (int c = 0; c < 127; ++c) t[c] = e4m3_value((uint8_t)c);
    return t;
  }();
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(v);
  if (a >= table[126]) return sign | 126;
  const int hi = (int)(std::upper_bound(table.begin(), table.end(), a) - table.begin());
  const int lo = hi - 1;  // table[lo] <= a < table[hi]
  const double dl = a - table[lo], dh = table[hi] - a;
  const int c = dl < dh ? lo : dh < dl ? hi : ((lo & 1) ? hi : lo);
  return sign | (uint8_t)c;
}

// Power-of-two scale of a row or column whose largest magnitude is amax:
// the smallest integer e with amax * 2^-e <= 448, so that every scaled value
// is finite in E4M3.  amax below 2^-100 (zero included), infinite or NaN:
// e = 0 (such a row's scaled values are then exact fp32 products, and 2^-e
// stays an ordinary fp32 power of two for every other row).
int fp8_scale_exp(double amax) {
  if (!(amax >= std::ldexp(1.0, -100)) || !std::isfinite(amax)) return 0;
  int e = -400;
  while (std::ldexp(amax, -e) > 448.0) ++e;
  return e;
}

// The nearest bf16 value to v (ties: even), as a double.
double bf16_round(double v) {
  const float f = (float)v;
  uint32_t bits;
  std::memcpy(&bits, &f, 4);
  const uint32_t lo_bits = bits & 0xFFFF0000u, hi_bits = lo_bits + 0x10000u;
  float lo, hi;
  std::memcpy(&lo, &lo_bits, 4);
  std::memcpy(&hi, &hi_bits, 4);
  const double dl = std::fabs(v - (double)lo), dh = std::fabs((double)hi - v);
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo_bits & 0x10000u) ? hi : lo;
}

}  // namespace

extern "C" {

int oracle_abi_version(void) { return 6; }

// [MC] §3 Gating: logits = x . Wg (+ bias) with the router math in fp32.
// The oracle forms the exact sum in double over the exact fp32 values of x
// and Wg (sum over i in index order), adds the bias, and rounds once to
// fp32: "the exact value rounded once".
//   x [T,h] (x_dtype), Wg [h,E] fp32 (row i holds the E gate weights of input
//   feature i), gate_bias [E] or NULL, logits [T,E] fp32 out.
void oracle_router_logits(int64_t T, int h, int E, const void* x, int x_dtype,
                          const float* Wg, const float* gate_bias, float* logits,
                          int nthreads) {
  parallel_for(T, nthreads, [&](int64_t t) {
    std::vector<double> acc(E, 0.0);
    for (int i = 0; i < h; ++i) {
      const double xi = value_at(x, x_dtype, t * (int64_t)h + i);
      const float* wrow = Wg + (int64_t)i * E;
      for (int e = 0; e < E; ++e) acc[e] += xi * (double)wrow[e];
    }
    for (int e = 0; e < E; ++e) {
      double l = acc[e] + (gate_bias ? (double)gate_bias[e] : 0.0);
      logits[t * E + e] = (float)l;
    }
  });
}

// [MC] §5 Score function (topk_routing_with_score_function):
//  SOFTMAX_POST : scores, idx = topk(logits); probs = softmax(scores) over the k.
//  SOFTMAX_PRE  : scores = softmax(logits) over all E; probs, idx = topk(scores).
//  SIGMOID      : s = sigmoid(logits); idx = topk(s + expert_bias) (the bias
//                 only chooses); probs = s[idx] / (sum s[idx] + 1e-20).
//  SQRTSOFTPLUS : s = sqrt(softplus(logits)), softplus(l) = log(1 + e^l);
//                 choice and weights as for SIGMOID.
// Selection is done on fp32 values (the router dtype of [MC] §3); each
// score is formed in double and rounded once to fp32 before it is compared.
//
// Group-limited top-k (the page passes num_groups and group_topk to
// compute_topk but does not print its body).  Reading, the group-limited
// routing of DeepSeek-V3: the E experts form num_groups contiguous groups
// of E/num_groups; a group's score is the sum of its m = k/group_topk largest
// selection scores (in double, largest first, rounded once to fp32); the
// group_topk groups with the largest scores are kept (equal scores: lower
// group index first) and the top-k is taken over the kept groups' experts
// only.  num_groups <= 1 switches grouping off.
//
// Outputs: topk_idx [T,k] (slot order = selection score, descending),
// topk_prob [T,k] fp32, margin [T] = the smallest gap between consecutive
// selection scores among the k+1 largest of the eligible experts (so both
// the chosen set and the slot order of the k chosen are decided by it) and,
// with groups, (group_topk-th - next group score); +inf where there is no
// gap.  The margin is used by the input conditioner, not by the method.
void oracle_topk_scores(int64_t T, int E, int k, int score, int num_groups, int group_topk,
                        const float* logits, const float* expert_bias, int32_t* topk_idx,
                        float* topk_prob, float* margin, int nthreads) {
  const double inf = std::numeric_limits<double>::infinity();
  parallel_for(T, nthreads, [&](int64_t t) {
    const float* l = logits + t * E;
    std::vector<float> s(E), sel(E);
    if (score == SCORE_SOFTMAX_POST) {
      for (int e = 0; e < E; ++e) s[e] = sel[e] = l[e];
    } else if (score == SCORE_SOFTMAX_PRE) {
      double m = -inf;
      for (int e = 0; e < E; ++e) m = std::max(m, (double)l[e]);
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += std::exp((double)l[e] - m);
      for (int e = 0; e < E; ++e) s[e] = sel[e] = (float)(std::exp((double)l[e] - m) / z);
    } else {
      for (int e = 0; e < E; ++e) {
        const double x = (double)l[e];
        if (score == SCORE_SIGMOID) {
          s[e] = (float)(1.0 / (1.0 + std::exp(-x)));
        } else {
          // log(1 + e^x), written so that e^x cannot overflow
          const double softplus = std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x)));
          s[e] = (float)std::sqrt(softplus);
        }
        // scores_for_routing = scores + expert_bias, an fp32 addition
        sel[e] = expert_bias ? (float)(s[e] + expert_bias[e]) : s[e];
      }
    }
    // experts a token may choose (all, or those of the kept groups)
    std::vector<float> cand(sel);
    double group_margin = inf;
    if (num_groups > 1) {
      const int per = E / num_groups, m = k / group_topk;
      std::vector<float> gscore(num_groups);
      std::vector<int32_t> top(m);
      for (int g = 0; g < num_groups; ++g) {
        topk_desc(sel.data() + (int64_t)g * per, per, m, top.data());
        double sum = 0.0;
        for (int j = 0; j < m; ++j) sum += (double)sel[g * per + top[j]];
        gscore[g] = (float)sum;
      }
      const int gk = std::min(num_groups, group_topk + 1);
      std::vector<int32_t> gidx(gk);
      topk_desc(gscore.data(), num_groups, gk, gidx.data());
      std::vector<char> kept(num_groups, 0);
      for (int j = 0; j < group_topk; ++j) kept[gidx[j]] = 1;
      for (int e = 0; e < E; ++e)
        if (!kept[e / per]) cand[e] = -std::numeric_limits<float>::infinity();
      if (group_topk < num_groups)
        group_margin = (double)gscore[gidx[group_topk - 1]] - (double)gscore[gidx[group_topk]];
    }
    const int kk = std::min(E, k + 1);
    std::vector<int32_t> idx(kk);
    topk_desc(cand.data(), E, kk, idx.data());
    int32_t* oi = topk_idx + t * k;
    float* op = topk_prob + t * k;
    for (int j = 0; j < k; ++j) oi[j] = idx[j];
    if (margin) {
      double em = inf;
      for (int j = 0; j + 1 < kk && std::isfinite(cand[idx[j + 1]]); ++j)
        em = std::min(em, (double)cand[idx[j]] - (double)cand[idx[j + 1]]);
      margin[t] = (float)std::min(em, group_margin);
    }
    if (score == SCORE_SOFTMAX_POST) {
      double m = (double)s[idx[0]];
      double z = 0.0;
      for (int j = 0; j < k; ++j) z += std::exp((double)s[idx[j]] - m);
      for (int j = 0; j < k; ++j) op[j] = (float)(std::exp((double)s[idx[j]] - m) / z);
    } else if (score == SCORE_SOFTMAX_PRE) {
      for (int j = 0; j < k; ++j) op[j] = s[idx[j]];
    } else {
      double z = 0.0;
      for (int j = 0; j < k; ++j) z += (double)s[idx[j]];
      for (int j = 0; j < k; ++j) op[j] = (float)((double)s[idx[j]] / (z + 1e-20));
    }
  });
}

// [MC] §8 Token dropping: get_capacity(num_tokens = T*k, E, capacity_factor).
// The pages print the call but not its body; the reading used here is
// ceil((T*k / E) * capacity_factor), raised to min_capacity.  Returns -1
// (dropless) when capacity_factor <= 0.
int64_t oracle_capacity(int64_t T, int E, int k, double capacity_factor, int64_t min_capacity) {
  if (capacity_factor <= 0.0) return -1;
  double c = std::ceil(((double)T * (double)k / (double)E) * capacity_factor);
  int64_t cap = (int64_t)c;
  if (cap < min_capacity) cap = min_capacity;
  return cap;
}

// [MC] §8 apply_router_token_dropping, per expert column:
//  - capacity > T: every routed pair is kept;
//  - policy "probs": keep the `capacity` routed tokens with the largest
//    probability (equal probabilities: lower token index kept -- the pages'
//    topk(..., sorted=False) leaves this open);
//  - policy "position": keep the first `capacity` routed tokens in token
//    order (the plain reading of topk over the 0/1 routing map).
// Dropped pairs get probability 0 (final_probs = probs * final_map) and no
// renormalisation follows.  keep [T,k] u8 out; topk_prob updated in place;
// kept_per_expert [E] out.
void oracle_capacity_drop(int64_t T, int E, int k, int64_t capacity, int policy,
                          const int32_t* topk_idx, float* topk_prob, uint8_t* keep,
                          int32_t* kept_per_expert) {
  for (int64_t p = 0; p < T * k; ++p) keep[p] = 1;
  for (int e = 0; e < E; ++e) kept_per_expert[e] = 0;
  // candidate pairs per expert, in token order
  std::vector<std::vector<int64_t>> cand(E);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) cand[topk_idx[t * k + j]].push_back(t * k + j);
  for (int e = 0; e < E; ++e) {
    std::vector<int64_t>& c = cand[e];
    if (capacity >= 0 && capacity <= T && (int64_t)c.size() > capacity) {
      std::vector<int64_t> order = c;
      if (policy == DROP_PROBS) {
        std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
          return topk_prob[a] > topk_prob[b];  // stable: ties stay in token order
        });
      }
      for (size_t r = (size_t)capacity; r < order.size(); ++r) {
        keep[order[r]] = 0;
        topk_prob[order[r]] = 0.0f;
      }
    }
    int32_t n = 0;
    for (int64_t p : c) n += keep[p];
    kept_per_expert[e] = n;
  }
}

// [MC] §9 Token dispatcher (sequence-major -> expert-major) and [DS] §8
// step 4 "permute tokens into expert order".  The pages print no permute
// code; the reading: expert-major, and inside one expert ascending token
// index (a stable permutation).  offsets [E+1] = exclusive prefix of the
// kept counts; row_map [T,k] = row of pair (t,j) or -1 if dropped;
// row_token [rows] = source token of each row.  Returns the row count.
int64_t oracle_permute(int64_t T, int E, int k, const int32_t* topk_idx, const uint8_t* keep,
                       int32_t* offsets, int32_t* row_map, int32_t* row_token) {
  std::vector<int64_t> count(E, 0);
  for (int64_t p = 0; p < T * k; ++p)
    if (!keep || keep[p]) count[topk_idx[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + count[e]);
  std::vector<int64_t> cursor(E);
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int64_t p = t * k + j;
      if (keep && !keep[p]) {
        row_map[p] = -1;
        continue;
      }
      int64_t r = cursor[topk_idx[p]]++;
      row_map[p] = (int32_t)r;
      if (row_token) row_token[r] = (int32_t)t;
    }
  }
  return offsets[E];
}

// [MC] §8 apply_router_token_dropping with pad_to_capacity: final_map =
// capacity_mask, the `capacity` tokens chosen per expert column of the dense
// [T,E] probability map (capacity > T: every token).  Under capacity an expert
// has fewer routed tokens than it keeps, so its capacity_mask is its routed
// tokens plus tokens whose probability in that column is 0; the pages'
// topk(..., sorted=False) leaves open which of those equal zeros are taken,
// and the reading is the one used for every tie here: lower token index
// first.  Over capacity it is the kept set of oracle_capacity_drop.  In map
// form: start from the kept pairs (keep [T,k]) and give each expert column
// min(capacity, T) ones, adding the lowest-index tokens that are not yet
// set.  map [T,E] u8 out; padded_per_expert [E] out (the column sums).
void oracle_pad_to_capacity(int64_t T, int E, int k, int64_t capacity, const int32_t* topk_idx,
                            const uint8_t* keep, uint8_t* map, int32_t* padded_per_expert) {
  for (int64_t i = 0; i < T * E; ++i) map[i] = 0;
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j)
      if (keep[t * k + j]) map[t * E + topk_idx[t * k + j]] = 1;
  const int64_t quota = capacity > T ? T : capacity;
  for (int e = 0; e < E; ++e) {
    int64_t n = 0;
    for (int64_t t = 0; t < T; ++t) n += map[t * E + e];
    for (int64_t t = 0; t < T && n < quota; ++t) {
      if (!map[t * E + e]) {
        map[t * E + e] = 1;
        ++n;
      }
    }
    padded_per_expert[e] = (int32_t)n;
  }
}

// [MC] §9 Token dispatcher from a [T,E] routing map (the dispatcher permutes
// by the map: expert-major, ascending token index inside an expert).  Rows of
// expert e are the tokens t with map[t,e] = 1; row_map [T,k] gives the row of
// each kept pair (t,j) (its expert's column is set in the map) and -1 for the
// others; row_token [rows] the source token of each row; offsets [E+1].
// Returns the row count (the sum of the map).
int64_t oracle_permute_map(int64_t T, int E, int k, const uint8_t* map, const int32_t* topk_idx,
                           const uint8_t* keep, int32_t* offsets, int32_t* row_map,
                           int32_t* row_token) {
  std::vector<int64_t> count(E, 0);
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) count[e] += map[t * E + e];
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + count[e]);
  std::vector<int64_t> cursor(E);
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  std::vector<int64_t> row_of((size_t)(T * E), -1);
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e)
      if (map[t * E + e]) {
        const int64_t r = cursor[e]++;
        row_of[(size_t)(t * E + e)] = r;
        if (row_token) row_token[r] = (int32_t)t;
      }
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int64_t p = t * k + j;
      row_map[p] = keep[p] ? (int32_t)row_of[(size_t)(t * E + topk_idx[p])] : -1;
    }
  return offsets[E];
}

// [MC] §10 Experts (grouped expert MLP), one row at a time.  The expert MLP
// is SwiGLU (the pages name the grouped MLP but not its activation):
//   a = x.W1[e], g = x.W3[e], H = silu(a) * g with silu(a) = a / (1 + exp(-a)),
//   Y = H.W2[e]
// with W1/W3 [E,h,f] (row i = input feature i) and W2 [E,f,h].  Sums in
// double over the exact inputs; H is kept in double (not rounded).
//   rows: x_rows [R,h] (x_dtype) are the inputs; row_expert [R] their experts;
//   h_mid [R,f] (double, may be NULL) and y_rows [R,h] (double) out.
void oracle_expert_rows(int64_t R, int h, int f, const void* x_rows, int x_dtype,
                        const int32_t* row_expert, const void* W1, const void* W3,
                        const void* W2, int w_dtype, double* h_mid, double* y_rows,
                        int nthreads) {
  parallel_for(R, nthreads, [&](int64_t r) {
    const int64_t e = row_expert[r];
    std::vector<double> xv(h), a(f, 0.0), g(f, 0.0), H(f), y(h, 0.0);
    for (int i = 0; i < h; ++i) xv[i] = value_at(x_rows, x_dtype, r * (int64_t)h + i);
    const int64_t w13 = e * (int64_t)h * f;
    for (int i = 0; i < h; ++i) {
      const double xi = xv[i];
      const int64_t base = w13 + (int64_t)i * f;
      for (int c = 0; c < f; ++c) {
        a[c] += xi * value_at(W1, w_dtype, base + c);
        g[c] += xi * value_at(W3, w_dtype, base + c);
      }
    }
    for (int c = 0; c < f; ++c) H[c] = a[c] / (1.0 + std::exp(-a[c])) * g[c];
    const int64_t w2 = e * (int64_t)f * h;
    for (int c = 0; c < f; ++c) {
      const double hc = H[c];
      const int64_t base = w2 + (int64_t)c * h;
      for (int n = 0; n < h; ++n) y[n] += hc * value_at(W2, w_dtype, base + n);
    }
    if (h_mid)
      for (int c = 0; c < f; ++c) h_mid[r * (int64_t)f + c] = H[c];
    for (int n = 0; n < h; ++n) y_rows[r * (int64_t)h + n] = y[n];
  });
}

// [MC] §2 combine / [DS] §8 step 8 "unpermute and combine outputs with gate
// weights": y[t] = sum over kept slots j (in slot order) of
// topk_prob[t,j] * y_perm[row_map[t,j]], in double.  A token whose pairs
// were all dropped gets 0.  y_perm [rows,h] double, y [T,h] double out.
void oracle_combine(int64_t T, int k, int h, const double* y_perm, const int32_t* row_map,
                    const float* topk_prob, double* y, int nthreads) {
  parallel_for(T, nthreads, [&](int64_t t) {
    double* out = y + t * (int64_t)h;
    for (int n = 0; n < h; ++n) out[n] = 0.0;
    for (int j = 0; j < k; ++j) {
      int32_t r = row_map[t * k + j];
      if (r < 0) continue;
      const double p = (double)topk_prob[t * k + j];
      const double* src = y_perm + (int64_t)r * h;
      for (int n = 0; n < h; ++n) out[n] += p * src[n];
    }
  });
}

// A second, independent route to the layer output, for validating the
// oracle on tiny inputs only: every expert is evaluated on every token (no
// permutation, no row bookkeeping) and weighted by the token's kept
// probability for that expert (0 if the expert was not selected or the
// pair was dropped).  y [T,h] double out.
void oracle_forward_dense(int64_t T, int h, int E, int k, int f, const void* x, int x_dtype,
                          const int32_t* topk_idx, const float* topk_prob, const uint8_t* keep,
                          const void* W1, const void* W3, const void* W2, int w_dtype, double* y,
                          int nthreads) {
  parallel_for(T, nthreads, [&](int64_t t) {
    std::vector<double> out(h, 0.0), yrow(h);
    for (int e = 0; e < E; ++e) {
      double w = 0.0;
      for (int j = 0; j < k; ++j)
        if (topk_idx[t * k + j] == e && (!keep || keep[t * k + j])) w = (double)topk_prob[t * k + j];
      // evaluate expert e on token t regardless of w
      int32_t ee = e;
      std::vector<uint8_t> xrow(h * (x_dtype == DT_F32 ? 4 : 2));
      std::memcpy(xrow.data(), (const uint8_t*)x + t * (int64_t)h * (x_dtype == DT_F32 ? 4 : 2),
                  xrow.size());
      oracle_expert_rows(1, h, f, xrow.data(), x_dtype, &ee, W1, W3, W2, w_dtype, nullptr,
                         yrow.data(), 1);
      for (int n = 0; n < h; ++n) out[n] += w * yrow[n];
    }
    for (int n = 0; n < h; ++n) y[t * (int64_t)h + n] = out[n];
  });
}

// ------------------------------------------------------------ FP8 experts
// FP8 variant of the grouped expert MLP ([MC] §10 experts; the Megatron Core
// report names FP8 GEMMs as its most effective single optimisation but
// prints no scaling recipe).  Reading used here: E4M3 values with one
// power-of-two scale per token row of the activations and one per output
// channel of every weight matrix (the scale of fp8_scale_exp), fp32-exact
// dequantisation value = code value * 2^e.

// Row quantisation: x [rows, cols] (x_dtype) -> codes [rows, cols] and
// scales [rows] (= 2^e of each row's largest magnitude).
void oracle_quantize_rows_e4m3(int64_t rows, int cols, const void* x, int x_dtype,
                               uint8_t* codes, float* scales, int nthreads) {
  parallel_for(rows, nthreads, [&](int64_t r) {
    double amax = 0.0;
    for (int c = 0; c < cols; ++c)
      amax = std::max(amax, std::fabs(value_at(x, x_dtype, r * (int64_t)cols + c)));
    const int e = fp8_scale_exp(amax);
    scales[r] = (float)std::ldexp(1.0, e);
    for (int c = 0; c < cols; ++c)
      codes[r * (int64_t)cols + c] =
          e4m3_code(std::ldexp(value_at(x, x_dtype, r * (int64_t)cols + c), -e));
  });
}

// Weight quantisation per output channel: W [E][K][N] (w_dtype) -> codes
// [E][N][K] (K contiguous: each output channel's weights in a row) and
// scales [E][N] (2^e of the channel's largest magnitude over K).
void oracle_quantize_cols_e4m3(int64_t E, int K, int N, const void* W, int w_dtype,
                               uint8_t* codes, float* scales, int nthreads) {
  parallel_for(E * N, nthreads, [&](int64_t en) {
    const int64_t e = en / N, n = en % N;
    const int64_t base = e * (int64_t)K * N + n;
    double amax = 0.0;
    for (int k = 0; k < K; ++k) amax = std::max(amax, std::fabs(value_at(W, w_dtype, base + (int64_t)k * N)));
    const int ex = fp8_scale_exp(amax);
    scales[en] = (float)std::ldexp(1.0, ex);
    for (int k = 0; k < K; ++k)
      codes[en * (int64_t)K + k] = e4m3_code(std::ldexp(value_at(W, w_dtype, base + (int64_t)k * N), -ex));
  });
}

// SwiGLU expert rows on FP8 operands:
//   a = (sum_i x(i) w1(c,i)) * sx * s1(c),  g likewise with W3,
//   H = silu(a) * g, rounded to bf16 (the stored intermediate), then
//   quantised per row (hq, hs) and
//   y(n) = (sum_c h(c) w2(n,c)) * hs * s2(n)
// where x(i), w(c,i), h(c) are E4M3 code values; sums in double.
//   xq [R,h] codes, xs [R]; W1q/W3q [E,f,h] codes, s1/s3 [E,f];
//   W2q [E,h,f] codes, s2 [E,h]; h_mid [R,f] (bf16 values, may be NULL),
//   hq [R,f] codes and hs [R] (may be NULL), y_rows [R,h] out.
void oracle_expert_rows_fp8(int64_t R, int h, int f, const uint8_t* xq, const float* xs,
                            const int32_t* row_expert, const uint8_t* W1q, const float* s1,
                            const uint8_t* W3q, const float* s3, const uint8_t* W2q,
                            const float* s2, double* h_mid, uint8_t* hq, float* hs,
                            double* y_rows, int nthreads) {
  parallel_for(R, nthreads, [&](int64_t r) {
    const int64_t e = row_expert[r];
    std::vector<double> xv(h), H(f);
    for (int i = 0; i < h; ++i) xv[i] = e4m3_value(xq[r * (int64_t)h + i]);
    double amax = 0.0;
    for (int c = 0; c < f; ++c) {
      const uint8_t* w1 = W1q + (e * f + c) * (int64_t)h;
      const uint8_t* w3 = W3q + (e * f + c) * (int64_t)h;
      double a = 0.0, g = 0.0;
      for (int i = 0; i < h; ++i) {
        a += xv[i] * e4m3_value(w1[i]);
        g += xv[i] * e4m3_value(w3[i]);
      }
      a *= (double)xs[r] * (double)s1[e * f + c];
      g *= (double)xs[r] * (double)s3[e * f + c];
      H[c] = bf16_round(a / (1.0 + std::exp(-a)) * g);
      amax = std::max(amax, std::fabs(H[c]));
    }
    const int ex = fp8_scale_exp(amax);
    const double scale = std::ldexp(1.0, ex);
    std::vector<double> hv(f);
    for (int c = 0; c < f; ++c) {
      const uint8_t code = e4m3_code(std::ldexp(H[c], -ex));
      hv[c] = e4m3_value(code);
      if (hq) hq[r * (int64_t)f + c] = code;
      if (h_mid) h_mid[r * (int64_t)f + c] = H[c];
    }
    if (hs) hs[r] = (float)scale;
    for (int n = 0; n < h; ++n) {
      const uint8_t* w2 = W2q + (e * h + n) * (int64_t)f;
      double y = 0.0;
      for (int c = 0; c < f; ++c) y += hv[c] * e4m3_value(w2[c]);
      y_rows[r * (int64_t)h + n] = y * scale * (double)s2[e * h + n];
    }
  });
}

// ------------------------------------------------------------ backward
// Gradient of L = sum(dy * y) through the layer for fixed routing decisions
// (top-k choice, capacity drop): the training-side counterpart of the
// forward above, derived by the chain rule from the same definitions.
// y weights each expert output by the forward's fp32 combine weight
// (topk_prob, an input as a training step saves it), so dY uses that value;
// the derivatives of the scores are taken in double.
// Discrete decisions carry no gradient; the expert bias only chooses and
// gets none.  Per kept pair (t,j) of expert e with weight p:
//   dY = p dy[t],  dp = <dy[t], Y>,  dH = dY . W2[e]^T,
//   da = dH * g * silu'(a),  dg = dH * silu(a)   (silu'(a) = s (1 + a (1 - s)), s = sigmoid(a)),
//   dx[t] += da . W1[e]^T + dg . W3[e]^T,
//   dW2[e] += H^T dY,  dW1[e] += x^T da,  dW3[e] += x^T dg,
// and through the router: dlogits from dp by the score function's
// derivative (only the k chosen experts carry a weight; dropped pairs have
// dp = 0 but stay in the renormalisation), then
//   dWg = x^T dlogits,  dgate_bias = sum_t dlogits,  dx[t] += dlogits[t] . Wg^T.
// All sums in double over the exact inputs.  Outputs: dx [T,h], dWg [h,E],
// dgb [E], dW1/dW3 [E,h,f], dW2 [E,f,h] (all three may be NULL: not formed),
// dlogits [T,E] (may be NULL).
void oracle_backward(int64_t T, int h, int E, int k, int f, int score, const void* x,
                     int x_dtype, const float* Wg, const float* gate_bias,
                     const float* expert_bias, const void* W1, const void* W3, const void* W2,
                     int w_dtype, const int32_t* topk_idx, const float* topk_prob,
                     const uint8_t* keep, const void* dy,
                     int dy_dtype, double* dx, double* dWg, double* dgb, double* dW1, double* dW3,
                     double* dW2, double* dlogits_out, int nthreads) {
  // logits, as the forward forms them (exact sum rounded once to fp32)
  std::vector<float> logits((size_t)T * E);
  oracle_router_logits(T, h, E, x, x_dtype, Wg, gate_bias, logits.data(), nthreads);
  std::vector<double> dl((size_t)T * E, 0.0);
  // per kept pair: da, dg ([f]) and dY ([h]) for the weight gradients
  std::vector<double> pda((size_t)T * k * f, 0.0), pdg((size_t)T * k * f, 0.0);
  std::vector<double> pH((size_t)T * k * f, 0.0), pdY((size_t)T * k * h, 0.0);
  parallel_for(T, nthreads, [&](int64_t t) {
    const float* l = logits.data() + t * E;
    std::vector<double> s(E), xv(h), dyv(h), dxt(h, 0.0);
    for (int i = 0; i < h; ++i) {
      xv[i] = value_at(x, x_dtype, t * (int64_t)h + i);
      dyv[i] = value_at(dy, dy_dtype, t * (int64_t)h + i);
    }
    // scores s (double) and the chosen-expert weights p_j (before the drop)
    for (int e = 0; e < E; ++e) {
      const double z = (double)l[e];
      if (score == SCORE_SIGMOID) s[e] = 1.0 / (1.0 + std::exp(-z));
      else if (score == SCORE_SQRTSOFTPLUS) s[e] = std::sqrt(std::max(z, 0.0) + std::log1p(std::exp(-std::fabs(z))));
      else s[e] = z;
    }
    if (score == SCORE_SOFTMAX_PRE) {
      double m = -std::numeric_limits<double>::infinity(), zsum = 0.0;
      for (int e = 0; e < E; ++e) m = std::max(m, s[e]);
      for (int e = 0; e < E; ++e) zsum += std::exp(s[e] - m);
      for (int e = 0; e < E; ++e) s[e] = std::exp(s[e] - m) / zsum;
    }
    std::vector<double> p(k), dp(k, 0.0);
    const int32_t* idx = topk_idx + t * k;
    if (score == SCORE_SOFTMAX_POST) {
      double m = s[idx[0]], zsum = 0.0;
      for (int j = 0; j < k; ++j) m = std::max(m, s[idx[j]]);
      for (int j = 0; j < k; ++j) zsum += std::exp(s[idx[j]] - m);
      for (int j = 0; j < k; ++j) p[j] = std::exp(s[idx[j]] - m) / zsum;
    } else if (score == SCORE_SOFTMAX_PRE) {
      for (int j = 0; j < k; ++j) p[j] = s[idx[j]];
    } else {
      double zsum = 0.0;
      for (int j = 0; j < k; ++j) zsum += s[idx[j]];
      for (int j = 0; j < k; ++j) p[j] = s[idx[j]] / (zsum + 1e-20);
    }
    // experts of the kept pairs
    for (int j = 0; j < k; ++j) {
      if (keep && !keep[t * k + j]) continue;
      const int64_t e = idx[j], pr = t * k + j;
      std::vector<double> a(f, 0.0), g(f, 0.0), H(f), Y(h, 0.0);
      for (int i = 0; i < h; ++i) {
        const int64_t base = (e * h + i) * (int64_t)f;
        for (int c = 0; c < f; ++c) {
          a[c] += xv[i] * value_at(W1, w_dtype, base + c);
          g[c] += xv[i] * value_at(W3, w_dtype, base + c);
        }
      }
      for (int c = 0; c < f; ++c) H[c] = a[c] / (1.0 + std::exp(-a[c])) * g[c];
      for (int c = 0; c < f; ++c) {
        const int64_t base = (e * f + c) * (int64_t)h;
        for (int n = 0; n < h; ++n) Y[n] += H[c] * value_at(W2, w_dtype, base + n);
      }
      double dot = 0.0;
      for (int n = 0; n < h; ++n) dot += dyv[n] * Y[n];
      dp[j] = dot;
      // y weights Y by the forward's fp32 combine weight, so that is dY's factor
      const double pf = (double)topk_prob[pr];
      double* dYp = &pdY[pr * h];
      for (int n = 0; n < h; ++n) dYp[n] = pf * dyv[n];
      for (int c = 0; c < f; ++c) {
        const int64_t base = (e * f + c) * (int64_t)h;
        double dH = 0.0;
        for (int n = 0; n < h; ++n) dH += dYp[n] * value_at(W2, w_dtype, base + n);
        const double sg = 1.0 / (1.0 + std::exp(-a[c]));
        pda[pr * f + c] = dH * g[c] * sg * (1.0 + a[c] * (1.0 - sg));
        pdg[pr * f + c] = dH * a[c] * sg;
        pH[pr * f + c] = H[c];
      }
      for (int i = 0; i < h; ++i) {
        const int64_t base = (e * h + i) * (int64_t)f;
        double acc = 0.0;
        for (int c = 0; c < f; ++c)
          acc += pda[pr * f + c] * value_at(W1, w_dtype, base + c) +
                 pdg[pr * f + c] * value_at(W3, w_dtype, base + c);
        dxt[i] += acc;
      }
    }
    // router: dlogits from dp through the score function
    double* dlt = &dl[t * E];
    if (score == SCORE_SOFTMAX_POST) {
      double sdp = 0.0;
      for (int j = 0; j < k; ++j) sdp += p[j] * dp[j];
      for (int j = 0; j < k; ++j) dlt[idx[j]] += p[j] * (dp[j] - sdp);
    } else if (score == SCORE_SOFTMAX_PRE) {
      std::vector<double> ds(E, 0.0);
      for (int j = 0; j < k; ++j) ds[idx[j]] += dp[j];
      double sds = 0.0;
      for (int e = 0; e < E; ++e) sds += s[e] * ds[e];
      for (int e = 0; e < E; ++e) dlt[e] = s[e] * (ds[e] - sds);
    } else {
      double zsum = 0.0, spd = 0.0;
      for (int j = 0; j < k; ++j) zsum += s[idx[j]];
      const double Z = zsum + 1e-20;
      for (int j = 0; j < k; ++j) spd += dp[j] * s[idx[j]];
      for (int j = 0; j < k; ++j) {
        const int e = idx[j];
        const double ds = dp[j] / Z - spd / (Z * Z);
        const double z = (double)l[e];
        const double deriv = score == SCORE_SIGMOID ? s[e] * (1.0 - s[e])
                                                    : (1.0 / (1.0 + std::exp(-z))) / (2.0 * s[e]);
        dlt[e] += ds * deriv;
      }
    }
    (void)expert_bias;  // choice only: no gradient
    for (int i = 0; i < h; ++i) {
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += dlt[e] * (double)Wg[(int64_t)i * E + e];
      dx[t * (int64_t)h + i] = dxt[i] + acc;
    }
  });
  // router weight and bias gradients
  parallel_for(h, nthreads, [&](int64_t i) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += value_at(x, x_dtype, t * (int64_t)h + i) * dl[t * E + e];
      dWg[i * E + e] = acc;
    }
  });
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int64_t t = 0; t < T; ++t) acc += dl[t * E + e];
    dgb[e] = acc;
  }
  // expert weight gradients, per expert (pairs in token order)
  if (dW1 && dW3 && dW2) parallel_for(E, nthreads, [&](int64_t e) {
    for (int64_t i = 0; i < (int64_t)h * f; ++i) dW1[e * (int64_t)h * f + i] = dW3[e * (int64_t)h * f + i] = 0.0;
    for (int64_t i = 0; i < (int64_t)f * h; ++i) dW2[e * (int64_t)f * h + i] = 0.0;
    for (int64_t t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        if (topk_idx[t * k + j] != e || (keep && !keep[t * k + j])) continue;
        const int64_t pr = t * k + j;
        for (int i = 0; i < h; ++i) {
          const double xi = value_at(x, x_dtype, t * (int64_t)h + i);
          double* w1 = dW1 + (e * h + i) * (int64_t)f;
          double* w3 = dW3 + (e * h + i) * (int64_t)f;
          for (int c = 0; c < f; ++c) {
            w1[c] += xi * pda[pr * f + c];
            w3[c] += xi * pdg[pr * f + c];
          }
        }
        for (int c = 0; c < f; ++c) {
          double* w2 = dW2 + (e * f + c) * (int64_t)h;
          const double Hc = pH[pr * f + c];
          for (int n = 0; n < h; ++n) w2[n] += Hc * pdY[pr * h + n];
        }
      }
  });
  if (dlogits_out)
    for (size_t i = 0; i < dl.size(); ++i) dlogits_out[i] = dl[i];
}

// Selected weight gradients of one expert, for checks at sizes where the
// whole backward is out of reach: the expert's R rows are x_rows [R,h] with
// combine weights p [R] and output gradients dy_rows [R,h] (the rows of dy
// of the tokens behind them); W1e, W3e [h,f] and W2e [f,h] are its weights.
// With the definitions of oracle_backward (dY = p dy, a = x.W1, g = x.W3,
// H = silu(a) g, dH = dY.W2^T, da = dH g silu'(a), dg = dH silu(a)):
//   for each c of rows_c (n2 of them):  dW2_rows[q,:] = sum_r H[r,c] dY[r,:]
//   for each c of cols_c (n13):         dW1_cols[:,q] = sum_r x[r,:] da[r,c]
//                                       dW3_cols[:,q] = sum_r x[r,:] dg[r,c]
// Only column c of a, g, H, dH is needed for index c.  All sums in double.
void oracle_expert_wgrad_cols(int64_t R, int h, int f, const void* x_rows, int x_dtype,
                              const float* p, const void* dy_rows, int dy_dtype, const void* W1e,
                              const void* W3e, const void* W2e, int w_dtype, int n2,
                              const int32_t* rows_c, int n13, const int32_t* cols_c,
                              double* dW2_rows, double* dW1_cols, double* dW3_cols,
                              int nthreads) {
  parallel_for(n2 + n13, nthreads, [&](int64_t q) {
    const bool second = q < n2;
    const int64_t c = second ? rows_c[q] : cols_c[q - n2];
    std::vector<double> acc1(h, 0.0), acc3(h, 0.0);
    for (int64_t r = 0; r < R; ++r) {
      double a = 0.0, g = 0.0;
      for (int i = 0; i < h; ++i) {
        const double xi = value_at(x_rows, x_dtype, r * h + i);
        a += xi * value_at(W1e, w_dtype, (int64_t)i * f + c);
        g += xi * value_at(W3e, w_dtype, (int64_t)i * f + c);
      }
      const double sg = 1.0 / (1.0 + std::exp(-a));
      const double pr = (double)p[r];
      if (second) {
        const double H = a * sg * g;
        for (int n = 0; n < h; ++n) acc1[n] += H * pr * value_at(dy_rows, dy_dtype, r * h + n);
      } else {
        double dH = 0.0;
        for (int n = 0; n < h; ++n)
          dH += pr * value_at(dy_rows, dy_dtype, r * h + n) * value_at(W2e, w_dtype, c * h + n);
        const double da = dH * g * sg * (1.0 + a * (1.0 - sg));
        const double dg = dH * a * sg;
        for (int i = 0; i < h; ++i) {
          const double xi = value_at(x_rows, x_dtype, r * h + i);
          acc1[i] += xi * da;
          acc3[i] += xi * dg;
        }
      }
    }
    if (second) {
      for (int n = 0; n < h; ++n) dW2_rows[q * h + n] = acc1[n];
    } else {
      const int64_t qq = q - n2;
      for (int i = 0; i < h; ++i) {
        dW1_cols[(int64_t)i * n13 + qq] = acc1[i];
        dW3_cols[(int64_t)i * n13 + qq] = acc3[i];
      }
    }
  });
}

// The E4M3 value of every code 0..255 (for the pins).
void oracle_e4m3_values(double* out) {
  for (int c = 0; c < 256; ++c) out[c] = e4m3_value((uint8_t)c);
}
// E4M3 codes of n doubles (for the pins).
void oracle_e4m3_codes(int64_t n, const double* v, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(v[i]);
}

}  // extern "C"
