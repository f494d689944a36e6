"""Pins of the CPU oracle against facts other than itself: exact integer
cases, closed forms, special cases that reduce to library routines (scipy's
expit/softmax, numpy matmul on one-hot inputs), brute force over all k-subsets,
and invariants (probabilities sum to 1, kept counts = min(assigned, cap),
permutation round trip, dense vs permuted evaluation).  CPU only.
"""

import itertools

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- router --

def test_logits_one_hot_pick_rows_of_Wg():
    # x = e_i selects row i of Wg [h,E]; a transposed Wg would pick a column.
    h, E = 6, 4
    Wg = rng(1).standard_normal((h, E)).astype(np.float32)
    x = np.eye(h, dtype=np.float32)
    np.testing.assert_array_equal(oracle.router_logits(x, Wg), Wg)


def test_logits_integer_exact():
    # small integers: every partial sum is exact, so the result is the exact
    # integer matmul.
    r = rng(2)
    x = r.integers(-4, 5, (9, 33)).astype(np.float32)
    Wg = r.integers(-3, 4, (33, 5)).astype(np.float32)
    b = r.integers(-2, 3, (5,)).astype(np.float32)
    want = (x.astype(np.int64) @ Wg.astype(np.int64) + b.astype(np.int64)).astype(np.float32)
    np.testing.assert_array_equal(oracle.router_logits(x, Wg, b), want)


def test_logits_bias_only():
    b = np.array([0.5, -1.25, 3.0], np.float32)
    x = np.zeros((2, 4), np.float32)
    Wg = rng(3).standard_normal((4, 3)).astype(np.float32)
    np.testing.assert_array_equal(oracle.router_logits(x, Wg, b), np.stack([b, b]))


def test_logits_bf16_widening_matches_f32():
    import torch
    xf = rng(4).standard_normal((5, 16)).astype(np.float32)
    xb = torch.from_numpy(xf).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    widened = xb.to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.bf16_bits_to_f32(bits), widened)
    Wg = rng(5).standard_normal((16, 4)).astype(np.float32)
    np.testing.assert_array_equal(oracle.router_logits(bits, Wg), oracle.router_logits(widened, Wg))


def _brute_topk_set(sel, k):
    """The k-subset with the largest sum of selection scores (all subsets)."""
    best, best_sum = None, -np.inf
    for S in itertools.combinations(range(sel.size), k):
        s = float(np.sum(sel[list(S)].astype(np.float64)))
        if s > best_sum:
            best, best_sum = set(S), s
    return best


@pytest.mark.parametrize("score", ["softmax_post", "softmax_pre", "sigmoid"])
@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_brute_force(score, k):
    E, T = 6, 40
    logits = rng(10 + k).standard_normal((T, E)).astype(np.float32)
    eb = rng(20).uniform(-0.1, 0.1, E).astype(np.float32) if score == "sigmoid" else None
    idx, prob, margin = oracle.topk_scores(logits, k, score, eb)
    for t in range(T):
        l = logits[t].astype(np.float64)
        if score == "softmax_post":
            sel = l
        elif score == "softmax_pre":
            sel = softmax(l)
        else:
            sel = expit(l) + eb
        assert set(idx[t].tolist()) == _brute_topk_set(sel, k)
        # slots ordered by selection score, descending
        assert np.all(np.diff(sel[idx[t]]) <= 0)


def test_post_softmax_probs_sum_to_one_and_logistic_closed_form():
    logits = rng(30).standard_normal((200, 8)).astype(np.float32) * 3
    idx, prob, _ = oracle.topk_scores(logits, 2, "softmax_post")
    assert np.all(np.abs(prob.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    l0 = np.take_along_axis(logits, idx[:, :1], 1)[:, 0].astype(np.float64)
    l1 = np.take_along_axis(logits, idx[:, 1:2], 1)[:, 0].astype(np.float64)
    # two-way softmax is the logistic function of the logit gap
    np.testing.assert_allclose(prob[:, 0], expit(l0 - l1), rtol=1e-6)


def test_post_softmax_top1_is_exactly_one():
    logits = rng(31).standard_normal((50, 16)).astype(np.float32)
    _, prob, _ = oracle.topk_scores(logits, 1, "softmax_post")
    assert np.all(prob == 1.0)


def test_pre_softmax_matches_scipy_and_full_k_sums_to_one():
    logits = rng(32).standard_normal((64, 8)).astype(np.float32) * 2
    idx, prob, _ = oracle.topk_scores(logits, 8, "softmax_pre")
    want = softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(prob, np.take_along_axis(want, idx, 1), rtol=1e-6)
    assert np.all(np.abs(prob.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    idx2, prob2, _ = oracle.topk_scores(logits, 2, "softmax_pre")
    np.testing.assert_allclose(prob2, np.take_along_axis(want, idx2, 1), rtol=1e-6)


def test_sigmoid_without_bias_selects_top_logits():
    logits = rng(33).standard_normal((100, 16)).astype(np.float32)
    idx, prob, _ = oracle.topk_scores(logits, 4, "sigmoid")
    want_idx = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :4]
    np.testing.assert_array_equal(idx, want_idx)
    s = expit(np.take_along_axis(logits, idx, 1).astype(np.float64))
    np.testing.assert_allclose(prob, s / s.sum(1, keepdims=True), rtol=1e-6)
    assert np.all(np.abs(prob.astype(np.float64).sum(1) - 1.0) <= 1e-6)


def test_sigmoid_bias_only_chooses():
    # a large bias forces experts 3 and 5; their weights stay sigmoid(logit)
    logits = rng(34).standard_normal((30, 8)).astype(np.float32)
    eb = np.zeros(8, np.float32)
    eb[[3, 5]] = 10.0
    idx, prob, _ = oracle.topk_scores(logits, 2, "sigmoid", eb)
    assert all(set(r) == {3, 5} for r in idx.tolist())
    s = expit(np.take_along_axis(logits, idx, 1).astype(np.float64))
    np.testing.assert_allclose(prob, s / s.sum(1, keepdims=True), rtol=1e-6)


def test_ties_take_lower_expert_index():
    logits = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]], np.float32)
    idx, _, margin = oracle.topk_scores(logits, 2, "softmax_post")
    assert idx.tolist() == [[1, 2]]
    assert margin[0] == 0.0


def test_margin_is_smallest_gap_among_top_k_plus_one():
    # the set of k experts and their slot order are both decided by the margin
    logits = rng(35).standard_normal((20, 8)).astype(np.float32)
    _, _, margin = oracle.topk_scores(logits, 3, "softmax_post")
    srt = -np.sort(-logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(margin, np.diff(-srt[:, :4], axis=1).min(axis=1), rtol=1e-6)
    _, _, m_all = oracle.topk_scores(logits, 8, "softmax_post")  # k = E: the order of all 8
    np.testing.assert_allclose(m_all, np.diff(-srt, axis=1).min(axis=1), rtol=1e-6)
    _, _, m_one = oracle.topk_scores(logits[:, :1], 1, "softmax_post")  # one expert: no gap
    assert np.all(np.isinf(m_one))


# --------------------------------------------------------------- capacity --

def _random_routing(seed, T, E, k):
    r = rng(seed)
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    prob = r.uniform(0.01, 1.0, (T, k)).astype(np.float32)
    return idx, prob


@pytest.mark.parametrize("policy", ["probs", "position"])
@pytest.mark.parametrize("cap", [0, 1, 3, 7, 40])
def test_drop_counts_and_kept_set(policy, cap):
    T, E, k = 40, 5, 2
    idx, prob = _random_routing(40 + cap, T, E, k)
    prob_out, keep, kept = oracle.capacity_drop(idx, prob, E, cap, policy)
    assigned = np.bincount(idx.reshape(-1), minlength=E)
    np.testing.assert_array_equal(kept, np.minimum(assigned, cap))
    # dropped pairs get 0, kept pairs keep their probability (no renormalisation)
    np.testing.assert_array_equal(prob_out, np.where(keep == 1, prob, 0.0).astype(np.float32))
    for e in range(E):
        pairs = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        for (t, j) in pairs:
            if policy == "probs":
                better = sum(1 for (u, i) in pairs
                             if prob[u, i] > prob[t, j] or (prob[u, i] == prob[t, j] and u < t))
            else:
                better = sum(1 for (u, i) in pairs if u < t)
            assert keep[t, j] == (1 if better < cap else 0)


def test_capacity_above_T_keeps_everything():
    idx, prob = _random_routing(50, 12, 3, 2)
    cap = oracle.capacity(12, 3, 2, 100.0)
    assert cap > 12
    prob_out, keep, kept = oracle.capacity_drop(idx, prob, 3, cap, "probs")
    assert keep.all()
    np.testing.assert_array_equal(prob_out, prob)


def test_route_with_capacity_end_to_end():
    # skewed gate bias so that drops happen
    r = rng(51)
    T, h, E, k = 300, 16, 6, 1
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = (0.3 * r.standard_normal((h, E))).astype(np.float32)
    gb = np.array([2.0, 0, 0, 0, 0, 0], np.float32)
    out = oracle.route(x, Wg, k, "softmax_pre", gate_bias=gb, capacity_factor=1.0)
    assert out["capacity"] == 50
    assert out["assigned"][0] > 50
    np.testing.assert_array_equal(out["tokens_per_expert"], np.minimum(out["assigned"], 50))


# ---------------------------------------------------------------- permute --

@pytest.mark.parametrize("seed", [60, 61, 62])
def test_permute_invariants(seed):
    T, E, k = 57, 7, 3
    idx, prob = _random_routing(seed, T, E, k)
    keep = (rng(seed + 100).uniform(size=(T, k)) > 0.2).astype(np.uint8)
    offsets, row_map, row_token = oracle.permute(idx, keep, E)
    counts = np.array([int(((idx == e) & (keep == 1)).sum()) for e in range(E)])
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    R = offsets[-1]
    rows = row_map[keep == 1]
    assert sorted(rows.tolist()) == list(range(R))            # bijection onto [0,R)
    assert np.all(row_map[keep == 0] == -1)
    for t in range(T):
        for j in range(k):
            if keep[t, j]:
                r_ = row_map[t, j]
                assert row_token[r_] == t
                assert offsets[idx[t, j]] <= r_ < offsets[idx[t, j] + 1]
    for e in range(E):                                         # stable inside a segment
        assert np.all(np.diff(row_token[offsets[e]:offsets[e + 1]]) > 0)


def test_permute_combine_round_trip_identity_experts():
    # identity experts: feeding x_perm straight into combine gives x * sum(kept p)
    T, h, E, k = 33, 12, 5, 2
    x = rng(70).standard_normal((T, h)).astype(np.float32)
    idx, prob = _random_routing(71, T, E, k)
    prob, keep, _ = oracle.capacity_drop(idx, prob, E, 9, "probs")
    offsets, row_map, row_token = oracle.permute(idx, keep, E)
    x_perm = x[row_token].astype(np.float64)
    y = oracle.combine(x_perm, row_map, prob)
    want = x.astype(np.float64) * prob.astype(np.float64).sum(1, keepdims=True)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_combine_closed_form_constant_rows():
    T, k, h = 4, 2, 3
    row_map = np.array([[0, 3], [1, -1], [-1, -1], [2, 4]], np.int32)
    prob = np.array([[0.5, 0.25], [1.0, 0.0], [0.0, 0.0], [0.125, 2.0]], np.float32)
    y_perm = np.repeat(np.array([[1.0], [2.0], [4.0], [8.0], [16.0]]), h, axis=1)
    y = oracle.combine(y_perm, row_map, prob)
    want = np.array([0.5 * 1 + 0.25 * 8, 1.0 * 2, 0.0, 0.125 * 4 + 2.0 * 16])
    np.testing.assert_array_equal(y, np.repeat(want[:, None], h, axis=1))


# ---------------------------------------------------------------- experts --

def _weights(seed, E, h, f, scale=0.3):
    r = rng(seed)
    return tuple((scale * r.standard_normal(s)).astype(np.float32)
                 for s in ((E, h, f), (E, h, f), (E, f, h)))


def test_expert_one_hot_closed_form():
    # x = e_i: a = W1[e][i,:], g = W3[e][i,:] and y = (silu(a) * g) . W2[e]
    E, h, f = 3, 5, 7
    W1, W3, W2 = _weights(80, E, h, f)
    rows, experts = [], []
    for e in range(E):
        for i in range(h):
            v = np.zeros(h, np.float32)
            v[i] = 1.0
            rows.append(v)
            experts.append(e)
    y, hm = oracle.expert_rows(np.array(rows), np.array(experts), W1, W3, W2, want_h_mid=True)
    for r_, (e, i) in enumerate(itertools.product(range(E), range(h))):
        a = W1[e, i].astype(np.float64)
        g = W3[e, i].astype(np.float64)
        H = a * expit(a) * g
        np.testing.assert_allclose(hm[r_], H, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(y[r_], H @ W2[e].astype(np.float64), rtol=1e-12, atol=1e-15)


def test_expert_zero_gate_or_up_gives_zero():
    E, h, f = 2, 6, 4
    W1, W3, W2 = _weights(81, E, h, f)
    x = rng(82).standard_normal((5, h)).astype(np.float32)
    ex = np.array([0, 1, 1, 0, 1], np.int32)
    assert np.all(oracle.expert_rows(x, ex, np.zeros_like(W1), W3, W2) == 0.0)  # silu(0) = 0
    assert np.all(oracle.expert_rows(x, ex, W1, np.zeros_like(W3), W2) == 0.0)


def test_expert_linear_in_W2_and_W3():
    E, h, f = 2, 6, 5
    W1, W3, W2 = _weights(83, E, h, f)
    _, _, W2b = _weights(84, E, h, f)
    x = rng(85).standard_normal((6, h)).astype(np.float32)
    ex = np.array([0, 1, 0, 1, 1, 0], np.int32)
    y = oracle.expert_rows(x, ex, W1, W3, W2)
    yb = oracle.expert_rows(x, ex, W1, W3, W2b)
    np.testing.assert_allclose(oracle.expert_rows(x, ex, W1, W3, W2 + W2b), y + yb,
                               rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(oracle.expert_rows(x, ex, W1, W3 * 2, W2), 2 * y,
                               rtol=1e-12, atol=1e-15)


def test_expert_uses_its_own_weights():
    E, h, f = 4, 5, 3
    W1, W3, W2 = _weights(86, E, h, f)
    x = rng(87).standard_normal((1, h)).astype(np.float32)
    ys = [oracle.expert_rows(x, np.array([e], np.int32), W1, W3, W2)[0] for e in range(E)]
    for e in range(E):  # zeroing expert e's down-projection only affects expert e
        W2z = W2.copy()
        W2z[e] = 0
        for e2 in range(E):
            y2 = oracle.expert_rows(x, np.array([e2], np.int32), W1, W3, W2z)[0]
            if e2 == e:
                assert np.all(y2 == 0)
            else:
                np.testing.assert_array_equal(y2, ys[e2])


# ------------------------------------------------------------------ whole --

@pytest.mark.parametrize("score,k,cf", [("softmax_post", 2, 0.0), ("softmax_pre", 1, 1.0),
                                        ("sigmoid", 3, 0.0), ("softmax_post", 2, 0.75)])
def test_forward_permuted_equals_dense(score, k, cf):
    T, h, E, f = 24, 8, 5, 6
    r = rng(90)
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = (0.5 * r.standard_normal((h, E))).astype(np.float32)
    eb = r.uniform(-0.1, 0.1, E).astype(np.float32) if score == "sigmoid" else None
    W1, W3, W2 = _weights(91, E, h, f)
    out = oracle.forward(x, Wg, W1, W3, W2, k, score, expert_bias=eb, capacity_factor=cf)
    if cf > 0:
        assert (out["keep"] == 0).any()
    yd = oracle.forward_dense(x, out["topk_idx"], out["topk_prob"], out["keep"], W1, W3, W2)
    np.testing.assert_allclose(out["y"], yd, rtol=1e-12, atol=1e-14)


def test_forward_bf16_inputs_equal_widened_f32():
    import torch
    T, h, E, k, f = 16, 8, 4, 2, 8
    r = rng(95)
    xf = torch.from_numpy(r.standard_normal((T, h)).astype(np.float32)).to(torch.bfloat16)
    Ws = [torch.from_numpy((0.3 * r.standard_normal(s)).astype(np.float32)).to(torch.bfloat16)
          for s in ((E, h, f), (E, h, f), (E, f, h))]
    Wg = (0.5 * r.standard_normal((h, E))).astype(np.float32)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    a = oracle.forward(bits(xf), Wg, *[bits(w) for w in Ws], k, "softmax_post")
    b = oracle.forward(xf.float().numpy(), Wg, *[w.float().numpy() for w in Ws], k, "softmax_post")
    np.testing.assert_array_equal(a["y"], b["y"])


# ----------------------------------------------------------- shared expert --

def test_shared_expert_one_hot_closed_form():
    # x = e_i: y_shared = (silu(W1s[i,:]) * W3s[i,:]) . W2s for every token,
    # whatever the routing; a transposed W1s/W3s (or W2s) would pick a column.
    T, h, E, k, f, fs = 7, 7, 3, 2, 4, 5
    r = rng(100)
    x = np.eye(h, dtype=np.float32)[r.permutation(h)[:T]]
    Wg = r.standard_normal((h, E)).astype(np.float32)
    W1, W3, W2 = _weights(101, E, h, f)
    W1s, W3s, W2s = (r.standard_normal(s).astype(np.float32) for s in ((h, fs), (h, fs), (fs, h)))
    out = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post", W1s=W1s, W3s=W3s, W2s=W2s)
    for t in range(T):
        i = int(np.argmax(x[t]))
        a, g = W1s[i].astype(np.float64), W3s[i].astype(np.float64)
        H = a * expit(a) * g
        np.testing.assert_allclose(out["h_mid_s"][t], H, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(out["y_shared"][t], H @ W2s.astype(np.float64),
                                   rtol=1e-12, atol=1e-14)
    # the layer output is the routed output plus the shared one
    np.testing.assert_allclose(out["y"], out["y_routed"] + out["y_shared"], rtol=0, atol=0)


def test_shared_expert_equals_a_routed_expert_with_probability_one():
    # one routed expert, top-1 post-softmax (p = 1 exactly) and identical
    # weights: the routed output and the shared one coincide, and y doubles
    T, h, f = 9, 6, 5
    r = rng(102)
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = r.standard_normal((h, 1)).astype(np.float32)
    W1, W3, W2 = _weights(103, 1, h, f)
    out = oracle.forward(x, Wg, W1, W3, W2, 1, "softmax_post", W1s=W1[0], W3s=W3[0], W2s=W2[0])
    assert np.all(out["topk_prob"] == 1.0)
    np.testing.assert_array_equal(out["y_shared"], out["y_routed"])
    np.testing.assert_array_equal(out["y"], 2.0 * out["y_routed"])


def test_shared_expert_zero_down_projection_leaves_routed_output():
    T, h, E, k, f, fs = 10, 8, 4, 2, 6, 4
    r = rng(104)
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = r.standard_normal((h, E)).astype(np.float32)
    W1, W3, W2 = _weights(105, E, h, f)
    W1s, W3s = (r.standard_normal((h, fs)).astype(np.float32) for _ in range(2))
    base = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post")
    out = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post", W1s=W1s, W3s=W3s,
                         W2s=np.zeros((fs, h), np.float32))
    assert np.all(out["y_shared"] == 0.0)
    np.testing.assert_array_equal(out["y"], base["y"])


# ------------------------------------------------ router variants (sqrtsoftplus, groups) --

def _sqrtsoftplus(l):
    return np.sqrt(np.logaddexp(0.0, np.asarray(l, np.float64)))


def test_sqrtsoftplus_all_experts_closed_form():
    # k = E: every expert is chosen, in descending score order, with weight s / sum(s)
    T, E = 7, 6
    logits = (3.0 * rng(110).standard_normal((T, E))).astype(np.float32)
    idx, prob, _ = oracle.topk_scores(logits, E, "sqrtsoftplus")
    s = _sqrtsoftplus(logits).astype(np.float32).astype(np.float64)
    for t in range(T):
        np.testing.assert_array_equal(idx[t], np.argsort(-s[t], kind="stable"))
        np.testing.assert_allclose(prob[t], s[t][idx[t]] / s[t].sum(), rtol=1e-6)


def test_sqrtsoftplus_large_logits_do_not_overflow():
    logits = np.array([[100.0, -100.0, 0.0, 88.0]], np.float32)
    idx, prob, _ = oracle.topk_scores(logits, 4, "sqrtsoftplus")
    s = np.array([10.0, np.sqrt(np.log1p(np.exp(-100.0))), np.sqrt(np.log(2.0)), np.sqrt(88.0)])
    assert list(idx[0]) == [0, 3, 2, 1]
    np.testing.assert_allclose(prob[0], s[idx[0]] / s.sum(), rtol=1e-6)


def test_sqrtsoftplus_bias_only_chooses():
    T, E, k = 5, 6, 2
    logits = rng(111).standard_normal((T, E)).astype(np.float32)
    eb = np.zeros(E, np.float32)
    eb[4] = 10.0  # expert 4 always chosen, its weight from the unbiased score
    idx, prob, _ = oracle.topk_scores(logits, k, "sqrtsoftplus", eb)
    s = _sqrtsoftplus(logits).astype(np.float32).astype(np.float64)
    for t in range(T):
        assert idx[t, 0] == 4
        other = max((e for e in range(E) if e != 4), key=lambda e: (s[t, e], -e))
        assert idx[t, 1] == other
        np.testing.assert_allclose(prob[t], s[t][idx[t]] / s[t][idx[t]].sum(), rtol=1e-6)


def _grouped_brute_force(sel, k, G, gk):
    """Group-limited choice by exhaustive search: the kept groups are the
    gk-subset with the largest total group score (group score = the sum of the
    group's k//gk largest values, each group's best m-subset found by
    enumeration); the chosen experts are the k-subset of the kept groups'
    experts with the largest total score, listed by score."""
    E = sel.shape[0]
    per, m = E // G, k // gk
    gscore = []
    for g in range(G):
        vals = sel[g * per:(g + 1) * per].astype(np.float64)
        gscore.append(max(sum(c) for c in itertools.combinations(vals, m)))
    groups = max(itertools.combinations(range(G), gk), key=lambda c: sum(gscore[g] for g in c))
    elig = [e for e in range(E) if e // per in groups]
    best = max(itertools.combinations(elig, k), key=lambda c: sum(float(sel[e]) for e in c))
    return sorted(best, key=lambda e: -float(sel[e]))


@pytest.mark.parametrize("score,E,k,G,gk", [("softmax_post", 8, 2, 4, 2), ("sigmoid", 12, 4, 4, 2),
                                            ("sqrtsoftplus", 12, 3, 3, 1),
                                            ("softmax_pre", 8, 4, 2, 2)])
def test_group_limited_topk_brute_force(score, E, k, G, gk):
    T = 40
    r = rng(112)
    logits = r.standard_normal((T, E)).astype(np.float32)
    eb = r.uniform(-0.1, 0.1, E).astype(np.float32) if score in ("sigmoid", "sqrtsoftplus") else None
    idx, prob, margin = oracle.topk_scores(logits, k, score, eb, num_groups=G, group_topk=gk)
    # selection scores as the pages define them (fp32 values)
    if score == "softmax_post":
        sel = logits
    elif score == "softmax_pre":
        from scipy.special import softmax as sm
        sel = sm(logits.astype(np.float64), axis=1).astype(np.float32)
    else:
        s = expit(logits.astype(np.float64)) if score == "sigmoid" else _sqrtsoftplus(logits)
        sel = s.astype(np.float32) + (eb if eb is not None else 0)
    for t in range(T):
        assert list(idx[t]) == _grouped_brute_force(sel[t], k, G, gk), t
        assert margin[t] >= 0


def test_group_limited_special_cases_equal_ungrouped():
    T, E, k = 30, 16, 4
    logits = rng(113).standard_normal((T, E)).astype(np.float32)
    base = oracle.topk_scores(logits, k, "sigmoid")
    for G, gk in ((1, 1), (2, 2), (4, 4)):   # one group, or every group kept
        got = oracle.topk_scores(logits, k, "sigmoid", num_groups=G, group_topk=gk)
        np.testing.assert_array_equal(got[0], base[0])
        np.testing.assert_array_equal(got[1], base[1])


def test_group_limited_keeps_experts_inside_chosen_groups():
    # group 1's best two scores dominate, group 0 has the single best expert:
    # with one group kept, group 1 wins (sum of top-2) although it lacks the max
    logits = np.array([[5.0, -9.0, -9.0, -9.0, 4.0, 3.9, -9.0, -9.0]], np.float32)
    idx, prob, margin = oracle.topk_scores(logits, 2, "softmax_post", num_groups=2, group_topk=1)
    assert list(idx[0]) == [4, 5]
    # eligible scores 4.0, 3.9, then -9; group scores 7.9 against -4.0
    np.testing.assert_allclose(margin[0], min(4.0 - 3.9, 3.9 - (-9.0), (4.0 + 3.9) - (5.0 - 9.0)),
                               rtol=1e-6)
    idx_u, _, _ = oracle.topk_scores(logits, 2, "softmax_post")
    assert list(idx_u[0]) == [0, 4]
