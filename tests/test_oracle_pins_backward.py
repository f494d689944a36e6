"""Pins of the oracle's backward against facts other than itself: central
finite differences of the (separately pinned) forward for every score
function, with capacity drops and group-limited routing; Euler's identity
for the parameters the output is linear in (W2, W3: sum(W * dW) = L for
L = sum(dy * y)); and the cases where the router gets no gradient (top-1
after softmax: p == 1).  Routing decisions are held fixed, as in the
method: inputs are drawn with clear top-k margins and each perturbed
forward is checked to route identically.  CPU only.
"""

import numpy as np
import pytest

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, T=6, h=8, E=4, f=6, eb=False):
    r = rng(seed)
    p = {"x": r.standard_normal((T, h)).astype(np.float32),
         "Wg": (0.7 * r.standard_normal((h, E))).astype(np.float32),
         "gate_bias": (0.1 * r.standard_normal(E)).astype(np.float32),
         "W1": (0.5 * r.standard_normal((E, h, f))).astype(np.float32),
         "W3": (0.5 * r.standard_normal((E, h, f))).astype(np.float32),
         "W2": (0.5 * r.standard_normal((E, f, h))).astype(np.float32),
         "expert_bias": r.uniform(-0.1, 0.1, E).astype(np.float32) if eb else None}
    dy = r.standard_normal((T, h)).astype(np.float32)
    return p, dy


def _loss(p, dy, k, score, cf, groups):
    out = oracle.forward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], k, score, p["gate_bias"],
                         p["expert_bias"], capacity_factor=cf, num_groups=groups[0],
                         group_topk=groups[1])
    return float(np.sum(dy.astype(np.float64) * out["y"])), out


CASES = [("softmax_post", 2, 0.0, (0, 0), False), ("softmax_pre", 2, 0.0, (0, 0), False),
         ("sigmoid", 3, 0.0, (0, 0), True), ("sqrtsoftplus", 2, 0.0, (0, 0), True),
         ("softmax_pre", 1, 0.75, (0, 0), False), ("sigmoid", 2, 0.0, (2, 1), True),
         ("softmax_post", 2, 0.9, (0, 0), False)]


@pytest.mark.parametrize("score,k,cf,groups,eb", CASES)
def test_backward_matches_finite_differences(score, k, cf, groups, eb):
    p, dy = _problem(140 + k + int(10 * cf) + groups[0], eb=eb)
    L0, base = _loss(p, dy, k, score, cf, groups)
    if cf > 0:
        assert (base["keep"] == 0).any()
    g = oracle.backward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], k, score, base["topk_idx"],
                        base["topk_prob"], base["keep"], dy, p["gate_bias"], p["expert_bias"])
    names = {"x": "dx", "Wg": "dWg", "gate_bias": "dgate_bias", "W1": "dW1", "W3": "dW3",
             "W2": "dW2"}
    r = rng(7)
    checked = 0
    for name, gname in names.items():
        arr = p[name]
        for flat in r.choice(arr.size, size=min(arr.size, 12), replace=False):
            idx = np.unravel_index(flat, arr.shape)
            v = float(arr[idx])
            d = 1e-3 * max(1.0, abs(v))
            plus, minus = dict(p), dict(p)
            plus[name] = arr.copy()
            minus[name] = arr.copy()
            plus[name][idx] = np.float32(v + d)
            minus[name][idx] = np.float32(v - d)
            lp, op = _loss(plus, dy, k, score, cf, groups)
            lm, om = _loss(minus, dy, k, score, cf, groups)
            same = all(np.array_equal(o["topk_idx"], base["topk_idx"]) and
                       np.array_equal(o["keep"], base["keep"]) for o in (op, om))
            if not same:  # the routing moved: no derivative there
                continue
            step = float(plus[name][idx]) - float(minus[name][idx])
            fd = (lp - lm) / step
            an = g[gname][idx]
            # parameters that reach the router pass through the forward's fp32
            # roundings of logits and probabilities (about 1e-7 relative), which
            # the central difference divides by 2e-3: 1e-4 of noise, hence 1e-3
            tol = 1e-3 if name in ("x", "Wg", "gate_bias") else 2e-5
            assert abs(fd - an) <= tol * (abs(an) + 1.0), (name, idx, fd, an)
            checked += 1
    assert checked >= 50


@pytest.mark.parametrize("score,k", [("softmax_post", 2), ("sigmoid", 3)])
def test_backward_euler_identity_for_linear_parameters(score, k):
    # y is linear in W2 and in W3 (routing fixed): sum(W * dW) = sum(dy * y)
    p, dy = _problem(150, T=9, E=5, eb=(score == "sigmoid"))
    L, base = _loss(p, dy, k, score, 0.0, (0, 0))
    g = oracle.backward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], k, score, base["topk_idx"],
                        base["topk_prob"], base["keep"], dy, p["gate_bias"], p["expert_bias"])
    for w, dw in (("W2", "dW2"), ("W3", "dW3")):
        np.testing.assert_allclose(np.sum(p[w].astype(np.float64) * g[dw]), L, rtol=1e-10)


def test_top1_after_softmax_gives_the_router_no_gradient():
    p, dy = _problem(151)
    _, base = _loss(p, dy, 1, "softmax_post", 0.0, (0, 0))
    g = oracle.backward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], 1, "softmax_post",
                        base["topk_idx"], base["topk_prob"], base["keep"], dy, p["gate_bias"])
    assert np.all(g["dlogits"] == 0.0) and np.all(g["dWg"] == 0.0)
    assert np.all(g["dgate_bias"] == 0.0)


def test_backward_is_linear_in_dy_and_zero_for_dropped_tokens():
    p, dy = _problem(152, T=10)
    _, base = _loss(p, dy, 1, "softmax_pre", 0.5, (0, 0))
    args = (p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], 1, "softmax_pre", base["topk_idx"],
            base["topk_prob"], base["keep"])
    g1 = oracle.backward(*args, dy, p["gate_bias"])
    g2 = oracle.backward(*args, 4.0 * dy, p["gate_bias"])  # a power of two: exact in fp32
    for key in g1:
        np.testing.assert_allclose(g2[key], 4.0 * g1[key], rtol=1e-12, atol=1e-14)
    dropped = np.nonzero(base["keep"][:, 0] == 0)[0]
    assert dropped.size > 0
    # a dropped token reaches no expert; only the router term remains
    router_only = g1["dlogits"][dropped] @ p["Wg"].astype(np.float64).T
    np.testing.assert_allclose(g1["dx"][dropped], router_only, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("score,k,cf", [("softmax_post", 2, 0.0), ("sigmoid", 3, 0.0),
                                        ("softmax_pre", 1, 0.75)])
def test_expert_wgrad_cols_match_the_full_backward(score, k, cf):
    # the column oracle (used where the full backward is out of reach) against
    # the finite-difference-pinned backward: every row of dW2[e] and every
    # column of dW1[e] / dW3[e], from the expert's kept rows in token order
    p, dy = _problem(160 + k, T=12, E=3, eb=(score == "sigmoid"))
    _, base = _loss(p, dy, k, score, cf, (0, 0))
    g = oracle.backward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], k, score, base["topk_idx"],
                        base["topk_prob"], base["keep"], dy, p["gate_bias"], p["expert_bias"])
    f = p["W1"].shape[-1]
    checked = 0
    for e in range(3):
        pairs = [(t, j) for t in range(12) for j in range(k)
                 if base["topk_idx"][t, j] == e and base["keep"][t, j]]
        if not pairs:
            continue
        rows = np.array([t for t, _ in pairs])
        prob = np.array([base["topk_prob"][t, j] for t, j in pairs], np.float32)
        c = oracle.expert_wgrad_cols(p["x"][rows], prob, dy[rows], p["W1"][e], p["W3"][e],
                                     p["W2"][e], np.arange(f), np.arange(f))
        np.testing.assert_allclose(c["dW2_rows"], g["dW2"][e], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(c["dW1_cols"], g["dW1"][e], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(c["dW3_cols"], g["dW3"][e], rtol=1e-12, atol=1e-14)
        checked += 1
    assert checked >= 2


def test_weight_grads_off_leaves_the_rest_unchanged():
    p, dy = _problem(165)
    _, base = _loss(p, dy, 2, "softmax_post", 0.0, (0, 0))
    args = (p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], 2, "softmax_post", base["topk_idx"],
            base["topk_prob"], base["keep"], dy, p["gate_bias"])
    full = oracle.backward(*args)
    part = oracle.backward(*args, weight_grads=False)
    for key in ("dx", "dWg", "dgate_bias", "dlogits"):
        assert np.array_equal(full[key], part[key]), key
    assert part["dW1"] is None and part["dW2"] is None


@pytest.mark.parametrize("score,k,cf", [("softmax_post", 2, 0.0), ("sigmoid", 3, 0.0),
                                        ("softmax_pre", 1, 0.75)])
def test_shared_expert_backward_matches_finite_differences(score, k, cf):
    # the layer with a shared expert (y = routed + SwiGLU_s(x)): routed
    # backward + oracle.shared_backward against central differences of the
    # whole forward, for x and the shared weights
    p, dy = _problem(170 + k, eb=(score == "sigmoid"))
    r = rng(171)
    h = p["x"].shape[1]
    fs = 5
    p.update({"W1s": (0.5 * r.standard_normal((h, fs))).astype(np.float32),
              "W3s": (0.5 * r.standard_normal((h, fs))).astype(np.float32),
              "W2s": (0.5 * r.standard_normal((fs, h))).astype(np.float32)})

    def loss(q):
        out = oracle.forward(q["x"], q["Wg"], q["W1"], q["W3"], q["W2"], k, score,
                             q["gate_bias"], q["expert_bias"], capacity_factor=cf,
                             W1s=q["W1s"], W3s=q["W3s"], W2s=q["W2s"])
        return float(np.sum(dy.astype(np.float64) * out["y"])), out

    L0, base = loss(p)
    g = oracle.backward(p["x"], p["Wg"], p["W1"], p["W3"], p["W2"], k, score, base["topk_idx"],
                        base["topk_prob"], base["keep"], dy, p["gate_bias"], p["expert_bias"])
    gs = oracle.shared_backward(p["x"], p["W1s"], p["W3s"], p["W2s"], dy)
    grads = {"x": g["dx"] + gs["dx"], "W1s": gs["dW1s"], "W3s": gs["dW3s"], "W2s": gs["dW2s"]}
    pick = rng(172)
    checked = 0
    for name, an_all in grads.items():
        arr = p[name]
        for flat in pick.choice(arr.size, size=min(arr.size, 12), replace=False):
            idx = np.unravel_index(flat, arr.shape)
            v = float(arr[idx])
            d = 1e-3 * max(1.0, abs(v))
            plus, minus = dict(p), dict(p)
            plus[name], minus[name] = arr.copy(), arr.copy()
            plus[name][idx] = np.float32(v + d)
            minus[name][idx] = np.float32(v - d)
            lp, op = loss(plus)
            lm, om = loss(minus)
            if not all(np.array_equal(o["topk_idx"], base["topk_idx"]) and
                       np.array_equal(o["keep"], base["keep"]) for o in (op, om)):
                continue
            fd = (lp - lm) / (float(plus[name][idx]) - float(minus[name][idx]))
            an = an_all[idx]
            tol = 1e-3 if name == "x" else 2e-5   # x reaches the router's fp32 roundings
            assert abs(fd - an) <= tol * (abs(an) + 1.0), (name, idx, fd, an)
            checked += 1
    assert checked >= 30
