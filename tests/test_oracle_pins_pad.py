"""Pins of the oracle's pad_to_capacity routing map and of the permutation by
a routing map (apply_router_token_dropping with pad_to_capacity, §8 of the
Megatron Core page; the dispatcher's permutation by the map, §9).

The page writes the padded map as capacity_mask: per expert column of the
dense [T,E] routing probabilities, the `capacity` largest entries (topk along
the tokens), every token when capacity > T.  The oracle builds it the other
way round, from the kept pairs, filling each column up to min(capacity, T)
with the lowest-index free tokens.  These tests rebuild capacity_mask the
page's way (a per-column sort of the dense probabilities, ties to the lower
token index: the reading for the ties the page leaves open) and compare; they
also check the map permutation against the pair permutation on an unpadded
map, and that padding rows never reach the layer output.
"""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _routing(seed, T, E, k, skew=None):
    """A seeded top-k routing with probabilities (softmax over the k)."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(size=(T, E))
    if skew is not None:
        logits += skew
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, idx, axis=1)
    p = np.exp(sel - sel[:, :1])
    p = (p / p.sum(axis=1, keepdims=True)).astype(np.float32)
    return idx, p


def _capacity_mask(idx, prob, E, cap, policy):
    """capacity_mask of the page: per column of the dense [T,E] matrix (the
    probabilities, or the 0/1 routing map for 'position'), the min(cap, T)
    largest entries, equal entries taken in ascending token order."""
    T, k = idx.shape
    dense = np.zeros((T, E), np.float64)
    for j in range(k):
        dense[np.arange(T), idx[:, j]] = prob[:, j] if policy == "probs" else 1.0
    mask = np.zeros((T, E), np.uint8)
    q = min(cap, T)
    for e in range(E):
        order = np.lexsort((np.arange(T), -dense[:, e]))  # value descending, then token
        mask[order[:q], e] = 1
    return mask, dense


@pytest.mark.parametrize("policy", ["probs", "position"])
@pytest.mark.parametrize("seed,T,E,k,cf", [(1, 200, 8, 2, 1.0), (2, 333, 6, 1, 1.5),
                                          (3, 97, 16, 4, 0.5), (4, 64, 4, 2, 3.0)])
def test_padded_map_is_the_pages_capacity_mask(policy, seed, T, E, k, cf):
    skew = np.linspace(1.5, -1.5, E)  # uneven loads: experts over and under capacity
    idx, prob = _routing(seed, T, E, k, skew)
    cap = oracle.capacity(T, E, k, cf)
    prob_final, keep, kept = oracle.capacity_drop(idx, prob, E, cap, policy)
    m, n = oracle.pad_to_capacity_map(idx, keep, E, cap)
    want, dense = _capacity_mask(idx, prob, E, cap, policy)
    assert np.array_equal(m, want)
    assert np.array_equal(n, want.sum(axis=0))
    # final_probs = routing_probs * final_map: the kept pairs keep their
    # probability, dropped pairs get 0, padding entries carry 0
    fp = dense * m if policy == "probs" else None
    for j in range(k):
        col = m[np.arange(T), idx[:, j]]
        assert np.array_equal(keep[:, j].astype(bool), col.astype(bool))
        if fp is not None:
            assert np.array_equal(prob_final[:, j].astype(np.float64),
                                  fp[np.arange(T), idx[:, j]])
    assert (n == min(cap, T)).all()
    assert ((m.sum(axis=0) > kept) | (kept >= min(cap, T))).all()


def test_capacity_above_tokens_gives_every_token_to_every_expert():
    idx, prob = _routing(5, 50, 8, 2)
    cap = oracle.capacity(50, 8, 2, 40.0)
    assert cap > 50
    _, keep, _ = oracle.capacity_drop(idx, prob, 8, cap, "probs")
    m, n = oracle.pad_to_capacity_map(idx, keep, 8, cap)
    assert m.all() and (n == 50).all()


@pytest.mark.parametrize("seed,T,E,k", [(6, 300, 8, 2), (7, 129, 5, 3), (8, 1000, 32, 4)])
def test_map_permutation_equals_pair_permutation_without_padding(seed, T, E, k):
    idx, prob = _routing(seed, T, E, k, np.linspace(1, -1, E))
    cap = oracle.capacity(T, E, k, 1.0)
    _, keep, _ = oracle.capacity_drop(idx, prob, E, cap, "probs")
    kept_map = np.zeros((T, E), np.uint8)
    t, j = np.nonzero(keep)
    kept_map[t, idx[t, j]] = 1
    a = oracle.permute_map(kept_map, idx, keep)
    b = oracle.permute(idx, keep, E)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_padded_permutation_rows_are_the_map_in_token_order():
    T, E, k = 240, 6, 2
    idx, prob = _routing(9, T, E, k, np.linspace(2, -2, E))
    cap = oracle.capacity(T, E, k, 1.25)
    _, keep, _ = oracle.capacity_drop(idx, prob, E, cap, "probs")
    m, n = oracle.pad_to_capacity_map(idx, keep, E, cap)
    offsets, row_map, row_token = oracle.permute_map(m, idx, keep)
    assert np.array_equal(np.diff(offsets), n)
    for e in range(E):
        seg = row_token[offsets[e]:offsets[e + 1]]
        assert np.array_equal(seg, np.flatnonzero(m[:, e]))  # ascending, exactly the column
    for tt in range(T):
        for jj in range(k):
            r = row_map[tt, jj]
            if keep[tt, jj]:
                e = idx[tt, jj]
                assert offsets[e] <= r < offsets[e + 1] and row_token[r] == tt
            else:
                assert r == -1


@pytest.mark.parametrize("policy", ["probs", "position"])
def test_padding_never_reaches_the_output(policy):
    rng = np.random.default_rng(10)
    T, h, E, k, f = 160, 16, 6, 2, 24
    x = rng.normal(size=(T, h)).astype(np.float32)
    Wg = (rng.normal(size=(h, E)) * 0.5).astype(np.float32)
    gb = np.linspace(1.0, -1.0, E).astype(np.float32)
    W1 = (rng.normal(size=(E, h, f)) * 0.2).astype(np.float32)
    W3 = (rng.normal(size=(E, h, f)) * 0.2).astype(np.float32)
    W2 = (rng.normal(size=(E, f, h)) * 0.2).astype(np.float32)
    kw = dict(gate_bias=gb, capacity_factor=1.25, drop_policy=policy)
    a = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post", pad_to_capacity=True, **kw)
    b = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post", **kw)
    cap = a["capacity"]
    assert (a["tokens_per_expert"] == min(cap, T)).all()
    assert int(a["offsets"][-1]) == E * min(cap, T) > int(b["offsets"][-1])  # padding rows exist
    assert np.array_equal(a["y"], b["y"])  # bit for bit: padding rows carry no weight
    assert np.array_equal(a["keep"], b["keep"]) and np.array_equal(a["topk_prob"], b["topk_prob"])
    # every padded row is that expert's MLP of its token
    assert np.array_equal(a["x_perm"], x[a["row_token"]])
