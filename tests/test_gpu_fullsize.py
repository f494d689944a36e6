"""Parity at every workload's full size, in the launch configuration the
benchmark times (the same C-ABI stage calls and kernels).

Checked in full: routing (topk_idx, keep, tokens_per_expert bit-exact,
probabilities within tolerance), the permutation (expert_offsets, row_map
bit-exact; every permuted row equal to its source token row), and
moe_forward reproducing the staged output bit for bit.

The expert MLP and the combine are checked on a covering set of rows that
the oracle evaluates one by one, every column of each: in every expert that
has rows, every 128-row block of its rows (the grouped GEMM's row tile; a
256-row SM-pair tile is two of them) contributes its first and last row and
two seeded rows from each of its 32-row quarters (one epilogue warp each),
so each expert's partly filled tail block is checked.  The layer output y is
checked on a seeded token sample (with capacity drops, half of it tokens
with a dropped pair), all k of each token's rows evaluated by the oracle.
The oracle takes one expert's weights at a time, copied to the host, so
host memory stays bounded.  The grouped expert MLP is section 10 (Experts)
and the combine section 2 of the Megatron Core walkthrough
(r00kie-liu.github.io).
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import (assert_close, assert_equal, assert_probs, condition_inputs, gpu_forward,
                       gpu_stages, np_view, to_np)

pytestmark = pytest.mark.gpu

ROW_BLOCK = 128      # rows of one grouped-GEMM tile (half of an SM-pair tile)
WARP_ROWS = 32       # rows drained by one epilogue warp
ROWS_PER_WARP = 2    # seeded rows checked in each 32-row quarter of a block
Y_TOKENS = 48        # tokens whose output row y is checked
WEIGHT_CHUNK = 1 << 30   # expert weight bytes copied to the host at a time


@pytest.fixture(scope="module", params=sorted(synthetic.WORKLOADS))
def full(request):
    w = synthetic.WORKLOADS[request.param]
    torch.cuda.empty_cache()
    inp = synthetic.generate(w, device="cuda")
    r = condition_inputs(w, inp)
    b = gpu_stages(w, inp, with_routing_map=False)
    torch.cuda.synchronize()
    yield w, inp, r, b
    del inp, b
    torch.cuda.empty_cache()


def test_routing_full(full):
    w, inp, r, b = full
    assert_equal("topk_idx", to_np(b.topk_idx), r["topk_idx"])
    assert_equal("keep", to_np(b.keep), r["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), r["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), r["topk_prob"])
    if w.capacity_factor > 0:
        assert (r["keep"] == 0).any()


def test_permutation_full(full):
    w, inp, r, b = full
    if w.pad_to_capacity:  # the permutation of the padded routing map
        assert_equal("routing_map", to_np(b.routing_map), r["routing_map"])
        offsets, row_map, row_token = oracle.permute_map(r["routing_map"], r["topk_idx"],
                                                         r["keep"])
    else:
        offsets, row_map, row_token = oracle.permute(r["topk_idx"], r["keep"], w.E)
    assert_equal("expert_offsets", to_np(b.expert_offsets), offsets)
    assert_equal("row_map", to_np(b.row_map), row_map)
    R = int(offsets[-1])
    src = inp["x"][torch.from_numpy(row_token).long().to(inp["x"].device)]
    got = b.x_perm[:R]
    if got.dtype == torch.bfloat16:
        got, src = got.view(torch.int16), src.view(torch.int16)
    assert torch.equal(got, src)


def _oracle_permutation(w, r):
    if w.pad_to_capacity:
        return oracle.permute_map(r["routing_map"], r["topk_idx"], r["keep"])
    return oracle.permute(r["topk_idx"], r["keep"], w.E)


def _covering_rows(offsets, rng):
    """Rows of x_perm that cover every (expert, 128-row block): the block's
    first and last row and seeded rows of each of its 32-row quarters."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for b0 in range(lo, hi, ROW_BLOCK):
            b1 = min(b0 + ROW_BLOCK, hi)
            rows += [b0, b1 - 1]
            for q0 in range(b0, b1, WARP_ROWS):
                rows += rng.integers(q0, min(q0 + WARP_ROWS, b1), ROWS_PER_WARP).tolist()
    return np.unique(np.array(rows, np.int64))


def _y_tokens(w, r, rng):
    order = rng.permutation(w.T)
    if w.capacity_factor > 0:
        dropped = order[(r["keep"][order] == 0).any(axis=1)][:Y_TOKENS // 2]
        kept = order[(r["keep"][order] == 1).all(axis=1)][:Y_TOKENS - len(dropped)]
        return np.sort(np.concatenate([dropped, kept]))
    return np.sort(order[:Y_TOKENS])


def _expert_chunks(experts, bytes_per_expert):
    per = max(1, WEIGHT_CHUNK // max(1, bytes_per_expert))
    for i in range(0, len(experts), per):
        yield experts[i:i + per]


def _oracle_rows(w, inp, rows, row_expert, row_token):
    """Oracle h_mid and y_perm of the given x_perm rows, one chunk of experts'
    weights on the host at a time."""
    f, h = w.f, w.h
    y = np.empty((len(rows), h), np.float64)
    hm = np.empty((len(rows), f), np.float64)
    x = inp["x"]
    experts = np.unique(row_expert)
    esize = 3 * h * f * inp["W1"].element_size()
    for chunk in _expert_chunks(list(experts), esize):
        sel = np.nonzero(np.isin(row_expert, chunk))[0]
        local = {int(e): i for i, e in enumerate(chunk)}
        idx = torch.tensor([int(e) for e in chunk], device=inp["W1"].device)
        W = {n: np_view(inp[n].index_select(0, idx).cpu()) for n in ("W1", "W3", "W2")}
        toks = torch.from_numpy(row_token[rows[sel]]).long().to(x.device)
        xr = np_view(x.index_select(0, toks).cpu())
        re = np.array([local[int(e)] for e in row_expert[sel]], np.int32)
        ys, hs = oracle.expert_rows(xr, re, W["W1"], W["W3"], W["W2"], want_h_mid=True)
        y[sel], hm[sel] = ys, hs
    return y, hm


def test_covering_outputs_full(full):
    w, inp, r, b = full
    offsets, row_map, row_token = _oracle_permutation(w, r)
    rng = np.random.default_rng(1234)
    cover = _covering_rows(offsets, rng)
    toks = _y_tokens(w, r, rng)
    tok_rows = row_map[toks].reshape(-1)
    rows = np.unique(np.concatenate([cover, tok_rows[tok_rows >= 0]]).astype(np.int64))
    row_expert = np.searchsorted(offsets, rows, side="right") - 1
    y_rows, h_rows = _oracle_rows(w, inp, rows, row_expert, row_token)

    # every column of every covering row (and of the y tokens' rows)
    g = torch.from_numpy(rows).to(b.h_mid.device)
    assert_close("h_mid", to_np(b.h_mid.index_select(0, g)), h_rows,
                 "bf16_stored" if w.dtype == "bf16" else w.dtype)
    assert_close("y_perm", to_np(b.y_perm.index_select(0, g)), y_rows, w.dtype)
    # every (expert, block) with rows is covered
    blocks = {(int(e), (int(rw) - int(offsets[e])) // ROW_BLOCK) for e, rw in zip(row_expert, rows)}
    want_blocks = sum(-(-int(offsets[e + 1] - offsets[e]) // ROW_BLOCK) for e in range(w.E))
    assert len(blocks) == want_blocks

    # the output rows of the sampled tokens, from the oracle's rows
    pos = {int(rw): i for i, rw in enumerate(rows)}
    local_map = np.array([[pos[int(rw)] if rw >= 0 else -1 for rw in row_map[t]] for t in toks],
                         np.int32)
    y_ref = oracle.combine(y_rows, local_map, r["topk_prob"][toks])
    tsel = torch.from_numpy(toks).to(b.y.device)
    if w.shared_f > 0:
        x_cpu = inp["x"].index_select(0, tsel).cpu()
        ys, hs = oracle.shared_expert(np_view(x_cpu), *(np_view(inp[n].cpu()) for n in
                                                       ("W1s", "W3s", "W2s")), want_h_mid=True)
        assert_close("h_mid_s", to_np(b.h_mid_s[tsel]), hs,
                     "bf16_stored" if w.dtype == "bf16" else w.dtype)
        assert_close("y_shared", to_np(b.y_shared[tsel]), ys, w.dtype)
        y_ref = y_ref + ys
    assert_close("y", to_np(b.y[tsel]), y_ref, w.dtype)
    if w.capacity_factor > 0:
        all_dropped = (r["keep"][toks] == 0).all(axis=1)
        assert (r["keep"][toks] == 0).any()
        assert np.all(y_ref[all_dropped] == 0)


def test_forward_reproduces_stages_full(full):
    w, inp, r, b = full
    y, idx, prob, tpe = gpu_forward(w, inp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(tpe, b.tokens_per_expert)
    assert torch.equal(y, b.y)
