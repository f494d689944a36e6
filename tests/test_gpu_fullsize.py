"""Parity at every workload's full size, in the launch configuration the
benchmark times (the same C-ABI stage calls and kernels).

Checked in full: routing (topk_idx, keep, tokens_per_expert bit-exact,
probabilities within tolerance), the permutation (expert_offsets, row_map
bit-exact; every permuted row equal to its source token row), and
moe_forward reproducing the staged output bit for bit.  Checked on a seeded
sample of tokens that the oracle evaluates one by one: each sampled token's
expert rows (h_mid, y_perm) and its output row y.  The sample is limited to
a few dozen experts so that the oracle only needs those experts' weights.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import (assert_close, assert_equal, assert_probs, condition_inputs, gpu_forward,
                       gpu_stages, np_view, to_np)

pytestmark = pytest.mark.gpu

MAX_EXPERTS = {"tiny_fp32": 8, "mixtral": 8, "dsv3": 48, "dsv3_grouped": 48, "dsv3_shared": 48,
               "qwen3": 48, "switch": 32, "switch_pad": 32}
MAX_TOKENS = 32


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


def _sample_tokens(w, r):
    """Seeded token sample whose kept pairs touch at most MAX_EXPERTS experts;
    with capacity drops, half of the sample has a dropped pair."""
    rng = np.random.default_rng(1234)
    order = rng.permutation(w.T)
    if w.capacity_factor > 0:
        dropped = order[(r["keep"][order] == 0).any(axis=1)]
        kept = order[(r["keep"][order] == 1).all(axis=1)]
        order = np.concatenate([np.stack([dropped[:MAX_TOKENS // 2],
                                          kept[:MAX_TOKENS // 2]], 1).reshape(-1), kept])
    experts, toks = set(), []
    for t in order:
        es = set(r["topk_idx"][t][r["keep"][t] == 1].tolist())
        if len(experts | es) > MAX_EXPERTS[w.name]:
            continue
        experts |= es
        toks.append(int(t))
        if len(toks) == MAX_TOKENS:
            break
    return np.array(sorted(toks)), sorted(experts)


def test_sampled_outputs_full(full):
    w, inp, r, b = full
    toks, experts = _sample_tokens(w, r)
    assert len(toks) >= 3
    sub = {e: i for i, e in enumerate(experts)}
    W = {n: np_view(torch.stack([inp[n][e] for e in experts]).cpu()) for n in ("W1", "W3", "W2")}
    x_cpu = inp["x"][torch.from_numpy(toks).to(inp["x"].device)].cpu()
    k = w.k
    pairs = [(i, j) for i, t in enumerate(toks) for j in range(k) if r["keep"][t, j]]
    rows_x = np.stack([np_view(x_cpu)[i] for i, _ in pairs])
    rows_e = np.array([sub[int(r["topk_idx"][toks[i], j])] for i, j in pairs], np.int32)
    y_rows, h_rows = oracle.expert_rows(rows_x, rows_e, W["W1"], W["W3"], W["W2"],
                                        want_h_mid=True)
    # GPU rows of those pairs
    gpu_rows = torch.tensor([int(to_np(b.row_map[toks[i], j])) for i, j in pairs],
                            device=b.h_mid.device)
    assert_close("h_mid", to_np(b.h_mid[gpu_rows]), h_rows,
                 "bf16_stored" if w.dtype == "bf16" else w.dtype)
    assert_close("y_perm", to_np(b.y_perm[gpu_rows]), y_rows, w.dtype)
    # oracle combine of the sampled tokens
    local_map = np.full((len(toks), k), -1, np.int32)
    for n, (i, j) in enumerate(pairs):
        local_map[i, j] = n
    y_ref = oracle.combine(y_rows, local_map, r["topk_prob"][toks])
    tsel = torch.from_numpy(toks).to(b.y.device)
    if w.shared_f > 0:
        ys, hs = oracle.shared_expert(np_view(x_cpu), *(np_view(inp[n].cpu()) for n in
                                                       ("W1s", "W3s", "W2s")), want_h_mid=True)
        assert_close("h_mid_s", to_np(b.h_mid_s[tsel]), hs,
                     "bf16_stored" if w.dtype == "bf16" else w.dtype)
        assert_close("y_shared", to_np(b.y_shared[tsel]), ys, w.dtype)
        y_ref = y_ref + ys
    assert_close("y", to_np(b.y[tsel]), y_ref, w.dtype)
    if w.capacity_factor > 0:
        all_dropped = (r["keep"][toks] == 0).all(axis=1)
        assert np.all(y_ref[all_dropped] == 0)


def test_forward_reproduces_stages_full(full):
    w, inp, r, b = full
    y, idx, prob, tpe = gpu_forward(w, inp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(tpe, b.tokens_per_expert)
    assert torch.equal(y, b.y)
