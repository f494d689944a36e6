"""pad_to_capacity on the GPU against the oracle (apply_router_token_dropping
with pad_to_capacity, §8 of the Megatron Core page, and the dispatcher's
permutation by the padded routing map, §9).

Every expert's input holds exactly min(capacity, T) rows: its kept pairs and,
under capacity, the lowest-index tokens not routed to it, in token order.
Checked bit for bit: the padded routing map, tokens_per_expert, the expert
offsets, row_map and every permuted row; h_mid, y_perm (padding rows
included) and y within the parity tolerances.  Padding rows carry no combine
weight, so the layer output equals the unpadded layer's bit for bit (each
output row of the grouped GEMM depends on its own row only).  Also: the
padded moe_forward reproduces the staged calls, moe_permute_map on an
unpadded routing map gives moe_permute's result, and the backward of the
padded layer gives the unpadded layer's gradients (the oracle backward of the
same routing; the padding rows' gradients are zero) within the criteria of
the bf16 and fp32 backward tests.
"""

import pytest
import torch

import synthetic
from moe_cases import (assert_equal, compare_all, gpu_config, gpu_forward, gpu_stages,
                       make_case, oracle_forward, to_dev, to_np)

pytestmark = pytest.mark.gpu

CASES = {
    # Switch-like top-1: 4 hot experts dropped to capacity, the rest padded
    "switch_probs": synthetic.scaled("switch", T=4096, h=256, f=256, seed=14,
                                     pad_to_capacity=True),
    "switch_position": synthetic.scaled("switch", T=2048, h=256, f=256, seed=15,
                                        drop_policy="position", pad_to_capacity=True),
    # top-2 of 8 with two hot experts: drops and padding in one layer
    "top2_hot": synthetic.scaled("mixtral", T=700, h=256, f=256, capacity_factor=1.0,
                                 gate_bias="hot:2:2.5", seed=71, pad_to_capacity=True),
    # capacity above T: every token goes to every expert
    "capacity_above_tokens": synthetic.scaled("mixtral", T=300, h=256, f=128,
                                              capacity_factor=20.0, seed=72,
                                              pad_to_capacity=True),
    # fp32 experts (SIMT GEMM)
    "tiny_fp32": synthetic.scaled("tiny_fp32", T=500, capacity_factor=1.1, seed=73,
                                  pad_to_capacity=True),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, r = make_case(w)
    ref = oracle_forward(w, inp)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    return w, inp, ref, dinp, b


def test_padded_layer_matches_oracle(case):
    w, inp, ref, dinp, b = case
    assert_equal("routing_map", to_np(b.routing_map), ref["routing_map"])
    compare_all(w, inp, ref, b)
    q = min(ref["capacity"], w.T)
    assert (to_np(b.tokens_per_expert) == q).all()
    assert int(ref["offsets"][-1]) == w.E * q


def test_padding_never_reaches_the_output(case):
    w, inp, ref, dinp, b = case
    from dataclasses import replace
    # the unpadded layer over the same fp32 y_perm and combine kernel as the padded one
    u = gpu_stages(replace(w, pad_to_capacity=False), dinp, fp32_combine=True)
    torch.cuda.synchronize()
    for n in ("topk_idx", "topk_prob", "keep"):
        assert torch.equal(getattr(u, n), getattr(b, n)), n
    assert torch.equal(u.y, b.y)


def test_padded_forward_reproduces_stages(case):
    w, inp, ref, dinp, b = case
    y, idx, prob, tpe = gpu_forward(w, dinp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(prob, b.topk_prob)
    assert torch.equal(tpe, b.tokens_per_expert)
    assert torch.equal(y, b.y)


@pytest.mark.parametrize("name,w", [
    ("mixtral", synthetic.scaled("mixtral", T=600, h=512, f=384, seed=11)),
    ("switch_drop", synthetic.scaled("switch", T=4096, h=256, f=256, seed=14)),
    ("qwen3", synthetic.scaled("qwen3", T=1024, h=512, f=384, seed=13)),
])
def test_permute_map_equals_permute_without_padding(name, w):
    import mixture_experts_layer_fp32_gb300 as moe
    inp, _ = make_case(w)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)  # moe_route with the routing map, moe_permute
    cfg = gpu_config(w)
    x_perm = torch.empty_like(b.x_perm)
    row_map = torch.empty_like(b.row_map)
    offsets = torch.empty_like(b.expert_offsets)
    moe.permute_map(cfg, dinp["x"], b.routing_map, b.topk_idx, b.keep, x_perm, row_map, offsets,
                    b.ws)
    moe.check(b.ws)
    R = int(b.expert_offsets[-1])
    assert torch.equal(offsets, b.expert_offsets)
    assert torch.equal(row_map, b.row_map)
    assert torch.equal(x_perm[:R], b.x_perm[:R])


@pytest.mark.parametrize("name", ["switch_probs", "top2_hot", "tiny_fp32"])
def test_padded_backward_matches_oracle(name):
    import mixture_experts_layer_fp32_gb300 as moe
    import oracle
    from moe_cases import assert_close, np_view
    from test_gpu_backward import assert_grad
    w = CASES[name]
    inp, r = make_case(w)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)
    cfg = gpu_config(w)
    dy = torch.randn((w.T, w.h), generator=torch.Generator().manual_seed(420)).to(
        moe.act_dtype(cfg))
    g = moe.Grads(cfg)
    ws = moe.alloc_workspace_backward(cfg)
    moe.backward(cfg, dinp["x"], dinp["Wg"], dinp["gate_bias"], dinp["W1"], dinp["W3"],
                 dinp["W2"], b, dy.cuda(), g, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    ref = oracle.backward(np_view(inp["x"]), np_view(inp["Wg"]), np_view(inp["W1"]),
                          np_view(inp["W3"]), np_view(inp["W2"]), w.k, w.score, r["topk_idx"],
                          r["topk_prob"], r["keep"], np_view(dy), np_view(inp["gate_bias"]),
                          np_view(inp["expert_bias"]))
    for n in ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2"):
        got = to_np(getattr(g, n))
        if w.dtype == "f32":
            assert_close(n, got, ref[n], "f32")
        elif n == "dWg" and not ref[n].any():  # top-1 after softmax: nothing reaches the router
            assert not got.any()
        elif n == "dgate_bias" and not ref[n].any():
            assert not got.any()
        else:
            assert_grad(n, got, ref[n])
