"""GPU parity: the CUDA path through the C ABI against the CPU oracle on
seeded inputs at sizes the oracle finishes in seconds.  Each shrunk
workload keeps its routing structure and spans several GEMM tiles with
ragged tails (rows per expert not a multiple of 128).
"""

import numpy as np
import pytest
import torch

import synthetic
from moe_cases import (assert_close, assert_equal, assert_probs, gpu_forward, gpu_stages,
                       make_case, oracle_forward, to_dev, to_np)

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32": synthetic.WORKLOADS["tiny_fp32"],
    "tiny_fp32_ragged": synthetic.scaled("tiny_fp32", T=1000, h=136, f=200, seed=10),
    "mixtral_small": synthetic.scaled("mixtral", T=600, h=512, f=384, seed=11),
    "dsv3_small": synthetic.scaled("dsv3", T=300, h=512, f=256, seed=12),
    "qwen3_small": synthetic.scaled("qwen3", T=1024, h=512, f=384, seed=13),
    "switch_small": synthetic.scaled("switch", T=4096, h=256, f=256, seed=14),
    "switch_small_position": synthetic.scaled("switch", T=2048, h=256, f=256, seed=15,
                                              drop_policy="position"),
    # one expert with ~7000 routed tokens: more drop candidates than the
    # drop kernel keeps in shared memory (4096), so its keys are re-read
    "switch_one_hot": synthetic.scaled("switch", T=12000, h=256, f=256, E=8, seed=16,
                                       gate_bias="hot:1:4.6"),
    # fp32 x with 64 experts: the large-E router GEMM's fp32 operand path, one
    # K split whose last 16-wide K tile is half past h = 136 (zero-filled)
    "fp32_e64": synthetic.scaled("qwen3", T=777, h=136, f=64, E=64, k=4, dtype="f32",
                                 seed=17),
    # 192 experts: 64-wide expert tiles, 3 of them, and 8 experts per top-k lane
    "e192": synthetic.scaled("qwen3", T=700, h=512, f=128, E=192, k=6, seed=18),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, r = make_case(w)
    ref = oracle_forward(w, inp)
    dinp = to_dev(inp)
    out = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    return w, inp, ref, dinp, out


def test_routing_bit_exact(case):
    w, inp, ref, dinp, b = case
    assert_equal("topk_idx", to_np(b.topk_idx), ref["topk_idx"])
    assert_equal("keep", to_np(b.keep), ref["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), ref["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), ref["topk_prob"])
    rm = np.zeros((w.T, w.E), np.uint8)
    t_idx, s_idx = np.nonzero(ref["keep"])
    rm[t_idx, ref["topk_idx"][t_idx, s_idx]] = 1
    assert_equal("routing_map", to_np(b.routing_map), rm)
    if w.capacity_factor > 0:
        assert (ref["keep"] == 0).any(), "this workload is meant to drop tokens"


def test_permutation_bit_exact(case):
    w, inp, ref, dinp, b = case
    assert_equal("expert_offsets", to_np(b.expert_offsets), ref["offsets"])
    assert_equal("row_map", to_np(b.row_map), ref["row_map"])
    R = int(ref["offsets"][-1])
    got = b.x_perm[:R].detach().cpu()
    want = inp["x"][torch.from_numpy(ref["row_token"]).long()]
    assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                       want.view(torch.int16) if want.dtype == torch.bfloat16 else want)


def test_expert_mlp(case):
    w, inp, ref, dinp, b = case
    R = int(ref["offsets"][-1])
    assert_close("h_mid", to_np(b.h_mid[:R]), ref["h_mid"],
                 "bf16_stored" if w.dtype == "bf16" else w.dtype)
    assert_close("y_perm", to_np(b.y_perm[:R]), ref["y_perm"], w.dtype)


def test_output(case):
    w, inp, ref, dinp, b = case
    assert_close("y", to_np(b.y), ref["y"], w.dtype)


def test_forward_matches_stages(case):
    # moe_forward runs the same kernels with the same launch shapes
    w, inp, ref, dinp, b = case
    y, idx, prob, tpe = gpu_forward(w, dinp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(tpe, b.tokens_per_expert)
    assert torch.equal(prob, b.topk_prob)
    assert torch.equal(y, b.y)
