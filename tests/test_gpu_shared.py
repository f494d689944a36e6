"""The shared expert (one SwiGLU MLP every token goes through, added to the
routed output) against the oracle: the staged calls (moe_shared_expert +
moe_combine_shared) on the bf16 tensor-core path and the fp32 SIMT path,
moe_forward_shared (shared path on the library's second stream) reproducing
the staged output bit for bit, and the degenerate batches."""

import pytest
import torch

import synthetic
from moe_cases import compare_all, gpu_forward, gpu_stages, make_case, oracle_forward, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # fs spans three 128-column fc1 tiles; T spans several pair tiles plus a tail
    "dsv3_shared_small": synthetic.scaled("dsv3_shared", T=900, h=512, f=256, E=32,
                                          shared_f=384, seed=81),
    # fewer than 768 rows: the single-SM kernel, T not a multiple of 128
    "mixtral_shared_small": synthetic.scaled("mixtral", T=300, h=256, f=128, shared_f=256,
                                             seed=82),
    "tiny_fp32_shared": synthetic.scaled("tiny_fp32", T=200, h=136, f=200, shared_f=72, seed=83),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    return w, inp, ref, dinp, b


def test_shared_stages_match_oracle(case):
    w, inp, ref, dinp, b = case
    compare_all(w, inp, ref, b)


def test_forward_shared_reproduces_stages(case):
    w, inp, ref, dinp, b = case
    y, idx, prob, tpe = gpu_forward(w, dinp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(prob, b.topk_prob)
    assert torch.equal(y, b.y)


def test_forward_shared_repeated_calls_are_deterministic(case):
    w, inp, ref, dinp, b = case
    y1 = gpu_forward(w, dinp)[0]
    y2 = gpu_forward(w, dinp)[0]
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T", [0, 1])
def test_shared_degenerate_batches(T):
    w = synthetic.scaled("mixtral", T=T, h=256, f=128, shared_f=128, seed=84)
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    compare_all(w, inp, ref, b)
    y = gpu_forward(w, dinp)[0]
    assert torch.equal(y, b.y)
