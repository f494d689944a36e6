"""fc2 with the combine in its epilogue (moe_grouped_fc2_combine), on the
GPU through the C ABI.

The combine is y[t] = sum over kept slots j, in slot order, of
p[t,j] * Y[row(t,j)], in fp32, rounded once to the output dtype (0 for a
token with no kept slot): the Megatron Core walkthrough
(r00kie-liu.github.io), section 10 Experts and section 2 (the combine).
Top-1 rows go, weighted, straight to their token's output row; with k >= 2
the epilogue that stores the last of a token's rows sums them.  Either way
the arithmetic is the combine kernel's, so the output must equal
moe_grouped_fc2 followed by moe_combine bit for bit, on both tensor-core
kernels, with every dropped token's row zero; and it is checked against
the oracle.
"""

import numpy as np
import pytest
import torch

import synthetic
from moe_cases import assert_close, gpu_config, gpu_stages, make_case, oracle_forward, to_dev
from moe_cases import to_np

pytestmark = pytest.mark.gpu

CASES = {
    # Switch-shaped: four hot experts over capacity, so tokens are dropped
    "switch_drop": synthetic.scaled("switch", T=4096, h=512, f=256, seed=61),
    # one hot expert with ~7000 candidates (the drop's keys re-read), few experts
    "switch_one_hot": synthetic.scaled("switch", T=12000, h=256, f=256, E=8, seed=62,
                                       gate_bias="hot:1:4.6"),
    # top-1 without drops: every token has a row; ~1000 rows per expert (pair tiles)
    "top1_dropless": synthetic.scaled("mixtral", T=4000, h=256, f=384, E=4, k=1, seed=63),
    # fp32: the two kernels behind the same call
    "top1_fp32": synthetic.scaled("tiny_fp32", T=700, h=136, f=200, k=1, seed=64),
    # top-2, ~1000 rows per expert, 4 n-tiles of fc2: rows of a token in different tiles
    "top2": synthetic.scaled("mixtral", T=2000, h=1024, f=256, E=4, seed=65),
    # top-8 over 128 experts with Zipf loads: eight rows per token to add up
    "top8_zipf": synthetic.scaled("qwen3", T=1500, h=512, f=256, seed=66),
    # top-8 sigmoid with the selection bias, 64 experts
    "top8_sigmoid": synthetic.scaled("dsv3", T=600, h=768, f=256, E=64, seed=67),
    # top-2 with capacity drops: tokens with one kept slot and with none
    "top2_drop": synthetic.scaled("switch", T=3000, h=256, f=256, E=8, k=2, seed=68,
                                  capacity_factor=0.6),
    # fp32 top-2: fc2 and the combine kernel behind the same call
    "top2_fp32": synthetic.scaled("tiny_fp32", T=500, h=136, f=200, seed=69),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    d = to_dev(inp)
    b = gpu_stages(w, d)  # route, permute, fc1, fc2, combine (unfused)
    torch.cuda.synchronize()
    return w, inp, ref, d, b


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_fused_equals_fc2_then_combine(case, kernel, monkeypatch):
    # gpu_stages ran the staged calls the forward uses: fc2 + combine over the
    # fp32 y_perm (top-1, fp32), or fc2_f16s + combine_f16s (bf16, k >= 2)
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, ref, d, b = case
    monkeypatch.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
    cfg = gpu_config(w)
    for _ in range(2):  # a second call on the same workspace gives the same bits
        y = torch.full_like(b.y, float("nan"))
        moe.grouped_fc2_combine(cfg, b.h_mid, b.expert_offsets, d["W2"], b.row_map, b.topk_prob,
                                y, b.ws)
        moe.check(b.ws)
        bits = torch.int16 if y.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(y.view(bits), b.y.view(bits))
    dropped = (to_np(b.keep) == 0).all(axis=1)
    if w.capacity_factor > 0:
        assert dropped.any()
    assert (to_np(y)[dropped] == 0).all()
    assert_close("y", to_np(y), ref["y"], w.dtype)


def _decode(y16, y16_exp):
    """Values of the fp16 y_perm: fp16 * 2^exp per 32-column chunk (float64)."""
    v = y16.double().cpu()
    e = torch.repeat_interleave(y16_exp.cpu().long(), 32, dim=1)
    return (v * torch.pow(2.0, e.double())).numpy()


def test_f16s_y_perm_against_fp32(case):
    # the fp16 y_perm against the fp32 one from the same fc2 products: each chunk's
    # scale puts its largest magnitude in [2^14, 2^15] (2^15 when it rounds up to
    # it), so every value is within
    # 2^-11 of its magnitude (round to nearest fp16) plus the fp16 underflow step
    w, inp, ref, d, b = case
    if not hasattr(b, "y16"):
        pytest.skip("this layer combines over the fp32 y_perm")
    R = int(b.expert_offsets[-1].item())
    got = _decode(b.y16[:R], b.y16_exp[:R])
    want = to_np(b.y_perm[:R]).astype(np.float64)
    chunk_max = np.abs(want).reshape(R, -1, 32).max(axis=2)
    floor = np.repeat(chunk_max * 2.0 ** -29, 32, axis=1)
    assert (np.abs(got - want) <= 2.0 ** -11 * np.abs(want) + floor).all()
    h16 = np.abs(b.y16[:R].float().cpu().numpy()).reshape(R, -1, 32).max(axis=2)
    nz = chunk_max > 0
    assert ((h16[nz] >= 2.0 ** 14) & (h16[nz] <= 2.0 ** 15)).all()
