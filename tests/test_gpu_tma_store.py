"""The two stores of the grouped GEMM's fp32 and fp16 outputs give the same bits.

fc2's y_perm (fp32, or fp16 with a scale per 32 columns for bf16 top-k
layers), the E4M3 fc2's y_perm and the backward's fp32 dx (fc1's dgrad
over [W1 ; W3], and the router's dx on the dense tensor-core path) leave the
accumulator either through TMA tile stores of 32 x 32 blocks (a warp whose 32
rows all belong to the tile's expert) or through masked row-segment stores (a
warp whose rows cross the expert's end, or an accumulating dgrad).  Each
output element is the same fp32 accumulator value either way, so the layer
run with MOE_TC_TMA_OUT=0 (row-segment stores only) and with the default
must agree bit for bit, on the one-SM kernel and on SM pairs.  Parity with the
oracle is covered by the forward, E4M3 and backward parity tests; here the
shapes put expert ends inside and at the edges of 32-row warps (ragged
offsets) and include an expert with no rows.
"""

import pytest
import torch

import synthetic
from moe_cases import gpu_config, gpu_stages, make_case, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # ragged offsets: most experts end inside a 32-row warp
    "mixtral_ragged": synthetic.scaled("mixtral", T=777, h=512, f=384, seed=501),
    # 64 experts, 4 of them hot: many row blocks of whole warps, some experts empty
    "dsv3_hot": synthetic.scaled("dsv3", T=512, h=512, f=256, E=64, k=4,
                                 gate_bias="hot:4:3", seed=502),
    # every expert padded to its capacity of 320 rows: only whole warps
    "switch_pad": synthetic.scaled("switch", T=2048, h=256, f=256, E=8, seed=503,
                                   pad_to_capacity=True),
}


def _forward(w, d, mp, tma, kernel):
    mp.setenv("MOE_TC_TMA_OUT", "1" if tma else "0")
    mp.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
    b = gpu_stages(w, d)
    torch.cuda.synchronize()
    return b


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_stores_agree(name, kernel):
    w = CASES[name]
    inp, _ = make_case(w)
    d = to_dev(inp)
    with pytest.MonkeyPatch.context() as mp:
        a = _forward(w, d, mp, True, kernel)
        b = _forward(w, d, mp, False, kernel)
    R = int(a.expert_offsets[-1])
    assert R > 0
    assert torch.equal(a.expert_offsets, b.expert_offsets)
    assert torch.equal(a.y_perm[:R], b.y_perm[:R])
    if hasattr(a, "y16"):  # the fp16 y_perm: 32 x 64 TMA boxes or per-lane row stores
        assert torch.equal(a.y16[:R].view(torch.int16), b.y16[:R].view(torch.int16))
        assert torch.equal(a.y16_exp[:R], b.y16_exp[:R])
    assert torch.equal(a.y, b.y)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_e4m3_forward_stores_agree(kernel):
    import mixture_experts_layer_fp32_gb300 as moe
    w = CASES["mixtral_ragged"]
    inp, _ = make_case(w)
    d = to_dev(inp)
    cfg = gpu_config(w)
    q = moe.E4m3Experts(cfg, d["W1"], d["W3"], d["W2"])
    ws = moe.alloc_workspace_e4m3(cfg)
    outs = []
    with pytest.MonkeyPatch.context() as mp:
        mp.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
        for tma in (True, False):
            mp.setenv("MOE_TC_TMA_OUT", "1" if tma else "0")
            y = torch.empty((w.T, w.h), dtype=moe.act_dtype(cfg), device="cuda")
            moe.forward_e4m3(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], q, y, ws)
            moe.check(ws)
            torch.cuda.synchronize()
            outs.append(y)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("name", ["mixtral_ragged", "dsv3_hot"])
def test_backward_stores_agree(name, kernel):
    import mixture_experts_layer_fp32_gb300 as moe
    w = CASES[name]
    inp, _ = make_case(w)
    d = to_dev(inp)
    cfg = gpu_config(w)
    dy = torch.randn((w.T, w.h), generator=torch.Generator().manual_seed(510)).to(
        moe.act_dtype(cfg)).cuda()
    grads = []
    with pytest.MonkeyPatch.context() as mp:
        for tma in (True, False):
            b = _forward(w, d, mp, tma, kernel)
            g = moe.Grads(cfg)
            ws = moe.alloc_workspace_backward(cfg)
            moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b, dy,
                         g, ws)
            moe.check(ws)
            torch.cuda.synchronize()
            grads.append(g)
    for n in ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(grads[0], n), getattr(grads[1], n)), n
