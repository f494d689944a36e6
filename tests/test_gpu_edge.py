"""Edge cases of the GPU path against the oracle: empty and one-token
batches, every token on one expert (others empty), a single expert, k = E,
a capacity that cannot bind, min_capacity above the formula, and the
device-side index checks (bad ids are skipped and reported, never read)."""

import numpy as np
import pytest
import torch

import synthetic
from moe_cases import compare_all, gpu_config, gpu_stages, make_case, oracle_forward, to_dev, to_np

pytestmark = pytest.mark.gpu


def _run(w, tweak=None):
    inp, _ = make_case(w)
    if tweak:
        tweak(inp)
        from moe_cases import condition_inputs
        condition_inputs(w, inp)
    ref = oracle_forward(w, inp)
    b = gpu_stages(w, to_dev(inp))
    torch.cuda.synchronize()
    compare_all(w, inp, ref, b)
    return inp, ref, b


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_token(dtype):
    _run(synthetic.scaled("mixtral", T=1, h=256, f=128, dtype=dtype, seed=41))


def test_empty_batch():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=0, h=256, f=128, seed=42)
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    d = to_dev(synthetic.generate(w, device="cpu"))
    b.tokens_per_expert.fill_(7)
    moe.route(cfg, d["x"], d["Wg"], None, None, b.topk_idx, b.topk_prob, b.keep,
              b.tokens_per_expert, None, b.ws)
    moe.permute(cfg, d["x"], b.topk_idx, b.keep, b.x_perm, b.row_map, b.expert_offsets, b.ws)
    moe.grouped_mlp(cfg, b.x_perm, b.expert_offsets, d["W1"], d["W3"], d["W2"], b.h_mid,
                    b.y_perm, b.ws)
    moe.combine(cfg, b.y_perm, b.row_map, b.topk_prob, b.y)
    moe.forward(cfg, d["x"], d["Wg"], None, None, d["W1"], d["W3"], d["W2"], b.y, b.ws)
    moe.check(b.ws)
    assert int(b.tokens_per_expert.sum()) == 0
    assert int(b.expert_offsets.abs().sum()) == 0


def test_all_tokens_on_one_expert():
    # a large gate bias on expert 3: one expert gets every token, the rest are empty
    w = synthetic.scaled("qwen3", T=700, h=256, f=128, k=1, gate_bias=None, seed=43)

    def tweak(inp):
        gb = torch.zeros(w.E)
        gb[3] = 50.0
        inp["gate_bias"] = gb
    inp, ref, b = _run(w, tweak)
    tpe = to_np(b.tokens_per_expert)
    assert tpe[3] == w.T and tpe.sum() == w.T


def test_single_expert():
    _run(synthetic.scaled("mixtral", T=300, h=256, f=256, E=1, k=1, seed=44))


def test_topk_equals_num_experts():
    _run(synthetic.scaled("mixtral", T=333, h=256, f=128, E=4, k=4, seed=45))


def test_sigmoid_top8_of_8():
    _run(synthetic.scaled("dsv3", T=200, h=256, f=128, E=8, k=8, seed=46))


def test_capacity_that_cannot_bind():
    w = synthetic.scaled("switch", T=512, h=256, f=128, capacity_factor=200.0, seed=47)
    inp, ref, b = _run(w)
    assert ref["keep"].all()


def test_min_capacity_above_formula():
    w = synthetic.scaled("switch", T=2048, h=256, f=128, capacity_factor=0.05, min_capacity=40,
                         seed=48)
    inp, ref, b = _run(w)
    assert ref["capacity"] == 40
    assert to_np(b.tokens_per_expert).max() == 40


def test_fp32_many_experts_sigmoid():
    _run(synthetic.scaled("dsv3", T=160, h=64, f=48, dtype="f32", E=256, k=8, x_std=1.0,
                          seed=49))


def test_bad_expert_id_is_skipped_and_reported():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=64, h=256, f=128, seed=50)
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    x = torch.randn(w.T, w.h, device="cuda").to(torch.bfloat16)
    idx = torch.stack([torch.arange(w.T) % w.E, (torch.arange(w.T) + 1) % w.E], 1).int().cuda()
    idx[5, 1] = w.E          # out of range
    idx[9, 0] = -3           # out of range
    moe.permute(cfg, x, idx, None, b.x_perm, b.row_map, b.expert_offsets, b.ws)
    with pytest.raises(moe.MoeError) as ei:
        moe.check(b.ws)
    assert ei.value.code == 5  # MOE_ERR_DEVICE_CHECK
    rm = to_np(b.row_map)
    assert rm[5, 1] == -1 and rm[9, 0] == -1
    assert int(b.expert_offsets[-1]) == 2 * w.T - 2
    moe.check(b.ws)  # cleared by the previous read


def test_inconsistent_offsets_are_rejected_by_the_gemm():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=64, h=256, f=128, seed=51)
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    d = to_dev(synthetic.generate(w, device="cpu"))
    bad = torch.tensor([0, 10, 5, 20, 30, 40, 50, 60, 64], dtype=torch.int32, device="cuda")
    b.h_mid.fill_(1.0)
    moe.grouped_fc1(cfg, b.x_perm, bad, d["W1"], d["W3"], b.h_mid, b.ws)
    with pytest.raises(moe.MoeError) as ei:
        moe.check(b.ws)
    assert ei.value.code == 5
    assert bool((b.h_mid == 1.0).all())  # nothing written
    too_many = torch.tensor([0, 10, 20, 30, 40, 50, 60, 64, 129], dtype=torch.int32,
                            device="cuda")   # beyond the T*k rows of the buffers
    moe.grouped_fc2(cfg, b.h_mid, too_many, d["W2"], b.y_perm, b.ws)
    with pytest.raises(moe.MoeError):
        moe.check(b.ws)
