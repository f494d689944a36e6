"""The opt-in router on the tensor cores (MOE_ROUTER_TC=1; bf16 layers with
more experts than the fused small-E kernel takes), on the GPU through the C
ABI.  The layer's default router stays on the CUDA cores (fp32 FMA).

The gating step computes logits = x . Wg with the router math in fp32 (the
Megatron Core walkthrough, r00kie-liu.github.io, section 3 Gating).  The
library splits each fp32 gate weight v into three bf16 pieces p0 + p1 + p2
(p0 = bf16(v), p1 = bf16(v - p0), p2 = bf16(v - p0 - p1); together they hold
v's 24 significant bits), multiplies the bf16 activations by each piece on
the tensor cores (products exact in fp32, fp32 accumulation) and adds the
three partial logits in piece order before the top-k.

  * a pin of the split itself: one-hot activation rows make each logit one
    gate weight, (p0 + p1) + p2 in fp32, which is v exactly; the weights of a
    row differ only in their lowest 6 significand bits, so a piece lost or
    misplaced turns the top-k into ties (or the wrong order) -- the
    expected experts and weights follow from Wg alone;
  * on the workloads' shapes the routing equals the oracle's bit for bit
    and the CUDA-core fp32 GEMM's (the default), weights within the parity
    tolerance; at the workloads' full sizes, against the oracle.
"""

import numpy as np
import pytest
import torch

import synthetic
from moe_cases import PROB_ATOL, PROB_RTOL, assert_equal, assert_probs, gpu_config, make_case
from moe_cases import oracle_forward, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_router(monkeypatch):
    monkeypatch.setenv("MOE_ROUTER_TC", "1")


def _route(w, d, cfg=None):
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = cfg or gpu_config(w)
    b = moe.Buffers(cfg)
    moe.route(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], b.topk_idx, b.topk_prob,
              b.keep, b.tokens_per_expert, None, b.ws)
    moe.check(b.ws)
    torch.cuda.synchronize()
    return b


@pytest.mark.parametrize("E,k,T", [(64, 4, 512), (256, 8, 300), (12, 3, 700), (128, 8, 129)])
def test_split_pieces_pin(E, k, T):
    import mixture_experts_layer_fp32_gb300 as moe
    h = 256
    rng = np.random.default_rng(1000 + E)
    # row kk of Wg: 1 + (a * 64 + perm(e)) * 2^-23, a random 17-bit prefix per
    # row: the experts of a row differ in the lowest 6 of the 23 fraction bits
    a = rng.integers(0, 1 << 17, size=(h, 1))
    perm = np.argsort(rng.random((h, E)), axis=1)
    m = a * 64 + perm
    Wg = (1.0 + m * 2.0 ** -23).astype(np.float32)
    assert np.array_equal((Wg.astype(np.float64) - 1.0) * 2.0 ** 23, m)  # exact in fp32
    rows = np.arange(T) % h
    x = np.zeros((T, h), np.float32)
    x[np.arange(T), rows] = 1.0
    cfg = moe.config(T, h, E, k, 128, score="softmax_post")
    d = {"x": torch.from_numpy(x).to(torch.bfloat16).cuda(),
         "Wg": torch.from_numpy(Wg).cuda(), "gate_bias": None, "expert_bias": None}
    b = _route(None, d, cfg)
    logits = Wg[rows].astype(np.float64)  # token t's logits: Wg row t % h, exactly
    want_idx = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert_equal("topk_idx", to_np(b.topk_idx), want_idx)
    sel = np.take_along_axis(logits, want_idx, axis=1)
    p = np.exp(sel - sel.max(axis=1, keepdims=True))
    assert_probs(to_np(b.topk_prob), p / p.sum(axis=1, keepdims=True))
    assert (to_np(b.tokens_per_expert) == np.bincount(want_idx.ravel(), minlength=E)).all()


CASES = {
    "qwen3": synthetic.scaled("qwen3", T=1000, h=512, f=128, seed=111),
    "dsv3_grouped": synthetic.scaled("dsv3_grouped", T=700, h=768, f=128, seed=112),
    "switch_drop": synthetic.scaled("switch", T=3000, h=256, f=128, seed=113),
    "E20_k3": synthetic.scaled("mixtral", T=901, h=512, f=128, E=20, k=3, seed=114),
    "sqrtsoftplus_E36": synthetic.scaled("dsv3", T=640, h=256, f=128, E=36, k=6,
                                         score="sqrtsoftplus", seed=115),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    assert w.dtype == "bf16" and w.E > 8 and w.E % 4 == 0
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp, want_h_mid=False)
    return w, inp, ref, to_dev(inp)


def test_tensor_core_router_matches_oracle(case):
    w, inp, ref, d = case
    b = _route(w, d)
    assert_equal("topk_idx", to_np(b.topk_idx), ref["topk_idx"])
    assert_equal("keep", to_np(b.keep), ref["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), ref["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), ref["topk_prob"])
    if w.capacity_factor > 0:
        assert (ref["keep"] == 0).any()


def test_tensor_core_router_matches_cuda_cores(case, monkeypatch):
    w, inp, ref, d = case
    tc = _route(w, d)
    monkeypatch.delenv("MOE_ROUTER_TC")
    cc = _route(w, d)
    assert torch.equal(tc.topk_idx, cc.topk_idx)
    assert torch.equal(tc.keep, cc.keep)
    assert torch.equal(tc.tokens_per_expert, cc.tokens_per_expert)
    got, want = to_np(tc.topk_prob).astype(np.float64), to_np(cc.topk_prob).astype(np.float64)
    assert np.all(np.abs(got - want) <= PROB_RTOL * np.abs(want) + PROB_ATOL)


@pytest.fixture(scope="module", params=["dsv3", "qwen3", "switch"])
def full(request):
    from moe_cases import condition_inputs
    w = synthetic.WORKLOADS[request.param]
    torch.cuda.empty_cache()
    inp = synthetic.generate(w, device="cuda")
    r = condition_inputs(w, inp)
    yield w, inp, r
    del inp
    torch.cuda.empty_cache()


def test_full_size_routing(full, monkeypatch):
    # the workloads' full sizes, with the K split the library picks (four
    # 1024-long accumulation chains at h = 4096, five at h = 7168, one at 1024)
    w, inp, r = full
    b = _route(w, inp)
    assert_equal("topk_idx", to_np(b.topk_idx), r["topk_idx"])
    assert_equal("keep", to_np(b.keep), r["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), r["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), r["topk_prob"])
