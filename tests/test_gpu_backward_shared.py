"""The layer backward with a shared expert on the GPU against the oracle.

moe_backward_shared: the routed gradients plus the shared expert's, dx
holding both paths before its one rounding; moe_shared_expert_backward: the
shared expert alone, its dx added to a caller fp32 buffer.  The oracle is the
routed backward plus oracle.shared_backward (the routed formula for one
expert of weight 1, pinned by finite differences of the forward with its
shared expert).  Criteria as in test_gpu_backward.py: relative L2 error <=
1e-2 per gradient, every element within 0.15 of the gradient's RMS.  Cases:
a DeepSeek-V3-like layer with fs % 256 == 128 (a half last tile in the
shared fc2 dgrad) and a Mixtral-like one with T >= 768 (the shared GEMMs on
SM pairs by the automatic rule); each with the GEMMs forced onto single SMs
and onto SM pairs.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import gpu_config, gpu_stages, make_case, np_view, rms, to_dev, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "dsv3_fs384": synthetic.scaled("dsv3_shared", T=400, h=512, f=256, E=32, k=4, shared_f=384,
                                   seed=181),
    "mixtral_fs256": synthetic.scaled("mixtral", T=900, h=512, f=256, E=4, shared_f=256,
                                      seed=182),
}


def _assert_grad(name, got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, name
    assert np.all(np.isfinite(got)), name
    r = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert r <= 1e-2, "%s: relative L2 error %g > 1e-2" % (name, r)
    err = np.abs(got - want).max()
    assert err <= 0.15 * rms(want), "%s: max error %g > 0.15 * RMS %g" % (name, err, rms(want))


@pytest.fixture(scope="module",
                params=[(n, k) for n in sorted(CASES) for k in ("single", "pair")],
                ids=lambda p: "%s-%s" % p)
def case(request):
    import mixture_experts_layer_fp32_gb300 as moe
    name, kernel = request.param
    w = CASES[name]
    inp, r = make_case(w)
    gen = torch.Generator().manual_seed(190)
    dy = torch.randn((w.T, w.h), generator=gen).to(torch.bfloat16)
    d = to_dev(inp)
    b = gpu_stages(w, d)
    cfg = gpu_config(w)
    g, gs = moe.Grads(cfg), moe.SharedGrads(cfg, w.shared_f)
    ws = moe.alloc_workspace_backward_shared(cfg, w.shared_f)
    with pytest.MonkeyPatch.context() as mp:
        mp.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
        moe.backward_shared(cfg, w.shared_f, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"],
                            d["W2"], d["W1s"], d["W3s"], d["W2s"], b, dy.cuda(), g, gs, ws)
        moe.check(ws)
        torch.cuda.synchronize()
    ref = oracle.backward(np_view(inp["x"]), np_view(inp["Wg"]), np_view(inp["W1"]),
                          np_view(inp["W3"]), np_view(inp["W2"]), w.k, w.score, r["topk_idx"],
                          r["topk_prob"], r["keep"], np_view(dy), np_view(inp["gate_bias"]),
                          np_view(inp["expert_bias"]))
    refs = oracle.shared_backward(np_view(inp["x"]), np_view(inp["W1s"]), np_view(inp["W3s"]),
                                  np_view(inp["W2s"]), np_view(dy))
    return w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs


def test_token_gradient_with_shared_expert(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    _assert_grad("dx", to_np(g.dx), ref["dx"] + refs["dx"])


def test_shared_weight_gradients(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    for n in ("dW1s", "dW3s", "dW2s"):
        _assert_grad(n, to_np(getattr(gs, n)), refs[n])


def test_routed_gradients_unchanged_by_the_shared_path(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    for n in ("dWg", "dgate_bias", "dW1", "dW3", "dW2"):
        _assert_grad(n, to_np(getattr(g, n)), ref[n])


def test_shared_expert_backward_alone_adds_to_dx(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    start = torch.full((w.T, w.h), 0.25, dtype=torch.float32, device="cuda")
    acc = start.clone()
    gs2 = moe.SharedGrads(cfg, w.shared_f)
    moe.shared_expert_backward(cfg, w.shared_f, d["x"], d["W1s"], d["W3s"], d["W2s"], b.h_mid_s,
                               dy.cuda(), acc, gs2, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    _assert_grad("dx_s", to_np(acc - start), refs["dx"])
    # the same kernels as inside moe_backward_shared (automatic kernel choice)
    for n in ("dW1s", "dW3s", "dW2s"):
        _assert_grad(n, to_np(getattr(gs2, n)), refs[n])


def test_backward_shared_is_deterministic(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    outs = []
    for _ in range(2):
        g2, gs2 = moe.Grads(cfg), moe.SharedGrads(cfg, w.shared_f)
        moe.backward_shared(cfg, w.shared_f, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"],
                            d["W2"], d["W1s"], d["W3s"], d["W2s"], b, dy.cuda(), g2, gs2, ws)
        outs.append((g2, gs2))
    torch.cuda.synchronize()
    for n in ("dx", "dWg", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(outs[0][0], n), getattr(outs[1][0], n)), n
    for n in ("dW1s", "dW3s", "dW2s"):
        assert torch.equal(getattr(outs[0][1], n), getattr(outs[1][1], n)), n
