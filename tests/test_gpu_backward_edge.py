"""Edge cases of the layer backward on the GPU against the oracle's backward:
an empty batch (every gradient zero), one token, every token on one expert
(the others get exact zeros), a single expert (softmax over one logit: no
router gradient), k = E, and sigmoid top-8 of 8.  Criteria as in
test_gpu_backward.py (relative L2 <= 1e-2, elements within 0.15 of the RMS),
with the RMS taken over the entries the oracle makes nonzero: with one token
most experts have no rows, and their exact zeros (checked as such) would
shrink a whole-array RMS.  Gradients the oracle makes exactly zero must be
exactly zero."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import gpu_config, gpu_stages, make_case, np_view, rms, to_dev, to_np

pytestmark = pytest.mark.gpu

NAMES = ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2")


def _assert_grad(name, got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, name
    assert np.all(np.isfinite(got)), name
    if not np.any(want):
        assert not np.any(got), "%s: expected exact zeros" % name
        return
    r = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert r <= 1e-2, "%s: relative L2 error %g > 1e-2" % (name, r)
    assert not np.any(got[want == 0]), "%s: nonzero where the oracle is exactly zero" % name
    scale = rms(want[want != 0])
    err = np.abs(got - want).max()
    assert err <= 0.15 * scale, "%s: max error %g > 0.15 * RMS %g" % (name, err, scale)


def _backward(w, tweak=None):
    import mixture_experts_layer_fp32_gb300 as moe
    inp, r = make_case(w)
    if tweak:
        tweak(inp)
        from moe_cases import condition_inputs
        r = condition_inputs(w, inp)
    d = to_dev(inp)
    b = gpu_stages(w, d)
    cfg = gpu_config(w)
    dy = torch.randn((w.T, w.h), generator=torch.Generator().manual_seed(200)).to(torch.bfloat16)
    g = moe.Grads(cfg)
    for n in NAMES:  # every output is overwritten
        getattr(g, n).fill_(float("nan"))
    ws = moe.alloc_workspace_backward(cfg)
    moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b, dy.cuda(),
                 g, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    ref = oracle.backward(np_view(inp["x"]), np_view(inp["Wg"]), np_view(inp["W1"]),
                          np_view(inp["W3"]), np_view(inp["W2"]), w.k, w.score, r["topk_idx"],
                          r["topk_prob"], r["keep"], np_view(dy), np_view(inp["gate_bias"]),
                          np_view(inp["expert_bias"]))
    for n in NAMES:
        _assert_grad(n, to_np(getattr(g, n)), ref[n])
    return r, g, ref


def test_backward_empty_batch():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=0, h=256, f=128, seed=201)
    cfg = gpu_config(w)
    d = to_dev(synthetic.generate(w, device="cpu"))
    b = gpu_stages(w, d)
    g = moe.Grads(cfg)
    for n in NAMES:
        getattr(g, n).fill_(float("nan"))
    ws = moe.alloc_workspace_backward(cfg)
    dy = torch.empty((0, w.h), dtype=torch.bfloat16, device="cuda")
    moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b, dy, g, ws)
    moe.check(ws)
    for n in NAMES[1:]:  # no tokens: every parameter gradient is zero
        assert not torch.any(getattr(g, n)), n


def test_backward_one_token():
    _backward(synthetic.scaled("mixtral", T=1, h=256, f=128, seed=202))


def test_backward_all_tokens_on_one_expert():
    w = synthetic.scaled("qwen3", T=700, h=256, f=128, k=1, gate_bias=None, seed=203)

    def tweak(inp):
        gb = torch.zeros(w.E)
        gb[3] = 50.0
        inp["gate_bias"] = gb
    r, g, ref = _backward(w, tweak)
    assert r["tokens_per_expert"][3] == w.T
    others = [e for e in range(w.E) if e != 3]
    for n in ("dW1", "dW3", "dW2"):
        assert not torch.any(getattr(g, n)[others]), n


def test_backward_single_expert():
    r, g, ref = _backward(synthetic.scaled("mixtral", T=300, h=256, f=256, E=1, k=1, seed=204))
    assert not torch.any(g.dWg)  # softmax over one logit: no router gradient


def test_backward_topk_equals_num_experts():
    _backward(synthetic.scaled("mixtral", T=333, h=256, f=128, E=4, k=4, seed=205))


def test_backward_sigmoid_top8_of_8():
    _backward(synthetic.scaled("dsv3", T=200, h=256, f=128, E=8, k=8, seed=206))
