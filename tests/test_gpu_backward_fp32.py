"""The layer backward of fp32 layers on the GPU against the oracle's backward.

For MOE_F32 every backward GEMM runs on the FMA units (the SIMT grouped
kernels: fc2's dgrad with W2 read in place, fc1's products recomputed with
the SwiGLU backward in the epilogue, fc1's dgrad over [W1 ; W3], the
per-expert wgrads) and every intermediate stays fp32, so the gradients meet
the fp32 forward's tolerance: each element within 1e-4 of (|exact| + RMS).
Cases: the tiny fp32 layer, ragged shapes (h = 136, f = 200), capacity drops,
sigmoid routing over 64 experts (the router's gradients stay on the FMA
units in fp32), and a shared expert (moe_backward_shared and
moe_shared_expert_backward).  Experts without rows get exact zeros.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import assert_close, gpu_config, gpu_stages, make_case, np_view, to_dev, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synthetic.WORKLOADS["tiny_fp32"],
    "ragged": synthetic.scaled("tiny_fp32", T=1000, h=136, f=200, seed=401),
    "drops": synthetic.scaled("tiny_fp32", T=700, capacity_factor=1.0, gate_bias="hot:2:3",
                              seed=402),
    "sigmoid_e64": synthetic.scaled("dsv3", T=300, h=64, f=48, E=64, k=4, dtype="f32",
                                    seed=403),
    "shared": synthetic.scaled("dsv3_shared", T=200, h=64, f=48, E=16, k=2, dtype="f32",
                               shared_f=72, seed=404),
}

NAMES = ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2")


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    import mixture_experts_layer_fp32_gb300 as moe
    w = CASES[request.param]
    inp, r = make_case(w)
    dy = torch.randn((w.T, w.h), generator=torch.Generator().manual_seed(410))
    d = to_dev(inp)
    b = gpu_stages(w, d)
    cfg = gpu_config(w)
    g = moe.Grads(cfg)
    for n in NAMES:  # every output is overwritten
        getattr(g, n).fill_(float("nan"))
    gs = None
    if w.shared_f:
        gs = moe.SharedGrads(cfg, w.shared_f)
        ws = moe.alloc_workspace_backward_shared(cfg, w.shared_f)
        moe.backward_shared(cfg, w.shared_f, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"],
                            d["W2"], d["W1s"], d["W3s"], d["W2s"], b, dy.cuda(), g, gs, ws)
    else:
        ws = moe.alloc_workspace_backward(cfg)
        moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b,
                     dy.cuda(), g, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    ref = oracle.backward(np_view(inp["x"]), np_view(inp["Wg"]), np_view(inp["W1"]),
                          np_view(inp["W3"]), np_view(inp["W2"]), w.k, w.score, r["topk_idx"],
                          r["topk_prob"], r["keep"], np_view(dy), np_view(inp["gate_bias"]),
                          np_view(inp["expert_bias"]))
    refs = None
    if w.shared_f:
        refs = oracle.shared_backward(np_view(inp["x"]), np_view(inp["W1s"]),
                                      np_view(inp["W3s"]), np_view(inp["W2s"]), np_view(dy))
    return w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs


def test_token_gradient_fp32(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    want = ref["dx"] + (refs["dx"] if refs else 0.0)
    assert_close("dx", to_np(g.dx), want, "f32")


def test_router_gradients_fp32(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    assert_close("dWg", to_np(g.dWg), ref["dWg"], "f32")
    assert_close("dgate_bias", to_np(g.dgate_bias), ref["dgate_bias"], "f32")


def test_expert_weight_gradients_fp32(case):
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    for n in ("dW1", "dW3", "dW2"):
        got = to_np(getattr(g, n))
        for e in range(w.E):
            if r["tokens_per_expert"][e] == 0:
                assert np.all(got[e] == 0.0), (n, e)
            else:
                assert_close("%s[%d]" % (n, e), got[e], ref[n][e], "f32")


def test_shared_gradients_fp32(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    if not w.shared_f:
        pytest.skip("no shared expert")
    for n in ("dW1s", "dW3s", "dW2s"):
        assert_close(n, to_np(getattr(gs, n)), refs[n], "f32")
    # the shared expert's backward alone adds its dx to a caller buffer
    start = torch.full((w.T, w.h), 0.5, dtype=torch.float32, device="cuda")
    acc = start.clone()
    gs2 = moe.SharedGrads(cfg, w.shared_f)
    moe.shared_expert_backward(cfg, w.shared_f, d["x"], d["W1s"], d["W3s"], d["W2s"], b.h_mid_s,
                               dy.cuda(), acc, gs2, ws)
    moe.check(ws)
    assert_close("dx_s", to_np(acc - start), refs["dx"], "f32")
    for n in ("dW1s", "dW3s", "dW2s"):
        assert torch.equal(getattr(gs2, n), getattr(gs, n)), n


def test_backward_fp32_is_deterministic(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, d, b, dy, cfg, g, gs, ws, ref, refs = case
    if w.shared_f:
        pytest.skip("covered by the routed cases")
    g2 = moe.Grads(cfg)
    moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b, dy.cuda(),
                 g2, ws)
    moe.check(ws)
    for n in NAMES:
        assert torch.equal(getattr(g, n), getattr(g2, n)), n
