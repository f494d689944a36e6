"""The C-ABI calls captured into CUDA graphs and replayed.

The library's calls only enqueue work on the given stream (one-time set-up
-- kernel attributes, the cluster occupancy query, the driver entry point --
happens on a first call, made here before capture; tensor maps are kernel
parameters by value; the shared expert forks to the library's second stream
and joins back with events, which stream capture records as graph edges).
So a forward, a forward with the shared expert and a backward can be
captured once and replayed: each replay must give bit for bit what a direct
call gives, also after the inputs are rewritten in place between replays.
"""

import pytest
import torch

import synthetic
from moe_cases import gpu_config, gpu_stages, make_case, to_dev

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Capture fn() into a CUDA graph on a side stream (after one direct call)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _redraw(t, seed):
    gen = torch.Generator().manual_seed(seed)
    t.copy_(torch.randn(t.shape, generator=gen).to(t.dtype))


@pytest.mark.parametrize("name,w", [
    ("mixtral", synthetic.scaled("mixtral", T=1000, h=512, f=256, E=4, seed=301)),
    ("dsv3_shared", synthetic.scaled("dsv3_shared", T=300, h=512, f=256, E=32, k=4,
                                     shared_f=256, seed=302)),
])
def test_forward_replays_in_a_graph(name, w):
    import mixture_experts_layer_fp32_gb300 as moe
    inp, _ = make_case(w)
    d = to_dev(inp)
    cfg = gpu_config(w)
    fs = w.shared_f
    ws = moe.alloc_workspace_shared(cfg, fs) if fs else moe.alloc_workspace(cfg)
    y = torch.empty((w.T, w.h), dtype=moe.act_dtype(cfg), device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    prob = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    tpe = torch.empty((w.E,), dtype=torch.int32, device="cuda")

    def fwd():
        if fs:
            moe.forward_shared(cfg, fs, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], d["W1"],
                               d["W3"], d["W2"], d["W1s"], d["W3s"], d["W2s"], y, ws, idx, prob,
                               tpe)
        else:
            moe.forward(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], d["W1"], d["W3"],
                        d["W2"], y, ws, idx, prob, tpe)

    g = _capture(fwd)
    for rnd in range(3):
        if rnd:
            _redraw(d["x"], 310 + rnd)   # new tokens in the captured buffer
        fwd()
        moe.check(ws)
        want = (y.clone(), idx.clone(), prob.clone(), tpe.clone())
        for t in (y, idx, prob, tpe):
            t.zero_()
        g.replay()
        moe.check(ws)
        for got, ref in zip((y, idx, prob, tpe), want):
            assert torch.equal(got, ref), name


def test_backward_replays_in_a_graph():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("qwen3", T=400, h=256, f=256, E=64, seed=303)  # tensor-core router grads
    inp, _ = make_case(w)
    d = to_dev(inp)
    b = gpu_stages(w, d)
    cfg = gpu_config(w)
    dy = torch.randn((w.T, w.h), generator=torch.Generator().manual_seed(304)).to(
        torch.bfloat16).cuda()
    grads = moe.Grads(cfg)
    ws = moe.alloc_workspace_backward(cfg)

    def bwd():
        moe.backward(cfg, d["x"], d["Wg"], d["gate_bias"], d["W1"], d["W3"], d["W2"], b, dy,
                     grads, ws)

    g = _capture(bwd)
    names = ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2")
    for rnd in range(2):
        if rnd:
            _redraw(dy, 305)
        bwd()
        moe.check(ws)
        want = {n: getattr(grads, n).clone() for n in names}
        for n in names:
            getattr(grads, n).zero_()
        g.replay()
        moe.check(ws)
        for n in names:
            assert torch.equal(getattr(grads, n), want[n]), n
