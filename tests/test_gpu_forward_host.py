"""moe_forward_host: batches in host memory, copies pipelined with compute
on the library's copy streams.  Every batch's output must equal moe_forward
on the same input bit for bit (the same kernels), whether batches have
their own host buffers or share one (stride 0)."""

import pytest
import torch

import synthetic
from moe_cases import gpu_config, make_case, to_dev

pytestmark = pytest.mark.gpu


def _inputs(w, batches):
    inp, _ = make_case(w)
    d = to_dev(inp)
    xs = [inp["x"]] + [synthetic.redraw_x_rows(w, 100 + b, w.T) for b in range(batches - 1)]
    return d, torch.stack([x.contiguous() for x in xs]).pin_memory()


def _device_forward(moe, cfg, d, x):
    ws = moe.alloc_workspace(cfg)
    y = torch.empty((cfg.num_tokens, cfg.hidden), dtype=moe.act_dtype(cfg), device="cuda")
    moe.forward(cfg, x.cuda(), d["Wg"], d["gate_bias"], d["expert_bias"], d["W1"], d["W3"],
                d["W2"], y, ws)
    moe.check(ws)
    return y.cpu()


@pytest.mark.parametrize("name,B", [("mixtral", 5), ("tiny_fp32", 3), ("switch", 4)])
def test_forward_host_batches_equal_forward(name, B):
    import mixture_experts_layer_fp32_gb300 as moe
    base = synthetic.WORKLOADS[name]
    w = base if name == "tiny_fp32" else synthetic.scaled(name, T=700, h=512, f=256, seed=101)
    cfg = gpu_config(w)
    d, x_host = _inputs(w, B)
    y_host = torch.full((B, w.T, w.h), float("nan"), dtype=x_host.dtype).pin_memory()
    ws = moe.alloc_workspace_host(cfg)
    moe.forward_host(cfg, x_host, y_host, d["Wg"], d["gate_bias"], d["expert_bias"], d["W1"],
                     d["W3"], d["W2"], ws)
    torch.cuda.current_stream().synchronize()
    moe.check(ws)
    for b in range(B):
        want = _device_forward(moe, cfg, d, x_host[b])
        assert torch.equal(y_host[b], want), b


def test_forward_host_stride_zero_reuses_buffers():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=300, h=256, f=128, seed=102)
    cfg = gpu_config(w)
    d, x_host = _inputs(w, 1)
    x1 = x_host[0].clone().pin_memory()
    y1 = torch.empty((w.T, w.h), dtype=x1.dtype).pin_memory()
    ws = moe.alloc_workspace_host(cfg)
    moe.forward_host(cfg, x1, y1, d["Wg"], d["gate_bias"], d["expert_bias"], d["W1"], d["W3"],
                     d["W2"], ws, num_batches=7)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(y1, _device_forward(moe, cfg, d, x1))


def test_forward_host_zero_batches_and_empty_tokens():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=0, h=256, f=128, seed=103)
    cfg = gpu_config(w)
    d = to_dev(synthetic.generate(w))
    x = torch.empty((2, 0, w.h), dtype=torch.bfloat16).pin_memory()
    y = torch.empty((2, 0, w.h), dtype=torch.bfloat16).pin_memory()
    ws = moe.alloc_workspace_host(cfg)
    moe.forward_host(cfg, x, y, d["Wg"], None, None, d["W1"], d["W3"], d["W2"], ws)
    moe.forward_host(cfg, x, y, d["Wg"], None, None, d["W1"], d["W3"], d["W2"], ws,
                     num_batches=0)
    torch.cuda.current_stream().synchronize()
    moe.check(ws)


def test_forward_host_shared_batches_equal_forward_shared():
    # the shared-expert variant: each batch forks the shared expert onto the
    # library's side stream inside the copy pipeline
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("dsv3_shared", T=300, h=512, f=256, E=32, k=4, shared_f=256, seed=111)
    cfg = gpu_config(w)
    B = 4
    d, x_host = _inputs(w, B)
    y_host = torch.full((B, w.T, w.h), float("nan"), dtype=x_host.dtype).pin_memory()
    ws = moe.alloc_workspace_host_shared(cfg, w.shared_f)
    moe.forward_host_shared(cfg, w.shared_f, x_host, y_host, d["Wg"], d["gate_bias"],
                            d["expert_bias"], d["W1"], d["W3"], d["W2"], d["W1s"], d["W3s"],
                            d["W2s"], ws)
    moe.check(ws)
    torch.cuda.synchronize()
    ws1 = moe.alloc_workspace_shared(cfg, w.shared_f)
    for b in range(B):
        y = torch.empty((w.T, w.h), dtype=moe.act_dtype(cfg), device="cuda")
        moe.forward_shared(cfg, w.shared_f, x_host[b].cuda(), d["Wg"], d["gate_bias"],
                           d["expert_bias"], d["W1"], d["W3"], d["W2"], d["W1s"], d["W3s"],
                           d["W2s"], y, ws1)
        moe.check(ws1)
        assert torch.equal(y_host[b], y.cpu()), b


def test_forward_host_e4m3_batches_equal_forward_e4m3():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=700, h=512, f=256, seed=112)
    cfg = gpu_config(w)
    B = 4
    d, x_host = _inputs(w, B)
    q = moe.E4m3Experts(cfg, d["W1"], d["W3"], d["W2"])
    y_host = torch.full((B, w.T, w.h), float("nan"), dtype=x_host.dtype).pin_memory()
    ws = moe.alloc_workspace_host_e4m3(cfg)
    moe.forward_host_e4m3(cfg, x_host, y_host, d["Wg"], d["gate_bias"], d["expert_bias"], q, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    ws1 = moe.alloc_workspace_e4m3(cfg)
    for b in range(B):
        y = torch.empty((w.T, w.h), dtype=moe.act_dtype(cfg), device="cuda")
        moe.forward_e4m3(cfg, x_host[b].cuda(), d["Wg"], d["gate_bias"], d["expert_bias"], q, y,
                         ws1)
        moe.check(ws1)
        assert torch.equal(y_host[b], y.cpu()), b
