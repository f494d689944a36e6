"""Failure detection on the GPU without a GPU fault: a bounded wait is made to
run out (a barrier nothing signals), the kernel returns, the error word in
the workspace reports MOE_ERR_TIMEOUT through moe_check, and the context is
still usable for a normal forward afterwards."""

import pytest
import torch

import synthetic
from moe_cases import assert_close, gpu_stages, make_case, oracle_forward, to_dev, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import mixture_experts_layer_fp32_gb300 as moe
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    moe.selftest_wait_timeout(ws, 2_000_000)           # ~1 ms of SM cycles
    with pytest.raises(moe.MoeError) as ei:
        moe.check(ws)
    assert ei.value.code == 6                           # MOE_ERR_TIMEOUT
    moe.check(ws)                                       # the word was cleared
    # the context still runs the layer correctly
    w = synthetic.scaled("mixtral", T=200, h=256, f=128, seed=61)
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    b = gpu_stages(w, to_dev(inp))
    torch.cuda.synchronize()
    assert_close("y", to_np(b.y), ref["y"], w.dtype)


def test_timeout_reports_once_for_repeated_failures():
    import mixture_experts_layer_fp32_gb300 as moe
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        moe.selftest_wait_timeout(ws, 100_000)
    with pytest.raises(moe.MoeError) as ei:
        moe.check(ws)
    assert ei.value.code == 6
