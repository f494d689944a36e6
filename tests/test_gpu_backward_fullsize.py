"""The layer backward at the Mixtral-shaped workload's full size (T=8192,
h=4096, E=8, top-2, f=14336), in the launch configuration `bench.py --pass
backward` times: moe_backward after the staged forward, with the SM-pair
dgrad / recompute / wgrad kernels and the small-E router kernels.

The oracle cannot form the whole backward at this size (each expert's weight
gradient alone is ~2048 rows x 4096 x 14336 products in double), so it checks
samples against its own routing and permutation:
  * dx of a seeded sample of tokens: a token's dx depends on that token
    alone, so the oracle backward over the sample gives it exactly;
  * whole rows dW2[e][c, :] and whole columns dW1[e][:, c], dW3[e][:, c] for
    seeded (e, c), from all of expert e's rows;
with the criteria of the small-size backward tests (relative L2 error <=
1e-2, every element within 0.15 of the sample's RMS).  Also: every gradient
finite, and a second backward bitwise identical.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import condition_inputs, gpu_config, gpu_stages, np_view, rms, to_np

pytestmark = pytest.mark.gpu

N_TOKENS = 16
N_EXPERTS = 2
N_COLS = 3


def _host(t):
    """A device tensor (or None) as the oracle's numpy input."""
    return None if t is None else np_view(t.cpu())


def _rel_l2(got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    return np.linalg.norm(got - want) / np.linalg.norm(want)


def _assert_grad(name, got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), name
    r = _rel_l2(got, want)
    assert r <= 1e-2, "%s: relative L2 error %g > 1e-2" % (name, r)
    err = np.abs(got - want).max()
    assert err <= 0.15 * rms(want), "%s: max error %g > 0.15 * RMS %g" % (name, err, rms(want))


@pytest.fixture(scope="module")
def full():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.WORKLOADS["mixtral"]
    torch.cuda.empty_cache()
    inp = synthetic.generate(w, device="cuda")
    r = condition_inputs(w, inp)
    b = gpu_stages(w, inp, with_routing_map=False)
    gen = torch.Generator().manual_seed(w.seed + 7)
    dy = torch.randn((w.T, w.h), generator=gen).to(torch.bfloat16)
    cfg = gpu_config(w)
    g = moe.Grads(cfg)
    ws = moe.alloc_workspace_backward(cfg)
    moe.backward(cfg, inp["x"], inp["Wg"], inp["gate_bias"], inp["W1"], inp["W3"], inp["W2"], b,
                 dy.cuda(), g, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    yield w, inp, r, b, dy, cfg, g, ws
    del inp, b, g, ws
    torch.cuda.empty_cache()


def test_gradients_finite_full(full):
    w, inp, r, b, dy, cfg, g, ws = full
    for n in ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2"):
        assert bool(torch.isfinite(getattr(g, n).float()).all()), n


def test_sampled_token_gradients_full(full):
    w, inp, r, b, dy, cfg, g, ws = full
    toks = np.sort(np.random.default_rng(2024).choice(w.T, N_TOKENS, replace=False))
    tsel = torch.from_numpy(toks).to(inp["x"].device)
    x_s = _host(inp["x"][tsel])
    W = {n: _host(inp[n]) for n in ("W1", "W3", "W2")}
    ref = oracle.backward(x_s, _host(inp["Wg"]), W["W1"], W["W3"], W["W2"], w.k, w.score,
                          r["topk_idx"][toks], r["topk_prob"][toks], r["keep"][toks],
                          np_view(dy[torch.from_numpy(toks)]), _host(inp.get("gate_bias")),
                          _host(inp.get("expert_bias")), weight_grads=False)
    _assert_grad("dx (sampled tokens)", to_np(g.dx[tsel]), ref["dx"])


def test_sampled_weight_gradients_full(full):
    w, inp, r, b, dy, cfg, g, ws = full
    offsets, row_map, row_token = oracle.permute(r["topk_idx"], r["keep"], w.E)
    rng = np.random.default_rng(2025)
    x_all = _host(inp["x"])
    dy_all = np_view(dy)
    for e in sorted(rng.choice(w.E, N_EXPERTS, replace=False)):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        assert hi > lo
        tok = row_token[lo:hi]
        # the slot of each row, for its combine weight
        slot = np.array([int(np.nonzero(row_map[t] == q)[0][0]) for q, t in zip(range(lo, hi), tok)])
        p = r["topk_prob"][tok, slot].astype(np.float32)
        cols = np.sort(rng.choice(w.f, N_COLS, replace=False))
        rows_c = np.sort(rng.choice(w.f, N_COLS, replace=False))
        ref = oracle.expert_wgrad_cols(x_all[tok], p, dy_all[tok], _host(inp["W1"][e]),
                                       _host(inp["W3"][e]), _host(inp["W2"][e]), rows_c, cols)
        for q, c in enumerate(rows_c):
            _assert_grad("dW2[%d][%d, :]" % (e, c), to_np(g.dW2[e, c]), ref["dW2_rows"][q])
        for q, c in enumerate(cols):
            _assert_grad("dW1[%d][:, %d]" % (e, c), to_np(g.dW1[e, :, c]), ref["dW1_cols"][:, q])
            _assert_grad("dW3[%d][:, %d]" % (e, c), to_np(g.dW3[e, :, c]), ref["dW3_cols"][:, q])


def test_backward_deterministic_full(full):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, b, dy, cfg, g, ws = full
    g2 = moe.Grads(cfg)
    moe.backward(cfg, inp["x"], inp["Wg"], inp["gate_bias"], inp["W1"], inp["W3"], inp["W2"], b,
                 dy.cuda(), g2, ws)
    moe.check(ws)
    torch.cuda.synchronize()
    for n in ("dx", "dWg", "dgate_bias", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(g, n), getattr(g2, n)), n
