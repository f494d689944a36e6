"""The FP8 (E4M3) expert path against the oracle's FP8 arithmetic.

Bit-exact: the quantisers (per-row codes and power-of-two scales of x and
of bf16 matrices with crafted rounding ties; per-channel K-major codes of
the expert weights), the routing, the permutation and the permuted code
rows.  Within tolerance: the bf16 SwiGLU output (one bf16 ulp), its E4M3
codes (equal up to rare one-code flips where GPU and oracle round the
SwiGLU output differently), y_perm and y (2e-2 of the RMS beyond the
output's own rounding, plus, where a code flipped, the most that flip can
move the element: one E4M3 step times the row scale times the W2 entry).  Both tensor-core GEMM kernels are forced on the
same cases; moe_forward_e4m3 reproduces the staged calls bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import (BF16_RMS_TOL, assert_close, assert_equal, assert_probs, cf32, gpu_config,
                       half_ulp_bf16, make_case, np_view, rms, to_dev, to_np)

pytestmark = pytest.mark.gpu


def _bits(t):
    return np_view(t.detach().cpu())


def _gpu_quantize_rows(x):
    import mixture_experts_layer_fp32_gb300 as moe
    codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty((x.shape[0],), dtype=torch.float32, device="cuda")
    moe.quantize_rows_e4m3(x.cuda().contiguous(), codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(300, 512), (100, 4096), (70, 6144), (40, 16384),
                                       (33, 14336), (20, 20480), (9, 33280)])
def test_quantize_rows_bit_exact_with_ties_and_ranges(rows, cols):
    # a warp per row (<= 2048 values), a CTA per row (<= 32768), the wide fallback
    r = np.random.default_rng(130)
    x = (r.standard_normal((rows, cols)) * np.exp(r.uniform(-30, 30, (rows, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1, :] = 2.0 ** -105                      # below 2^-100: scale 1
    # rounding ties in E4M3 (midpoints of neighbouring codes) at scale 1
    mids = np.array([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, 13.5, 240.0, 208.0, 448.0])
    x[2, :mids.size] = mids
    x[2, mids.size:] = 0.5
    x[3, :mids.size] = -mids
    xb = torch.from_numpy(x).to(torch.bfloat16)
    codes, scales = _gpu_quantize_rows(xb)
    want_c, want_s = oracle.quantize_rows_e4m3(_bits(xb))
    assert_equal("codes", codes, want_c)
    assert_equal("scales", scales.view(np.uint32), want_s.view(np.uint32))


def test_quantize_experts_bit_exact():
    import mixture_experts_layer_fp32_gb300 as moe
    w = synthetic.scaled("mixtral", T=16, h=512, f=384, E=3, seed=131)
    inp = synthetic.generate(w)
    inp["W2"][1, 7, :] *= 1e3                   # a channel with a far larger range
    cfg = gpu_config(w)
    q = moe.E4m3Experts(cfg, inp["W1"].cuda(), inp["W3"].cuda(), inp["W2"].cuda())
    torch.cuda.synchronize()
    want = oracle.quantize_experts_e4m3(_bits(inp["W1"]), _bits(inp["W3"]), _bits(inp["W2"]))
    for n in ("W1q", "W3q", "W2q"):
        assert_equal(n, getattr(q, n).cpu().numpy(), want[n])
    for n in ("s1", "s3", "s2"):
        assert_equal(n, getattr(q, n).cpu().numpy().view(np.uint32), want[n].view(np.uint32))


CASES = {
    "mixtral_e4": synthetic.scaled("mixtral", T=1200, h=512, f=384, E=4, seed=132),
    "qwen3_sparse": synthetic.scaled("qwen3", T=300, h=256, f=256, seed=133),
    "switch_drop": synthetic.scaled("switch", T=2048, h=256, f=256, seed=134),
    "dsv3_grouped": synthetic.scaled("dsv3_grouped", T=400, h=512, f=256, E=64, seed=135),
    # pad_to_capacity: x quantised per token, code rows and scales placed by the padded map
    "switch_pad": synthetic.scaled("switch", T=2048, h=256, f=256, seed=136,
                                   pad_to_capacity=True),
    "top2_pad": synthetic.scaled("mixtral", T=600, h=512, f=384, E=4, capacity_factor=1.0,
                                 gate_bias="hot:1:2", seed=137, pad_to_capacity=True),
}


def oracle_forward_e4m3(w, inp):
    q = oracle.quantize_experts_e4m3(_bits(inp["W1"]), _bits(inp["W3"]), _bits(inp["W2"]))
    return oracle.forward_fp8(_bits(inp["x"]), _bits(inp["Wg"]), q, w.k, w.score,
                              np_view(inp["gate_bias"]), np_view(inp["expert_bias"]),
                              cf32(w), w.min_capacity, w.drop_policy,
                              num_groups=w.num_groups, group_topk=w.group_topk,
                              pad_to_capacity=w.pad_to_capacity)


def gpu_stages_e4m3(w, d):
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    ws = moe.alloc_workspace_e4m3(cfg)
    q = moe.E4m3Experts(cfg, d["W1"], d["W3"], d["W2"])
    R = moe.max_rows(cfg)
    b.x_perm_q = torch.empty((R, w.h), dtype=torch.uint8, device="cuda")
    b.x_perm_s = torch.empty((R,), dtype=torch.float32, device="cuda")
    b.h_q = torch.empty((R, w.f), dtype=torch.uint8, device="cuda")
    b.h_s = torch.empty((R,), dtype=torch.float32, device="cuda")
    moe.route(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], b.topk_idx, b.topk_prob,
              b.keep, b.tokens_per_expert, b.routing_map if w.pad_to_capacity else None, ws)
    if w.pad_to_capacity:
        moe.permute_map_e4m3(cfg, d["x"], b.routing_map, b.topk_idx, b.keep, b.x_perm_q,
                             b.x_perm_s, b.row_map, b.expert_offsets, ws)
    else:
        moe.permute_e4m3(cfg, d["x"], b.topk_idx, b.keep, b.x_perm_q, b.x_perm_s, b.row_map,
                         b.expert_offsets, ws)
    moe.grouped_mlp_e4m3(cfg, b.x_perm_q, b.x_perm_s, b.expert_offsets, q, b.h_mid, b.h_q,
                         b.h_s, b.y_perm, ws)
    # the forward's fc2 and combine: y_perm as fp16 with a scale per 32 columns
    b.y16 = torch.empty((R, w.h), dtype=torch.float16, device="cuda")
    b.y16_exp = torch.empty((R, w.h // 32), dtype=torch.int8, device="cuda")
    moe.grouped_fc2_e4m3_f16s(cfg, b.h_mid, b.expert_offsets, q, b.h_q, b.h_s, b.y16, b.y16_exp,
                              ws)
    moe.combine_f16s(cfg, b.y16, b.y16_exp, b.row_map, b.topk_prob, b.y)
    moe.check(ws)
    b.q, b.ws_e4m3 = q, ws
    return b


def flip_allowance(hq_gpu, ref, q, E, h):
    """Per element of y_perm [R, h]: the most the permitted one-code flips of
    the SwiGLU codes (GPU and oracle rounding a bf16 SwiGLU value that sits on
    an E4M3 rounding boundary to neighbouring codes) can move it.  For each
    flipped code (row r, column j): the larger E4M3 step beside the oracle's
    code, times the row scale, times |W2| of the row's expert in column j,
    dequantised -- oracle values only; the GPU's codes give the positions."""
    vals = oracle.e4m3_values()
    hq_ref = ref["hq"].astype(np.int32)
    R = hq_ref.shape[0]
    bound = np.zeros((R, h))
    rows, cols = np.nonzero(hq_gpu != hq_ref)
    row_expert = np.repeat(np.arange(E), np.diff(ref["offsets"]))
    for r, j in zip(rows, cols):
        c = int(hq_ref[r, j])
        mag, sign = c & 0x7F, c & 0x80
        step = max(abs(vals[(mag + dm) | sign] - vals[c]) for dm in (-1, 1)
                   if 0 <= mag + dm <= 0x7E)
        e = row_expert[r]
        w2 = np.abs(vals[q["W2q"][e, :, j]] * q["s2"][e].astype(np.float64))
        bound[r] += step * float(ref["hs"][r]) * w2
    return bound


def assert_bf16_close_allowing(name, got, want, allowance):
    """assert_close(..., "bf16") with a per-element allowance added to the
    2e-2 * RMS bound."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape and np.all(np.isfinite(got)), name
    excess = np.abs(got - want) - half_ulp_bf16(want) - allowance
    tol = BF16_RMS_TOL * rms(want)
    assert excess.max() <= tol, "%s: max err beyond rounding and flips %g > %g" % (
        name, excess.max(), tol)


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, _ = make_case(w)
    ref = oracle_forward_e4m3(w, inp)
    return w, inp, ref, to_dev(inp)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_e4m3_layer_matches_oracle(case, kernel, monkeypatch):
    w, inp, ref, d = case
    monkeypatch.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
    b = gpu_stages_e4m3(w, d)
    torch.cuda.synchronize()
    check_layer(w, inp, ref, b)


def check_layer(w, inp, ref, b):
    """Every stage of gpu_stages_e4m3's result against the FP8 oracle."""
    assert_equal("topk_idx", to_np(b.topk_idx), ref["topk_idx"])
    assert_equal("keep", to_np(b.keep), ref["keep"])
    assert_probs(to_np(b.topk_prob), ref["topk_prob"])
    assert_equal("expert_offsets", to_np(b.expert_offsets), ref["offsets"])
    assert_equal("row_map", to_np(b.row_map), ref["row_map"])
    R = int(ref["offsets"][-1])
    assert_equal("x_perm_q", to_np(b.x_perm_q[:R]), ref["xq"][ref["row_token"]])
    assert_equal("x_perm_scale", to_np(b.x_perm_s[:R]).view(np.uint32),
                 ref["xs"][ref["row_token"]].view(np.uint32))
    assert_close("h_mid", to_np(b.h_mid[:R]), ref["h_mid"], "bf16_stored")
    hq = to_np(b.h_q[:R]).astype(np.int32)
    diff = hq != ref["hq"].astype(np.int32)
    assert diff.mean() < 2e-3, diff.mean()
    if diff.any():  # only neighbouring codes, and only where the row scales agree
        same_scale = to_np(b.h_s[:R]) == ref["hs"]
        d_rows = np.nonzero(diff)[0]
        assert np.all(np.abs(hq - ref["hq"].astype(np.int32))[diff][same_scale[d_rows]] == 1)
    # a flipped code moves its row of y_perm by up to one E4M3 step times the
    # row's W2 column; every other element is held to the plain bound
    q = oracle.quantize_experts_e4m3(_bits(inp["W1"]), _bits(inp["W3"]), _bits(inp["W2"]))
    allow = flip_allowance(hq, ref, q, w.E, w.h)
    assert_bf16_close_allowing("y_perm", to_np(b.y_perm[:R]), ref["y_perm"], allow)
    # the fp16 y_perm: within 2^-11 of the fp32 one (plus the fp16 underflow step of its chunk)
    got = b.y16[:R].double().cpu() * torch.pow(2.0, torch.repeat_interleave(
        b.y16_exp[:R].cpu().long(), 32, dim=1).double())
    want = b.y_perm[:R].double().cpu()
    cmax = torch.repeat_interleave(want.abs().reshape(R, -1, 32).amax(dim=2), 32, dim=1)
    assert ((got - want).abs() <= 2.0 ** -11 * want.abs() + 2.0 ** -29 * cmax).all()
    # y: each token's slots add p times their rows' allowances
    rm = ref["row_map"].reshape(w.T, w.k)
    p = np.abs(ref["topk_prob"].reshape(w.T, w.k).astype(np.float64))
    allow_y = np.zeros((w.T, w.h))
    for j in range(w.k):
        ok = rm[:, j] >= 0
        allow_y[ok] += p[ok, j, None] * allow[rm[ok, j]]
    assert_bf16_close_allowing("y", to_np(b.y), ref["y"], allow_y)


def test_e4m3_forward_reproduces_stages(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, ref, d = case
    b = gpu_stages_e4m3(w, d)
    cfg = gpu_config(w)
    ws = moe.alloc_workspace_e4m3(cfg)
    y = torch.empty_like(b.y)
    idx = torch.empty_like(b.topk_idx)
    moe.forward_e4m3(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], b.q, y, ws, idx)
    moe.check(ws)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(y, b.y)


def test_e4m3_close_to_the_bf16_layer(case):
    # quantisation error of the whole layer against the unquantised oracle
    w, inp, ref, d = case
    from moe_cases import oracle_forward
    exact = oracle_forward(w, inp)
    rel = np.sqrt(np.mean((ref["y"] - exact["y"]) ** 2) / np.mean(exact["y"] ** 2))
    assert rel < 0.1, rel


def test_e4m3_rejects_fp32_config():
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = moe.config(T=16, h=256, E=4, k=2, f=128, dtype="f32")
    with pytest.raises(moe.MoeError):
        moe.workspace_size_e4m3(cfg)


def test_e4m3_stage_halves_equal_grouped_mlp(case):
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, ref, d = case
    b = gpu_stages_e4m3(w, d)
    cfg = gpu_config(w)
    h_mid = torch.empty_like(b.h_mid)
    h_q = torch.empty_like(b.h_q)
    h_s = torch.empty_like(b.h_s)
    y_perm = torch.empty_like(b.y_perm)
    moe.grouped_fc1_e4m3(cfg, b.x_perm_q, b.x_perm_s, b.expert_offsets, b.q, h_mid, b.ws_e4m3)
    moe.grouped_fc2_e4m3(cfg, h_mid, b.expert_offsets, b.q, h_q, h_s, y_perm, b.ws_e4m3)
    moe.check(b.ws_e4m3)
    R = int(ref["offsets"][-1])
    assert torch.equal(h_mid[:R], b.h_mid[:R])
    assert torch.equal(h_q[:R], b.h_q[:R])
    assert torch.equal(y_perm[:R], b.y_perm[:R])
