"""Pins of the oracle's FP8 (E4M3) arithmetic against facts other than
itself: the format's known code points, PyTorch's float8_e4m3fn conversion
(a library routine) over every in-range bf16 value, the round trip of every
finite code, the power-of-two scale rule checked by its defining
inequalities, and closed forms of the FP8 expert on one-hot rows.  CPU only.
"""

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def test_e4m3_known_code_points():
    v = oracle.e4m3_values()
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0          # largest finite
    assert v[0x08] == 2.0 ** -6                             # smallest normal
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9  # subnormals
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    finite = v[:127]
    assert np.all(np.diff(finite) > 0)                      # codes 0..126 increase


def test_e4m3_round_trip_of_every_finite_code():
    v = oracle.e4m3_values()
    codes = np.array([c for c in range(256) if not np.isnan(v[c])])
    np.testing.assert_array_equal(oracle.e4m3_codes(v[codes]), codes)


def test_e4m3_codes_match_torch_on_every_bf16_value_in_range():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (bits << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    vals = vals[ok]
    want = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(oracle.e4m3_codes(vals), want.numpy())


def test_e4m3_ties_to_even_and_saturation():
    # midpoints between neighbouring codes go to the even code
    assert list(oracle.e4m3_codes([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10])) == \
        [0x38, 0x3A, 0x02, 0x00]
    # beyond the largest finite value: saturate, keep the sign; NaN -> NaN code
    assert list(oracle.e4m3_codes([449.0, 464.0, 1e30, -1e30, np.nan])) == \
        [0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantize_rows_scale_rule_and_codes(dtype):
    r = rng(120)
    x = (r.standard_normal((64, 96)) * np.exp(r.uniform(-20, 20, (64, 1)))).astype(np.float32)
    x[3] = 0.0
    x[5, :] = 448.0                                   # exactly representable, scale 1
    if dtype == "bf16":
        x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
        arg = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        arg = x
    codes, scales = oracle.quantize_rows_e4m3(arg)
    amax = np.abs(x.astype(np.float64)).max(axis=1)
    for i in range(x.shape[0]):
        s = float(scales[i])
        e = int(np.round(np.log2(s)))
        assert s == 2.0 ** e                                           # a power of two
        if amax[i] == 0:
            assert e == 0 and np.all(codes[i] == 0)
            continue
        assert amax[i] / 2.0 ** e <= 448.0 < amax[i] / 2.0 ** (e - 1)  # the smallest such e
        want = torch.from_numpy((x[i] / s).astype(np.float32)).to(torch.float8_e4m3fn)
        np.testing.assert_array_equal(codes[i], want.view(torch.uint8).numpy())
    assert scales[5] == 1.0


def test_scale_rule_edges():
    x = np.zeros((4, 8), np.float32)
    x[0, 0] = 2.0 ** -101           # below 2^-100: scale 1, codes 0
    x[1, 0] = 2.0 ** -99            # smallest e: 2^-99 / 2^e <= 448 -> e = -107
    x[2, 0] = np.float32(3.4e38)    # largest magnitudes: e = 120
    x[3, 0] = np.inf                # infinite: scale 1, saturated code
    codes, scales = oracle.quantize_rows_e4m3(x)
    assert scales[0] == 1.0 and codes[0, 0] == 0
    assert scales[1] == 2.0 ** -107 and oracle.e4m3_values()[codes[1, 0]] == 256.0
    assert scales[2] == 2.0 ** 120
    assert scales[3] == 1.0 and codes[3, 0] == 0x7E


def test_quantize_cols_is_rows_of_the_transpose():
    W = rng(121).standard_normal((3, 40, 24)).astype(np.float32)
    W[1, :, 7] *= 1e4
    codes, scales = oracle.quantize_cols_e4m3(W)
    assert codes.shape == (3, 24, 40) and scales.shape == (3, 24)
    for e in range(3):
        c2, s2 = oracle.quantize_rows_e4m3(np.ascontiguousarray(W[e].T))
        np.testing.assert_array_equal(codes[e], c2)
        np.testing.assert_array_equal(scales[e], s2)


def _dequant_cols(codes, scales):
    v = oracle.e4m3_values()
    return v[codes] * scales[..., None].astype(np.float64)      # [E,N,K]


def test_fp8_expert_one_hot_closed_form():
    # x = 256 * e_i: the smallest power of two s with 256 / s <= 448 is 1, so the
    # row holds one code of value 256 -> a = 256 * W1q[c][i] * s1[c] exactly, and
    # h, its bf16 rounding and its row quantisation follow in closed form.
    E, h, f = 2, 6, 5
    r = rng(122)
    W1, W3 = (r.standard_normal((E, h, f)).astype(np.float32) for _ in range(2))
    W2 = r.standard_normal((E, f, h)).astype(np.float32)
    q = oracle.quantize_experts_e4m3(W1, W3, W2)
    w1 = _dequant_cols(q["W1q"], q["s1"])
    w3 = _dequant_cols(q["W3q"], q["s3"])
    w2 = _dequant_cols(q["W2q"], q["s2"])
    rows, experts = [], []
    for e in range(E):
        for i in range(h):
            v = np.zeros(h, np.float32)
            v[i] = 256.0
            rows.append(v)
            experts.append(e)
    xq, xs = oracle.quantize_rows_e4m3(np.array(rows))
    assert np.all(xs == 1.0)
    out = oracle.expert_rows_fp8(xq, xs, np.array(experts, np.int32), q)
    for n_, (e, i) in enumerate([(e, i) for e in range(E) for i in range(h)]):
        a, g = 256.0 * w1[e, :, i], 256.0 * w3[e, :, i]
        H = torch.from_numpy(a * expit(a) * g).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(out["h_mid"][n_], H)        # bf16 rounding, exact
        hq, hs = oracle.quantize_rows_e4m3(H[None].astype(np.float32))
        np.testing.assert_array_equal(out["hq"][n_], hq[0])
        y = (oracle.e4m3_values()[hq[0]] * float(hs[0])) @ w2[e].T
        np.testing.assert_allclose(out["y_rows"][n_], y, rtol=1e-12, atol=1e-12)


def test_fp8_forward_close_to_the_unquantised_layer():
    # the FP8 layer differs from the bf16 one only by quantisation: a few % of RMS
    T, h, E, k, f = 48, 64, 4, 2, 32
    r = rng(123)
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = (0.1 * r.standard_normal((h, E))).astype(np.float32)
    W1, W3 = ((0.1 * r.standard_normal((E, h, f))).astype(np.float32) for _ in range(2))
    W2 = (0.1 * r.standard_normal((E, f, h))).astype(np.float32)
    ref = oracle.forward(x, Wg, W1, W3, W2, k, "softmax_post")
    q = oracle.quantize_experts_e4m3(W1, W3, W2)
    out = oracle.forward_fp8(x, Wg, q, k, "softmax_post")
    np.testing.assert_array_equal(out["topk_idx"], ref["topk_idx"])   # routing is not quantised
    rel = np.sqrt(np.mean((out["y"] - ref["y"]) ** 2) / np.mean(ref["y"] ** 2))
    assert 1e-4 < rel < 0.1, rel


def test_fp8_padded_forward_equals_unpadded():
    # pad_to_capacity adds rows of probability 0: the FP8 layer's output is
    # unchanged bit for bit, and each padded row is its token's code row
    T, h, E, k, f = 120, 32, 6, 2, 32
    r = rng(124)
    x = r.standard_normal((T, h)).astype(np.float32)
    Wg = (0.2 * r.standard_normal((h, E))).astype(np.float32)
    gb = np.linspace(1.0, -1.0, E).astype(np.float32)
    W1, W3 = ((0.1 * r.standard_normal((E, h, f))).astype(np.float32) for _ in range(2))
    W2 = (0.1 * r.standard_normal((E, f, h))).astype(np.float32)
    q = oracle.quantize_experts_e4m3(W1, W3, W2)
    a = oracle.forward_fp8(x, Wg, q, k, "softmax_post", gate_bias=gb, capacity_factor=1.25,
                           pad_to_capacity=True)
    b = oracle.forward_fp8(x, Wg, q, k, "softmax_post", gate_bias=gb, capacity_factor=1.25)
    cap = a["capacity"]
    assert int(a["offsets"][-1]) == E * min(cap, T) > int(b["offsets"][-1])
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["xq"][a["row_token"]].shape[0], a["offsets"][-1])
