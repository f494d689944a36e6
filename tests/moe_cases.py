"""Shared helpers of the parity tests: seeded inputs conditioned on the
routing margin (using the oracle), oracle runs, GPU runs through the C ABI,
and the comparisons with their tolerances.

Tolerances (fixed here, used by every parity test):
  * integer / index outputs (topk_idx, keep, tokens_per_expert, offsets,
    row_map) and permuted rows: bit-exact;
  * router probabilities: |gpu - oracle| <= 1e-5 * |oracle| + 1e-6;
  * fp32 outputs: |gpu - oracle| <= 1e-4 * (|oracle| + RMS(oracle))
    (1e-4 relative, with an RMS floor for entries near zero where a
    relative bound is meaningless for any summation order);
  * bf16 outputs: max (|gpu - oracle| - half_ulp_bf16(oracle)) <= 2e-2 * RMS(oracle)
    -- the bound applies to the error beyond the output's own rounding to
    bf16, which alone reaches 2^-8 * max|y| (more than 2e-2 * RMS whenever
    max|y| > 5 RMS, e.g. with dropped tokens' zero rows);
  * bf16-stored intermediates (h_mid): |gpu - oracle| <= 2^-7 * |oracle| +
    1e-2 * RMS(oracle) -- the SwiGLU output is heavy-tailed, so bf16
    storage rounding of its largest entries alone exceeds 2e-2 * RMS; the
    layer output y is near-Gaussian and keeps the 2e-2 * RMS bound.
"""

import numpy as np
import torch

import oracle
import synthetic

MARGIN = 1e-3        # selection-score gap between the k-th and (k+1)-th expert
CAP_MARGIN = 1e-5    # probability gap at each overflowing expert's capacity boundary
PROB_RTOL, PROB_ATOL = 1e-5, 1e-6
F32_RTOL = 1e-4
BF16_RMS_TOL = 2e-2
BF16_ULP = 2.0 ** -7
BF16_STORED_RMS_TOL = 1e-2


def cf32(w):
    """The capacity factor as the layer gets it: an fp32 field of the config
    (0.6 arrives as 0.60000002384...).  The oracle is given the same value, so
    that ceil(T*k/E * cf) is the same number on both sides."""
    return float(np.float32(w.capacity_factor))


def np_view(t):
    """A CPU torch tensor as the numpy array the oracle takes."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _cap_boundary_bad(r, w):
    """Tokens sitting on a capacity boundary closer than CAP_MARGIN."""
    cap = r["capacity"]
    if cap < 0 or cap >= w.T or w.drop_policy != "probs":
        return []
    idx, p = r["topk_idx"], r["topk_prob_raw"]
    bad = []
    for e in np.nonzero(r["assigned"] > cap)[0]:
        tok, slot = np.nonzero(idx == e)
        pe = p[tok, slot].astype(np.float64)
        order = np.argsort(-pe, kind="stable")
        if pe[order[cap - 1]] - pe[order[cap]] < CAP_MARGIN:
            bad.append(int(tok[order[cap]]))
    return bad


def condition_inputs(w, inp, max_rounds=64, nthreads=0):
    """Redraw x rows until every token's top-k margin is >= MARGIN (and the
    capacity boundaries are clear).  Only redrawn rows are routed again.
    Returns the oracle routing of the final x.  `inp["x"]` is updated in
    place (CPU or CUDA tensor)."""
    x = inp["x"]
    Wg = np_view(inp["Wg"])
    gb, eb = np_view(inp["gate_bias"]), np_view(inp["expert_bias"])
    x_cpu = x.detach().to("cpu").clone()
    logits = oracle.router_logits(np_view(x_cpu), Wg, gb, nthreads)
    groups = (w.num_groups, w.group_topk)
    idx, prob, margin = oracle.topk_scores(logits, w.k, w.score, eb, nthreads, *groups)
    for rnd in range(max_rounds):
        part = {"capacity": oracle.capacity(w.T, w.E, w.k, cf32(w), w.min_capacity),
                "topk_idx": idx, "topk_prob_raw": prob,
                "assigned": np.bincount(idx.reshape(-1), minlength=w.E)}
        bad = sorted(set(np.nonzero(margin < MARGIN)[0].tolist()) |
                     set(_cap_boundary_bad(part, w)))
        if not bad:
            break
        rows = torch.tensor(bad)
        x_cpu[rows] = synthetic.redraw_x_rows(w, rnd, len(bad))
        sub = oracle.router_logits(np_view(x_cpu[rows]), Wg, gb, nthreads)
        i2, p2, m2 = oracle.topk_scores(sub, w.k, w.score, eb, nthreads, *groups)
        idx[bad], prob[bad], margin[bad] = i2, p2, m2
    else:
        raise RuntimeError("margin conditioning did not converge")
    x.copy_(x_cpu.to(x.device))
    r = oracle.route(np_view(x_cpu), Wg, w.k, w.score, gb, eb, cf32(w),
                     w.min_capacity, w.drop_policy, nthreads, *groups,
                     pad_to_capacity=w.pad_to_capacity)
    assert np.all(r["margin"] >= MARGIN)
    return r


def make_case(w, device="cpu", nthreads=0):
    inp = synthetic.generate(w, device=device)
    r = condition_inputs(w, inp, nthreads=nthreads)
    return inp, r


def oracle_forward(w, inp, nthreads=0, want_h_mid=True):
    shared = {}
    if w.shared_f > 0:
        shared = {n: np_view(inp[n]) for n in ("W1s", "W3s", "W2s")}
    return oracle.forward(np_view(inp["x"]), np_view(inp["Wg"]), np_view(inp["W1"]),
                          np_view(inp["W3"]), np_view(inp["W2"]), w.k, w.score,
                          np_view(inp["gate_bias"]), np_view(inp["expert_bias"]),
                          cf32(w), w.min_capacity, w.drop_policy, nthreads,
                          want_h_mid=want_h_mid, num_groups=w.num_groups,
                          group_topk=w.group_topk, pad_to_capacity=w.pad_to_capacity, **shared)


def gpu_config(w):
    import mixture_experts_layer_fp32_gb300 as moe
    return moe.config(w.T, w.h, w.E, w.k, w.f, w.score, w.dtype, w.capacity_factor,
                      w.min_capacity, w.drop_policy, w.num_groups, w.group_topk,
                      w.pad_to_capacity)


def to_dev(inp, device="cuda"):
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in inp.items()}


def uses_f16s(w):
    """bf16 layers with k >= 2 (no padding, no shared expert): the forward
    combines over y_perm stored as fp16 with a power-of-two scale per 32
    columns (moe_grouped_fc2_f16s + moe_combine_f16s)."""
    return w.dtype == "bf16" and w.k > 1 and not w.pad_to_capacity and w.shared_f == 0


def gpu_stages(w, dinp, with_routing_map=True, fp32_combine=False):
    """Run the stages through the C ABI as the forward does; returns the
    Buffers object.  y_perm (fp32, moe_grouped_fc2) is always computed for
    the intermediate checks; y comes from the combine the forward uses (for
    uses_f16s layers the fp16 y_perm path, its y16 / y16_exp kept on the
    Buffers) unless fp32_combine."""
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    moe.route(cfg, dinp["x"], dinp["Wg"], dinp["gate_bias"], dinp["expert_bias"], b.topk_idx,
              b.topk_prob, b.keep, b.tokens_per_expert,
              b.routing_map if (with_routing_map or w.pad_to_capacity) else None, b.ws)
    if w.pad_to_capacity:  # the padded routing map drives the permutation
        moe.permute_map(cfg, dinp["x"], b.routing_map, b.topk_idx, b.keep, b.x_perm, b.row_map,
                        b.expert_offsets, b.ws)
    else:
        moe.permute(cfg, dinp["x"], b.topk_idx, b.keep, b.x_perm, b.row_map, b.expert_offsets,
                    b.ws)
    moe.grouped_fc1(cfg, b.x_perm, b.expert_offsets, dinp["W1"], dinp["W3"], b.h_mid, b.ws)
    moe.grouped_fc2(cfg, b.h_mid, b.expert_offsets, dinp["W2"], b.y_perm, b.ws)
    if w.shared_f > 0:
        b.h_mid_s = torch.empty((w.T, w.shared_f), dtype=moe.act_dtype(cfg), device="cuda")
        b.y_shared = torch.empty((w.T, w.h), dtype=torch.float32, device="cuda")
        moe.shared_expert(cfg, w.shared_f, dinp["x"], dinp["W1s"], dinp["W3s"], dinp["W2s"],
                          b.h_mid_s, b.y_shared, b.ws)
        if w.dtype == "bf16" and not w.pad_to_capacity and not fp32_combine:
            # the shared forward's path: the fp16 y_perm and its combine with the shared row
            b.y16 = torch.empty((b.y_perm.shape[0], w.h), dtype=torch.float16, device="cuda")
            b.y16_exp = torch.empty((b.y_perm.shape[0], w.h // 32), dtype=torch.int8,
                                    device="cuda")
            moe.grouped_fc2_f16s(cfg, b.h_mid, b.expert_offsets, dinp["W2"], b.y16, b.y16_exp,
                                 b.ws)
            moe.combine_f16s(cfg, b.y16, b.y16_exp, b.row_map, b.topk_prob, b.y,
                             y_shared=b.y_shared)
        else:
            moe.combine_shared(cfg, b.y_perm, b.row_map, b.topk_prob, b.y_shared, b.y)
    elif uses_f16s(w) and not fp32_combine:
        b.y16 = torch.empty((b.y_perm.shape[0], w.h), dtype=torch.float16, device="cuda")
        b.y16_exp = torch.empty((b.y_perm.shape[0], w.h // 32), dtype=torch.int8, device="cuda")
        moe.grouped_fc2_f16s(cfg, b.h_mid, b.expert_offsets, dinp["W2"], b.y16, b.y16_exp, b.ws)
        moe.combine_f16s(cfg, b.y16, b.y16_exp, b.row_map, b.topk_prob, b.y)
    else:
        moe.combine(cfg, b.y_perm, b.row_map, b.topk_prob, b.y)
    moe.check(b.ws)
    return b


def gpu_forward(w, dinp):
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = gpu_config(w)
    ws = moe.alloc_workspace(cfg)
    y = torch.empty((w.T, w.h), dtype=moe.act_dtype(cfg), device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    prob = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    tpe = torch.empty((w.E,), dtype=torch.int32, device="cuda")
    if w.shared_f > 0:
        ws = moe.alloc_workspace_shared(cfg, w.shared_f)
        moe.forward_shared(cfg, w.shared_f, dinp["x"], dinp["Wg"], dinp["gate_bias"],
                           dinp["expert_bias"], dinp["W1"], dinp["W3"], dinp["W2"], dinp["W1s"],
                           dinp["W3s"], dinp["W2s"], y, ws, idx, prob, tpe)
    else:
        moe.forward(cfg, dinp["x"], dinp["Wg"], dinp["gate_bias"], dinp["expert_bias"],
                    dinp["W1"], dinp["W3"], dinp["W2"], y, ws, idx, prob, tpe)
    moe.check(ws)
    return y, idx, prob, tpe


# ------------------------------------------------------------ comparisons

def assert_equal(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    bad = np.nonzero(got != want)
    assert bad[0].size == 0, "%s: %d mismatches, first at %s: got %s want %s" % (
        name, bad[0].size, tuple(b[0] for b in bad), got[tuple(b[0] for b in bad)],
        want[tuple(b[0] for b in bad)])


def assert_probs(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want) - (PROB_RTOL * np.abs(want) + PROB_ATOL)
    assert np.all(err <= 0), "probs: max excess %g" % err.max()


def half_ulp_bf16(v):
    """Half the bf16 spacing at |v| (the largest error of a correct rounding)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def rms(a):
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def assert_close(name, got, want, dtype):
    """got: GPU values (any float), want: oracle float64."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if want.size == 0:
        return
    assert np.all(np.isfinite(got)), "%s: non-finite GPU values" % name
    r = rms(want)
    d = np.abs(got - want)
    if dtype == "bf16":
        # error beyond the output's own rounding to bf16 (half an ulp of the
        # exact value), bounded by 2e-2 * RMS
        excess = d - half_ulp_bf16(want)
        tol = BF16_RMS_TOL * r
        assert excess.max() <= tol, "%s: max err beyond rounding %g > %g (= 2e-2 * RMS %g)" % (
            name, excess.max(), tol, r)
    elif dtype == "bf16_stored":
        # a bf16-stored intermediate: one bf16 ulp (2^-7 relative) for the
        # storage rounding plus 1e-2 * RMS for the accumulation
        lim = BF16_ULP * np.abs(want) + BF16_STORED_RMS_TOL * r
        i = np.argmax(d - lim)
        assert d.reshape(-1)[i] <= lim.reshape(-1)[i], "%s: err %g > %g (want %g)" % (
            name, d.reshape(-1)[i], lim.reshape(-1)[i], want.reshape(-1)[i])
    else:
        lim = (F32_RTOL * (np.abs(want) + r)).reshape(-1)
        d = d.reshape(-1)
        i = int(np.argmax(d - lim))
        assert d[i] <= lim[i], "%s: err %g > %g at %d (want %g)" % (name, d[i], lim[i], i,
                                                                      want.reshape(-1)[i])


def to_np(t):
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def compare_all(w, inp, ref, b):
    """Every output of a staged GPU run against the oracle (small cases)."""
    assert_equal("topk_idx", to_np(b.topk_idx), ref["topk_idx"])
    assert_equal("keep", to_np(b.keep), ref["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), ref["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), ref["topk_prob"])
    assert_equal("expert_offsets", to_np(b.expert_offsets), ref["offsets"])
    assert_equal("row_map", to_np(b.row_map), ref["row_map"])
    R = int(ref["offsets"][-1])
    got = b.x_perm[:R].detach().cpu()
    want = inp["x"].detach().cpu()[torch.from_numpy(ref["row_token"]).long()]
    if got.dtype == torch.bfloat16:
        got, want = got.view(torch.int16), want.view(torch.int16)
    assert torch.equal(got, want)
    assert_close("h_mid", to_np(b.h_mid[:R]), ref["h_mid"],
                 "bf16_stored" if w.dtype == "bf16" else w.dtype)
    assert_close("y_perm", to_np(b.y_perm[:R]), ref["y_perm"], w.dtype)
    if w.shared_f > 0:
        assert_close("h_mid_s", to_np(b.h_mid_s), ref["h_mid_s"],
                     "bf16_stored" if w.dtype == "bf16" else w.dtype)
        assert_close("y_shared", to_np(b.y_shared), ref["y_shared"], w.dtype)
    assert_close("y", to_np(b.y), ref["y"], w.dtype)
