"""CPU oracle of the MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The product (the CUDA library under
`mixture_experts_layer_fp32_gb300/` and its binding) never imports it; the
two share no code.  The arithmetic lives in `moe_oracle.cpp` (plain C++,
double precision); this module only marshals numpy arrays.

Inputs are numpy arrays: fp32 arrays, or uint16 arrays holding bf16 bit
patterns (widened exactly inside the oracle).
"""

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIBDIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_LIBDIR, "libmoe_oracle.so")
_lib = None

SCORES = {"softmax_post": 0, "softmax_pre": 1, "sigmoid": 2, "sqrtsoftplus": 3}
POLICIES = {"probs": 0, "position": 1}


def build(force=False):
    """Compile the oracle into oracle/_build/libmoe_oracle.so (g++, -O2)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.oracle_router_logits.argtypes = [i64, i32, i32, vp, i32, vp, vp, vp, i32]
        L.oracle_topk_scores.argtypes = [i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32]
        L.oracle_capacity.argtypes = [i64, i32, i32, dbl, i64]
        L.oracle_capacity.restype = i64
        L.oracle_capacity_drop.argtypes = [i64, i32, i32, i64, i32, vp, vp, vp, vp]
        L.oracle_permute.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_permute.restype = i64
        L.oracle_pad_to_capacity.argtypes = [i64, i32, i32, i64, vp, vp, vp, vp]
        L.oracle_permute_map.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp, vp]
        L.oracle_permute_map.restype = i64
        L.oracle_expert_rows.argtypes = [i64, i32, i32, vp, i32, vp, vp, vp, vp, i32, vp, vp, i32]
        L.oracle_combine.argtypes = [i64, i32, i32, vp, vp, vp, vp, i32]
        L.oracle_forward_dense.argtypes = [i64, i32, i32, i32, i32, vp, i32, vp, vp, vp,
                                           vp, vp, vp, i32, vp, i32]
        L.oracle_quantize_rows_e4m3.argtypes = [i64, i32, vp, i32, vp, vp, i32]
        L.oracle_quantize_cols_e4m3.argtypes = [i64, i32, i32, vp, i32, vp, vp, i32]
        L.oracle_expert_rows_fp8.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             vp, vp, vp, vp, i32]
        L.oracle_backward.argtypes = [i64, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp,
                                      vp, vp, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                      vp, i32]
        L.oracle_expert_wgrad_cols.argtypes = [i64, i32, i32, vp, i32, vp, vp, i32, vp, vp, vp,
                                               i32, i32, vp, i32, vp, vp, vp, vp, i32]
        L.oracle_e4m3_values.argtypes = [vp]
        L.oracle_e4m3_codes.argtypes = [i64, vp, vp]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a):
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError("oracle inputs are float32 or uint16 (bf16 bits), got %s" % a.dtype)


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.asarray(a)
    if dtype is not None:
        a = a.astype(dtype, copy=False)
    return np.ascontiguousarray(a)


def bf16_bits_to_f32(a):
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def router_logits(x, Wg, gate_bias=None, nthreads=0):
    x = _c(x)
    Wg = _c(Wg, np.float32)
    gate_bias = _c(gate_bias, np.float32)
    T, h = x.shape
    E = Wg.shape[1]
    out = np.empty((T, E), np.float32)
    _load().oracle_router_logits(T, h, E, _ptr(x), _dtype_code(x), _ptr(Wg), _ptr(gate_bias),
                                 _ptr(out), nthreads)
    return out


def topk_scores(logits, k, score, expert_bias=None, nthreads=0, num_groups=0, group_topk=0):
    """Scores and top-k of [MC] §5; num_groups > 1 turns on group-limited
    top-k (group_topk of num_groups groups kept)."""
    logits = _c(logits, np.float32)
    expert_bias = _c(expert_bias, np.float32)
    T, E = logits.shape
    if num_groups > 1:
        assert E % num_groups == 0 and 1 <= group_topk <= min(num_groups, k)
        assert k <= group_topk * (E // num_groups)
    idx = np.empty((T, k), np.int32)
    prob = np.empty((T, k), np.float32)
    margin = np.empty((T,), np.float32)
    _load().oracle_topk_scores(T, E, k, SCORES[score], int(num_groups), int(group_topk),
                               _ptr(logits), _ptr(expert_bias), _ptr(idx), _ptr(prob),
                               _ptr(margin), nthreads)
    return idx, prob, margin


def capacity(T, E, k, capacity_factor, min_capacity=0):
    return int(_load().oracle_capacity(T, E, k, float(capacity_factor), int(min_capacity)))


def capacity_drop(topk_idx, topk_prob, E, cap, policy="probs"):
    topk_idx = _c(topk_idx, np.int32)
    prob = np.array(topk_prob, dtype=np.float32, copy=True)
    T, k = topk_idx.shape
    keep = np.empty((T, k), np.uint8)
    kept = np.empty((E,), np.int32)
    _load().oracle_capacity_drop(T, E, k, cap, POLICIES[policy], _ptr(topk_idx), _ptr(prob),
                                 _ptr(keep), _ptr(kept))
    return prob, keep, kept


def permute(topk_idx, keep, E):
    topk_idx = _c(topk_idx, np.int32)
    keep = _c(keep, np.uint8)
    T, k = topk_idx.shape
    offsets = np.empty((E + 1,), np.int32)
    row_map = np.empty((T, k), np.int32)
    row_token = np.empty((T * k,), np.int32)
    R = _load().oracle_permute(T, E, k, _ptr(topk_idx), _ptr(keep), _ptr(offsets),
                               _ptr(row_map), _ptr(row_token))
    return offsets, row_map, row_token[:R].copy()


def pad_to_capacity_map(topk_idx, keep, E, cap):
    """final_map of apply_router_token_dropping with pad_to_capacity: every
    expert column holds min(cap, T) tokens (the kept pairs, then the
    lowest-index tokens not yet set).  Returns (map [T,E] u8, column sums)."""
    topk_idx = _c(topk_idx, np.int32)
    keep = _c(keep, np.uint8)
    T, k = topk_idx.shape
    m = np.empty((T, E), np.uint8)
    n = np.empty((E,), np.int32)
    _load().oracle_pad_to_capacity(T, E, k, int(cap), _ptr(topk_idx), _ptr(keep), _ptr(m), _ptr(n))
    return m, n


def permute_map(routing_map, topk_idx, keep):
    """Permutation by a [T,E] routing map: rows of expert e are its tokens in
    ascending order; row_map [T,k] holds the rows of the kept pairs."""
    routing_map = _c(routing_map, np.uint8)
    topk_idx = _c(topk_idx, np.int32)
    keep = _c(keep, np.uint8)
    T, E = routing_map.shape
    k = topk_idx.shape[1]
    offsets = np.empty((E + 1,), np.int32)
    row_map = np.empty((T, k), np.int32)
    row_token = np.empty((int(routing_map.sum()),), np.int32)
    R = _load().oracle_permute_map(T, E, k, _ptr(routing_map), _ptr(topk_idx), _ptr(keep),
                                   _ptr(offsets), _ptr(row_map), _ptr(row_token))
    return offsets, row_map, row_token[:R].copy()


def expert_rows(x_rows, row_expert, W1, W3, W2, want_h_mid=False, nthreads=0):
    """SwiGLU expert MLP on rows; returns y_rows [R,h] (and h_mid [R,f]) in float64."""
    x_rows = _c(x_rows)
    row_expert = _c(row_expert, np.int32)
    W1, W3, W2 = _c(W1), _c(W3), _c(W2)
    R, h = x_rows.shape
    f = W1.shape[-1]
    wd = _dtype_code(W1)
    assert _dtype_code(W3) == wd and _dtype_code(W2) == wd
    y = np.empty((R, h), np.float64)
    hm = np.empty((R, f), np.float64) if want_h_mid else None
    _load().oracle_expert_rows(R, h, f, _ptr(x_rows), _dtype_code(x_rows), _ptr(row_expert),
                               _ptr(W1), _ptr(W3), _ptr(W2), wd, _ptr(hm), _ptr(y), nthreads)
    return (y, hm) if want_h_mid else y


def combine(y_perm, row_map, topk_prob, nthreads=0):
    y_perm = _c(y_perm, np.float64)
    row_map = _c(row_map, np.int32)
    topk_prob = _c(topk_prob, np.float32)
    T, k = row_map.shape
    h = y_perm.shape[1]
    y = np.empty((T, h), np.float64)
    _load().oracle_combine(T, k, h, _ptr(y_perm), _ptr(row_map), _ptr(topk_prob), _ptr(y),
                           nthreads)
    return y


def forward_dense(x, topk_idx, topk_prob, keep, W1, W3, W2, nthreads=0):
    x = _c(x)
    topk_idx = _c(topk_idx, np.int32)
    topk_prob = _c(topk_prob, np.float32)
    keep = _c(keep, np.uint8)
    W1, W3, W2 = _c(W1), _c(W3), _c(W2)
    T, h = x.shape
    E, _, f = W1.shape
    k = topk_idx.shape[1]
    y = np.empty((T, h), np.float64)
    _load().oracle_forward_dense(T, h, E, k, f, _ptr(x), _dtype_code(x), _ptr(topk_idx),
                                 _ptr(topk_prob), _ptr(keep), _ptr(W1), _ptr(W3), _ptr(W2),
                                 _dtype_code(W1), _ptr(y), nthreads)
    return y


def route(x, Wg, k, score, gate_bias=None, expert_bias=None, capacity_factor=0.0,
          min_capacity=0, drop_policy="probs", nthreads=0, num_groups=0, group_topk=0,
          pad_to_capacity=False):
    """Router + optional capacity drop (and, with pad_to_capacity, the padded
    routing map: "routing_map", with tokens_per_expert its column sums).
    Returns a dict of numpy arrays."""
    T = x.shape[0]
    E = Wg.shape[1]
    logits = router_logits(x, Wg, gate_bias, nthreads)
    idx, prob, margin = topk_scores(logits, k, score, expert_bias, nthreads, num_groups,
                                    group_topk)
    assigned = np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)
    cap = capacity(T, E, k, capacity_factor, min_capacity)
    prob_final, keep, kept = capacity_drop(idx, prob, E, cap, drop_policy)
    out = {"logits": logits, "topk_idx": idx, "topk_prob_raw": prob, "margin": margin,
           "assigned": assigned, "capacity": cap, "topk_prob": prob_final, "keep": keep,
           "tokens_per_expert": kept}
    if pad_to_capacity:
        assert cap >= 0, "pad_to_capacity needs a capacity factor"
        m, padded = pad_to_capacity_map(idx, keep, E, cap)
        out.update({"routing_map": m, "tokens_per_expert": padded, "kept_per_expert": kept})
    return out


def shared_expert(x, W1s, W3s, W2s, want_h_mid=False, nthreads=0):
    """The shared expert of the Megatron Core page (§11; the layer forward of
    §2 adds it: hidden = shared_expert(hidden_in) + routed output): one SwiGLU
    MLP applied to every token, no router.  It is the same SwiGLU row
    computation as a routed expert, with every row on the single expert 0.
    W1s/W3s [h,fs], W2s [fs,h].  Returns y_shared [T,h] (and h_mid_s [T,fs])
    in float64."""
    x = _c(x)
    T = x.shape[0]
    expert = np.zeros(T, np.int32)
    return expert_rows(x, expert, _c(W1s)[None], _c(W3s)[None], _c(W2s)[None],
                       want_h_mid=want_h_mid, nthreads=nthreads)


def forward(x, Wg, W1, W3, W2, k, score, gate_bias=None, expert_bias=None,
            capacity_factor=0.0, min_capacity=0, drop_policy="probs", nthreads=0,
            want_h_mid=False, W1s=None, W3s=None, W2s=None, num_groups=0, group_topk=0,
            pad_to_capacity=False):
    """The whole layer: route -> drop -> permute -> SwiGLU experts -> combine,
    plus the shared expert's output when W1s/W3s/W2s are given (added to the
    routed sum in double: y = sum_j p_j Y_j + Y_shared).  pad_to_capacity:
    the experts run on the padded routing map's rows (the padding rows carry
    no combine weight)."""
    r = route(x, Wg, k, score, gate_bias, expert_bias, capacity_factor, min_capacity,
              drop_policy, nthreads, num_groups, group_topk, pad_to_capacity)
    E = Wg.shape[1]
    if pad_to_capacity:
        offsets, row_map, row_token = permute_map(r["routing_map"], r["topk_idx"], r["keep"])
    else:
        offsets, row_map, row_token = permute(r["topk_idx"], r["keep"], E)
    row_expert = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    x_perm = np.ascontiguousarray(np.asarray(x)[row_token])
    res = expert_rows(x_perm, row_expert, W1, W3, W2, want_h_mid=want_h_mid, nthreads=nthreads)
    y_perm, h_mid = (res if want_h_mid else (res, None))
    y = combine(y_perm, row_map, r["topk_prob"], nthreads)
    if W1s is not None:
        y_shared, h_mid_s = shared_expert(x, W1s, W3s, W2s, want_h_mid=True, nthreads=nthreads)
        r.update({"y_routed": y, "y_shared": y_shared, "h_mid_s": h_mid_s})
        y = y + y_shared
    r.update({"offsets": offsets, "row_map": row_map, "row_token": row_token,
              "x_perm": x_perm, "y_perm": y_perm, "h_mid": h_mid, "y": y})
    return r


# ------------------------------------------------------------------- FP8 --

def e4m3_values():
    """The value of every E4M3 code 0..255 (float64; NaN for the NaN codes)."""
    out = np.empty(256, np.float64)
    _load().oracle_e4m3_values(_ptr(out))
    return out


def e4m3_codes(v):
    """E4M3 codes (nearest, ties to even, saturating at 448) of float64 values."""
    v = _c(np.asarray(v, np.float64), np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_codes(v.size, _ptr(v), _ptr(out))
    return out


def quantize_rows_e4m3(x, nthreads=0):
    """Per-row power-of-two-scaled E4M3: x [rows, cols] -> (codes, scales [rows])."""
    x = _c(x)
    rows, cols = x.shape
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows,), np.float32)
    _load().oracle_quantize_rows_e4m3(rows, cols, _ptr(x), _dtype_code(x), _ptr(codes),
                                      _ptr(scales), nthreads)
    return codes, scales


def quantize_cols_e4m3(W, nthreads=0):
    """Per-output-channel E4M3 of W [E,K,N] -> (codes [E,N,K], scales [E,N])."""
    W = _c(W)
    E, K, N = W.shape
    codes = np.empty((E, N, K), np.uint8)
    scales = np.empty((E, N), np.float32)
    _load().oracle_quantize_cols_e4m3(E, K, N, _ptr(W), _dtype_code(W), _ptr(codes),
                                      _ptr(scales), nthreads)
    return codes, scales


def quantize_experts_e4m3(W1, W3, W2, nthreads=0):
    """The FP8 form of the expert weights: dict of W1q/W3q [E,f,h], W2q [E,h,f]
    codes and s1/s3 [E,f], s2 [E,h] scales."""
    W1q, s1 = quantize_cols_e4m3(W1, nthreads)
    W3q, s3 = quantize_cols_e4m3(W3, nthreads)
    W2q, s2 = quantize_cols_e4m3(W2, nthreads)
    return {"W1q": W1q, "s1": s1, "W3q": W3q, "s3": s3, "W2q": W2q, "s2": s2}


def expert_rows_fp8(xq, xs, row_expert, q, nthreads=0):
    """FP8 SwiGLU rows: returns dict y_rows [R,h], h_mid [R,f] (bf16 values),
    hq [R,f] codes, hs [R] scales (float64 / uint8 / float32)."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    row_expert = _c(row_expert, np.int32)
    R, h = xq.shape
    f = q["W1q"].shape[1]
    y = np.empty((R, h), np.float64)
    hm = np.empty((R, f), np.float64)
    hq = np.empty((R, f), np.uint8)
    hs = np.empty((R,), np.float32)
    _load().oracle_expert_rows_fp8(R, h, f, _ptr(xq), _ptr(xs), _ptr(row_expert),
                                   _ptr(_c(q["W1q"], np.uint8)), _ptr(_c(q["s1"], np.float32)),
                                   _ptr(_c(q["W3q"], np.uint8)), _ptr(_c(q["s3"], np.float32)),
                                   _ptr(_c(q["W2q"], np.uint8)), _ptr(_c(q["s2"], np.float32)),
                                   _ptr(hm), _ptr(hq), _ptr(hs), _ptr(y), nthreads)
    return {"y_rows": y, "h_mid": hm, "hq": hq, "hs": hs}


def forward_fp8(x, Wg, q, k, score, gate_bias=None, expert_bias=None, capacity_factor=0.0,
                min_capacity=0, drop_policy="probs", nthreads=0, num_groups=0, group_topk=0,
                pad_to_capacity=False):
    """The layer with FP8 experts: route -> drop -> permute -> (x quantised per
    token) FP8 SwiGLU experts -> combine.  q: quantize_experts_e4m3(...).
    pad_to_capacity: the experts run on the padded routing map's rows, as in
    forward()."""
    r = route(x, Wg, k, score, gate_bias, expert_bias, capacity_factor, min_capacity,
              drop_policy, nthreads, num_groups, group_topk, pad_to_capacity)
    E = Wg.shape[1]
    if pad_to_capacity:
        offsets, row_map, row_token = permute_map(r["routing_map"], r["topk_idx"], r["keep"])
    else:
        offsets, row_map, row_token = permute(r["topk_idx"], r["keep"], E)
    row_expert = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    xq, xs = quantize_rows_e4m3(x, nthreads)
    res = expert_rows_fp8(xq[row_token], xs[row_token], row_expert, q, nthreads)
    y = combine(res["y_rows"], row_map, r["topk_prob"], nthreads)
    r.update({"offsets": offsets, "row_map": row_map, "row_token": row_token, "xq": xq,
              "xs": xs, "y_perm": res["y_rows"], "h_mid": res["h_mid"], "hq": res["hq"],
              "hs": res["hs"], "y": y})
    return r


# -------------------------------------------------------------- backward --

def backward(x, Wg, W1, W3, W2, k, score, topk_idx, topk_prob, keep, dy, gate_bias=None,
             expert_bias=None, nthreads=0, weight_grads=True):
    """Gradients of sum(dy * y) for the routing decisions topk_idx / keep and
    the combine weights topk_prob (as route() returns them).  Returns a dict of float64 arrays: dx [T,h],
    dWg [h,E], dgate_bias [E], dW1/dW3 [E,h,f], dW2 [E,f,h], dlogits [T,E];
    weight_grads=False leaves the expert weight gradients out (None)."""
    x, dy = _c(x), _c(dy)
    Wg = _c(Wg, np.float32)
    gate_bias = _c(gate_bias, np.float32)
    expert_bias = _c(expert_bias, np.float32)
    W1, W3, W2 = _c(W1), _c(W3), _c(W2)
    topk_idx = _c(topk_idx, np.int32)
    topk_prob = _c(topk_prob, np.float32)
    keep = _c(keep, np.uint8)
    T, h = x.shape
    E = Wg.shape[1]
    f = W1.shape[-1]
    wd = _dtype_code(W1)
    out = {"dx": np.empty((T, h)), "dWg": np.empty((h, E)), "dgate_bias": np.empty(E),
           "dW1": np.empty((E, h, f)) if weight_grads else None,
           "dW3": np.empty((E, h, f)) if weight_grads else None,
           "dW2": np.empty((E, f, h)) if weight_grads else None,
           "dlogits": np.empty((T, E))}
    _load().oracle_backward(T, h, E, k, f, SCORES[score], _ptr(x), _dtype_code(x), _ptr(Wg),
                            _ptr(gate_bias), _ptr(expert_bias), _ptr(W1), _ptr(W3), _ptr(W2), wd,
                            _ptr(topk_idx), _ptr(topk_prob), _ptr(keep), _ptr(dy),
                            _dtype_code(dy),
                            _ptr(out["dx"]), _ptr(out["dWg"]), _ptr(out["dgate_bias"]),
                            _ptr(out["dW1"]), _ptr(out["dW3"]), _ptr(out["dW2"]),
                            _ptr(out["dlogits"]), nthreads)
    return out


def shared_backward(x, W1s, W3s, W2s, dy, nthreads=0):
    """Gradients of sum(dy * Y_shared) for the shared expert (weights W1s,
    W3s [h,fs], W2s [fs,h]): the routed backward of ONE expert that every
    token reaches with weight 1 (E = 1, k = 1, softmax after top-1: the
    softmax over one logit is exactly 1 and passes no gradient to the
    router).  Returns float64 dx [T,h], dW1s, dW3s [h,fs], dW2s [fs,h]."""
    x = _c(x)
    T, h = x.shape
    one = np.zeros((T, 1), np.int32)
    g = backward(x, np.zeros((h, 1), np.float32), _c(W1s)[None], _c(W3s)[None], _c(W2s)[None],
                 1, "softmax_post", one, np.ones((T, 1), np.float32), np.ones((T, 1), np.uint8),
                 dy, nthreads=nthreads)
    assert not np.any(g["dlogits"]), "one expert of weight 1 passes no router gradient"
    return {"dx": g["dx"], "dW1s": g["dW1"][0], "dW3s": g["dW3"][0], "dW2s": g["dW2"][0]}


def expert_wgrad_cols(x_rows, p, dy_rows, W1e, W3e, W2e, rows_c, cols_c, nthreads=0):
    """Selected weight gradients of ONE expert from its rows: x_rows [R,h],
    combine weights p [R], dy_rows [R,h] (dy of the tokens behind the rows),
    weights W1e/W3e [h,f], W2e [f,h].  Returns float64 arrays dW2 rows
    [len(rows_c), h] (dW2[c, :] for c in rows_c) and dW1 / dW3 columns
    [h, len(cols_c)] (dW1[:, c] for c in cols_c)."""
    x_rows, dy_rows = _c(x_rows), _c(dy_rows)
    p = _c(p, np.float32)
    W1e, W3e, W2e = _c(W1e), _c(W3e), _c(W2e)
    rows_c = _c(np.asarray(rows_c), np.int32)
    cols_c = _c(np.asarray(cols_c), np.int32)
    R, h = x_rows.shape
    f = W1e.shape[1]
    n2, n13 = rows_c.size, cols_c.size
    d2 = np.empty((n2, h))
    d1 = np.empty((h, n13))
    d3 = np.empty((h, n13))
    _load().oracle_expert_wgrad_cols(R, h, f, _ptr(x_rows), _dtype_code(x_rows), _ptr(p),
                                     _ptr(dy_rows), _dtype_code(dy_rows), _ptr(W1e), _ptr(W3e),
                                     _ptr(W2e), _dtype_code(W1e), n2, _ptr(rows_c), n13,
                                     _ptr(cols_c), _ptr(d2), _ptr(d1), _ptr(d3), nthreads)
    return {"dW2_rows": d2, "dW1_cols": d1, "dW3_cols": d3}
