"""ctypes binding of libmoe_gb300.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
Tensors are torch CUDA tensors (contiguous); the current torch stream is
passed to the library.  There is no CPU or PyTorch fallback: if the
library is missing, `lib()` raises.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_gb300.so")

SCORE = {"softmax_post": 0, "softmax_pre": 1, "sigmoid": 2, "sqrtsoftplus": 3}
DTYPE = {"f32": 0, "bf16": 1}
DROP_POLICY = {"probs": 0, "position": 1}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_CHECK", 6: "MOE_ERR_TIMEOUT"}

# every function declared in include/moe.h
EXPORTS = ["moe_abi_version", "moe_status_string", "moe_last_cuda_error", "moe_capacity",
           "moe_workspace_size", "moe_max_rows", "moe_route", "moe_permute", "moe_grouped_mlp",
           "moe_grouped_fc1", "moe_grouped_fc2", "moe_combine", "moe_forward", "moe_check",
           "moe_permute_noalloc", "moe_selftest_wait_timeout", "moe_shared_expert",
           "moe_combine_shared", "moe_workspace_size_shared", "moe_forward_shared",
           "moe_probe_fp32_fma", "moe_workspace_size_host", "moe_forward_host",
           "moe_quantize_rows_e4m3", "moe_quantize_experts_e4m3", "moe_workspace_size_e4m3",
           "moe_permute_e4m3", "moe_grouped_mlp_e4m3", "moe_forward_e4m3",
           "moe_grouped_fc1_e4m3", "moe_grouped_fc2_e4m3", "moe_workspace_size_backward",
           "moe_backward", "moe_workspace_size_backward_shared", "moe_backward_shared",
           "moe_shared_expert_backward", "moe_workspace_size_host_shared",
           "moe_forward_host_shared", "moe_workspace_size_host_e4m3", "moe_forward_host_e4m3",
           "moe_permute_map", "moe_permute_map_e4m3", "moe_grouped_fc2_combine",
           "moe_grouped_fc2_f16s", "moe_combine_f16s", "moe_grouped_fc2_e4m3_f16s"]


class MoeConfig(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("ffn_hidden", ctypes.c_int32), ("score", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("drop_policy", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("min_capacity", ctypes.c_int32),
                ("num_groups", ctypes.c_int32), ("group_topk", ctypes.c_int32),
                ("pad_to_capacity", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, code, where, detail=""):
        self.code = code
        msg = "%s failed: %s" % (where, STATUS.get(code, code))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_gb300.so is not built (expected at %s); run "
                               "mixture_experts_layer_fp32_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
        cfgp = ctypes.POINTER(MoeConfig)
        sig = {
            "moe_abi_version": ([], i32),
            "moe_status_string": ([i32], ctypes.c_char_p),
            "moe_last_cuda_error": ([], ctypes.c_char_p),
            "moe_capacity": ([cfgp, ctypes.POINTER(i64)], i32),
            "moe_workspace_size": ([cfgp, ctypes.POINTER(sz)], i32),
            "moe_max_rows": ([cfgp, ctypes.POINTER(i64)], i32),
            "moe_route": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_permute": ([cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_permute_map": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_permute_map_e4m3": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_grouped_mlp": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_grouped_fc1": ([cfgp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_grouped_fc2": ([cfgp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_combine": ([cfgp, vp, vp, vp, vp, vp], i32),
            "moe_grouped_fc2_combine": ([cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_grouped_fc2_f16s": ([cfgp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_combine_f16s": ([cfgp, vp, vp, vp, vp, vp, vp, vp], i32),
            "moe_forward": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_check": ([vp, vp, ctypes.POINTER(i32)], i32),
            "moe_permute_noalloc": ([cfgp, vp, vp, vp, vp, vp, vp, vp], i32),
            "moe_selftest_wait_timeout": ([vp, sz, i64, vp], i32),
            "moe_shared_expert": ([cfgp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_combine_shared": ([cfgp, vp, vp, vp, vp, vp, vp], i32),
            "moe_workspace_size_shared": ([cfgp, i32, ctypes.POINTER(sz)], i32),
            "moe_forward_shared": ([cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    vp, vp, sz, vp], i32),
            "moe_probe_fp32_fma": ([i64, vp, ctypes.POINTER(ctypes.c_double), vp], i32),
            "moe_workspace_size_host": ([cfgp, ctypes.POINTER(sz)], i32),
            "moe_forward_host": ([cfgp, i32, vp, sz, vp, sz, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                                 i32),
            "moe_quantize_rows_e4m3": ([i64, i32, vp, vp, vp, vp], i32),
            "moe_quantize_experts_e4m3": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp], i32),
            "moe_workspace_size_e4m3": ([cfgp, ctypes.POINTER(sz)], i32),
            "moe_permute_e4m3": ([cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_grouped_mlp_e4m3": ([cfgp] + [vp] * 13 + [vp, sz, vp], i32),
            "moe_forward_e4m3": ([cfgp] + [vp] * 14 + [vp, sz, vp], i32),
            "moe_grouped_fc1_e4m3": ([cfgp] + [vp] * 8 + [vp, sz, vp], i32),
            "moe_grouped_fc2_e4m3": ([cfgp] + [vp] * 7 + [vp, sz, vp], i32),
            "moe_grouped_fc2_e4m3_f16s": ([cfgp] + [vp] * 8 + [vp, sz, vp], i32),
            "moe_workspace_size_backward": ([cfgp, ctypes.POINTER(sz)], i32),
            "moe_backward": ([cfgp] + [vp] * 20 + [vp, sz, vp], i32),
            "moe_workspace_size_backward_shared": ([cfgp, i32, ctypes.POINTER(sz)], i32),
            "moe_backward_shared": ([cfgp, i32] + [vp] * 27 + [vp, sz, vp], i32),
            "moe_shared_expert_backward": ([cfgp, i32] + [vp] * 10 + [vp, sz, vp], i32),
            "moe_workspace_size_host_shared": ([cfgp, i32, ctypes.POINTER(sz)], i32),
            "moe_forward_host_shared": ([cfgp, i32, i32, vp, sz, vp, sz] + [vp] * 9 +
                                        [vp, sz, vp], i32),
            "moe_workspace_size_host_e4m3": ([cfgp, ctypes.POINTER(sz)], i32),
            "moe_forward_host_e4m3": ([cfgp, i32, vp, sz, vp, sz] + [vp] * 9 + [vp, sz, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def config(T, h, E, k, f, score="softmax_post", dtype="bf16", capacity_factor=0.0,
           min_capacity=0, drop_policy="probs", num_groups=0, group_topk=0,
           pad_to_capacity=False):
    return MoeConfig(int(T), int(h), int(E), int(k), int(f), SCORE[score], DTYPE[dtype],
                     DROP_POLICY[drop_policy], float(capacity_factor), int(min_capacity),
                     int(num_groups), int(group_topk), int(bool(pad_to_capacity)))


def _check(code, where):
    if code != 0:
        detail = lib().moe_last_cuda_error().decode() if code == 4 else ""
        raise MoeError(code, where, detail)


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _host(t):
    """Pointer of a HOST tensor (the host-I/O entry point's batches)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if t.is_cuda:
        raise ValueError("x_host / y_host must be host tensors (ideally pinned)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _ws(ws):
    return _p(ws), ws.numel() * ws.element_size()


def act_dtype(cfg):
    return torch.float32 if cfg.dtype == DTYPE["f32"] else torch.bfloat16


def capacity(cfg):
    v = ctypes.c_int64()
    _check(lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(v)), "moe_capacity")
    return v.value


def workspace_size(cfg):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(v)), "moe_workspace_size")
    return v.value


def max_rows(cfg):
    v = ctypes.c_int64()
    _check(lib().moe_max_rows(ctypes.byref(cfg), ctypes.byref(v)), "moe_max_rows")
    return v.value


def alloc_workspace(cfg, device="cuda"):
    """Zero-filled workspace of moe_workspace_size(cfg) bytes."""
    return torch.zeros(workspace_size(cfg), dtype=torch.uint8, device=device)


def route(cfg, x, Wg, gate_bias, expert_bias, topk_idx, topk_prob, keep, tokens_per_expert,
          routing_map, ws):
    w, wb = _ws(ws)
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(Wg), _p(gate_bias), _p(expert_bias),
                           _p(topk_idx), _p(topk_prob), _p(keep), _p(tokens_per_expert),
                           _p(routing_map), w, wb, _stream()), "moe_route")


def permute(cfg, x, topk_idx, keep, x_perm, row_map, expert_offsets, ws):
    w, wb = _ws(ws)
    _check(lib().moe_permute(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(keep), _p(x_perm),
                             _p(row_map), _p(expert_offsets), w, wb, _stream()), "moe_permute")


def permute_map(cfg, x, routing_map, topk_idx, keep, x_perm, row_map, expert_offsets, ws):
    """moe_permute_map: the permutation driven by a [T,E] routing map."""
    w, wb = _ws(ws)
    _check(lib().moe_permute_map(ctypes.byref(cfg), _p(x), _p(routing_map), _p(topk_idx),
                                 _p(keep), _p(x_perm), _p(row_map), _p(expert_offsets), w, wb,
                                 _stream()), "moe_permute_map")


def permute_noalloc(cfg, x, topk_idx, keep, x_perm, row_map, expert_offsets):
    """moe_permute without a workspace (scratch in a fixed array inside the
    library; for callers that cannot provide device memory)."""
    _check(lib().moe_permute_noalloc(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(keep),
                                     _p(x_perm), _p(row_map), _p(expert_offsets), _stream()),
           "moe_permute_noalloc")


def grouped_fc1(cfg, x_perm, expert_offsets, W1, W3, h_mid, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc1(ctypes.byref(cfg), _p(x_perm), _p(expert_offsets), _p(W1),
                                 _p(W3), _p(h_mid), w, wb, _stream()), "moe_grouped_fc1")


def grouped_fc2(cfg, h_mid, expert_offsets, W2, y_perm, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc2(ctypes.byref(cfg), _p(h_mid), _p(expert_offsets), _p(W2),
                                 _p(y_perm), w, wb, _stream()), "moe_grouped_fc2")


def grouped_mlp(cfg, x_perm, expert_offsets, W1, W3, W2, h_mid, y_perm, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_mlp(ctypes.byref(cfg), _p(x_perm), _p(expert_offsets), _p(W1),
                                 _p(W3), _p(W2), _p(h_mid), _p(y_perm), w, wb, _stream()),
           "moe_grouped_mlp")


def grouped_fc2_combine(cfg, h_mid, expert_offsets, W2, row_map, topk_prob, y, ws):
    """moe_grouped_fc2_combine: fc2 and the combine of a top-1 layer in one call."""
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc2_combine(ctypes.byref(cfg), _p(h_mid), _p(expert_offsets),
                                         _p(W2), _p(row_map), _p(topk_prob), _p(y), w, wb,
                                         _stream()), "moe_grouped_fc2_combine")


def grouped_fc2_f16s(cfg, h_mid, expert_offsets, W2, y16, y16_exp, ws):
    """moe_grouped_fc2_f16s: fc2 with y_perm as fp16 (y16, torch.float16
    [R, h]) and one power-of-two exponent per 32 columns (y16_exp, int8)."""
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc2_f16s(ctypes.byref(cfg), _p(h_mid), _p(expert_offsets), _p(W2),
                                      _p(y16), _p(y16_exp), w, wb, _stream()),
           "moe_grouped_fc2_f16s")


def combine_f16s(cfg, y16, y16_exp, row_map, topk_prob, y, y_shared=None):
    """moe_combine_f16s: the combine over that y_perm (plus the shared
    expert's fp32 output y_shared, if given)."""
    _check(lib().moe_combine_f16s(ctypes.byref(cfg), _p(y16), _p(y16_exp), _p(row_map),
                                  _p(topk_prob), _p(y_shared), _p(y), _stream()),
           "moe_combine_f16s")


def combine(cfg, y_perm, row_map, topk_prob, y):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(y_perm), _p(row_map), _p(topk_prob), _p(y),
                             _stream()), "moe_combine")


def forward(cfg, x, Wg, gate_bias, expert_bias, W1, W3, W2, y, ws, topk_idx=None,
            topk_prob=None, tokens_per_expert=None):
    w, wb = _ws(ws)
    _check(lib().moe_forward(ctypes.byref(cfg), _p(x), _p(Wg), _p(gate_bias), _p(expert_bias),
                             _p(W1), _p(W3), _p(W2), _p(y), _p(topk_idx), _p(topk_prob),
                             _p(tokens_per_expert), w, wb, _stream()), "moe_forward")


def workspace_size_shared(cfg, fs):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_shared(ctypes.byref(cfg), int(fs), ctypes.byref(v)),
           "moe_workspace_size_shared")
    return v.value


def alloc_workspace_shared(cfg, fs, device="cuda"):
    """Zero-filled workspace for forward_shared (moe_workspace_size_shared bytes)."""
    return torch.zeros(workspace_size_shared(cfg, fs), dtype=torch.uint8, device=device)


def shared_expert(cfg, fs, x, W1s, W3s, W2s, h_mid_s, y_shared, ws):
    w, wb = _ws(ws)
    _check(lib().moe_shared_expert(ctypes.byref(cfg), int(fs), _p(x), _p(W1s), _p(W3s), _p(W2s),
                                   _p(h_mid_s), _p(y_shared), w, wb, _stream()),
           "moe_shared_expert")


def combine_shared(cfg, y_perm, row_map, topk_prob, y_shared, y):
    _check(lib().moe_combine_shared(ctypes.byref(cfg), _p(y_perm), _p(row_map), _p(topk_prob),
                                    _p(y_shared), _p(y), _stream()), "moe_combine_shared")


def forward_shared(cfg, fs, x, Wg, gate_bias, expert_bias, W1, W3, W2, W1s, W3s, W2s, y, ws,
                   topk_idx=None, topk_prob=None, tokens_per_expert=None):
    w, wb = _ws(ws)
    _check(lib().moe_forward_shared(ctypes.byref(cfg), int(fs), _p(x), _p(Wg), _p(gate_bias),
                                    _p(expert_bias), _p(W1), _p(W3), _p(W2), _p(W1s), _p(W3s),
                                    _p(W2s), _p(y), _p(topk_idx), _p(topk_prob),
                                    _p(tokens_per_expert), w, wb, _stream()),
           "moe_forward_shared")


def workspace_size_host(cfg):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_host(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_workspace_size_host")
    return v.value


def alloc_workspace_host(cfg, device="cuda"):
    """Zero-filled workspace for forward_host (moe_workspace_size_host bytes)."""
    return torch.zeros(workspace_size_host(cfg), dtype=torch.uint8, device=device)


def forward_host(cfg, x_host, y_host, Wg, gate_bias, expert_bias, W1, W3, W2, ws,
                 num_batches=None):
    """The forward over host batches x_host [B,T,h] -> y_host [B,T,h] (or one
    [T,h] buffer reused num_batches times, stride 0), copies pipelined with
    compute on the library's copy streams.  Asynchronous on the current
    stream."""
    T, h = cfg.num_tokens, cfg.hidden
    if num_batches is None:
        num_batches = x_host.shape[0] if x_host.dim() == 3 else 1
    xs = x_host[0].numel() * x_host.element_size() if x_host.dim() == 3 else 0
    ys = y_host[0].numel() * y_host.element_size() if y_host.dim() == 3 else 0
    for t, stride in ((x_host, xs), (y_host, ys)):
        per = T * h * t.element_size()
        if (t.numel() * t.element_size()) < (per if stride == 0 else per * num_batches):
            raise ValueError("host buffer smaller than its batches")
    w, wb = _ws(ws)
    _check(lib().moe_forward_host(ctypes.byref(cfg), int(num_batches), _host(x_host), xs,
                                  _host(y_host), ys, _p(Wg), _p(gate_bias), _p(expert_bias),
                                  _p(W1), _p(W3), _p(W2), w, wb, _stream()), "moe_forward_host")


def _host_batches(cfg, x_host, y_host, num_batches):
    """Batch count and byte strides of host buffers [B,T,h] (or [T,h] reused)."""
    T, h = cfg.num_tokens, cfg.hidden
    if num_batches is None:
        num_batches = x_host.shape[0] if x_host.dim() == 3 else 1
    xs = x_host[0].numel() * x_host.element_size() if x_host.dim() == 3 else 0
    ys = y_host[0].numel() * y_host.element_size() if y_host.dim() == 3 else 0
    for t, stride in ((x_host, xs), (y_host, ys)):
        per = T * h * t.element_size()
        if (t.numel() * t.element_size()) < (per if stride == 0 else per * num_batches):
            raise ValueError("host buffer smaller than its batches")
    return num_batches, xs, ys


def workspace_size_host_shared(cfg, fs):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_host_shared(ctypes.byref(cfg), int(fs), ctypes.byref(v)),
           "moe_workspace_size_host_shared")
    return v.value


def alloc_workspace_host_shared(cfg, fs, device="cuda"):
    return torch.zeros(workspace_size_host_shared(cfg, fs), dtype=torch.uint8, device=device)


def forward_host_shared(cfg, fs, x_host, y_host, Wg, gate_bias, expert_bias, W1, W3, W2, W1s,
                        W3s, W2s, ws, num_batches=None):
    """forward_host with the shared expert (moe_forward_shared per batch)."""
    n, xs, ys = _host_batches(cfg, x_host, y_host, num_batches)
    w, wb = _ws(ws)
    _check(lib().moe_forward_host_shared(ctypes.byref(cfg), int(fs), int(n), _host(x_host), xs,
                                         _host(y_host), ys, _p(Wg), _p(gate_bias),
                                         _p(expert_bias), _p(W1), _p(W3), _p(W2), _p(W1s),
                                         _p(W3s), _p(W2s), w, wb, _stream()),
           "moe_forward_host_shared")


def workspace_size_host_e4m3(cfg):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_host_e4m3(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_workspace_size_host_e4m3")
    return v.value


def alloc_workspace_host_e4m3(cfg, device="cuda"):
    return torch.zeros(workspace_size_host_e4m3(cfg), dtype=torch.uint8, device=device)


def forward_host_e4m3(cfg, x_host, y_host, Wg, gate_bias, expert_bias, q, ws, num_batches=None):
    """forward_host with E4M3 experts (moe_forward_e4m3 per batch); q: E4m3Experts."""
    n, xs, ys = _host_batches(cfg, x_host, y_host, num_batches)
    w, wb = _ws(ws)
    _check(lib().moe_forward_host_e4m3(ctypes.byref(cfg), int(n), _host(x_host), xs,
                                       _host(y_host), ys, _p(Wg), _p(gate_bias), _p(expert_bias),
                                       _p(q.W1q), _p(q.s1), _p(q.W3q), _p(q.s3), _p(q.W2q),
                                       _p(q.s2), w, wb, _stream()), "moe_forward_host_e4m3")


# ------------------------------------------------------------- E4M3 experts

def quantize_rows_e4m3(x, codes, scales):
    """x [rows, cols] bf16 -> codes [rows, cols] uint8, scales [rows] fp32."""
    rows, cols = x.shape
    _check(lib().moe_quantize_rows_e4m3(rows, cols, _p(x), _p(codes), _p(scales), _stream()),
           "moe_quantize_rows_e4m3")


class E4m3Experts:
    """The expert weights in E4M3 (device tensors): W1q/W3q [E,f,h], W2q [E,h,f]
    uint8 codes, s1/s3 [E,f] and s2 [E,h] fp32 scales."""

    def __init__(self, cfg, W1, W3, W2):
        E, h, f = cfg.num_experts, cfg.hidden, cfg.ffn_hidden
        d = W1.device
        self.W1q = torch.empty((E, f, h), dtype=torch.uint8, device=d)
        self.W3q = torch.empty((E, f, h), dtype=torch.uint8, device=d)
        self.W2q = torch.empty((E, h, f), dtype=torch.uint8, device=d)
        self.s1 = torch.empty((E, f), dtype=torch.float32, device=d)
        self.s3 = torch.empty((E, f), dtype=torch.float32, device=d)
        self.s2 = torch.empty((E, h), dtype=torch.float32, device=d)
        _check(lib().moe_quantize_experts_e4m3(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2),
                                               _p(self.W1q), _p(self.W3q), _p(self.W2q),
                                               _p(self.s1), _p(self.s3), _p(self.s2), _stream()),
               "moe_quantize_experts_e4m3")


def workspace_size_e4m3(cfg):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_e4m3(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_workspace_size_e4m3")
    return v.value


def alloc_workspace_e4m3(cfg, device="cuda"):
    return torch.zeros(workspace_size_e4m3(cfg), dtype=torch.uint8, device=device)


def permute_map_e4m3(cfg, x, routing_map, topk_idx, keep, x_perm_q, x_perm_scale, row_map,
                     expert_offsets, ws):
    """moe_permute_map_e4m3: the E4M3 permutation by the padded routing map."""
    w, wb = _ws(ws)
    _check(lib().moe_permute_map_e4m3(ctypes.byref(cfg), _p(x), _p(routing_map), _p(topk_idx),
                                      _p(keep), _p(x_perm_q), _p(x_perm_scale), _p(row_map),
                                      _p(expert_offsets), w, wb, _stream()),
           "moe_permute_map_e4m3")


def permute_e4m3(cfg, x, topk_idx, keep, x_perm_q, x_perm_scale, row_map, expert_offsets, ws):
    w, wb = _ws(ws)
    _check(lib().moe_permute_e4m3(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(keep), _p(x_perm_q),
                                  _p(x_perm_scale), _p(row_map), _p(expert_offsets), w, wb,
                                  _stream()), "moe_permute_e4m3")


def grouped_mlp_e4m3(cfg, x_perm_q, x_perm_scale, expert_offsets, q, h_mid, h_q, h_scale,
                     y_perm, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_mlp_e4m3(ctypes.byref(cfg), _p(x_perm_q), _p(x_perm_scale),
                                      _p(expert_offsets), _p(q.W1q), _p(q.s1), _p(q.W3q),
                                      _p(q.s3), _p(q.W2q), _p(q.s2), _p(h_mid), _p(h_q),
                                      _p(h_scale), _p(y_perm), w, wb, _stream()),
           "moe_grouped_mlp_e4m3")


def grouped_fc1_e4m3(cfg, x_perm_q, x_perm_scale, expert_offsets, q, h_mid, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc1_e4m3(ctypes.byref(cfg), _p(x_perm_q), _p(x_perm_scale),
                                      _p(expert_offsets), _p(q.W1q), _p(q.s1), _p(q.W3q),
                                      _p(q.s3), _p(h_mid), w, wb, _stream()),
           "moe_grouped_fc1_e4m3")


def grouped_fc2_e4m3(cfg, h_mid, expert_offsets, q, h_q, h_scale, y_perm, ws):
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc2_e4m3(ctypes.byref(cfg), _p(h_mid), _p(expert_offsets),
                                      _p(q.W2q), _p(q.s2), _p(h_q), _p(h_scale), _p(y_perm), w,
                                      wb, _stream()), "moe_grouped_fc2_e4m3")


def grouped_fc2_e4m3_f16s(cfg, h_mid, expert_offsets, q, h_q, h_scale, y16, y16_exp, ws):
    """moe_grouped_fc2_e4m3_f16s: the E4M3 fc2 into the fp16 y_perm (a
    power-of-two scale per 32 columns), for combine_f16s."""
    w, wb = _ws(ws)
    _check(lib().moe_grouped_fc2_e4m3_f16s(ctypes.byref(cfg), _p(h_mid), _p(expert_offsets),
                                           _p(q.W2q), _p(q.s2), _p(h_q), _p(h_scale), _p(y16),
                                           _p(y16_exp), w, wb, _stream()),
           "moe_grouped_fc2_e4m3_f16s")


def forward_e4m3(cfg, x, Wg, gate_bias, expert_bias, q, y, ws, topk_idx=None, topk_prob=None,
                 tokens_per_expert=None):
    w, wb = _ws(ws)
    _check(lib().moe_forward_e4m3(ctypes.byref(cfg), _p(x), _p(Wg), _p(gate_bias),
                                  _p(expert_bias), _p(q.W1q), _p(q.s1), _p(q.W3q), _p(q.s3),
                                  _p(q.W2q), _p(q.s2), _p(y), _p(topk_idx), _p(topk_prob),
                                  _p(tokens_per_expert), w, wb, _stream()), "moe_forward_e4m3")


# ------------------------------------------------------------------ backward

def workspace_size_backward(cfg):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_backward(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_workspace_size_backward")
    return v.value


def alloc_workspace_backward(cfg, device="cuda"):
    return torch.zeros(workspace_size_backward(cfg), dtype=torch.uint8, device=device)


class Grads:
    """Gradient buffers of one backward (dx bf16, the rest fp32)."""

    def __init__(self, cfg, device="cuda"):
        T, h, E, f = cfg.num_tokens, cfg.hidden, cfg.num_experts, cfg.ffn_hidden
        d = torch.device(device)
        self.dx = torch.empty((T, h), dtype=act_dtype(cfg), device=d)
        self.dWg = torch.empty((h, E), dtype=torch.float32, device=d)
        self.dgate_bias = torch.empty((E,), dtype=torch.float32, device=d)
        self.dW1 = torch.empty((E, h, f), dtype=torch.float32, device=d)
        self.dW3 = torch.empty((E, h, f), dtype=torch.float32, device=d)
        self.dW2 = torch.empty((E, f, h), dtype=torch.float32, device=d)


def backward(cfg, x, Wg, gate_bias, W1, W3, W2, saved, dy, g, ws):
    """saved: a Buffers object after the staged forward (topk_idx, topk_prob,
    row_map, expert_offsets, x_perm, h_mid, y_perm); g: Grads."""
    w, wb = _ws(ws)
    _check(lib().moe_backward(ctypes.byref(cfg), _p(x), _p(Wg), _p(gate_bias), _p(W1), _p(W3),
                              _p(W2), _p(saved.topk_idx), _p(saved.topk_prob), _p(saved.row_map),
                              _p(saved.expert_offsets), _p(saved.x_perm), _p(saved.h_mid),
                              _p(saved.y_perm), _p(dy), _p(g.dx), _p(g.dWg), _p(g.dgate_bias),
                              _p(g.dW1), _p(g.dW3), _p(g.dW2), w, wb, _stream()), "moe_backward")


class SharedGrads:
    """The shared expert's weight gradients (fp32): dW1s, dW3s [h,fs], dW2s [fs,h]."""

    def __init__(self, cfg, fs, device="cuda"):
        h = cfg.hidden
        d = torch.device(device)
        self.dW1s = torch.empty((h, fs), dtype=torch.float32, device=d)
        self.dW3s = torch.empty((h, fs), dtype=torch.float32, device=d)
        self.dW2s = torch.empty((fs, h), dtype=torch.float32, device=d)


def workspace_size_backward_shared(cfg, fs):
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size_backward_shared(ctypes.byref(cfg), int(fs), ctypes.byref(v)),
           "moe_workspace_size_backward_shared")
    return v.value


def alloc_workspace_backward_shared(cfg, fs, device="cuda"):
    return torch.zeros(workspace_size_backward_shared(cfg, fs), dtype=torch.uint8, device=device)


def backward_shared(cfg, fs, x, Wg, gate_bias, W1, W3, W2, W1s, W3s, W2s, saved, dy, g, gs, ws):
    """The layer backward with the shared expert: saved as for backward() plus
    h_mid_s; g: Grads (dx includes the shared path), gs: SharedGrads."""
    w, wb = _ws(ws)
    _check(lib().moe_backward_shared(
        ctypes.byref(cfg), int(fs), _p(x), _p(Wg), _p(gate_bias), _p(W1), _p(W3), _p(W2),
        _p(W1s), _p(W3s), _p(W2s), _p(saved.topk_idx), _p(saved.topk_prob), _p(saved.row_map),
        _p(saved.expert_offsets), _p(saved.x_perm), _p(saved.h_mid), _p(saved.y_perm),
        _p(saved.h_mid_s), _p(dy), _p(g.dx), _p(g.dWg), _p(g.dgate_bias), _p(g.dW1), _p(g.dW3),
        _p(g.dW2), _p(gs.dW1s), _p(gs.dW3s), _p(gs.dW2s), w, wb, _stream()),
        "moe_backward_shared")


def shared_expert_backward(cfg, fs, x, W1s, W3s, W2s, h_mid_s, dy, dx_acc, gs, ws):
    """The shared expert's backward alone: its dx is ADDED to dx_acc (fp32 [T,h])."""
    w, wb = _ws(ws)
    _check(lib().moe_shared_expert_backward(ctypes.byref(cfg), int(fs), _p(x), _p(W1s), _p(W3s),
                                            _p(W2s), _p(h_mid_s), _p(dy), _p(dx_acc),
                                            _p(gs.dW1s), _p(gs.dW3s), _p(gs.dW2s), w, wb,
                                            _stream()), "moe_shared_expert_backward")


def probe_fp32_fma(iters, out):
    """Enqueue the FP32 FMA-rate probe; returns the flops it performs (time it
    with CUDA events on the current stream).  `out`: float32 device buffer of
    4 * SM-count elements."""
    flops = ctypes.c_double()
    _check(lib().moe_probe_fp32_fma(int(iters), _p(out), ctypes.byref(flops), _stream()),
           "moe_probe_fp32_fma")
    return flops.value


def selftest_wait_timeout(ws, limit_cycles):
    """Enqueue a bounded wait that is made to run out (see include/moe.h)."""
    w, wb = _ws(ws)
    _check(lib().moe_selftest_wait_timeout(w, wb, int(limit_cycles), _stream()),
           "moe_selftest_wait_timeout")


def check(ws):
    """Synchronises the current stream and raises if a kernel flagged an error."""
    info = ctypes.c_int32(0)
    code = lib().moe_check(_p(ws), _stream(), ctypes.byref(info))
    if code != 0:
        raise MoeError(code, "device check", "info=%d" % info.value)


class Buffers:
    """Device buffers of one forward, allocated with torch (plumbing only)."""

    def __init__(self, cfg, device="cuda"):
        T, h, E, k, f = cfg.num_tokens, cfg.hidden, cfg.num_experts, cfg.topk, cfg.ffn_hidden
        R = max_rows(cfg)
        dt = act_dtype(cfg)
        d = torch.device(device)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=d)
        self.topk_prob = torch.empty((T, k), dtype=torch.float32, device=d)
        self.keep = torch.empty((T, k), dtype=torch.uint8, device=d)
        self.tokens_per_expert = torch.empty((E,), dtype=torch.int32, device=d)
        self.routing_map = torch.empty((T, E), dtype=torch.uint8, device=d)
        self.x_perm = torch.empty((R, h), dtype=dt, device=d)
        self.row_map = torch.empty((T, k), dtype=torch.int32, device=d)
        self.expert_offsets = torch.empty((E + 1,), dtype=torch.int32, device=d)
        self.h_mid = torch.empty((R, f), dtype=dt, device=d)
        self.y_perm = torch.empty((R, h), dtype=torch.float32, device=d)
        self.y = torch.empty((T, h), dtype=dt, device=d)
        self.ws = alloc_workspace(cfg, d)
