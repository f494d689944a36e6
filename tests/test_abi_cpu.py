"""The C ABI without a GPU: the library builds and loads, exports every
function that include/moe.h declares, and rejects bad arguments on the host
before anything would be enqueued (no call here reaches the CUDA runtime)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
FAKE = 0x10000          # a 16-byte-aligned address that is never dereferenced
MISALIGNED = 0x10004


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_fp32_gb300 import build
    build.build()
    import mixture_experts_layer_fp32_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_mlp", "moe_combine", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_function(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(moe.EXPORTS) == declared_functions()
    assert moe.lib().moe_abi_version() == 4
    assert moe.lib().moe_status_string(3) == b"MOE_ERR_WORKSPACE"


def _status(moe, fn, *args):
    return getattr(moe.lib(), fn)(*args)


def _cfgp(cfg):
    return ctypes.byref(cfg)


@pytest.mark.parametrize("field,value,want", [
    ("num_tokens", -1, INVALID), ("hidden", 0, INVALID), ("num_experts", 0, INVALID),
    ("topk", 0, INVALID), ("ffn_hidden", -8, INVALID),
    ("dtype", 2, INVALID), ("drop_policy", 5, INVALID), ("min_capacity", -1, INVALID),
    ("num_experts", 257, UNSUPPORTED), ("topk", 9, UNSUPPORTED), ("hidden", 4100, UNSUPPORTED),
    ("score", 4, INVALID), ("num_groups", -1, INVALID), ("group_topk", -2, INVALID),
    ("ffn_hidden", 1500, UNSUPPORTED), ("hidden", 4092, UNSUPPORTED),
])
def test_config_validation(moe, field, value, want):
    cfg = moe.config(T=64, h=4096, E=8, k=2, f=1536)
    setattr(cfg, field, value)
    size = ctypes.c_size_t()
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == want


def test_topk_larger_than_experts(moe):
    cfg = moe.config(T=64, h=4096, E=4, k=5, f=1536)
    size = ctypes.c_size_t()
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == UNSUPPORTED


def test_fp32_path_accepts_small_multiples_of_8(moe):
    cfg = moe.config(T=64, h=136, E=8, k=2, f=200, dtype="f32")
    size = ctypes.c_size_t()
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == OK
    assert size.value > 0


def test_capacity_matches_reading(moe):
    cfg = moe.config(T=32768, h=1024, E=64, k=1, f=4096, score="softmax_pre",
                     capacity_factor=1.25)
    assert moe.capacity(cfg) == 640
    assert moe.capacity(moe.config(T=10, h=256, E=4, k=2, f=128, capacity_factor=1.1)) == 6
    assert moe.capacity(moe.config(T=10, h=256, E=4, k=2, f=128)) == -1


def _route_args(cfg, ws_bytes, **over):
    a = dict(x=FAKE, Wg=FAKE, gb=None, eb=None, idx=FAKE, prob=FAKE, keep=FAKE, tpe=FAKE, rm=None,
             ws=FAKE, ws_bytes=ws_bytes, stream=None)
    a.update(over)
    return (ctypes.byref(cfg), a["x"], a["Wg"], a["gb"], a["eb"], a["idx"], a["prob"], a["keep"],
            a["tpe"], a["rm"], a["ws"], a["ws_bytes"], a["stream"])


def test_route_rejects_null_misaligned_and_small_workspace(moe):
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536)
    need = moe.workspace_size(cfg)
    lib = moe.lib()
    assert lib.moe_route(*_route_args(cfg, need, x=None)) == INVALID
    assert lib.moe_route(*_route_args(cfg, need, idx=None)) == INVALID
    assert lib.moe_route(*_route_args(cfg, need, x=MISALIGNED)) == INVALID
    assert lib.moe_route(*_route_args(cfg, need, ws=None)) == INVALID
    assert lib.moe_route(*_route_args(cfg, need - 1)) == WORKSPACE


def test_forward_and_stage_argument_checks(moe):
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536)
    need = moe.workspace_size(cfg)
    lib = moe.lib()
    # moe_forward: W2 missing
    assert lib.moe_forward(ctypes.byref(cfg), FAKE, FAKE, None, None, FAKE, FAKE, None, FAKE,
                           None, None, None, FAKE, need, None) == INVALID
    # moe_permute: x_perm misaligned
    assert lib.moe_permute(ctypes.byref(cfg), FAKE, FAKE, None, MISALIGNED, FAKE, FAKE, FAKE,
                           need, None) == INVALID
    # moe_grouped_fc1: workspace too small
    assert lib.moe_grouped_fc1(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16,
                               None) == WORKSPACE
    # moe_combine: y missing
    assert lib.moe_combine(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, None) == INVALID
    # moe_check: no workspace
    assert lib.moe_check(None, None, None) == INVALID


def test_fc2_combine_host_checks(moe):
    lib = moe.lib()
    top1 = moe.config(T=128, h=1024, E=8, k=1, f=512)
    need = moe.workspace_size(top1)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None]
    # padding rows have no slot to combine into
    pad = moe.config(T=128, h=1024, E=8, k=1, f=512, capacity_factor=1.0, pad_to_capacity=True)
    assert lib.moe_grouped_fc2_combine(ctypes.byref(pad), *args[:-2],
                                       moe.workspace_size(pad), None) == UNSUPPORTED
    # missing or misaligned pointers, short workspace
    bad = list(args)
    bad[6] = None  # y
    assert lib.moe_grouped_fc2_combine(ctypes.byref(top1), *bad) == INVALID
    bad = list(args)
    bad[0] = MISALIGNED  # h_mid
    assert lib.moe_grouped_fc2_combine(ctypes.byref(top1), *bad) == INVALID
    bad = list(args)
    bad[7] = need - 1
    assert lib.moe_grouped_fc2_combine(ctypes.byref(top1), *bad) == WORKSPACE


def test_permute_noalloc_host_checks(moe):
    lib = moe.lib()
    big = moe.config(T=70000, h=256, E=256, k=8, f=128)
    assert lib.moe_permute_noalloc(ctypes.byref(big), FAKE, FAKE, None, FAKE, FAKE, FAKE,
                                   None) == UNSUPPORTED
    small = moe.config(T=100, h=256, E=8, k=2, f=128)
    assert lib.moe_permute_noalloc(ctypes.byref(small), None, FAKE, None, FAKE, FAKE, FAKE,
                                   None) == INVALID


def test_binding_refuses_cpu_tensors(moe):
    import torch
    cfg = moe.config(T=4, h=256, E=4, k=2, f=128)
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        moe.permute(cfg, x, x, None, x, x, x, x)


def test_selftest_wait_timeout_host_checks(moe):
    lib = moe.lib()
    assert lib.moe_selftest_wait_timeout(None, 4096, 1000, None) == INVALID
    assert lib.moe_selftest_wait_timeout(FAKE, 100, 1000, None) == INVALID     # too small for the error word
    assert lib.moe_selftest_wait_timeout(FAKE, 4096, 0, None) == INVALID
    assert lib.moe_selftest_wait_timeout(MISALIGNED, 4096, 1000, None) == INVALID


def test_shared_expert_host_checks(moe):
    lib = moe.lib()
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536)
    size = ctypes.c_size_t()
    assert lib.moe_workspace_size_shared(ctypes.byref(cfg), 0, ctypes.byref(size)) == INVALID
    assert lib.moe_workspace_size_shared(ctypes.byref(cfg), 200, ctypes.byref(size)) == UNSUPPORTED
    assert lib.moe_workspace_size_shared(ctypes.byref(cfg), 256, ctypes.byref(size)) == OK
    # routed workspace + h_mid_s [T,256] bf16 + y_shared [T,h] fp32
    assert size.value >= moe.workspace_size(cfg) + 128 * 256 * 2 + 128 * 4096 * 4
    f32 = moe.config(T=16, h=136, E=4, k=2, f=200, dtype="f32")
    assert lib.moe_workspace_size_shared(ctypes.byref(f32), 72, ctypes.byref(size)) == OK
    need = moe.workspace_size(cfg)
    # moe_shared_expert: x missing, then a misaligned W2s
    assert lib.moe_shared_expert(ctypes.byref(cfg), 256, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 need, None) == INVALID
    assert lib.moe_shared_expert(ctypes.byref(cfg), 256, FAKE, FAKE, FAKE, MISALIGNED, FAKE, FAKE,
                                 FAKE, need, None) == INVALID
    # moe_forward_shared: the routed workspace size is too small for it
    assert lib.moe_forward_shared(ctypes.byref(cfg), 256, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, need,
                                  None) == WORKSPACE
    # moe_combine_shared: y_shared is optional but must be aligned
    assert lib.moe_combine_shared(ctypes.byref(cfg), FAKE, FAKE, FAKE, MISALIGNED, FAKE,
                                  None) == INVALID


def test_backward_shared_host_checks(moe):
    lib = moe.lib()
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536)
    size, base = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.moe_workspace_size_backward(ctypes.byref(cfg), ctypes.byref(base)) == OK
    assert lib.moe_workspace_size_backward_shared(ctypes.byref(cfg), 0, ctypes.byref(size)) == INVALID
    assert lib.moe_workspace_size_backward_shared(ctypes.byref(cfg), 200,
                                                  ctypes.byref(size)) == UNSUPPORTED
    assert lib.moe_workspace_size_backward_shared(ctypes.byref(cfg), 256, ctypes.byref(size)) == OK
    # the routed backward's workspace + dH_s [T,256] + dA_s [T,512] bf16
    assert size.value >= base.value + 128 * 256 * 2 + 128 * 512 * 2
    need = size.value
    # fp32 runs the backward on the FMA units: fp32 gradient buffers
    f32 = moe.config(T=16, h=136, E=4, k=2, f=200, dtype="f32")
    f32_size, f32_base = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.moe_workspace_size_backward(ctypes.byref(f32), ctypes.byref(f32_base)) == OK
    assert lib.moe_workspace_size_backward_shared(ctypes.byref(f32), 72,
                                                  ctypes.byref(f32_size)) == OK
    assert f32_size.value >= f32_base.value + 16 * 72 * 4 + 16 * 144 * 4
    # moe_backward_shared: W1s missing, then a misaligned dW2s, then the routed-only workspace
    args = [FAKE] * 27
    args[6] = None                                   # W1s
    assert lib.moe_backward_shared(ctypes.byref(cfg), 256, *args, FAKE, need, None) == INVALID
    args = [FAKE] * 27
    args[26] = MISALIGNED                            # dW2s
    assert lib.moe_backward_shared(ctypes.byref(cfg), 256, *args, FAKE, need, None) == INVALID
    args = [FAKE] * 27
    assert lib.moe_backward_shared(ctypes.byref(cfg), 256, *args, FAKE, base.value,
                                   None) == WORKSPACE
    # moe_shared_expert_backward: dx_acc missing; an fp32 call with too small a workspace
    assert lib.moe_shared_expert_backward(ctypes.byref(cfg), 256, FAKE, FAKE, FAKE, FAKE, FAKE,
                                          FAKE, None, FAKE, FAKE, FAKE, FAKE, need,
                                          None) == INVALID
    assert lib.moe_shared_expert_backward(ctypes.byref(f32), 72, FAKE, FAKE, FAKE, FAKE, FAKE,
                                          FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f32_base.value,
                                          None) == WORKSPACE


@pytest.mark.parametrize("E,k,G,gk,want", [
    (256, 8, 8, 4, OK), (256, 8, 1, 0, OK), (256, 8, 0, 5, OK),   # off when num_groups <= 1
    (256, 8, 6, 2, UNSUPPORTED),    # E not a multiple of the groups
    (256, 8, 64, 4, UNSUPPORTED),   # more than 32 groups
    (256, 8, 8, 0, UNSUPPORTED), (256, 8, 8, 9, UNSUPPORTED),  # group_topk out of [1, min(G,k)]
    (16, 4, 4, 1, OK), (16, 6, 4, 1, UNSUPPORTED),  # k above group_topk * E/G
    (8, 2, 4, 4, UNSUPPORTED),      # group_topk above k
])
def test_group_limited_config_validation(moe, E, k, G, gk, want):
    cfg = moe.config(T=64, h=4096, E=E, k=k, f=1536, score="sigmoid", num_groups=G, group_topk=gk)
    size = ctypes.c_size_t()
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == want


def test_config_struct_matches_header(moe):
    # field order and size of moe_config in include/moe.h
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct moe_config \{(.*?)\} moe_config;", text, re.S).group(1)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in moe.MoeConfig._fields_]
    assert ctypes.sizeof(moe.MoeConfig) == 4 * len(fields)


def test_forward_host_host_checks(moe):
    lib = moe.lib()
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536)
    size = ctypes.c_size_t()
    assert lib.moe_workspace_size_host(ctypes.byref(cfg), ctypes.byref(size)) == OK
    need = size.value
    assert need >= moe.workspace_size(cfg) + 4 * 128 * 4096 * 2
    row = 128 * 4096 * 2
    call = lambda nb, x, xs, y, ys, ws_bytes: lib.moe_forward_host(
        ctypes.byref(cfg), nb, x, xs, y, ys, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, ws_bytes,
        None)
    assert call(-1, FAKE, 0, FAKE, 0, need) == INVALID
    assert call(2, None, 0, FAKE, 0, need) == INVALID           # no input buffer
    assert call(2, FAKE, 0, FAKE, row - 2, need) == INVALID     # output batches overlap
    assert call(2, FAKE, row, FAKE, row, need - 1) == WORKSPACE  # routed ws is not enough
    assert call(0, FAKE, 0, FAKE, 0, need) == OK                 # nothing to do, nothing enqueued


def _declared_arg_counts():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(moe_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_header(moe):
    counts = _declared_arg_counts()
    lib = moe.lib()
    for name in moe.EXPORTS:
        assert len(getattr(lib, name).argtypes) == counts[name], name


def test_pad_to_capacity_configuration(moe):
    size = ctypes.c_size_t()
    lib = moe.lib()
    # needs a capacity factor, and is 0 or 1
    cfg = moe.config(T=64, h=4096, E=8, k=2, f=1536, pad_to_capacity=True)
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == INVALID
    cfg = moe.config(T=64, h=4096, E=8, k=2, f=1536, capacity_factor=1.0)
    cfg.pad_to_capacity = 2
    assert _status(moe, "moe_workspace_size", _cfgp(cfg), ctypes.byref(size)) == INVALID
    # the permuted buffers hold E * min(capacity, T) rows when that is more than T*k
    sw = dict(T=32768, h=1024, E=64, k=1, f=4096, score="softmax_pre", capacity_factor=1.25)
    assert moe.max_rows(moe.config(**sw, pad_to_capacity=True)) == 64 * 640
    assert moe.max_rows(moe.config(**sw)) == 32768
    assert moe.workspace_size(moe.config(**sw, pad_to_capacity=True)) > \
        moe.workspace_size(moe.config(**sw))
    assert moe.max_rows(moe.config(T=100, h=256, E=8, k=2, f=128, capacity_factor=20.0,
                                   pad_to_capacity=True)) == 8 * 100
    assert moe.max_rows(moe.config(T=1000, h=256, E=8, k=2, f=128, capacity_factor=0.5,
                                   pad_to_capacity=True)) == 2000
    # the E4M3 and backward buffers hold the padded rows
    cfg = moe.config(T=128, h=4096, E=8, k=2, f=1536, capacity_factor=1.0, pad_to_capacity=True)
    assert _status(moe, "moe_workspace_size_e4m3", _cfgp(cfg), ctypes.byref(size)) == OK
    e4m3_need = size.value
    # the E4M3 pair permutation refuses padding; its map permutation needs it
    assert lib.moe_permute_e4m3(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                FAKE, e4m3_need, None) == INVALID
    plain = moe.config(T=128, h=4096, E=8, k=2, f=1536, capacity_factor=1.0)
    assert lib.moe_permute_map_e4m3(ctypes.byref(plain), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    FAKE, FAKE, FAKE, e4m3_need, None) == INVALID
    assert _status(moe, "moe_workspace_size_backward", _cfgp(cfg), ctypes.byref(size)) == OK
    padded = size.value
    cfg.pad_to_capacity = 0
    assert _status(moe, "moe_workspace_size_backward", _cfgp(cfg), ctypes.byref(size)) == OK
    assert padded >= size.value
    cfg.pad_to_capacity = 1
    need = moe.workspace_size(cfg)
    # the pair permutation cannot place padding rows; the route must return the map
    assert lib.moe_permute(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need,
                           None) == INVALID
    assert lib.moe_permute_noalloc(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   None) == INVALID
    assert lib.moe_route(*_route_args(cfg, need, rm=None)) == INVALID
    # moe_permute_map checks its map and buffers like the other stages
    assert lib.moe_permute_map(ctypes.byref(cfg), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               need, None) == INVALID
    assert lib.moe_permute_map(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, MISALIGNED, FAKE,
                               FAKE, FAKE, need, None) == INVALID
    assert lib.moe_permute_map(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               need - 1, None) == WORKSPACE
