"""moe_permute_noalloc against moe_permute, on the GPU through the C ABI.

moe_permute_noalloc is for callers that cannot give the library device
memory beyond their inputs and outputs (a memory budget fixed at start-up, a
host framework that forbids allocating outside its pools, a path that must
not call cudaMalloc/cudaFree because they may synchronise the device).  Its
scratch is a fixed array inside the library, shared by all calls.  Two calls
in a row, with different shapes, must each match moe_permute exactly (a
permutation is index and byte work: bit-exact).  This file is collected
last so that a stop at the first failure has already run every other test.
"""

import pytest
import torch

import synthetic
from moe_cases import gpu_config, to_dev

pytestmark = pytest.mark.gpu

# sizes go up and down so that stale counters from the previous call would
# show; the second case has 137 tiles of 2048 pairs (more than 128), so its
# scan and ranking run as two launches on the fixed array
CASES = [synthetic.scaled("qwen3", T=1500, h=256, f=128, seed=31),
         synthetic.scaled("mixtral", T=140000, h=256, f=128, seed=34),
         synthetic.scaled("switch", T=3000, h=256, f=128, seed=32),
         synthetic.scaled("mixtral", T=700, h=256, f=128, seed=33)]


def _routed(w):
    import mixture_experts_layer_fp32_gb300 as moe
    cfg = gpu_config(w)
    d = to_dev(synthetic.generate(w, device="cpu", with_experts=False))
    b = moe.Buffers(cfg)
    moe.route(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], b.topk_idx, b.topk_prob,
              b.keep, b.tokens_per_expert, None, b.ws)
    return cfg, d, b


def test_permute_noalloc_matches_permute_on_consecutive_calls():
    import mixture_experts_layer_fp32_gb300 as moe
    for w in CASES:
        cfg, d, b = _routed(w)
        moe.permute(cfg, d["x"], b.topk_idx, b.keep, b.x_perm, b.row_map, b.expert_offsets, b.ws)
        moe.check(b.ws)
        R = int(b.expert_offsets[-1].item())
        for _ in range(2):
            x_perm = torch.full_like(b.x_perm, float("nan"))
            row_map = torch.full_like(b.row_map, -7)
            offsets = torch.full_like(b.expert_offsets, -7)
            moe.permute_noalloc(cfg, d["x"], b.topk_idx, b.keep, x_perm, row_map, offsets)
            torch.cuda.synchronize()
            assert torch.equal(offsets, b.expert_offsets)
            assert torch.equal(row_map, b.row_map)
            assert torch.equal(x_perm[:R].view(torch.int16), b.x_perm[:R].view(torch.int16))


def test_permute_noalloc_rejects_oversized_config():
    import mixture_experts_layer_fp32_gb300 as moe
    # ceil(T*k/2048) * E counters: 560000 pairs -> 274 tiles x 256 experts > 65536
    cfg = moe.config(T=70000, h=256, E=256, k=8, f=128)
    with pytest.raises(moe.MoeError) as ei:
        moe.permute_noalloc(cfg, None, None, None, None, None, torch.empty(257, dtype=torch.int32,
                                                                          device="cuda"))
    assert ei.value.code == 2  # MOE_ERR_UNSUPPORTED
