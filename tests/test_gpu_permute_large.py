"""The permutation above 128 tiles of 2048 token-slot pairs, on the GPU
through the C ABI, against the oracle.

Up to 128 tiles the scan of the per-tile counts and the in-tile ranking run
in one launch; beyond, they run as two launches (a one-CTA scan, then one
CTA per tile ranking).  None of the five workloads reaches that branch (the
largest has 64 tiles), so these cases do: the dispatcher's stable
expert-major permutation of the Megatron Core walkthrough (r00kie-liu.github.io),
section 9 Token dispatcher.  A permutation is index and byte work: bit-exact.

The Switch-shaped case also takes its capacity-drop candidate lists through
the same two-launch branch (the candidate lists are the permutation of all
routed pairs), section 8 Token dropping of the same page.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from moe_cases import assert_equal, assert_probs, gpu_config, make_case, to_dev, to_np

pytestmark = pytest.mark.gpu

PAIRS_PER_TILE = 2048
FUSED_MAX_TILES = 128

CASES = {
    # 320,000 pairs = 157 tiles over 128 experts with Zipf loads
    "qwen3_T40000": synthetic.scaled("qwen3", T=40000, h=256, f=128, seed=41),
    # 280,000 pairs = 137 tiles over 8 experts
    "mixtral_T140000": synthetic.scaled("mixtral", T=140000, h=256, f=128, seed=42),
    # 300,000 pairs = 147 tiles; four hot experts over capacity (5860), so the
    # drop's candidate lists take the two-launch branch too
    "switch_T300000": synthetic.scaled("switch", T=300000, h=256, f=128, seed=43),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def large(request):
    import mixture_experts_layer_fp32_gb300 as moe
    w = CASES[request.param]
    assert -(-w.T * w.k // PAIRS_PER_TILE) > FUSED_MAX_TILES
    inp, r = make_case(w)
    d = to_dev({n: inp[n] for n in ("x", "Wg", "gate_bias", "expert_bias")})
    cfg = gpu_config(w)
    b = moe.Buffers(cfg)
    moe.route(cfg, d["x"], d["Wg"], d["gate_bias"], d["expert_bias"], b.topk_idx, b.topk_prob,
              b.keep, b.tokens_per_expert, None, b.ws)
    moe.permute(cfg, d["x"], b.topk_idx, b.keep, b.x_perm, b.row_map, b.expert_offsets, b.ws)
    moe.check(b.ws)
    torch.cuda.synchronize()
    return w, inp, r, d, b


def test_routing_large(large):
    w, inp, r, d, b = large
    assert_equal("topk_idx", to_np(b.topk_idx), r["topk_idx"])
    assert_equal("keep", to_np(b.keep), r["keep"])
    assert_equal("tokens_per_expert", to_np(b.tokens_per_expert), r["tokens_per_expert"])
    assert_probs(to_np(b.topk_prob), r["topk_prob"])
    if w.capacity_factor > 0:
        assert (r["keep"] == 0).any()


def test_permutation_large(large):
    w, inp, r, d, b = large
    offsets, row_map, row_token = oracle.permute(r["topk_idx"], r["keep"], w.E)
    assert_equal("expert_offsets", to_np(b.expert_offsets), offsets)
    assert_equal("row_map", to_np(b.row_map), row_map)
    R = int(offsets[-1])
    want = d["x"][torch.from_numpy(row_token).long().to(d["x"].device)]
    assert torch.equal(b.x_perm[:R].view(torch.int16), want.view(torch.int16))


def test_permutation_large_repeats(large):
    # the second call reuses the same workspace counters: nothing may carry over
    import mixture_experts_layer_fp32_gb300 as moe
    w, inp, r, d, b = large
    cfg = gpu_config(w)
    row_map = torch.full_like(b.row_map, -7)
    offsets = torch.full_like(b.expert_offsets, -7)
    moe.permute(cfg, d["x"], b.topk_idx, b.keep, b.x_perm, row_map, offsets, b.ws)
    moe.check(b.ws)
    assert torch.equal(row_map, b.row_map)
    assert torch.equal(offsets, b.expert_offsets)
    assert np.all(np.diff(to_np(offsets)) >= 0)
