"""Router variants against the oracle on the GPU: the sqrtsoftplus score
and group-limited top-k (alone and together, with every score function and
with capacity drops), and every score function on the fused small-E router
(E <= 8).  Routing and the permutation are bit-exact, outputs within the
tolerances of the other parity tests."""

import pytest
import torch

import synthetic
from moe_cases import compare_all, gpu_forward, gpu_stages, make_case, oracle_forward, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    "sqrtsoftplus_bias": synthetic.scaled("dsv3", T=500, h=512, f=256, E=64,
                                          score="sqrtsoftplus", seed=91),
    "sqrtsoftplus_no_bias": synthetic.scaled("mixtral", T=400, h=256, f=128, E=16, k=4,
                                             score="sqrtsoftplus", seed=92),
    # DeepSeek-V3's routing on a smaller expert set: 8 groups of 8, 4 kept, top-2 sums
    "grouped_sigmoid": synthetic.scaled("dsv3_grouped", T=600, h=512, f=256, E=64, seed=93),
    "grouped_sqrtsoftplus": synthetic.scaled("dsv3_grouped", T=600, h=512, f=256, E=64,
                                             score="sqrtsoftplus", seed=94),
    # skewed loads (gate bias) with 4 groups of 32, 2 kept
    "grouped_softmax_post": synthetic.scaled("qwen3", T=700, h=256, f=128, num_groups=4,
                                             group_topk=2, seed=95),
    # top-1 over 8 groups of 8 with one group kept, plus capacity drops
    "grouped_softmax_pre_drop": synthetic.scaled("switch", T=3000, h=256, f=256, E=64,
                                                 num_groups=8, group_topk=1, seed=96),
    # 32 groups (the largest number) of 8 experts
    "grouped_32_groups": synthetic.scaled("dsv3_grouped", T=300, h=256, f=128, E=256,
                                          num_groups=32, group_topk=8, seed=97),
    # E <= 8 without groups: the fused logits + top-k kernel, every score
    # function, expert counts that leave idle lanes in a token's 8-lane
    # segment, capacity drops, and the largest h whose gate rows it stages
    "small_e_sigmoid_bias": synthetic.scaled("dsv3", T=500, h=512, f=256, E=8, k=4, seed=81),
    "small_e_sqrtsoftplus_bias": synthetic.scaled("dsv3", T=500, h=512, f=256, E=8, k=2,
                                                  score="sqrtsoftplus", seed=82),
    "small_e_softmax_post_E5_k3": synthetic.scaled("mixtral", T=700, h=512, f=128, E=5, k=3,
                                                   seed=83),
    "small_e_softmax_pre_drop_E6": synthetic.scaled("switch", T=2000, h=256, f=256, E=6,
                                                    gate_bias="hot:1:3", seed=84),
    "small_e_max_hidden": synthetic.scaled("mixtral", T=300, h=6144, f=128, seed=85),
    # fp32 activations (4 features per 16-byte vector, h not a multiple of
    # the 128 features a warp covers per step) with several score functions;
    # fewer 4-token groups than SMs
    "small_e_fp32_sigmoid_bias": synthetic.scaled("dsv3", T=400, h=136, f=64, E=8, k=3,
                                                  dtype="f32", seed=86),
    "small_e_fp32_softmax_pre_drop": synthetic.scaled("switch", T=1500, h=200, f=64, E=7,
                                                      dtype="f32", gate_bias="hot:1:3",
                                                      seed=87),
    "small_e_few_tokens": synthetic.scaled("mixtral", T=100, h=4096, f=128, seed=88),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    dinp = to_dev(inp)
    b = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    return w, inp, ref, dinp, b


def test_variant_matches_oracle(case):
    w, inp, ref, dinp, b = case
    compare_all(w, inp, ref, b)
    if w.capacity_factor > 0:
        assert (ref["keep"] == 0).any()


def test_variant_forward_reproduces_stages(case):
    w, inp, ref, dinp, b = case
    y, idx, prob, tpe = gpu_forward(w, dinp)
    assert torch.equal(idx, b.topk_idx)
    assert torch.equal(prob, b.topk_prob)
    assert torch.equal(y, b.y)


def test_groups_chosen_are_within_kept_groups(case):
    w, inp, ref, dinp, b = case
    if w.num_groups <= 1:
        pytest.skip("no groups")
    per = w.E // w.num_groups
    groups = (b.topk_idx.long() // per).cpu()
    for row in groups:
        assert len(set(row.tolist())) <= w.group_topk


def test_one_group_equals_ungrouped():
    w = synthetic.scaled("dsv3", T=400, h=256, f=128, E=32, seed=98)
    inp, _ = make_case(w)
    dinp = to_dev(inp)
    a = gpu_stages(w, dinp)
    b = gpu_stages(synthetic.scaled(w, num_groups=1, group_topk=1), dinp)
    c = gpu_stages(synthetic.scaled(w, num_groups=4, group_topk=4), dinp)  # every group kept
    torch.cuda.synchronize()
    for other in (b, c):
        assert torch.equal(a.topk_idx, other.topk_idx)
        assert torch.equal(a.topk_prob, other.topk_prob)
        assert torch.equal(a.y, other.y)
