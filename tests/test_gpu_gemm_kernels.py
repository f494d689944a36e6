"""Both tensor-core grouped GEMM kernels against the oracle on the same
inputs: the one-SM kernel (128-row tiles) and the SM-pair kernel (256-row
tiles, the MMA shared by a 2-CTA cluster), each forced through the
MOE_TC_PAIR override.  The cases put the pair tile's boundaries everywhere
it matters: experts with rows a multiple of 256, with a tail that ends in
the first or the second CTA's half, with fewer rows than one half, and
empty experts; plus the automatic choice on a shape that selects pairs.
In the boundary case, tails of 1, 44, 100 and exactly 128 rows leave the
pair's second CTA without rows; tails of 148 and 255 fill it in part.
"""

import numpy as np
import pytest
import torch

import synthetic
from moe_cases import compare_all, gpu_stages, make_case, oracle_forward, to_dev, to_np

pytestmark = pytest.mark.gpu

CASES = {
    # ~1000 rows per expert: 3 full pair tiles and a tail in the second half
    "mixtral_e4": synthetic.scaled("mixtral", T=2000, h=512, f=384, E=4, seed=71),
    # ~75 rows per expert: the second CTA's rows are all past the expert's end
    "qwen3_sparse": synthetic.scaled("qwen3", T=300, h=256, f=256, seed=72),
    # capacity drop: kept rows per expert capped, several n-tiles in fc2
    "switch_cap": synthetic.scaled("switch", T=3000, h=512, f=256, E=8, seed=73),
    # larger K: several 64-wide K stages per tile and a deep ring wrap-around
    "dsv3_deepk": synthetic.scaled("dsv3", T=700, h=1536, f=512, E=16, k=4, seed=74),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w = CASES[request.param]
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    return w, inp, ref, to_dev(inp)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_grouped_gemm_kernel(case, kernel, monkeypatch):
    w, inp, ref, dinp = case
    monkeypatch.setenv("MOE_TC_PAIR", "1" if kernel == "pair" else "0")
    b = gpu_stages(w, dinp)
    torch.cuda.synchronize()
    compare_all(w, inp, ref, b)


def test_experts_on_pair_boundaries(monkeypatch):
    # rows per expert: 0, 128, 256, 300, 511, 1, 100 and the rest (404)
    w = synthetic.scaled("mixtral", T=1700, h=256, f=128, E=8, k=1, gate_bias=None, seed=75)
    inp, _ = make_case(w)
    counts = [0, 128, 256, 300, 511, 1, 100]
    counts.append(w.T - sum(counts))
    owner = np.repeat(np.arange(w.E), counts)
    rng = np.random.default_rng(75)
    rng.shuffle(owner)
    # steer every token to its expert with a large per-token logit margin:
    # x rows get a strong component along the owner's gate column
    Wg = inp["Wg"].double().numpy()
    x = inp["x"].float().numpy().astype(np.float64)
    col = Wg[:, owner].T / np.linalg.norm(Wg[:, owner].T, axis=1, keepdims=True)
    x = x + 30.0 * col
    xt = torch.from_numpy(x).to(inp["x"].dtype)
    inp["x"] = xt
    from moe_cases import condition_inputs
    condition_inputs(w, inp)
    ref = oracle_forward(w, inp)
    got = np.bincount(ref["topk_idx"][:, 0], minlength=w.E)
    assert (got == 0).any() and (got % 256 != 0).any()
    d = to_dev(inp)
    for kernel in ("0", "1"):
        monkeypatch.setenv("MOE_TC_PAIR", kernel)
        b = gpu_stages(w, d)
        torch.cuda.synchronize()
        compare_all(w, inp, ref, b)


def test_automatic_choice_selects_pairs_and_matches(monkeypatch):
    # 2048 rows per expert on average: the default rule takes the pair kernel
    monkeypatch.delenv("MOE_TC_PAIR", raising=False)
    w = synthetic.scaled("mixtral", T=4096, h=256, f=256, E=4, seed=76)
    inp, _ = make_case(w)
    ref = oracle_forward(w, inp)
    b = gpu_stages(w, to_dev(inp))
    torch.cuda.synchronize()
    compare_all(w, inp, ref, b)
    assert to_np(b.tokens_per_expert).sum() == w.T * w.k
