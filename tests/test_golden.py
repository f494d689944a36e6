"""The oracle against hand-derived values (tests/golden/*.json, each citing the
page and section it follows).  CPU only."""

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _num(v):
    if isinstance(v, str):
        sign = -1.0 if v.startswith("-") else 1.0
        return sign * math.log(float(v.lstrip("-")[2:]))
    return float(v)


def _logits_via_one_hot(logit_rows):
    """Router inputs whose exact logits are the given rows: x = one-hot rows,
    Wg row i = the i-th wanted logit vector (x.Wg picks row i)."""
    L = np.array([[_num(v) for v in row] for row in logit_rows], dtype=np.float32)
    T, E = L.shape
    x = np.eye(T, dtype=np.float32)
    return x, L  # h = T, Wg = L [h,E]


@pytest.mark.parametrize("case", _load("router_cases.json")["cases"], ids=lambda c: c["name"])
def test_router_golden(case):
    x, Wg = _logits_via_one_hot(case["logits"])
    eb = None if case["expert_bias"] is None else np.array(case["expert_bias"], np.float32)
    r = oracle.route(x, Wg, case["k"], case["score"], expert_bias=eb)
    np.testing.assert_array_equal(r["topk_idx"], np.array(case["topk_idx"]))
    np.testing.assert_allclose(r["topk_prob"], np.array(case["topk_prob"]), rtol=2e-7, atol=1e-7)


@pytest.mark.parametrize("case", _load("capacity_cases.json")["capacity"],
                         ids=lambda c: "T%d_E%d_k%d_cf%g" % (c["T"], c["E"], c["k"], c["cf"]))
def test_capacity_golden(case):
    assert oracle.capacity(case["T"], case["E"], case["k"], case["cf"],
                           case["min_capacity"]) == case["capacity"]


def test_capacity_dropless():
    assert oracle.capacity(100, 4, 2, 0.0) == -1


@pytest.mark.parametrize("case", _load("capacity_cases.json")["drop"], ids=lambda c: c["name"])
def test_drop_golden(case):
    prob, keep, kept = oracle.capacity_drop(np.array(case["topk_idx"], np.int32),
                                            np.array(case["topk_prob"], np.float32),
                                            case["E"], case["capacity"], case["policy"])
    np.testing.assert_array_equal(keep, np.array(case["keep"]))
    np.testing.assert_array_equal(prob, np.array(case["topk_prob_out"], np.float32))
    np.testing.assert_array_equal(kept, np.array(case["kept_per_expert"]))


@pytest.mark.parametrize("case", _load("permute_cases.json")["cases"], ids=lambda c: c["name"])
def test_permute_golden(case):
    offsets, row_map, row_token = oracle.permute(np.array(case["topk_idx"], np.int32),
                                                 np.array(case["keep"], np.uint8), case["E"])
    np.testing.assert_array_equal(offsets, case["offsets"])
    np.testing.assert_array_equal(row_map, case["row_map"])
    np.testing.assert_array_equal(row_token, case["row_token"])
