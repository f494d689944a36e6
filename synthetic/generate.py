"""Seeded tensor generation for the MoE workloads.

Every tensor comes from its own torch.Generator sub-stream, keyed by the
workload seed, a tensor id and (for expert weights) the expert index, so
that one expert's weights can be regenerated alone and a margin-failing x
row can be redrawn without touching anything else.  Values are drawn in
fp32 and rounded once to the workload dtype (bf16 rounding is
round-to-nearest-even by torch).
"""

import math
from functools import lru_cache

import numpy as np
import torch

from .workloads import Workload

# tensor ids of the sub-streams
_ID_X = 1
_ID_WG = 2
_ID_W1 = 3
_ID_W3 = 4
_ID_W2 = 5
_ID_EXPERT_BIAS = 6
_ID_EXPERT_RANK = 7
_ID_W1S = 8
_ID_W3S = 9
_ID_W2S = 10
_ID_X_REDRAW = 1000


def _mix(*parts: int) -> int:
    """splitmix64 finaliser over the parts: a well-spread 63-bit seed."""
    z = 0x9E3779B97F4A7C15
    for p in parts:
        z = (z + (p & 0xFFFFFFFFFFFFFFFF) + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        z = z ^ (z >> 31)
    return z & 0x7FFFFFFFFFFFFFFF


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*parts))
    return g


def _torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _normal(shape, std, gen, device, dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def logit_std(w: Workload) -> float:
    """Standard deviation of one gate logit x.Wg[:,e] for x, Wg i.i.d. normal."""
    return math.sqrt(w.h) * w.x_std * w.gate_std


def expert_weights(w: Workload, which: str, e: int, device="cpu", seed=None):
    """W1[e] or W3[e] ([h,f]) or W2[e] ([f,h]) in the workload dtype; with
    which = W1s / W3s ([h,shared_f]) or W2s ([shared_f,h]) the shared expert's."""
    seed = w.seed if seed is None else seed
    tid = {"W1": _ID_W1, "W3": _ID_W3, "W2": _ID_W2,
           "W1s": _ID_W1S, "W3s": _ID_W3S, "W2s": _ID_W2S}[which]
    f = w.shared_f if which.endswith("s") else w.f
    shape = (w.h, f) if which[:2] in ("W1", "W3") else (f, w.h)
    return _normal(shape, w.w_std, _gen(device, seed, tid, e), device, _torch_dtype(w))


def redraw_x_rows(w: Workload, rnd: int, n: int, device="cpu", seed=None):
    """n fresh x rows from the redraw sub-stream of round `rnd`."""
    seed = w.seed if seed is None else seed
    return _normal((n, w.h), w.x_std, _gen(device, seed, _ID_X_REDRAW + rnd), device,
                   _torch_dtype(w))


def generate(w: Workload, device="cpu", seed=None, with_experts=True):
    """All inputs of one MoE layer forward, as torch tensors on `device`.

    Returns a dict with x [T,h], Wg [h,E] fp32, gate_bias [E] fp32 or None,
    expert_bias [E] fp32 or None and, if `with_experts`, W1/W3 [E,h,f] and
    W2 [E,f,h] in the workload dtype (plus W1s/W3s [h,shared_f] and W2s
    [shared_f,h] when the workload has a shared expert).
    """
    seed = w.seed if seed is None else seed
    dt = _torch_dtype(w)
    out = {
        "x": _normal((w.T, w.h), w.x_std, _gen(device, seed, _ID_X), device, dt),
        "Wg": _normal((w.h, w.E), w.gate_std, _gen(device, seed, _ID_WG), device,
                      torch.float32),
        "gate_bias": None,
        "expert_bias": None,
    }
    gb = calibrate_gate_bias(w)
    if gb is not None:
        out["gate_bias"] = torch.from_numpy(gb).to(device)
    if w.expert_bias is not None:
        kind, a = w.expert_bias.split(":")
        assert kind == "uniform"
        a = float(a)
        u = torch.rand((w.E,), generator=_gen(device, seed, _ID_EXPERT_BIAS), device=device,
                       dtype=torch.float32)
        out["expert_bias"] = (u * (2 * a) - a).contiguous()
    if with_experts:
        for name, shape in (("W1", (w.E, w.h, w.f)), ("W3", (w.E, w.h, w.f)),
                            ("W2", (w.E, w.f, w.h))):
            t = torch.empty(shape, dtype=dt, device=device)
            for e in range(w.E):
                t[e] = expert_weights(w, name, e, device=device, seed=seed)
            out[name] = t
        if w.shared_f > 0:
            for name in ("W1s", "W3s", "W2s"):
                out[name] = expert_weights(w, name, 0, device=device, seed=seed)
    return out


# --------------------------------------------------------------------------
# gate-bias calibration (a probability computation on i.i.d. Gaussian logits)
# --------------------------------------------------------------------------

def _expert_ranks(w: Workload) -> np.ndarray:
    """rank[e] in 0..E-1: a seeded permutation deciding which expert is hot."""
    g = torch.Generator().manual_seed(_mix(w.seed, _ID_EXPERT_RANK))
    perm = torch.randperm(w.E, generator=g).numpy()
    rank = np.empty(w.E, dtype=np.int64)
    rank[perm] = np.arange(w.E)
    return rank


def target_probabilities(w: Workload):
    """Per-expert probability that a token selects the expert (sums to k).

    zipf:s  - p(rank r) = min(0.995, c * r^-s), c water-filled so that the
              p sum to k (an expert can take a token at most once, so the
              head of a raw Zipf law is clipped).
    hot:n:m - n experts at m times the mean k/E, the others share the rest.
    """
    if w.gate_bias is None:
        return None
    kind, *args = w.gate_bias.split(":")
    E, k = w.E, w.k
    rank = _expert_ranks(w)
    if kind == "zipf":
        s = float(args[0])
        base = (np.arange(E) + 1.0) ** (-s)
        lo, hi = 0.0, 1e6
        for _ in range(200):
            c = 0.5 * (lo + hi)
            if np.minimum(0.995, c * base).sum() > k:
                hi = c
            else:
                lo = c
        by_rank = np.minimum(0.995, lo * base)
        by_rank *= k / by_rank.sum()
        return by_rank[rank]
    if kind == "hot":
        n, mult = int(args[0]), float(args[1])
        hot_p = mult * k / E
        cold_p = (k - n * hot_p) / (E - n)
        return np.where(rank < n, hot_p, cold_p)
    raise ValueError(w.gate_bias)


def _selection_probabilities(b: np.ndarray, sigma: float, k: int) -> np.ndarray:
    """P(expert e is among the k largest of l_j + b_j), l_j ~ iid N(0, sigma^2).

    For a given value z of expert e's standardised logit, the others exceed
    it independently with probabilities q_j = Phi((b_j - b_e)/sigma - z); the
    count of those is Poisson-binomial and e is selected iff fewer than k
    exceed.  The outer expectation over z is a trapezoid sum on [-9, 9].
    """
    from scipy.special import ndtr
    E = b.shape[0]
    z = np.arange(-9.0, 9.0 + 1e-9, 0.05)
    wz = np.exp(-0.5 * z * z) / math.sqrt(2 * math.pi) * 0.05
    d = (b[None, :] - b[:, None]) / sigma            # d[e, j]
    state = np.zeros((z.size, E, k))
    state[:, :, 0] = 1.0
    for j in range(E):
        q = ndtr(d[:, j][None, :] - z[:, None])       # [Q, E]
        q[:, j] = 0.0                                 # an expert does not compete with itself
        q = q[:, :, None]
        shifted = np.concatenate([np.zeros_like(state[:, :, :1]), state[:, :, :-1]], axis=2)
        state = state * (1.0 - q) + shifted * q
    return (state.sum(axis=2) * wz[:, None]).sum(axis=0)


@lru_cache(maxsize=None)
def _calibrate_cached(w: Workload):
    from scipy.special import ndtri
    target = target_probabilities(w)
    sigma = logit_std(w)
    b = np.zeros(w.E)
    t = np.clip(target, 1e-9, 1 - 1e-9)
    for _ in range(80):
        p = np.clip(_selection_probabilities(b, sigma, w.k), 1e-12, 1 - 1e-12)
        if np.max(np.abs(p - target)) < 2e-5:
            break
        b += 0.8 * sigma * (ndtri(t) - ndtri(p))
        b -= b.mean()
    return b.astype(np.float32)


def calibrate_gate_bias(w: Workload):
    """Gate-logit bias [E] (fp32) giving the workload's target expert loads.

    None when the workload has no gate bias.  The bias is a property of the
    distribution (logit std sqrt(h)*x_std*gate_std), not of the drawn
    tensors, so the loads reached by one draw scatter around the target.
    """
    if w.gate_bias is None:
        return None
    return _calibrate_cached(w).copy()
