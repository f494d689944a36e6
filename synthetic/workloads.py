"""The five MoE-layer workloads and a helper to shrink them for parity tests.

Shapes and value distributions follow the problem statement of the pages on
the single-GPU MoE layer forward (hidden [T,h], gate W [h,E], top-k, capacity
factor, expert weights W1/W3 [E,h,f] and W2 [E,f,h]).  Names:

* ``tiny_fp32``  - T=256, h=128, E=8, top-2 softmax (renormalised), f=256,
  everything fp32, x and all weights ~N(0, 0.02), seed 0.
* ``mixtral``    - Mixtral-8x7B-shaped: T=8192, h=4096, E=8, top-2 softmax,
  f=14336, bf16 activations/weights, fp32 gate.
* ``dsv3``       - DeepSeek-V3-shaped: T=4096, h=7168, E=256, top-8 sigmoid
  scores with a selection-only expert bias ~U(-0.1, 0.1), f=2048.
* ``qwen3``      - Qwen3-235B-shaped: T=16384, h=4096, E=128, top-8 softmax,
  f=1536, expert loads skewed to Zipf(s=1.1) through a gate-logit bias.
* ``switch``     - Switch-style top-1 with capacity factor 1.25: T=32768,
  h=1024, E=64, f=4096, four hot experts at 4x the mean load, so drops occur.
* ``dsv3_grouped`` - ``dsv3`` with DeepSeek-V3's group-limited routing: the 256
  experts form 8 groups of 32 and each token may only choose among the 4
  groups whose two best selection scores sum highest.
* ``dsv3_shared`` - ``dsv3`` plus one shared expert of width 2048 (DeepSeek-V3
  has one shared expert as wide as a routed one) that every token goes
  through, added to the routed output.
"""

from dataclasses import dataclass, replace
from typing import Optional

SCORE_SOFTMAX_POST = "softmax_post"  # top-k on logits, softmax over the k (renormalised)
SCORE_SOFTMAX_PRE = "softmax_pre"    # softmax over all E, then top-k, no renormalisation
SCORE_SIGMOID = "sigmoid"            # sigmoid, choice-only expert bias, renormalised


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    k: int
    f: int
    score: str
    dtype: str                 # "f32" or "bf16": x, W1/W3/W2, h_mid and y
    seed: int
    x_std: float
    w_std: float
    gate_std: float
    capacity_factor: float = 0.0   # <= 0 means dropless
    min_capacity: int = 0
    drop_policy: str = "probs"     # "probs" or "position"
    gate_bias: Optional[str] = None      # None, "zipf:<s>" or "hot:<n>:<mult>"
    expert_bias: Optional[str] = None    # None or "uniform:<a>" (selection only)
    shared_f: int = 0              # > 0: a shared expert of this SwiGLU width
    num_groups: int = 0            # > 1: group-limited top-k over this many expert groups
    group_topk: int = 0            # groups kept per token when num_groups > 1
    pad_to_capacity: bool = False  # every expert padded to its capacity (needs a capacity factor)
    description: str = ""

    @property
    def dropless(self) -> bool:
        return self.capacity_factor <= 0.0


WORKLOADS = {
    "tiny_fp32": Workload(
        name="tiny_fp32", T=256, h=128, E=8, k=2, f=256,
        score=SCORE_SOFTMAX_POST, dtype="f32", seed=0,
        x_std=0.02, w_std=0.02, gate_std=0.02,
        description="tiny fp32 MoE fwd: T=256, h=128, E=8, top-2 softmax "
                    "(renormalised), SwiGLU f=256, dropless; x,W ~N(0,0.02), seed 0"),
    "mixtral": Workload(
        name="mixtral", T=8192, h=4096, E=8, k=2, f=14336,
        score=SCORE_SOFTMAX_POST, dtype="bf16", seed=2,
        x_std=1.0, w_std=0.02, gate_std=0.02,
        description="Mixtral-8x7B-shaped MoE fwd bf16: T=8192, h=4096, E=8, top-2 "
                    "softmax, SwiGLU f=14336, dropless; x~N(0,1), weights ~N(0,0.02), "
                    "gate logits fp32"),
    "dsv3": Workload(
        name="dsv3", T=4096, h=7168, E=256, k=8, f=2048,
        score=SCORE_SIGMOID, dtype="bf16", seed=3,
        x_std=1.0, w_std=0.02, gate_std=0.02, expert_bias="uniform:0.1",
        description="DeepSeek-V3-shaped fine-grained MoE fwd bf16: T=4096, h=7168, "
                    "E=256, top-8 sigmoid + selection bias ~U(-0.1,0.1), renormalised, "
                    "SwiGLU f=2048, dropless"),
    "qwen3": Workload(
        name="qwen3", T=16384, h=4096, E=128, k=8, f=1536,
        score=SCORE_SOFTMAX_POST, dtype="bf16", seed=4,
        x_std=1.0, w_std=0.02, gate_std=0.02, gate_bias="zipf:1.1",
        description="Qwen3-235B-shaped MoE fwd bf16: T=16384, h=4096, E=128, top-8 "
                    "softmax renormalised, SwiGLU f=1536, dropless; expert loads "
                    "follow Zipf(s=1.1)"),
    "switch": Workload(
        name="switch", T=32768, h=1024, E=64, k=1, f=4096,
        score=SCORE_SOFTMAX_PRE, dtype="bf16", seed=5,
        x_std=1.0, w_std=0.02, gate_std=0.02,
        capacity_factor=1.25, gate_bias="hot:4:4",
        description="Switch-style top-1 with capacity drop bf16: T=32768, h=1024, "
                    "E=64, capacity factor 1.25, SwiGLU f=4096, 4 hot experts at 4x "
                    "mean load"),
}
WORKLOADS["dsv3_grouped"] = replace(
    WORKLOADS["dsv3"], name="dsv3_grouped", num_groups=8, group_topk=4,
    description="dsv3 with group-limited routing: 8 expert groups of 32, the 4 best groups "
                "(group score = sum of its top-2 selection scores) kept per token")
WORKLOADS["switch_pad"] = replace(
    WORKLOADS["switch"], name="switch_pad", pad_to_capacity=True,
    description="switch with pad_to_capacity: every expert's input padded to its capacity "
                "(640 rows; 40960 rows in all) with tokens of probability 0")
WORKLOADS["dsv3_shared"] = replace(
    WORKLOADS["dsv3"], name="dsv3_shared", shared_f=2048,
    description="dsv3 plus one shared SwiGLU expert (width 2048) applied to every token and "
                "added to the routed output")


def scaled(name_or_workload, **overrides) -> Workload:
    """A copy of a workload with some fields replaced (e.g. smaller T, h, f).

    The routing structure (score function, k, E, bias recipe, capacity
    factor) is kept unless overridden, so a shrunk case still exercises the
    same path.
    """
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    if "name" not in overrides:
        overrides["name"] = w.name + "_scaled"
    return replace(w, **overrides)

