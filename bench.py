"""Benchmark of the GB300 MoE layer forward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference] [--no-e2e] [--no-cpu-baseline]

A step is one MoE layer forward -- route, permute, grouped SwiGLU fc1,
fc2, combine -- over one batch of T synthetic tokens already resident in
HBM.  Each stage is bracketed by CUDA events on the stream the kernels are
launched on; the L2 is flushed (a 512 MB write) between timed steps,
outside the events.  `value` is tokens/s over all ranks (weak scaling:
every rank runs its own replica of the workload, there is no exchange).
`e2e` repeats the measurement through moe_forward with the step's input
copied from pinned host memory and the output copied back inside the
timed region.  `cpu_baseline` times the CPU oracle on a bounded sample of
the same workload on the host cores.

--impl reference times the CPU oracle alone on the same workload (a
bounded sample of tokens per step) and prints the same JSON line with
"impl": "reference".
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "MoE fwd tokens/sec"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mixtral"
STAGES = ["route", "permute", "fc1", "fc2", "combine"]
# experts averaging at least this many rows run on the SM-pair GEMM kernel
# (the library's selection rule; MOE_TC_PAIR=0/1 overrides it)
PAIR_MIN_ROWS = 768


def fused_top1(w, fp8=False):
    """Top-1 bf16 layers without padding or a shared expert run fc2 and the
    combine as one call (moe_grouped_fc2_combine: the combine in fc2's
    epilogue)."""
    return (w.k == 1 and w.dtype == "bf16" and not w.pad_to_capacity and w.shared_f == 0
            and not fp8)


def uses_f16s(w, fp8=False):
    """bf16 layers with k >= 2 (no padding, no shared expert) and every E4M3
    layer keep y_perm as fp16 with a power-of-two scale per 32 columns
    (moe_grouped_fc2_f16s or moe_grouped_fc2_e4m3_f16s, then moe_combine_f16s),
    as moe_forward and moe_forward_e4m3 do."""
    if fp8:
        return True
    if w.dtype != "bf16" or w.pad_to_capacity:
        return False
    return w.k > 1 or w.shared_f > 0  # top-1 without a shared expert: fc2+combine fused


def router_on_tc(w):
    """The opt-in tensor-core router (MOE_ROUTER_TC=1 in the environment, off
    by default: the layer keeps the tensor cores to the expert GEMMs): bf16
    layers with more experts than the fused small-E router, E % 4 == 0, the
    gate weights split into three bf16 pieces (the library's rule)."""
    fused = w.E <= 8 and w.k <= w.E and w.num_groups <= 1 and w.h <= 6144
    return (w.dtype == "bf16" and w.E % 4 == 0 and not fused
            and os.environ.get("MOE_ROUTER_TC", "")[:1] == "1")


def router_ksplit(w):
    """K splits of the tensor-core router GEMM: fp32 accumulation chains of at
    most 1024 products, at most 5 splits (the library's rule)."""
    force = os.environ.get("MOE_ROUTER_KSPLIT", "")
    S = int(force[0]) if force[:1].isdigit() and force[0] != "0" else -(-w.h // 1024)
    return max(1, min(S, 5, w.h // 64))


def stages_of(w, fp8=False):
    """Timed stages of one forward (the shared expert between fc2 and combine)."""
    if fused_top1(w, fp8):
        return STAGES[:3] + ["fc2+combine"]
    return STAGES[:4] + (["shared"] if w.shared_f > 0 else []) + STAGES[4:]


def gemm_kernel_name(w, rows, stage):
    force = os.environ.get("MOE_TC_PAIR", "")
    pair = rows >= (1 if stage == "shared" else w.E) * PAIR_MIN_ROWS
    if force[:1] in ("0", "1"):
        pair = force[:1] == "1"
    base = "tc_grouped_pair_kernel" if pair else "tc_grouped_kernel"
    return "%s<%s>" % (base, "FC1" if stage in ("fc1", "shared") else "FC2")
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay of the step (an extra measurement)")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "e4m3"],
                    help="expert GEMM operands: bf16 (the default workload) or E4M3 (FP8 "
                         "experts, weights quantised once outside the timed region)")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward"],
                    help="time the layer forward (the default) or its backward (after one "
                         "staged forward; dy seeded)")
    ap.add_argument("--override", default="",
                    help="comma list of workload fields to replace, e.g. T=2048,f=3584 "
                         "(a shrunk case for profiling captures)")
    return ap.parse_args()


def workload_of(args):
    w = synthetic.WORKLOADS[args.workload]
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        typed = {k: type(getattr(w, k))(v) for k, v in kv.items()}
        w = synthetic.scaled(w, name=w.name + "_" + args.override.replace(",", "_"), **typed)
    return w


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def workload_desc(w):
    return {"workload": w.description, "name": w.name, "T": w.T, "h": w.h, "E": w.E, "k": w.k,
            "f": w.f, "score": w.score, "capacity_factor": w.capacity_factor,
            "shared_f": w.shared_f, "num_groups": w.num_groups, "group_topk": w.group_topk,
            "l2": "flushed between timed steps (512 MB write outside the events)"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        if not enabled:
            return
        fd, self.path = tempfile.mkstemp(prefix="moe_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: power above the midpoint of the observed range
        thr = 0.5 * (min(power) + max(power))
        loaded = [s for s, p in zip(sm, power) if p >= thr] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


# ---------------------------------------------------------------- traffic

def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source has not changed since it was captured (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    ent = d.get(kernel, {}).get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, "mixture_experts_layer_fp32_gb300", "csrc", ent["source"])
    with open(src, "rb") as fh:
        if hashlib.sha256(fh.read()).hexdigest() != ent["sha256"]:
            return None
    return ent["dram_bytes_per_launch"]


# ---------------------------------------------------------------- native arm

def kernels_per_forward(w, cfg, fp8=False):
    import mixture_experts_layer_fp32_gb300 as moe
    cap = moe.capacity(cfg)
    drops = 0 <= cap < w.T
    # logits and top-k (one fused kernel when E <= 8 without groups and h <= 6144,
    # the library's rule); the permutation index is hist + scan/rank (one
    # kernel up to 128 tiles of 2048 pairs, else scan and rank), run again for
    # the drop candidates before the select kernel
    fused = w.E <= 8 and w.k <= w.E and w.num_groups <= 1 and w.h <= 6144
    index = 2 if -(-w.T * w.k // 2048) <= 128 else 3
    # the tensor-core router: split of the gate weights, logits GEMM, top-k
    logits = 1 if fused else 3 if router_on_tc(w) else 2
    route = logits + (index + 1 if drops else 0) + (1 if w.pad_to_capacity else 0)
    if w.pad_to_capacity:  # permutation by the padded map: hist, scan, rank, gather
        # E4M3: x quantised per token first, the scales gathered, the SwiGLU rows quantised
        return route + 4 + 1 + 1 + (2 if w.shared_f > 0 else 0) + (3 if fp8 else 0) + 1
    shared = 2 if w.shared_f > 0 else 0  # the shared expert's fc1 and fc2
    quant = 1 if fp8 else 0           # E4M3: the SwiGLU rows before fc2 (x is quantised by the copy)
    return route + index + 1 + 1 + 1 + shared + quant + 1  # permute index + copy, fc1, fc2, combine


def stage_work(w, R, fp8=False, active=None, y16=False, kept=None):
    """Algorithmic work of each stage (bytes moved or flops), per forward.
    fp8: E4M3 expert operands (1-byte codes of x_perm, the weights and the
    SwiGLU output; fc2 also reads the bf16 SwiGLU output once to quantise it).
    active: experts with at least one row (only their weights are read;
    default all E)."""
    b = 4 if w.dtype == "f32" else 2
    q = 1 if fp8 else b          # bytes of a GEMM operand element
    T, h, E, k, f = w.T, w.h, w.E, w.k, w.f
    A = E if active is None else active
    yb = 2 + 1 / 32 if y16 else 4  # bytes of a y_perm value: fp16 + exponent byte, or fp32
    K = R if kept is None else kept  # rows the combine reads (padding rows have no slot)
    return {
        "route": {"bytes": T * h * b + h * E * 4 + T * k * (4 + 4 + 1),
                  "flops": 2 * T * h * E},
        "permute": {"bytes": T * h * b + R * h * q + T * k * (4 + 1 + 4)},
        "fc1": {"flops": 4 * R * h * f, "bytes": 2 * A * h * f * q + R * h * q + R * f * b},
        "fc2": {"flops": 2 * R * f * h,
                "bytes": A * f * h * q + R * f * b + (2 * R * f if fp8 else 0) + R * h * yb,
                "bytes_algorithmic": A * f * h * q + R * f * b + (2 * R * f if fp8 else 0)
                + R * h * b},
        "combine": {"bytes": K * h * yb + T * h * b + T * k * 8 + (T * h * 4 if w.shared_f else 0),
                    # the scope's algorithmic bytes: y_perm in the activation dtype
                    "bytes_algorithmic": K * h * b + T * h * b},
        # top-1: fc2 writes each row, weighted, straight into the token's output
        # row (no y_perm); dropped tokens' rows are zeroed
        "fc2+combine": {"flops": 2 * R * f * h,
                        "bytes": A * f * h * q + R * f * b + T * h * b + T * k * 8,
                        "bytes_algorithmic": A * f * h * q + R * f * b + T * h * b},
        "shared": {"flops": 6 * T * h * w.shared_f,
                   "bytes": 3 * h * w.shared_f * b + T * h * b + 2 * T * w.shared_f * b + T * h * 4},
    }


def run_native(args, rank, world, local):
    import mixture_experts_layer_fp32_gb300 as moe

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload_of(args)
    inp = synthetic.generate(w, device=dev, seed=w.seed + 1000 * rank)
    cfg = moe.config(w.T, w.h, w.E, w.k, w.f, w.score, w.dtype, w.capacity_factor,
                     w.min_capacity, w.drop_policy, w.num_groups, w.group_topk,
                     w.pad_to_capacity)
    b = moe.Buffers(cfg, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fp8 = args.precision == "e4m3"
    stage_names = stages_of(w, fp8)
    # the backward reads the forward's fp32 y_perm: its staged forward keeps it
    f16s = uses_f16s(w, fp8) and args.which == "forward"
    if f16s:  # y_perm as fp16 + one exponent byte per 32 columns
        y16 = torch.empty((b.y_perm.shape[0], w.h), dtype=torch.float16, device=dev)
        y16_exp = torch.empty((b.y_perm.shape[0], w.h // 32), dtype=torch.int8, device=dev)
    if w.shared_f > 0:
        h_mid_s = torch.empty((w.T, w.shared_f), dtype=moe.act_dtype(cfg), device=dev)
        y_shared = torch.empty((w.T, w.h), dtype=torch.float32, device=dev)

    if fp8:
        if w.dtype != "bf16" or w.shared_f > 0:
            raise SystemExit("--precision e4m3 needs a bf16 workload without a shared expert")
        q = moe.E4m3Experts(cfg, inp["W1"], inp["W3"], inp["W2"])  # once, outside the timing
        b.ws = moe.alloc_workspace_e4m3(cfg, dev)
        Rmax = moe.max_rows(cfg)
        xq = torch.empty((Rmax, w.h), dtype=torch.uint8, device=dev)
        xs = torch.empty((Rmax,), dtype=torch.float32, device=dev)
        hq = torch.empty((Rmax, w.f), dtype=torch.uint8, device=dev)
        hs = torch.empty((Rmax,), dtype=torch.float32, device=dev)

    def step(ev=None):
        if ev: ev[0].record(stream)
        moe.route(cfg, inp["x"], inp["Wg"], inp["gate_bias"], inp["expert_bias"], b.topk_idx,
                  b.topk_prob, b.keep, b.tokens_per_expert,
                  b.routing_map if w.pad_to_capacity else None, b.ws)
        if ev: ev[1].record(stream)
        if fp8:
            if w.pad_to_capacity:
                moe.permute_map_e4m3(cfg, inp["x"], b.routing_map, b.topk_idx, b.keep, xq, xs,
                                     b.row_map, b.expert_offsets, b.ws)
            else:
                moe.permute_e4m3(cfg, inp["x"], b.topk_idx, b.keep, xq, xs, b.row_map,
                                 b.expert_offsets, b.ws)
            if ev: ev[2].record(stream)
            moe.grouped_fc1_e4m3(cfg, xq, xs, b.expert_offsets, q, b.h_mid, b.ws)
            if ev: ev[3].record(stream)
            moe.grouped_fc2_e4m3_f16s(cfg, b.h_mid, b.expert_offsets, q, hq, hs, y16, y16_exp,
                                      b.ws)
        else:
            if w.pad_to_capacity:  # the padded routing map drives the permutation
                moe.permute_map(cfg, inp["x"], b.routing_map, b.topk_idx, b.keep, b.x_perm,
                                b.row_map, b.expert_offsets, b.ws)
            else:
                moe.permute(cfg, inp["x"], b.topk_idx, b.keep, b.x_perm, b.row_map,
                            b.expert_offsets, b.ws)
            if ev: ev[2].record(stream)
            moe.grouped_fc1(cfg, b.x_perm, b.expert_offsets, inp["W1"], inp["W3"], b.h_mid,
                            b.ws)
            if ev: ev[3].record(stream)
            if fused_top1(w):
                moe.grouped_fc2_combine(cfg, b.h_mid, b.expert_offsets, inp["W2"], b.row_map,
                                        b.topk_prob, b.y, b.ws)
                if ev: ev[4].record(stream)
                return
            if f16s:
                moe.grouped_fc2_f16s(cfg, b.h_mid, b.expert_offsets, inp["W2"], y16, y16_exp, b.ws)
            else:
                moe.grouped_fc2(cfg, b.h_mid, b.expert_offsets, inp["W2"], b.y_perm, b.ws)
        if ev: ev[4].record(stream)
        if w.shared_f > 0:
            moe.shared_expert(cfg, w.shared_f, inp["x"], inp["W1s"], inp["W3s"], inp["W2s"],
                              h_mid_s, y_shared, b.ws)
            if ev: ev[5].record(stream)
            if f16s:
                moe.combine_f16s(cfg, y16, y16_exp, b.row_map, b.topk_prob, b.y,
                                 y_shared=y_shared)
            else:
                moe.combine_shared(cfg, b.y_perm, b.row_map, b.topk_prob, y_shared, b.y)
        elif f16s:
            moe.combine_f16s(cfg, y16, y16_exp, b.row_map, b.topk_prob, b.y)
        else:
            moe.combine(cfg, b.y_perm, b.row_map, b.topk_prob, b.y)
        if ev: ev[-1].record(stream)

    fma_tflops = fp32_fma_rate(moe, dev, stream)
    for _ in range(args.warmup):
        step()
    moe.check(b.ws)
    R = int(b.expert_offsets[-1].item())
    tpe = b.tokens_per_expert.cpu().numpy()
    if args.which == "backward":
        if w.shared_f > 0:
            b.h_mid_s = h_mid_s  # saved by the shared expert's forward
        return run_backward(args, moe, w, cfg, inp, b, R, flush, stream, world, rank, local)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
              for _ in range(args.steps)]
    clocks = ClockSampler(local, enabled=not args.no_clocks and rank == 0)
    if clocks.proc is not None:
        time.sleep(0.5)  # let the sampler start before the timed region
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(events[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()
    moe.check(b.ws)

    stage_ms = {s: [events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps)]
                for j, s in enumerate(stage_names)}
    step_ms = [events[i][0].elapsed_time(events[i][-1]) for i in range(args.steps)]
    ms = sum(step_ms) / len(step_ms)
    ms_all, tokens_per_s = job_throughput(ms, w.T, world)

    # ---- e2e: through the C ABI with host (pinned) input and output, copies
    # inside the timed region
    e2e = None
    if not args.no_e2e:
        x_host = inp["x"].cpu().pin_memory()
        y_host = torch.empty(b.y.shape, dtype=b.y.dtype).pin_memory()
        if fp8:
            ws2 = moe.alloc_workspace_host_e4m3(cfg, dev)

            def run(n):
                moe.forward_host_e4m3(cfg, x_host, y_host, inp["Wg"], inp["gate_bias"],
                                      inp["expert_bias"], q, ws2, num_batches=n)
            api = ("moe_forward_host_e4m3 (C ABI): %d batches from a pinned host buffer, each "
                   "batch's H2D input and D2H output copy inside the timed region, pipelined on "
                   "the library's copy streams" % args.steps)
        elif w.shared_f > 0:
            ws2 = moe.alloc_workspace_host_shared(cfg, w.shared_f, dev)

            def run(n):
                moe.forward_host_shared(cfg, w.shared_f, x_host, y_host, inp["Wg"],
                                        inp["gate_bias"], inp["expert_bias"], inp["W1"],
                                        inp["W3"], inp["W2"], inp["W1s"], inp["W3s"], inp["W2s"],
                                        ws2, num_batches=n)
            api = ("moe_forward_host_shared (C ABI): %d batches from a pinned host buffer, each "
                   "batch's H2D input and D2H output copy inside the timed region, pipelined on "
                   "the library's copy streams" % args.steps)
        else:
            # moe_forward_host: every step's input copied from the pinned host buffer and its
            # output copied back (stride 0: one buffer reused), the copies of neighbouring
            # steps overlapping the compute of the current one
            ws2 = moe.alloc_workspace_host(cfg, dev)

            def run(n):
                moe.forward_host(cfg, x_host, y_host, inp["Wg"], inp["gate_bias"],
                                 inp["expert_bias"], inp["W1"], inp["W3"], inp["W2"], ws2,
                                 num_batches=n)
            api = ("moe_forward_host (C ABI): %d batches from a pinned host buffer, each batch's "
                   "H2D input and D2H output copy inside the timed region, pipelined on the "
                   "library's copy streams" % args.steps)

        run(max(1, args.warmup))
        torch.cuda.synchronize()
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        a.record(stream)
        run(args.steps)
        c.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        moe.check(ws2)
        e2e_ms = max_over_ranks(a.elapsed_time(c) / args.steps, world)
        e2e = {"value": world * w.T / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
               "d2h_bytes_per_step": y_host.numel() * y_host.element_size(),
               "api": api,
               "l2": "not flushed between e2e steps; the expert weights read every step "
                     "(%.0f MB) %s the 129 MB L2" % (
                         3 * w.E * w.h * w.f * (4 if w.dtype == "f32" else 2) / 1e6,
                         "exceed" if 3 * w.E * w.h * w.f * (4 if w.dtype == "f32" else 2)
                         > 129e6 else "fit in")}

    # ---- the same step captured once into a CUDA graph and replayed: the same
    # kernels on the same buffers, without the launch gaps between them (the
    # L2 flush stays outside the graph, between replays)
    graph = None
    if not args.no_graph:
        step()
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            step()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            gev[i][0].record(stream)
            cg.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        moe.check(b.ws)
        g_ms = max_over_ranks(sum(a.elapsed_time(c) for a, c in gev) / args.steps, world)
        graph = {"value": world * w.T / (g_ms / 1e3), "unit": UNIT, "ms_per_step": g_ms,
                 "api": "the timed step's C-ABI calls captured once into a CUDA graph, "
                        "replayed per step (L2 flushed between replays)"}
        del cg

    if rank != 0:
        return None

    peaks = measured_peaks()
    kept = int(b.keep.sum().item())
    work = stage_work(w, R, fp8, active=int(np.count_nonzero(tpe)), y16=f16s, kept=kept)
    stages = {}
    for s in stage_names:
        t = sum(stage_ms[s]) / len(stage_ms[s])
        ent = {"ms": t, "share": t / ms}
        if "flops" in work[s]:
            ent["tflops"] = work[s]["flops"] / (t * 1e-3) / 1e12
        if "bytes" in work[s]:
            ent["gbs"] = work[s]["bytes"] / (t * 1e-3) / 1e9
            if s in ("route", "permute", "combine"):
                ent["hbm_frac"] = ent["gbs"] / peaks["hbm_gbs"]
        if "bytes_algorithmic" in work[s]:
            # y_perm counted in the activation dtype (2 bytes for bf16) although
            # the library stores it in fp32: the fraction of HBM on those bytes
            ent["gbs_algorithmic"] = work[s]["bytes_algorithmic"] / (t * 1e-3) / 1e9
            ent["frac_algorithmic"] = ent["gbs_algorithmic"] / peaks["hbm_gbs"]
        stages[s] = ent
    if router_on_tc(w):
        # the logits on the tensor cores: three bf16 pieces of the gate weights,
        # so 3x the algorithmic flops run as MMAs (columns padded to 256)
        S = router_ksplit(w)
        t = stages["route"]["ms"] * 1e-3
        stages["route"]["tensor_tflops"] = 3 * work["route"]["flops"] / t / 1e12
        stages["route"]["tensor_frac"] = stages["route"]["tensor_tflops"] / peaks["bf16_tflops"]
        stages["route"]["logit_partials"] = 3 * S
    elif w.E >= 64:
        # the fp32 router GEMM at E >= 64 is bound by the FMA pipe: its fraction
        # of the FMA rate measured in this run (the small-E router is HBM-bound)
        stages["route"]["alu_frac"] = stages["route"]["tflops"] / fma_tflops
    peaks["fp32_fma_tflops"] = fma_tflops
    fc2_name = "fc2+combine" if "fc2+combine" in stages else "fc2"
    gemm_ms = stages["fc1"]["ms"] + stages[fc2_name]["ms"]
    gemm_tflops = (work["fc1"]["flops"] + work[fc2_name]["flops"]) / (gemm_ms * 1e-3) / 1e12

    dom = max(stage_names, key=lambda s: stages[s]["ms"])
    # a GEMM whose FLOP per algorithmic byte is below the ridge (peak FLOP/s
    # over peak bytes/s) is bound by HBM (DeepSeek-V3's 22.5 GB of weights
    # over ~128 rows per expert): it is measured against the HBM peak
    ridge = (2.0 if fp8 else 1.0) * peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    gemm_hbm_bound = dom in ("fc1", "fc2") and work[dom].get("bytes") and \
        work[dom]["flops"] / work[dom]["bytes"] < ridge
    if dom in ("fc1", "fc2") and w.dtype == "bf16" and not gemm_hbm_bound:
        # E4M3 MMAs: the measured bf16 peak x the nominal FP8/bf16 ratio (4.5 / 2.25)
        ratio = 2.0 if fp8 else 1.0
        roof = {"kernel": gemm_kernel_name(w, w.T * w.k, dom) + ("[E4M3]" if fp8 else ""),
                "bound": "tensor", "achieved": stages[dom]["tflops"],
                "peak": ratio * peaks["bf16_tflops"], "unit": "TFLOP/s"}
    elif gemm_hbm_bound:
        name = gemm_kernel_name(w, w.T * w.k, dom) if w.dtype == "bf16" else \
            "simt_grouped_kernel<%s>" % ("FC1" if dom == "fc1" else "FC2")
        roof = {"kernel": name + ("[E4M3]" if fp8 else ""),
                "bound": "hbm", "achieved": stages[dom].get("gbs"),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "tensor_frac": stages[dom]["tflops"] / ((2.0 if fp8 else 1.0) * peaks["bf16_tflops"])}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": stages[dom].get("gbs"),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["achieved"] else None
    if roof["bound"] == "tensor" and peaks.get("bf16_tflops_sustained"):
        roof["frac_of_sustained_peak"] = roof["achieved"] / (
            (2.0 if fp8 else 1.0) * peaks["bf16_tflops_sustained"])
    roof["peak_source"] = "%s (MEASURED_PEAKS.json burst%s)" % (
        peaks["source"], " x 2, the nominal E4M3/bf16 ratio" if fp8 else "") \
        if peaks["source"] == "measured" else "fallback"
    roof["traffic"] = None if fp8 else recorded_traffic(dom, w.name)
    roof["algorithmic_per_launch"] = work[dom].get("flops") if roof["unit"] == "TFLOP/s" \
        else work[dom].get("bytes")

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all,
        # the per-step event times' median and spread beside the mean the value uses
        "step_ms_stats": {"median": statistics.median(step_ms), "min": min(step_ms),
                          "max": max(step_ms)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 experts, bf16 activations" if fp8 else w.dtype,
        "data": "synthetic (seeded, x~N(0,%g), weights~N(0,%g), random-init)" % (w.x_std, w.w_std),
        "config": dict(workload_desc(w), parallelism="replicas" if world > 1 else "single",
                       precision=args.precision),
        "grouped_gemm_tflops": gemm_tflops,
        "stages": stages,
        "rows": R, "tokens_per_expert_cv": float(np.std(tpe) / max(np.mean(tpe), 1e-9)),
        "roofline": roof,
        "e2e": e2e,
        "graph": graph,
        "gpu_launches": kernels_per_forward(w, cfg, fp8) * args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
        "peaks": peaks,
    }
    return line


def fp32_fma_rate(moe, dev, stream, iters=4096, reps=5):
    """FP32 FMA TFLOP/s of this GPU (the library's FMA-chain probe, best of
    `reps` event-timed launches after one warm-up launch)."""
    out = torch.zeros(4 * torch.cuda.get_device_properties(dev).multi_processor_count,
                      dtype=torch.float32, device=dev)
    moe.probe_fp32_fma(iters, out)
    best = None
    for _ in range(reps):
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        flops = moe.probe_fp32_fma(iters, out)
        c.record(stream)
        c.synchronize()
        t = a.elapsed_time(c) * 1e-3
        best = t if best is None or t < best else best
    return flops / best / 1e12


def run_backward(args, moe, w, cfg, inp, b, R, flush, stream, world, rank, local):
    """Time moe_backward (the saved buffers of one staged forward, a seeded dy)."""
    if args.precision != "bf16" or w.pad_to_capacity:
        raise SystemExit("--pass backward needs --precision bf16 and no pad_to_capacity")
    dev = b.y.device
    g = torch.Generator(device="cpu").manual_seed(w.seed + 7)
    dy = torch.randn((w.T, w.h), generator=g).to(moe.act_dtype(cfg)).to(dev)
    grads = moe.Grads(cfg, dev)
    fs = w.shared_f
    if fs > 0:
        sgrads = moe.SharedGrads(cfg, fs, dev)
        ws = moe.alloc_workspace_backward_shared(cfg, fs, dev)
    else:
        ws = moe.alloc_workspace_backward(cfg, dev)

    def bwd():
        if fs > 0:  # moe_backward_shared: the routed layer and the shared expert
            moe.backward_shared(cfg, fs, inp["x"], inp["Wg"], inp["gate_bias"], inp["W1"],
                                inp["W3"], inp["W2"], inp["W1s"], inp["W3s"], inp["W2s"], b, dy,
                                grads, sgrads, ws)
        else:
            moe.backward(cfg, inp["x"], inp["Wg"], inp["gate_bias"], inp["W1"], inp["W3"],
                         inp["W2"], b, dy, grads, ws)

    for _ in range(max(3, args.warmup)):
        bwd()
    moe.check(ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local, enabled=not args.no_clocks and rank == 0)
    if clocks.proc is not None:
        time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        bwd()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    moe.check(ws)
    ms = sum(a.elapsed_time(c) for a, c in ev) / args.steps
    ms_all, tokens_per_s = job_throughput(ms, w.T, world)
    if rank != 0:
        return None
    peaks = measured_peaks()
    if w.dtype != "bf16":  # the fp32 backward runs on the FMA units: their rate, measured now
        peaks["fp32_fma_tflops"] = fp32_fma_rate(moe, dev, stream)
    # expert GEMMs of the backward: fc2 dgrad 2Rfh, fc1 recompute 4Rhf, fc1
    # dgrad 4Rhf, wgrad 2Rfh + 4Rhf; the shared expert the same over T rows
    gemm_flops = 16 * R * w.h * w.f + 16 * w.T * w.h * fs
    achieved = gemm_flops / (ms * 1e-3) / 1e12
    return {
        "metric": "MoE bwd tokens/sec", "value": tokens_per_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded inputs and dy, random-init weights)",
        "config": dict(workload_desc(w), parallelism="replicas" if world > 1 else "single",
                       precision=args.precision, pass_="backward"),
        "rows": R,
        "roofline": ({"kernel": "whole backward (expert GEMM flops / backward time)",
                      "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                      "traffic": None, "algorithmic_per_launch": gemm_flops}
                     if w.dtype == "bf16" else
                     {"kernel": "whole backward (expert GEMM flops / backward time), FMA units",
                      "bound": "alu", "achieved": achieved,
                      "peak": peaks.get("fp32_fma_tflops"), "unit": "TFLOP/s",
                      "frac": achieved / peaks["fp32_fma_tflops"]
                      if peaks.get("fp32_fma_tflops") else None,
                      "traffic": None, "algorithmic_per_launch": gemm_flops}),
        "e2e": None,
        "gpu_launches": backward_launches(w) * args.steps,
        "clocks": clk,
        "peaks": peaks,
    }


def backward_launches(w):
    """Kernels moe_backward launches for workload w: router logits (two on
    the tensor cores: the weight split and the GEMM), combine backward,
    router backward, the router's parameter and token gradients
    (tensor-core path for E % 64 == 0: two bf16 splits, the dWg GEMM, its
    fold, dgate_bias, the dx GEMM; else dWg (+ its split reduction), dgate_bias,
    dx), three dgrad/recompute GEMMs, the token-gradient combine, three
    wgrad GEMMs."""
    if w.dtype == "bf16" and w.E >= 64 and w.E % 64 == 0:
        router = 6
    else:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        small = w.E <= 32
        tiles = (w.h + 511) // 512 if small else ((w.h + 63) // 64) * ((w.E + 63) // 64)
        S = min(-(-4 * sms // tiles), -(-w.T // (64 if small else 256)), 128 if small else 32)
        router = 3 + (1 if S > 1 else 0)
    logits = 2 if router_on_tc(w) else 1  # the tensor-core logits: weight split + GEMM
    return logits + 2 + router + 3 + 1 + 3 + (6 if w.shared_f > 0 else 0)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The largest per-rank value (the slowest replica sets the job time)."""
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms_local, tokens_per_rank, world, device="cuda"):
    """Whole-job tokens/s of `world` replicas: all ranks' tokens over the
    slowest rank's step time.  Returns (max ms per step, tokens/s)."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, world * tokens_per_rank / (ms / 1e3)


# ---------------------------------------------------------------- oracle timing

def np_view(t):
    """A CPU tensor as the numpy array the oracle takes (bf16 as uint16 bits)."""
    if t is None:
        return None
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_sample_run(w, inp_cpu, tokens, nthreads=0):
    """Oracle forward on the given token rows; returns seconds."""
    import oracle
    x = inp_cpu["x"][torch.from_numpy(tokens)]
    t0 = time.perf_counter()
    shared = {n: np_view(inp_cpu[n]) for n in ("W1s", "W3s", "W2s")} if w.shared_f > 0 else {}
    oracle.forward(np_view(x), np_view(inp_cpu["Wg"]), np_view(inp_cpu["W1"]),
                   np_view(inp_cpu["W3"]), np_view(inp_cpu["W2"]), w.k, w.score,
                   np_view(inp_cpu["gate_bias"]), np_view(inp_cpu["expert_bias"]),
                   0.0 if w.capacity_factor <= 0 else w.capacity_factor * w.T / len(tokens),
                   w.min_capacity, w.drop_policy, nthreads, **shared)
    return time.perf_counter() - t0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_inputs(w, device_inputs=None):
    """The workload's inputs on the host (copied from the device if given)."""
    if device_inputs is not None:
        return {k: (None if v is None else v.detach().cpu()) for k, v in device_inputs.items()}
    return synthetic.generate(w, device="cpu")


def cpu_baseline(w, inp_cpu, budget_s=15.0):
    """Oracle tokens/s on the host cores: a 4-token probe sizes one timed
    sample of about `budget_s` seconds."""
    cores = host_cores()
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(w.T, size=min(4, w.T), replace=False))
    per_token = oracle_sample_run(w, inp_cpu, probe, cores) / len(probe)
    n = int(min(w.T, max(4, budget_s / max(per_token, 1e-6))))
    toks = np.sort(rng.choice(w.T, size=n, replace=False))
    sec = oracle_sample_run(w, inp_cpu, toks, cores)
    # the same oracle on one thread: a smaller sample (about budget_s / 2)
    n1 = int(min(n, max(2, 0.5 * budget_s / max(per_token * cores, 1e-6))))
    toks1 = np.sort(rng.choice(w.T, size=n1, replace=False))
    sec1 = oracle_sample_run(w, inp_cpu, toks1, 1)
    return {"value": n / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu": cpu_model(), "seconds": sec,
            "sample": "%d random tokens (fixed seed) of the %s workload; oracle forward (route, "
                      "permute, SwiGLU experts, combine) in double on %d threads"
                      % (n, w.name, cores),
            "one_thread": {"value": n1 / sec1, "unit": UNIT, "cores": 1, "seconds": sec1,
                           "sample": "%d random tokens of the same workload, one thread" % n1}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = workload_of(args)
    inp_cpu = cpu_inputs(w)
    cores = host_cores()
    rng = np.random.default_rng(1)
    sample = 8 if w.T * w.k * w.h * w.f > 1e11 else 64
    for _ in range(min(args.warmup, 1)):
        oracle_sample_run(w, inp_cpu, np.sort(rng.choice(w.T, sample, replace=False)), cores)
    times = []
    for _ in range(args.steps):
        toks = np.sort(rng.choice(w.T, sample, replace=False))
        times.append(oracle_sample_run(w, inp_cpu, toks, cores))
    sec = sum(times) / len(times)
    value = sample / sec
    desc = ("%d random tokens of the %s workload per step; CPU oracle (double) on %d threads"
            % (sample, w.name, cores))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_desc(w), parallelism="replicas" if world > 1 else "single",
                           precision=args.precision),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_native(args, rank, world, local)
    if line is not None and world == 1 and not args.no_cpu_baseline:
        import mixture_experts_layer_fp32_gb300 as moe  # noqa: F401
        w = workload_of(args)
        dev_inp = synthetic.generate(w, device="cuda", seed=w.seed)
        inp_cpu = cpu_inputs(w, dev_inp)
        del dev_inp
        line["cpu_baseline"] = cpu_baseline(w, inp_cpu)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
