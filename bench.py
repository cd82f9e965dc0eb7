#!/usr/bin/env python
"""MoE layer forward benchmark on GB300.

One step = one moe_forward (router, dispatch, grouped expert FFN, combine) over
one batch of n synthetic tokens with the layer's weights resident in HBM.
Default workload: the largest one-GPU layer, fine-grained experts plus a shared
expert (n=16384, d=7168, d_ff=2048, E=256, top-8, shared SwiGLU expert of
d_ff=2048, bf16).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--n N]
  python bench.py --impl reference ...   # the fp64 CPU oracle on a bounded sample

Multi-GPU (torchrun, one rank per GPU): each rank runs its own batch with its
own copy of the weights (data parallel, no collective on the data path); the
reported value is all ranks' tokens / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import moe_synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per launch of the dominant kernel from an ncu
# capture of the same workload and kernel version (profiles/ has the summary).
MEASURED_TRAFFIC = {
    ("finegrained_shared_bf16", 16384, "ffn_up"): 22.632e9 + 0.534e9,
    ("mixtral_bf16", 4096, "ffn_up"): 1.973e9 + 0.229e9,
    ("gptoss_prefill_zipf_mxfp4", 8192, "ffn_up"): 1.080e9 + 0.368e9,
    ("gptoss_decode_mxfp4", 64, "ffn_up"): 1.03e9 + 0.00734e9,
    # the fused small-batch launch (one launch of the rotation's first batch)
    ("gptoss_decode_mxfp4", 1, "fused"): 53.94e6 + 0.247e6,
    ("gptoss_decode_mxfp4", 4, "fused"): 201.95e6 + 4.56e6,
    ("gptoss_decode_mxfp4", 16, "fused"): 710.3e6 + 6.21e6,
    ("gptoss_decode_nvfp4", 1, "fused"): 57.05e6 + 0.138e6,
    ("gptoss_decode_nvfp4", 8, "fused"): 407.5e6 + 4.95e6,
}
L2_BYTES = 129 * 1024 * 1024
# a timed loop at least this long runs at the power-capped clock: the sustained
# bf16 peak (measured over a seconds-long loop) is its denominator
SUSTAINED_LOOP_S = 2.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default="finegrained_shared_bf16", choices=sorted(moe_synth.CONFIGS))
    p.add_argument("--n", type=int, default=None, help="override the token count")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layers", type=int, default=1,
                   help="MoE layers per step (independently seeded weights, run in sequence)")
    p.add_argument("--cpu-sample", type=int, default=None,
                   help="tokens in the oracle's timed sample")
    p.add_argument("--pool-fraction", type=float, default=None,
                   help="small-batch MXFP4 workloads: run moe_forward_pooled with this share of "
                        "each layer's experts resident in a slot pool (the rest read from the "
                        "backing arrays)")
    return p.parse_args(argv)


# --------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def job_throughput(units_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job units/s: all ranks' units over the (max-over-ranks) time."""
    return units_per_rank * world / seconds


# -------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ roofline

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


DECODE_MAX_PAIRS = 256   # the library's small-batch MXFP4 path (n*k up to this)
DECODE_BATCHES = 8       # token batches rotated through in decode timing


def is_decode(cfg) -> bool:
    return cfg.weight_dtype in ("mxfp4", "nvfp4") and cfg.n * cfg.k <= DECODE_MAX_PAIRS


def layer_bytes(cfg, active_experts):
    """Algorithmic bytes of one small-batch layer: each selected expert's weights
    (codes + scales) once, the router's weights, x in and y out."""
    return (active_experts * moe_synth.weight_bytes_per_expert(cfg)
            + cfg.E * cfg.d * 2 + 2 * cfg.n * cfg.d * 2)


def dominant_kernel(cfg, active_experts=None, fused=False):
    """(stage name, bound, algorithmic units per launch, unit) of the dominant kernel.

    Tensor-bound workloads: the up-projection grouped GEMM (W1 and W3, 2/3 of the
    expert FLOPs with SwiGLU), FLOPs = 2 * (n*k) * d * d_ff * (2 for SwiGLU, else 1).
    Small-batch FP4 (decode) run as one fused launch: that launch, whose bytes are
    the whole layer's (layer_bytes).  Small-batch FP4 run as chained launches: the
    up-projection kernel streams the selected experts' W1/W3 codes and scales once,
    reads the tokens' x rows and writes h: bytes = u * mats * d_ff * (d/2 + d/32)
    + n*k*d*2 + n*k*d_ff*2 (MXFP4; NVFP4 has d/16 scale bytes per row and one fp32
    scale per matrix).
    """
    mats = 2 if cfg.act == "swiglu" else 1
    if is_decode(cfg) and fused:
        u = active_experts if active_experts is not None else min(cfg.E, cfg.n * cfg.k)
        return "fused", "hbm", layer_bytes(cfg, u), "GB/s"
    if is_decode(cfg):
        u = active_experts if active_experts is not None else min(cfg.E, cfg.n * cfg.k)
        P = cfg.n * cfg.k
        scale_bytes = cfg.d // 16 if cfg.weight_dtype == "nvfp4" else cfg.d // 32
        extra = 4 if cfg.weight_dtype == "nvfp4" else 0
        nbytes = (u * mats * (cfg.d_ff * (cfg.d // 2 + scale_bytes) + extra)
                  + P * cfg.d * 2 + P * cfg.d_ff * 2)
        return "ffn_up", "hbm", nbytes, "GB/s"
    flops = 2 * cfg.n * cfg.k * cfg.d * cfg.d_ff * mats
    return "ffn_up", "tensor", flops, "TFLOP/s"


def make_event(timing=True, external=False):
    if external:
        try:
            return torch.cuda.Event(enable_timing=timing, external=True)
        except TypeError:
            return None
    return torch.cuda.Event(enable_timing=timing)


# -------------------------------------------------------------- CPU baseline

def host_copy(inputs_dev):
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs_dev.items()}


def oracle_sample(cfg, inputs_host, tokens: int, seed: int):
    """A bounded sample of the workload for the fp64 oracle: `tokens` seeded rows
    of x with the full layer's weights."""
    g = torch.Generator().manual_seed(seed)
    rows = torch.sort(torch.randperm(cfg.n, generator=g)[:tokens]).values
    sub = dict(inputs_host)
    sub["x"] = inputs_host["x"][rows]
    return cfg.scaled(n=int(rows.numel())), sub


def time_oracle_step(scfg, sub):
    from oracle import moe_oracle as O   # the CPU baseline leg is the oracle as it stands
    t0 = time.perf_counter()
    O.forward(scfg, sub)
    return time.perf_counter() - t0


def default_cpu_sample(cfg):
    return {"tiny_switch_fp32": 256, "mixtral_bf16": 4096, "gptoss_decode_mxfp4": cfg.n,
            "gptoss_decode_nvfp4": cfg.n,
            "gptoss_prefill_zipf_mxfp4": 256, "finegrained_shared_bf16": 2048}.get(cfg.name, 64)


# ----------------------------------------------------------------- our arm

def workload_name(cfg):
    return moe_synth.describe(cfg)


def run_ours(args):
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    from mixture_experts_layer_moe_gb300 import build as _b
    if rank == 0 or world == 1:
        _b.build()
    barrier(device)
    from mixture_experts_layer_moe_gb300 import moe

    cfg = moe_synth.CONFIGS[args.config]
    if args.n:
        cfg = cfg.scaled(n=args.n)
    # each rank draws its own token batch; the weights are the same layer
    inputs = moe_synth.make_inputs(cfg, seed=args.seed, device=device)
    if rank:
        g = torch.Generator(device=device).manual_seed(args.seed + 1000 * rank)
        x = torch.randn(inputs["x"].shape, generator=g, device=device, dtype=torch.float32)
        inputs["x"] = (x * cfg.x_std).to(inputs["x"].dtype)
    w = moe.make_weights(inputs)
    ws = moe.alloc_workspace(cfg, device)
    y = torch.empty(cfg.n, cfg.d, dtype=inputs["x"].dtype, device=device)
    mid = [torch.empty_like(y) for _ in range(2)]
    # further layers of the stack: their own seeded weights, same shapes.
    # Each layer reads its own token batch (layer l of step i the batch
    # i + l of the rotation) rather than the previous layer's output: a chain
    # of these random layers, which has none of a model's residual
    # connections, collapses onto a few experts (n = 64: 116 experts with
    # tokens in layer 0, 8 from layer 9 on), a routing no model step has.
    # The layers still run one after another on one stream.
    layer_inputs = [inputs] + [moe_synth.make_stack_inputs(cfg, l, seed=args.seed, device=device)
                               for l in range(1, args.layers)]
    layer_w = [w] + [moe.make_weights(li) for li in layer_inputs[1:]]

    # expert-slot indirection: a seeded resident set per layer, copied into a
    # slot pool; the classification of every layer lands in its own counts
    pools, pool_keep, pool_counts = [], [], []
    if args.pool_fraction is not None:
        if not is_decode(cfg):
            raise SystemExit("--pool-fraction applies to small-batch MXFP4 workloads")
        resident = round(args.pool_fraction * cfg.E)
        n_slots = max(1, resident)
        for l, li in enumerate(layer_inputs):
            table = moe_synth.make_slot_table(cfg.E, n_slots, resident, seed=args.seed + 31 * l)
            tensors = moe_synth.make_pool(li, table, n_slots, device=device)
            table_dev = table.to(device)
            pool_keep.append((tensors, table_dev))
            pools.append(moe.make_pool(table_dev, tensors))
            pool_counts.append(torch.zeros(4, dtype=torch.int32, device=device))
        pool_state = torch.empty(cfg.E, dtype=torch.int32, device=device)
        pool_miss = torch.empty(cfg.E, dtype=torch.int32, device=device)

    ccfg = moe.make_config(cfg)   # the C struct once, as a caller would build it

    def run_layers(x_in, y_out, hook=None, active=None, batch=0):
        """Layer 0 .. L-1 in sequence; the stage hook instruments layer 0.
        Layer 0 reads x_in, layer l > 0 token batch batch + l of the rotation.
        active (a list): receives each layer's count of experts with tokens."""
        for l in range(args.layers):
            cur = x_in if l == 0 else x_pool[(batch + l) % len(x_pool)]
            out = y_out if l == args.layers - 1 else mid[l % 2]
            if pools:
                if l == 0 and hook is not None:
                    moe.moe_forward_pooled_staged(ccfg, cur, layer_w[l], pools[l], out, pool_state,
                                                  pool_miss, pool_counts[l], ws, hook, stream)
                else:
                    moe.moe_forward_pooled(ccfg, cur, layer_w[l], pools[l], out, pool_state,
                                           pool_miss, pool_counts[l], ws, stream)
            elif l == 0 and hook is not None:
                moe.moe_forward_staged(ccfg, cur, layer_w[l], out, ws, hook, stream)
            else:
                moe.moe_forward(ccfg, cur, layer_w[l], out, ws, stream)
            if active is not None:
                torch.cuda.synchronize(device)
                active.append(int((counts > 0).sum().item()))
    # a non-default stream: CUDA graphs cannot be captured on the legacy default stream
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)

    stage_names = moe.STAGES
    launches = {"n": 0}
    # Small-batch MXFP4 steps read only the selected experts (tens of MB, below
    # L2): rotate over seeded token batches so each step routes differently and
    # its experts come from HBM, as in a real decode loop.
    n_batches = DECODE_BATCHES if is_decode(cfg) else 1
    x_pool = [inputs["x"]]
    for r in range(1, n_batches):
        gr = torch.Generator(device=device).manual_seed(args.seed + 7919 * r + 1000 * rank)
        xr = torch.randn(inputs["x"].shape, generator=gr, device=device, dtype=torch.float32)
        x_pool.append((xr * cfg.x_std).to(inputs["x"].dtype))

    end_stage = stage_names.index("end")
    seen_order = []   # stage ids in the order the hook reports them (one step)

    def step(i, events=None, active=None):
        def hook(stage, kernels):
            if events is not None:
                events[stage].record(stream)
            if not seen_order or seen_order[-1] != end_stage:
                seen_order.append(stage)
            if stage == end_stage:
                launches["n"] = kernels
        run_layers(x_pool[i % n_batches], y, hook, active, batch=i)

    L = moe.moe_workspace_layout_of(cfg)
    counts = ws[L["counts"]:L["counts"] + 4 * cfg.E].view(torch.int32)
    # experts with tokens, per token batch: layer 0 (the instrumented one) and
    # the whole stack
    active_per_batch, stack_active_per_batch, served = [], [], []
    for i in range(max(args.warmup, n_batches)):
        per_layer = [] if i < n_batches else None
        step(i, active=per_layer)
        if i < n_batches:
            active_per_batch.append(per_layer[0])
            stack_active_per_batch.append(per_layer)
            for pc in pool_counts:
                c4 = pc.tolist()
                served.append(c4[moe.POOL_SERVED] / c4[moe.POOL_LOOKUPS])
    torch.cuda.synchronize(device)
    st, detail = moe.moe_status_check(ws)
    if st != 0:
        raise RuntimeError(f"device status {moe.status_string(st)} ({detail})")
    fused = stage_names.index("fused") in seen_order
    step_units = [dominant_kernel(cfg, active_per_batch[i % n_batches], fused)[2]
                  for i in range(args.steps)]
    active = statistics.mean(active_per_batch[i % n_batches] for i in range(args.steps))
    dom_stage, bound, _, dom_unit = dominant_kernel(cfg, fused=fused)
    dom_units = statistics.mean(step_units)

    # The timed region: K steps captured into one CUDA graph (external event
    # nodes between stages) and replayed once; eager launches if capture fails.
    timing = "cuda_graph"
    graph = None
    plain = None
    ev = [[make_event(external=True) for _ in stage_names] for _ in range(args.steps)]
    if any(e is None for row in ev for e in row):
        print("bench: torch.cuda.Event(external=True) unavailable; timing eager launches",
              file=sys.stderr)
        timing = "eager"
    else:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(args.steps):
                    step(i, ev[i])
            plain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(plain, stream=stream):
                for i in range(args.steps):
                    step(i)
            torch.cuda.synchronize(device)
        except Exception as exc:  # capture unsupported here: time eager launches instead
            print(f"bench: CUDA graph capture failed ({exc!r}); timing eager launches",
                  file=sys.stderr)
            graph, timing = None, "eager"
            torch.cuda.synchronize(device)
    if graph is None:
        ev = [[make_event() for _ in stage_names] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    # timed region: the K steps (the graph without stage events when captured),
    # then the same K steps with the stage events for the per-stage breakdown
    with ClockSampler(device.index) as clocks:
        start.record(stream)
        if plain is not None:
            plain.replay()
        else:
            for i in range(args.steps):
                step(i, ev[i])
        stop.record(stream)
        if graph is not None:
            graph.replay()
        torch.cuda.synchronize(device)
    barrier(device)
    elapsed = start.elapsed_time(stop) / 1e3
    t_job = max_over_ranks(elapsed, device)
    kernels_per_step = launches["n"] * args.layers
    st, detail = moe.moe_status_check(ws)
    if st != 0:
        raise RuntimeError(f"device status {moe.status_string(st)} ({detail})")

    # per-stage durations (CUDA events on the launching stream, inside the
    # timed region): each stage runs from its event to the next stage's
    stage_ms = {}
    for s, nxt in zip(seen_order, seen_order[1:]):
        stage_ms[stage_names[s]] = statistics.mean(
            ev[i][s].elapsed_time(ev[i][nxt]) for i in range(args.steps))
    dom_ms = stage_ms[dom_stage]
    del graph, plain

    # end to end: every step copies its x from pinned host memory, runs the
    # layer through the C ABI and copies y back to pinned host memory.  For
    # copies of a megabyte or more, as a serving loop would, they run on their
    # own streams with double buffers: step i + 1's input copy and step i - 1's
    # output copy overlap step i's layer, and each step's layer waits for its
    # own input copy.  Smaller copies stay on the layer's stream, in order
    # (the extra stream calls would cost more host time than the copies).
    x_host = inputs["x"].cpu().pin_memory()
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inputs["x"]) for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def e2e_steps(count, first_event):
        done = [None] * count
        out = [None] * count
        h2d.wait_event(first_event)
        d2h.wait_event(first_event)
        for i in range(count):
            b = i % 2
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(done[i - 2])          # x_dev[b] no longer read
                x_dev[b].copy_(x_host, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(h2d)
            stream.wait_event(ready)
            if i >= 2:
                stream.wait_event(out[i - 2])            # y_dev[b] copied out
            run_layers(x_dev[b], y_dev[b])
            done[i] = torch.cuda.Event()
            done[i].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done[i])
                y_host[b].copy_(y_dev[b], non_blocking=True)
                out[i] = torch.cuda.Event()
                out[i].record(d2h)
        stream.wait_event(out[count - 1])

    copy_bytes = 2 * x_host.numel() * x_host.element_size()
    overlap = copy_bytes >= (1 << 20)

    def e2e_serial(count, first_event):
        for _ in range(count):
            x_dev[0].copy_(x_host, non_blocking=True)
            run_layers(x_dev[0], y_dev[0])
            y_host[0].copy_(y_dev[0], non_blocking=True)

    if not overlap:
        e2e_steps = e2e_serial  # noqa: F811
    warm = torch.cuda.Event()
    warm.record(stream)
    e2e_steps(2, warm)
    torch.cuda.synchronize(device)
    barrier(device)
    # two clocks around the same loop: the host's wall clock (it includes
    # every call's enqueue cost on this thread, the binding's ctypes calls
    # among them, and any host stall between steps) and CUDA events on the
    # layer's stream; the reported value is the wall-clock one
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    e0.record(stream)
    e2e_steps(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize(device)
    h1 = time.perf_counter()
    t_e2e = max_over_ranks(h1 - h0, device)
    t_e2e_events = max_over_ranks(e0.elapsed_time(e1) / 1e3, device)
    st, detail = moe.moe_status_check(ws)
    if st != 0:
        raise RuntimeError(f"device status {moe.status_string(st)} ({detail})")

    peaks, peak_src = load_peaks()
    step_bytes = (active if is_decode(cfg) else cfg.E) * moe_synth.weight_bytes_per_expert(cfg)
    if n_batches > 1:
        l2_note = (f"{n_batches} seeded token batches rotate through the timed steps, so each "
                   f"step routes to other experts ({step_bytes / 1e6:.1f} MB of expert weights "
                   f"per step on average; L2 is {L2_BYTES / 1e6:.0f} MB)")
    else:
        l2_note = (f"inputs larger than L2: {step_bytes / 1e9:.3f} GB of expert weights read per "
                   f"step" if step_bytes > L2_BYTES else
                   f"expert weights read per step ({step_bytes / 1e6:.1f} MB) fit in L2 and are "
                   f"not flushed: the step may run from L2")
    # the dominant kernel's duration comes from the stage-event replay that
    # follows the plain one, so its kernels run inside a loop of 2 x K steps:
    # the sustained (power-capped) peak applies when that loop lasts seconds,
    # the burst peak otherwise
    loop_s = 2 * elapsed
    if bound == "tensor":
        sustained = loop_s >= SUSTAINED_LOOP_S and "bf16_tflops_sustained" in peaks
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        peak_kind = (f"bf16 sustained: kernel timed inside a {loop_s:.1f} s loop" if sustained else
                     f"bf16 burst: kernel timed inside a {loop_s:.2f} s loop")
        achieved = dom_units / (dom_ms / 1e3) / 1e12
    else:
        peak = peaks["hbm_gbs"]
        peak_kind = "hbm copy"
        achieved = dom_units / (dom_ms / 1e3) / 1e9
    per_launch = ({"flops_per_launch": dom_units} if bound == "tensor"
                  else {"bytes_per_launch": dom_units, "active_experts_mean": active})
    if is_decode(cfg):
        # the whole layer (stack) against HBM on its algorithmic bytes: each
        # layer's selected experts' weights once each, the router's weights,
        # x in and y out
        stack_active = statistics.mean(sum(stack_active_per_batch[i % n_batches])
                                       for i in range(args.steps))
        stack_bytes = (stack_active * moe_synth.weight_bytes_per_expert(cfg)
                       + (cfg.E * cfg.d * 2 + 2 * cfg.n * cfg.d * 2) * args.layers)
        layer_gbs = stack_bytes / (t_job / args.steps) / 1e9
        per_launch["whole_layer"] = {
            "bytes_per_step": stack_bytes, "achieved": layer_gbs, "unit": "GB/s",
            "frac": layer_gbs / peaks["hbm_gbs"],
            "bytes": "selected experts' weights (codes + scales) + router weights + x + y",
            **({"active_experts_per_layer_first_batch": stack_active_per_batch[0]}
               if args.layers > 1 else {})}

    out = {
        "metric": ("MoE-layer tokens/s" if args.layers == 1 else
                   f"MoE-stack tokens/s ({args.layers} layers per step)"),
        "value": job_throughput(cfg.n * args.steps, world, t_job),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_job / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32" if cfg.act_dtype == "f32" else "bf16",
        "data": "synthetic (seeded normal x and weights; MXFP4 codes/scales uniform)",
        "config": {
            "workload": workload_name(cfg),
            "tokens_per_rank": cfg.n,
            "layers_per_step": args.layers,
            **({"stack": "independently seeded layers run in sequence on one stream; layer l "
                         "reads its own token batch (a chain of these random layers without "
                         "residual connections collapses onto a few experts)"}
               if args.layers > 1 else {}),
            "parallelism": f"dp{world} (independent token batches, replicated weights)",
            "l2": l2_note,
            "timing": timing,
            **({"expert_pool": {
                "resident_fraction": args.pool_fraction,
                "resident_experts_per_layer": round(args.pool_fraction * cfg.E),
                "lookups_served_fraction": statistics.mean(served),
                "path": "moe_forward_pooled (resident experts read from their pool slots, the "
                        "others from the backing arrays)"}} if pools else {}),
        },
        "e2e": {"value": job_throughput(cfg.n * args.steps, world, t_e2e), "unit": "tokens/s",
                "clock": "host wall clock around the loop (enqueue + copies + layer)",
                "value_gpu_events": job_throughput(cfg.n * args.steps, world, t_e2e_events),
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host[0].numel() * y_host[0].element_size(),
                "copies": ("pinned host buffers; input and output copies on their own streams, "
                           "double-buffered: step i+1's input and step i-1's output copies "
                           "overlap step i's layer") if overlap else
                          "pinned host buffers; copies in order on the layer's stream"},
        "gpu_launches": kernels_per_step * args.steps,
        "roofline": {"kernel": dom_stage, "bound": bound, "achieved": achieved, "peak": peak,
                     "unit": dom_unit, "frac": achieved / peak,
                     "peak_source": f"{peak_src} ({peak_kind})",
                     "traffic": (MEASURED_TRAFFIC.get((cfg.name, cfg.n, dom_stage))
                                 if args.layers == 1 else None), **per_launch},
        "stages_ms": stage_ms,
        "clocks": clocks.summary(),
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.layers == 1:
        tokens = args.cpu_sample or default_cpu_sample(cfg)
        del x_host, y_host, x_dev
        scfg, sub = oracle_sample(cfg, host_copy(inputs), tokens, args.seed)
        secs = time_oracle_step(scfg, sub)
        out["cpu_baseline"] = {"value": scfg.n / secs, "unit": "tokens/s",
                               "cores": torch.get_num_threads(), "kind": "oracle",
                               "sample": f"{scfg.n} of {cfg.n} token rows, full layer weights, "
                                         f"fp64 oracle, {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    cfg = moe_synth.CONFIGS[args.config]
    if args.n:
        cfg = cfg.scaled(n=args.n)
    device = "cuda" if torch.cuda.is_available() else "cpu"
    inputs = host_copy(moe_synth.make_inputs(cfg, seed=args.seed, device=device))
    # size each step's sample so that warm-up + timed steps take about two minutes:
    # the first warm-up step measures the oracle's rate on a small sample
    budget_s = 120.0
    tokens = args.cpu_sample or min(cfg.n, 32)
    times, done = [], 0
    scfg = None
    for i in range(args.warmup + args.steps):
        scfg, sub = oracle_sample(cfg, inputs, tokens, args.seed + i)
        secs = time_oracle_step(scfg, sub)
        if i == 0 and not args.cpu_sample:
            per_step = budget_s / max(1, args.warmup + args.steps - 1)
            tokens = int(max(1, min(cfg.n, scfg.n * per_step / max(secs, 1e-3))))
        if i >= args.warmup:
            times.append(secs)
            done += scfg.n
    total = sum(times)
    value = done / total
    out = {
        "impl": "reference",
        "metric": "MoE-layer tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same generator and seed as the GPU arm)",
        "config": {"workload": workload_name(cfg), "tokens_per_rank": cfg.n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": torch.get_num_threads(),
                         "kind": "oracle",
                         "sample": f"{done // len(times)} of {cfg.n} token rows per step "
                                   f"(seeded rows), full layer weights"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
