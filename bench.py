"""Benchmark of the MoE expert layer on GB300.

One step = one whole layer (router, top-k, align, gate_up+SwiGLU, down, combine,
shared expert) over one batch of seeded synthetic tokens.  Default workload: the
speculative-verify layer, T=8 tokens (1 target + 7 draft positions), d=2048,
E=256 routed experts, top-8 renormalised, I=512, shared expert I=512, bf16.

Prints one JSON line (rank 0).  `value` = tokens/s of the whole job with inputs
resident in HBM; `e2e` = the same through the C ABI with the step's x copied from
pinned host memory and out copied back inside the timed region.

L2: the 129 MB L2 is not allowed to serve weights across steps: steps rotate
over several device copies of the full weight set (together well over 2x L2),
and over several token batches.

--impl reference times the fp64 CPU oracle (the only reference there is: the
source pages publish no code for this layer) on the same workload, metric and
unit, on the host cores.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s & achieved HBM GB/s (T=8 verify) vs roofline; prefill TFLOP/s"
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="verify_t8")
    p.add_argument("--also", default="tiny,verify_t64,verify_t64_skew,int4_t32,prefill_t4096",
                   help="further workloads measured in the same run ('none' = none); each "
                        "gets its own entry under 'workloads' in the JSON line")
    p.add_argument("--copies", type=int, default=0, help="weight copies to rotate (0 = auto)")
    p.add_argument("--batches", type=int, default=8, help="token batches to rotate")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def ranks_max(vals, dev):
    """Element-wise max of `vals` over the ranks of the process group (each
    rank's own values when there is none): per-step times, so the job's time
    is its slowest replica's."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(T, world, ms_per_step):
    """Whole-job throughput: every replica processes T tokens per step, and
    the step time is the max over ranks."""
    return world * T / (ms_per_step * 1e-3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- byte model
def algorithmic(shape, ids_list):
    """Per-step algorithmic bytes (whole layer and gate_up stage) and flops,
    averaged over the token batches' actual routing.  Touched experts only; no
    padding, no intermediates beyond the stage's own inputs/outputs."""
    s = shape
    if s.fmt == "int4":
        gu_e = 2 * s.I * (s.d // 2 + s.d // s.group * 2)
        dn_e = s.d * (s.I // 2 + s.I // s.group * 2)
    else:
        gu_e = 2 * s.I * s.d * 2
        dn_e = s.d * s.I * 2
    sh_gu = 2 * s.Is * s.d * 2
    sh_dn = s.d * s.Is * 2
    router = s.E * s.d * 2
    x = s.T * s.d * 2
    out = s.T * s.d * 2
    layer_b, gu_b, touched = [], [], []
    for ids in ids_list:
        n = len(set(ids.reshape(-1).tolist()))
        touched.append(n)
        layer_b.append(n * (gu_e + dn_e) + sh_gu + sh_dn + (s.d * 2 if s.Is else 0) + router + x + out)
        gu_b.append(n * gu_e + sh_gu + x)
    flops = 2 * s.T * s.k * 3 * s.I * s.d + 2 * s.T * 3 * s.Is * s.d + 2 * s.T * s.E * s.d
    return {"layer_bytes": statistics.mean(layer_b), "gate_up_bytes": statistics.mean(gu_b),
            "touched": statistics.mean(touched), "flops": flops}


def tensor_core_path(s):
    """Whether the library runs this layer's expert stages as grouped tcgen05
    GEMMs (its dispatch rule: T >= 256, bf16 routed weights, 128-row align
    blocks, I % 128 == 0, d % 256 == 0, shared expert absent or as wide)."""
    return (s.T >= 256 and s.fmt == "bf16" and s.block % 128 == 0 and s.I % 128 == 0
            and s.d % 256 == 0 and s.Is in (0, s.I))


def gate_up_flops(s):
    """Algorithmic flops of the gate_up stage: real routed rows (no padding)
    plus the shared expert."""
    return 2 * s.T * s.k * 2 * s.I * s.d + 2 * s.T * 2 * s.Is * s.d


def kernel_traffic(src_name, workload, algorithmic_bytes):
    """DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
    capture recorded in profiles/gate_up_<workload>.json -- scaled from the
    captured token batch to this run's by the algorithmic bytes -- or None when
    the kernel source changed since the capture."""
    prof = os.path.join(ROOT, "profiles", f"gate_up_{workload}.json")
    src = os.path.join(ROOT, "moe_expert_layer_gemv_gb300", "csrc", src_name)
    try:
        rec = json.load(open(prof))
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("source_sha256") == h:
            return rec["dram_bytes_per_launch"] * algorithmic_bytes / rec["algorithmic_bytes_of_capture"]
    except (OSError, ValueError, KeyError):
        pass
    return None


# --------------------------------------------------------------------------- CPU oracle
def host_cores():
    """Cores this process may run on (torchrun sets OMP_NUM_THREADS=1 for
    multi-process jobs, so the oracle is given this count explicitly)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_tokens_per_s(inp, seconds, nthreads=0, chunk=0):
    """Time the fp64 oracle on the workload's batch until `seconds`: whole
    batches, or (chunk > 0) successive runs of `chunk` of its tokens."""
    import oracle
    from moe_expert_layer_gemv_gb300 import inputs as I

    s = inp["shape"]
    fmt = oracle.BF16 if s.fmt == "bf16" else oracle.INT4
    conv = I.bits if s.fmt == "bf16" else (lambda t: t.numpy())
    ex = {"format": fmt, "group": s.group, "gate_up": conv(inp["gate_up"]), "down": conv(inp["down"]),
          "gate_up_scales": None if inp["gate_up_scales"] is None else I.bits(inp["gate_up_scales"]),
          "down_scales": None if inp["down_scales"] is None else I.bits(inp["down_scales"])}
    sh = None
    if s.Is:
        sh = {"gate_up": I.bits(inp["shared_gate_up"]), "down": I.bits(inp["shared_down"]),
              "gate_w": I.bits(inp["w_sg"])}
    dims = {"T": s.T, "d": s.d, "E": s.E, "k": s.k, "I": s.I, "Is": s.Is,
            "renormalize": int(s.renormalize)}
    xb, rb = I.bits(inp["x"]), I.bits(inp["router_w"])
    import numpy as np

    tokens, t0 = 0, time.perf_counter()
    while True:
        if chunk > 0:
            sel = (tokens + np.arange(chunk, dtype=np.int32)) % s.T
            oracle.layer(xb, rb, ex, sh, dims, tokens=sel, nthreads=nthreads)
            tokens += chunk
        else:
            oracle.layer(xb, rb, ex, sh, dims, nthreads=nthreads)
            tokens += s.T
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    threads = nthreads if nthreads > 0 else oracle.max_threads()
    return tokens / el, threads, tokens, el


def run_reference(args, shape):
    """The reference arm: the fp64 CPU oracle on the host cores."""
    from moe_expert_layer_gemv_gb300 import inputs as I

    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = I.make_inputs(shape, seed=0)
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_tokens_per_s(inp, 0.0, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_tokens_per_s(inp, 0.0, nthreads=cores)
    el = time.perf_counter() - t0
    v = args.steps * shape.T / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": shape.name, "T": shape.T, "d": shape.d,
                                            "E": shape.E, "top_k": shape.k, "I": shape.I,
                                            "I_shared": shape.Is, "weights": shape.fmt},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} full steps of {shape.T} tokens, fp64, "
                                       f"OpenMP over tokens"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def measure(shape, args, dev, world, local, inp0, e2e):
    """Time one workload on this rank's GPU.

    Region A: `steps` layer calls with inputs resident in HBM between two
    events (the value), then the same calls as up to 5 rounds with an event at
    each boundary to check their spread (when the rounds vary by more than 3 %,
    region A is run once more).  Region B: the same steps through
    moe_layer_forward_timed, events at the stage boundaries (an event between
    two kernels also stops the second from starting early, so stage times
    include each stage's launch; region A has none of that).  Region C (e2e):
    x copied from pinned host memory and out copied back inside the timed
    loop.  Weight copies rotate so that the bytes in flight exceed L2 several
    times over."""
    import torch
    import torch.distributed as dist

    from moe_expert_layer_gemv_gb300 import abi
    from moe_expert_layer_gemv_gb300 import inputs as I
    from moe_expert_layer_gemv_gb300.layer import MoeLayer

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 0
    layer0 = MoeLayer(inp0, dev)
    w_bytes = sum(t.numel() * t.element_size() for t in
                  [layer0.router_w, layer0.gate_up, layer0.down] +
                  [t for t in [layer0.gate_up_scales, layer0.down_scales] if t is not None] +
                  ([layer0.s_gate_up, layer0.s_down, layer0.w_sg] if shape.Is else []))
    ncopy = args.copies or max(2, math.ceil(4 * max(l2, 128 << 20) / w_bytes))
    layers = [layer0] + [MoeLayer(inp0, dev) for _ in range(ncopy - 1)]
    xs = [I.make_x(shape, seed=100 + b).to(dev) for b in range(args.batches)]
    outs = [torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=dev) for _ in xs]
    ids_dev = [torch.empty((shape.T, shape.k), dtype=torch.int32, device=dev) for _ in xs]
    for b, x in enumerate(xs):
        layers[0].forward(x, outs[b], topk_ids=ids_dev[b])
    torch.cuda.synchronize()
    ids_host = [t.cpu().numpy() for t in ids_dev]
    alg = algorithmic(shape, ids_host)

    def step(i, stream=None):
        b = i % len(xs)
        layers[i % ncopy].forward(xs[b], outs[b], stream=stream)

    steps = args.steps
    clocks = ClockSampler(local) if e2e else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # The warm-up runs right before the timed region (no idle GPU in between).
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    def region_a():
        # The timed region: exactly `steps` layer calls between two events, so
        # that nothing in the stream breaks the programmatic launch chain from
        # one layer to the next.
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        n0 = abi.moe_kernel_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms_a = e0.elapsed_time(e1) / steps
        n_launch = abi.moe_kernel_launch_count() - n0
        # Spread check, not part of the value: the same calls again as up to
        # five rounds with an event at each boundary (each boundary event also
        # ends one launch chain, so rounds read a little slower than the value).
        nr = min(5, steps)
        cut = [round(r * steps / nr) for r in range(nr + 1)]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nr + 1)]
        ev[0].record()
        for r in range(nr):
            for i in range(cut[r], cut[r + 1]):
                step(i)
            ev[r + 1].record()
        torch.cuda.synchronize()
        per = [ev[r].elapsed_time(ev[r + 1]) / (cut[r + 1] - cut[r]) for r in range(nr)]
        cv = statistics.pstdev(per) / statistics.mean(per)
        return (ms_a, n_launch,
                {"n": nr, "us_per_step": [round(v * 1e3, 2) for v in per],
                 "median_us": statistics.median(per) * 1e3, "cv": cv})

    ms, launches, rounds = region_a()
    first_cv = ranks_max([rounds["cv"]], dev)[0]  # every rank takes the same decision
    if first_cv > 0.03:
        if world > 1:
            dist.barrier()
        ms, launches, rounds = region_a()
        rounds["rerun_after_cv"] = first_cv

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(abi.MOE_EV_COUNT)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        b = i % len(xs)
        layers[i % ncopy].forward_timed(xs[b], outs[b], evs[i])
    torch.cuda.synchronize()
    stage_names = ["route_align", "gate_up", "down", "combine"]
    stage_ms = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, n in enumerate(stage_names)}
    ms_timed = statistics.mean(e[0].elapsed_time(e[-1]) for e in evs)

    res = {"ms": ms, "launches": launches, "rounds": rounds, "stage_ms": stage_ms,
           "ms_timed": ms_timed, "alg": alg, "ncopy": ncopy, "w_bytes": w_bytes,
           "batches": len(xs)}
    if e2e:
        x_host = [x.cpu().pin_memory() for x in xs]
        out_host = [torch.empty((shape.T, shape.d), dtype=torch.bfloat16).pin_memory() for _ in xs]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall = time.perf_counter()
        e0.record()
        for i in range(steps):
            b = i % len(xs)
            xs[b].copy_(x_host[b], non_blocking=True)
            layers[i % ncopy].forward(xs[b], outs[b])
            out_host[b].copy_(outs[b], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res["t_wall"] = time.perf_counter() - t_wall
        res["ms_e2e"] = e0.elapsed_time(e1) / steps
    if clocks:
        res["clocks"] = clocks.stop()
    del layers, layer0, xs, outs
    torch.cuda.empty_cache()
    return res


def measure_chain(shape, args, dev, inp0, n_layers=16):
    """A decode step's MoE layers back to back: n_layers calls, each reading
    the previous call's output, captured once into a CUDA graph (programmatic
    dependent launch between every pair of kernels, inside and across layers)
    and replayed; layers alternate between weight copies so that HBM, not L2,
    serves the weights.  Each layer routes its own input (the previous
    layer's output), so the bytes are counted from every layer's own routing.
    Returns (per-layer microseconds: device time, events around the replays;
    the algorithmic bytes per layer averaged over the chain)."""
    import torch

    from moe_expert_layer_gemv_gb300 import inputs as I
    from moe_expert_layer_gemv_gb300.layer import MoeLayer

    copies = [MoeLayer(inp0, dev) for _ in range(2)]
    acts = [torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=dev)
            for _ in range(n_layers + 1)]
    ids = [torch.empty((shape.T, shape.k), dtype=torch.int32, device=dev)
           for _ in range(n_layers)]
    xs = [I.make_x(shape, seed=300 + b).to(dev) for b in range(4)]

    def chain():
        for i in range(n_layers):
            copies[i % 2].forward(acts[i], acts[i + 1], topk_ids=ids[i])

    acts[0].copy_(xs[0])
    chain()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for i in range(max(3, args.warmup)):
        acts[0].copy_(xs[i % 4])
        g.replay()
    torch.cuda.synchronize()
    reps = max(5, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        acts[0].copy_(xs[i % 4])
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_layers)
    layer_bytes = algorithmic(shape, [t.cpu().numpy() for t in ids])["layer_bytes"]
    del g, copies, acts, xs, ids
    torch.cuda.empty_cache()
    return us, layer_bytes


def roofline_of(shape, m, peaks, peak_kind):
    """Dominant kernel (the gate_up stage) against its roofline, and the layer
    figures, from one measure() result."""
    alg, ms = m["alg"], m["ms"]
    gu_ms = m["stage_ms"]["gate_up"]
    achieved = alg["gate_up_bytes"] / (gu_ms * 1e-3) / 1e9
    tc = tensor_core_path(shape)
    traffic = kernel_traffic("grouped_tc.cu" if tc else "expert_gemv.cu", shape.name,
                             alg["gate_up_bytes"])
    kname = ("grouped_tc_kernel<gate_up, N=256>" if tc else
             f"gate_up_kernel<{'int4' if shape.fmt == 'int4' else 'bf16'}>")
    roof = {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes": alg["gate_up_bytes"], "peak_source": peak_kind}
    if tc:
        gtf = gate_up_flops(shape) / (gu_ms * 1e-3) / 1e12
        roof["tensor"] = {
            "achieved": gtf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": gtf / peaks["bf16_tflops"],
            "note": "gate_up algorithmic flops (real rows) / stage time vs measured bf16 burst peak"}
    layer = {"layer_us": ms * 1e3,
             "layer_hbm_gbs": alg["layer_bytes"] / (ms * 1e-3) / 1e9,
             "layer_roofline_frac": alg["layer_bytes"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
             "layer_tflops": alg["flops"] / (ms * 1e-3) / 1e12,
             "touched_experts": alg["touched"],
             "stage_us": {k: v * 1e3 for k, v in m["stage_ms"].items()},
             "timed_pass_us": m["ms_timed"] * 1e3,
             "rounds": m["rounds"]}
    if tc:
        layer["layer_tensor_frac"] = layer["layer_tflops"] / peaks["bf16_tflops"]
    return roof, layer


def config_of(shape, world, m):
    return {"workload": shape.name, "T": shape.T, "d": shape.d, "E": shape.E, "top_k": shape.k,
            "I": shape.I, "I_shared": shape.Is, "weights": shape.fmt,
            **({"skew": "router rows of 16 hot experts x4"} if shape.skew else {}),
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": f"rotate {m['ncopy']} device copies of all weights "
                  f"({m['ncopy'] * m['w_bytes'] / 1e9:.2f} GB) and {m['batches']} token batches"}


def main():
    args = parse()
    from moe_expert_layer_gemv_gb300 import inputs as I

    shape = I.shape(args.workload)
    if args.impl == "reference":
        run_reference(args, shape)
        return

    import torch
    import torch.distributed as dist

    from moe_expert_layer_gemv_gb300 import abi, build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    abi.load()

    # CPU baseline first (before heavy GPU allocations), rank 0 only, N=1 only.
    cpu = None
    inp0 = I.make_inputs(shape, seed=0)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, threads, ntok, el = oracle_tokens_per_s(inp0, args.cpu_seconds, nthreads=host_cores())
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{ntok // shape.T} whole steps ({ntok} tokens) of the {shape.name} "
                         f"workload, {el:.1f} s, fp64 OpenMP over tokens"}
        ch = min(shape.T, 8)
        v1, _, ntok1, el1 = oracle_tokens_per_s(inp0, args.cpu_seconds / 5, nthreads=1, chunk=ch)
        cpu["one_thread"] = {"value": v1, "unit": UNIT, "cores": 1,
                             "sample": f"{ntok1} tokens of the same batch, {ch} per call, "
                                       f"{el1:.1f} s"}

    m = measure(shape, args, dev, world, local, inp0, e2e=True)
    chain = measure_chain(shape, args, dev, inp0) if shape.T <= 128 else None
    del inp0
    ms, ms_e2e = ranks_max([m["ms"], m["ms_e2e"]], dev)
    peaks, peak_kind = measured_peaks()
    m["ms"] = ms
    roof, layer = roofline_of(shape, m, peaks, peak_kind)

    # The other workloads: same protocol (regions A and B), each its own entry.
    others = {}
    if chain is not None:
        chain_us, chain_bytes = chain
        chain_us = ranks_max([chain_us], dev)[0]
        others[f"{shape.name}_chain16_graph"] = {
            "config": {**config_of(shape, world, m), "layers": 16,
                       "note": "16 chained layer calls (each reads the previous output), one "
                               "CUDA graph, two weight copies alternating; bytes from every "
                               "layer's own routing of its input"},
            "value": job_tokens_per_s(shape.T, world, chain_us * 1e-3), "unit": UNIT,
            "layer_us": chain_us, "layer_bytes": chain_bytes,
            "layer_hbm_gbs": chain_bytes / (chain_us * 1e-6) / 1e9,
            "layer_roofline_frac": chain_bytes / (chain_us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    for name in [w for w in args.also.split(",") if w not in ("", "none", shape.name)]:
        sh = I.shape(name)
        mo = measure(sh, args, dev, world, local, I.make_inputs(sh, seed=0), e2e=False)
        mo["ms"] = ranks_max([mo["ms"]], dev)[0]
        r2, l2 = roofline_of(sh, mo, peaks, peak_kind)
        others[name] = {"config": config_of(sh, world, mo), "value": job_tokens_per_s(sh.T, world, mo["ms"]),
                        "unit": UNIT, "ms_per_step": mo["ms"], "gpu_launches": mo["launches"],
                        **l2, "roofline": r2,
                        "dtype": "bf16" if sh.fmt == "bf16" else "int4g32+bf16"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": job_tokens_per_s(shape.T, world, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            # operands as stored (bf16, or int4 codes with bf16 group scales), fp32 accumulate
            "dtype": "bf16" if shape.fmt == "bf16" else "int4g32+bf16",
            "data": "synthetic",
            "config": config_of(shape, world, m),
            **layer,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": job_tokens_per_s(shape.T, world, ms_e2e), "unit": UNIT,
                    "h2d_bytes_per_step": shape.T * shape.d * 2,
                    "d2h_bytes_per_step": shape.T * shape.d * 2,
                    "wall_value": args.steps * world * shape.T / m["t_wall"]},
            "gpu_launches": m["launches"],
            "clocks": m["clocks"],
            "workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
