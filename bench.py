"""Benchmark: the 30-layer MoE decode stack (B=1, H=2048, I=768, E=128, top-2)
on one GB300, through the C ABI of libmoe.so.

Prints ONE JSON line (rank 0).  A step is one decode token through all 30
layers (router GEMV, softmax/top-k, grouping, grouped gate_up/SiLU*up, down
and combine, with the residual add), one fused persistent kernel launch.

  value     tokens/s of the whole job (sum over ranks / max-over-ranks time),
            inputs resident in HBM, L2 flushed (256 MiB memset) before every
            timed step, timed with CUDA events on the launching stream;
  e2e       the same metric through the public Python API with pinned HOST
            buffers: x copied in, the stack run, x copied out, each step;
  roofline  algorithmic bytes per launch (each layer's bf16 router plus each
            unique selected expert once) / mean launch time, against the
            measured HBM copy bandwidth;
  cpu_baseline  the CPU oracle on a bounded sample of the same workload;
  configs   sub-records measured in the same run for the other workloads
            (tiny layer, uniform-routing sweep B = 1..64, skewed-routing
            sweep B = 1..128, prefill-sized layer): ms, tokens/s, algorithmic
            bytes, GB/s and fraction of the peak, unique experts, reuse,
            near-tie tokens and kernel launches per step; and the dense
            counterpart of the stack (E=1, top-1, I=1536: the same active
            bytes per layer), with moe_over_dense_time beside the headline;
            and the stack as a pre-norm stack (RMSNorm fused).

--impl reference times the CPU oracle itself on this workload (rank 0 only).
--workload {uniform,skewed,prefill,tiny} times one layer of that workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and achieved HBM GB/s (unique-expert bytes) vs roofline"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="fused", choices=["fused", "unfused"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="bound on the oracle's CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=30,
                    help="layers in the stack (30 = the workload; fewer only for profiling captures)")
    ap.add_argument("--workload", default="stack",
                    choices=["stack", "uniform", "skewed", "prefill", "tiny", "dense"],
                    help="stack = the 30-layer decode stack (the headline); dense = its dense SwiGLU "
                         "counterpart (E=1, top-1, I=1536); the others time one layer")
    ap.add_argument("--batch", type=int, default=None, help="tokens per step for a single-layer workload")
    ap.add_argument("--experts", type=int, default=None,
                    help="experts of a single-layer workload (fewer only for scaled profiling captures)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the sub-records of the other workloads in the default run")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps per sub-record")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_throughput(local_ms, units_per_rank, pg=None, device="cpu"):
    """Whole-job throughput of N replicas: every rank processed
    `units_per_rank` units in `local_ms`; the job took the slowest rank's
    time.  Returns (max-over-ranks ms, units of all ranks per second)."""
    import torch
    world = 1
    if pg is not None:
        world = pg.get_world_size()
        t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        local_ms = float(t.item())
    return local_ms, units_per_rank * world / (local_ms / 1000.0)


def hbm_peak(path=None):
    """HBM roofline peak in GB/s: the measured copy bandwidth from
    MEASURED_PEAKS.json (a numeric entry whose key path names HBM and a
    bandwidth, the burst figure first: kernels here are timed per launch; a
    value below 100 is taken as TB/s), else the fallback."""
    p = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p)) if os.path.exists(p) else None
    except Exception:
        d = None
    found = []

    def walk(o, key_path):
        if isinstance(o, dict):
            for k, v in o.items():
                walk(v, key_path + "/" + str(k).lower())
        elif isinstance(o, (int, float)) and not isinstance(o, bool) and o > 0:
            found.append((key_path, float(o)))

    walk(d, "")
    unrelated = ("clock", "mhz", "freq", "mib", "size", "bytes", "count", "util", "pct", "frac")
    cands = [(k, v) for k, v in found if "hbm" in k and not any(u in k for u in unrelated)]
    if cands:
        cands.sort(key=lambda kv: ("burst" not in kv[0], "sustain" in kv[0], kv[0]))
        v = cands[0][1]
        return (v * 1000.0 if v < 100 else v), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_decode_layer_gemv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "moe.h"), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        rec = d.get(f"{kernel}@{workload}")
        if rec and rec.get("source_hash") == kernel_source_hash():
            return rec.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.2)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle
def oracle_stack_sample(layers_cpu_fn, x0_list, k, seconds, n_layers=30):
    """Run the CPU oracle on whole tokens through the stack (cycling through
    x0_list) until `seconds` of oracle time accumulate (at least one token).  layers_cpu_fn(l, ids)
    returns the layer's weights as the oracle takes them (host arrays),
    fetching only the experts in ids.  Returns (tokens, oracle_seconds)."""
    import numpy as np
    import oracle
    done, spent = 0, 0.0
    # cycle through the given tokens until the time is spent
    for i in range(100000):
        x = np.array(x0_list[i % len(x0_list)], dtype=np.float32, copy=True)
        for l in range(n_layers):
            wr, bias = layers_cpu_fn(l, None)
            t0 = time.perf_counter()
            lo = oracle.router(x, wr, bias)
            ids, w = oracle.topk(lo, k)
            spent += time.perf_counter() - t0
            gu, dn = layers_cpu_fn(l, ids)
            t0 = time.perf_counter()
            x = oracle.experts(x, gu, dn, ids, w, wr.shape[0], residual=x)
            spent += time.perf_counter() - t0
        done += 1
        if spent >= seconds:
            break
    return done, spent


def cpu_model():
    try:
        for ln in open("/proc/cpuinfo"):
            k = ln.split(":")[0].strip().lower()
            if k in ("model name", "cpu part", "hardware"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_threads()))
    import numpy as np
    import torch
    from moe_decode_layer_gemv_gb300 import accounting, synth
    w = synth.STACK
    cache = {}

    def layer_cpu(l, ids):
        key = ("r", l)
        if key not in cache:
            cache[key] = (synth.bf16_bits(synth.normal_bf16((w.E, w.H), w.sigma_router, args.seed,
                                                             10 + 3 * l, 0, "cpu")), None)
        if ids is None:
            return cache[key]
        gu, dn = {}, {}
        for e in np.unique(ids):
            e = int(e)
            kg = ("g", l, e)
            if kg not in cache:
                cache[kg] = (synth.bf16_bits(synth.normal_bf16((2 * w.I, w.H), w.sigma_expert, args.seed,
                                                                11 + 3 * l, e, "cpu")),
                             synth.bf16_bits(synth.normal_bf16((w.H, w.I), w.sigma_expert, args.seed,
                                                                12 + 3 * l, e, "cpu")))
            gu[e], dn[e] = cache[kg]
        return gu, dn

    xs = [synth.make_x(w, s, seed=args.seed, device="cpu").numpy() for s in range(args.warmup + args.steps)]
    per_step = max(1.0, args.cpu_seconds / max(args.steps, 1))
    for s in range(args.warmup):
        oracle_stack_sample(layer_cpu, [xs[s]], w.top_k, 0.0)
    total_tok, total_t = 0, 0.0
    for s in range(args.steps):
        n, t = oracle_stack_sample(layer_cpu, [xs[args.warmup + s]], w.top_k, per_step)
        total_tok += n
        total_t += t
    value = total_tok * w.B / total_t
    cores = int(os.environ.get("OMP_NUM_THREADS", cpu_threads()))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total_t / max(total_tok, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": w.name, "layers": w.layers, "B": w.B, "H": w.H,
                                         "I": w.I, "E": w.E, "top_k": w.top_k},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"{total_tok} whole tokens through all 30 layers (CPU-drawn weights)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ single layer
def near_tie_count(api, xs, lw, k, stream):
    """Tokens whose k-th and (k+1)-th router logits are within 1e-5 (the
    near ties the parity rules exempt), over the given inputs; None when
    k == E.  Statistics only, computed outside any timed region."""
    import torch
    E = lw["w_router"].shape[0]
    if k >= E:
        return None
    n = 0
    for x in xs:
        _, _, lg = api.route(x, lw["w_router"], k, bias=lw.get("bias"), stream=stream)
        srt = torch.sort(lg, dim=1, descending=True).values
        n += int(((srt[:, k - 1] - srt[:, k]) < 1e-5).sum())
    return n


def step_statuses(api, status, what):
    """Per-step device status words (one int32 per call): any bit other than
    the value-dependent ones ends the run; a non-finite or out-of-range router
    value -- the no-norm 30-layer stack's residual stream overflows for some
    inputs, see the design notes -- is counted and reported instead.
    Returns the number of steps that saw one."""
    value_bits = api.MOE_DEV_NONFINITE | api.MOE_DEV_RANGE
    sts = [int(v) for v in status[:, 0].cpu().tolist()]
    for v in sts:
        if v & ~value_bits:
            raise SystemExit(f"{what}: device status {v}: {api.status_string(v & ~value_bits)}")
    return sum(1 for v in sts if v)


def measure_layer(api, accounting, synth, w, dev, steps, warmup, flags=0, seed=0, flush=None, lw=None):
    """One MoE layer per step on fresh inputs, L2 flushed before each timed
    step, CUDA events on the launching stream.  Returns the sub-record."""
    import numpy as np
    import torch
    lw = lw if lw is not None else synth.make_layer(w, 0, seed=seed, device=dev)
    nsteps = warmup + steps
    xs = [synth.make_x(w, s, seed=seed, device=dev) for s in range(nsteps)]
    y = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    ids = torch.empty((w.B, w.top_k), dtype=torch.int32, device=dev)
    rw = torch.empty((w.B, w.top_k), dtype=torch.float32, device=dev)
    ws = api.new_workspace(w.B, w.H, w.I, w.E, w.top_k, dev)
    status = api.new_status(dev)
    flush = flush if flush is not None else torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        api.layer_forward(xs[i], lw["w_router"], lw["gate_up"], lw["down"], w.top_k, bias=lw["bias"],
                          flags=flags, out=y, ids_out=ids, w_out=rw, workspace=ws, status=status,
                          stream=stream)

    for i in range(warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    uniq = []
    launches = 0
    for s in range(steps):
        flush.zero_()
        n0 = api.launch_count()
        ev[s][0].record(stream)
        step(warmup + s)
        ev[s][1].record(stream)
        launches += api.launch_count() - n0
        uniq.append(ids.clone())
    torch.cuda.synchronize()
    st = int(status.item())
    if st != 0:
        raise SystemExit(f"{w.name} B={w.B}: device status {st}: {api.status_string(st)}")
    times_ms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = statistics.mean(times_ms)
    us = [len(np.unique(u.cpu().numpy())) for u in uniq]
    bytes_step = statistics.mean(accounting.layer_bytes(w.H, w.I, w.E, u) for u in us)
    achieved = bytes_step / (mean_ms / 1e3) / 1e9
    peak, _ = hbm_peak()
    try:
        ties = near_tie_count(api, xs[warmup:], lw, w.top_k, stream)
    except Exception as exc:  # statistics only: never fail the timing
        print(f"near-tie count skipped: {exc}", file=sys.stderr)
        ties = None
    return {"workload": w.name, "B": w.B, "H": w.H, "I": w.I, "E": w.E, "top_k": w.top_k,
            "ms": mean_ms, "tokens_per_s": w.B / (mean_ms / 1e3), "bytes_per_step": bytes_step,
            "hbm_gbs": achieved, "frac": achieved / peak, "unique_experts": statistics.mean(us),
            "reuse": statistics.mean(w.B * w.top_k / u for u in us), "near_tie_tokens": ties,
            "launches_per_step": launches / steps, "steps": steps}


def run_layer_workload(args):
    """One MoE layer per step (uniform / skewed / prefill-sized / tiny), or
    the dense stack."""
    rank, world, local = dist_env()
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from moe_decode_layer_gemv_gb300 import accounting, build, synth
    build.build()
    from moe_decode_layer_gemv_gb300 import api
    if args.workload == "dense":
        flags = api.MOE_F_UNFUSED if args.mode == "unfused" else 0
        with ClockSampler(local) as clk:
            rec = measure_stack(api, accounting, synth, synth.DENSE, dev, args.steps, args.warmup, flags, args.seed)
        peak, peak_src = hbm_peak()
        w = synth.DENSE
        line = {"metric": METRIC, "value": rec["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "weights_dtype": "bf16",
                "data": "synthetic", "mode": args.mode, "l2_flush": "256 MiB memset before every timed step",
                "config": {"workload": w.name, "layers": w.layers, "B": w.B, "H": w.H, "I": w.I, "E": w.E,
                           "top_k": w.top_k},
                "us_per_layer": rec["us_per_layer"], "hbm_gbs": rec["hbm_gbs"],
                "roofline": {"bound": "hbm", "achieved": rec["hbm_gbs"], "peak": peak, "unit": "GB/s",
                             "frac": rec["frac"], "peak_source": peak_src, "traffic": None,
                             "bytes_per_launch": rec["bytes_per_step"]},
                "gpu_launches": int(round(rec["launches_per_step"] * args.steps)), "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
        return
    base = {"uniform": synth.UNIFORM, "skewed": synth.SKEWED, "prefill": synth.PREFILL,
            "tiny": synth.TINY}[args.workload]
    w = base.with_batch(args.batch) if args.batch else base
    if args.experts:
        import dataclasses
        w = dataclasses.replace(w, E=args.experts, name=f"{w.name}_e{args.experts}")
    flags = api.MOE_F_UNFUSED if args.mode == "unfused" else 0
    with ClockSampler(local) as clk:
        rec = measure_layer(api, accounting, synth, w, dev, args.steps, args.warmup, flags, args.seed)
    peak, peak_src = hbm_peak()
    line = {"metric": METRIC, "value": rec["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "weights_dtype": "bf16",
            "data": "synthetic", "mode": args.mode, "l2_flush": "256 MiB memset before every timed step",
            "config": {"workload": w.name, "layers": 1, "B": w.B, "H": w.H, "I": w.I, "E": w.E,
                       "top_k": w.top_k},
            "unique_experts_mean": rec["unique_experts"], "reuse_mean": rec["reuse"],
            "near_tie_tokens": rec["near_tie_tokens"], "hbm_gbs": rec["hbm_gbs"],
            "roofline": {"bound": "hbm", "achieved": rec["hbm_gbs"], "peak": peak, "unit": "GB/s",
                         "frac": rec["frac"], "peak_source": peak_src, "traffic": None,
                         "bytes_per_launch": rec["bytes_per_step"]},
            "gpu_launches": int(round(rec["launches_per_step"] * args.steps)),
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def measure_stack(api, accounting, synth, w, dev, steps, warmup, flags=0, seed=0, flush=None, norm=False,
                  fp8=False, nvfp4=False, layers=None):
    """One token through an L-layer stack per step (L2 flushed before each
    timed step, CUDA events on the launching stream); norm=True makes it a
    pre-norm stack (RMSNorm fused into the router and residual add), fp8=True
    gives it block-scaled FP8 expert weights, nvfp4=True NVFP4 ones.
    Returns the sub-record."""
    import numpy as np
    import torch
    if nvfp4:
        if layers is None:
            layers = [synth.make_layer_nvfp4(w, l, seed=seed, device=dev) for l in range(w.layers)]
        for lw in layers:  # only the codes and scales stay resident
            lw.pop("gate_up", None)
            lw.pop("down", None)
        sw = api.StackWeightsNVFP4(layers)
        fwd = lambda xb, **kw: api.stack_forward_nvfp4_(xb, sw, w.top_k, **kw)
        lbytes = accounting.layer_bytes_nvfp4
    elif fp8:
        if layers is None:
            layers = [synth.make_layer_fp8(w, l, seed=seed, device=dev) for l in range(w.layers)]
        for lw in layers:  # only the codes and scales stay resident
            lw.pop("gate_up", None)
            lw.pop("down", None)
        sw = api.StackWeightsFP8(layers)
        fwd = lambda xb, **kw: api.stack_forward_fp8_(xb, sw, w.top_k, **kw)
        lbytes = accounting.layer_bytes_fp8
    else:
        layers = [synth.make_layer(w, l, seed=seed, device=dev) for l in range(w.layers)]
        if norm:
            for l, lw in enumerate(layers):
                lw["norm"] = synth.norm_weights(w.H, l, seed=seed, device=dev)
        sw = api.StackWeights(layers)
        fwd = ((lambda xb, **kw: api.stack_forward_norm_(xb, sw, w.top_k, eps=1e-6, **kw)) if norm else
               (lambda xb, **kw: api.stack_forward_(xb, sw, w.top_k, **kw)))
        lbytes = accounting.layer_bytes
    xs = [synth.make_x(w, s, seed=seed, device=dev) for s in range(warmup + steps)]
    xbuf = torch.empty_like(xs[0])
    ids = torch.empty((w.layers, w.B, w.top_k), dtype=torch.int32, device=dev)
    ws = api.new_workspace(w.B, w.H, w.I, w.E, w.top_k, dev)
    status = torch.zeros((warmup + steps, 4), dtype=torch.int32, device=dev)  # one 16-byte-aligned word per call
    st_of = [status[i, :1] for i in range(warmup + steps)]
    flush = flush if flush is not None else torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        flush.zero_()
        xbuf.copy_(xs[i])
        fwd(xbuf, flags=flags, ids_out=ids, workspace=ws, status=st_of[i], stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    uniq, launches = [], 0
    for s in range(steps):
        flush.zero_()
        xbuf.copy_(xs[warmup + s])
        n0 = api.launch_count()
        ev[s][0].record(stream)
        fwd(xbuf, flags=flags, ids_out=ids, workspace=ws, status=st_of[warmup + s], stream=stream)
        ev[s][1].record(stream)
        launches += api.launch_count() - n0
        uniq.append(ids.clone())
    torch.cuda.synchronize()
    value_flag_steps = step_statuses(api, status[warmup:], w.name)
    mean_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    u_layers = [len(np.unique(u.cpu().numpy()[l])) for u in uniq for l in range(w.layers)]
    bytes_step = statistics.mean(
        sum(lbytes(w.H, w.I, w.E, len(np.unique(u.cpu().numpy()[l]))) for l in range(w.layers))
        for u in uniq)
    achieved = bytes_step / (mean_ms / 1e3) / 1e9
    peak, _ = hbm_peak()
    del layers, sw
    torch.cuda.empty_cache()
    return {"workload": w.name + ("_rmsnorm" if norm else "") + ("_fp8_block128" if fp8 else "")
            + ("_nvfp4" if nvfp4 else ""), "B": w.B, "H": w.H, "I": w.I, "E": w.E,
            "top_k": w.top_k, "layers": w.layers,
            "ms": mean_ms, "tokens_per_s": w.B / (mean_ms / 1e3), "us_per_layer": 1000.0 * mean_ms / w.layers,
            "bytes_per_step": bytes_step, "hbm_gbs": achieved, "frac": achieved / peak,
            "unique_experts": statistics.mean(u_layers), "launches_per_step": launches / steps, "steps": steps,
            "value_flag_steps": value_flag_steps}


def config_records(api, accounting, synth, dev, steps, warmup, seed=0):
    """Sub-records for every workload besides the stack: the tiny layer, the
    uniform-routing sweep, the skewed-routing sweep and the prefill-sized
    layer (one layer per step each, measured in this run)."""
    import torch
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {}
    out["tiny"] = measure_layer(api, accounting, synth, synth.TINY, dev, steps, warmup, 0, seed, flush)
    for base in (synth.UNIFORM, synth.SKEWED):
        lw = synth.make_layer(base, 0, seed=seed, device=dev)
        for B in base.batches:
            key = f"{'uniform' if base is synth.UNIFORM else 'skewed'}_B{B}"
            out[key] = measure_layer(api, accounting, synth, base.with_batch(B), dev, steps, warmup, 0, seed,
                                     flush, lw=lw)
            if B > 4:
                # the split dispatch: only the experts with >= 8 routes on the
                # tensor cores, the rest on the CUDA-core streaming GEMV
                out[key + "_split_tc"] = measure_layer(api, accounting, synth, base.with_batch(B), dev, steps,
                                                       warmup, api.MOE_F_SPLIT_TC, seed, flush, lw=lw)
            if base is synth.SKEWED and B > 4:
                # the step's most chosen experts kept in L2 across steps (an L2
                # policy on the weight copies; the same flush between steps)
                out[key + "_hot_l2"] = measure_layer(api, accounting, synth, base.with_batch(B), dev, steps, warmup,
                                                     api.MOE_F_HOT_L2, seed, flush, lw=lw)
        del lw
        torch.cuda.empty_cache()
    out["prefill"] = measure_layer(api, accounting, synth, synth.PREFILL, dev, steps, warmup, 0, seed, flush)
    torch.cuda.empty_cache()
    # the dense counterpart of the stack (one expert, top-1, same active bytes
    # per layer): the dense-vs-MoE comparison of the first page
    out["dense_stack"] = measure_stack(api, accounting, synth, synth.DENSE, dev, steps, warmup, 0, seed, flush)
    # the stack as a pre-norm stack: RMSNorm fused into the router and residual add
    out["stack_rmsnorm"] = measure_stack(api, accounting, synth, synth.STACK, dev, steps, warmup, 0, seed, flush,
                                         norm=True)
    # the stack with block-scaled FP8 experts (E4M3 codes, fp32 scale per 128x128 block)
    out["stack_fp8"] = measure_stack(api, accounting, synth, synth.STACK, dev, steps, warmup, 0, seed, flush,
                                     fp8=True)
    # the stack with NVFP4 experts (E2M1 codes, E4M3 scale per 16 weights, fp32 per matrix)
    out["stack_nvfp4"] = measure_stack(api, accounting, synth, synth.STACK, dev, steps, warmup, 0, seed, flush,
                                       nvfp4=True)
    # one layer of the uniform-routing workload with FP8 experts over the batch
    # sweep (decode kernel up to B=4, the CUDA-core phase kernels beyond), then
    # the same with NVFP4 experts
    base = synth.UNIFORM
    fp8_layer = [synth.make_layer_fp8(base, 0, seed=seed, device=dev)]
    for B in base.batches:
        out[f"uniform_B{B}_fp8"] = measure_stack(api, accounting, synth, base.with_batch(B), dev, steps, warmup, 0,
                                                 seed, flush, fp8=True, layers=fp8_layer)
    del fp8_layer
    torch.cuda.empty_cache()
    # and with NVFP4 experts
    nvfp4_layer = [synth.make_layer_nvfp4(base, 0, seed=seed, device=dev)]
    for B in base.batches:
        out[f"uniform_B{B}_nvfp4"] = measure_stack(api, accounting, synth, base.with_batch(B), dev, steps, warmup, 0,
                                                   seed, flush, nvfp4=True, layers=nvfp4_layer)
    del nvfp4_layer
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------------- ours
def stack_near_ties(api, sw, layers, x0, k, stream):
    """Near ties along one token's path through the stack (layer by layer,
    outside the timed region): tokens x layers whose k-th and (k+1)-th logits
    are within 1e-5."""
    import torch
    x = x0.clone()
    n = 0
    for lw in layers:
        n += near_tie_count(api, [x], lw, k, stream) or 0
        y, _, _ = api.layer_forward(x, lw["w_router"], lw["gate_up"], lw["down"], k, bias=lw.get("bias"),
                                    residual=x, stream=stream)
        x = y
    torch.cuda.synchronize()
    return n


def run_ours(args):
    rank, world, local = dist_env()
    import numpy as np
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    from moe_decode_layer_gemv_gb300 import accounting, build, synth
    build.build()
    from moe_decode_layer_gemv_gb300 import api
    w = synth.STACK
    if args.layers != w.layers:
        w = synth.Workload(f"stack{args.layers}_b1_h2048_i768_e128_k2", B=w.B, H=w.H, I=w.I, E=w.E,
                           top_k=w.top_k, layers=args.layers, residual=True)
    flags = api.MOE_F_UNFUSED if args.mode == "unfused" else 0
    layers = [synth.make_layer(w, l, seed=args.seed + 7919 * rank, device=dev) for l in range(w.layers)]
    sw = api.StackWeights(layers)
    nsteps = args.warmup + args.steps
    xs = [synth.make_x(w, s, seed=args.seed + 7919 * rank, device=dev) for s in range(nsteps)]
    xbuf = torch.empty_like(xs[0])
    ids = torch.empty((w.layers, w.B, w.top_k), dtype=torch.int32, device=dev)
    ws = api.new_workspace(w.B, w.H, w.I, w.E, w.top_k, dev)
    status = torch.zeros((nsteps, 4), dtype=torch.int32, device=dev)  # one 16-byte-aligned word per call
    st_of = [status[i, :1] for i in range(nsteps)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        xbuf.copy_(xs[i])
        api.stack_forward_(xbuf, sw, w.top_k, flags=flags, ids_out=ids, workspace=ws, status=st_of[i],
                           stream=stream)

    for i in range(args.warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    uniq = []
    launches = 0
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.nvtx.range_push("timed")
        for s in range(args.steps):
            i = args.warmup + s
            flush.zero_()
            xbuf.copy_(xs[i])
            n0 = api.launch_count()
            ev[s][0].record(stream)
            api.stack_forward_(xbuf, sw, w.top_k, flags=flags, ids_out=ids, workspace=ws, status=st_of[i],
                               stream=stream)
            ev[s][1].record(stream)
            launches += api.launch_count() - n0
            uniq.append(ids.clone())
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
    times_ms = [a.elapsed_time(b) for a, b in ev]
    value_flag_steps = step_statuses(api, status[args.warmup:], w.name)
    total_ms, value = job_throughput(sum(times_ms), w.B * args.steps, pg, dev)
    # algorithmic bytes: per layer the router + each unique selected expert once
    bytes_steps, u_layers = [], []
    for u in uniq:
        un = u.cpu().numpy()
        ul = [len(np.unique(un[l])) for l in range(w.layers)]
        u_layers += ul
        bytes_steps.append(sum(accounting.layer_bytes(w.H, w.I, w.E, n) for n in ul))
    bytes_per_launch = statistics.mean(bytes_steps)
    mean_ms = statistics.mean(times_ms)
    achieved = bytes_per_launch / (mean_ms / 1000.0) / 1e9
    peak, peak_src = hbm_peak()
    clocks = clk.summary()
    ties = None
    if rank == 0:
        try:
            ties = sum(stack_near_ties(api, sw, layers, xs[args.warmup + s], w.top_k, stream)
                       for s in range(min(args.steps, 5)))
        except Exception as exc:  # statistics only
            print(f"near-tie count skipped: {exc}", file=sys.stderr)

    # ---- e2e: public API, pinned host buffers, copies inside the timed
    # region; no L2 flush (a user's call has none, and every step reads
    # 582 MB of weights, over four times the 129 MB L2)
    e2e = None
    if not args.no_e2e:
        xh = [xs[args.warmup + s].cpu().pin_memory() for s in range(args.steps)]
        e2e_status = torch.zeros((args.steps, 4), dtype=torch.int32, device=dev)
        e2e_st = [e2e_status[s, :1] for s in range(args.steps)]
        out_h = torch.empty_like(xh[0]).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(args.steps):
            xbuf.copy_(xh[s], non_blocking=True)
            api.stack_forward_(xbuf, sw, w.top_k, flags=flags, ids_out=ids, workspace=ws,
                               status=e2e_st[s], stream=stream)
            out_h.copy_(xbuf, non_blocking=True)
            stream.synchronize()
        e2e_s = time.perf_counter() - t0
        step_statuses(api, e2e_status, w.name + " (e2e)")
        nbytes = xh[0].numel() * 4
        e2e = {"value": w.B * args.steps * world / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "l2_flush": "none (per-step weights exceed L2)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "weights_dtype": "bf16", "data": "synthetic",
        "mode": args.mode, "l2_flush": "256 MiB memset before every timed step, outside the events",
        "config": {"workload": w.name, "layers": w.layers, "B": w.B, "H": w.H, "I": w.I, "E": w.E,
                   "top_k": w.top_k},
        "hbm_gbs": achieved,
        "us_per_layer": 1000.0 * mean_ms / w.layers,
        "unique_experts_per_layer": statistics.mean(u_layers),
        "reuse": w.B * w.top_k / statistics.mean(u_layers),
        "near_tie_token_layers": ties,
        # timed steps whose token overflowed the no-norm stack (non-finite or
        # out-of-range router values; the work done is the same)
        "value_flag_steps": value_flag_steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": recorded_traffic("moe_stack_fused", w.name),
                     "kernel": "decode_kernel (one launch = 30 layers)",
                     "bytes_per_launch": bytes_per_launch},
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        os.environ.setdefault("OMP_NUM_THREADS", str(cpu_threads()))
        cache = {}

        def layer_cpu(l, ids_np):
            lw = layers[l]
            if ("r", l) not in cache:
                cache[("r", l)] = (synth.bf16_bits(lw["w_router"]), None)
            if ids_np is None:
                return cache[("r", l)]
            gu, dn = {}, {}
            for e in np.unique(ids_np):
                e = int(e)
                if ("g", l, e) not in cache:
                    cache[("g", l, e)] = (synth.bf16_bits(lw["gate_up"][e]), synth.bf16_bits(lw["down"][e]))
                gu[e], dn[e] = cache[("g", l, e)]
            return gu, dn

        x_np = [xs[args.warmup + s].cpu().numpy() for s in range(args.steps)]
        n, t = oracle_stack_sample(layer_cpu, x_np, w.top_k, args.cpu_seconds, w.layers)
        line["cpu_baseline"] = {"value": n * w.B / t, "unit": "tokens/s",
                                "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": f"{n} whole tokens through all {w.layers} layers (same weights, "
                                          f"{t:.1f} s of oracle time)"}
    if rank == 0 and not args.no_configs and world == 1:
        del layers, sw
        torch.cuda.empty_cache()
        line["configs"] = config_records(api, accounting, synth, dev, args.config_steps, 3, args.seed)
        dense = line["configs"].get("dense_stack")
        if dense:  # per-token time of the MoE stack over its dense counterpart (same active bytes)
            line["moe_over_dense_time"] = mean_ms / dense["ms"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "stack":
        run_layer_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
