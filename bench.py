#!/usr/bin/env python3
"""Benchmark: causal attention forward + backward on GB300 through the C ABI.

One step = one pass of the whole path over one batch: rca_attn_fwd, then the
three backward stages (preprocess, main, dQ convert). Workload: B=4, H=16,
T=2048, Dh=64, bf16 operands with fp32 accumulation (override with --workload).

Prints ONE JSON line (rank 0). FLOP convention (algorithmic, causal half):
forward = 4*B*Hq*T^2*Dh/2, backward = 2.5 x forward (five GEMM-shaped products
including the recompute of P); a step counts 3.5 x forward.

Under torchrun each rank runs its own independent batch of (batch, head) units
(no data exchange): weak scaling, value = all ranks' FLOPs / max rank time.
`--impl reference` times the fp64 CPU oracle instead (rank 0 only).
"""

from __future__ import annotations

import os

# The CPU oracle legs run one BLAS thread per worker thread; set before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import concurrent.futures as cf
import hashlib
import json
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from causal_head_attention_gb300.inputs import (  # noqa: E402
    BY_NAME,
    DEC_GQA,
    DEC_MHA,
    HEADLINE,
    make_inputs,
    make_paged_inputs,
)

L2_BYTES = 129 * 1024 * 1024


def fwd_flops(w) -> float:
    return 4.0 * w.B * w.Hq * w.T * w.T * w.Dh / 2.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# Source files each profiled kernel is built from (its device code, the shared
# device helpers and its host launcher).
KERNEL_SOURCES = {
    "fwd": ("fwd.cuh", "tc.cuh", "rca_attn.cu"),
    "bwd_main": ("bwd.cuh", "bwd_sub.cuh", "tc.cuh", "rca_attn.cu"),
    "bwd_preprocess": ("bwd.cuh", "tc.cuh", "rca_attn.cu"),
    "bwd_dq_convert": ("bwd.cuh", "tc.cuh", "rca_attn.cu"),
    "decode": ("decode.cu", "decode.h", "tc.cuh"),
}


def src_digest(kernel: str | None = None) -> str:
    """Digest of the kernel sources (all of csrc/, or those `kernel` is built from)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_head_attention_gb300", "csrc")
    names = sorted(os.listdir(csrc)) if kernel is None else sorted(KERNEL_SOURCES[kernel])
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("src_digest") != src_digest(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.out = None

    def start(self):
        try:
            self.out = open(f"/tmp/rca_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def rank_workload(w, rank: int):
    """This rank's batch: same shapes, its own seed, so ranks process distinct
    (batch, head) units with nothing to exchange (weak scaling)."""
    from dataclasses import replace

    return w if rank == 0 else replace(w, seed=w.seed + 1000 * rank)


def aggregate_tflops(step_flops: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return step_flops * world / (ms_per_step_max * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample(w, budget_s: float, max_groups: int | None = None):
    """Run the fp64 oracle (fwd + bwd) on whole (batch, KV-head) groups of the
    workload, one worker thread per host core, until budget_s has elapsed.
    Returns (causal FLOPs done, seconds, threads, groups)."""
    import oracle

    threads = len(os.sched_getaffinity(0))
    q, k, v, do = make_inputs(w)
    q64, k64, v64, do64 = (x.double().numpy() for x in (q, k, v, do))
    groups = [(b, kv) for b in range(w.B) for kv in range(w.Hkv)]
    if max_groups is not None:
        groups = groups[:max_groups]
    per_group = 3.5 * 4.0 * w.group * w.T * w.T * w.Dh / 2.0
    done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        it = iter(groups)
        futs = set()
        for _ in range(threads):
            g = next(it, None)
            if g is not None:
                futs.add(ex.submit(oracle.group_reference, q64, k64, v64, do64, g[0], g[1]))
        while futs:
            fin, futs = cf.wait(futs, return_when=cf.FIRST_COMPLETED)
            done += len(fin)
            if time.perf_counter() - t0 < budget_s:
                for _ in fin:
                    g = next(it, None)
                    if g is not None:
                        futs.add(ex.submit(oracle.group_reference, q64, k64, v64, do64, g[0], g[1]))
    dt = time.perf_counter() - t0
    return done * per_group, dt, threads, done


def input_sets(w) -> tuple[int, int]:
    """(number of rotating input copies, bytes of one copy): enough distinct
    copies of a step's inputs that together they exceed twice the L2 size."""
    es = 2 if w.dtype == "bf16" else 4
    set_bytes = es * w.B * w.T * w.Dh * (2 * w.Hq + 2 * w.Hkv)
    return max(2, -(-2 * L2_BYTES // set_bytes) + 1), set_bytes


def config_for(w, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    nsets, set_bytes = input_sets(w)
    return {"workload": w.describe(), "name": w.name, "global_batch": w.B * world, "seq_len": w.T,
            "heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.Dh, "parallelism": f"independent units x{world}",
            "l2": f"GPU arm: {nsets} rotating input sets ({nsets * set_bytes / 2**20:.0f} MiB) > L2",
            "flop_convention": "fwd 4*B*H*T^2*Dh/2; bwd 2.5x fwd; step 3.5x fwd"}


def launches_per_step(w) -> int:
    """Kernels this library launches per training step: forward, preprocess,
    backward main, dQ conversion; fp32 storage adds the four bf16 hi/lo splits
    of Q, dO, K and V."""
    return 4 if w.dtype == "bf16" else 8


def nominal_tflops(sms: int, sm_mhz: float, dtype: str) -> float:
    """Nominal dense tensor peak at the sampled SM clock: SMs x 8192 bf16
    FLOP per clock per SM (one M=128 N=256 K=16 tcgen05 MMA per 128 cycles),
    half that for TF32 operands."""
    per_clk = 8192.0 if dtype == "bf16" else 4096.0
    return sms * per_clk * sm_mhz * 1e6 / 1e12


def spread(xs) -> dict:
    """Mean, median, 10th and 90th percentile of a list of per-step times (ms)."""
    s = sorted(xs)
    n = len(s)

    def pct(p):
        i = (n - 1) * p
        lo, hi = int(i), min(int(i) + 1, n - 1)
        return s[lo] + (s[hi] - s[lo]) * (i - lo)

    return {"mean": sum(s) / n, "median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9)}


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    steps = []
    flops_step = None
    threads = len(os.sched_getaffinity(0))
    for s in range(args.warmup + args.steps):
        fl, dt, threads, n = oracle_sample(w, 0.0, max_groups=threads)
        if s >= args.warmup:
            steps.append(dt)
            flops_step = fl
            n_groups = n
    t = sum(steps)
    value = flops_step * len(steps) / t / 1e12
    line = {
        "impl": "reference", "metric": args.metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_for(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_groups} of {w.B * w.Hkv} (batch, KV-head) groups per step, fwd+bwd, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, w, world, rank, local):
    import causal_head_attention_gb300 as rca

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    P = peaks()

    q0, k0, v0, do0 = make_inputs(rank_workload(w, rank))
    nsets, set_bytes = input_sets(w)
    assert set_bytes == sum(x.numel() * x.element_size() for x in (q0, k0, v0, do0))
    # Distinct copies of the same inputs, so each step reads memory the previous
    # steps evicted from L2.
    base = tuple(x.to(dev) for x in (q0, k0, v0, do0))
    sets = [base] + [tuple(x.clone() for x in base) for _ in range(nsets - 1)]
    out = torch.empty_like(sets[0][0])
    lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=dev)
    dq = torch.empty_like(sets[0][0])
    dk = torch.empty_like(sets[0][1])
    dv = torch.empty_like(sets[0][2])
    ws = rca.workspace_for(sets[0][0], sets[0][1])

    def step(i, ev=None):
        q, k, v, do = sets[i % nsets]
        if ev is not None:
            ev[0].record(stream)
        rca.rca_attn_fwd(q, k, v, out, lse, stream)
        if ev is not None:
            ev[1].record(stream)
        rca.rca_attn_bwd_preprocess(out, lse, do, ws, Hkv=w.Hkv, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        rca.rca_attn_bwd_main(q, k, v, do, dk, dv, ws, stream)
        if ev is not None:
            ev[3].record(stream)
        rca.rca_attn_bwd_dq_convert(dq, ws, Hkv=w.Hkv, stream=stream)
        if ev is not None:
            ev[4].record(stream)

    # Warm-up: exactly W untimed steps. The clock sampler runs from here to the
    # end of a >= 1 s run of the same step right after the timed region, so its
    # samples (100 ms apart) cover the GPU under this load, the timed steps
    # included.
    clk = ClockSampler(local)
    clk.start()
    for i in range(args.warmup):
        step(i)
    n_warm = args.warmup
    rca.rca_stream_status(stream)

    # Timed region: exactly K steps with nothing between the launches, so each
    # kernel's launch overlaps the tail of the one before (the library launches
    # them with programmatic dependent launch; an event recorded between two
    # kernels would serialise them again).
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(n_warm + i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    # Per-kernel durations: the same K steps once more, with an event between
    # every two launches on the launching stream. These intervals include each
    # kernel's full launch gap (events take away the overlap), so they are
    # upper bounds on the kernels' own durations.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(n_warm + args.steps + i, evs[i])
    torch.cuda.synchronize(dev)
    # The same step again, untimed, for at least min_warmup_s: clock samples
    # under load (the timed steps alone last only milliseconds).
    t_c = time.perf_counter()
    n_clock = 0
    while time.perf_counter() - t_c < args.min_warmup_s:
        step(n_warm + 2 * args.steps + n_clock)
        n_clock += 1
        if n_clock % 64 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = clk.stop()
    if clocks is not None:
        clocks["window"] = (f"{args.warmup} warm-up + {args.steps} timed steps + {args.steps} steps with "
                            f"per-kernel events + {n_clock} more steps "
                            f"({time.perf_counter() - t_c:.1f} s) after the timed region")
    rca.rca_stream_status(stream)
    total_ms = t_start.elapsed_time(t_end)
    per = {"fwd": [], "bwd_preprocess": [], "bwd_main": [], "bwd_dq_convert": []}
    names = list(per)
    for e in evs:
        for j, n in enumerate(names):
            per[n].append(e[j].elapsed_time(e[j + 1]))
    avg = {n: sum(v) / len(v) for n, v in per.items()}
    step_spread = spread([e[0].elapsed_time(e[4]) for e in evs])
    step_spread["pass"] = "per-kernel pass (an event between every two launches)"

    ms = max_over_ranks(total_ms, world) / args.steps
    F = fwd_flops(w)
    step_flops = 3.5 * F
    value = aggregate_tflops(step_flops, world, ms)

    es = 2 if w.dtype == "bf16" else 4
    n_q = w.B * w.T * w.Hq * w.Dh
    n_kv = w.B * w.T * w.Hkv * w.Dh
    Tpad = -(-w.T // 128) * 128
    pre_bytes = 2 * n_q * es + 4 * w.B * w.Hq * w.T + 8 * w.B * w.Hq * Tpad + 4 * n_q
    cvt_bytes = 4 * n_q + es * n_q
    peak_tc = P["bf16_tflops"] if w.dtype == "bf16" else P["bf16_tflops"] / 2.0
    kern = {
        "fwd": {"bound": "tensor", "flops": F, "ms": avg["fwd"]},
        "bwd_main": {"bound": "tensor", "flops": 2.5 * F, "ms": avg["bwd_main"]},
        "bwd_preprocess": {"bound": "hbm", "bytes": pre_bytes, "ms": avg["bwd_preprocess"]},
        "bwd_dq_convert": {"bound": "hbm", "bytes": cvt_bytes, "ms": avg["bwd_dq_convert"]},
    }
    for n, d in kern.items():
        if d["bound"] == "tensor":
            d["achieved"] = d["flops"] / (d["ms"] * 1e-3) / 1e12
            d["unit"] = "TFLOP/s"
            d["frac"] = d["achieved"] / peak_tc
        else:
            d["achieved"] = d["bytes"] / (d["ms"] * 1e-3) / 1e9
            d["unit"] = "GB/s"
            d["frac"] = d["achieved"] / P["hbm_gbs"]
        d["share"] = d["ms"] / sum(avg.values())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    peak_nom = nominal_tflops(sms, clk_mhz, w.dtype)
    for d in kern.values():
        if d["bound"] == "tensor":
            d["frac_of_nominal"] = d["achieved"] / peak_nom
    bwd_ms = avg["bwd_preprocess"] + avg["bwd_main"] + avg["bwd_dq_convert"]
    bwd_tflops = 2.5 * F / (bwd_ms * 1e-3) / 1e12
    fracs = {
        "fwd_frac_of_peak": kern["fwd"]["frac"],
        "bwd_frac_of_peak": bwd_tflops / peak_tc,
        "fwd_frac_of_nominal": kern["fwd"]["achieved"] / peak_nom,
        "bwd_frac_of_nominal": bwd_tflops / peak_nom,
    }
    dom = max(kern, key=lambda n: kern[n]["ms"])
    dk_ = kern[dom]
    roofline = {
        "kernel": dom, "bound": dk_["bound"], "achieved": dk_["achieved"],
        "peak": peak_tc if dk_["bound"] == "tensor" else P["hbm_gbs"], "unit": dk_["unit"],
        "frac": dk_["frac"], "traffic": ncu_traffic(dom, w.name),
        "peak_source": f"{P['source']} (bf16 burst{'; tf32 = bf16/2 nominal ratio' if w.dtype != 'bf16' else ''})",
        "peak_nominal": peak_nom,
        "peak_nominal_source": f"{sms} SMs x {8192 if w.dtype == 'bf16' else 4096} FLOP/clk/SM x {clk_mhz:.0f} MHz "
                               "(median sampled SM clock)",
        "frac_of_nominal": dk_.get("frac_of_nominal"),
        **fracs,
    }

    # End to end: pinned host inputs -> device -> fwd+bwd -> outputs back to
    # pinned host, every step. Measured two ways: serial (one stream: copy in,
    # compute, copy out) and pipelined the way a training loop double-buffers
    # (two device buffer sets; step n's inputs go up on a copy stream while step
    # n-1 computes and step n-2's results come down on another, ordered by
    # events). Both move every step's bytes inside the timed region; the
    # pipelined one is the reported value.
    e2e = None
    if not args.no_e2e:
        hin = tuple(x.pin_memory() for x in (q0, k0, v0, do0))
        dev_in = [sets[0], tuple(torch.empty_like(x) for x in sets[0])]
        dev_out = [(out, lse, dq, dk, dv), tuple(torch.empty_like(x) for x in (out, lse, dq, dk, dv))]
        host_out = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in dev_out[0]) for _ in range(2)]
        s_up = torch.cuda.Stream(dev)
        s_down = torch.cuda.Stream(dev)
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]
        for e in ev_comp + ev_down:
            e.record(stream)

        def compute(b, st):
            q, k, v, do = dev_in[b]
            o, l, gq, gk, gv = dev_out[b]
            rca.rca_attn_fwd(q, k, v, o, l, st)
            rca.rca_attn_bwd(q, k, v, o, l, do, gq, gk, gv, ws, st)

        def serial_step(n):
            for d, h in zip(dev_in[0], hin):
                d.copy_(h, non_blocking=True)
            compute(0, stream)
            for h, d in zip(host_out[0], dev_out[0]):
                h.copy_(d, non_blocking=True)

        def piped_step(n):
            b = n % 2
            with torch.cuda.stream(s_up):
                s_up.wait_event(ev_comp[b])  # step n-2 has finished reading these inputs
                for d, h in zip(dev_in[b], hin):
                    d.copy_(h, non_blocking=True)
                ev_up[b].record(s_up)
            stream.wait_event(ev_up[b])
            stream.wait_event(ev_down[b])  # step n-2's results have left these outputs
            compute(b, stream)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_comp[b])
                for h, d in zip(host_out[b], dev_out[b]):
                    h.copy_(d, non_blocking=True)
                ev_down[b].record(s_down)

        def timed(step_fn):
            for n in range(2):
                step_fn(n)
            torch.cuda.synchronize(dev)
            barrier(world)
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(s_up)
            stream.wait_event(a)
            s_down.wait_event(a)
            for n in range(args.steps):
                step_fn(n)
            stream.wait_event(ev_down[(args.steps - 1) % 2])
            z.record(stream)
            torch.cuda.synchronize(dev)
            rca.rca_stream_status(stream)
            return max_over_ranks(a.elapsed_time(z), world) / args.steps

        ser_ms = timed(serial_step)
        e_ms = timed(piped_step)
        h2d = sum(x.numel() * x.element_size() for x in hin)
        d2h = sum(x.numel() * x.element_size() for x in host_out[0])
        e2e = {"value": aggregate_tflops(step_flops, world, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "schedule": "double-buffered: inputs up and results down on two copy streams, overlapping compute",
               "serial": {"value": aggregate_tflops(step_flops, world, ser_ms), "ms_per_step": ser_ms}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, dt, threads, n = oracle_sample(w, args.cpu_budget)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} of {w.B * w.Hkv} (batch, KV-head) groups of the same workload, fwd+bwd, fp64, "
                         f"{dt:.1f} s"}

    fused_qkv = varlen = None
    if rank == 0 and not args.no_extras:
        fused_qkv = bench_fused_qkv(w, dev, stream, max(5, args.steps // 2), 3)
        varlen = bench_varlen(w, dev, stream, max(5, args.steps // 2), 3)

    mat = None
    if rank == 0 and not args.no_extras and w.B * w.Hq * w.T * w.T * 4 <= 2 ** 31:
        mat = bench_materialized(w, dev, stream, max(3, args.steps // 5), 2, P)

    decode = None
    if rank == 0 and not args.no_decode:
        decode = [bench_decode(dw, dev, stream, args.decode_steps, 5,
                               0.0 if (args.no_cpu_baseline or world > 1) else args.decode_cpu_budget, P)
                  for dw in (DEC_MHA, DEC_GQA)]

    if rank == 0:
        line = {
            "metric": args.metric, "value": value, "unit": "TFLOP/s", **fracs,
            "n_gpus": world, "steps": args.steps,
            "warmup": n_warm, "ms_per_step": ms, "step_ms": step_spread, "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32 (tf32 MMA)", "data": "synthetic",
            "config": config_for(w, world),
            "roofline": roofline,
            "min_convention": {
                "note": "backward counted as 2 x forward (no recompute), step as 3 x forward",
                "bwd_tflops": 2.0 * F / (bwd_ms * 1e-3) / 1e12,
                "step_tflops": aggregate_tflops(3.0 * F, world, ms),
            },
            "kernels": {n: {k2: (round(v2, 6) if isinstance(v2, float) else v2) for k2, v2 in d.items()}
                        for n, d in kern.items()},
            "kernels_timing": ("second pass of the same K steps with an event between every two launches; "
                               "each interval includes the kernel's launch gap"),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": launches_per_step(w) * args.steps,
            "paged_decode": decode,
            "materialized": mat,
            "fused_qkv": fused_qkv,
            "varlen": varlen,
            "src_digest": src_digest(),
        }
        print(json.dumps(line), flush=True)
    return 0


def bench_varlen(w, dev, stream, steps, warmup):
    """Variable-length batch on the workload's shape: sequence lengths drawn
    uniform in [1, T] (seeded), right padding. Tiles made only of padding are
    left out; the effective rate counts only the causal work of the real tokens."""
    import causal_head_attention_gb300 as rca

    q0, k0, v0, do0 = make_inputs(w)
    q, k, v, do = (x.to(dev) for x in (q0, k0, v0, do0))
    g = torch.Generator().manual_seed(w.seed + 100)
    lens_h = torch.randint(1, w.T + 1, (w.B,), generator=g, dtype=torch.int32)
    lens = lens_h.to(dev)
    out, lse = torch.empty_like(q), torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = rca.varlen_workspace_for(q, k)

    def step():
        rca.rca_attn_fwd_varlen(q, k, v, lens, out, lse, ws, stream)
        rca.rca_attn_bwd_varlen(q, k, v, out, lse, do, lens, dq, dk, dv, ws, stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    rca.rca_stream_status(stream)
    ms = a.elapsed_time(b) / steps
    real_flops = 3.5 * sum(4.0 * w.Hq * int(n) * int(n) * w.Dh / 2.0 for n in lens_h)
    return {"workload": w.describe(), "lens": [int(x) for x in lens_h], "ms_per_step": ms,
            "effective_tflops": real_flops / (ms * 1e-3) / 1e12,
            "note": "tiles made only of padding are skipped (planned on the device); the rate counts real tokens"}


def bench_fused_qkv(w, dev, stream, steps, warmup):
    """Fused projection layout on one workload: a training step (forward +
    backward) reading q, k, v in place from qkv [B,T,(Hq+2Hkv)Dh] and writing
    dqkv in place, against the same step with the split and concatenation
    copies a caller of the separate-tensor entry points would need."""
    import causal_head_attention_gb300 as rca

    q0, k0, v0, do0 = make_inputs(w)
    B, T, Hq, Dh, Hkv = w.B, w.T, w.Hq, w.Dh, w.Hkv
    qkv = torch.cat([q0.reshape(B, T, -1), k0.reshape(B, T, -1), v0.reshape(B, T, -1)], dim=2).to(dev)
    dout = do0.reshape(B, T, Hq * Dh).to(dev)
    out = torch.empty((B, T, Hq * Dh), dtype=qkv.dtype, device=dev)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
    dqkv = torch.empty_like(qkv)
    ws = torch.empty(rca.rca_attn_bwd_workspace_size(B, Hq, Hkv, T, Dh, qkv.dtype), dtype=torch.uint8, device=dev)

    def fused():
        rca.rca_attn_fwd_qkv(qkv, Hq, Hkv, out, lse, stream)
        rca.rca_attn_bwd_qkv(qkv, Hq, Hkv, out, lse, dout, dqkv, ws, stream)

    def with_copies():
        q = qkv[:, :, : Hq * Dh].reshape(B, T, Hq, Dh).contiguous()
        k = qkv[:, :, Hq * Dh: (Hq + Hkv) * Dh].reshape(B, T, Hkv, Dh).contiguous()
        v = qkv[:, :, (Hq + Hkv) * Dh:].reshape(B, T, Hkv, Dh).contiguous()
        o = torch.empty_like(q)
        rca.rca_attn_fwd(q, k, v, o, lse, stream)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rca.rca_attn_bwd(q, k, v, o, lse, dout.reshape(B, T, Hq, Dh), dq, dk, dv, ws, stream)
        torch.cat([dq.reshape(B, T, -1), dk.reshape(B, T, -1), dv.reshape(B, T, -1)], dim=2, out=dqkv)

    res = {}
    for name, fn in (("fused", fused), ("separate_with_copies", with_copies)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        rca.rca_stream_status(stream)
        ms = a.elapsed_time(b) / steps
        res[name] = {"ms_per_step": ms, "tflops": 3.5 * fwd_flops(w) / (ms * 1e-3) / 1e12}
    res["workload"] = w.describe()
    res["note"] = "inputs stay in L2 between steps here (one buffer set); compare the two arms, not the headline"
    return res


def bench_materialized(w, dev, stream, steps, warmup, P):
    """Materialized path on one workload: CUDA-event time of rca_attn_materialized_fwd
    and _bwd (probabilities kept, dprobs = None), and of the fused causal softmax
    and its VJP alone on [B*Hq, T, T] fp32 rows (HBM-bound; bytes below)."""
    import causal_head_attention_gb300 as rca

    q0, k0, v0, do0 = make_inputs(w)
    q, k, v, do = (x.to(dev) for x in (q0, k0, v0, do0))
    out = torch.empty_like(q)
    E, T = w.B * w.Hq, w.T
    probs = torch.empty((w.B, w.Hq, T, T), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.Hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(rca.rca_attn_materialized_workspace_size(w.B, w.Hq, w.Hkv, T, w.Dh, q.dtype),
                     dtype=torch.uint8, device=dev)

    def timed(fn, n):
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        rca.rca_stream_status(stream)
        return a.elapsed_time(b) / n

    fwd_ms = timed(lambda i: rca.rca_attn_materialized_fwd(q, k, v, out, probs, lse, ws, stream), steps)
    bwd_ms = timed(lambda i: rca.rca_attn_materialized_bwd(q, k, v, probs, do, None, dq, dk, dv, ws, stream), steps)
    # The softmax and its VJP alone, on two row buffers each larger than L2.
    scale = 1.0 / (w.Dh ** 0.5)
    s = [torch.randn((E, T, T), device=dev) for _ in range(2)]
    g = [torch.randn((E, T, T), device=dev) for _ in range(2)]
    lse2 = torch.empty((E, T), device=dev)
    sm_ms = timed(lambda i: rca.rca_causal_softmax(s[i % 2], lse2, scale, stream), steps)
    smb_ms = timed(lambda i: rca.rca_causal_softmax_bwd(s[i % 2], g[i % 2], None, scale, stream), steps)
    # The backward call runs the VJP tiled by 128 columns (dS only where its products read it).
    smbt_ms = timed(lambda i: rca.rca_causal_softmax_bwd_tiled(s[i % 2], g[i % 2], None, 128, scale, stream), steps)
    mb = materialized_bytes(E, T)
    full = mb["full"]
    sm_bytes, smb_bytes, smbt_bytes = mb["softmax"], mb["softmax_bwd"], mb["softmax_bwd_tiled128"]
    # Forward call: the probabilities written once as whole rows and read once by
    # P V (S is formed twice on the tensor cores and never stored); the
    # [B,T,H,Dh] operands are small beside them.
    fwd_bytes = mb["fwd"]
    # Backward products over the kept triangle (dP, dQ, dK, dV), each 2 * Dh FLOPs
    # per kept score and one [T, T] triangle streamed once (dP written; dS, dS, P
    # read): the backward call minus the tiled VJP it runs, timed alone.
    prod_flops = 2.0 * w.Dh * (E * T * (T + 1) / 2) * 4
    prod_bytes = mb["bwd_products"]
    prod_ms = bwd_ms - smbt_ms

    def roof(nbytes, ms):
        a = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": a, "peak": P["hbm_gbs"], "unit": "GB/s", "frac": a / P["hbm_gbs"],
                "bytes_per_launch": nbytes, "us": ms * 1e3}

    return {
        "workload": w.describe(), "name": w.name, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "probs_bytes": full,
        "fwd": dict(roof(fwd_bytes, fwd_ms), how="whole forward call: probabilities written once (whole rows), "
                    "read once by P V; row statistics from a first pass over recomputed S"),
        "bwd_products": {"ms": prod_ms, "tflops": prod_flops / (prod_ms * 1e-3) / 1e12,
                         "gbs": prod_bytes / (prod_ms * 1e-3) / 1e9,
                         "frac_hbm": prod_bytes / (prod_ms * 1e-3) / 1e9 / P["hbm_gbs"], "bytes": prod_bytes,
                         "how": "backward call time minus the VJP tiled by 128 columns (the form it runs), "
                                "timed alone"},
        "causal_softmax": roof(sm_bytes, sm_ms), "causal_softmax_bwd": roof(smb_bytes, smb_ms),
        "causal_softmax_bwd_tiled128": roof(smbt_bytes, smbt_ms),
        "note": "all kernels are this library's: tensor-core products over the kept triangle of tiles only, "
                "the fused causal softmax and its VJP",
        "gpu_launches": {"per_fwd": 4 if w.dtype == "bf16" else 7, "per_bwd": 5 if w.dtype == "bf16" else 9},
    }


def materialized_bytes(E: int, T: int) -> dict:
    """Algorithmic HBM bytes of the materialised path's pieces on E [T, T] fp32
    row blocks: `tri` the kept (lower) half, `full` whole rows; the forward
    call writes the probabilities once (whole rows) and reads them once (P V);
    the standalone softmax reads the kept half and writes whole rows and LSE;
    its VJP reads P and dP where kept and writes whole rows, or, tiled by 128,
    row i up to the end of its diagonal tile; the four backward products each
    stream one kept triangle."""
    tri = E * T * (T + 1) // 2 * 4
    full = E * T * T * 4
    return {
        "tri": tri, "full": full,
        "fwd": full + tri,
        "softmax": tri + full + E * T * 4,
        "softmax_bwd": 2 * tri + full,
        "softmax_bwd_tiled128": 2 * tri + E * sum(min(T, 128 * (i // 128 + 1)) for i in range(T)) * 4,
        "bwd_products": 4 * tri,
    }


def decode_bytes(w, lens) -> int:
    """Algorithmic HBM bytes of one paged decode call: every cached K and V row
    once, the query, the page-table entries in use, the lengths, and the output
    and LSE written once."""
    es = 2 if w.dtype == "bf16" else 4
    n = [int(x) for x in lens]
    kv = sum(n) * w.Hkv * w.Dh * 2 * es
    table = sum(-(-x // w.page_size) for x in n) * 4
    return kv + 2 * w.B * w.Hq * w.Dh * es + w.B * w.Hq * 4 + table + w.B * 4


def bench_decode(w, dev, stream, steps, warmup, cpu_budget, P):
    """Paged decode on one workload: CUDA-event time per call (decode kernel plus
    the combine kernel) over `steps` calls that alternate between two copies of
    the pools (each larger than L2)."""
    import causal_head_attention_gb300 as rca

    q0, kp0, vp0, table0, lens0 = make_paged_inputs(w)
    q, table, lens = (x.to(dev) for x in (q0, table0, lens0))
    pools = [(kp0.to(dev), vp0.to(dev))]
    pools.append(tuple(x.clone() for x in pools[0]))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    n_ws = rca.rca_paged_decode_workspace_size(w.B, w.Hq, w.Hkv, w.Dh, w.page_size, w.max_pages, q.dtype)
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)

    def call(i):
        kp, vp = pools[i % 2]
        rca.rca_paged_decode(q, kp, vp, table, lens, out, lse, ws, stream)

    for i in range(warmup):
        call(i)
    torch.cuda.synchronize(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        call(i)
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    rca.rca_stream_status(stream)
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
    ms = sum(per) / steps
    nbytes = decode_bytes(w, lens0)
    gbs = nbytes / (ms * 1e-3) / 1e9

    # End to end: query, table and lengths from pinned host memory (the cache
    # stays resident, as a serving cache does), output and LSE back to the host,
    # every call. The per-call inputs sit in one pinned staging buffer and the
    # device buffers the call reads are views of one allocation, likewise the
    # results, so each direction is a single copy (as a serving loop packs them).
    def packed(tensors, host_src):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-t.numel() * t.element_size() // 256) * 256
        dbuf = torch.empty(n, dtype=torch.uint8, device=dev)
        hbuf = torch.empty(n, dtype=torch.uint8).pin_memory()
        views = []
        for t, o, h in zip(tensors, offs, host_src):
            nb = t.numel() * t.element_size()
            views.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
            if h is not None:
                hbuf[o:o + nb].copy_(h.contiguous().view(-1).view(torch.uint8))
        return dbuf, hbuf, views

    din, hin, (qe, te, le) = packed((q, table, lens), (q0, table0, lens0))
    dout_, hout, (oe, lsee) = packed((out, lse), (None, None))

    def e2e_call(i):
        din.copy_(hin, non_blocking=True)
        kp, vp = pools[i % 2]
        rca.rca_paged_decode(qe, kp, vp, te, le, oe, lsee, ws, stream)
        hout.copy_(dout_, non_blocking=True)

    for i in range(2):
        e2e_call(i)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        e2e_call(i)
    b.record(stream)
    torch.cuda.synchronize(dev)
    rca.rca_stream_status(stream)
    e_ms = a.elapsed_time(b) / steps
    assert torch.equal(oe, out), "packed end-to-end call disagrees with the device-resident call"

    cpu = None
    if cpu_budget > 0:
        import numpy as np

        import oracle

        order = np.argsort(-lens0.numpy())  # longest requests first, then as many as the budget allows
        q64, k64, v64 = (x.double().numpy() for x in (q0, kp0, vp0))
        t0 = time.perf_counter()
        done_bytes, nreq = 0, 0
        for bi in order:
            one = slice(int(bi), int(bi) + 1)
            oracle.paged_decode(q64[one], k64, v64, table0.numpy()[one], lens0.numpy()[one])
            done_bytes += int(lens0[bi]) * w.Hkv * w.Dh * 2 * (2 if w.dtype == "bf16" else 4)
            nreq += 1
            if time.perf_counter() - t0 > cpu_budget:
                break
        dt = time.perf_counter() - t0
        cpu = {"value": done_bytes / dt / 1e9, "unit": "GB/s of K/V", "cores": 1, "kind": "oracle",
               "sample": f"{nreq} of {w.B} requests (longest first), fp64, {dt:.1f} s"}

    return {
        "workload": w.describe(), "name": w.name, "metric": "paged decode K/V streaming GB/s",
        "us_per_call": ms * 1e3, "us_min": per[0] * 1e3,
        "calls_per_s": 1e3 / ms, "tokens_per_s": w.B * 1e3 / ms,
        "roofline": {"kernel": "decode_mma_kernel" if w.dtype == "bf16" and w.Hq // w.Hkv >= 2 else "decode_kernel",
                     "bound": "hbm", "achieved": gbs, "peak": P["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / P["hbm_gbs"], "bytes_per_call": nbytes,
                     "traffic": ncu_traffic("decode", w.name)},
        "e2e": {"us_per_call": e_ms * 1e3, "h2d_bytes_per_call": hin.numel(), "d2h_bytes_per_call": hout.numel(),
                "copies": "one packed host-to-device and one device-to-host copy per call"},
        "l2": "2 rotating pool copies, each larger than L2",
        "cpu_baseline": cpu,
        "gpu_launches": 2 * steps,
    }


def profile_case(case: str, w) -> int:
    """One small invocation of a kernel family on cuda:0, untimed, for profiler
    captures: three forward calls (fwd), three backward calls after one
    forward (bwd), or two materialized forward + backward calls on the
    workload's shape cut to one batch row (materialized: [1, Hq, T, T] fp32
    probabilities, 1 GiB at T = 8192, 256 MiB at the headline T)."""
    from dataclasses import replace

    import causal_head_attention_gb300 as rca

    if case == "materialized":
        w = replace(w, B=1)
    q, k, v, do = (x.cuda() for x in make_inputs(w))
    if case == "fwd":
        for _ in range(3):
            rca.attention_forward(q, k, v)
    elif case == "bwd":
        out, lse = rca.attention_forward(q, k, v)
        for _ in range(3):
            rca.attention_backward(q, k, v, out, lse, do)
    else:
        for _ in range(2):
            out, probs, lse = rca.materialized_forward(q, k, v)
            rca.materialized_backward(q, k, v, probs, do)
    torch.cuda.synchronize()
    rca.rca_stream_status()
    print(json.dumps({"profile_case": case, "workload": w.describe()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE.name, choices=sorted(BY_NAME))
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="after the timed steps, the same step runs untimed at least this long "
                         "(clock samples under load)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the paged decode measurement")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the fused-layout, variable-length and materialized-path measurements")
    ap.add_argument("--decode-steps", type=int, default=50)
    ap.add_argument("--decode-cpu-budget", type=float, default=3.0)
    ap.add_argument("--profile-case", choices=["fwd", "bwd", "materialized"],
                    help="run one small untimed invocation of a kernel family (for profiler captures) and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.metric = "causal attn fwd+bwd TFLOP/s at B4 H16 T2048 Dh64 BF16; % of GB300 tensor peak"
    w = BY_NAME[args.workload]
    if args.profile_case:
        return profile_case(args.profile_case, w)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, w, world, rank)
    else:
        rc = run_gpu(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
