#!/usr/bin/env python
"""Benchmark of the recurrent-state decode step on GB300.

Headline workload (one "step" = one batched decode step = 8,192 state
updates): GDN, batch 256, 16 q/k heads shared by 32 value heads, dk = dv =
128, FP32 states, bf16 q/k/v, per-token per-head decay, 64 consecutive
steps of synthetic inputs cycled.  Metric: state updates per second (whole
job, all ranks) and the decode kernel's achieved HBM bandwidth against the
measured copy bandwidth.

Also reported, each on its own workload: the KDA FP32 step, the KDA mixed
FP16/INT8 step, mixed-layout speculative replay (1..8 accepted tokens), and
dasc checkpoint pack / restore (36 layers x 64 checkpoints).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torch.distributed.run, one rank per GPU, each rank an
independent replica (the decode path shards by sequence with no exchange).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from recurrent_state_gb300 import inputs as gen  # noqa: E402

METRIC = "state-updates/sec and achieved HBM GB/s (% of GB300 peak) at batch 256"
UNIT = "state-updates/s"
GDN = dict(B=256, Hk=16, Hv=32, d=128)
KDA = dict(B=256, Hk=32, Hv=32, d=128)
BENCH_STEPS_DATA = 64   # distinct input steps, cycled


# --------------------------------------------------------------------------
# algorithmic bytes (what the step must move at minimum)
# --------------------------------------------------------------------------
def decode_bytes(B, Hk, Hv, d, head_bytes, in_size, per_channel, o_size=4, tokens=1):
    state = 2 * B * Hv * head_bytes
    qk = 2 * B * Hk * d * in_size * tokens
    v = B * Hv * d * in_size * tokens
    alpha = B * Hv * (d if per_channel else 1) * 4 * tokens
    beta = B * Hv * 4 * tokens
    o = B * Hv * d * o_size * tokens
    return state + qk + v + alpha + beta + o


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# sources of the headline kernel (the FP32 step kernel at d = 128)
HEADLINE_SOURCES = ("rs_device.cuh", "rs_internal.h", "rs_step.cuh", "rs_step_f32_d128.cu")


def kernel_sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "recurrent_state_gb300", "csrc")
    for f in HEADLINE_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("sources") != kernel_sources_hash():
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            self.path = f"/tmp/rs_clocks_{os.getpid()}.csv"
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[3]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(loaded)}


# --------------------------------------------------------------------------
# the oracle as CPU baseline (host cores, bounded sample)
# --------------------------------------------------------------------------
class OracleSample:
    """The oracle's GDN decode step on host threads over a bounded sample of
    the B=256 workload's (sequence, head) items."""

    def __init__(self):
        import oracle as orc
        self.orc = orc
        self.w = gen.decode_workload(steps=1, per_channel=False, in_dtype="bf16", seed=0, **GDN)
        self.items = GDN["B"] * GDN["Hv"]
        self.pool = self.w.state0.copy()
        self.o = np.zeros((GDN["B"], GDN["Hv"], GDN["d"]), np.float32)
        self.threads = os.cpu_count() or 1
        w = self.w
        self.args = (w.q[0], w.k[0], w.v[0], w.alpha[0], w.beta[0])
        t0 = time.perf_counter()
        orc.decode_f32(self.pool, w.slot_idx, *self.args, items=(0, 16))
        self.per_item = (time.perf_counter() - t0) / 16

    def size_for(self, seconds):
        n = int(seconds * self.threads / max(self.per_item, 1e-9))
        return int(min(self.items, max(self.threads, n)))

    def run(self, n_items):
        bounds = np.linspace(0, n_items, self.threads + 1).astype(int)

        def work(i):
            self.orc.decode_f32(self.pool, self.w.slot_idx, *self.args, o=self.o,
                                items=(int(bounds[i]), int(bounds[i + 1])))
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=self.threads) as ex:
            list(ex.map(work, range(self.threads)))
        return time.perf_counter() - t0

    def describe(self, n_items):
        return (f"{n_items} of the {self.items} (sequence, head) state updates of one GDN decode "
                f"step (B=256, Hv=32, d=128), split over {self.threads} threads")


def cpu_baseline(target_seconds=12.0):
    """About target_seconds of oracle work: repeated passes over (a sample of)
    the batch's items, timed as a whole."""
    s = OracleSample()
    n = s.size_for(target_seconds)
    per_pass = max(n * s.per_item / s.threads, 1e-6)
    passes = max(1, int(round(target_seconds / per_pass)))
    dt = sum(s.run(n) for _ in range(passes))
    # the same oracle on one host thread, about 2 s of work
    n1 = int(min(s.items, max(1, 2.0 / max(s.per_item, 1e-9))))
    t0 = time.perf_counter()
    s.orc.decode_f32(s.pool, s.w.slot_idx, *s.args, o=s.o, items=(0, n1))
    dt1 = time.perf_counter() - t0
    return {"value": n * passes / dt, "unit": UNIT, "cores": s.threads, "kind": "oracle",
            "sample": f"{passes} pass(es) over " + s.describe(n), "seconds": dt,
            "single_thread": {"value": n1 / dt1, "unit": UNIT, "items": n1, "seconds": dt1}}


# --------------------------------------------------------------------------
# GPU measurement
# --------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import recurrent_state_gb300 as rs
    from recurrent_state_gb300 import build as rsbuild

    if rank == 0 or not os.path.exists(rsbuild.LIB_PATH):
        rsbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def to_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    # ---------------- headline: GDN decode, FP32 state --------------------
    w = gen.decode_workload(steps=BENCH_STEPS_DATA, per_channel=False, in_dtype="bf16",
                            seed=rank, **GDN)
    lay = rs.Layout("fp32", GDN["d"], GDN["Hv"], GDN["Hk"])
    pool = to_dev(w.state0)
    slots = to_dev(w.slot_idx)
    q, k, v = to_bf16(w.q_bits), to_bf16(w.k_bits), to_bf16(w.v_bits)
    al, be = to_dev(w.alpha), to_dev(w.beta)
    o = torch.empty((GDN["B"], GDN["Hv"], GDN["d"]), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(i):
        t = i % BENCH_STEPS_DATA
        rs.gdn_decode_update(lay, pool, slots, q[t], k[t], v[t], al[t], be[t], o=o, status=status)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        _barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        ev1.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
    dt = ev0.elapsed_time(ev1) / 1e3
    dt_max = _max_over_ranks(dt, world)
    assert int(status.item()) == 0
    updates = GDN["B"] * GDN["Hv"]
    alg = decode_bytes(GDN["B"], GDN["Hk"], GDN["Hv"], GDN["d"], lay.head_bytes, 2, False)
    per_launch = dt / args.steps
    achieved = alg / per_launch / 1e9

    # ---------------- e2e: host buffers through the C ABI ----------------
    # Each step's inputs sit in pinned host memory as one slab [q | k | v |
    # alpha | beta] (every part 16-byte aligned); a copy stream moves step
    # i + 1's slab into one of two device buffers while step i's kernel runs,
    # and a third stream copies o back.  Events order the buffer reuse.
    parts = [w.q_bits.view(np.uint8).reshape(BENCH_STEPS_DATA, -1),
             w.k_bits.view(np.uint8).reshape(BENCH_STEPS_DATA, -1),
             w.v_bits.view(np.uint8).reshape(BENCH_STEPS_DATA, -1),
             w.alpha.view(np.uint8).reshape(BENCH_STEPS_DATA, -1),
             w.beta.view(np.uint8).reshape(BENCH_STEPS_DATA, -1)]
    sizes = [x.shape[1] for x in parts]
    assert all(n % 16 == 0 for n in sizes)
    offs = np.cumsum([0] + sizes)
    slab_h = torch.from_numpy(np.ascontiguousarray(np.concatenate(parts, axis=1))).pin_memory()
    slab_d = [torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev) for _ in range(2)]
    o_d = [torch.empty_like(o) for _ in range(2)]
    oh = torch.empty((2,) + tuple(o.shape), dtype=torch.float32).pin_memory()

    def views(buf):
        def part(j, dt, shape):
            return buf[int(offs[j]):int(offs[j + 1])].view(dt).view(shape)
        return (part(0, torch.bfloat16, q[0].shape), part(1, torch.bfloat16, k[0].shape),
                part(2, torch.bfloat16, v[0].shape), part(3, torch.float32, al[0].shape),
                part(4, torch.float32, be[0].shape))
    ins = [views(b_) for b_ in slab_d]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e_ in ev_comp + ev_out:
        e_.record(stream)

    def e2e_step(i):
        t, j = i % BENCH_STEPS_DATA, i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[j])        # step i - 2 finished reading this buffer
            slab_d[j].copy_(slab_h[t], non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])           # step i - 2's o has been copied out
        qs, ks, vs, as_, bs = ins[j]
        rs.gdn_decode_update(lay, pool, slots, qs, ks, vs, as_, bs, o=o_d[j], stream=stream)
        ev_comp[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            oh[j].copy_(o_d[j], non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(world)
    ev0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    for j in range(2):
        stream.wait_event(ev_out[j])           # the last outputs are on the host
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_dt = _max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world)
    h2d = int(offs[-1])
    d2h = o.numel() * 4

    result = {
        "metric": METRIC, "value": job_value(world, args.steps, updates, dt_max), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt_max / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "GDN decode step, B=256, Hk=16, Hv=32, dk=dv=128, FP32 state, "
                               "bf16 q/k/v, 64 input steps cycled",
                   "global_batch": GDN["B"] * world, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (512 MiB state pool per rank)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": profiled_traffic("step_gdn_f32_b256"),
                     "algorithmic_bytes_per_launch": alg,
                     "kernel": "rs::step_kernel<128, FP32, GDN>"},
        "e2e": {"value": job_value(world, args.steps, updates, e2e_dt), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    del pool, q, k, v, al, be
    torch.cuda.empty_cache()
    if not args.skip_extra:
        result["kernels"] = extra_kernels(args, rs, torch, dev, peak, world)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline()
    if "kernels" in result:
        # the packed-layout and multi-token lines in short, last in the line
        # (the most-read end of a long record), most important last
        keep = [n for n in result["kernels"] if n.startswith(("ckpt_", "kda_prefill", "gdn_prefill", "kda_replay"))]
        keep += [n for n in result["kernels"] if n.startswith(("kda_decode_damp", "gdn_decode_mixed",
                                                                "kda_decode_mixed"))]
        result["packed_summary"] = {
            n: {"ms": round(result["kernels"][n]["ms"], 4),
                "frac": round(result["kernels"][n]["frac_of_peak"], 3)} for n in keep}
    return result


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world):
    """Largest value over the ranks (the elapsed time of the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, steps, units_per_step, dt_max):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (every rank runs its own replica of the workload)."""
    return world * steps * units_per_step / dt_max


# Median of the per-launch times of the last _time call (s) and its repeat count.
_LAST_MEDIAN = {"s": None, "n": 0}


def _time(torch, fn, iters, warm=3, repeats=20):
    """Seconds per launch: ``iters`` launches split into up to five windows of
    back-to-back launches (CUDA events around each window), and the median of
    the windows' means, so that one stall of the host between two launches
    cannot move the figure; also times ``max(repeats, 20)`` launches one by
    one, each between its own pair of events, and keeps their median."""
    warm = max(3, warm)
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    nw = max(1, min(5, iters))
    per_w = max(1, iters // nw)
    means, k = [], warm
    for _ in range(nw):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(per_w):
            fn(k)
            k += 1
        e1.record()
        torch.cuda.synchronize()
        means.append(e0.elapsed_time(e1) / 1e3 / per_w)
    mean = sorted(means)[nw // 2]
    n = max(repeats, 20)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i, (a, b) in enumerate(ev):
        a.record()
        fn(k + i)
        b.record()
    torch.cuda.synchronize()
    per = sorted(a.elapsed_time(b) / 1e3 for a, b in ev)
    _LAST_MEDIAN["s"], _LAST_MEDIAN["n"] = per[n // 2], n
    return mean


def rotation(torch, pool, dev):
    """The pool and enough copies of it that consecutive launches, taking them
    in turn, read at least four L2 capacities of distinct state: every launch
    then reads its state from HBM, not from what the previous launch left in
    L2."""
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2 ** 20
    n = max(1, -(-4 * l2 // (pool.numel() * pool.element_size())))
    return [pool] + [pool.clone() for _ in range(n - 1)]


def rot_info(pools):
    return {"pools_rotated": len(pools),
            "rotation_bytes": sum(p.numel() * p.element_size() for p in pools)}


EXTRA = ("gdn_tiny", "gdn_fp32", "kda_fp32", "kda_mixed", "gdn_mixed", "kda_damp", "replay_mixed", "replay_fp32",
         "kda_mixed_fused", "kda_mixed_fused_wide", "gdn_mixed_fused", "kda_damp_fused", "replay_mixed_fused", "replay_sweep",
         "prefill_fp32", "prefill_mixed_fused", "prefill_chunked",
         "pack_gdn", "restore_gdn", "pack_kda", "restore_kda", "pack_int8_gdn", "restore_int8_gdn",
         "pack_int8_kda", "restore_int8_kda", "pack_mixed", "restore_mixed")


# The five workload configurations as named presets of secondary kernels:
# the small GDN case, GDN and KDA decode with FP32 state, KDA on the mixed
# layout (decode and replay, both requantisation modes), dasc pack/restore.
PRESETS = {
    "tiny": ["gdn_tiny"],
    "gdn": ["gdn_fp32"],
    "kda": ["kda_fp32"],
    "kda_mixed": ["kda_mixed", "kda_mixed_fused", "kda_mixed_fused_wide", "replay_mixed", "replay_mixed_fused",
                  "replay_sweep"],
    "ckpt": ["pack_gdn", "restore_gdn", "pack_kda", "restore_kda"],
}


def extra_kernels(args, rs, torch, dev, peak, world, only=None):
    """The other hot-path kernels, each timed alone on its own workload."""
    out = {}
    iters = max(3, min(args.steps, 200))
    warm = max(3, min(args.warmup, 10))
    want = set(only) if only else set(EXTRA)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def to_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    # FP32 pipe peak for the multi-token kernels, whose arithmetic per state byte is 4.5-32x a decode
    # step's: every SM's 128 FP32 lanes retiring one FMA (2 FLOP) per cycle at the 2,070 MHz maximum
    # SM clock.  Their FP32 work per state element and token is 7 FLOP (decay multiply, and the FMAs of
    # the prediction, the write and the readout).
    fp32_peak = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * 2.07e9

    def rec(name, sec, alg, updates, extra=None, tile_tokens=None):
        gbs = alg / sec / 1e9
        out[name] = {"ms": sec * 1e3, "GB/s": gbs, "frac_of_peak": gbs / peak,
                     "algorithmic_bytes": alg, "state_updates_per_s": updates / sec if updates else None}
        if _LAST_MEDIAN["s"] is not None:
            out[name].update({"ms_median": _LAST_MEDIAN["s"] * 1e3, "median_of": _LAST_MEDIAN["n"]})
            _LAST_MEDIAN["s"] = None
        if tile_tokens:
            fl = tile_tokens * 128 * 128 * 7
            out[name].update({"fp32_flops": fl, "TFLOP/s": fl / sec / 1e12, "frac_of_fp32_peak": fl / sec / fp32_peak})
        if extra:
            out[name].update(extra)

    B = getattr(args, "batch", None) or 256
    if "gdn_tiny" in want:
        # small GDN case: B=4, 4 heads, dk=dv=64, FP32 state and inputs (launch-bound; correctness size)
        w = gen.decode_workload(B=4, Hk=4, Hv=4, d=64, steps=16, per_channel=False, in_dtype="f32", seed=0,
                                tiny_gdn=True)
        lay = rs.Layout("fp32", 64, 4, 4)
        pool = to_dev(w.state0)
        q, k, v = to_dev(w.q), to_dev(w.k), to_dev(w.v)
        al, be, slots = to_dev(w.alpha), to_dev(w.beta), to_dev(w.slot_idx)
        o = torch.empty((4, 4, 64), device=dev)
        sec = _time(torch, lambda i: rs.gdn_decode_update(lay, pool, slots, q[i % 16], k[i % 16], v[i % 16],
                                                          al[i % 16], be[i % 16], o=o), iters, warm)
        rec("gdn_decode_fp32_tiny_b4_d64", sec, decode_bytes(4, 4, 4, 64, lay.head_bytes, 4, False), 16)
        # the same 16 steps captured once in a CUDA graph and replayed: launch cost without the
        # host-side call path
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for i in range(16):
                rs.gdn_decode_update(lay, pool, slots, q[i], k[i], v[i], al[i], be[i], o=o)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(16):
                rs.gdn_decode_update(lay, pool, slots, q[i], k[i], v[i], al[i], be[i], o=o)
        sec = _time(torch, lambda i: graph.replay(), max(3, iters // 16), warm) / 16
        _LAST_MEDIAN["s"] /= 16  # per launch, like the mean
        rec("gdn_decode_fp32_tiny_b4_d64_graph", sec, decode_bytes(4, 4, 4, 64, lay.head_bytes, 4, False), 16,
            {"launches_per_graph": 16})
    if "gdn_fp32" in want:
        nsteps = 8
        g_cfg = dict(GDN, B=B)
        w = gen.decode_workload(steps=nsteps, per_channel=False, in_dtype="bf16", seed=2, **g_cfg)
        lay = rs.Layout("fp32", 128, GDN["Hv"], GDN["Hk"])
        pool = to_dev(w.state0)
        q, k, v = to_bf16(w.q_bits), to_bf16(w.k_bits), to_bf16(w.v_bits)
        al, be, slots = to_dev(w.alpha), to_dev(w.beta), to_dev(w.slot_idx)
        o = torch.empty((B, GDN["Hv"], 128), device=dev)
        sec = _time(torch, lambda i: rs.gdn_decode_update(
            lay, pool, slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al[i % nsteps],
            be[i % nsteps], o=o), iters, warm)
        rec(f"gdn_decode_fp32_b{B}", sec, decode_bytes(B, 16, 32, 128, lay.head_bytes, 2, False),
            B * 32)
        del pool, q, k, v
        torch.cuda.empty_cache()
    KDA_B = dict(KDA, B=B)
    MIXED_KEYS = {"kda_fp32", "kda_mixed", "gdn_mixed", "kda_damp", "replay_mixed", "replay_fp32",
                  "kda_mixed_fused", "kda_mixed_fused_wide", "gdn_mixed_fused", "kda_damp_fused",
                  "replay_mixed_fused", "replay_sweep"}
    if want & MIXED_KEYS:
        nsteps = 8
        w = gen.decode_workload(steps=nsteps, per_channel=True, in_dtype="bf16", seed=1,
                                horizon=(2.0, 8192.0), **KDA_B)
        q, k, v = to_bf16(w.q_bits), to_bf16(w.k_bits), to_bf16(w.v_bits)
        al, be = to_dev(w.alpha), to_dev(w.beta)
        slots = to_dev(w.slot_idx)
        o = torch.empty((B, KDA["Hv"], KDA["d"]), device=dev)
        f32 = rs.Layout("fp32", 128, KDA["Hv"], KDA["Hk"])
        hi = gen.hi_rows(KDA["Hv"], 128, 16, seed=1)
        mix = rs.Layout("mixed", 128, KDA["Hv"], KDA["Hk"], k_hi=16, hi_rows=hi)
        # the same pool format with the fused requantisation arithmetic
        mixf = rs.Layout("mixed", 128, KDA["Hv"], KDA["Hk"], k_hi=16, hi_rows=hi, quant="fused")
        pool = to_dev(w.state0)
        mpool = mix.empty_pool(B, device=dev)
        rs.state_convert(f32, pool, mix, mpool, torch.arange(B, dtype=torch.int32, device=dev))
        mpools = rotation(torch, mpool, dev)  # 155 MB each at batch 256: rotated past L2
        R_m = len(mpools)
        if "kda_fp32" in want:
            sec = _time(torch, lambda i: rs.kda_decode_update(
                f32, pool, slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al[i % nsteps],
                be[i % nsteps], o=o), iters, warm)
            rec(f"kda_decode_fp32_b{B}", sec, decode_bytes(B, 32, 32, 128, f32.head_bytes, 2, True),
                B * 32)
        if "kda_mixed" in want:
            sec = _time(torch, lambda i: rs.kda_decode_update(
                mix, mpools[i % R_m], slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al[i % nsteps],
                be[i % nsteps], o=o), iters, warm)
            rec(f"kda_decode_mixed_b{B}", sec, decode_bytes(B, 32, 32, 128, mix.head_bytes, 2, True),
                B * 32, rot_info(mpools))
        if "kda_mixed_fused" in want:
            sec = _time(torch, lambda i: rs.kda_decode_update(
                mixf, mpools[i % R_m], slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al[i % nsteps],
                be[i % nsteps], o=o), iters, warm)
            rec(f"kda_decode_mixed_fused_b{B}", sec, decode_bytes(B, 32, 32, 128, mix.head_bytes, 2, True),
                B * 32, {"quant": "fused", **rot_info(mpools)})
        if "kda_mixed_fused_wide" in want:
            # the same kernel on four copies of the batch (4 B sequences, built on the device): the
            # per-launch fixed cost (pipeline fill and the last round of tiles) weighs a quarter as much
            R = 4
            wpool = mpool.repeat(R, 1, 1)  # 619 MB: larger than four L2 capacities by itself
            wq, wk, wv = q.repeat(1, R, 1, 1), k.repeat(1, R, 1, 1), v.repeat(1, R, 1, 1)
            wal, wbe = al.repeat(1, R, 1, 1), be.repeat(1, R, 1)
            wslots = torch.arange(R * B, dtype=torch.int32, device=dev)
            wo = torch.empty((R * B, KDA["Hv"], KDA["d"]), device=dev)
            sec = _time(torch, lambda i: rs.kda_decode_update(
                mixf, wpool, wslots, wq[i % nsteps], wk[i % nsteps], wv[i % nsteps], wal[i % nsteps],
                wbe[i % nsteps], o=wo), iters, warm)
            rec(f"kda_decode_mixed_fused_b{R * B}", sec,
                decode_bytes(R * B, 32, 32, 128, mix.head_bytes, 2, True), R * B * 32,
                {"quant": "fused", "inputs": f"the batch-{B} workload repeated {R} times"})
            del wpool, wq, wk, wv, wal, wbe, wo
            torch.cuda.empty_cache()
        al_g = al[..., 0].contiguous()  # one decay per (sequence, head) for the GDN form
        if "gdn_mixed" in want:
            sec = _time(torch, lambda i: rs.gdn_decode_update(
                mix, mpools[i % R_m], slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al_g[i % nsteps],
                be[i % nsteps], o=o), iters, warm)
            rec(f"gdn_decode_mixed_b{B}_h32", sec,
                decode_bytes(B, 32, 32, 128, mix.head_bytes, 2, False), B * 32, rot_info(mpools))
        if "gdn_mixed_fused" in want:
            sec = _time(torch, lambda i: rs.gdn_decode_update(
                mixf, mpools[i % R_m], slots, q[i % nsteps], k[i % nsteps], v[i % nsteps], al_g[i % nsteps],
                be[i % nsteps], o=o), iters, warm)
            rec(f"gdn_decode_mixed_fused_b{B}_h32", sec,
                decode_bytes(B, 32, 32, 128, mix.head_bytes, 2, False), B * 32,
                {"quant": "fused", **rot_info(mpools)})
        for dkey, quant in (("kda_damp", "ieee"), ("kda_damp_fused", "fused")):
            if dkey not in want:
                continue
            # DAMP-exact storage: INT8 groups of 32 along dv, value scaling
            damp = rs.Layout("damp", 128, KDA["Hv"], KDA["Hk"], k_hi=16, hi_rows=hi,
                             value_scales=gen.value_scales(KDA["Hv"], 128, seed=1), quant=quant)
            dpool = damp.empty_pool(B, device=dev)
            rs.state_convert(f32, pool, damp, dpool, torch.arange(B, dtype=torch.int32, device=dev))
            dpools = rotation(torch, dpool, dev)
            sec = _time(torch, lambda i: rs.kda_decode_update(
                damp, dpools[i % len(dpools)], slots, q[i % nsteps], k[i % nsteps], v[i % nsteps],
                al[i % nsteps], be[i % nsteps], o=o), iters, warm)
            suffix = "_fused" if quant == "fused" else ""
            rec(f"kda_decode_damp_g32{suffix}_b{B}", sec,
                decode_bytes(B, 32, 32, 128, damp.head_bytes, 2, True), B * 32,
                {"bits_per_value": damp.bits_per_value(), "quant": quant, **rot_info(dpools)})
            del dpool, dpools
        if want & {"replay_mixed", "replay_fp32", "replay_mixed_fused", "replay_sweep"}:
            T = 8
            n_acc = gen.n_accept(B, T, seed=1)
            tok = int(n_acc.sum())

            def bt(x):
                return np.ascontiguousarray(np.swapaxes(x[:T], 0, 1))
            rq, rk, rv = to_bf16(bt(w.q_bits)), to_bf16(bt(w.k_bits)), to_bf16(bt(w.v_bits))
            ra, rb = to_dev(bt(w.alpha)), to_dev(bt(w.beta))
            ro = torch.empty((B, T, 32, 128), device=dev)
            nd = to_dev(n_acc)
            per_tok = 2 * 32 * 128 * 2 + 32 * 128 * 2 + 32 * 128 * 4 + 32 * 4 + 32 * 128 * 4
            if "replay_mixed" in want:
                sec = _time(torch, lambda i: rs.spec_replay_update(
                    mix, True, mpools[i % R_m], slots, nd, rq, rk, rv, ra, rb, o=ro), iters, warm)
                rec(f"kda_replay_mixed_b{B}_T8", sec, 2 * B * 32 * mix.head_bytes + tok * per_tok,
                    tok * 32, {"accepted_tokens": tok, "n_accept": "uniform 1..8", **rot_info(mpools)},
                    tile_tokens=tok * 32)
            if "replay_mixed_fused" in want:
                sec = _time(torch, lambda i: rs.spec_replay_update(
                    mixf, True, mpools[i % R_m], slots, nd, rq, rk, rv, ra, rb, o=ro), iters, warm)
                rec(f"kda_replay_mixed_fused_b{B}_T8", sec, 2 * B * 32 * mix.head_bytes + tok * per_tok,
                    tok * 32, {"accepted_tokens": tok, "n_accept": "uniform 1..8", "quant": "fused",
                               **rot_info(mpools)}, tile_tokens=tok * 32)
            if "replay_fp32" in want:
                sec = _time(torch, lambda i: rs.spec_replay_update(
                    f32, True, pool, slots, nd, rq, rk, rv, ra, rb, o=ro), iters, warm)
                rec(f"kda_replay_fp32_b{B}_T8", sec, 2 * B * 32 * f32.head_bytes + tok * per_tok,
                    tok * 32, {"accepted_tokens": tok}, tile_tokens=tok * 32)
            if "replay_sweep" in want:
                # every sequence accepts exactly Tn tokens of the 8-token window, both layouts' mixed modes
                for Tn in (1, 2, 4, 8):
                    nfix = torch.full((B,), Tn, dtype=torch.int32, device=dev)
                    for lay, qname in ((mix, "ieee"), (mixf, "fused")):
                        sec = _time(torch, lambda i: rs.spec_replay_update(
                            lay, True, mpools[i % R_m], slots, nfix, rq, rk, rv, ra, rb, o=ro), iters, warm)
                        rec(f"kda_replay_mixed_{qname}_b{B}_n{Tn}", sec,
                            2 * B * 32 * mix.head_bytes + B * Tn * per_tok, B * Tn * 32,
                            {"accepted_tokens": B * Tn, "n_accept": f"all {Tn}", "quant": qname,
                             **rot_info(mpools)}, tile_tokens=B * Tn * 32)
        del pool, mpool, mpools
        torch.cuda.empty_cache()

    # prefill chunks: KDA, 32 heads, a chunk of 32 tokens per sequence
    if want & {"prefill_fp32", "prefill_mixed_fused"}:
        Lc = 32
        w = gen.decode_workload(steps=Lc, per_channel=True, in_dtype="bf16", seed=3,
                                horizon=(2.0, 8192.0), **KDA_B)

        def bt(x):
            return np.ascontiguousarray(np.swapaxes(x, 0, 1))
        pq, pk, pv = to_bf16(bt(w.q_bits)), to_bf16(bt(w.k_bits)), to_bf16(bt(w.v_bits))
        pa, pb = to_dev(bt(w.alpha)), to_dev(bt(w.beta))
        slots = to_dev(w.slot_idx)
        po = torch.empty((B, Lc, 32, 128), device=dev)
        f32 = rs.Layout("fp32", 128, KDA["Hv"], KDA["Hk"])
        pool = to_dev(w.state0)
        per_tok = 2 * 32 * 128 * 2 + 32 * 128 * 2 + 32 * 128 * 4 + 32 * 4 + 32 * 128 * 4
        if "prefill_fp32" in want:
            sec = _time(torch, lambda i: rs.prefill_update(f32, True, pool, slots, pq, pk, pv, pa, pb, o=po),
                        max(3, iters // 10), warm)
            rec(f"kda_prefill_fp32_b{B}_L{Lc}", sec, 2 * B * 32 * f32.head_bytes + B * Lc * per_tok,
                B * 32 * Lc, {"chunk_tokens": Lc}, tile_tokens=B * 32 * Lc)
        if "prefill_mixed_fused" in want:
            hi = gen.hi_rows(KDA["Hv"], 128, 16, seed=3)
            mixf = rs.Layout("mixed", 128, KDA["Hv"], KDA["Hk"], k_hi=16, hi_rows=hi, quant="fused")
            mpool = mixf.empty_pool(B, device=dev)
            rs.state_convert(f32, pool, mixf, mpool, torch.arange(B, dtype=torch.int32, device=dev))
            ppools = rotation(torch, mpool, dev)
            sec = _time(torch, lambda i: rs.prefill_update(mixf, True, ppools[i % len(ppools)], slots, pq, pk,
                                                           pv, pa, pb, o=po), max(3, iters // 10), warm)
            rec(f"kda_prefill_mixed_fused_b{B}_L{Lc}", sec, 2 * B * 32 * mixf.head_bytes + B * Lc * per_tok,
                B * 32 * Lc, {"chunk_tokens": Lc, "quant": "fused", **rot_info(ppools)},
                tile_tokens=B * 32 * Lc)
            del mpool, ppools
        del pool, pq, pk, pv, pa, pb, po
        torch.cuda.empty_cache()

    # prefill in the chunk-parallel form on the tensor cores: FP32 state, KDA and GDN, 32 and 64 tokens
    if "prefill_chunked" in want:
        for kda, Lc in ((True, 32), (True, 64), (False, 32)):
            cfg = dict(KDA_B) if kda else dict(GDN, B=B)
            w = gen.decode_workload(steps=Lc, per_channel=kda, in_dtype="bf16", seed=4,
                                    horizon=(2.0, 8192.0) if kda else (4.0, 4096.0), **cfg)

            def bt(x):
                return np.ascontiguousarray(np.swapaxes(x, 0, 1))
            pq, pk, pv = to_bf16(bt(w.q_bits)), to_bf16(bt(w.k_bits)), to_bf16(bt(w.v_bits))
            pa, pb = to_dev(bt(w.alpha)), to_dev(bt(w.beta))
            slots = to_dev(w.slot_idx)
            Hk, Hv = cfg["Hk"], cfg["Hv"]
            po = torch.empty((B, Lc, Hv, 128), device=dev)
            f32 = rs.Layout("fp32", 128, Hv, Hk)
            pool = to_dev(w.state0)  # 512 MiB: larger than four L2 capacities
            qk_tok = 2 * Hk * 128 * 2 / Hv          # q and k (bf16) per value head and token
            per_tok = Hv * (qk_tok + 128 * 2 + (128 * 4 if kda else 4) + 4 + 128 * 4)
            sec = _time(torch, lambda i: rs.prefill_update(f32, kda, pool, slots, pq, pk, pv, pa, pb, o=po,
                                                           chunked=True), max(3, iters // 10), warm)
            rec(f"{'kda' if kda else 'gdn'}_prefill_chunked_fp32_b{B}_L{Lc}", sec,
                2 * B * Hv * f32.head_bytes + int(B * Lc * per_tok), B * Hv * Lc,
                {"chunk_tokens": Lc, "form": "chunk-parallel, tcgen05 kind::tf32 (3 products per pair)"},
                tile_tokens=B * Hv * Lc)
            if kda and Lc == 32:  # the same on the mixed FP16/INT8 state, fused arithmetic, rotated pools
                hi = gen.hi_rows(Hv, 128, 16, seed=4)
                mixf = rs.Layout("mixed", 128, Hv, Hk, k_hi=16, hi_rows=hi, quant="fused")
                mpool = mixf.empty_pool(w.state0.shape[0], device=dev)
                rs.state_convert(f32, pool, mixf, mpool,
                                 torch.arange(w.state0.shape[0], dtype=torch.int32, device=dev))
                ppools = rotation(torch, mpool, dev)
                sec = _time(torch, lambda i: rs.prefill_update(mixf, kda, ppools[i % len(ppools)], slots, pq, pk,
                                                               pv, pa, pb, o=po, chunked=True),
                            max(3, iters // 10), warm)
                rec(f"kda_prefill_chunked_mixed_fused_b{B}_L{Lc}", sec,
                    2 * B * Hv * mixf.head_bytes + int(B * Lc * per_tok), B * Hv * Lc,
                    {"chunk_tokens": Lc, "quant": "fused", "form": "chunk-parallel, tcgen05 kind::tf32",
                     **rot_info(ppools)}, tile_tokens=B * Hv * Lc)
                del mpool, ppools
                # and on DAMP-exact tiles (INT8 groups of 32, value scaling)
                cs = gen.value_scales(Hv, 128, seed=4)
                dmp = rs.Layout("damp", 128, Hv, Hk, k_hi=16, hi_rows=hi, value_scales=cs, quant="fused")
                dpool = dmp.empty_pool(w.state0.shape[0], device=dev)
                rs.state_convert(f32, pool, dmp, dpool,
                                 torch.arange(w.state0.shape[0], dtype=torch.int32, device=dev))
                dpools = rotation(torch, dpool, dev)
                sec = _time(torch, lambda i: rs.prefill_update(dmp, kda, dpools[i % len(dpools)], slots, pq, pk,
                                                               pv, pa, pb, o=po, chunked=True),
                            max(3, iters // 10), warm)
                rec(f"kda_prefill_chunked_damp_fused_b{B}_L{Lc}", sec,
                    2 * B * Hv * dmp.head_bytes + int(B * Lc * per_tok), B * Hv * Lc,
                    {"chunk_tokens": Lc, "quant": "fused", "form": "chunk-parallel, tcgen05 kind::tf32",
                     **rot_info(dpools)}, tile_tokens=B * Hv * Lc)
                del dpool, dpools
            del pool, pq, pk, pv, pa, pb, po
            torch.cuda.empty_cache()

    # dasc pack / restore: 36 layers, 64 checkpoints, 64 pool slots
    for unit, p, name in ((0, 0.5, "gdn"), (1, 0.45, "kda")):
        if not want & {f"pack_{name}", f"restore_{name}", f"pack_int8_{name}", f"restore_int8_{name}"}:
            continue
        nslot = n = getattr(args, "slots", None) or 64
        L, Hv, d = 36, 32, 128
        keep = gen.keep_mask(L, Hv if unit == 0 else Hv * d, p, seed=unit)
        src, dst = gen.ckpt_slots(nslot, n, seed=unit)
        lay = rs.Layout("fp32", d, Hv, 1)
        plan = rs.Plan(lay, keep, "head" if unit == 0 else "channel").upload()
        big = torch.empty((L, nslot, Hv, d, d), device=dev)
        big.normal_()
        ckpt = plan.empty_ckpt_pool(n, device=dev)
        sd, dd = to_dev(src), to_dev(dst)
        kept_bytes = int(plan.offsets[-1]) * plan.unit_bytes * n
        full_bytes = L * Hv * d * d * 4 * n
        rs.ckpt_pack(plan, big, sd, dd, ckpt)
        if f"pack_{name}" in want:
            sec = _time(torch, lambda i: rs.ckpt_pack(plan, big, sd, dd, ckpt), max(3, iters // 10), warm)
            rec(f"ckpt_pack_{name}", sec, 2 * kept_bytes, 0,
                {"checkpoints_per_s": n / sec, "C_temp": keep.size / max(int(keep.sum()), 1)})
        if f"restore_{name}" in want:
            sec = _time(torch, lambda i: rs.ckpt_restore(plan, ckpt, dd, big, sd), max(3, iters // 10),
                        warm)
            rec(f"ckpt_restore_{name}", sec, kept_bytes + full_bytes, 0, {"checkpoints_per_s": n / sec})
        del ckpt
        # dasc INT8 checkpoint of the same plan: quantise at pack, dequantise at restore
        if want & {f"pack_int8_{name}", f"restore_int8_{name}"}:
            ck8 = plan.empty_int8_ckpt_pool(n, device=dev)
            rows = plan.int8_codes_bytes // d
            int8_bytes = (plan.int8_codes_bytes + 4 * rows) * n
            kept_f32 = rows * d * 4 * n
            rs.ckpt_pack_int8(plan, big, sd, dd, ck8)
            if f"pack_int8_{name}" in want:
                sec = _time(torch, lambda i: rs.ckpt_pack_int8(plan, big, sd, dd, ck8), max(3, iters // 10),
                            warm)
                rec(f"ckpt_pack_int8_{name}", sec, kept_f32 + int8_bytes, 0,
                    {"checkpoints_per_s": n / sec, "bytes_vs_fp32": kept_f32 / int8_bytes})
            if f"restore_int8_{name}" in want:
                sec = _time(torch, lambda i: rs.ckpt_restore_int8(plan, ck8, dd, big, sd),
                            max(3, iters // 10), warm)
                rec(f"ckpt_restore_int8_{name}", sec, int8_bytes + full_bytes, 0, {"checkpoints_per_s": n / sec})
            del ck8
        del big
        torch.cuda.empty_cache()
    # whole mixed FP16/INT8 heads (18,880 B) in and out of checkpoints
    if want & {"pack_mixed", "restore_mixed"}:
        nslot = n = getattr(args, "slots", None) or 64
        L, Hv, d = 36, 32, 128
        keep = gen.keep_mask(L, Hv, 0.5, seed=0)
        src, dst = gen.ckpt_slots(nslot, n, seed=0)
        hi = gen.hi_rows(Hv, d, 16, seed=1)
        mix = rs.Layout("mixed", d, Hv, Hv, k_hi=16, hi_rows=hi)
        plan = rs.Plan(mix, keep, "head").upload()
        big = torch.randint(0, 255, (L, nslot, Hv, mix.head_bytes), dtype=torch.uint8, device=dev)
        ckpt = plan.empty_ckpt_pool(n, device=dev)
        sd, dd = to_dev(src), to_dev(dst)
        kept_bytes = int(plan.offsets[-1]) * plan.unit_bytes * n
        full_bytes = L * Hv * mix.head_bytes * n
        rs.ckpt_pack(plan, big, sd, dd, ckpt)
        if "pack_mixed" in want:
            sec = _time(torch, lambda i: rs.ckpt_pack(plan, big, sd, dd, ckpt), max(3, iters // 10), warm)
            rec("ckpt_pack_mixed_gdn", sec, 2 * kept_bytes, 0, {"checkpoints_per_s": n / sec})
        if "restore_mixed" in want:
            sec = _time(torch, lambda i: rs.ckpt_restore(plan, ckpt, dd, big, sd), max(3, iters // 10), warm)
            rec("ckpt_restore_mixed_gdn", sec, kept_bytes + full_bytes, 0, {"checkpoints_per_s": n / sec})
        del big, ckpt
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------
# reference arm: the oracle on host cores
# --------------------------------------------------------------------------
def run_reference(args, budget_seconds=100.0):
    s = OracleSample()
    total = args.warmup + args.steps
    n = s.size_for(budget_seconds / total)
    for _ in range(args.warmup):
        s.run(n)
    t_all = 0.0
    for _ in range(args.steps):
        t_all += s.run(n)
    value = n * args.steps / t_all
    updates = GDN["B"] * GDN["Hv"]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": updates / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "GDN decode step, B=256, Hk=16, Hv=32, dk=dv=128, FP32 state, "
                               "bf16 q/k/v", "global_batch": GDN["B"], "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": s.threads, "kind": "oracle",
                         "sample": s.describe(n) + " per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--batch", type=int, default=None,
                    help="batch of the decode kernels in --only mode (default 256)")
    ap.add_argument("--slots", type=int, default=None,
                    help="pool slots and checkpoints of the pack/restore kernels (default 64)")
    ap.add_argument("--only", default=None,
                    help="comma list of secondary kernels to time alone (" + ",".join(EXTRA) + ")")
    ap.add_argument("--config", choices=sorted(PRESETS), default=None,
                    help="time one workload configuration's kernels alone (a named --only list)")
    args = ap.parse_args()
    if args.config:
        args.only = ",".join(PRESETS[args.config] + ([args.only] if args.only else []))
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if args.only:
        import torch
        import recurrent_state_gb300 as rs
        from recurrent_state_gb300 import build as rsbuild
        rsbuild.build()
        names = [x for x in args.only.split(",") if x]
        bad = [x for x in names if x not in EXTRA]
        if bad:
            raise SystemExit(f"unknown kernel(s) {bad}; choose from {EXTRA}")
        torch.cuda.set_device(local_rank)
        res = extra_kernels(args, rs, torch, torch.device("cuda", local_rank), measured_peaks()[0],
                            1, only=names)
        print(json.dumps({"only": res}), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
