#!/usr/bin/env python3
"""Benchmark: causal NeoX-rotary self-attention forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole op (rotary + QK^T + causal online softmax + PV +
epilogue, one kernel launch) over the GPT-NeoX-20B-shaped workload (B=2, H=64,
S=2048, D=96, rotary_dim=24) unless --workload says otherwise.  Inputs are seeded,
synthetic and already resident in HBM when the timed region starts; L2 is flushed
before every step, outside the per-step CUDA-event interval (a 256 MB write, then a
256 MB read of another buffer, so that no dirty line of the flush is written back
inside the step).
Metric: causal FLOPs 2*B*H*S^2*D per step / kernel time, in TFLOP/s, and that figure
as a fraction of the measured dense bf16 tensor peak.

N > 1 (torchrun): every rank runs its own copy of the workload on its own seed (weak
scaling; the op has no exchange step), the timing is the max over ranks, and the
value is the FLOPs of all ranks over that time.

--impl reference times the fp64 CPU oracle (the test oracle, as it stands) on the
host cores on a bounded sample of the same workload per step; rank 0 only.

--workload NAME-decode measures the incremental decode instead (neox_attn_decode: one
new token per sequence against a resident K/V cache), in GB/s of cache read per step,
against the measured HBM copy bandwidth (1 GPU).
One JSON line on stdout (rank 0); everything else goes to stderr.

--pass bwd times the backward (neox_attn_bwd) on a prefill workload instead: 5 B H S^2 D
algorithmic FLOPs per step in TFLOP/s, the forward's out/lse and a seeded dout resident.

--pass proj times the query_key_value projection that produces the packed qkv
(neox_attn_qkv_proj: x[B*S, H*D] times w[H*D, 3*H*D] plus bias, query/key slots rotated
in the epilogue): 2 M K N FLOPs per step in TFLOP/s against the same bf16 peak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from causal_rope_self_neox_b300.workloads import (DECODE_WORKLOADS, WORKLOADS, bf16_bits,  # noqa: E402
                                                  make_decode_inputs, make_qkv)

METRIC = "causal RoPE attention fwd TFLOP/s and % of B300 bf16 tensor peak"
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed before every step, outside the event interval: a 256 MB write, then a 256 MB read of "
           "another buffer, so L2 holds clean unrelated lines (no write-back of the flush inside the step)")


class L2Flush:
    """Evicts L2 between timed steps: writes one buffer larger than L2, then reads another,
    so the step starts with neither its inputs nor dirty lines of the flush in L2."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)
        self.torch = torch

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.sink)
FALLBACK_BF16_TFLOPS = 1800.0
FALLBACK_HBM_GBS = 6400.0
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), \
            float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


FWD_KERNEL_SOURCES = ("attn_ws.cuh", "attn_common.cuh", "ptx.cuh", "rotary.cuh", "tile_layout.cuh")
DEC_KERNEL_SOURCES = ("decode.cuh", "attn_common.cuh", "ptx.cuh", "tile_layout.cuh", "neox_attn.cu")
BWD_KERNEL_SOURCES = ("attn_bwd.cuh", "attn_common.cuh", "ptx.cuh", "tile_layout.cuh", "neox_attn.cu")


def code_only(text: str) -> str:
    """C/C++/CUDA source with its comments and blank lines removed and trailing whitespace
    trimmed (string and character literals kept as they are), so that a comment edit
    leaves the hash of the compiled code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (l.rstrip() for l in "".join(out).split("\n"))
    return "\n".join(l for l in lines if l)


def kernel_source_hash(sources=FWD_KERNEL_SOURCES) -> str:
    """Hash of the code (comments excluded) of the sources a kernel is compiled and launched
    from (by default the prefill kernel's)."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "causal_rope_self_neox_b300", "csrc", name)) as fh:
            h.update(name.encode())
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, prefix: str = "attn_fwd_ws", sources=FWD_KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary of this workload
    (profiles/<prefix>_<workload>.txt, `key: value` lines), if it was taken on the
    current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.txt")
    prof = {}
    try:
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith(("#", " ")):
                    k, v = line.split(":", 1)
                    prof[k.strip()] = v.strip()
    except OSError:
        return None, "no ncu summary"
    if prof.get("source_hash") != kernel_source_hash(sources):
        return None, "kernel changed since the ncu capture"
    try:
        return float(prof["dram_bytes_per_launch"]), os.path.relpath(path, ROOT)
    except (KeyError, ValueError):
        return None, "summary without dram_bytes_per_launch"


# ------------------------------------------------------------------ clocks ----
class ClockSampler:
    FIELDS = ("index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception as e:  # nvidia-smi missing: record nothing
            log("clock sampling unavailable:", e)
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

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None}


def clocks_rejected(c) -> bool:
    if any(r in c["reasons"] for r in BAD_REASONS):
        return True
    if c["sm_mhz"] and c["sm_max_mhz"] and c["sm_mhz"] < 0.5 * c["sm_max_mhz"] and "sw_power_cap" not in c["reasons"]:
        return True
    return False


# ------------------------------------------------------------- CPU oracle ----
def cpu_baseline(w, qkv_cpu):
    import oracle
    threads = oracle.default_threads()
    bits = bf16_bits(qkv_cpu)
    t0 = time.perf_counter()
    oracle.fwd(bits, w.B, w.S, w.H, w.D, w.rotary_dim, w.rotary_base, threads=threads)
    dt = time.perf_counter() - t0
    used = min(threads, w.B * w.H)
    return {"value": w.flops / dt / 1e12, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
            "seconds": dt,
            "sample": f"the whole workload ({w.B * w.H} heads x {w.S} rows), one pass, fp64, {used} threads"}


def run_reference(args, w):
    """The oracle as the reference arm: each step is a bounded sample of whole heads (with
    --alibi, of the ALiBi oracle: the same work per head, with the slopes of a model of as
    many heads as the sample holds)."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    threads = oracle.default_threads()
    qkv = make_qkv(w.B, w.S, w.H, w.D, w.seed, w.k_scale)
    bits_all = bf16_bits(qkv)
    head_flops = 2.0 * w.S * w.S * w.D
    alibi = bool(getattr(args, "alibi", False))

    def fwd_heads(bits, n, thr):
        if alibi:
            return oracle.fwd_alibi(bits, 1, w.S, n, w.D, threads=thr)
        return oracle.fwd(bits, 1, w.S, n, w.D, w.rotary_dim, w.rotary_base, threads=thr)

    # calibrate: one head on one thread
    one = bf16_bits(qkv[:1, :, :1].contiguous())
    t0 = time.perf_counter()
    fwd_heads(one, 1, 1)
    per_head_1t = time.perf_counter() - t0
    budget = 120.0
    per_step_budget = budget / max(1, args.steps + args.warmup)
    heads = int(max(1, min(w.B * w.H, per_step_budget / per_head_1t * threads)))
    heads = min(heads, w.H)
    sub = bf16_bits(qkv[:1, :, :heads].contiguous())
    used = min(threads, heads)
    run = lambda: fwd_heads(sub, heads, used)
    flops = heads * head_flops
    sample = f"{heads} of {w.B * w.H} heads x {w.S} rows per step, fp64" + \
        (f", ALiBi with the slopes of a {heads}-head model" if alibi else "")
    # a head runs on one thread: a step takes about per_head_1t * ceil(heads / used)
    if not alibi and per_head_1t * -(-heads // used) > 1.5 * per_step_budget:
        # too long for the budget: evenly spaced query rows of head (0, 0) on all threads,
        # counted at their exact causal cost 4 (i + 1) D, so the whole run stays near it
        one = bf16_bits(qkv[:1, :, :1].contiguous())

        def row_sample(n):
            r_i = np.unique(np.linspace(0, w.S - 1, n).astype(np.int64))
            return r_i, np.stack([np.zeros_like(r_i), np.zeros_like(r_i), r_i], axis=1)

        _, probe = row_sample(16)  # calibrate: 16 evenly spaced rows on all threads
        t0 = time.perf_counter()
        oracle.fwd_rows(one, 1, w.S, 1, w.D, w.rotary_dim, w.rotary_base, probe, threads=threads)
        per16 = time.perf_counter() - t0
        rows_i, rows = row_sample(int(min(w.S, max(1, 16 * per_step_budget / per16))))
        used = min(threads, len(rows_i))
        run = lambda: oracle.fwd_rows(one, 1, w.S, 1, w.D, w.rotary_dim, w.rotary_base, rows, threads=used)
        flops = float(np.sum(4.0 * (rows_i + 1) * w.D))
        heads = 0
        sample = f"{len(rows_i)} evenly spaced query rows of one of {w.B * w.H} heads per step, fp64"
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    del bits_all
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "sample_heads_per_step": heads, "l2": "n/a (CPU)",
                   **({"rotation": "none: ALiBi bias -m_h (i - j) instead (the ALiBi oracle)"} if alibi else {})},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_bwd(args, w):
    """The backward oracle as the reference arm of the backward line: each step is a
    bounded sample of whole heads of batch 0, timed on the host cores."""
    import oracle
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import torch
    threads = oracle.default_threads()
    qkv = make_qkv(w.B, w.S, w.H, w.D, w.seed, w.k_scale)
    dout = torch.randn((w.B, w.S, w.H, w.D), generator=torch.Generator().manual_seed(w.seed + 7)).to(torch.bfloat16)
    head_flops = 5.0 * w.S * w.S * w.D
    t0 = time.perf_counter()  # calibrate: one head on one thread
    oracle.bwd(bf16_bits(qkv[:1, :, :1].contiguous()), bf16_bits(dout[:1, :, :1].contiguous()), 1, w.S, 1, w.D,
               w.rotary_dim, w.rotary_base, threads=1)
    per_head_1t = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    heads = int(max(1, min(w.H, per_step_budget / per_head_1t * threads)))
    q1 = bf16_bits(qkv[:1, :, :heads].contiguous())
    g1 = bf16_bits(dout[:1, :, :heads].contiguous())
    used = min(threads, heads)
    for _ in range(args.warmup):
        oracle.bwd(q1, g1, 1, w.S, heads, w.D, w.rotary_dim, w.rotary_base, threads=used)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.bwd(q1, g1, 1, w.S, heads, w.D, w.rotary_dim, w.rotary_base, threads=used)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = heads * head_flops * args.steps / total / 1e12
    line = {
        "metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "pass": "backward", "sample_heads_per_step": heads, "l2": "n/a (CPU)"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": f"{heads} of {w.B * w.H} heads x {w.S} rows per step, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- rank timing ----
def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's value (a timing); the identity with no process group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (total_ms / 1e3) / 1e12


# ------------------------------------------------------------------ GPU arm ----
def run_ours(args, w):
    import torch
    import causal_rope_self_neox_b300 as na

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        log(f"note: --gpus {args.gpus} but WORLD_SIZE {world}; using WORLD_SIZE")
    dist = None
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    qkv_cpu = make_qkv(w.B, w.S, w.H, w.D, w.seed + rank, w.k_scale)
    qkv = qkv_cpu.to(dev)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    rotation = {"auto": na.NEOX_ROTATION_AUTO, "fused": na.NEOX_ROTATION_FUSED, "pre": na.NEOX_ROTATION_PRE}[args.rotation]
    # the placement the library takes (the header's documented rule for "auto")
    pre = args.rotation == "pre" or (args.rotation == "auto" and w.rotary_dim >= 64 and w.rotary_dim % 16 == 0)

    if args.alibi:
        pre = False

    def step(q=qkv, o=out, l_=lse):
        if args.alibi:
            rc = na.neox_attn_fwd_alibi(q.data_ptr(), w.B, w.S, w.H, w.D, o.data_ptr(), l_.data_ptr(), sh)
        else:
            rc = na.neox_attn_fwd_ex(q.data_ptr(), w.B, w.S, w.H, w.D, w.rotary_dim, w.rotary_base, o.data_ptr(),
                                     l_.data_ptr(), rotation, sh)
        if rc != 0:
            raise na.NeoxAttnError(rc, "neox_attn_fwd_alibi" if args.alibi else "neox_attn_fwd_ex")

    for _ in range(args.warmup):
        flush()
        step()
    na.check_device_error()
    if not bool(torch.isfinite(lse).all()):
        raise RuntimeError("non-finite lse after warm-up")

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(local_rank)
    try:
        u = str(props.uuid)
        gpu_id = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass

    def timed():
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        with ClockSampler(gpu_id) as cs:
            t0 = time.perf_counter()
            for i in range(args.steps):
                flush()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
        barrier()
        ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return ms, wall, cs.summary()

    ms, wall, clocks = timed()
    retried = False
    if clocks_rejected(clocks):
        log("clock record rejected", clocks, "- measuring once more")
        ms, wall, clocks = timed()
        retried = True
    na.check_device_error()

    total_ms = max_over_ranks(sum(ms), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(w.flops, world, args.steps, total_ms)

    # end to end through the public API: every step copies its qkv in from pinned host memory,
    # runs the kernel and copies out + lse back to pinned host memory.  The steps are
    # pipelined on three streams (step k's input copy, step k-1's kernel and step k-2's result
    # copy run at once; two device buffers of each), so a step costs about its slowest copy.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_in = qkv_cpu.pin_memory()
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    host_lse = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    dev_in = [torch.empty_like(qkv) for _ in range(2)]
    dev_out = [torch.empty_like(out) for _ in range(2)]
    dev_lse = [torch.empty_like(lse) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for k in range(n):
            bb = k % 2
            if k >= 2:
                s_in.wait_event(ev_done[bb])  # the kernel of step k-2 has read dev_in[bb]
            with torch.cuda.stream(s_in):
                dev_in[bb].copy_(host_in, non_blocking=True)
            ev_in[bb].record(s_in)
            stream.wait_event(ev_in[bb])
            if k >= 2:
                stream.wait_event(ev_out[bb])  # dev_out[bb] of step k-2 is back on the host
            step(dev_in[bb], dev_out[bb], dev_lse[bb])
            ev_done[bb].record(stream)
            s_out.wait_event(ev_done[bb])
            with torch.cuda.stream(s_out):
                host_out[bb].copy_(dev_out[bb], non_blocking=True)
                host_lse[bb].copy_(dev_lse[bb], non_blocking=True)
            ev_out[bb].record(s_out)

    e2e_run(2)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(e2e_steps)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    na.check_device_error()

    if rank == 0:
        peak, peak_sus, hbm, src = load_peaks()
        per_gpu = w.flops / (ms_per_step / 1e3) / 1e12
        traffic, tsrc = profiled_traffic(("alibi_" if args.alibi else "pre_" if pre else "") + w.name)
        alg_bytes = 2 * w.B * w.S * w.H * 3 * w.D + 2 * w.B * w.S * w.H * w.D + 4 * w.B * w.H * w.S
        D = w.D
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, K x k_scale)",
            "config": {**w.describe(), "l2": L2_NOTE,
                       "rotation": ("none: ALiBi bias -m_h (i - j) instead (neox_attn_fwd_alibi)" if args.alibi else
                                    f"{args.rotation} -> " + ("pre-rotation pass + attention kernel" if pre
                                                              else "fused in the attention kernel")),
                       "parallelism": f"replicas x{world} (each rank its own workload; no collective on the data path)"},
            "roofline": {"bound": "tensor", "achieved": per_gpu, "peak": peak, "unit": "TFLOP/s",
                         "frac": per_gpu / peak, "traffic": traffic,
                         "peak_kind": f"{src} dense bf16 burst (cuBLAS, kernel timed alone)",
                         "frac_of_sustained": per_gpu / peak_sus,
                         "kernel": f"attn_fwd_ws_kernel<D={D}>", "traffic_source": tsrc,
                         "algorithmic_flops_per_launch": w.flops,
                         "hbm_secondary": {"algorithmic_bytes_per_launch": alg_bytes,
                                           "achieved_gbs": alg_bytes / (ms_per_step / 1e3) / 1e9,
                                           "peak_gbs": hbm}},
            "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
            "clocks_retried": retried,
            "e2e": {"value": world * w.flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
                    "d2h_bytes_per_step": host_out[0].numel() * host_out[0].element_size() + host_lse[0].numel() * 4,
                    "steps": e2e_steps, "ms_per_step": e2e_ms,
                    "path": ("pinned host qkv -> device, " + ("neox_attn_fwd_alibi" if args.alibi else "neox_attn_fwd_ex")
                             + " (C ABI), out + lse -> pinned host; steps pipelined on three streams")},
            "gpu_launches": (2 if pre else 1) * args.steps,
            "wall_s_timed_region": wall,
            "kernel_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
        }
        if world == 1 and not args.no_cpu_baseline and not args.alibi:
            line["cpu_baseline"] = cpu_baseline(w, qkv_cpu)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ backward ----
BWD_METRIC = "causal NeoX-rotary attention backward TFLOP/s (5 B H S^2 D algorithmic FLOPs per step)"


def run_bwd(args, w):
    """One step = one neox_attn_bwd call (delta, the tcgen05 backward kernel, dq rotation
    back) on the workload, with the forward's out and lse and a seeded dout resident."""
    import torch
    import causal_rope_self_neox_b300 as na

    if int(os.environ.get("RANK", "0")) != 0:
        return 0  # one GPU: the backward line is a single-replica measurement
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    qkv_cpu = make_qkv(w.B, w.S, w.H, w.D, w.seed, w.k_scale)
    g = torch.Generator().manual_seed(w.seed + 7)
    dout_cpu = torch.randn((w.B, w.S, w.H, w.D), generator=g).to(torch.bfloat16)
    qkv, dout = qkv_cpu.to(dev), dout_cpu.to(dev)
    out, lse = na.attn_fwd(qkv, w.rotary_dim, w.rotary_base)
    dqkv = torch.empty_like(qkv)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flops = 2.5 * w.flops  # five S^2 D contractions over the causal half, against the forward's two

    def step(q=qkv, o=out, l_=lse, gg=dout):
        rc = na.neox_attn_bwd(q.data_ptr(), o.data_ptr(), l_.data_ptr(), gg.data_ptr(), w.B, w.S, w.H, w.D,
                              w.rotary_dim, w.rotary_base, dqkv.data_ptr(), sh)
        if rc != 0:
            raise na.NeoxAttnError(rc, "neox_attn_bwd")

    for _ in range(args.warmup):
        flush()
        step()
    na.check_device_error()
    if not bool(torch.isfinite(dqkv.float()).all()):
        raise RuntimeError("non-finite gradients after warm-up")
    props = torch.cuda.get_device_properties(dev)
    gpu_id = "0"
    try:
        u = str(props.uuid)
        gpu_id = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as cs:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    clocks = cs.summary()
    na.check_device_error()
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_per_step = sum(ms) / len(ms)
    tflops = flops / (ms_per_step / 1e3) / 1e12
    # end to end: qkv, out, lse, dout in from pinned host memory, dqkv back
    hq, ho, hl, hg = qkv_cpu.pin_memory(), out.cpu().pin_memory(), lse.cpu().pin_memory(), dout_cpu.pin_memory()
    hd = torch.empty(dqkv.shape, dtype=dqkv.dtype).pin_memory()
    dq_, do_, dl_, dg_ = torch.empty_like(qkv), torch.empty_like(out), torch.empty_like(lse), torch.empty_like(dout)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for d_, h_ in ((dq_, hq), (do_, ho), (dl_, hl), (dg_, hg)):
            d_.copy_(h_, non_blocking=True)
        step(dq_, do_, dl_, dg_)
        hd.copy_(dqkv, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    na.check_device_error()
    peak, peak_sus, hbm, src = load_peaks()
    traffic, tsrc = profiled_traffic(w.name, "attn_bwd", BWD_KERNEL_SOURCES)
    line = {
        "metric": BWD_METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 qkv and dout)",
        "config": {**w.describe(), "pass": "backward", "l2": L2_NOTE},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "traffic": traffic, "traffic_source": tsrc,
                     "peak_kind": f"{src} dense bf16 burst (cuBLAS, kernel timed alone)",
                     "kernel": f"attn_bwd_kernel<D={w.D}> + delta + dq kernels (all in the timed step)",
                     "algorithmic_flops_per_launch": flops},
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "e2e": {"value": flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, ho, hl, hg)),
                "d2h_bytes_per_step": hd.numel() * 2, "steps": e2e_steps, "ms_per_step": e2e_ms,
                "path": "pinned host qkv, out, lse, dout -> device, neox_attn_bwd (C ABI), dqkv -> pinned host"},
        "gpu_launches": 3 * args.steps,
        "wall_s_timed_region": wall,
        "kernel_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
    }
    if not args.no_cpu_baseline:
        import oracle
        used = oracle.default_threads()
        nh = min(w.H, used)  # one head per host thread, batch 0
        q1 = qkv_cpu[:1, :, :nh].contiguous()
        g1 = dout_cpu[:1, :, :nh].contiguous()
        t0 = time.perf_counter()
        oracle.bwd(bf16_bits(q1), bf16_bits(g1), 1, w.S, nh, w.D, w.rotary_dim, w.rotary_base, used)
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 2.5 * 2 * nh * w.S * w.S * w.D / secs / 1e12, "unit": "TFLOP/s",
                                "cores": used, "kind": "oracle", "seconds": secs,
                                "sample": f"{nh} of the {w.B * w.H} heads (batch 0), fp64, {used} threads"}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------ qkv projection ----
PROJ_METRIC = "fused query_key_value projection (+bias, +rotary epilogue) TFLOP/s and % of B300 bf16 tensor peak"
PROJ_KERNEL_SOURCES = ("qkv_proj.cuh", "attn_common.cuh", "ptx.cuh")


def proj_shape(w):
    """(M tokens, K hidden, N = 3 H D) of the workload's query_key_value projection."""
    return w.B * w.S, w.H * w.D, 3 * w.H * w.D


def run_proj(args, w):
    """One step = one neox_attn_qkv_proj call: x[B*S, hidden] times w[hidden, 3 H D] plus
    bias, the query/key slots rotated in the epilogue (rotary_dim of the workload), packed
    qkv out.  2 M K N algorithmic FLOPs per step."""
    import torch
    import causal_rope_self_neox_b300 as na
    from causal_rope_self_neox_b300.workloads import proj_inputs

    if int(os.environ.get("RANK", "0")) != 0:
        return 0  # one GPU: a single-replica measurement
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    M, K, N = proj_shape(w)
    x_cpu, w_cpu, b_cpu = proj_inputs(w)
    x, wt, b = x_cpu.to(dev), w_cpu.to(dev), b_cpu.to(dev)
    qkv = torch.empty((w.B, w.S, w.H, 3, w.D), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flops = 2.0 * M * K * N

    def step(xx=x, out=qkv):
        rc = na.neox_attn_qkv_proj(xx.data_ptr(), wt.data_ptr(), b.data_ptr(), w.B, w.S, K, w.H, w.D, w.rotary_dim,
                                   w.rotary_base, out.data_ptr(), sh)
        if rc != 0:
            raise na.NeoxAttnError(rc, "neox_attn_qkv_proj")

    for _ in range(args.warmup):
        flush()
        step()
    na.check_device_error()
    if not bool(torch.isfinite(qkv.float()).all()):
        raise RuntimeError("non-finite projection after warm-up")
    props = torch.cuda.get_device_properties(dev)
    gpu_id = "0"
    try:
        u = str(props.uuid)
        gpu_id = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as cs:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    clocks = cs.summary()
    na.check_device_error()
    ms = [a.elapsed_time(b_) for a, b_ in zip(starts, ends)]
    ms_per_step = sum(ms) / len(ms)
    tflops = flops / (ms_per_step / 1e3) / 1e12
    # end to end: the token rows in from pinned host memory, the packed qkv back; the
    # weight and bias stay resident, as a model's parameters do
    hx = x_cpu.pin_memory()
    hq = torch.empty(qkv.shape, dtype=qkv.dtype).pin_memory()
    dx = torch.empty_like(x)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        dx.copy_(hx, non_blocking=True)
        step(dx)
        hq.copy_(qkv, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    na.check_device_error()
    peak, peak_sus, hbm, src = load_peaks()
    traffic, tsrc = profiled_traffic(w.name, "qkv_proj", PROJ_KERNEL_SOURCES)
    line = {
        "metric": PROJ_METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded x ~ N(0,1), w ~ N(0,1)/sqrt(hidden), bias ~ N(0,0.25), bf16)",
        "config": {**w.describe(), "pass": "qkv_proj", "M": M, "hidden": K, "N": N, "l2": L2_NOTE},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "traffic": traffic, "traffic_source": tsrc,
                     "peak_kind": f"{src} dense bf16 burst (cuBLAS, kernel timed alone)",
                     "kernel": f"qkv_proj_kernel<NT={192 if w.D == 96 else 256}>",
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": 2 * (M * K + K * N + N + M * N)},
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "e2e": {"value": flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hq.numel() * 2, "steps": e2e_steps,
                "ms_per_step": e2e_ms,
                "path": "pinned host x -> device, neox_attn_qkv_proj (C ABI), qkv -> pinned host; w, bias resident"},
        "gpu_launches": args.steps,
        "wall_s_timed_region": wall,
        "kernel_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
    }
    if not args.no_cpu_baseline:
        import oracle
        used = oracle.default_threads()
        rows = list(range(min(M, 2 * used)))  # a bounded sample of token rows
        t0 = time.perf_counter()
        oracle.qkv_proj_rotated(bf16_bits(x_cpu), bf16_bits(w_cpu), bf16_bits(b_cpu), w.B, w.S, w.H, w.D,
                                w.rotary_dim, w.rotary_base, rows=rows, threads=used)
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 2.0 * len(rows) * K * N / secs / 1e12, "unit": "TFLOP/s", "cores": used,
                                "kind": "oracle", "seconds": secs,
                                "sample": f"{len(rows)} of the {M} token rows, fp64, {used} threads"}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_proj(args, w):
    """The projection oracle as the reference arm: each step a bounded sample of token rows."""
    import oracle
    from causal_rope_self_neox_b300.workloads import proj_inputs
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    threads = oracle.default_threads()
    M, K, N = proj_shape(w)
    x_cpu, w_cpu, b_cpu = proj_inputs(w)
    xb, wb, bb = bf16_bits(x_cpu), bf16_bits(w_cpu), bf16_bits(b_cpu)
    t0 = time.perf_counter()  # calibrate: one row on one thread
    oracle.qkv_proj(xb, wb, bb, rows=[0], threads=1)
    per_row_1t = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(M, per_step_budget / per_row_1t * threads)))
    rows = list(range(n))
    used = min(threads, n)
    run = lambda: oracle.qkv_proj_rotated(xb, wb, bb, w.B, w.S, w.H, w.D, w.rotary_dim, w.rotary_base, rows=rows,
                                          threads=used)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2.0 * n * K * N * args.steps / total / 1e12
    line = {
        "metric": PROJ_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "pass": "qkv_proj", "M": M, "hidden": K, "N": N, "sample_rows_per_step": n,
                   "l2": "n/a (CPU)"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": f"{n} of {M} token rows per step, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------- decode workloads ----
DECODE_METRIC = "incremental decode: KV-cache GB/s read per step (and tokens/s)"


def run_reference_decode(args, w):
    """The fp64 decode oracle as the reference arm of a decode line: each step decodes a
    bounded sample of whole sequences (every head, every cached key) on the host cores, so
    that the run stays within about two minutes; GB/s counts the sample's share of the
    step's algorithmic bytes."""
    import oracle
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    new_cpu, kc_cpu, vc_cpu = make_decode_inputs(w.B, w.H, w.Smax, w.D, w.seed)
    threads = oracle.default_threads()
    alg_bytes = w.cache_bytes_read + w.B * w.H * 3 * w.D * 2 + w.B * w.H * w.D * 2 * 2 + w.B * w.H * w.D * 2 \
        + w.B * w.H * 4
    per_seq_bytes = alg_bytes / w.B

    def run(nseq, used):
        oracle.decode(bf16_bits(new_cpu[:nseq].contiguous()), bf16_bits(kc_cpu[:nseq].contiguous()),
                      bf16_bits(vc_cpu[:nseq].contiguous()), [w.pos] * nseq, nseq, w.H, w.Smax, w.D, w.rotary_dim,
                      w.rotary_base, used)

    t0 = time.perf_counter()  # calibrate: one sequence
    run(1, threads)
    per_seq = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    nseq = int(max(1, min(w.B, per_step_budget / max(per_seq, 1e-9))))
    for _ in range(args.warmup):
        run(nseq, threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run(nseq, threads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = nseq * per_seq_bytes * args.steps / total / 1e9
    sample = f"{nseq} of {w.B} sequences per step (all {w.H} heads, {w.pos + 1} keys each), fp64"
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "sample_sequences_per_step": nseq, "l2": "n/a (CPU)"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, w):
    """One step = one neox_attn_decode call: a new token for each of B sequences at
    position pos against a cache of pos tokens (every cached key and value read once)."""
    import torch
    import causal_rope_self_neox_b300 as na

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    new_cpu, kc_cpu, vc_cpu = make_decode_inputs(w.B, w.H, w.Smax, w.D, w.seed)
    new, kc, vc = new_cpu.to(dev), kc_cpu.to(dev), vc_cpu.to(dev)
    pos_cpu = torch.full((w.B,), w.pos, dtype=torch.int32)
    pos = pos_cpu.to(dev)
    out = torch.empty((w.B, w.H, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(n=new, p_=pos):
        rc = na.neox_attn_decode(n.data_ptr(), kc.data_ptr(), vc.data_ptr(), p_.data_ptr(), w.B, w.H, w.Smax, w.D,
                                 w.rotary_dim, w.rotary_base, out.data_ptr(), lse.data_ptr(), sh)
        if rc != 0:
            raise na.NeoxAttnError(rc, "neox_attn_decode")

    for _ in range(args.warmup):
        flush()
        step()
    na.check_device_error()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = "0"
    try:
        u = str(props.uuid)
        gpu_id = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as cs:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    clocks = cs.summary()
    na.check_device_error()
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_per_step = sum(ms) / len(ms)
    # algorithmic bytes: cached K and V rows read, the new token's projections read, its
    # k and v appended, out and lse written
    alg_bytes = w.cache_bytes_read + w.B * w.H * 3 * w.D * 2 + w.B * w.H * w.D * 2 * 2 + w.B * w.H * w.D * 2 \
        + w.B * w.H * 4
    gbs = alg_bytes / (ms_per_step / 1e3) / 1e9
    # end to end: the new token's projections and positions in, out and lse back (the cache stays resident)
    host_new, host_pos = new_cpu.pin_memory(), pos_cpu.pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dn, dp = torch.empty_like(new), torch.empty_like(pos)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        dn.copy_(host_new, non_blocking=True)
        dp.copy_(host_pos, non_blocking=True)
        step(dn, dp)
        host_out.copy_(out, non_blocking=True)
        host_lse.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    na.check_device_error()
    _, _, hbm, src = load_peaks()
    traffic, tsrc = profiled_traffic(w.name, "attn_decode", DEC_KERNEL_SOURCES)
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 caches and new tokens)",
        "tokens_per_s": w.B / (ms_per_step / 1e3),
        "config": {**w.describe(), "l2": L2_NOTE},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": traffic, "traffic_source": tsrc, "peak_kind": f"{src} HBM copy bandwidth",
                     "kernel": f"attn_decode_kernel<D={w.D}> (one launch per step)",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "e2e": {"value": alg_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": host_new.numel() * 2 + host_pos.numel() * 4,
                "d2h_bytes_per_step": host_out.numel() * 2 + host_lse.numel() * 4, "steps": e2e_steps,
                "ms_per_step": e2e_ms,
                "path": "pinned host new-token qkv + positions -> device, neox_attn_decode (C ABI), out + lse -> pinned host"},
        "gpu_launches": args.steps,
        "wall_s_timed_region": wall,
        "kernel_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
    }
    if not args.no_cpu_baseline:
        import oracle
        nb_, kb, vb = bf16_bits(new_cpu), bf16_bits(kc_cpu), bf16_bits(vc_cpu)
        used = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.decode(nb_, kb, vb, [w.pos] * w.B, w.B, w.H, w.Smax, w.D, w.rotary_dim, w.rotary_base, used)
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": alg_bytes / secs / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
                                "seconds": secs,
                                "sample": f"the whole step ({w.B * w.H} heads x {w.pos + 1} keys), fp64, {used} threads"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS), default="neox20b")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--alibi", action="store_true",
                    help="time the ALiBi forward (neox_attn_fwd_alibi) on the workload's shape instead")
    ap.add_argument("--rotation", choices=["auto", "fused", "pre"], default="auto",
                    help="where the forward applies the rotary embedding (neox_attn_fwd_ex placement)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "proj"], default="fwd",
                    help="bwd: time the backward (neox_attn_bwd) on a prefill workload; proj: the "
                         "query_key_value projection that feeds it (neox_attn_qkv_proj)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in DECODE_WORKLOADS:  # the decode path (a separate op, its own metric)
        if args.impl == "reference":
            return run_reference_decode(args, DECODE_WORKLOADS[args.workload])
        return run_decode(args, DECODE_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.pass_ == "bwd":
        if args.impl == "reference":
            return run_reference_bwd(args, w)
        return run_bwd(args, w)
    if args.pass_ == "proj":
        if args.impl == "reference":
            return run_reference_proj(args, w)
        return run_proj(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
