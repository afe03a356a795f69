#!/usr/bin/env python
"""Benchmark of the LoCo data-parallel hot path on GB300.

Workload (default): a Llama-2-7B-shaped bf16 gradient bucket (6,738,415,616
elements), 4-bit codes, block 256, W = 8 simulated ranks held as 8 packed
buffers in one HBM.  One step is one pass of the whole hot path:

  loco_compress      rank 0's bucket: compensate, quantise, pack, error update
  loco_decode_reduce the 8 ranks' packed buckets -> fp32 mean
  loco_adam_step     the same 8 buffers decoded, averaged and fed to Adam(W)

Ranks 1..7's packed buffers are produced before timing by compressing their
own seeded gradients.  Inputs (176 GB live) are far larger than L2, so no L2
flush is needed between steps.

value = gradient bytes processed per second: compress counts N*2 bytes (bf16
gradient), decode-reduce and the fused Adam each count W*N*2 bytes (the
gradient-equivalent of the W contributions they consume).  Decode-reduce and
the fused Adam decode the same W packed buffers, so those W*N*2 bytes are
counted twice, and the mean that decode-reduce writes is not consumed inside
the timed step (the fused step re-derives it): value is the metric's
definitional sum, not a traffic figure.  The traffic figures are each
kernel's roofline fraction (algorithmic HBM bytes / its CUDA-event time / the
measured HBM copy bandwidth) and, for the whole step, "step_hbm": all
kernels' algorithmic bytes / ms_per_step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl loco|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step on a one-GPU-per-process box); value sums the
ranks' units over the slowest rank's time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compress & decode-reduce GB/s of gradient processed; % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e datasheet rate, shown beside the measured-peak fraction


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="loco", choices=["loco", "reference"])
    ap.add_argument("--workload", default="llama2-7b",
                    help="llama2-7b (default), tinyllama, mixtral, or flat:<log2 n> (bf16, 4-bit, block 256, W 8)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="host-to-device copy streams of the end-to-end leg (inputs split across them)")
    ap.add_argument("--error-storage", default="fp32", choices=["fp32", "int8"],
                    help="compensation error kept in fp32 (default) or as int8 codes + per-block step")
    ap.add_argument("--optimizer", default="adam", choices=["adam", "sgd"],
                    help="optimizer fused with the receiver average (default adam)")
    ap.add_argument("--param-bf16", action="store_true", help="also write the bf16 copy of the updated parameters")
    ap.add_argument("--fixed-scale", type=float, default=None,
                    help="paper-literal fixed quantisation scale s (e.g. 524288 = 2^19) instead of blockwise absmax")
    ap.add_argument("--bits", type=int, default=None, choices=[4, 8], help="override the workload's code width")
    ap.add_argument("--block", type=int, default=None, help="override the workload's scale block (power of two)")
    ap.add_argument("--ranks", type=int, default=None, help="override the workload's W simulated ranks (1..16)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="leave out the timed oracle sample (for sweeps; the default run reports it)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- workload

def workload(name: str, bits=None, block=None, ranks=None):
    """The named workload, with its code width, block or rank count replaced
    where given (the name then records the change)."""
    import dataclasses
    from bit_gradient_compression_gb300 import workloads as wl
    if name == "llama2-7b":
        w = wl.LLAMA2_7B
    elif name == "tinyllama":
        w = wl.TINYLLAMA
    elif name == "mixtral":
        w = wl.MIXTRAL_MOE
    elif name.startswith("flat:"):
        import torch
        n = 1 << int(name.split(":")[1])
        w = wl.Workload(f"flat-bf16-2^{name.split(':')[1]}", n, torch.bfloat16, 4, 256, 8, 1, "flat")
    else:
        raise SystemExit(f"unknown workload {name}")
    over = {k: v for k, v in (("bits", bits), ("block", block), ("W", ranks)) if v is not None and v != getattr(w, k)}
    if over:
        tag = ",".join(f"{k}={v}" for k, v in over.items())
        w = dataclasses.replace(w, name=f"{w.name}[{tag}]", **over)
    return w


def kernel_bytes(n, gsize, bits, block, W, e8=False, optimizer="adam", bf16_out=False):
    nb = -(-n // block)
    cb = nb * block * bits // 8
    sb = nb * 4
    opt_state = 24 if optimizer == "adam" else 8   # param (+ m, v) read and written
    return {
        # int8 error: codes read + written (2 B) and the block step read + written; fp32: 4 B read + 4 B written
        "compress": n * gsize + (2 * n + 2 * sb if e8 else 8 * n) + cb + sb,
        "decode_reduce": W * (cb + sb) + 4 * n,
        optimizer: W * (cb + sb) + opt_state * n + (2 * n if bf16_out else 0),
    }


def grad_units(n, gsize, W, optimizer="adam"):
    return {"compress": n * gsize, "decode_reduce": W * n * gsize, optimizer: W * n * gsize}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each timed kernel (and its launcher) is built from; abi.cu is host validation.
_COMMON = ("device_common.cuh", "loco_internal.h")
KERNEL_SOURCES = {
    "compress": ("compress.cu",) + _COMMON,
    "decode_reduce": ("decode_reduce.cu", "receiver_common.cuh") + _COMMON,
    "adam": ("adam.cu", "receiver_common.cuh") + _COMMON,
    "sgd": ("sgd.cu", "receiver_common.cuh") + _COMMON,
}


def code_of(text: str) -> str:
    """C/C++ source with comments removed and whitespace collapsed: what a change
    to a kernel's code alters and a change to its comments does not."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(kernel: str, read=None) -> str:
    """Hash of the code (comments aside) of the sources one kernel is built from,
    stored with its ncu counters.  read(name) -> text overrides reading the file."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_gradient_compression_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        if read is None:
            with open(os.path.join(csrc, f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(f.encode() + code_of(text).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, units: int, n_elems: int, workload_name: str):
    """DRAM bytes per launch of this kernel on this workload from the committed
    ncu capture (profiles/ncu_traffic.json); None for another workload or when
    the kernel sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if (d.get("workload") != workload_name or d.get("n_elements") != n_elems or kernel not in d.get("kernels", {})
            or d["kernels"][kernel].get("source_hash") != source_hash(kernel)):
        return None
    return d["kernels"][kernel]["dram_bytes"]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", self.gpu_id],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        busy = [s for s, p in zip(sm, power) if p > 0] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def host_mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except Exception:
        return None
    return None


def gpu_uuid(dev) -> str:
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        return "GPU-" + str(u)
    except Exception:
        return str(dev.index or 0)


# ----------------------------------------------------------------------------- CPU oracle (baseline)

def prefix_layout(layout, count):
    out, tot = [], 0
    for name, n in layout:
        if tot >= count:
            break
        take_n = min(n, count - tot)
        out.append((name, take_n))
        tot += take_n
    return out


def oracle_sample(w, S, seed=7):
    """Host inputs for an S-element prefix of the workload: rank 0's gradient,
    the error, W ranks' packed buffers (ranks 1.. compressed by the oracle,
    untimed), parameters and Adam state."""
    import numpy as np
    import torch

    import oracle
    from bit_gradient_compression_gb300 import workloads as wl

    def grad(r):
        t = torch.empty(S, dtype=w.grad_dtype)
        if w.kind == "llm":
            lay = prefix_layout(w.layout, S)
            sig_rng = np.random.default_rng(wl.seed_for(seed, 1, r))
            sig = 10.0 ** sig_rng.uniform(-5.0, -2.0, size=len(w.layout))[:len(lay)]
            gen = torch.Generator().manual_seed(wl.seed_for(seed, 1, r))
            off = 0
            for (nm, n), s in zip(lay, sig):
                t[off:off + n].copy_(torch.randn(n, generator=gen) * float(s))
                off += n
        else:
            w.fill(t, wl.seed_for(seed, 1, r))
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16).copy()
        return t.numpy().copy()

    codes, scales = [], []
    for r in range(1, w.W):
        c, s = oracle.compress(grad(r), np.zeros(S, np.float32), 1, bits=w.bits, block=w.block, beta=0.9,
                               kappa=4.0, threads=os.cpu_count() or 1)
        codes.append(c)
        scales.append(s)
    g0 = grad(0)
    e = np.zeros(S, np.float32)
    rng = np.random.default_rng(3)
    p = rng.uniform(-0.02, 0.02, S).astype(np.float32)
    return g0, e, codes, scales, p, np.zeros(S, np.float32), np.zeros(S, np.float32)


def oracle_step(w, S, inp, step, threads, optimizer="adam"):
    import oracle
    g0, e, codes, scales, p, m, v = inp
    c0, s0 = oracle.compress(g0, e, step, bits=w.bits, block=w.block, beta=0.9, kappa=4.0, reset_period=512,
                             threads=threads)
    allc, alls = [c0] + codes, [s0] + scales
    oracle.decode_reduce(allc, alls, S, bits=w.bits, block=w.block, threads=threads)
    if optimizer == "sgd":
        oracle.sgd_step(allc, alls, S, p, bits=w.bits, block=w.block, lr=1e-3, threads=threads)
    else:
        oracle.adam_step(allc, alls, S, p, m, v, step, bits=w.bits, block=w.block, lr=1e-4, beta1=0.9, beta2=0.95,
                         eps=1e-8, threads=threads)


def cpu_baseline(w, S, steps, warmup, optimizer="adam"):
    """Times the oracle, as it stands, on all host cores over an S-element sample
    of the step (fp32 error, absmax scale, the given optimizer)."""
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    inp = oracle_sample(w, S)
    gsize = 2 if "bf16" in str(w.grad_dtype) else 4
    for k in range(warmup):
        oracle_step(w, S, inp, k + 1, threads, optimizer)
    t0 = time.perf_counter()
    for k in range(steps):
        oracle_step(w, S, inp, warmup + k + 1, threads, optimizer)
    dt = (time.perf_counter() - t0) / steps
    units = sum(grad_units(S, gsize, w.W, optimizer).values())
    # the same oracle on one thread, over a smaller prefix (a few hundred ms of work)
    S1 = min(S, 1 << 24)
    inp1 = inp if S1 == S else oracle_sample(w, S1)
    t1 = time.perf_counter()
    oracle_step(w, S1, inp1, warmup + steps + 1, 1, optimizer)
    dt1 = time.perf_counter() - t1
    units1 = sum(grad_units(S1, gsize, w.W, optimizer).values())
    return {"value": units / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {S:,} elements of the {w.name} bucket (rank 0 compress + decode-reduce + "
                      f"{'SGD' if optimizer == 'sgd' else 'Adam'} over W={w.W} ranks, fp32 error, absmax scale), "
                      f"{steps} timed step(s) after {warmup} warm-up, same gradient law on host",
            "ms_per_step": dt * 1e3,
            "single_thread": {"value": units1 / dt1 / 1e9, "unit": UNIT, "cores": 1,
                              "sample": f"first {S1:,} elements, one step", "ms_per_step": dt1 * 1e3}}


# ----------------------------------------------------------------------------- multi-rank

def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over all ranks (a no-op on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def all_ranks_agree(ok: bool, device) -> bool:
    """True only if `ok` holds on every rank (a no-op on one rank), so that a
    leg with collectives inside is entered by all ranks or by none."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return bool(ok)
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def whole_job_value(units_per_rank_step: int, world: int, ms_per_step_max: float) -> float:
    """Units every rank processed in one step, over the slowest rank's step time (GB/s)."""
    return world * units_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


# ----------------------------------------------------------------------------- GPU arm

def run_e2e(args, L, w, cfg, n, nb, cb, g, compress, update, codes, scales, mean, world, dist, h2d, d2h):
    """The step through the public API with its inputs coming from page-locked
    host memory and its output (rank 0's packed buffer, the bytes a rank sends)
    going back to it, every step, inside the timed region.

    Copies run on their own streams and overlap the kernels of the previous
    step: device inputs are double-buffered (set k % 2), and event waits order
    every copy against the kernels that read or write the same buffers."""
    import torch
    W = len(codes)
    dev = g.device
    comp = torch.cuda.current_stream()
    nS = max(1, args.e2e_copy_streams)
    s_ins, s_out = [torch.cuda.Stream() for _ in range(nS)], torch.cuda.Stream()
    hosts = []

    def host_like(t):
        # page-locked at allocation (measured ~3 % faster to copy than registering pageable memory)
        h = torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
        hosts.append(h)
        return h

    g_h = host_like(g)
    g_h.copy_(g)
    codes_h = [host_like(codes[r]) for r in range(1, W)]
    scales_h = [host_like(scales[r]) for r in range(1, W)]
    for r in range(1, W):
        codes_h[r - 1].copy_(codes[r])
        scales_h[r - 1].copy_(scales[r])
    out_c, out_s = host_like(codes[0]), host_like(scales[0])
    # second device set: gradient, ranks 1..W-1 packed buffers, rank 0 output
    sets = [(g, codes, scales),
            (torch.empty_like(g), [torch.empty_like(c) for c in codes], [torch.empty_like(x) for x in scales])]
    torch.cuda.synchronize()
    # This machine's host link, measured on the same page-locked buffer just before
    # the timed region (it varies between boxes), reported beside the e2e number.
    probe_n = min(g_h.numel() * g_h.element_size(), 4 << 30)
    src = g_h.view(torch.uint8)[:probe_n]
    dst = g.view(torch.uint8)[:probe_n]
    link = []
    for dst_, src_ in ((dst, src), (src, dst)):
        dst_.copy_(src_, non_blocking=True)
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(3):  # a single copy can be far slower than the link sustains: keep the best of three
            a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(comp)
            dst_.copy_(src_, non_blocking=True)
            b0.record(comp)
            torch.cuda.synchronize()
            best = max(best, probe_n / (a0.elapsed_time(b0) * 1e-3) / 1e9)
        link.append(best)
    # the whole input set of one step, copied once as the loop copies it (one pass per buffer, in
    # order, on the first copy stream): what the loop's inputs alone take on this machine
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(s_ins[0])
    with torch.cuda.stream(s_ins[0]):
        sets[1][0].copy_(g_h, non_blocking=True)
        for r in range(1, W):
            sets[1][1][r].copy_(codes_h[r - 1], non_blocking=True)
            sets[1][2][r].copy_(scales_h[r - 1], non_blocking=True)
    b0.record(s_ins[0])
    torch.cuda.synchronize()
    full_set_GBps = h2d / (a0.elapsed_time(b0) * 1e-3) / 1e9
    # the same link with the copy split over the copy streams, as the loop issues it
    parts = [(i * probe_n // nS, (i + 1) * probe_n // nS) for i in range(nS)]
    best = 0.0
    for _ in range(3):
        a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(comp)
        for st, (lo, hi) in zip(s_ins, parts):
            st.wait_event(a0)
            with torch.cuda.stream(st):
                dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
        for st in s_ins:
            comp.wait_stream(st)
        b0.record(comp)
        torch.cuda.synchronize()
        best = max(best, probe_n / (a0.elapsed_time(b0) * 1e-3) / 1e9)
    link.append(best)
    g.copy_(g_h)
    torch.cuda.synchronize()
    K = args.e2e_steps
    ev = lambda: torch.cuda.Event()
    comp_done, c0_done, out_done = [[ev() for _ in range(K)] for _ in range(3)]
    g_done, in_done = [[[ev() for _ in range(nS)] for _ in range(K)] for _ in range(2)]
    # each copy stream takes one contiguous part of the gradient, then its share of ranks 1..W-1
    gparts = [(i * n // nS, (i + 1) * n // nS) for i in range(nS)]
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for st in s_ins:
        st.wait_event(a)
    s_out.wait_event(a)
    for k in range(K):
        gk, ck, sk = sets[k % 2]
        for i, st in enumerate(s_ins):         # inputs of step k
            with torch.cuda.stream(st):
                if k >= 2:
                    st.wait_event(comp_done[k - 2])
                lo, hi = gparts[i]
                gk[lo:hi].copy_(g_h[lo:hi], non_blocking=True)
                g_done[k][i].record(st)
        for r in range(1, W):
            st = s_ins[(r - 1) % nS]
            with torch.cuda.stream(st):
                ck[r].copy_(codes_h[r - 1], non_blocking=True)
                sk[r].copy_(scales_h[r - 1], non_blocking=True)
        for i, st in enumerate(s_ins):
            in_done[k][i].record(st)
        for e_ in g_done[k]:
            comp.wait_event(e_)
        if k >= 2:
            comp.wait_event(out_done[k - 2])   # rank 0's buffer of set k % 2 has left
        compress(gk, k + 1, ck[0], sk[0], stream=comp)
        c0_done[k].record(comp)
        for e_ in in_done[k]:
            comp.wait_event(e_)                # ranks 1..W-1 arrived
        L.loco_decode_reduce(cfg, ck, sk, n, mean, stream=comp)
        update(ck, sk, k + 1, stream=comp)
        comp_done[k].record(comp)
        with torch.cuda.stream(s_out):         # output of step k
            s_out.wait_event(c0_done[k])
            out_c.copy_(ck[0], non_blocking=True)
            out_s.copy_(sk[0], non_blocking=True)
            out_done[k].record(s_out)
    comp.wait_event(out_done[K - 1])
    for e_ in in_done[K - 1]:
        comp.wait_event(e_)
    b.record(comp)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    hosts.clear()
    del sets[1]
    return (ms, h2d, d2h, link + [full_set_GBps])


def run_loco(args, rank, world):
    import torch
    import torch.distributed as dist

    from bit_gradient_compression_gb300 import loco as L
    from bit_gradient_compression_gb300 import workloads as wl

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.workload, args.bits, args.block, args.ranks)
    n, bits, block, W = w.n, w.bits, w.block, w.W
    gsize = 2 if w.grad_dtype == torch.bfloat16 else 4
    # beta weights the previous error; the 8-bit storage needs weight on the new error (see loco.h)
    cfg = L.make_config(bits=bits, block=block, beta=0.9 if args.error_storage == "fp32" else 0.1,
                        err_scale_mult=4.0, reset_period=512, fixed_scale=args.fixed_scale)
    opt = args.optimizer
    pb16 = torch.empty(n, dtype=torch.int16, device=dev) if args.param_bf16 else None
    hp = L.make_adam(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)

    # ---- resident buffers (setup, untimed)
    e8 = args.error_storage == "int8"
    g = torch.empty(n, dtype=w.grad_dtype, device=dev)
    if e8:
        e = (torch.zeros(n, dtype=torch.int8, device=dev), torch.zeros(nb, dtype=torch.float32, device=dev))
    else:
        e = torch.zeros(n, dtype=torch.float32, device=dev)

    def compress(grad, step, c, sc, stream=None):
        if e8:
            L.loco_compress_e8(cfg, grad, e[0], e[1], step, c, sc, stream=stream)
        else:
            L.loco_compress(cfg, grad, e, step, c, sc, stream=stream)

    def zero_error():
        if e8:
            e[0].zero_()
            e[1].zero_()
        else:
            e.zero_()
    codes = [torch.empty(cb, dtype=torch.uint8, device=dev) for _ in range(W)]
    scales = [torch.empty(nb, dtype=torch.float32, device=dev) for _ in range(W)]
    for r in range(1, W):
        w.fill(g, wl.seed_for(7, 1, r))
        zero_error()
        compress(g, 1, codes[r], scales[r])
    w.fill(g, wl.seed_for(7, 1, 0))
    zero_error()
    mean = torch.empty(n, dtype=torch.float32, device=dev)
    param = wl.fill_uniform(torch.empty(n, device=dev), 3, -0.02, 0.02)
    m = torch.zeros(n, device=dev) if opt == "adam" else None
    v = torch.zeros(n, device=dev) if opt == "adam" else None
    torch.cuda.synchronize()

    def update(ck, sk, k, stream=None):
        if opt == "sgd":
            L.loco_sgd_step(cfg, ck, sk, n, param, 1e-3, param_bf16=pb16, stream=stream)
        elif pb16 is not None:
            L.loco_adam_step_bf16(cfg, ck, sk, n, param, m, v, pb16, hp, k, stream=stream)
        else:
            L.loco_adam_step(cfg, ck, sk, n, param, m, v, hp, k, stream=stream)

    stream = torch.cuda.current_stream()
    step_no = [0]

    def one_step(ev=None):
        step_no[0] += 1
        k = step_no[0]
        if ev:
            ev[0].record(stream)
        compress(g, k, codes[0], scales[0])
        if ev:
            ev[1].record(stream)
        L.loco_decode_reduce(cfg, codes, scales, n, mean)
        if ev:
            ev[2].record(stream)
        update(codes, scales, k)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_uuid(dev)) if rank == 0 else None
    if clocks:
        clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        one_step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = t_start.elapsed_time(t_end)
    per_kernel = {
        "compress": statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs),
        "decode_reduce": statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs),
        opt: statistics.mean(ev[2].elapsed_time(ev[3]) for ev in evs),
    }

    # ---- e2e: host buffers in page-locked memory, copies inside the timed region
    e2e = None
    h2d = n * gsize + (W - 1) * (cb + 4 * nb)
    d2h = cb + 4 * nb
    need = h2d + d2h
    avail = host_mem_available()
    local_ranks = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))  # ranks sharing this host's memory
    e2e_skip = None
    if args.e2e_steps <= 0:
        e2e_skip = "disabled"
    elif avail is not None and need > 0.6 * avail / local_ranks:
        e2e_skip = (f"host buffers need {need / 1e9:.1f} GB per rank, {avail / 1e9:.1f} GB available "
                    f"for {local_ranks} rank(s)")
    else:
        free_dev = torch.cuda.mem_get_info(dev)[0]
        if h2d + d2h > 0.9 * free_dev:
            e2e_skip = f"second device buffer set needs {(h2d + d2h) / 1e9:.1f} GB, {free_dev / 1e9:.1f} GB free"
    if not all_ranks_agree(e2e_skip is None, dev) and e2e_skip is None:
        e2e_skip = "skipped on another rank"
    if e2e_skip is None:
        e2e = run_e2e(args, L, w, cfg, n, nb, cb, g, compress, update, codes, scales, mean, world, dist, h2d, d2h)

    units_step = sum(grad_units(n, gsize, W, opt).values())
    t_ms, e2e_max = max_over_ranks([total_ms / args.steps, e2e[0] if e2e else 0.0], dev)
    if e2e:
        e2e = (e2e_max,) + tuple(e2e[1:])
    if rank != 0:
        return None

    hbm, hbm_kind = peaks()
    default_step = not e8 and opt == "adam" and pb16 is None and args.fixed_scale is None
    kb = kernel_bytes(n, gsize, bits, block, W, e8, opt, pb16 is not None)
    step_bytes = sum(kb.values())
    roof = {}
    for k, ms in per_kernel.items():
        ach = kb[k] / (ms * 1e-3) / 1e9
        roof[k] = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                   "frac": round(ach / hbm, 4), "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4), "ms": round(ms, 4),
                   "traffic": ncu_traffic(k, kb[k], n, w.name) if default_step else None,
                   "algorithmic_bytes": kb[k],
                   "grad_GBps": round(grad_units(n, gsize, W, opt)[k] / (ms * 1e-3) / 1e9, 1),
                   "peak_source": f"{hbm_kind} (MEASURED_PEAKS.json hbm_gbs)" if hbm_kind == "measured" else
                   "fallback"}
    dominant = max(per_kernel, key=per_kernel.get)
    value = whole_job_value(units_step, world, t_ms)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_elements": n, "grad_dtype": "bf16" if gsize == 2 else "fp32",
                   "bits": bits, "block": block, "W": W, "beta": cfg.beta, "kappa": 4.0,
                   "error_storage": args.error_storage, "optimizer": opt,
                   "step": ("loco_compress_e8" if e8 else "loco_compress") + "(rank 0) + loco_decode_reduce(W) + "
                           + {"adam": "loco_adam_step" + ("_bf16" if pb16 is not None else ""),
                              "sgd": "loco_sgd_step" + (" (bf16 copy)" if pb16 is not None else "")}[opt] + "(W)",
                   "scale": "absmax" if args.fixed_scale is None else f"fixed s={args.fixed_scale:g}",
                   "l2": "inputs larger than L2 (no flush needed)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU, W ranks simulated in HBM"},
        "roofline": dict(roof[dominant], kernel=dominant),
        "roofline_kernels": roof,
        "step_hbm": {"algorithmic_bytes": step_bytes, "achieved": round(step_bytes / (t_ms * 1e-3) / 1e9, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(step_bytes / (t_ms * 1e-3) / 1e9 / hbm, 4),
                     "what": "algorithmic HBM bytes of all kernels of one step / ms_per_step"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }
    if e2e_skip:
        out["e2e"] = {"value": None, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "skipped": e2e_skip}
    if e2e:
        e2e_ms, h2d, d2h, link = e2e
        out["e2e"] = {"value": round(whole_job_value(units_step, world, e2e_ms), 1), "unit": UNIT,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                      "steps": args.e2e_steps,
                      "host_link_GBps": {"h2d": round(link[0], 1), "d2h": round(link[1], 1),
                                         f"h2d_{args.e2e_copy_streams}_streams": round(link[2], 1),
                                         "h2d_step_inputs": round(link[3], 1)},
                      "copy_streams": args.e2e_copy_streams,
                      "copy_bound_ms_per_step": round(h2d / (max(link[0], link[2]) * 1e9) * 1e3, 1),
                      "achieved_h2d_GBps": round(h2d / (e2e_ms * 1e-3) / 1e9, 1),
                      "what": "page-locked host -> device: rank 0 gradient + ranks 1..W-1 packed buffers "
                              "(split over the copy streams); device -> page-locked host: rank 0's packed buffer; "
                              "copies on their own streams overlap the previous step's kernels (double-buffered "
                              "device inputs)"}
    return out


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        w = workload(args.workload, args.bits, args.block, args.ranks)
        S = min(w.n, 1 << 25)
        cb = cpu_baseline(w, S, args.steps, args.warmup)
        out = {"impl": "reference", "metric": METRIC, "value": round(cb["value"], 3), "unit": UNIT,
               "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(cb["ms_per_step"], 3), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f32", "data": "synthetic",
               "config": {"workload": w.name, "n_elements": w.n, "sample_elements": S, "bits": w.bits,
                          "block": w.block, "W": w.W},
               "cpu_baseline": cb,
               "e2e": {"value": round(cb["value"], 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "note": "the reference arm is the CPU oracle (plain C, fp32) timed on the host cores"}
        print(json.dumps(out), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    out = run_loco(args, rank, world)
    if rank == 0 and args.no_cpu_baseline:
        out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    elif rank == 0:
        w = workload(args.workload, args.bits, args.block, args.ranks)
        S = min(w.n, 1 << 27)
        try:
            out["cpu_baseline"] = cpu_baseline(w, S, 1, 1, args.optimizer)
        except Exception as ex:  # the GPU numbers stand without it
            out["cpu_baseline"] = {"value": None, "error": repr(ex)}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
