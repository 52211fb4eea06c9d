"""Falcon throughput on GB300: tokens/s through the C ABI, roofline, oracle baseline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one full forward pass of the workload (all its segments) over one
batch of synthetic input already resident in HBM; for the backward workloads
(`*_bwd_*`) one falcon_bwd call (every gradient). Rank 0 prints one JSON line.
Under torchrun each rank runs the whole workload on its own GPU (sequences are
independent, so there is no data-path collective: weak scaling); the value is
all ranks' tokens over the slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def _algorithmic_bytes(w, es):
    """Bytes every step must move at least once: inputs read, outputs written."""
    BH = w.batch * w.heads
    tok = BH * w.seqlen
    per_seg = tok * (2 * w.dk + w.dv) * es + tok * w.dv * es + tok * 4 * (w.dv if w.variant in ("falcon2", "falcon2a") else 1) \
        + tok * 4 + BH * w.dk * w.dv * 4
    tail = BH * (w.window * w.dk + (w.window - 1) * w.dv) * es
    total = w.segments * (per_seg + tail)
    total += (w.segments - 1) * (BH * w.dk * w.dv * 4 + tail)  # S0 and tail read by later segments
    total += (BH * w.dk * w.dv * 4 if w.nonzero_s0 else 0) + (tail if w.pos0 > 0 else 0)  # the first call's
    return total


def _launches_per_call(w, kernel_id):
    """Kernels one falcon_fwd call launches on the path `kernel_id` takes."""
    if kernel_id == 5:  # [window normalisers,] [tensor-core chunk maps,] chunk maps, [compose, groups,] apply
        n = -(-w.seqlen // w.chunk)
        tc = w.variant in ("falcon3", "falcon3a") and w.window == 4 and w.chunk == 32 and w.dtype == "bf16" \
            and w.dk == 64 and w.dv == 64
        return (1 if w.variant == "falcon3" else 0) + (1 if tc else 0) + 1 + (2 if n > 16 else 0) + 1
    return 1


def _chunk_flops(w):
    """Flops of the method's chunk algebra per call (each product once, 2 flops per multiply-add, at
    the workload's own sizes). Per (b, h) chunk of C tokens with dk = dv = d and R = C W unknown rows
    (W = 1 but for Falcon-3 / 3A, whose rows are the chunk's (token, window slot) pairs): the solve
    variants (Falcon-1, 2, 3) form G = X_w X_w^T (R R d), Q X_w^T (C R d), X_w S_n (R d d), Q S_n
    (C d d), the triangular solve (R R d / 2), P R (C R d) and X_w^T diag(w) R (d R d); the
    inner-product variants (1A, 2A, 3A) form Q X_w^T, Q S_n, P Y and X_w^T diag(w) Y. Falcon-2's
    per-column solves and reads add up to the same counts as Falcon-1's."""
    C, d = w.chunk, w.dk
    R = C * (w.window if w.variant in ("falcon3", "falcon3a") else 1)
    if w.variant in ("falcon1", "falcon2", "falcon3"):
        per = 2 * (1.5 * R * R * d + 2 * C * R * d + 2 * R * d * d + C * d * d)
    elif w.variant in ("falcon1a", "falcon2a", "falcon3a"):
        per = 2 * (2 * C * R * d + C * d * d + R * d * d)
    else:
        return None
    n = -(-w.seqlen // C)
    return per * w.batch * w.heads * n * w.segments


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model", "hardware")):
                return line.split(":", 1)[1].strip()
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("cpu part"):
                return "cpu part " + line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def _kernel_digest(files=None):
    """Digest of the kernel sources (all of csrc/, or the listed files of it)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "weight_linear_attention_gb300", "csrc")
    for f in sorted(files or os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _traffic(workload, kernel_id):
    """DRAM bytes per launch from a committed ncu summary, only if taken on the current sources of the
    kernels that path launches (the entry lists them)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{workload}:{kernel_id}")
    if not e or e.get("kernel_digest") != _kernel_digest(e.get("sources")):
        return None
    return e.get("dram_bytes_per_step")


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, gpu_index):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f".clocks_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
        return dist, rank, world, local
    return None, rank, world, local


def _job_value(world, tokens_per_rank_step, steps, max_total_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time (weak scaling)."""
    return world * tokens_per_rank_step * steps / (max_total_ms / 1e3)


def _barrier_max(dist, value):
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, w):
    """The oracle (fp64 C recurrence) as it stands, timed on the host cores."""
    import oracle
    from weight_linear_attention_gb300 import inputs as I

    dist, rank, world, _ = _dist_setup()
    if rank != 0:
        return
    oracle.build()
    inp = I.make_inputs(w, seed=0)
    cores = os.cpu_count() or 1
    # Bounded sample: the first `bs` batch rows of every segment, all heads, all tokens.
    bs = max(1, min(w.batch, args.ref_batch))
    segs = []
    for s in range(w.segments):
        sl = slice(s * w.seqlen, (s + 1) * w.seqlen)
        segs.append({n: inp[n][:bs, :, sl] for n in ("q", "k", "v", "beta", "lam")})

    S_first, tail_first = _oracle_start(w, inp, bs)

    def step():
        S, tail = S_first, tail_first
        for s, x in enumerate(segs):
            _, S, tail = oracle.falcon_ref_fwd(w.variant_id, x["q"], x["k"], x["v"], x["beta"], x["lam"], S, tail,
                                               pos=w.pos0 + s * w.seqlen, window=w.window, eps=w.eps,
                                               eps_gamma=w.eps_gamma, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    tokens = bs * w.seqlen * w.segments * args.steps
    value = tokens / el
    sample = f"batch rows 0..{bs - 1} of {w.batch}, all {w.heads} heads, all {w.seqlen * w.segments} tokens"
    line = {
        "impl": "reference", "metric": "falcon_fwd_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "seq_len": w.seqlen * w.segments,
                   "d": w.dk, "chunk": w.chunk, "variant": w.variant, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, budget_s=4.0):
    """The oracle on the host cores: enough batch rows of the first segment that every core has a
    sequence, each measurement repeating the sample for about `budget_s` seconds; the median of three
    such measurements with all cores and one with a single thread."""
    import oracle
    from weight_linear_attention_gb300 import inputs as I

    oracle.build()
    cores = os.cpu_count() or 1
    inp = I.make_inputs(w, seed=0)
    bs = max(1, min(w.batch, -(-cores // w.heads)))
    x = {n: inp[n][:bs, :, :w.seqlen] for n in ("q", "k", "v", "beta", "lam")}
    S0, tail = _oracle_start(w, inp, bs)

    def measure(nthreads, rows):
        xs = {n: t[:rows] for n, t in x.items()}
        s0 = S0[:rows] if S0 is not None else None
        tl = (tail[0][:rows], tail[1][:rows]) if tail is not None else None
        runs, t0 = 0, time.perf_counter()
        while True:
            oracle.falcon_ref_fwd(w.variant_id, xs["q"], xs["k"], xs["v"], xs["beta"], xs["lam"], s0, tl,
                                  pos=w.pos0, window=w.window, eps=w.eps, eps_gamma=w.eps_gamma, nthreads=nthreads)
            runs += 1
            if time.perf_counter() - t0 > budget_s or runs >= 100000:
                break
        return runs * rows * w.seqlen / (time.perf_counter() - t0)

    threads = min(cores, bs * w.heads)
    vals = [measure(threads, bs) for _ in range(3)]
    one = measure(1, 1)
    return {"value": statistics.median(vals), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "runs": vals, "one_thread": one, "cpu_model": _cpu_model(),
            "sample": f"batch rows 0..{bs - 1} of {w.batch} ({bs * w.heads} sequences of {w.seqlen} tokens, "
                      f"first segment) repeated for ~{budget_s:.0f} s per measurement; median of 3 with "
                      f"{threads} threads; one_thread: batch row 0 with 1 thread"}


def _oracle_start(w, inp, bs):
    """The first call's S0 and tail, as the oracle takes them, for the first `bs` batch rows."""
    import numpy as np

    S0 = inp["S0"][:bs] if inp.get("S0") is not None else None
    tail = None
    if inp.get("tail") is not None:
        keys = inp["tail"].view(w.batch, w.heads, 1, w.dk)[:bs].double().numpy()
        tail = (keys, np.zeros((bs, w.heads, 0, w.dv)))
    return S0, tail


def _pipelined_ms(n_steps, warm, h2d, compute, d2h):
    """Milliseconds per step of a host-to-host pipeline: step i uses device buffer set b = i % 2; its
    host->device copies run on a copy-in stream, its compute on a compute stream, its device->host
    copies on a copy-out stream, so that step i's compute overlaps the copies of steps i + 1 and i - 1.
    Events order every reuse of a set (the copy-in of step i waits for step i - 2's compute; the
    compute of step i for step i - 2's copy-out). Timed from before the first copy-in to after the
    last copy-out, with CUDA events."""
    import torch

    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def one(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(ev_c[b])
        with torch.cuda.stream(s_in):
            h2d(b)
        ev_in[b].record(s_in)
        s_c.wait_event(ev_in[b])
        if used[b]:
            s_c.wait_event(ev_out[b])
        compute(b, s_c)
        ev_c[b].record(s_c)
        s_out.wait_event(ev_c[b])
        with torch.cuda.stream(s_out):
            d2h(b)
        ev_out[b].record(s_out)
        used[b] = True

    for i in range(warm):
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(n_steps):
        one(warm + i)
    e1.record(s_out)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n_steps


def _e2e(args, w, host_segs, sets, launch):
    """Same metric through the C ABI with host buffers: every step copies its inputs from pinned host
    memory to the device, runs the forward pass and copies the output back, the copies of
    neighbouring steps overlapping its compute (two device buffer sets)."""
    import torch

    B, H, Ts, dv = w.batch, w.heads, w.seqlen, w.dv
    hsegs = [{n: t.pin_memory() for n, t in hs.items()} for hs in host_segs]
    # every segment's output, and the final state and tail of the last segment (the call's result)
    last = sets[0][w.segments - 1]
    hout = [[torch.empty((B, H, Ts, dv), dtype=w.torch_dtype).pin_memory() for _ in range(w.segments)]
            for _ in range(2)]
    hS = [torch.empty_like(last["S"], device="cpu").pin_memory() for _ in range(2)]
    htail = [torch.empty_like(last["tail_out"], device="cpu").pin_memory() for _ in range(2)]
    h2d_bytes = sum(t.numel() * t.element_size() for hs in hsegs for t in hs.values())
    d2h_bytes = sum(t.numel() * t.element_size() for t in hout[0]) + hS[0].numel() * 4 + \
        htail[0].numel() * htail[0].element_size()

    def h2d(b):
        for s in range(w.segments):
            for n in hsegs[s]:
                sets[b][s][n].copy_(hsegs[s][n], non_blocking=True)

    def d2h(b):
        for s in range(w.segments):
            hout[b][s].copy_(sets[b][s]["out"], non_blocking=True)
        hS[b].copy_(sets[b][w.segments - 1]["S"], non_blocking=True)
        htail[b].copy_(sets[b][w.segments - 1]["tail_out"], non_blocking=True)

    ms = _pipelined_ms(max(3, min(args.steps, 50)), max(3, args.warmup), h2d, lambda b, st: launch(sets[b], st), d2h)
    return ms, h2d_bytes, d2h_bytes


def run_ours(args, w):
    import torch

    from weight_linear_attention_gb300 import build as fbuild
    from weight_linear_attention_gb300 import falcon as F
    from weight_linear_attention_gb300 import inputs as I

    dist, rank, world, local = _dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fbuild.build()
    F.load()
    es = 4 if w.dtype == "f32" else 2
    inp = I.make_inputs(w, seed=0)
    B, H, Ts, dk, dv, W = w.batch, w.heads, w.seqlen, w.dk, w.dv, w.window
    dims = [F.make_dims(B, H, Ts, dk, dv, window=W, dtype=F.FALCON_F32 if w.dtype == "f32" else F.FALCON_BF16,
                        pos=w.pos0 + s * Ts, eps=w.eps, eps_gamma=w.eps_gamma) for s in range(w.segments)]
    kernel_id = F.falcon_kernel_for(w.variant_id, dims[0], w.chunk)
    step_bytes = _algorithmic_bytes(w, es)
    nsets = max(2, -(-3 * L2_BYTES // step_bytes) + 1)  # rotating sets: > 3x L2 between reuses
    stream = torch.cuda.Stream(device=dev)
    tail_n = F.falcon_tail_bytes(dims[0]) // es

    def seg_inputs(s):
        sl = slice(s * Ts, (s + 1) * Ts)
        d = {n: inp[n][:, :, sl].contiguous() for n in ("q", "k", "v", "beta", "lam")}
        if s == 0:  # a workload that starts from a given state and tail
            d.update({n: inp[n].contiguous() for n in ("S0", "tail") if inp.get(n) is not None})
        return d

    host_segs = [seg_inputs(s) for s in range(w.segments)]
    sets = []
    for _ in range(nsets):
        segs = []
        for s in range(w.segments):
            d = {n: host_segs[s][n].to(dev) for n in host_segs[s]}
            d["out"] = torch.empty((B, H, Ts, dv), dtype=w.torch_dtype, device=dev)
            d["S"] = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
            d["tail_out"] = torch.empty(tail_n, dtype=w.torch_dtype, device=dev)
            segs.append(d)
        sets.append(segs)

    # one scratch workspace (the scan path's chunk maps, where that path runs), reused by every step
    ws = F.workspace_for(w.variant_id, dims[0], w.chunk, dev)

    def launch(segs, strm):
        for s, d in enumerate(segs):
            prev = segs[s - 1] if s > 0 else None
            S0 = prev["S"] if prev else d.get("S0")
            tail = prev["tail_out"] if prev else d.get("tail")
            st = F.falcon_fwd(w.variant_id, d["q"], d["k"], d["v"], d["beta"], d["lam"], S0, tail,
                              d["out"], d["S"], d["tail_out"], dims[s], w.chunk, ws, stream=strm.cuda_stream)
            if st != 0:
                raise F.FalconError(st)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(sets[i % nsets], stream)
        stream.synchronize()
        if F.falcon_device_status(stream.cuda_stream) != 0:
            raise SystemExit("device-side timeout during warm-up")
        # ---- clock sampling starts here and runs through a ~1 s soak of the same launches
        # (the last part of the warm-up) and the whole timed region.
        clocks = Clocks(local) if rank == 0 else None
        t_soak = time.perf_counter()
        i = 0
        while time.perf_counter() - t_soak < args.soak_s:
            launch(sets[i % nsets], stream)
            i += 1
            if i % 64 == 0:
                stream.synchronize()
        stream.synchronize()
        # ---- timed region: K steps back to back, CUDA events on the launching stream around all of them
        # (an event between steps would sit between one call's last kernel and the next call's first)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            launch(sets[i % nsets], stream)
        t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        clk = clocks.stop() if clocks else None
        total_ms = t_start.elapsed_time(t_end)
        if F.falcon_device_status(stream.cuda_stream) != 0:
            raise SystemExit("device-side timeout during the timed region")


    if args.no_e2e:
        e2e_ms, h2d, d2h = float("nan"), 0, 0
    else:
        e2e_ms, h2d, d2h = _e2e(args, w, host_segs, sets, launch)
    total_ms = _barrier_max(dist, total_ms)
    ms_step = total_ms / args.steps
    tokens_step = w.total_tokens
    value = _job_value(world, tokens_step, args.steps, total_ms)
    e2e_ms = _barrier_max(dist, e2e_ms)
    if rank != 0:
        return
    mean_launch = ms_step / w.segments  # one falcon_fwd call
    hbm, tfl, src = _peaks()
    achieved = step_bytes / (ms_step / 1e3) / 1e9
    line = {
        "metric": "falcon_fwd_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "variant": w.variant, "batch": B, "heads": H, "seq_len": Ts * w.segments,
                   "segments": w.segments, "d": dk, "chunk": w.chunk, "window": W,
                   "parallelism": f"dp{world} (independent sequences per GPU, no collective)",
                   "l2": f"rotating {nsets} input/output sets of {step_bytes / 1e6:.1f} MB (> L2 between reuses)",
                   "pos0": w.pos0,
                   "kernel": {1: "cuda-core chunk kernel", 4: "single-token kernel",
                              5: "scan path: chunk maps on the cuda-core kernel, associative scan over them "
                                 "with the outputs fused",
                              6: "fused tcgen05/TMA kernel, one persistent CTA per sequence",
                              7: "per-column tcgen05/TMA kernel, one persistent CTA per sequence"}.get(kernel_id, "?")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "scope": "one falcon_fwd call (all kernels it launches); per-kernel shares in profiles/",
                     "traffic": _traffic(w.name, kernel_id), "peak_source": src,
                     "algorithmic_bytes_per_step": step_bytes, "ms_per_call": mean_launch},
        "e2e": None if args.no_e2e else {"value": world * tokens_step / (e2e_ms / 1e3), "unit": "tokens/s",
                                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                         "pipeline": "copy-in of step i+1 and copy-out of step i-1 overlap the "
                                                     "compute of step i (two device buffer sets, three streams)"},
        "gpu_launches": args.steps * w.segments * _launches_per_call(w, kernel_id),
        "clocks": clk,
    }
    fl = _chunk_flops(w)
    if fl is not None:  # the same call against the tensor roofline (the method's own flops)
        tf = fl / (ms_step / 1e3) / 1e12
        line["roofline"]["tensor"] = {"achieved": tf, "peak": tfl, "unit": "TFLOP/s", "frac": tf / tfl,
                                      "flops_per_step": fl,
                                      "note": "chunk-algebra flops, each product once; peak = measured dense "
                                              "bf16 (the path mixes bf16 and tf32 products)"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------------------
# backward workloads (falcon_bwd)



def _bwd_groups(bh):
    """Groups of sequences one falcon_bwd call runs on streams of their own (three kernels each)."""
    return 4 if bh >= 16 else (2 if bh >= 4 else 1)


def _bwd_flops_per_chunk(w):
    """Flops of the chunk algebra the three backward kernels evaluate per 64-token chunk, each
    64 x 64 x 64 product counted once (2 flops per multiply-add) whatever the number of tf32 passes
    it takes: Falcon-1 prep 10 products and the triangular inverse (~1/3), the two scans 2,
    gradients 15; Falcon-1A prep 2, scans 2, gradients 9."""
    one = 2 * 64 ** 3
    return one * ((10 + 1 / 3 + 2 + 15) if w.variant == "falcon1" else (2 + 2 + 9))


def _bwd_bytes(w, es):
    """Bytes a backward step must move at least once: q, k, v, dout read (dtype), beta, lambda read,
    the fp32 gradients of q, k, v, beta, lambda written, dS_final read and dS0 written."""
    BH = w.batch * w.heads
    tok = BH * w.seqlen
    return tok * (2 * w.dk + 2 * w.dv) * es + tok * 8 + tok * (2 * w.dk + w.dv) * 4 + tok * 8 \
        + 2 * BH * w.dk * w.dv * 4 + (BH * w.dk * w.dv * 4 if w.nonzero_s0 else 0)


def cpu_baseline_bwd(w, budget_s=12.0):
    import torch

    from oracle import falcon_bwd as OB
    from weight_linear_attention_gb300 import inputs as I

    inp = I.make_inputs(w, seed=0, batch=1)
    inp.update(I.make_adjoints(w, seed=0, batch=1))
    runs, t0 = 0, time.perf_counter()
    while True:
        OB.falcon_ref_bwd(w.variant_id, inp["q"], inp["k"], inp["v"], inp["beta"], inp["lam"], inp["dout"],
                          inp["S0"], inp["dS_final"], eps=w.eps, eps_gamma=w.eps_gamma)
        runs += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": runs * w.seqlen / el, "unit": "tokens/s", "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{runs} runs of batch row 0 ({w.heads} heads x {w.seqlen} tokens), fp64 autograd, {el:.1f} s"}


def run_reference_bwd(args, w):
    _, rank, _, _ = _dist_setup()
    if rank != 0:
        return
    import torch

    from oracle import falcon_bwd as OB
    from weight_linear_attention_gb300 import inputs as I

    inp = I.make_inputs(w, seed=0, batch=1)
    inp.update(I.make_adjoints(w, seed=0, batch=1))

    def step():
        OB.falcon_ref_bwd(w.variant_id, inp["q"], inp["k"], inp["v"], inp["beta"], inp["lam"], inp["dout"],
                          inp["S0"], inp["dS_final"], eps=w.eps, eps_gamma=w.eps_gamma)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = w.seqlen * args.steps / el
    line = {
        "impl": "reference", "metric": "falcon_bwd_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "seq_len": w.seqlen, "d": w.dk,
                   "chunk": w.chunk, "variant": w.variant, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": torch.get_num_threads(), "kind": "oracle",
                         "sample": f"batch row 0 of {w.batch}, all {w.heads} heads, all {w.seqlen} tokens"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours_bwd(args, w):
    import torch

    from weight_linear_attention_gb300 import build as fbuild
    from weight_linear_attention_gb300 import falcon as F
    from weight_linear_attention_gb300 import inputs as I

    dist, rank, world, local = _dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fbuild.build()
    F.load()
    es = 4 if w.dtype == "f32" else 2
    B, H, T, dk, dv = w.batch, w.heads, w.seqlen, w.dk, w.dv
    inp = I.make_inputs(w, seed=0)
    inp.update(I.make_adjoints(w, seed=0))
    dims = F.make_dims(B, H, T, dk, dv, dtype=F.FALCON_F32 if w.dtype == "f32" else F.FALCON_BF16, eps=w.eps,
                       eps_gamma=w.eps_gamma)
    step_bytes = _bwd_bytes(w, es)
    nsets = max(2, -(-3 * L2_BYTES // step_bytes) + 1)
    names_in = [n for n in ("q", "k", "v", "beta", "lam", "S0", "dout", "dS_final") if inp.get(n) is not None]
    host = {n: inp[n].contiguous() for n in names_in}
    f32 = dict(dtype=torch.float32, device=dev)

    def new_set():
        d = {n: host[n].to(dev) for n in names_in}
        d.update(dq=torch.empty((B, H, T, dk), **f32), dk=torch.empty((B, H, T, dk), **f32),
                 dv=torch.empty((B, H, T, dv), **f32), dbeta=torch.empty((B, H, T), **f32),
                 dlam=torch.empty((B, H, T), **f32), dS0=torch.empty((B, H, dk, dv), **f32))
        return d

    sets = [new_set() for _ in range(nsets)]
    ws = torch.empty(F.falcon_bwd_workspace_bytes(w.variant_id, dims, w.chunk), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def launch(d, strm):
        st = F.falcon_bwd(w.variant_id, d["q"], d["k"], d["v"], d["beta"], d["lam"], d.get("S0"), None, d["dout"],
                          d["dS_final"], d["dq"], d["dk"], d["dv"], d["dbeta"], d["dlam"], d["dS0"], None, dims,
                          w.chunk, ws, stream=strm.cuda_stream)
        if st != 0:
            raise F.FalconError(st, "falcon_bwd")

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch(sets[i % nsets], stream)
        stream.synchronize()
        clocks = Clocks(local) if rank == 0 else None
        t_soak, i = time.perf_counter(), 0
        while time.perf_counter() - t_soak < args.soak_s:
            launch(sets[i % nsets], stream)
            i += 1
            if i % 16 == 0:
                stream.synchronize()
        stream.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            launch(sets[i % nsets], stream)
        e1.record(stream)
        stream.synchronize()
        if dist is not None:
            dist.barrier()
        clk = clocks.stop() if clocks else None
        total_ms = e0.elapsed_time(e1)
        if F.falcon_device_status(stream.cuda_stream) != 0:
            raise SystemExit("device-side timeout during the timed region")
        # end to end: pinned host inputs in, every gradient out, per step (pipelined as in _e2e)
        e2e = None
        if not args.no_e2e:
            hin = {n: host[n].pin_memory() for n in names_in}
            outs = ("dq", "dk", "dv", "dbeta", "dlam", "dS0")
            hout = [{n: torch.empty(sets[0][n].shape, dtype=torch.float32).pin_memory() for n in outs}
                    for _ in range(2)]

            def h2d(b):
                for n in names_in:
                    sets[b][n].copy_(hin[n], non_blocking=True)

            def d2h(b):
                for n in outs:
                    hout[b][n].copy_(sets[b][n], non_blocking=True)

            e2e_ms = _barrier_max(dist, _pipelined_ms(max(3, min(args.steps, 20)), 3, h2d,
                                                      lambda b, st: launch(sets[b], st), d2h))
            e2e = {"value": world * B * T / (e2e_ms / 1e3), "unit": "tokens/s",
                   "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
                   "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout[0].values()),
                   "pipeline": "copy-in of step i+1 and copy-out of step i-1 overlap the compute of step i "
                               "(two device buffer sets, three streams)"}
    total_ms = _barrier_max(dist, total_ms)
    ms_step = total_ms / args.steps
    value = _job_value(world, B * T, args.steps, total_ms)
    if rank != 0:
        return
    hbm, bf16_peak, src = _peaks()
    chunks = B * H * (-(-T // w.chunk))
    flops = _bwd_flops_per_chunk(w) * chunks
    achieved = flops / (ms_step / 1e3) / 1e12
    groups = _bwd_groups(B * H)
    line = {
        "metric": "falcon_bwd_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16-in/f32",
        "data": "synthetic",
        "config": {"workload": w.name, "variant": w.variant, "batch": B, "heads": H, "seq_len": T, "d": dk,
                   "chunk": w.chunk, "parallelism": f"dp{world} (independent sequences per GPU, no collective)",
                   "l2": f"rotating {nsets} input/gradient sets of {step_bytes / 1e6:.1f} MB (> L2 between reuses)",
                   "kernel": "backward: prep, chain and gradient kernels, every product tcgen05 bf16 with fp32 "
                             f"operands split into hi and lo; sequences in {groups} group(s) on their own streams"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": achieved / bf16_peak, "traffic": _traffic(w.name, "bwd"),
                     "scope": "one falcon_bwd call (all its kernels); flops of the chunk algebra, each product "
                              "counted once (bf16 tensor cores, 1-3 passes per product for fp32 accuracy)",
                     "peak_source": f"{src} dense bf16",
                     "flops_per_step": flops, "hbm_algorithmic_bytes_per_step": step_bytes,
                     "hbm_frac": step_bytes / (ms_step / 1e3) / 1e9 / hbm, "hbm_peak_source": src},
        "e2e": e2e,
        "gpu_launches": args.steps * 3 * groups,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--ref-batch", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0, help="seconds of warm-up launches under clock sampling")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--seqlen", type=int, default=None, help="override the workload's tokens per call")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from weight_linear_attention_gb300 import inputs as I

    w = I.WORKLOADS[args.workload or I.HEADLINE]
    if args.seqlen is not None:
        w = w.with_(seqlen=args.seqlen)
    if args.batch is not None:
        w = w.with_(batch=args.batch)
    if w.backward:
        (run_reference_bwd if args.impl == "reference" else run_ours_bwd)(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
