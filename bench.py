"""Benchmark of the FLASH GAU layer forward (mixed chunk attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the float64 CPU oracle arm

One step = one full forward (projection, chunk states, prefix scan, chunk
attention, output projection) over one batch of seeded synthetic input that
is resident in HBM.  L2 is flushed (a 512 MiB write) before every timed
step.  Per-stage device times come from CUDA events the library records on
the launching stream between its kernels.  Prints one JSON line (rank 0).
"""

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FLASH GAU layer forward tokens/sec at T=8192 causal; % of bf16 TC roofline"
DEFAULT_WORKLOAD = "long_causal_B2_T8192"
L2_FLUSH_BYTES = 512 << 20
# CUDA-core fp32 peak of a GB300, from unit counts and the clock: 152 SMs x
# 128 fp32 lanes x 2 flops per FMA x 2.07 GHz (maximum SM clock)
FP32_CORE_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def lib_backward_bytes(bd, weights, B, T, C, causal):
    import ctypes
    n = bd.lib().flash_gau_backward_workspace_bytes(B, T, C, ctypes.byref(weights.c),
                                                    int(bool(causal)), weights.dtype)
    if n == 0:
        raise RuntimeError("backward workspace size")
    return n


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return dict(hbm_gbs=float(m["hbm_gbs"]), bf16_tflops=float(m["bf16_tflops"]),
                    bf16_tflops_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


def stage_work(w):
    """Algorithmic work per launch of each stage: (flops, bytes)."""
    B, T, d, e, s, C = w["B"], w["T"], w["d"], w["e"], w["s"], w["C"]
    causal = w["causal"]
    io = 2 if w["dtype"] == "bf16" else 4
    M, G = B * T, T // C
    cbar = (C + 1) / 2.0 if causal else float(C)
    pre_rows = B * G if causal else B
    # causal with one chunk (FLASH-Quad): the global term is the empty sum,
    # so the bf16 schedule forms no chunk states and reads no prefix
    quad = causal and G == 1 and w["dtype"] == "bf16"
    lin = 0.0 if quad else 1.0
    return {
        "projection": (2.0 * M * d * (2 * e + s),
                       io * (M * d + d * (2 * e + s) + 2 * M * e + 4 * M * s)),
        "chunk_state": (2.0 * M * s * e, io * (M * s + M * e) + 4.0 * B * G * s * e),
        "prefix_scan": (float(B * G * s * e), 4.0 * B * G * s * e + io * pre_rows * s * e),
        # bf16 schedule: states written and read back in bf16 inside one kernel
        "chunk_state_scan": (lin * (2.0 * M * s * e + B * G * s * e),
                             lin * io * (M * s + M * e + 2 * B * G * s * e + pre_rows * s * e)),
        "chunk_attention": (2.0 * M * (cbar * s + cbar * e + lin * s * e),
                            io * (2 * M * e + (2 + lin) * M * s + lin * pre_rows * s * e + M * e)),
        "output": (2.0 * M * e * d, io * (M * e + e * d + M * d)),
    }


def traffic_record(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) < 4 or line.startswith("#"):
            continue
        k, src, sha, nbytes = parts[0], parts[1], parts[2], parts[3]
        wl = parts[4] if len(parts) > 4 else ""
        if k != kernel or wl != workload:
            continue
        try:
            cur = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        return float(nbytes) if cur == sha else None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(values, device):
    """Element-wise maximum of each rank's floats over the process group (the
    slowest rank sets a job's time); the values themselves when no group of
    more than one rank is running."""
    import torch
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: the tokens every rank processed over the
    slowest rank's time (ms)."""
    return tokens_per_rank * world / (ms * 1e-3)


def run_part(args, dev):
    """One component alone, a few calls, for profiling a kernel under ncu
    without the rest of the bench: the layer, the flash_block wrapper, the
    RoPE table, the backward, decode steps (B = 1, 16, 64), or the fp32
    layer on the small workload.  Returns a short record."""
    import torch
    import efficient_attention_transformer_gb300 as fg
    from efficient_attention_transformer_gb300 import binding as bd
    from efficient_attention_transformer_gb300.synthetic import WORKLOADS, make_inputs
    name = "tiny_causal_fp32_T256" if args.part == "fp32" else args.workload
    w = dict(WORKLOADS[name])
    B, T, d, e, s, C, causal = w["B"], w["T"], w["d"], w["e"], w["s"], w["C"], w["causal"]
    tdt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    inp = make_inputs(**w)
    W_uvz = np.concatenate([inp["W_u"], inp["W_v"], inp["W_z"]], axis=1)
    weights = fg.GauWeights(torch.tensor(W_uvz, dtype=tdt, device=dev),
                            torch.tensor(inp["W_o"], dtype=tdt, device=dev),
                            torch.tensor(inp["gamma"], dtype=torch.float32, device=dev),
                            torch.tensor(inp["beta"], dtype=torch.float32, device=dev),
                            torch.tensor(inp["relpos"], dtype=torch.float32, device=dev),
                            d, e, s)
    X = torch.tensor(inp["X"], dtype=tdt, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = args.warmup + args.steps
    calls = 0
    t0 = time.perf_counter()
    if args.part in ("layer", "fp32", "block"):
        ws = weights.new_workspace(B, T, C, causal, dev)
        out = torch.empty_like(X)
        g = torch.ones(d, dtype=torch.float32, device=dev)
        for _ in range(n):
            if args.part == "block":
                bd.block_forward(X, weights, C, causal, norm=bd.NORM_LAYER, norm_g=g, norm_b=g,
                                 out=out, workspace=ws, stream=stream)
            else:
                bd.forward(X, weights, C, causal, out=out, workspace=ws, stream=stream)
            calls += 1
        status = bd.workspace_status(ws)
    elif args.part == "rope":
        a = torch.ones(128, dtype=torch.float32, device=dev)
        tout = torch.empty(2 * 512 - 1, dtype=torch.float32, device=dev)
        for _ in range(n):
            bd.rope_toeplitz_bias(a, a, 512, out=tout, stream=stream)
            calls += 1
        status = 0
    elif args.part == "backward":
        dO = torch.tensor(np.random.default_rng(3000 + w["seed"]).normal(size=(B, T, d)),
                          dtype=tdt, device=dev)
        bws = torch.empty(lib_backward_bytes(bd, weights, B, T, C, causal), dtype=torch.uint8,
                          device=dev)
        for _ in range(n):
            bd.backward(X, dO, weights, C, causal, workspace=bws, stream=stream)
            calls += 1
        status = bd.workspace_status(bws)
    elif args.part == "decode":
        status = 0
        for Bd in (1, 16, 64):
            dec = bd.Decoder(weights, Bd, C)
            xs = torch.tensor(np.random.default_rng(4000 + Bd).normal(size=(Bd, d)), dtype=tdt,
                              device=dev)
            od = torch.empty_like(xs)
            for _ in range(n):
                dec.step(xs, out=od, stream=stream)
                calls += 1
            del dec
    else:
        raise ValueError("unknown part %r" % args.part)
    torch.cuda.synchronize()
    if status != 0:
        raise RuntimeError("kernel status %d in part %s" % (status, args.part))
    return {"part": args.part, "workload": name, "calls": calls,
            "wall_ms_per_call": round((time.perf_counter() - t0) * 1e3 / max(1, calls), 4)}


def run_ours(args, rank, world, local_rank):
    import torch
    import efficient_attention_transformer_gb300 as fg
    from efficient_attention_transformer_gb300 import binding as bd
    from efficient_attention_transformer_gb300.build import build
    from efficient_attention_transformer_gb300.synthetic import WORKLOADS, make_inputs

    build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if args.part != "all":
        return run_part(args, dev)
    w = dict(WORKLOADS[args.workload])
    B, T, d, e, s, C, causal = w["B"], w["T"], w["d"], w["e"], w["s"], w["C"], w["causal"]
    tdt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    inp = make_inputs(**w)
    W_uvz = np.concatenate([inp["W_u"], inp["W_v"], inp["W_z"]], axis=1)
    weights = fg.GauWeights(torch.tensor(W_uvz, dtype=tdt, device=dev),
                            torch.tensor(inp["W_o"], dtype=tdt, device=dev),
                            torch.tensor(inp["gamma"], dtype=torch.float32, device=dev),
                            torch.tensor(inp["beta"], dtype=torch.float32, device=dev),
                            torch.tensor(inp["relpos"], dtype=torch.float32, device=dev),
                            d, e, s)
    X = torch.tensor(inp["X"], dtype=tdt, device=dev)
    out = torch.empty_like(X)
    ws = weights.new_workspace(B, T, C, causal, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = bd.stage_names(weights.dtype, causal)
    nst = len(names)

    def step(evs):
        bd.forward(X, weights, C, causal, out=out, workspace=ws, stream=stream, stage_events=evs)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step(None)
    torch.cuda.synchronize()

    # timed region: K forwards, each bracketed by events on the launching
    # stream (no events between the kernels, so nothing breaks their overlap)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(1.0)
        ev0[k].record(stream)
        step(None)
        ev1[k].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    st = bd.workspace_status(ws)
    if st != 0:
        raise RuntimeError("kernel status %d after the timed region" % st)
    step_ms = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / args.steps

    # per-kernel split: the same forwards with the library's stage events
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
           for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(1.0)
        step(evs[k])
    torch.cuda.synchronize()
    per_stage = np.zeros(nst)
    split_ms = 0.0
    for k in range(args.steps):
        for j in range(nst):
            per_stage[j] += evs[k][j].elapsed_time(evs[k][j + 1])
        split_ms += evs[k][0].elapsed_time(evs[k][nst])
    per_stage /= args.steps
    split_ms /= args.steps
    step_ms, wall = max_over_ranks([step_ms, wall], dev)

    # ---- end to end: pinned host X in, O out, through the host-buffer entry
    # point (flash_gau_forward_host: its copies of one part of the batch
    # overlap the layer on another; the caller's stream waits for the last
    # output copy, so the events below bracket every copy)
    Xh = X.cpu().pin_memory()
    Oh = torch.empty_like(Xh).pin_memory()
    hws = torch.empty(bd.lib().flash_gau_forward_host_workspace_bytes(
        B, T, C, ctypes.byref(weights.c), int(bool(causal)), weights.dtype),
        dtype=torch.uint8, device=dev)

    def e2e_step():
        bd.forward_host(Xh, weights, C, causal, out=Oh, workspace=hws, stream=stream)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 200))
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    (e2e_ms,) = max_over_ranks([e2e_ms], dev)

    # the host link alone: plain pinned copies of the same bytes (X in, O
    # out), one way at a time and both ways at once on two streams, as the
    # bound the end-to-end figure is judged against
    Xd = torch.empty_like(X)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def copy_ms(h2d, d2h, n=20):
        for _ in range(3):
            if h2d:
                with torch.cuda.stream(s_in):
                    Xd.copy_(Xh, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    Oh.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(n):
            if h2d:
                with torch.cuda.stream(s_in):
                    Xd.copy_(Xh, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    Oh.copy_(out, non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        c1.record(stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / n

    nbytes = X.numel() * X.element_size()
    link = {"h2d_ms": copy_ms(True, False), "d2h_ms": copy_ms(False, True),
            "both_ms": copy_ms(True, True)}
    link = {k: round(v, 5) for k, v in link.items()}
    link["h2d_gbs"] = round(nbytes / (link["h2d_ms"] * 1e-3) / 1e9, 1)
    link["d2h_gbs"] = round(nbytes / (link["d2h_ms"] * 1e-3) / 1e9, 1)
    del Xd

    # ---- next row: the flash_block wrapper (LayerNorm, RoPE on the four heads,
    # residual) around the same layer on the same workload, timed the same way
    nrng = np.random.default_rng(1000 + w["seed"])
    norm_g = torch.tensor(nrng.normal(1.0, 0.1, d), dtype=torch.float32, device=dev)
    norm_b = torch.tensor(nrng.normal(0.0, 0.1, d), dtype=torch.float32, device=dev)

    def block_step():
        bd.block_forward(X, weights, C, causal, norm=bd.NORM_LAYER, norm_g=norm_g,
                         norm_b=norm_b, rope=True, residual=True, out=out, workspace=ws,
                         stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        block_step()
    blk_steps = max(1, min(args.steps, 200))
    b0 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
    b1 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
    torch.cuda.synchronize()
    for k in range(blk_steps):
        flush.fill_(1.0)
        b0[k].record(stream)
        block_step()
        b1[k].record(stream)
    torch.cuda.synchronize()
    block_ms = sum(a.elapsed_time(b) for a, b in zip(b0, b1)) / blk_steps
    if bd.workspace_status(ws) != 0:
        raise RuntimeError("kernel status after the flash_block runs")
    (block_ms,) = max_over_ranks([block_ms], dev)

    # ---- next row: the two ablations of the mixed chunk attention on the
    # same workload and weights: GlobalOnly (local term off: no chunk scores
    # are formed) and LocalOnly (global term off)
    ablations = {}
    for name, lin_sc, loc_sc in (("global_only", 1.0, 0.0), ("local_only", 0.0, 1.0)):
        wv = fg.GauWeights(weights.W_uvz, weights.W_o, weights.gamma, weights.beta,
                           weights.relpos, d, e, s, lin_sc, loc_sc)
        for _ in range(args.warmup):
            flush.fill_(1.0)
            bd.forward(X, wv, C, causal, out=out, workspace=ws, stream=stream)
        a0 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
        a1 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
        torch.cuda.synchronize()
        for k in range(blk_steps):
            flush.fill_(1.0)
            a0[k].record(stream)
            bd.forward(X, wv, C, causal, out=out, workspace=ws, stream=stream)
            a1[k].record(stream)
        torch.cuda.synchronize()
        (ab_ms,) = max_over_ranks([sum(x.elapsed_time(y) for x, y in zip(a0, a1)) / blk_steps],
                                  dev)
        if bd.workspace_status(ws) != 0:
            raise RuntimeError("kernel status after the %s runs" % name)
        ablations[name] = {"ms_per_step": round(ab_ms, 5),
                           "value": round(job_tokens_per_s(B * T, world, ab_ms), 1),
                           "unit": "tokens/s"}
        del wv

    # ---- next row: packed text, the chunk-masked global term: each batch
    # row holds four documents of G/4 chunks (ids 0..3), mean of the visible
    # chunk states
    G = T // C
    seg_ids = torch.tensor(np.repeat(np.arange(4), -(-G // 4))[:G][None, :].repeat(B, 0),
                           dtype=torch.int32, device=dev)

    def seg_step():
        bd.forward_segmented(X, weights, C, causal, seg_ids, True, out=out, workspace=ws,
                             stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        seg_step()
    s0 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
    s1 = [torch.cuda.Event(enable_timing=True) for _ in range(blk_steps)]
    torch.cuda.synchronize()
    for k in range(blk_steps):
        flush.fill_(1.0)
        s0[k].record(stream)
        seg_step()
        s1[k].record(stream)
    torch.cuda.synchronize()
    (seg_ms,) = max_over_ranks([sum(x.elapsed_time(y) for x, y in zip(s0, s1)) / blk_steps], dev)
    if bd.workspace_status(ws) != 0:
        raise RuntimeError("kernel status after the segmented runs")

    # ---- next row: the RoPE construction of the relative-position table
    # (windows of 512 and more), 128-wide learned vectors, C = 512
    trng = np.random.default_rng(2000 + w["seed"])
    ta = torch.tensor(trng.normal(0, 0.1, 128), dtype=torch.float32, device=dev)
    tb = torch.tensor(trng.normal(0, 0.1, 128), dtype=torch.float32, device=dev)
    tout = torch.empty(2 * 512 - 1, dtype=torch.float32, device=dev)
    for _ in range(3):
        bd.rope_toeplitz_bias(ta, tb, 512, out=tout, stream=stream)
    tn = 100
    te0, te1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    te0.record(stream)
    for _ in range(tn):
        bd.rope_toeplitz_bias(ta, tb, 512, out=tout, stream=stream)
    te1.record(stream)
    torch.cuda.synchronize()
    toeplitz_us = te0.elapsed_time(te1) * 1e3 / tn

    # ---- next row: the backward pass on the same workload (gradients of
    # sum(dO * O) for X and every parameter), dO seeded like X
    dO = torch.tensor(np.random.default_rng(3000 + w["seed"]).normal(size=(B, T, d)), dtype=tdt,
                      device=dev)
    bws = torch.empty(lib_backward_bytes(bd, weights, B, T, C, causal), dtype=torch.uint8,
                      device=dev)
    bd.backward(X, dO, weights, C, causal, workspace=bws, stream=stream)  # warm-up
    bn = 3
    be0, be1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    be0.record(stream)
    for _ in range(bn):
        bd.backward(X, dO, weights, C, causal, workspace=bws, stream=stream)
    be1.record(stream)
    torch.cuda.synchronize()
    (backward_ms,) = max_over_ranks([be0.elapsed_time(be1) / bn], dev)
    del bws

    # ---- next row: autoregressive decode at the workload's widths, B
    # sequences one token each per step, over two chunks (two folds of the
    # linear cache); plain calls and one step replayed as a CUDA graph
    decode = {}
    drng = np.random.default_rng(4000 + w["seed"])
    io_bytes = 2 if tdt == torch.bfloat16 else 4
    for Bd in (1, 16, 64):
        dec = bd.Decoder(weights, Bd, C)
        xs = torch.tensor(drng.normal(size=(Bd, d)), dtype=tdt, device=dev)
        od = torch.empty_like(xs)
        nsteps = 2 * C
        for _ in range(8):
            dec.step(xs, out=od, stream=stream)
        dec.reset()
        de0, de1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        de0.record(stream)
        for _ in range(nsteps):
            dec.step(xs, out=od, stream=stream)
        de1.record(stream)
        torch.cuda.synchronize()
        plain_us = de0.elapsed_time(de1) * 1e3 / nsteps
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            dec.step(xs, out=od, stream=cap)
        stream.wait_stream(cap)
        dec.reset()
        torch.cuda.synchronize()
        de0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(nsteps):
                graph.replay()
        de1.record(stream)
        torch.cuda.synchronize()
        graph_us = de0.elapsed_time(de1) * 1e3 / nsteps
        # bytes a step must move: both weight matrices once, and per
        # sequence the linear cache and on average half a chunk of cached
        # K_quad and V rows (fp32), plus the fold's share
        wbytes = io_bytes * (d * (2 * e + s) + e * d)
        sbytes = Bd * 4 * (s * e + (C // 2) * (s + e) + (C * (s + e) + 2 * s * e) // C)
        best = min(plain_us, graph_us)
        decode["B%d" % Bd] = {"us_per_step_plain": round(plain_us, 2),
                              "us_per_step_graph": round(graph_us, 2),
                              "tokens_per_s": round(Bd / (best * 1e-6), 1),
                              "gbs": round((wbytes + sbytes) / (best * 1e-6) / 1e9, 1)}
        del dec, graph

    # ---- the other workloads of the scope table, timed the same way (each
    # is also a parity case of the GPU tests)
    others = {}
    for wname in WORKLOADS:
        if wname == args.workload:
            continue
        ow = dict(WORKLOADS[wname])
        oi = make_inputs(**ow)
        otdt = torch.bfloat16 if ow["dtype"] == "bf16" else torch.float32
        owt = fg.GauWeights(
            torch.tensor(np.concatenate([oi["W_u"], oi["W_v"], oi["W_z"]], axis=1), dtype=otdt,
                         device=dev),
            torch.tensor(oi["W_o"], dtype=otdt, device=dev),
            torch.tensor(oi["gamma"], dtype=torch.float32, device=dev),
            torch.tensor(oi["beta"], dtype=torch.float32, device=dev),
            torch.tensor(oi["relpos"], dtype=torch.float32, device=dev),
            ow["d"], ow["e"], ow["s"])
        oX = torch.tensor(oi["X"], dtype=otdt, device=dev)
        oout = torch.empty_like(oX)
        ows = owt.new_workspace(ow["B"], ow["T"], ow["C"], ow["causal"], dev)
        for _ in range(3):
            flush.fill_(1.0)
            bd.forward(oX, owt, ow["C"], ow["causal"], out=oout, workspace=ows, stream=stream)
        on = 20
        o0 = [torch.cuda.Event(enable_timing=True) for _ in range(on)]
        o1 = [torch.cuda.Event(enable_timing=True) for _ in range(on)]
        torch.cuda.synchronize()
        for k in range(on):
            flush.fill_(1.0)
            o0[k].record(stream)
            bd.forward(oX, owt, ow["C"], ow["causal"], out=oout, workspace=ows, stream=stream)
            o1[k].record(stream)
        torch.cuda.synchronize()
        (oms,) = max_over_ranks([sum(a.elapsed_time(b) for a, b in zip(o0, o1)) / on], dev)
        if bd.workspace_status(ows) != 0:
            raise RuntimeError("kernel status after the %s runs" % wname)
        owork = stage_work(ow)
        onames = bd.stage_names(owt.dtype, ow["causal"])
        oflops = sum(owork[n][0] for n in onames)
        otf = oflops / (oms * 1e-3) / 1e12
        others[wname] = {"ms_per_step": round(oms, 5),
                         "value": round(job_tokens_per_s(ow["B"] * ow["T"], world, oms), 1),
                         "unit": "tokens/s", "tflops": round(otf, 2)}
        del owt, oX, oout, ows

    if rank != 0:
        return None
    peaks = _peaks()
    for wname, rec in others.items():
        # fp32 runs on the CUDA cores, bf16 on the tensor cores
        if WORKLOADS[wname]["dtype"] == "fp32":
            rec["frac_of_fp32_core_peak"] = round(rec["tflops"] / FP32_CORE_PEAK_TFLOPS, 4)
        else:
            rec["frac_of_bf16_peak"] = round(rec["tflops"] / peaks["bf16_tflops"], 4)
    work = stage_work(w)
    tokens = B * T * world
    # the stages this schedule runs (the table also lists the other dtype's)
    total_flops = sum(work[n][0] for n in names)
    stages = {}
    for j, n in enumerate(names):
        f, b = work[n]
        ms = float(per_stage[j])
        stages[n] = {"ms": round(ms, 5), "share": round(ms / per_stage.sum(), 4),
                     "bound": "tensor" if f / (peaks["bf16_tflops"] * 1e12) >=
                              b / (peaks["hbm_gbs"] * 1e9) else "hbm",
                     "tflops": round(f / (ms * 1e-3) / 1e12, 1),
                     "gbs": round(b / (ms * 1e-3) / 1e9, 1)}
    dom = names[int(np.argmax(per_stage))]
    f, b = work[dom]
    dom_ms = float(per_stage[names.index(dom)])
    # roofline: the bound is whichever of compute time and memory time at
    # peak is larger for the kernel's algorithmic work
    tensor_bound = f / (peaks["bf16_tflops"] * 1e12) >= b / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        achieved = f / (dom_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    else:
        achieved = b / (dom_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    layer_tflops = total_flops / (step_ms * 1e-3) / 1e12
    res = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(B * T, world, step_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w["dtype"],
        "data": "synthetic (seeded numpy normal draws; no dataset)",
        "config": {"workload": "%s: FLASH GAU forward B=%d T=%d d=%d e=%d s=%d C=%d %s %s"
                               % (args.workload, B, T, d, e, s, C,
                                  "causal" if causal else "non-causal", w["dtype"]),
                   "B": B, "T": T, "d": d, "e": e, "s": s, "C": C, "causal": causal,
                   "l2": "flushed before every timed step (512 MiB write)",
                   "parallelism": "replicas (one independent problem per GPU)"},
        "layer_tflops": round(layer_tflops, 1),
        "layer_frac_of_bf16_peak": round(layer_tflops / peaks["bf16_tflops"], 4),
        "roofline": {"bound": "tensor" if tensor_bound else "hbm", "kernel": dom,
                     "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4),
                     "peak_source": peaks["source"] + " (burst)",
                     "traffic": traffic_record(dom, args.workload)},
        "stages": stages,
        "gpu_launches": nst * args.steps,
        "wall_ms_per_step_incl_flush": round(wall * 1e3 / args.steps, 4),
        "ms_per_step_with_stage_events": round(split_ms, 5),
        "e2e": {"value": round(job_tokens_per_s(B * T, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(X.numel() * X.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "ms_per_step": round(e2e_ms, 5),
                "host_link": dict(
                    what="plain pinned copies of the same X and O bytes alone: the copy-only "
                         "time the overlapped call cannot beat (both_ms: both ways at once)",
                    **link)},
        "clocks": clocks,
        "next_rows": {"flash_block": {
            "what": "LayerNorm + RoPE on the four heads (global positions) + residual "
                    "around the same layer, same workload",
            "value": round(tokens / (block_ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(block_ms, 5),
            "extra_ms_over_layer": round(block_ms - step_ms, 5)},
            "backward": {
                "what": "gradients of sum(dO * O) for X, W_uvz, W_o, gamma, beta, relpos "
                        "(recomputes the forward's intermediates); every contraction on "
                        "the tensor cores (bf16 operands, fp32 accumulation; the chunk-level "
                        "ones batched over the chunks), sums, scans and elementwise steps "
                        "in fp32",
                "ms_per_call": round(backward_ms, 3),
                "value": round(tokens / (backward_ms * 1e-3), 1), "unit": "tokens/s",
                # two contractions per forward contraction, plus the recompute
                "algorithmic_tflops": round(2 * total_flops / (backward_ms * 1e-3) / 1e12, 2),
                "executed_tflops": round(3 * total_flops / (backward_ms * 1e-3) / 1e12, 2),
                "fp32_core_peak_tflops": round(FP32_CORE_PEAK_TFLOPS, 1)},
            "decode": dict(
                what="autoregressive decode step at the workload's widths (C = 256, causal): "
                     "B sequences, one token each per step, 2C steps; five kernels per step "
                     "(projection, chunk weights, chunk attention with the linear cache, "
                     "output, cache fold)",
                **decode),
            "global_only": dict(
                what="the layer with the local term switched off (local_scale = 0): "
                     "projection, chunk states, scan, Q_lin Prefix and the gate, output",
                **ablations["global_only"]),
            "local_only": dict(
                what="the layer with the global term switched off (lin_scale = 0)",
                **ablations["local_only"]),
            "segmented": {
                "what": "packed text: four documents per batch row (segment ids per chunk), "
                        "global term = mean of the visible chunk states of the document",
                "ms_per_step": round(seg_ms, 5),
                "value": round(tokens / (seg_ms * 1e-3), 1), "unit": "tokens/s"},
            "other_workloads": dict(
                what="the scope table's other workloads, same timing (L2 flushed, 20 steps); "
                     "algorithmic TFLOP/s against the bf16 tensor-core peak, or the fp32 "
                     "CUDA-core peak for the fp32 one",
                **others),
            "rope_toeplitz_bias": {
                "what": "relative-position table of the RoPE bias construction, C = 512, "
                        "128-wide vectors (1023 entries x 64 pairs), back-to-back launches",
                "us_per_call": round(toeplitz_us, 2)}},
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    return res


def _oracle_sample(w, tokens):
    """Oracle on a causal prefix of one sequence of the workload (a multiple
    of C tokens), returns (seconds, tokens)."""
    from efficient_attention_transformer_gb300.synthetic import make_inputs
    from oracle import flash_gau
    T = max(w["C"], min(w["T"], (tokens // w["C"]) * w["C"]))
    inp = make_inputs(1, T, w["d"], w["e"], w["s"], w["C"], w["dtype"], w["seed"])
    t0 = time.perf_counter()
    flash_gau(inp["X"], inp["W_u"], inp["W_v"], inp["W_z"], inp["W_o"], inp["gamma"],
              inp["beta"], inp["relpos"], w["C"], w["causal"])
    return time.perf_counter() - t0, T


def _threads():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


def cpu_baseline(w, budget_s=20.0):
    """The oracle as it stands on the host cores, on whole sequences of the
    workload repeated until about budget_s seconds of CPU work."""
    secs, toks, reps = 0.0, 0, 0
    while secs < budget_s and reps < 256:
        dt, T = _oracle_sample(w, w["T"])
        secs += dt
        toks += T
        reps += 1
    return {"value": round(toks / secs, 1), "unit": "tokens/s", "cores": _threads(),
            "kind": "oracle",
            "sample": "%d x one full sequence (B=1, T=%d) of the workload, float64 numpy oracle, "
                      "%.1f s" % (reps, w["T"], secs)}


def run_reference(args):
    """The oracle arm: each step runs the oracle on a causal prefix of one
    sequence, sized so that warmup + steps stay within a few minutes."""
    from efficient_attention_transformer_gb300.synthetic import WORKLOADS
    w = dict(WORKLOADS[args.workload])
    probe, T0 = _oracle_sample(w, w["C"])
    per_tok = probe / T0
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(budget / per_tok)
    for _ in range(args.warmup):
        _oracle_sample(w, tokens)
    secs, toks = 0.0, 0
    for _ in range(args.steps):
        dt, T = _oracle_sample(w, tokens)
        secs += dt
        toks += T
    v = toks / secs
    sample = ("causal prefix of one sequence, %d tokens per step, float64 numpy oracle"
              % (toks // max(1, args.steps)))
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "%s (oracle on a bounded sample)" % args.workload},
        "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "cores": _threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--part", default="all",
                    choices=["all", "layer", "block", "rope", "backward", "decode", "fp32"],
                    help="run one component alone (a profiling aid; prints a short record)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
