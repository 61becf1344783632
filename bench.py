"""Benchmark of the int4-g128 weight-streaming GEMV on GB300.

One step = one w4g128_decode_step call streaming the weight set of one
27B-class decoder layer at M = 1 (q, k, v 5120x6144; o 6144x5120; fused
gate+up 5120x34816; down 17408x5120 -- 208.9 MB of packed int4-g128 weights).
Steps rotate over 4 weight copies (836 MB > 4x the 129 MB L2), so every step
reads its weights from HBM.  The same step at M = 8 (speculative verify) is
timed alongside.  Inputs are seeded synthetic data with the value
distributions of the workload (codes uniform 0..15, scale U(0.002, 0.02),
min = -8 scale (1 + U(-0.1, 0.1)), x ~ N(0, 1)).

Before timing, sampled outputs of both M = 1 and M = 8 are checked against the
fp64 oracle; a mismatch voids the run (exit status 1, no number printed).

`--target layer|lm_head|single` instead runs a few untimed calls of one
workload (`single`: the matrix `--shape K,N`) and exits: the launch target
for profiler captures (no JSON line).

Prints ONE JSON line.  `--impl reference` times the fp64 CPU oracle instead
(the reference arm: the plain dequantise-then-multiply definition on the host
cores).  Under torchrun (N > 1) every rank streams its own copy of the layer
set (replicas; the path needs no exchange between GPUs) and rank 0 reports
the aggregate.
"""
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

METRIC = "int4-g128 GEMV HBM GB/s & % of GB300 peak at M=1 and M=8; µs/call"
LAYER = [("q", 5120, 6144), ("k", 5120, 6144), ("v", 5120, 6144), ("o", 6144, 5120),
         ("gate_up", 5120, 34816), ("down", 17408, 5120)]
# Single-call shapes timed for us/call: the square case, the four distinct
# layer shapes, the full-vocabulary lm_head and its first 131072 columns
# (a prefix view of the same packed buffer).
SHAPES = [("square", 4096, 4096), ("q_k_v", 5120, 6144), ("o", 6144, 5120), ("gate_up", 5120, 34816),
          ("down", 17408, 5120), ("lm_head", 5120, 248320), ("lm_head_slice", 5120, 131072)]
# The projections whose output feeds a residual add + RMS norm (attention
# output and MLP down), timed fused and plain.
NORM_SHAPES = [(6144, 5120), (17408, 5120)]
LM_HEAD = (5120, 248320)
N_LAYERS = 64
L2_BYTES = 129 * 1024 * 1024
SEED = 20260001
NCOPY = 4
PEAKS_FALLBACK = {"hbm_gbs": 6800.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "stream1_local_kernel_layer_m1.md")
KERNEL_SOURCES = [os.path.join(ROOT, "int4_weight_only_g128_gb300", "csrc", f)
                  for f in ("w4g128_stream.cu", "w4g128_ptx.cuh", "w4g128_internal.h")]


def weight_bytes(K, N):
    return K * N * 17 // 32


def algorithmic_bytes(M):
    """Packed weights + x + y bytes of one layer step."""
    return sum(weight_bytes(K, N) + 2 * M * K + 2 * M * N for _, K, N in LAYER)


def workload_config():
    return {
        "workload": "27B-class decoder layer weight stream: q,k,v 5120x6144, o 6144x5120, "
                    "gate+up 5120x34816, down 17408x5120; int4-g128 weights, bf16 x/y; "
                    "one w4g128_decode_step per step",
        "M": 1,
        "M_also_reported": [8],
        "weight_bytes_per_step": sum(weight_bytes(K, N) for _, K, N in LAYER),
        "algorithmic_bytes_per_step": algorithmic_bytes(1),
        "l2": f"inputs larger than L2: {NCOPY} rotating weight copies "
              f"({NCOPY * sum(weight_bytes(K, N) for _, K, N in LAYER) / 1e6:.0f} MB)",
        "seed": SEED,
    }


# --------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(dist, value, device):
    """The largest value over all ranks (the slowest rank's time); dist None
    means a single process."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbps(world, steps, bytes_per_step, seconds):
    """Whole-job throughput: each of `world` ranks streamed `steps` steps of its
    own copy of the workload in at most `seconds`."""
    return world * steps * bytes_per_step / seconds / 1e9


def dist_init(backend):
    import torch.distributed as dist
    ws, _, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return PEAKS_FALLBACK, "fallback"


def kernel_source_sha():
    """Hash of the kernel sources with comments and blank lines removed, so
    that a comment edit does not invalidate the profiled traffic."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(PROFILE_SUMMARY) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        s = line.strip().lstrip("-").strip()
        if ":" in s and s.startswith(("traffic_bytes_per_launch", "source_sha")):
            k, v = s.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != kernel_source_sha():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- CPU oracle

def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def time_oracle(budget_s, cols_hint=None, nthreads=0):
    """Times the fp64 oracle on the first `cols` columns of every layer
    matrix (nthreads 0: every core); returns (GB/s-equivalent of packed
    weight bytes, threads, sample, s)."""
    import numpy as np

    import oracle
    import synth
    O = oracle.Oracle()
    cores = nthreads or O.max_threads()

    def timed(cols):
        tot = 0.0
        nbytes = 0
        for i, (_, K, N) in enumerate(LAYER):
            sel = np.arange(cols)
            c, s, m = synth.columns(SEED, i, K, N, sel)
            x = synth.x(SEED, 100 + i, 1, K)
            t0 = time.perf_counter()
            O.gemm(x, c, s, m, nthreads=nthreads)
            tot += time.perf_counter() - t0
            nbytes += weight_bytes(K, cols) + 2 * K + 2 * cols
        return nbytes, tot

    cols = cols_hint or 64
    nbytes, t = timed(cols)
    if cols_hint is None:
        cols = int(max(16, min(4096, cols * budget_s / max(t, 1e-3))))
        cols -= cols % 16
        nbytes, t = timed(cols)
    sample = (f"fp64 oracle, first {cols} columns of each of the 6 layer matrices at M=1 "
              f"({sum(K * cols for _, K, _ in LAYER) / 1e6:.1f} M weights), {cores} threads")
    return nbytes / t / 1e9, cores, sample, t


def run_reference(args):
    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    # size one step so that warmup + steps finish within about a minute
    _, _, _, t_probe = time_oracle(0.0, cols_hint=32)
    per_step_budget = max(0.05, 60.0 / max(1, args.steps + args.warmup))
    cols = int(max(16, min(2048, 32 * per_step_budget / max(t_probe, 1e-3))))
    cols -= cols % 16
    for _ in range(args.warmup):
        time_oracle(0.0, cols_hint=cols)
    vals = []
    t_total = 0.0
    sample, cores = "", 1
    for _ in range(args.steps):
        v, cores, sample, t = time_oracle(0.0, cols_hint=cols)
        vals.append(v)
        t_total += t
    value = len(vals) / sum(1.0 / v for v in vals)  # harmonic mean = bytes-weighted throughput
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    record(args, out)
    return 0


# --------------------------------------------------------------------------- GPU arm

def run_ours(args):
    import numpy as np
    import torch

    import int4_weight_only_g128_gb300 as w
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init("nccl")
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream

    # ---- weights: NCOPY copies of the layer set, generated and packed on the device
    copies = []
    for cp in range(NCOPY):
        mats = []
        for i, (_, K, N) in enumerate(LAYER):
            codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
            s = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
            m = torch.empty_like(s)
            synth.fill_device(SEED, i, K, N, codes.data_ptr(), s.data_ptr(), m.data_ptr(), st)
            packed = torch.empty(w.w4g128_packed_bytes(K, N), dtype=torch.uint8, device="cuda")
            w.w4g128_pack(codes, s, m, K, N, packed)
            mats.append(packed)
            del codes, s, m
        copies.append(mats)
    torch.cuda.synchronize()

    def make_io(M):
        # the six x (and the six y) are slices of one contiguous buffer, 256-byte
        # aligned, so that the end-to-end run moves each direction in one copy
        xs_h = [synth.x(SEED, (100 if M == 1 else 200) + i, M, K) for i, (_, K, _) in enumerate(LAYER)]
        up = lambda n: -(-n // 128) * 128
        xoff = np.cumsum([0] + [up(x.size) for x in xs_h])
        yoff = np.cumsum([0] + [up(M * N) for _, _, N in LAYER])
        x_all = torch.zeros(int(xoff[-1]), dtype=torch.int16, device="cuda")
        y_all = torch.zeros(int(yoff[-1]), dtype=torch.int16, device="cuda")
        xs = [x_all[xoff[i]:xoff[i] + x.size] for i, x in enumerate(xs_h)]
        for xd, x in zip(xs, xs_h):
            xd.copy_(torch.from_numpy(x.reshape(-1).view(np.int16)))
        ys = [y_all[yoff[i]:yoff[i] + M * N] for i, (_, _, N) in enumerate(LAYER)]
        descs = [[(copies[c][i], xs[i], ys[i], K, N) for i, (_, K, N) in enumerate(LAYER)] for c in range(NCOPY)]
        nb = max(w.w4g128_decode_step_workspace_bytes(d, M) for d in descs)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        return xs_h, xs, ys, descs, ws, x_all, y_all

    MS = (1, 2, 4, 8, 16)
    io = {M: make_io(M) for M in MS}

    # ---- parity gate on sampled outputs (first and last weight copy)
    import oracle
    O = oracle.Oracle()
    worst = {}
    for M in MS:
        xs_h, xs, ys, descs, ws = io[M][:5]
        for c in (0, NCOPY - 1):
            w.w4g128_decode_step(descs[c], M, ws, stream=st)
            torch.cuda.synchronize()
            if w.w4g128_workspace_status(ws, st) != 0:
                print(json.dumps({"error": "device status word set: run void"}))
                return 1
            rng = np.random.default_rng(M * 10 + c)
            for i, (_, K, N) in enumerate(LAYER):
                cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 24)]))
                cc, ss, mm = synth.columns(SEED, i, K, N, cols)
                y_ref, a = O.gemm(xs_h[i], cc, ss, mm)
                y = oracle.bf16_bits_to_f64(ys[i].cpu().numpy().view(np.uint16).reshape(M, N)[:, cols])
                ok, ratio = oracle.accept(y, y_ref, a, O)
                if not ok.all():
                    print(json.dumps({"error": f"parity mismatch M={M} matrix={LAYER[i][0]}: run void"}))
                    return 1
                worst[M] = max(worst.get(M, 0.0), float(ratio.max()))

    def barrier():
        if dist is not None:
            dist.barrier()

    def capture(calls):
        """CUDA graph of the given launch callables (each takes the capture stream)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream().cuda_stream
            for f in calls:
                f(cs)
        return g

    def timed_graph(M, steps, warmup):
        """Replays a graph of `steps` decode_step calls (rotating weight copies);
        returns the max-over-ranks seconds of the whole replay."""
        _, _, _, descs, ws = io[M][:5]
        for i in range(warmup):
            w.w4g128_decode_step(descs[i % NCOPY], M, ws, stream=st)
        torch.cuda.synchronize()
        g = capture([lambda cs, i=i: w.w4g128_decode_step(descs[i % NCOPY], M, ws, stream=cs)
                     for i in range(steps)])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(dist, e0.elapsed_time(e1) * 1e-3, "cuda")

    # ---- clocks sampled over a soak of identical steps that ends with the timed region
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.perf_counter()
    _, _, _, descs1, ws1 = io[1][:5]
    k = 0
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(200):
            w.w4g128_decode_step(descs1[k % NCOPY], 1, ws1, stream=st)
            k += 1
        torch.cuda.synchronize()
    totals = {}
    for M in MS:
        totals[M] = timed_graph(M, args.steps, args.warmup)
    clk = clocks.stop()

    # informative only: the same step with one weight copy (209 MB, so the
    # 126 MB L2 holds part of it between steps)
    l2_warm = {}
    for M in (1, 8):
        _, _, _, descs_w, ws_w = io[M][:5]
        g = capture([lambda cs: w.w4g128_decode_step(descs_w[0], M, ws_w, stream=cs) for _ in range(50)])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        l2_warm[f"M{M}_us_per_step"] = round(e0.elapsed_time(e1) * 1e3 / 50, 3)
    total1, total8 = totals[1], totals[8]
    launch1, launch8 = total1 / args.steps, total8 / args.steps

    bytes1, bytes8 = algorithmic_bytes(1), algorithmic_bytes(8)
    value = aggregate_gbps(world, args.steps, bytes1, total1)
    value8 = aggregate_gbps(world, args.steps, bytes8, total8)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    by_m = {}
    for M in MS:
        gbs = algorithmic_bytes(M) / (totals[M] / args.steps) / 1e9
        by_m[str(M)] = {"us_per_step": round(1e6 * totals[M] / args.steps, 3), "GBps": round(gbs, 1),
                        "frac": round(gbs / peak, 4), "cost_ratio_vs_M1": round(totals[M] / total1, 4)}

    def pack_device(K, N, matrix_id):
        codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
        s_ = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
        m_ = torch.empty_like(s_)
        synth.fill_device(SEED, matrix_id, K, N, codes.data_ptr(), s_.data_ptr(), m_.data_ptr(), st)
        packed = torch.empty(w.w4g128_packed_bytes(K, N), dtype=torch.uint8, device="cuda")
        w.w4g128_pack(codes, s_, m_, K, N, packed, stream=st)
        return packed

    def graph_us(call, reps):
        for r in range(3):
            call(st, r)
        torch.cuda.synchronize()
        g = capture([lambda cs, r=r: call(cs, r) for r in range(reps)])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    # ---- single-matrix calls (gemv at M = 1, verify at M = 8), us per call, graph-timed over
    # enough rotating copies to exceed twice the L2
    per_call = {}
    lm_packed = None
    for si, (name, K, N) in enumerate(SHAPES):
        if name == "lm_head_slice":
            mats = [lm_packed]  # the first 131072 columns, in place
        else:
            first = pack_device(K, N, 50 + si)
            ncopy = max(1, -(-2 * L2_BYTES // weight_bytes(K, N)))
            mats = [first] + [first.clone() for _ in range(ncopy - 1)]
            if name == "lm_head":
                lm_packed = first
        for M in (1, 8):
            x = torch.from_numpy(synth.x(SEED, 300 + si, M, K).view(np.int16)).cuda()
            y = torch.empty(M * N, dtype=torch.int16, device="cuda")
            wsd = torch.empty(w.w4g128_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")

            def call(cs, r, M=M, K=K, N=N, wsd=wsd, x=x, y=y, mats=mats):
                if M == 1:
                    w.w4g128_gemv(mats[r % len(mats)], x, y, K, N, wsd, stream=cs)
                else:
                    w.w4g128_gemm_verify(mats[r % len(mats)], x, y, M, K, N, wsd, stream=cs)
            us = graph_us(call, 16 if weight_bytes(K, N) > L2_BYTES else 64)
            gbs = (weight_bytes(K, N) + 2 * M * (K + N)) / us / 1e3
            per_call[f"{name}_{K}x{N}_M{M}"] = {"us": round(us, 3), "GBps": round(gbs, 1),
                                                "frac": round(gbs / peak, 4), "copies": len(mats)}
        if name != "lm_head":
            del mats
    del lm_packed
    torch.cuda.synchronize()

    # ---- the product folded into the residual add + RMS norm, on the two projections a
    # norm follows (attention output, MLP down): fused call vs the plain call, us per call
    norm_fused = {}
    for si, (K, N) in enumerate(NORM_SHAPES):
        first = pack_device(K, N, 70 + si)
        ncopy = max(1, -(-2 * L2_BYTES // weight_bytes(K, N)))
        mats = [first] + [first.clone() for _ in range(ncopy - 1)]
        gam = torch.from_numpy(synth.norm_weight(SEED, 80 + si, N).view(np.int16)).cuda()
        for M in (1, 8):
            x = torch.from_numpy(synth.x(SEED, 310 + si, M, K).view(np.int16)).cuda()
            res = torch.from_numpy(synth.x(SEED, 320 + si, M, N).view(np.int16)).cuda()
            h = torch.empty(M * N, dtype=torch.int16, device="cuda")
            o = torch.empty(M * N, dtype=torch.int16, device="cuda")
            wsd = torch.empty(w.w4g128_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")

            def fcall(cs, r, M=M, K=K, N=N, wsd=wsd, x=x, res=res, h=h, o=o, mats=mats):
                w.w4g128_gemm_add_rmsnorm(mats[r % len(mats)], x, res, gam, 1e-6, h, o, M, K, N, 0, wsd,
                                          stream=cs)

            def pcall(cs, r, M=M, K=K, N=N, wsd=wsd, x=x, h=h, mats=mats):
                if M == 1:
                    w.w4g128_gemv(mats[r % len(mats)], x, h, K, N, wsd, stream=cs)
                else:
                    w.w4g128_gemm_verify(mats[r % len(mats)], x, h, M, K, N, wsd, stream=cs)
            us_f = graph_us(fcall, 64)
            us_p = graph_us(pcall, 64)
            norm_fused[f"{K}x{N}_M{M}"] = {"us_fused": round(us_f, 3), "us_product_only": round(us_p, 3),
                                           "added_us": round(us_f - us_p, 3)}
        del mats
    torch.cuda.synchronize()

    # ---- a dependent chain of single calls: o -> gate+up -> down, each x the previous y (down reads the first
    # 17408 outputs of gate+up: the activation between them is not part of the weight stream); the realistic
    # decode order, which one decode_step cannot batch
    chain = {}
    CHAIN = [(6144, 5120), (5120, 34816), (17408, 5120)]
    cbytes = sum(weight_bytes(K, N) for K, N in CHAIN)
    ncp = max(1, -(-2 * L2_BYTES // cbytes))
    cmats = [[pack_device(K, N, 90 + j) for j, (K, N) in enumerate(CHAIN)]]
    for _ in range(ncp - 1):
        cmats.append([m.clone() for m in cmats[0]])
    for M in (1, 8):
        x0 = torch.from_numpy(synth.x(SEED, 330, M, 6144).view(np.int16)).cuda()
        yo = torch.empty(M * 5120, dtype=torch.int16, device="cuda")
        yg = torch.empty(M * 34816, dtype=torch.int16, device="cuda")
        yd = torch.empty(M * 5120, dtype=torch.int16, device="cuda")
        wsc = torch.empty(max(w.w4g128_workspace_bytes(M, K, N) for K, N in CHAIN), dtype=torch.uint8,
                          device="cuda")

        def one(cs, r, M=M, x0=x0, yo=yo, yg=yg, yd=yd, wsc=wsc):
            ms = cmats[r % len(cmats)]
            if M == 1:
                w.w4g128_gemv(ms[0], x0, yo, 6144, 5120, wsc, stream=cs)
                w.w4g128_gemv(ms[1], yo, yg, 5120, 34816, wsc, stream=cs)
                w.w4g128_gemv(ms[2], yg, yd, 17408, 5120, wsc, stream=cs)  # x = y_gate_up[:17408]
            else:
                w.w4g128_gemm_verify(ms[0], x0, yo, M, 6144, 5120, wsc, stream=cs)
                w.w4g128_gemm_verify(ms[1], yo, yg, M, 5120, 34816, wsc, stream=cs)
                # rows of 34816 -> rows of 17408: a strided view is not a plain [M][K] array, so
                # the verify step reads the first M * 17408 values (each x row a slice of y)
                w.w4g128_gemm_verify(ms[2], yg, yd, M, 17408, 5120, wsc, stream=cs)
        us = graph_us(one, 32)
        chain[f"M{M}"] = {"us_per_chain": round(us, 3), "GBps": round(cbytes / us / 1e3, 1),
                          "frac": round(cbytes / us / 1e3 / peak, 4), "copies": len(cmats)}
    chain["chain"] = "o 6144x5120 -> gate+up 5120x34816 -> down 17408x5120, single calls, each x the previous y"
    del cmats
    torch.cuda.synchronize()

    # ---- host cost of one call (enqueue time while the GPU is busy): the list-of-tuples API, the
    # prepared DecodeStep, and a single gemv
    host_us = {}
    _, _, _, descs_h, ws_h = io[1][:5]
    step_h = w.DecodeStep(descs_h[0], 1, ws_h, stream=st)
    for name, fn in (("decode_step_list_api", lambda: w.w4g128_decode_step(descs_h[0], 1, ws_h, stream=st)),
                     ("decode_step_prepared", step_h.run)):
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(200):
            fn()
        host_us[name] = round((time.perf_counter() - t0) / 200 * 1e6, 2)
        torch.cuda.synchronize()

    # ---- the whole decode-step weight stream: 64 layer sets + the lm_head, one decode_step call
    full = {}
    fmats = [(K, N) for _ in range(N_LAYERS) for _, K, N in LAYER] + [LM_HEAD]
    fpacked = [pack_device(K, N, 1000 + j) for j, (K, N) in enumerate(fmats)]
    torch.cuda.synchronize()
    fbytes_w = sum(weight_bytes(K, N) for K, N in fmats)
    for M in (1, 8):
        xs_f = {}
        for K in sorted({K for K, _ in fmats}):
            xs_f[K] = torch.from_numpy(synth.x(SEED, 400 + K, M, K).view(np.int16)).cuda()
        ys_f = [torch.empty(M * N, dtype=torch.int16, device="cuda") for _, N in fmats]
        descs_f = [(fpacked[j], xs_f[K], ys_f[j], K, N) for j, (K, N) in enumerate(fmats)]
        wsf = torch.empty(w.w4g128_decode_step_workspace_bytes(descs_f, M), dtype=torch.uint8, device="cuda")
        w.w4g128_decode_step(descs_f, M, wsf, stream=st)
        torch.cuda.synchronize()
        if w.w4g128_workspace_status(wsf, st) != 0:
            print(json.dumps({"error": "device status word set in the full decode step: run void"}))
            return 1
        for j in (0, len(fmats) - 1):  # sampled parity: first layer matrix and the lm_head
            K, N = fmats[j]
            rng = np.random.default_rng(77 + M + j)
            cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 16)]))
            cc, ss, mm = synth.columns(SEED, 1000 + j, K, N, cols)
            y_ref, a = O.gemm(xs_f[K].cpu().numpy().view(np.uint16).reshape(M, K), cc, ss, mm)
            yv = oracle.bf16_bits_to_f64(ys_f[j].cpu().numpy().view(np.uint16).reshape(M, N)[:, cols])
            ok, ratio = oracle.accept(yv, y_ref, a, O)
            if not ok.all():
                print(json.dumps({"error": f"parity mismatch in the full decode step M={M}: run void"}))
                return 1
        us = graph_us(lambda cs, r: w.w4g128_decode_step(descs_f, M, wsf, stream=cs), 5)
        fb = fbytes_w + sum(2 * M * (K + N) for K, N in fmats)
        gbs = fb / us / 1e3
        full[f"M{M}"] = {"matrices": len(fmats), "weight_bytes": fbytes_w, "ms_per_step": round(us / 1e3, 4),
                         "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                         "steps_per_s": round(1e6 / us, 1)}
        del descs_f, ys_f, xs_f, wsf
    del fpacked
    torch.cuda.synchronize()

    # ---- live bandwidth probes: a pure read stream and a copy
    probe = {}
    nbp = 4 << 30
    buf = torch.empty(nbp, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    sink = torch.empty(max(16, w.w4g128_probe_sink_bytes()), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        w.w4g128_probe_read(buf, nbp, sink, stream=st)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        w.w4g128_probe_read(buf, nbp, sink, stream=st)
    e1.record(stream)
    torch.cuda.synchronize()
    probe["read_GBps"] = round(10 * nbp / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    half = nbp // 2
    src, dst = buf[:half], buf[half:]
    for _ in range(3):
        w.w4g128_probe_copy(src, dst, half, stream=st)
    e0.record(stream)
    for _ in range(10):
        w.w4g128_probe_copy(src, dst, half, stream=st)
    e1.record(stream)
    torch.cuda.synchronize()
    probe["copy_GBps_read_plus_write"] = round(10 * 2 * half / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    del buf, src, dst

    # ---- end to end through host buffers: pinned x in, y out, every step, eager C-ABI calls;
    # the layer's x and y each live in one contiguous buffer, moved in one copy per direction
    xs_h, xs, ys, descs, ws, x_all, y_all = io[1]
    x_pin = x_all.cpu().pin_memory()
    y_pin = torch.empty(y_all.numel(), dtype=torch.int16).pin_memory()
    h2d = x_pin.numel() * 2
    d2h = y_pin.numel() * 2
    # one w4g128_decode_step_host call per step: x in from pinned host memory, the layer streamed, y out
    steps_e2e = [w.DecodeStep(descs[c], 1, ws, stream=st, x_host=x_pin, x_dev=x_all, y_host=y_pin, y_dev=y_all)
                 for c in range(NCOPY)]
    for i in range(args.warmup):
        steps_e2e[i % NCOPY].run_host()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        steps_e2e[i % NCOPY].run_host()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_s = max_over_ranks(dist, e0.elapsed_time(e1) * 1e-3, "cuda")
    e2e_value = aggregate_gbps(world, args.steps, bytes1, e2e_s)

    if rank != 0:
        return 0

    achieved = bytes1 / launch1 / 1e9
    achieved8 = bytes8 / launch8 / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, sample, _ = time_oracle(args.cpu_budget)
        v1, _, sample1, _ = time_oracle(args.cpu_budget / 5, nthreads=1)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "single_thread": {"value": round(v1, 4), "sample": sample1}}

    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * total1 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(), timing="CUDA events around one CUDA-graph replay of `steps` "
                                                 "decode_step calls"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "peak_source": ("measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                                     if peak_kind == "measured" else "fallback 6.8 TB/s"),
                     "kernel": "stream1_local_kernel (M=1: activation packages built in each CTA) + fold1_kernel, per decode_step call"},
        "m8": {"value": round(value8, 1), "unit": "GB/s", "ms_per_step": round(1e3 * total8 / args.steps, 5),
               "achieved": round(achieved8, 1), "frac": round(achieved8 / peak, 4),
               "verify_cost_ratio_t8_over_t1": round(total8 / total1, 4)},
        "layer_step_by_M": by_m,
        "layer_step_one_copy_l2_warm_informative": l2_warm,
        "us_per_call": per_call,
        "residual_add_rmsnorm_us": norm_fused,
        "full_decode_step": full,
        "dependent_chain": chain,
        "host_us_per_call": host_us,
        "bandwidth_probes": probe,
        "frac_of_read_probe": {"m1": round(achieved / probe["read_GBps"], 4),
                               "m8": round(achieved8 / probe["read_GBps"], 4)},
        "parity": {"checked": "sampled columns of all 6 matrices, M=1 and M=8, vs fp64 oracle",
                   "worst_error_over_bound": {str(k): round(v, 5) for k, v in worst.items()}},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "w4g128_decode_step_host (one C call per step: x in, layer streamed, y out)"},
        "value_full_decode_step": {"workload": "64 x layer set + lm_head 5120x248320, 385 matrices, 14.04 GB, "
                                               "one decode_step call", "M1_GBps": full["M1"]["GBps"],
                                   "M8_GBps": full["M8"]["GBps"], "M1_frac": full["M1"]["frac"],
                                   "M8_frac": full["M8"]["frac"]},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "equivalent_tok_per_s_ceiling_full_27B_weight_set": round(achieved * 1e9 / 14044774400, 1),
        "measured_tok_per_s_full_decode_step_M1": full["M1"]["steps_per_s"],
    }
    print(json.dumps(out), flush=True)
    record(args, out)
    return 0


def record(args, out):
    """With --record DIR, append the line to DIR/<date>-<host>/bench.jsonl
    (the run history the tables of measured figures are written from)."""
    if not args.record:
        return
    import datetime
    import socket
    day = datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%d")
    d = os.path.join(args.record, f"{day}-{socket.gethostname()}")
    os.makedirs(d, exist_ok=True)
    line = dict(out, recorded_utc=datetime.datetime.now(datetime.timezone.utc).isoformat(timespec="seconds"))
    with open(os.path.join(d, "bench.jsonl"), "a") as f:
        f.write(json.dumps(line) + "\n")


def run_target(args):
    """Untimed calls of one workload for a profiler to capture: the layer set
    through w4g128_decode_step, or one matrix (the 5120 x 248320 lm_head, or
    --shape K,N) through w4g128_gemv (M = 1) / w4g128_gemm_verify (M > 1);
    each M in --m in turn.  Single matrices rotate over enough copies to
    exceed twice the L2, as in the timed run."""
    import numpy as np
    import torch

    import int4_weight_only_g128_gb300 as w
    import synth

    st = torch.cuda.current_stream().cuda_stream
    if args.target == "layer":
        shapes = [(K, N) for _, K, N in LAYER]
    elif args.target == "single":
        K, N = (int(v) for v in args.shape.split(","))
        shapes = [(K, N)]
    else:
        shapes = [(5120, 248320)]
    packed = []
    for i, (K, N) in enumerate(shapes):
        codes = torch.empty((K // 8) * N, dtype=torch.int32, device="cuda")
        s = torch.empty((K // 128) * N, dtype=torch.int16, device="cuda")
        m = torch.empty_like(s)
        synth.fill_device(SEED, i, K, N, codes.data_ptr(), s.data_ptr(), m.data_ptr(), st)
        pk = torch.empty(w.w4g128_packed_bytes(K, N), dtype=torch.uint8, device="cuda")
        w.w4g128_pack(codes, s, m, K, N, pk)
        packed.append(pk)
        del codes, s, m
    for M in [int(v) for v in args.m.split(",")]:
        xs = [torch.from_numpy(synth.x(SEED, 100 + i, M, K).view(np.int16)).cuda() for i, (K, _) in enumerate(shapes)]
        ys = [torch.empty(M * N, dtype=torch.int16, device="cuda") for _, N in shapes]
        descs = [(packed[i], xs[i], ys[i], K, N) for i, (K, N) in enumerate(shapes)]
        if args.target == "layer":
            ws = torch.empty(w.w4g128_decode_step_workspace_bytes(descs, M), dtype=torch.uint8, device="cuda")
            for _ in range(args.calls):
                w.w4g128_decode_step(descs, M, ws, stream=st)
        else:
            (pk, x, y, K, N), = descs
            ncopy = max(1, -(-2 * L2_BYTES // weight_bytes(K, N)))
            mats = [pk] + [pk.clone() for _ in range(ncopy - 1)]
            ws = torch.empty(w.w4g128_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
            for c in range(args.calls):
                if M == 1:
                    w.w4g128_gemv(mats[c % ncopy], x, y, K, N, ws, stream=st)
                else:
                    w.w4g128_gemm_verify(mats[c % ncopy], x, y, M, K, N, ws, stream=st)
            del mats
        torch.cuda.synchronize()
        if w.w4g128_workspace_status(ws, st) != 0:
            print("device status word set", file=sys.stderr)
            return 1
    print("ok")
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of identical untimed steps before timing")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--target", choices=["layer", "lm_head", "single"], help="profiler target: untimed calls, no JSON")
    ap.add_argument("--shape", default="4096,4096", help="with --target single: K,N of the matrix")
    ap.add_argument("--m", default="1", help="with --target: comma-separated M values")
    ap.add_argument("--calls", type=int, default=2, help="with --target: calls per M")
    ap.add_argument("--record", default=None, help="append the JSON line to DIR/<date>-<host>/bench.jsonl")
    args = ap.parse_args()
    if args.target:
        return run_target(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
