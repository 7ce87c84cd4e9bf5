#!/usr/bin/env python3
"""Throughput of the tensor-sliced MLP block forward+backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mtnlg] [--impl ours|reference]

One step = every micro-batch of the workload through mlp_fwd + mlp_bwd (all
slices in turn, partial sums reduced on the device, fp32 weight gradients
accumulated).  Prints one JSON line (rank 0).  Under torchrun each rank runs its
own replica of the workload (weak scaling, no collective on the data path).

Workload default: the MT-NLG-layer-shaped block, 2048 tokens, h 20480, ffn 81920,
t = 8 slices, one micro-batch; every input is seeded synthetic data.
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

NOMINAL_BF16_DENSE_TFLOPS = 2250.0
METRIC = "MLP block fwd+bwd TFLOP/s and % of GB300 dense-BF16 peak (1 GPU)"
UNIT = "TFLOP/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ----------------------------------------------------------------------------- ncu traffic
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "gemm_tc_dram_traffic.json")
GEMM_SOURCES = ["gemm_tc.cuh", "ptx.cuh", "block_math.cuh", "gemm_host.cuh"]
# Sustained peak only for timed regions at least this long (seconds); shorter
# regions run at the burst rate the driver measured with a 10-iteration matmul.
SUSTAINED_MIN_S = 3.0


def gemm_source_hash() -> str:
    """sha256 of the GEMM sources with // comments and blank lines removed, so that
    an edit of comments alone keeps a capture valid and any code change voids it."""
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "transformer_lm_megatron_gb300", "csrc", name)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update((code + "\n").encode())
    return h.hexdigest()


def gemm_traffic_per_launch(workload: str):
    """DRAM bytes (read + write) per GEMM launch of ``workload``, scaled from the
    committed ncu record (profiles/gemm_tc_dram_traffic.json: a capture of the six
    GEMM launches of one slice-sized block, scaled to a full launch by the units
    each processes), or None if there is no record for the workload or the GEMM
    code changed since it was taken (the record holds gemm_source_hash())."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None
    with open(TRAFFIC_RECORD) as fh:
        rec = json.load(fh)
    if rec.get("source_sha256") != gemm_source_hash():
        return None
    full = rec.get("scaled_to", {}).get(workload)
    if not full:
        return None
    return float(full["bytes_per_launch_avg"])


def step_time_summary(step_ms):
    """Median, min and max of per-step times (ms)."""
    v = sorted(step_ms)
    n = len(v)
    med = v[n // 2] if n % 2 else 0.5 * (v[n // 2 - 1] + v[n // 2])
    return {"median": med, "min": v[0], "max": v[-1]}


# the GB300's nominal HBM3e bandwidth (the spec sheet's figure), reported beside the measured one
NOMINAL_HBM_GBPS = 7900.0


def hbm_kernel_rooflines(trace, wl, peaks, reset_ms):
    """Achieved GB/s of the element-wise kernels against the measured HBM copy
    bandwidth, from algorithmic bytes (each tensor read or written once)."""
    T, h, F = wl.tokens, wl.h, wl.ffn
    summ = trace.summary()
    out = {}
    spec = {10: ("dropout backward + db (B1)", 4 * T * h + 4 * h),
            11: ("column sum da", 2 * T * F + 4 * F),
            15: ("transposed copies of X and dZ for B3/B4", 8 * T * h)}
    for kind, (name, nbytes) in spec.items():
        if kind in summ and summ[kind][0] > 0:
            ms = summ[kind][1] / summ[kind][0]
            gbs = nbytes / (ms / 1e3) / 1e9
            out[name] = {"bytes_per_launch": nbytes, "avg_ms": ms, "achieved_GBps": gbs,
                         "frac": gbs / peaks["hbm_gbs"], "frac_of_nominal": gbs / NOMINAL_HBM_GBPS}
    if reset_ms:
        nbytes = 4 * (2 * h * F + F + h)
        gbs = nbytes / (reset_ms / 1e3) / 1e9
        out["grad_accum_reset (R0)"] = {"bytes_per_launch": nbytes, "avg_ms": reset_ms, "achieved_GBps": gbs,
                                        "frac": gbs / peaks["hbm_gbs"], "frac_of_nominal": gbs / NOMINAL_HBM_GBPS,
                                        "note": "4 launches per call, timed alone"}
    out["peak_GBps"] = peaks["hbm_gbs"]
    out["nominal_GBps"] = NOMINAL_HBM_GBPS
    return out


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest of every rank's value (the slowest rank's time); value itself on one rank."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica (weak scaling)."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle sample
def oracle_sample_inputs(wl, weights_host, n_tokens: int, slice_index: int = 0):
    """Float64 inputs of the CPU sample: ``n_tokens`` tokens and slice ``slice_index``
    (A_i columns, B_i rows) of the workload's seeded weights."""
    from oracle import mlp_oracle as orc
    from transformer_lm_megatron_gb300 import inputs as gin

    A, a, B, b = weights_host
    f = wl.f
    cols = slice(slice_index * f, (slice_index + 1) * f)
    X, dO = gin.make_microbatch(n_tokens, wl.h, 0)
    dec = lambda t: orc.bf16_to_f64(gin.bf16_bits(t))  # noqa: E731
    return dec(X), dec(dO), dec(A[:, cols]), dec(a[cols]), dec(B[cols, :]), dec(b)


def oracle_sample(wl, sample_inputs):
    """Times the oracle (float64, host cores) forward+backward on a prepared sample.
    Returns (seconds, algorithmic flops of the sample)."""
    from oracle import mlp_oracle as orc
    X64, dO64, A_i, a_i, B_i, b64 = sample_inputs
    t0 = time.perf_counter()
    fw = orc.mlp_fwd(X64, A_i, a_i, B_i, b64, 1, wl.p, wl.seed, mirror=True)
    orc.mlp_bwd(dO64, X64, A_i, B_i, fw["U"], fw["Y"], fw["keep"], 1, wl.p, mirror=True)
    dt = time.perf_counter() - t0
    return dt, 12 * X64.shape[0] * wl.h * A_i.shape[1]


def sampled_parity(wl, weights, X, dO, buf, stream, n_rows=4):
    """Max |gpu - oracle| / max |oracle| per output over ``n_rows`` token rows of one
    micro-batch at the benchmarked size (the float64 oracle in its bf16-mirroring
    mode, full rows over all slices; the fp32 weight gradients need every token and
    are left to the test suite)."""
    import numpy as np
    import torch
    from oracle import mlp_oracle as orc
    from transformer_lm_megatron_gb300 import mlp
    rows = np.unique(np.linspace(0, wl.tokens - 1, n_rows).astype(np.int64))
    mlp.block_step(wl, weights, X, dO, buf, token_offset=0, slice_mode="all", stream=stream, accumulate=False)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    ridx = torch.as_tensor(rows, device=X.device)
    A, a, B, b = weights
    ref = orc.rows_fwd_bwd(rows, orc.Bf16Matrix(bits(X)), orc.Bf16Matrix(bits(dO)), orc.Bf16Matrix(bits(A)),
                           orc.bf16_to_f64(bits(a)), orc.Bf16Matrix(bits(B)), orc.bf16_to_f64(bits(b)), wl.t, wl.p,
                           wl.seed, 0, mirror=True)
    out = {"rows": [int(r) for r in rows], "oracle_mode": "bf16-mirroring, float64"}
    for name in ("U", "Y", "O", "dZ", "dU", "dX"):
        g = orc.bf16_to_f64(bits(getattr(buf, name).index_select(0, ridx)))
        r = ref[name]
        den = float(np.max(np.abs(r)))
        out[f"{name}_max_rel_err"] = float(np.max(np.abs(g - r)) / den) if den > 0 else float(np.max(np.abs(g)))
    out["tolerance"] = 1e-2
    return out


def workload_config(wl, slice_mode, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": wl.name, "tokens": wl.tokens, "h": wl.h, "ffn": wl.ffn, "t": wl.t,
            "micro_batches": wl.k, "dropout": wl.p, "slice_calls": slice_mode,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, all slices on-device",
            "l2": "inputs larger than L2 (bf16 weights %.1f GB, fp32 gradients %.1f GB)"
                  % (4 * wl.h * wl.ffn / 1e9, 8 * wl.h * wl.ffn / 1e9)}


def oracle_workload_time(wl, n_mb):
    """The whole oracle (float64 numpy on the host cores), forward + backward of the
    first n_mb micro-batches of a workload over all its slices, gradients summed:
    the CPU baseline of the smaller workloads."""
    from oracle import mlp_oracle as orc
    from transformer_lm_megatron_gb300 import inputs as gin
    dec = lambda t: orc.bf16_to_f64(gin.bf16_bits(t))  # noqa: E731
    A, a, B, b = (dec(x) for x in gin.make_weights(wl.h, wl.ffn))
    mbs = [tuple(dec(x) for x in gin.make_microbatch(wl.tokens, wl.h, j)) for j in range(n_mb)]
    t0 = time.perf_counter()
    for j, (X, dO) in enumerate(mbs):
        fw = orc.mlp_fwd(X, A, a, B, b, wl.t, wl.p, wl.seed, token_offset=j * wl.tokens, mirror=True)
        orc.mlp_bwd(dO, X, A, B, fw["U"], fw["Y"], fw["keep"], wl.t, wl.p, mirror=True)
    dt = time.perf_counter() - t0
    flops = 12 * wl.tokens * wl.h * wl.ffn * n_mb
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": _cpu_cores(), "kind": "oracle",
            "sample": f"{n_mb} of {wl.k} micro-batches, all {wl.t} slices, fwd+bwd, float64 numpy, {dt:.1f} s"}


def other_workloads(dev, stream, steps=5, warmup=2, cpu_oracle=True):
    """fwd+bwd TFLOP/s of the smaller named workloads, each step being all of its
    micro-batches (the first writes the gradients, the rest add).  The sweep runs
    one slice per call, as its workload description says; the others all slices
    per call.  Each step is timed as issued (eager) and as the replay of a CUDA graph
    captured from it: the library keeps no per-call host state that a replay would
    miss, and its device-side counters return to zero after every kernel."""
    import torch
    from transformer_lm_megatron_gb300 import inputs as gin
    from transformer_lm_megatron_gb300 import mlp
    out = {}
    for name in ("tiny", "small", "mid", "sweep1", "sweep4", "sweep16", "sweep32"):
        w = gin.WORKLOADS[name]
        mode = "each" if name.startswith("sweep") else "all"
        weights = gin.make_weights(w.h, w.ffn, device=dev)
        mbs = [gin.make_microbatch(w.tokens, w.h, j, device=dev) for j in range(min(w.k, 4))]
        buf = mlp.BlockBuffers(w.tokens, w.h, w.ffn, w.t, device=dev)

        def step(s=stream):
            for j in range(w.k):
                X, dO = mbs[j % len(mbs)]
                mlp.block_step(w, weights, X, dO, buf, token_offset=j * w.tokens, slice_mode=mode, stream=s,
                               accumulate=j > 0)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        # the same step captured once and replayed
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(torch.cuda.current_stream(dev))
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize(dev)
        gms = g0.elapsed_time(g1) / steps
        del graph
        out[name] = {"tokens": w.tokens, "h": w.h, "ffn": w.ffn, "t": w.t, "micro_batches": w.k,
                     "slice_calls": mode, "ms_per_step": ms, "TFLOPs": w.flops_total() / (ms / 1e3) / 1e12,
                     "graph_ms_per_step": gms, "graph_TFLOPs": w.flops_total() / (gms / 1e3) / 1e12}
        del weights, mbs, buf
        # the whole oracle on the host cores: every micro-batch of tiny and small, one of mid
        n_mb = {"tiny": w.k, "small": w.k, "mid": 1}.get(name)
        if cpu_oracle and n_mb:
            out[name]["cpu_oracle"] = oracle_workload_time(w, n_mb)
    if mlp.mlp_sync_status(stream) != mlp.MLP_OK:
        raise RuntimeError(mlp.last_error())
    return out




def attn_flops(tokens, h, seq_len):
    """Algorithmic FLOPs of one attention-block forward + backward: the QKV and
    output projections (8 T h^2 forward, twice that backward) and the attention
    products over the causal lower triangle only (Q K^T and P V: 2 T L h forward;
    dV, dP, dQ, dK: 4 T L h backward), i.e. half of the full L x L blocks."""
    return 24 * tokens * h * h + 6 * tokens * seq_len * h


def attn_bench(wl, dev, stream, args):
    import torch
    from transformer_lm_megatron_gb300 import mlp
    from transformer_lm_megatron_gb300 import inputs as gin
    c = dict(gin.ATTN_MTNLG)
    if args.attn_h:
        # the same head size (h / heads) and sequence at a smaller hidden size
        c["nh"] = args.attn_h * c["nh"] // c["h"]
        c["h"] = args.attn_h
    h, nh, t, L, T = c["h"], c["nh"], c["t"], c["seq_len"], c["tokens"]
    w, X, dOut = gin.make_attn_inputs(h, T, device=dev)
    buf = mlp.AttnBuffers(T, h, nh, L, device=dev)

    def step():
        mlp.attn_step(h, nh, t, L, wl.p, wl.seed, w, X, dOut, buf, accumulate=False, stream=stream)

    for _ in range(max(args.warmup, 3) if args.attn_only else 3):
        step()
    torch.cuda.synchronize(dev)
    n = args.steps if args.attn_only else 10
    tr = mlp.Trace(capacity=40 * n)
    tr.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    tr.stop()
    ms = e0.elapsed_time(e1) / n
    if mlp.mlp_sync_status(stream) != mlp.MLP_OK:
        raise RuntimeError(mlp.last_error())
    flops = attn_flops(T, h, L)
    summ = tr.summary()
    kernels = {mlp.TRACE_NAMES.get(k, str(k)): {"launches": v[0] // n, "ms_per_step": v[1] / n}
               for k, v in sorted(summ.items())}
    gemm_ms = summ.get(20, (0, 0.0, 0))[1] / n
    out = {"shape": dict(c), "flops_per_step": flops, "ms_per_step": ms, "value": flops / (ms / 1e3) / 1e12,
           "unit": "TFLOP/s", "gemm_ms_per_step": gemm_ms,
           "gemm_achieved_TFLOPs": flops / (gemm_ms / 1e3) / 1e12 if gemm_ms else None,
           "kernels": kernels,
           "note": "attention products counted over the causal lower triangle; tiles wholly above the diagonal "
                   "are skipped, the rest of each diagonal tile is computed and masked"}
    del buf, w
    return out


def adam_oracle_sample(n=1 << 22):
    """The Adam oracle (float64 numpy) on 4 Mi parameters, in the same unit as the GPU figure."""
    import numpy as np
    from oracle import adam_oracle as ado
    rng = np.random.default_rng(0)
    g, w = rng.standard_normal(n), rng.standard_normal(n) * 0.02
    m, v = np.zeros(n), np.zeros(n)
    t0 = time.perf_counter()
    ado.adam_step(g, w, m, v, 1, 5e-5, 0.9, 0.95, 1e-8, 0.1)
    dt = time.perf_counter() - t0
    return {"value": 30 * n / dt / 1e9, "unit": "GB/s (30 B per parameter)", "cores": _cpu_cores(),
            "kind": "oracle", "sample": f"{n} parameters, one step, float64 numpy, {dt * 1e3:.0f} ms"}


def _cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def _sample_weights_host(wl, device):
    """Slice-0 weights of the workload, drawn on ``device`` with the seeded generator, on the host."""
    from transformer_lm_megatron_gb300 import inputs as gin
    w = gin.make_weights(wl.h, wl.ffn, device=device)
    return tuple(x.cpu() for x in w)


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, wl, rank, world):
    """The CPU oracle timed on the host cores: each step is a bounded sample."""
    if rank != 0:
        return
    from transformer_lm_megatron_gb300 import inputs as gin
    w = gin.make_weights(wl.h, wl.ffn, device="cpu") if wl.h * wl.ffn <= 64 * 2**20 else None
    if w is None:
        import torch
        w = _sample_weights_host(wl, "cuda" if torch.cuda.is_available() else "cpu")
    n_tok = args.cpu_tokens
    sample = oracle_sample_inputs(wl, w, n_tok)
    del w
    for _ in range(args.warmup):
        oracle_sample(wl, sample)
    times, flops = [], 0
    for _ in range(args.steps):
        dt, fl = oracle_sample(wl, sample)
        times.append(dt)
        flops = fl
    total = sum(times)
    value = flops * args.steps / total / 1e12
    desc = f"{n_tok} of {wl.tokens} tokens x slice 0 of {wl.t} (f={wl.f}), fwd+bwd, float64 numpy, per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args.slice_mode, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cpu_cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def run_ours(args, wl, rank, world, dist):
    import torch
    from transformer_lm_megatron_gb300 import build as gb_build
    from transformer_lm_megatron_gb300 import inputs as gin
    from transformer_lm_megatron_gb300 import mlp

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gb_build.build()
    mlp.load()
    mlp.mlp_set_tile_scheduler({"default": -1, "static": 0, "dynamic": 1}[args.tile_scheduler])
    mlp.mlp_set_wgrad_transpose({"default": -1, "off": 0, "on": 1}[args.wgrad_transpose])
    if args.attn_only:
        # the attention block alone (the next row), e.g. for a counter capture of its kernels
        out = attn_bench(wl, dev, torch.cuda.current_stream(dev), args)
        if rank == 0:
            print(json.dumps({"attn_block": out}), flush=True)
        return

    weights = gin.make_weights(wl.h, wl.ffn, device=dev)
    mbs = [gin.make_microbatch(wl.tokens, wl.h, j, device=dev) for j in range(wl.k)]
    buf = mlp.BlockBuffers(wl.tokens, wl.h, wl.ffn, wl.t, device=dev)
    stream = torch.cuda.current_stream(dev)

    def reset():
        mlp.grad_accum_reset(wl.h, wl.ffn, buf.dA, buf.da, buf.dB, buf.db, stream=stream)

    def step():
        if args.reset_each_step:
            reset()
        # one optimizer step's worth of micro-batches: the first writes the fp32
        # gradients (accumulate = 0), the others add to them
        for j, (X, dO) in enumerate(mbs):
            mlp.block_step(wl, weights, X, dO, buf, token_offset=j * wl.tokens, slice_mode=args.slice_mode,
                           stream=stream, accumulate=(j > 0 or args.reset_each_step))

    mlp.grad_accum_reset(wl.h, wl.ffn, buf.dA, buf.da, buf.dB, buf.db, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if mlp.mlp_sync_status(stream) != mlp.MLP_OK:
        raise RuntimeError(mlp.last_error())

    # ---- timed region (device time, CUDA events on the launching stream)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    trace = mlp.Trace(capacity=args.steps * 80 * wl.k) if args.trace else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n_launch0 = mlp.mlp_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if trace:
        trace.start()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps - 1)]
    ev0.record(stream)
    for i in range(args.steps):
        step()
        if i < args.steps - 1:
            step_ev[i].record(stream)  # step boundaries, for the per-step spread
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if trace:
        trace.stop()
    bounds = [ev0] + step_ev + [ev1]
    step_ms = [bounds[i].elapsed_time(bounds[i + 1]) for i in range(args.steps)]
    n_launch = mlp.mlp_launch_count() - n_launch0

    # ---- the += form of the same step, inside the same clock record: the
    # accumulators are zeroed by grad_accum_reset OUTSIDE the event-timed region,
    # then every micro-batch adds its gradients (fp32 reduce-add epilogues).
    acc_form = None
    if not args.no_accumulate_form:
        def acc_step():
            for j, (X, dO) in enumerate(mbs):
                mlp.block_step(wl, weights, X, dO, buf, token_offset=j * wl.tokens, slice_mode=args.slice_mode,
                               stream=stream, accumulate=True)
        for _ in range(2):
            reset()
            acc_step()
        torch.cuda.synchronize(dev)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(2 * args.steps)]
        for i in range(args.steps):
            r0, r1 = pairs[2 * i]
            a0, a1 = pairs[2 * i + 1]
            r0.record(stream)
            reset()
            r1.record(stream)
            a0.record(stream)
            acc_step()
            a1.record(stream)
        torch.cuda.synchronize(dev)
        acc_ms = max_over_ranks(sum(pairs[2 * i + 1][0].elapsed_time(pairs[2 * i + 1][1]) for i in range(args.steps)),
                                dist, dev)
        reset_ms_total = sum(pairs[2 * i][0].elapsed_time(pairs[2 * i][1]) for i in range(args.steps))
        acc_form = {"value": job_throughput(wl.flops_total(), args.steps, world, acc_ms), "unit": UNIT,
                    "ms_per_step": acc_ms / args.steps, "reset_ms_per_step": reset_ms_total / args.steps,
                    "grad_init": "grad_accum_reset before each step, outside the timed events; every micro-batch "
                                 "adds (+=) into dA, da, dB, db",
                    "steps": args.steps}
    if dist is not None:
        dist.barrier()
    clock_info = clocks.stop() if clocks else None
    ms = ev0.elapsed_time(ev1)
    if mlp.mlp_sync_status(stream) != mlp.MLP_OK:
        raise RuntimeError(mlp.last_error())
    ms = max_over_ranks(ms, dist, dev)
    flops_step = wl.flops_total()
    value = job_throughput(flops_step, args.steps, world, ms)

    # ---- end to end through the public API: pinned host inputs in, results out.
    # Every micro-batch's X and dO are copied host->device and its O and dX
    # device->host inside the timed region.  The copies run on a second stream and
    # are double-buffered, so micro-batch g+1's inputs arrive while g computes and
    # g's outputs leave while g+1 computes.
    e2e = None
    if not args.no_e2e:
        hX = [X.cpu().pin_memory() for X, _ in mbs]
        hdO = [dO.cpu().pin_memory() for _, dO in mbs]
        hO = [torch.empty_like(X, device="cpu").pin_memory() for X, _ in mbs]
        hdX = [torch.empty_like(X, device="cpu").pin_memory() for X, _ in mbs]
        x_in = [torch.empty_like(mbs[0][0]) for _ in range(2)]
        do_in = [torch.empty_like(mbs[0][1]) for _ in range(2)]
        alt = mlp.BlockBuffers(wl.tokens, wl.h, wl.ffn, wl.t, device=dev)
        for name in ("dA", "da", "dB", "db"):  # one set of gradient accumulators
            setattr(alt, name, getattr(buf, name))
        bufs = [buf, alt]
        cs = torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n_steps, start_event):
            total = n_steps * wl.k
            cs.wait_event(start_event)

            def h2d(g):
                slot, j = g % 2, g % wl.k
                with torch.cuda.stream(cs):
                    if g >= 2:
                        cs.wait_event(comp_done[slot])  # micro-batch g-2 no longer reads this slot
                    x_in[slot].copy_(hX[j], non_blocking=True)
                    do_in[slot].copy_(hdO[j], non_blocking=True)
                    in_ready[slot].record(cs)

            h2d(0)
            for g in range(total):
                slot, j = g % 2, g % wl.k
                if g + 1 < total:
                    h2d(g + 1)
                stream.wait_event(in_ready[slot])
                if g >= 2:
                    stream.wait_event(out_done[slot])  # outputs of micro-batch g-2 have left
                mlp.block_step(wl, weights, x_in[slot], do_in[slot], bufs[slot], token_offset=j * wl.tokens,
                               slice_mode=args.slice_mode, stream=stream,
                               accumulate=(j > 0 or args.reset_each_step))
                comp_done[slot].record(stream)
                with torch.cuda.stream(cs):
                    cs.wait_event(comp_done[slot])
                    hO[j].copy_(bufs[slot].O, non_blocking=True)
                    hdX[j].copy_(bufs[slot].dX, non_blocking=True)
                    out_done[slot].record(cs)
            stream.wait_stream(cs)

        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_run(2, w0)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps, e0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ems = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        # the last step's outputs reached the host intact
        ok = torch.equal(hO[wl.k - 1], bufs[(args.steps * wl.k - 1) % 2].O.cpu())
        act = wl.tokens * wl.h * 2 * wl.k
        e2e = {"value": job_throughput(flops_step, args.steps, world, ems), "unit": UNIT,
               "h2d_bytes_per_step": 2 * act, "d2h_bytes_per_step": 2 * act, "ms_per_step": ems / args.steps,
               "copies": "H2D/D2H on a second stream, double-buffered across micro-batches",
               "outputs_checked": bool(ok)}

    # ---- next row: the mixed-precision Adam step over the block's parameters,
    # reading the fp32 gradients the step accumulated (30 bytes per parameter).
    adam = None
    if not args.no_adam:
        masters = [w.float() for w in weights]
        ms_state = [torch.zeros_like(x) for x in masters]
        vs_state = [torch.zeros_like(x) for x in masters]
        grads = [buf.dA, buf.da, buf.dB, buf.db]
        hp = dict(lr=5e-5, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, grad_scale=1.0 / wl.k)

        def adam_all(step):
            for gr, w32, mm, vv, w16 in zip(grads, masters, ms_state, vs_state, weights):
                mlp.adam_step(gr, w32, mm, vv, w16, step=step, stream=stream, **hp)

        for s_ in range(1, 3):
            adam_all(s_)
        torch.cuda.synchronize(dev)
        a_steps = 10
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for s_ in range(3, 3 + a_steps):
            adam_all(s_)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        a_ms = a0.elapsed_time(a1) / a_steps
        n_params = sum(x.numel() for x in masters)
        a_bytes = 30 * n_params
        adam = {"params": n_params, "ms_per_step": a_ms, "bytes_per_step": a_bytes,
                "achieved_GBps": a_bytes / (a_ms / 1e3) / 1e9, "launches_per_step": 4,
                "hyper": {k: v for k, v in hp.items()}}
        del masters, ms_state, vs_state

    # ---- the other named workloads (secondary figures; the headline is the MT-NLG layer)
    others = None
    if not args.no_others and wl.name == "mtnlg":
        others = other_workloads(dev, stream, cpu_oracle=(rank == 0 and world == 1 and not args.no_cpu_baseline))

    # ---- next row: the tensor-sliced self-attention block at the MT-NLG layer
    # shape (h 20480, 128 heads, t 8, one 2048-token sequence), forward + backward
    attn = None
    if not args.no_attn and wl.name == "mtnlg":
        attn = attn_bench(wl, dev, stream, args)

    # ---- HBM-bound kernels: the reset pass (R0) is not part of a step when the
    # first micro-batch writes the gradients, so it is traced here on its own.
    reset_ms = None
    if args.trace:
        rt = mlp.Trace(capacity=64)
        rt.start()
        for _ in range(3):
            mlp.grad_accum_reset(wl.h, wl.ffn, buf.dA, buf.da, buf.dB, buf.db, stream=stream)
        torch.cuda.synchronize(dev)
        rt.stop()
        reset_ms = sum(t for _, _, t in rt.entries) / 3

    if rank != 0:
        return
    peaks = _peaks()
    roofline = None
    if trace:
        timed_s = ms / 1e3
        if timed_s >= SUSTAINED_MIN_S:
            peak, kind = peaks["bf16_sustained"], f"bf16 dense sustained ({peaks['source']}; timed region {timed_s:.2f} s)"
        else:
            peak, kind = peaks["bf16_burst"], f"bf16 dense burst ({peaks['source']}; timed region {timed_s:.2f} s)"
        roofline = trace.roofline(peak, kind)
        if roofline is not None:
            roofline["hbm_kernels"] = hbm_kernel_rooflines(trace, wl, peaks, reset_ms)
            roofline["traffic"] = gemm_traffic_per_launch(wl.name)
            roofline["traffic_unit"] = ("bytes per GEMM launch (DRAM read + write; ncu capture of a slice-sized "
                                        "block scaled to a full launch, profiles/gemm_tc_dram_traffic.json)")
            roofline["algorithmic_bytes_per_launch"] = 2 * (wl.tokens * wl.h + wl.h * wl.ffn + wl.tokens * wl.ffn)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        w_host = tuple(x.cpu() for x in weights)
        dt, fl = oracle_sample(wl, oracle_sample_inputs(wl, w_host, args.cpu_baseline_tokens))
        del w_host
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": _cpu_cores(), "kind": "oracle",
               "sample": f"{args.cpu_baseline_tokens} of {wl.tokens} tokens x slice 0 of {wl.t} (f={wl.f}), fwd+bwd, "
                         f"float64 numpy, {dt:.1f} s"}
        cpu["parity"] = sampled_parity(wl, weights, mbs[0][0], mbs[0][1], buf, stream)
    if adam is not None:
        adam["peak_GBps"] = peaks["hbm_gbs"]
        adam["frac"] = adam["achieved_GBps"] / peaks["hbm_gbs"]
        if world == 1 and not args.no_cpu_baseline:
            adam["cpu_baseline"] = adam_oracle_sample()
    burst = peaks["bf16_burst"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "step_ms": step_time_summary(step_ms), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "pct_of_peak": 100.0 * value / (world * burst),
        "peak_tflops": {"value": burst, "kind": f"bf16 dense burst, {peaks['source']}"},
        # the nominal dense (no 2:4 sparsity) bf16 rate of a GB300, 2.25 PFLOP/s: the
        # stricter of the two denominators
        "pct_of_nominal_peak": 100.0 * value / (world * NOMINAL_BF16_DENSE_TFLOPS),
        "config": workload_config(wl, args.slice_mode, world),
        "run": {"tile_order": args.tile_scheduler,
                "wgrad_transposed_operands": args.wgrad_transpose,
                "grad_init": ("grad_accum_reset + every micro-batch adds (inside the timed region)"
                              if args.reset_each_step else
                              "first micro-batch of each step writes dA/da/dB/db, later ones add; no reset pass")},
        "gpu_launches": n_launch,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "accumulate_form": acc_form,
        "clocks": clock_info,
        "other_workloads": others,
        "next_rows": {"adam_step": adam, "attn_block": attn},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mtnlg")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--slice-mode", default="all", choices=["all", "each"])
    ap.add_argument("--cpu-tokens", type=int, default=32,
                    help="tokens of the oracle sample per step of the reference arm")
    ap.add_argument("--cpu-baseline-tokens", type=int, default=2048,
                    help="tokens of the timed oracle sample of this arm's cpu_baseline (10-15 s of CPU work on "
                         "16 cores for the MT-NLG layer's slice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-trace", dest="trace", action="store_false")
    ap.add_argument("--no-adam", action="store_true", help="skip the Adam-step measurement")
    ap.add_argument("--no-attn", action="store_true", help="skip the attention-block measurement")
    ap.add_argument("--no-others", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--attn-only", action="store_true",
                    help="time only the attention block (--steps timed, --warmup untimed steps)")
    ap.add_argument("--attn-h", type=int, default=0,
                    help="hidden size of the attention block (default 20480; the head size stays 160)")
    ap.add_argument("--tile-scheduler", default="default", choices=["default", "dynamic", "static"],
                    help="order in which the GEMMs hand out output tiles (results are bit-identical): "
                         "default = dynamic for the batched attention products only")
    ap.add_argument("--wgrad-transpose", default="default", choices=["default", "on", "off"],
                    help="whether the weight-gradient GEMMs read transposed copies of X and dZ (bit-identical "
                         "results): default = for GEMMs of 1e12 FLOP or more")
    ap.add_argument("--no-accumulate-form", action="store_true",
                    help="skip timing the += form (reset outside the timed region, every micro-batch adds)")
    ap.add_argument("--reset-each-step", action="store_true",
                    help="time grad_accum_reset + all micro-batches adding, instead of the first writing")
    args = ap.parse_args()

    from transformer_lm_megatron_gb300 import inputs as gin
    wl = gin.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    run_ours(args, wl, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
