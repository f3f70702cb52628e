#!/usr/bin/env python3
"""Throughput of the exact tiled attention library on GB300; prints ONE JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
  forward (causal) and backward (preprocess, dK/dV pass, dQ pass) at
  B=1, H=32, N=8192, d=128 — the top of the 1k-8k fwd/bwd sweep — and
  split-KV decode (16 splits + combine) at B=32, H=32, Nk=4096, d=128.
``value`` is forward+backward TFLOP/s (algorithmic FLOPs: 4 B H Nq Nk d / 2 for
the causal forward, 2.5x that for the backward) over the device time of those
kernels; decode KV-read GB/s is reported under ``decode``.  Inputs are resident
in HBM and larger than L2 (129 MB), so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path shards by head / batch with no exchange): ``value`` sums the ranks'
work over the slowest rank's time.  ``--impl reference`` times the fp64 CPU
oracle (the only other implementation there is) on the host cores, on a
bounded sample of the same workload, in the same metric.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd/bwd TFLOP/s (bf16, d=128, N 1k-8k, % of peak); decode KV-read GB/s"
B, H, N, D = 1, 32, 8192, 128
DEC_B, DEC_H, DEC_NK, DEC_SPLITS = 32, 32, 4096, 16
SCALE = 1.0 / math.sqrt(D)
FWD_FLOPS = 4.0 * B * H * N * N * D / 2          # causal
BWD_FLOPS = 2.5 * FWD_FLOPS
DKDV_FLOPS = BWD_FLOPS * 4 / 5                   # S, dP, dV, dK of the five products
DEC_BYTES = 2.0 * DEC_B * DEC_H * DEC_NK * D * 2  # K and V cache, read once
CONFIG = {
    "workload": "fwd+bwd causal B=1 H=32 N=8192 d=128 (top of the 1k-8k sweep); "
                "decode B=32 H=32 Nk=4096 d=128 16 splits",
    "fwd_bwd": {"B": B, "H": H, "N": N, "d": D, "causal": True, "scale": "1/sqrt(d)"},
    "decode": {"B": DEC_B, "H": DEC_H, "Nk": DEC_NK, "d": D, "splits": DEC_SPLITS},
    "inputs": "iid N(0,1) bf16, resident in HBM",
    "l2": "inputs larger than L2 (129 MB); no flush",
}
SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def peaks():
    """Measured HBM copy bandwidth and cuBLAS bf16 GEMM rate.  ``bf16`` is the
    burst figure (a GEMM timed alone at full clocks): the right denominator for
    the kernels timed here, whose timed regions last tens of milliseconds at the
    maximum SM clock.  ``bf16_sustained`` was taken over a seconds-long loop at
    power-capped clocks and is reported for context only."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16": float(m["bf16_tflops"]),
                "bf16_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + SMI_FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        def pump():
            for line in self.proc.stdout:
                self.rows.append((time.time(), [x.strip() for x in line.split(",")]))
        self.thread = threading.Thread(target=pump, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if len(r) > 9 and num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if len(r) > 9 and num(r[3]) is not None]
        reasons = set()
        for r in rows:
            if len(r) <= 9:
                continue
            for name, val in (("hw_slowdown", r[6]), ("hw_thermal_slowdown", r[7]),
                              ("sw_thermal_slowdown", r[8]), ("sw_power_cap", r[9])):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max([num(r[4]) or 0 for r in rows if len(r) > 4])}


def profiled_traffic(profile, source):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's source has changed since the capture (its hash no longer matches)."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        fields = dict(l.split(":", 1) for l in text.splitlines() if l.startswith(("traffic_bytes", "source_sha")))
        want = fields["source_sha256_16"].split()[0]
        src = os.path.join(ROOT, "exact_tiled_attention_21_gb300", "csrc", source)
        have = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return int(fields["traffic_bytes_per_launch"]) if want == have else None
    except (OSError, KeyError, ValueError):
        return None


def reduce_max(x, dist=None, device=None):
    """Max of a host float over all ranks (identity without a process group).
    The tensor lives on ``device`` (a CUDA device for NCCL, the CPU for gloo)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_rank, seconds_per_rank, world, dist=None, device=None):
    """Weak scaling over independent replicas: all ranks' work over the slowest rank's time."""
    return world * work_per_rank / reduce_max(seconds_per_rank, dist, device)


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample(seconds, max_rows=None, seed=2):
    """Time the fp64 oracle (naive materialised fwd + bwd) on 256-row query
    blocks of the fwd/bwd workload — head (0, 0), then (0, 1), ... — until
    ``seconds`` of CPU time have passed.  Returns (flops, secs, rows)."""
    import numpy as np
    from exact_tiled_attention_21_gb300 import synthetic as syn
    from oracle import naive
    flops, done, secs = 0.0, 0, 0.0
    for h in range(H):
        q, k, v, do = (syn.head(seed, tag, 0, h, N, D).double().numpy()
                       for tag in (syn.TAG_Q, syn.TAG_K, syn.TAG_V, syn.TAG_DO))
        t0 = time.perf_counter()
        for blk in np.random.default_rng(seed + h).permutation(N // 256):
            rows = np.arange(blk * 256, blk * 256 + 256)
            naive.forward(q[rows], k, v, SCALE, True, rows=rows, Nq=N)
            naive.backward(q[rows], k, v, do[rows], SCALE, True, rows=rows, Nq=N)
            flops += 4.0 * D * float((rows + 1).sum()) * 3.5  # causal row i sees i+1 keys; fwd + 2.5x bwd
            done += 256
            if secs + time.perf_counter() - t0 >= seconds or (max_rows and done >= max_rows):
                return flops, secs + time.perf_counter() - t0, done
        secs += time.perf_counter() - t0
    return flops, secs, done


def oracle_sample_o2(seconds, seed=2):
    """Time the C two-pass oracle (forward only, one thread per host core) on
    256-row query blocks of the fwd workload until ``seconds`` have passed.
    Returns (flops, secs, rows, threads)."""
    import numpy as np
    from exact_tiled_attention_21_gb300 import synthetic as syn
    from oracle import twopass
    threads = os.cpu_count() or 1
    flops, done, secs = 0.0, 0, 0.0
    for h in range(H):
        q, k, v = (syn.head(seed, tag, 0, h, N, D).double().numpy() for tag in (syn.TAG_Q, syn.TAG_K, syn.TAG_V))
        t0 = time.perf_counter()
        for blk in np.random.default_rng(seed + h).permutation(N // 256):
            rows = np.arange(blk * 256, blk * 256 + 256)
            twopass.forward(q[rows], k, v, SCALE, True, rows=rows, Nq=N, nthreads=threads)
            flops += 4.0 * D * float((rows + 1).sum())
            done += 256
            if secs + time.perf_counter() - t0 >= seconds:
                return flops, secs + time.perf_counter() - t0, done, threads
        secs += time.perf_counter() - t0
    return flops, secs, done, threads


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def run_reference(args, rank):
    if rank != 0:
        return 0
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step)
    tot_f, tot_t, tot_r = 0.0, 0.0, 0
    for _ in range(args.steps):
        f, t, r = oracle_sample(per_step)
        tot_f, tot_t, tot_r = tot_f + f, tot_t + t, tot_r + r
    value = tot_f / tot_t / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": CONFIG,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: numpy fp64 naive fwd+bwd of 256-row query blocks of heads "
                                   "(0,0), (0,1), ..., N=8192 causal, for %.1f s (%d rows in all)" % (per_step, tot_r)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ sweep
SWEEP_N = (1024, 2048, 4096, 8192)
LONG_N = 131072


def run_sweep(fa, dev, stream, g, barrier, sampler):
    """Every workload of the 1k-8k protocol and the other configurations, each
    timed on its own: the forward and the backward of B=1, H=32, d=128 causal at
    N = 1024 ... 8192; the forward at B=2, H=32, N=4096 causal and non-causal;
    the forward and backward under a causal 256-key sliding window (B=1, H=32,
    N=8192) and with per-sequence lengths 8192 / 5000 / 2500 / 700 (B=4, H=32,
    padded to 8192, causal), their FLOPs counted over the pairs the mask keeps;
    the long causal forward at N=131072 with its peak device memory; decode at
    B=32, H=32 for d=128 with Nk=4096 and Nk=4000 and for d=64, with 16 splits
    and with the automatic count; paged decode at B=32, Hq=32, Hkv=8 with 48-,
    80-, 40- and 20-token pages (d=128) and 48-token pages (d=64).  Each entry is
    the median over calls bracketed by CUDA events on the launching stream.  L2
    is flushed (a 256 MiB write) before every call whose inputs would otherwise
    stay in it; decode caches (>= 1 GiB) and paged caches (0.27-0.53 GB of K
    and V per call) are larger than L2.  Decode runs first and the long forward
    last, so the seconds-long full load of the latter cannot pull the clocks of
    the others down."""
    import torch
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def rnd(*shape, std=1.0):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        return (x * std).to(torch.bfloat16) if std != 1.0 else x.to(torch.bfloat16)

    def timed(call, reps, flush):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in evs:
            if flush:
                with torch.cuda.stream(stream):
                    flush_buf.fill_(1)
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)

    out = {"fwd_bwd_causal_B1_H32_d128": [], "fwd_B2_H32_N4096_d128": [], "decode_B32_H32": [],
           "decode_paged_B32_Hq32": [],
           "timing": "median of per-call CUDA-event times on the launching stream; L2 flushed before each "
                     "fwd/bwd call (256 MiB write, outside the events)",
           "bwd_modes": "bwd: fa_bwd (dK/dV pass + dQ pass, deterministic); bwd_fused: fa_bwd_fused (one pass, "
                        "dQ by fp32 reduce-adds, dQ bits vary run to run)",
           "_windows": {}}
    # decode shapes (the cache is read once per call; >= 1 GiB, larger than L2), each with the
    # headline's 16 splits and with the library's automatic count
    t0 = time.time()
    for nk, d in ((4096, 128), (4000, 128), (4096, 64)):
        q = rnd(DEC_B, DEC_H, d)
        kc, vc = rnd(DEC_B, DEC_H, nk, d), rnd(DEC_B, DEC_H, nk, d)
        o = torch.empty_like(q)
        lse = torch.empty(DEC_B, DEC_H, device=dev, dtype=torch.float32)
        for sp in (DEC_SPLITS, 0):
            ws = torch.empty(fa.fa_decode_workspace_bytes(DEC_B, DEC_H, nk, d, sp), dtype=torch.uint8,
                             device=dev)
            call = lambda: fa.fa_decode(q, kc, vc, o, lse, DEC_B, DEC_H, nk, d, 1.0 / math.sqrt(d), sp, ws,
                                        ws.numel(), stream)
            for _ in range(3):
                call()
            ms = timed(call, 20, False)
            byt = 2.0 * DEC_B * DEC_H * nk * d * 2
            out["decode_B32_H32"].append({"Nk": nk, "d": d, "splits": sp if sp > 0 else "auto", "ms": ms,
                                          "gbs": byt / (ms * 1e-3) / 1e9})
            del ws
        del q, kc, vc, o, lse
    # paged decode at page sizes beside the headline's 16 tokens: 48 and 80 (the tensor-core kernel in
    # 16-row boxes), 40 (8-row boxes) and 20 (not a multiple of 8: the CUDA-core kernel); 4080 tokens
    # (or the nearest whole number of pages below 4096) per sequence, pages in a random order,
    # automatic splits
    for hkv, page, d in ((8, 48, 128), (8, 80, 128), (8, 40, 128), (8, 20, 128), (8, 48, 64)):
        mp = DEC_NK // page
        npages = DEC_B * mp
        kp, vp = rnd(npages, hkv, page, d), rnd(npages, hkv, page, d)
        q = rnd(DEC_B, DEC_H, d)
        table = torch.randperm(npages, generator=torch.Generator().manual_seed(page)).to(torch.int32)
        table = table.reshape(DEC_B, mp).to(dev)
        lens = torch.full((DEC_B,), mp * page, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(DEC_B, DEC_H, device=dev, dtype=torch.float32)
        ws = torch.empty(fa.fa_decode_paged_workspace_bytes(DEC_B, DEC_H, d, 0), dtype=torch.uint8, device=dev)
        call = lambda: fa.fa_decode_paged(q, kp, vp, table, lens, o, lse, DEC_B, DEC_H, hkv, page, mp, npages, d,
                                          1.0 / math.sqrt(d), 0, ws, ws.numel(), stream)
        for _ in range(3):
            call()
        ms = timed(call, 20, False)
        byt = 2.0 * DEC_B * hkv * mp * page * d * 2
        out["decode_paged_B32_Hq32"].append({"Hkv": hkv, "page": page, "d": d, "tokens": mp * page, "ms": ms,
                                             "gbs": byt / (ms * 1e-3) / 1e9})
        del kp, vp, q, table, lens, o, lse, ws
    out["_windows"]["decode"] = (t0, time.time())
    t0 = time.time()
    for n in SWEEP_N:
        q, k, v, dO = (rnd(1, H, n, D) for _ in range(4))
        o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
        lse = torch.empty(1, H, n, device=dev, dtype=torch.float32)
        ws = torch.empty(fa.fa_bwd_workspace_bytes(1, H, n, n, D), dtype=torch.uint8, device=dev)
        fwd = lambda: fa.fa_fwd(q, k, v, o, lse, 1, H, n, n, D, SCALE, True, stream)
        bwd = lambda: fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, 1, H, n, n, D, SCALE, True, ws, ws.numel(),
                                stream)
        for _ in range(3):
            fwd()
            bwd()
        wsf = torch.empty(fa.fa_bwd_fused_workspace_bytes(1, H, n, n, D), dtype=torch.uint8, device=dev)
        bwdf = lambda: fa.fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, 1, H, n, n, D, SCALE, True, wsf,
                                       wsf.numel(), stream)
        for _ in range(3):
            bwdf()
        reps = 20 if n <= 2048 else 10
        f_ms = timed(fwd, reps, True)
        b_ms = timed(bwd, reps, True)
        bf_ms = timed(bwdf, reps, True)
        fl = 4.0 * H * n * n * D / 2
        out["fwd_bwd_causal_B1_H32_d128"].append(
            {"N": n, "fwd_ms": f_ms, "fwd_tflops": fl / (f_ms * 1e-3) / 1e12,
             "bwd_ms": b_ms, "bwd_tflops": 2.5 * fl / (b_ms * 1e-3) / 1e12,
             "bwd_fused_ms": bf_ms, "bwd_fused_tflops": 2.5 * fl / (bf_ms * 1e-3) / 1e12})
        del q, k, v, dO, o, dq, dk, dv, lse, ws, wsf
    for causal in (False, True):
        q, k, v = (rnd(2, H, 4096, D) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty(2, H, 4096, device=dev, dtype=torch.float32)
        fwd = lambda: fa.fa_fwd(q, k, v, o, lse, 2, H, 4096, 4096, D, SCALE, causal, stream)
        for _ in range(3):
            fwd()
        f_ms = timed(fwd, 10, True)
        fl = 4.0 * 2 * H * 4096 * 4096 * D / (2 if causal else 1)
        out["fwd_B2_H32_N4096_d128"].append({"causal": causal, "fwd_ms": f_ms,
                                             "fwd_tflops": fl / (f_ms * 1e-3) / 1e12})
        del q, k, v, o, lse
    # the mask variants: a causal sliding window of 256 keys, and per-sequence lengths in a padded
    # batch; their FLOPs count only the (query, key) pairs the mask keeps
    nw, win = 8192, 256
    q, k, v, dO = (rnd(1, H, nw, D) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(1, H, nw, device=dev, dtype=torch.float32)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, H, nw, nw, D), dtype=torch.uint8, device=dev)
    fwd = lambda: fa.fa_fwd_window(q, k, v, o, lse, 1, H, nw, nw, D, SCALE, win, stream)
    bwd = lambda: fa.fa_bwd_window(q, k, v, o, lse, dO, dq, dk, dv, 1, H, nw, nw, D, SCALE, win, ws, ws.numel(),
                                   stream)
    for _ in range(3):
        fwd()
        bwd()
    f_ms, b_ms = timed(fwd, 10, True), timed(bwd, 10, True)
    fl = 4.0 * H * (win * nw - win * (win - 1) / 2) * D  # query i sees min(i + 1, 256) keys
    out["window_B1_H32_N8192_d128_W256"] = {"fwd_ms": f_ms, "fwd_tflops": fl / (f_ms * 1e-3) / 1e12,
                                            "bwd_ms": b_ms, "bwd_tflops": 2.5 * fl / (b_ms * 1e-3) / 1e12}
    del q, k, v, dO, o, dq, dk, dv, lse, ws
    lens = [8192, 5000, 2500, 700]
    nb = len(lens)
    q, k, v, dO = (rnd(nb, H, nw, D) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(nb, H, nw, device=dev, dtype=torch.float32)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(nb, H, nw, nw, D), dtype=torch.uint8, device=dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    fwd = lambda: fa.fa_fwd_varlen(q, k, v, o, lse, sl, sl, nb, H, nw, nw, D, SCALE, True, stream)
    bwd = lambda: fa.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, sl, sl, nb, H, nw, nw, D, SCALE, True, ws,
                                   ws.numel(), stream)
    for _ in range(3):
        fwd()
        bwd()
    f_ms, b_ms = timed(fwd, 10, True), timed(bwd, 10, True)
    fl = 4.0 * H * sum(n * (n + 1) / 2 for n in lens) * D
    out["varlen_causal_B4_H32_N8192_d128"] = {"lens": lens, "fwd_ms": f_ms,
                                              "fwd_tflops": fl / (f_ms * 1e-3) / 1e12, "bwd_ms": b_ms,
                                              "bwd_tflops": 2.5 * fl / (b_ms * 1e-3) / 1e12}
    del q, k, v, dO, o, dq, dk, dv, lse, ws, sl
    out["_windows"]["short"] = (t0, time.time())

    # long causal forward (last: its seconds of full load can bring the power cap in).  Its
    # memory: the device's used bytes (cudaMemGetInfo, which sees every allocation, the
    # library's included) and the torch allocator's peak, both over the inputs' own
    # footprint; the library allocates nothing, so both stay at the floor.
    barrier()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    q, k, v = (rnd(1, H, LONG_N, D, std=0.5) for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty(1, H, LONG_N, device=dev, dtype=torch.float32)
    floor = 4 * q.numel() * 2 + lse.numel() * 4
    fwd = lambda: fa.fa_fwd(q, k, v, o, lse, 1, H, LONG_N, LONG_N, D, SCALE, True, stream)
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    fwd()
    torch.cuda.synchronize(dev)
    tl0 = time.time()
    l_ms = timed(fwd, 5, False)
    tl1 = time.time()
    free1 = torch.cuda.mem_get_info(dev)[0]
    peak = torch.cuda.max_memory_allocated(dev) - base
    fl = 4.0 * H * LONG_N * LONG_N * D / 2
    out["fwd_long_causal_B1_H32_N131072_d128"] = {
        "fwd_ms": l_ms, "fwd_tflops": fl / (l_ms * 1e-3) / 1e12, "inputs": "N(0, 0.5^2) bf16",
        "peak_mib": peak / 2**20, "floor_mib": floor / 2**20,
        "device_used_delta_mib": (free0 - free1) / 2**20,
        "memory_note": "peak_mib: the torch allocator's peak during the calls (counted from after the inputs "
                       "were made) minus what was allocated before the inputs; device_used_delta_mib: the "
                       "device's used memory after the calls minus before them (cudaMemGetInfo); floor = Q, K, "
                       "V, O bf16 + LSE fp32 (a materialised S would be 2 TiB)"}
    out["_windows"]["long"] = (tl0, tl1)
    del q, k, v, o, lse
    torch.cuda.empty_cache()

    del flush_buf
    torch.cuda.empty_cache()
    return out


def attention_bytes(rows, d, backward):
    """Algorithmic HBM bytes of one call over ``rows`` (b, h, position) rows with
    Nq = Nk: the forward reads Q, K, V and writes O (bf16) and the LSE (fp32); the
    backward reads Q, K, V, O, dO, writes dQ, dK, dV and reads the LSE and writes
    and reads D (fp32)."""
    return rows * (d * 2 * (8 if backward else 4) + 4 * (3 if backward else 1))


def roofline_of(tflops, ms, nbytes, pk):
    """(bound, fraction): the measured time against the larger of the tensor-peak
    time of the call's FLOPs and the HBM time of its algorithmic bytes."""
    t_tensor = tflops * ms / pk["bf16"]
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9) * 1e3
    return ("tensor" if t_tensor >= t_hbm else "hbm"), max(t_tensor, t_hbm) / ms


def add_roofline(e, rows, d, pk, keys=("fwd", "bwd", "bwd_fused")):
    for k in keys:
        if k + "_ms" in e:
            e[k + "_bound"], e[k + "_roofline_frac"] = roofline_of(
                e[k + "_tflops"], e[k + "_ms"], attention_bytes(rows, d, k != "fwd"), pk)


def finish_sweep(sw, pk, sampler):
    """Fractions of the measured peaks and the SM clocks sampled in each window.
    ``*_frac`` divides by the tensor peak; ``*_roofline_frac`` divides by the
    roofline of the call (tensor or HBM, whichever takes longer, named in ``*_bound``)."""
    for e in sw["fwd_bwd_causal_B1_H32_d128"]:
        e["fwd_frac"] = e["fwd_tflops"] / pk["bf16"]
        e["bwd_frac"] = e["bwd_tflops"] / pk["bf16"]
        e["bwd_fused_frac"] = e["bwd_fused_tflops"] / pk["bf16"]
        add_roofline(e, H * e["N"], D, pk)
    for e in sw["fwd_B2_H32_N4096_d128"]:
        e["fwd_frac"] = e["fwd_tflops"] / pk["bf16"]
        add_roofline(e, 2 * H * 4096, D, pk)
    for key, rows in (("window_B1_H32_N8192_d128_W256", H * 8192),
                      ("varlen_causal_B4_H32_N8192_d128", H * sum(sw["varlen_causal_B4_H32_N8192_d128"]["lens"]))):
        e = sw[key]
        e["fwd_frac"] = e["fwd_tflops"] / pk["bf16"]
        e["bwd_frac"] = e["bwd_tflops"] / pk["bf16"]
        add_roofline(e, rows, D, pk)
    lo = sw["fwd_long_causal_B1_H32_N131072_d128"]
    lo["fwd_frac"] = lo["fwd_tflops"] / pk["bf16"]
    add_roofline(lo, H * 131072, D, pk)
    for e in sw["decode_B32_H32"] + sw["decode_paged_B32_Hq32"]:
        e["frac_of_hbm"] = e["gbs"] / pk["hbm_gbs"]
    win = sw.pop("_windows")
    sw["peak_source"] = ("%s: bf16_tflops %.1f (burst) for TFLOP/s, hbm_gbs %.1f for GB/s"
                         % (pk["source"], pk["bf16"], pk["hbm_gbs"]))
    sw["clocks"] = {name: {k: v for k, v in sampler.summary(*w).items() if k != "samples"}
                    for name, w in win.items()}
    lo["clock_note"] = ("frac is of the burst peak; at the clock sampled in this entry's window "
                        "(sweep.clocks.long) the seconds-long sustained figure %.1f may be the fairer "
                        "denominator" % pk["bf16_sustained"])


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    import exact_tiled_attention_21_gb300 as fa

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    fa.load()
    stream = torch.cuda.current_stream(dev)

    g = torch.Generator(device=dev).manual_seed(1234 + rank)
    rnd = lambda *shape: torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    q, k, v, dO = (rnd(B, H, N, D) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    dq_, kc, vc = rnd(DEC_B, DEC_H, D), rnd(DEC_B, DEC_H, DEC_NK, D), rnd(DEC_B, DEC_H, DEC_NK, D)
    od = torch.empty_like(dq_)
    lsed = torch.empty(DEC_B, DEC_H, device=dev, dtype=torch.float32)
    dws = torch.empty(fa.fa_decode_workspace_bytes(DEC_B, DEC_H, DEC_NK, D, DEC_SPLITS),
                      dtype=torch.uint8, device=dev)
    bws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, N, D), dtype=torch.uint8, device=dev)
    LAUNCHES_PER_STEP = 6  # fwd 1, bwd 3, decode 2

    def step(ev=None):
        # the public calls a user makes: fa_fwd, fa_bwd (its three kernels, the dQ pass
        # overlapping the end of the dK/dV pass), fa_decode
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        fa.fa_fwd(q, k, v, o, lse, B, H, N, N, D, SCALE, True, stream)
        rec(1)
        fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, D, SCALE, True, bws, bws.numel(), stream)
        rec(2)
        fa.fa_decode(dq_, kc, vc, od, lsed, DEC_B, DEC_H, DEC_NK, D, SCALE, DEC_SPLITS, dws,
                     dws.numel(), stream)
        rec(3)

    def bwd_steps(ev=None):
        # the backward's three kernels through the step entry points, one by one between
        # events: their individual durations (same inputs; each waits for the one before)
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        fa.fa_bwd_preprocess(o, dO, delta, B, H, N, D, stream)
        rec(1)
        fa.fa_bwd_dkdv(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, D, SCALE, True, stream)
        rec(2)
        fa.fa_bwd_dq(q, k, v, lse, delta, dO, dq, B, H, N, N, D, SCALE, True, stream)
        rec(3)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
        bwd_steps()
    barrier()
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error during warm-up: %s" % detail)

    K_ALT = max(3, min(args.steps, 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    bevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    barrier()
    w0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    for i in range(args.steps):
        bwd_steps(bevs[i])
    barrier()
    # the single-pass backward (fa_bwd_fused) and the CTA-pair dK/dV pass, K calls each
    wsf = torch.empty(fa.fa_bwd_fused_workspace_bytes(B, H, N, N, D), dtype=torch.uint8, device=dev)
    fev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(3):
        fa.fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, D, SCALE, True, wsf, wsf.numel(), stream)
        fa.fa_bwd_dkdv_pair(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, D, SCALE, True, stream)
    barrier()
    fev[0].record(stream)
    for _ in range(K_ALT):
        fa.fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, D, SCALE, True, wsf, wsf.numel(), stream)
    fev[1].record(stream)
    fev[2].record(stream)
    for _ in range(K_ALT):
        fa.fa_bwd_dkdv_pair(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, D, SCALE, True, stream)
    fev[3].record(stream)
    barrier()
    bwd_fused_ms = fev[0].elapsed_time(fev[1]) / K_ALT
    dkdv_pair_ms = fev[2].elapsed_time(fev[3]) / K_ALT
    del wsf
    w1 = time.time()  # the clock record covers both passes
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the timed region: %s" % detail)

    total_ms = t_start.elapsed_time(t_end)
    comp = [0.0] * 3
    for e in evs:
        for j in range(3):
            comp[j] += e[j].elapsed_time(e[j + 1])
    bcomp = [0.0] * 3
    for e in bevs:
        for j in range(3):
            bcomp[j] += e[j].elapsed_time(e[j + 1])
    K = args.steps
    fwd_ms, bwd_ms, dec_ms = (c / K for c in comp)
    pre_ms, dkdv_ms, dq_ms = (c / K for c in bcomp)
    fb_ms = fwd_ms + bwd_ms

    maxall = lambda x: reduce_max(x, dist, dev)
    total_ms = maxall(total_ms)
    dec_ms_max = maxall(dec_ms)
    value = replica_throughput(FWD_FLOPS + BWD_FLOPS, fb_ms * 1e-3, world, dist, dev) / 1e12

    # ---- end to end through the public API, host buffers, copies inside the timed region
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    hq, hk, hv, hdO = (pin(t) for t in (q, k, v, dO))
    for h_, d_ in ((hq, q), (hk, k), (hv, v), (hdO, dO)):
        h_.copy_(d_)
    hqd = pin(dq_)
    hqd.copy_(dq_)
    ho, hl, hdq, hdk, hdv = pin(o), pin(lse), pin(dq), pin(dk), pin(dv)
    hod, hld = pin(od), pin(lsed)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdO))          # fwd + bwd step
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl, hdq, hdk, hdv))
    h2d_dec = hqd.numel() * hqd.element_size()                                     # decode step
    d2h_dec = sum(t.numel() * t.element_size() for t in (hod, hld))
    # the end-to-end runs take their own step count: the pipelined run's first copy-in and last
    # copy-out overlap no compute, which over 20 steps read 1026 TFLOP/s and over 60 1061
    e2e_steps = 60

    def e2e_step(ev):
        ev[0].record(stream)
        for d_, h_ in ((q, hq), (k, hk), (v, hv), (dO, hdO)):
            d_.copy_(h_, non_blocking=True)
        fa.fa_fwd(q, k, v, o, lse, B, H, N, N, D, SCALE, True, stream)
        fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, D, SCALE, True, bws, bws.numel(), stream)
        for h_, d_ in ((ho, o), (hl, lse), (hdq, dq), (hdk, dk), (hdv, dv)):
            h_.copy_(d_, non_blocking=True)
        ev[1].record(stream)
        dq_.copy_(hqd, non_blocking=True)
        fa.fa_decode(dq_, kc, vc, od, lsed, DEC_B, DEC_H, DEC_NK, D, SCALE, DEC_SPLITS, dws,
                     dws.numel(), stream)
        hod.copy_(od, non_blocking=True)
        hld.copy_(lsed, non_blocking=True)
        ev[2].record(stream)

    for _ in range(2):
        e2e_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    barrier()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        e2e_step(eev[i])
    barrier()
    e2e_fb_serial = maxall(sum(e[0].elapsed_time(e[1]) for e in eev) / e2e_steps)
    e2e_dec = maxall(sum(e[1].elapsed_time(e[2]) for e in eev) / e2e_steps)
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the end-to-end run: %s" % detail)

    # The same fwd + bwd step from host buffers, pipelined the way a training loop
    # feeds a GPU: step i+1's inputs copy in (stream s_in) and step i-1's results copy
    # out (s_out) while step i computes; three sets of device tensors rotate, so a
    # copy-in never waits for the copy-out of the set before it and the two
    # directions of the host link run at the same time.  Every step still moves its
    # own inputs in and its own results out inside the timed region; the time is
    # first copy-in to last copy-out over all steps.
    NSETS = 3
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sets = [(q, k, v, dO, o, lse, dq, dk, dv)] + [
        tuple(torch.empty_like(t) for t in (q, k, v, dO, o, lse, dq, dk, dv)) for _ in range(NSETS - 1)]
    bws_sets = [bws] + [torch.empty_like(bws) for _ in range(NSETS - 1)]

    def pipelined(nsteps, t0, t1):
        free = [None] * NSETS
        ready = [torch.cuda.Event() for _ in range(NSETS)]
        done = [torch.cuda.Event() for _ in range(NSETS)]
        t0.record(stream)
        s_in.wait_event(t0)
        for i in range(nsteps):
            b = i % NSETS
            q_, k_, v_, dO_, o_, lse_, dq2, dk2, dv2 = sets[b]
            if free[b] is not None:
                s_in.wait_event(free[b])
            with torch.cuda.stream(s_in):
                for d_, h_ in ((q_, hq), (k_, hk), (v_, hv), (dO_, hdO)):
                    d_.copy_(h_, non_blocking=True)
            ready[b].record(s_in)
            stream.wait_event(ready[b])
            ws_ = bws_sets[b]
            fa.fa_fwd(q_, k_, v_, o_, lse_, B, H, N, N, D, SCALE, True, stream)
            fa.fa_bwd(q_, k_, v_, o_, lse_, dO_, dq2, dk2, dv2, B, H, N, N, D, SCALE, True, ws_, ws_.numel(),
                      stream)
            done[b].record(stream)
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                for h_, d_ in ((ho, o_), (hl, lse_), (hdq, dq2), (hdk, dk2), (hdv, dv2)):
                    h_.copy_(d_, non_blocking=True)
            free[b] = torch.cuda.Event()
            free[b].record(s_out)
        t1.record(s_out)

    pipelined(3, torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    torch.cuda.synchronize(dev)
    barrier()
    pt0, pt1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipelined(e2e_steps, pt0, pt1)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_fb = maxall(pt0.elapsed_time(pt1) / e2e_steps)
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the pipelined end-to-end run: %s" % detail)

    # ---- paged grouped-query decode (next-row feature; timed separately, not part of the step)
    PG_HKV, PG_PAGE = 8, 16
    npages = DEC_B * (DEC_NK // PG_PAGE)
    kpg = rnd(npages, PG_HKV, PG_PAGE, D)
    vpg = rnd(npages, PG_HKV, PG_PAGE, D)
    perm = torch.randperm(npages, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    table = perm.reshape(DEC_B, DEC_NK // PG_PAGE).to(dev)
    lens = torch.full((DEC_B,), DEC_NK, dtype=torch.int32, device=dev)
    pws = torch.empty(fa.fa_decode_paged_workspace_bytes(DEC_B, DEC_H, D, 0), dtype=torch.uint8, device=dev)
    pg_call = lambda: fa.fa_decode_paged(dq_, kpg, vpg, table, lens, od, lsed, DEC_B, DEC_H, PG_HKV, PG_PAGE,
                                         DEC_NK // PG_PAGE, npages, D, SCALE, 0, pws, pws.numel(), stream)
    for _ in range(3):
        pg_call()
    barrier()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record(stream)
    for _ in range(20):
        pg_call()
    pe1.record(stream)
    barrier()
    pg_ms = pe0.elapsed_time(pe1) / 20
    pg_bytes = 2.0 * DEC_B * PG_HKV * DEC_NK * D * 2
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the paged decode run: %s" % detail)

    # ---- FP8 block-scaled forward (next-row feature; timed separately, not part of the step)
    def e4m3_bytes(*shape):  # finite e4m3 bytes of either sign (no NaN pattern)
        mag = torch.randint(0, 126, shape, generator=torch.Generator().manual_seed(7), dtype=torch.int32)
        sign = torch.randint(0, 2, shape, generator=torch.Generator().manual_seed(8), dtype=torch.int32) << 7
        return (mag | sign).to(torch.uint8).to(dev)
    f8q, f8k, f8v = (e4m3_bytes(1, H, N, D) for _ in range(3))
    f8sq = torch.full((H, N // 128), 1.0 / 64, device=dev)
    f8sk = f8sq.clone()
    f8sv = torch.full((H,), 1.0 / 64, device=dev)
    f8o = torch.empty(1, H, N, D, dtype=torch.bfloat16, device=dev)
    f8l = torch.empty(1, H, N, device=dev)
    f8ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(1, H, N, D), dtype=torch.uint8, device=dev)
    f8_call = lambda: fa.fa_fwd_fp8(f8q, f8k, f8v, f8sq, f8sk, f8sv, f8o, f8l, 1, H, N, N, D, SCALE, 1, f8ws,
                                    f8ws.numel(), stream)
    for _ in range(3):
        f8_call()
    barrier()
    fe0, fe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fe0.record(stream)
    for _ in range(20):
        f8_call()
    fe1.record(stream)
    barrier()
    f8_ms = fe0.elapsed_time(fe1) / 20
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the FP8 forward run: %s" % detail)

    # ---- the sweep over the other workloads (outside the timed step; each its own median)
    sw0 = time.time()
    sweep = run_sweep(fa, dev, stream, g, barrier, sampler) if not args.no_sweep else None
    sw1 = time.time()
    st, detail = fa.fa_get_last_device_error(stream)
    if st != 0:
        raise RuntimeError("device error in the sweep: %s" % detail)

    sampler.stop()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    pk = peaks()
    dkdv_tflops = DKDV_FLOPS / (dkdv_ms * 1e-3) / 1e12
    clocks = sampler.summary(w0, w1)
    if sweep is not None:
        finish_sweep(sweep, pk, sampler)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": CONFIG,
        "components": {
            "fwd_ms": fwd_ms, "fwd_tflops": FWD_FLOPS / (fwd_ms * 1e-3) / 1e12,
            "bwd_ms": bwd_ms,
            "bwd_tflops": BWD_FLOPS / (bwd_ms * 1e-3) / 1e12,
            "bwd_pre_ms": pre_ms, "bwd_dkdv_ms": dkdv_ms, "bwd_dq_ms": dq_ms,
            "bwd_kernels_note": "pre/dkdv/dq: the step entry points timed one by one after the timed region "
                                "(fa_bwd overlaps the dQ pass with the end of the dK/dV pass)",
            "bwd_fused_ms": bwd_fused_ms, "bwd_fused_tflops": BWD_FLOPS / (bwd_fused_ms * 1e-3) / 1e12,
            "bwd_fused_note": "fa_bwd_fused: the same backward in one pass over the key tiles (dQ^T = K^T dS^T on "
                              "the tensor cores, bulk fp32 reduce-adds; dQ bits vary run to run), %d back-to-back "
                              "calls" % K_ALT,
            "bwd_dkdv_pair_ms": dkdv_pair_ms,
            "bwd_dkdv_pair_note": "fa_bwd_dkdv_pair: the dK/dV pass on CTA pairs (cta_group::2), %d back-to-back "
                                  "calls; compare bwd_dkdv_ms" % K_ALT,
            "fwd_frac_of_peak": FWD_FLOPS / (fwd_ms * 1e-3) / 1e12 / pk["bf16"],
            "bwd_frac_of_peak": BWD_FLOPS / (bwd_ms * 1e-3) / 1e12 / pk["bf16"],
            "peak_source": "%s bf16_tflops (burst)" % pk["source"],
        },
        "decode": {"value": world * DEC_BYTES / (dec_ms_max * 1e-3) / 1e9, "unit": "GB/s",
                   "ms": dec_ms, "frac_of_hbm": DEC_BYTES / (dec_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "decode_paged": {"value": pg_bytes / (pg_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": pg_ms,
                         "config": "B=32 Hq=32 Hkv=8 page=16 Nk=4096 d=128, the library's automatic split count "
                                   "(grouped-query, paged)",
                         "frac_of_hbm": pg_bytes / (pg_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "fwd_fp8": {"value": FWD_FLOPS / (f8_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": f8_ms,
                    "config": "B=1 H=32 N=8192 d=128 causal, e4m3 q/k (one scale per 128 rows) and v (one per "
                              "head), including the V transpose into the workspace",
                    "frac_of_peak": FWD_FLOPS / (f8_ms * 1e-3) / 1e12 / (2 * pk["bf16"]),
                    "peak_source": "%s bf16_tflops (burst) x 2, the nominal dense fp8 / bf16 ratio "
                                   "(4.5 / 2.25 PFLOP/s); no fp8 peak is measured" % pk["source"]},
        "roofline": {
            "kernel": "bwd_dkdv_kernel<128>",
            "bound": "tensor",
            "achieved": dkdv_tflops,
            "peak": pk["bf16"],
            "peak_source": "%s bf16_tflops (burst): the kernel is timed in regions of tens of ms at the "
                           "sampled SM clock under \"clocks\"; the sustained %.1f was taken over seconds "
                           "at power-capped clocks" % (pk["source"], pk["bf16_sustained"]),
            "unit": "TFLOP/s",
            "frac": dkdv_tflops / pk["bf16"],
            "traffic": profiled_traffic("bwd_dkdv_kernel_causal_B1H32N8192.md", "fa_bwd.cu"),
            "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch; algorithmic "
                            "bytes are 4 x 64 MiB read (Q, K, V, dO) + 2 x 64 MiB written (dK, dV)",
            "algorithmic_per_launch": "4 of the 5 backward products: 4 * B*H*N*N*d FLOP (causal half of 8 B H N^2 d)",
            "duration_source": "fa_bwd_dkdv between CUDA events on the launching stream, K launches after the "
                               "fa_fwd/fa_bwd timed steps (inside fa_bwd its end overlaps the dQ pass)",
        },
        "e2e": {"value": world * (FWD_FLOPS + BWD_FLOPS) / (e2e_fb * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelined": "copies of neighbouring steps overlap this step's compute (separate copy-in and "
                             "copy-out streams, three rotating sets of device tensors)",
                "serial_value": world * (FWD_FLOPS + BWD_FLOPS) / (e2e_fb_serial * 1e-3) / 1e12,
                "decode_gbs": world * DEC_BYTES / (e2e_dec * 1e-3) / 1e9,
                "decode_h2d_bytes": h2d_dec, "decode_d2h_bytes": d2h_dec,
                "api": "fa_fwd + fa_bwd (and, serial, fa_decode) from pinned host buffers; KV cache resident"},
        "sweep": sweep,
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        f, t, r = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": "numpy fp64 naive fwd+bwd of %d query rows (256-row blocks of heads (0,0), "
                      "(0,1), ...), N=8192 causal, %.1f s" % (r, t)}
        f2, t2, r2, th2 = oracle_sample_o2(args.cpu_seconds / 3)
        line["cpu_baseline"]["o2_fwd"] = {
            "value": f2 / t2 / 1e12, "unit": "TFLOP/s", "cores": th2, "kind": "oracle (C two-pass, forward)",
            "sample": "forward of %d query rows (256-row blocks), N=8192 causal, %.1f s" % (r2, t2)}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ one kernel for a profiler
PROFILE_TARGETS = ("fwd", "dkdv", "dq", "fused", "pair", "window", "decode", "decode64", "paged", "paged48",
                   "paged20", "fp8")


def run_profile(target, launches):
    """Runs one kernel of the bench workload ``launches`` times (after one warm-up
    call) with only its own inputs on the device, for an ncu capture:
    fwd / dkdv / dq / fused / pair at B=1, H=32, N=8192, d=128 causal; window the
    forward under a causal 256-key window at the same size; decode at
    B=32, H=32, Nk=4096 (d=128 or d=64); paged at B=32, Hq=32, Hkv=8, page 16 (the
    tensor-core kernel), paged48 with 48-token pages, 85 per sequence (4080 tokens:
    the tensor-core kernel in 16-row boxes) and paged20 with 20-token pages, 204 per
    sequence (4080 tokens: the general kernel); fp8 the FP8 forward.  Prints one
    line; no timing."""
    import torch
    import exact_tiled_attention_21_gb300 as fa
    dev = torch.device("cuda", 0)
    fa.load()
    s = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev).manual_seed(99)
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    if target in ("fwd", "dkdv", "dq", "fused", "pair", "window"):
        q, k, v, dO = (rnd(B, H, N, D) for _ in range(4))
        o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
        lse = torch.empty(B, H, N, device=dev)
        delta = torch.empty(B, H, N, device=dev)
        fa.fa_fwd(q, k, v, o, lse, B, H, N, N, D, SCALE, True, s)
        fa.fa_bwd_preprocess(o, dO, delta, B, H, N, D, s)
        wsf = torch.empty(fa.fa_bwd_fused_workspace_bytes(B, H, N, N, D), dtype=torch.uint8, device=dev)
        call = {
            "fwd": lambda: fa.fa_fwd(q, k, v, o, lse, B, H, N, N, D, SCALE, True, s),
            "window": lambda: fa.fa_fwd_window(q, k, v, o, lse, B, H, N, N, D, SCALE, 256, s),
            "dkdv": lambda: fa.fa_bwd_dkdv(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, D, SCALE, True, s),
            "dq": lambda: fa.fa_bwd_dq(q, k, v, lse, delta, dO, dq, B, H, N, N, D, SCALE, True, s),
            "fused": lambda: fa.fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, D, SCALE, True, wsf,
                                             wsf.numel(), s),
            "pair": lambda: fa.fa_bwd_dkdv_pair(q, k, v, lse, delta, dO, dk, dv, B, H, N, N, D, SCALE, True, s),
        }[target]
    elif target in ("decode", "decode64"):
        d = 128 if target == "decode" else 64
        qd, kc, vc = rnd(DEC_B, DEC_H, d), rnd(DEC_B, DEC_H, DEC_NK, d), rnd(DEC_B, DEC_H, DEC_NK, d)
        od = torch.empty_like(qd)
        lsed = torch.empty(DEC_B, DEC_H, device=dev)
        ws = torch.empty(fa.fa_decode_workspace_bytes(DEC_B, DEC_H, DEC_NK, d, DEC_SPLITS), dtype=torch.uint8,
                         device=dev)
        call = lambda: fa.fa_decode(qd, kc, vc, od, lsed, DEC_B, DEC_H, DEC_NK, d, 1 / math.sqrt(d), DEC_SPLITS, ws,
                                    ws.numel(), s)
    elif target in ("paged", "paged48", "paged20"):
        hkv, page = 8, {"paged": 16, "paged48": 48, "paged20": 20}[target]
        npages = DEC_B * (DEC_NK // page)
        kp, vp = rnd(npages, hkv, page, D), rnd(npages, hkv, page, D)
        qd = rnd(DEC_B, DEC_H, D)
        table = torch.randperm(npages, generator=torch.Generator().manual_seed(5)).to(torch.int32)
        table = table.reshape(DEC_B, DEC_NK // page).to(dev)
        lens = torch.full((DEC_B,), (DEC_NK // page) * page, dtype=torch.int32, device=dev)
        od = torch.empty_like(qd)
        lsed = torch.empty(DEC_B, DEC_H, device=dev)
        ws = torch.empty(fa.fa_decode_paged_workspace_bytes(DEC_B, DEC_H, D, 0), dtype=torch.uint8, device=dev)
        call = lambda: fa.fa_decode_paged(qd, kp, vp, table, lens, od, lsed, DEC_B, DEC_H, hkv, page, DEC_NK // page,
                                          npages, D, SCALE, 0, ws, ws.numel(), s)
    else:  # fp8
        mk = lambda: torch.randint(0, 126, (1, H, N, D), generator=torch.Generator().manual_seed(7),
                                   dtype=torch.int32).to(torch.uint8).to(dev)
        q8, k8, v8 = mk(), mk(), mk()
        sq = torch.full((H, N // 128), 1.0 / 64, device=dev)
        sv = torch.full((H,), 1.0 / 64, device=dev)
        o = torch.empty(1, H, N, D, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(1, H, N, device=dev)
        ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(1, H, N, D), dtype=torch.uint8, device=dev)
        call = lambda: fa.fa_fwd_fp8(q8, k8, v8, sq, sq, sv, o, lse, 1, H, N, N, D, SCALE, 1, ws, ws.numel(), s)
    for _ in range(1 + launches):
        call()
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_last_device_error(s)
    print(json.dumps({"profile": target, "launches": 1 + launches, "device_error": st}), flush=True)
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-workload sweep (not timed in the step)")
    ap.add_argument("--profile", choices=PROFILE_TARGETS, default=None,
                    help="run one kernel of the workload a few times with only its own inputs (for ncu); no timing")
    ap.add_argument("--launches", type=int, default=2, help="with --profile: launches after one warm-up call")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.profile:
        return run_profile(args.profile, args.launches)
    if args.impl == "reference":
        return run_reference(args, rank)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
