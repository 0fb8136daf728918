"""Benchmark of the KVarN codec hot path on GB300 (libkvarn).

One step = the whole hot path once:
  * encode of one batch of completed blocks: 64 sequences x 8 kv heads x one 128-token block of
    bf16 K and V (a Qwen3-4B layer), 2-bit preset (kvarn_k2v2_g128), and
  * one decode-attention step over a 2-bit packed cache: batch 16, 32 query / 8 kv heads,
    head_dim 128, 32768 tokens per sequence, one bf16 query per head.
Inputs are seeded synthetic tensors already resident in HBM; the 302 MB packed cache is larger
than L2 and L2 is also flushed (a read-modify-write of 256 MiB) before every timed step.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle instead, on a
bounded sample of the same workload, scaled to the same unit.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-encode GB/s + 2-bit decode-attn us/step at 32k ctx; % of HBM peak"
ENC_SEQ, ENC_HKV = 64, 8
DEC_B, DEC_HQ, DEC_HKV, DEC_L = 16, 32, 8, 32768
WORKLOAD = ("encode 64 seq x 8 kv heads x 128-token block (K and V, bf16, 2-bit) + decode attention "
            "B=16, 32q/8kv heads, d=128, 32768-token 2-bit packed cache")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def enc_bytes(n_tiles_per_kind, k_bits=2, v_bits=2):
    inp = 2 * n_tiles_per_kind * 128 * 128 * 2
    out = n_tiles_per_kind * ((128 * 16 * k_bits + 512 + 4) + (128 * 16 * v_bits + 512 + 4))
    return inp, out


# Encode arithmetic per element, counted as the FP32 lane operations the encoder issues (a packed
# FFMA2/FADD2/FMUL2 on two elements is one lane operation for each): rotation 8 (4 butterfly stages
# in each of the two passes, the last including the 1/sqrt(128) scale); per normalisation iteration
# 6 (token and channel step: p = Y a, sum p, sum p^2) plus ~0.6 for their in-thread and cross-lane
# sums, 8 iterations = 53; W = Y / s2 1; quantisation 3 (W / g - Z, the saturating multiply, the
# rounding FFMA).  Min/max, conversions and packing are ALU-pipe work and are not counted.
ENC_FP32_LANE_OPS_PER_ELEMENT = 65
# FP32 lane-operation peak from unit counts and clock: 152 SMs x 128 lanes x 2.07 GHz = 40.3 T/s (a
# measured FFMA2 loop sustained 38.3 T/s at ~1990 MHz on this GPU).
FP32_LANE_PEAK_T = 152 * 128 * 2.07e9 / 1e12


def dec_bytes(k_bits=2, v_bits=2):
    tiles = DEC_B * DEC_HKV * (DEC_L // 128)
    cache = tiles * ((128 * 16 * k_bits + 512 + 4) + (128 * 16 * v_bits + 512 + 4))
    q = DEC_B * DEC_HQ * 128 * 2
    out = DEC_B * DEC_HQ * 128 * 4
    return cache, q, out


def ragged_dec_bytes(lens, Hq, Hkv, k_bits, v_bits):
    """Algorithmic bytes of one decode call over sequences of lengths `lens`: each (sequence, kv
    head) reads its L // 128 packed K and V tiles (codes, 512 B of parameters and a 4-byte factor
    each) and its L % 128 bf16 tail tokens of K and V; plus the bf16 queries and fp32 outputs."""
    tile = (128 * 16 * k_bits + 516) + (128 * 16 * v_bits + 516)
    cache = sum(Hkv * ((L // 128) * tile + (L % 128) * 128 * 2 * 2) for L in lens)
    return cache, len(lens) * Hq * 128 * 2, len(lens) * Hq * 128 * 4


# the sources each kernel's DRAM counters depend on (its own file and the headers it includes;
# include/kvarn.h is added to every set)
KERNEL_SOURCES = {
    "kvarn_decode_attention": ("decode_attn.cu", "kvarn_common.cuh", "tcgen05.cuh", "kvarn_internal.h"),
    "kvarn_encode_kv_blocks": ("encode.cu", "kvarn_common.cuh", "kvarn_internal.h"),
}


def source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_kv_cache_kvarn_gb300", "csrc")
    paths = [os.path.join(csrc, n) for n in KERNEL_SOURCES[kernel]] + [os.path.join(ROOT, "include", "kvarn.h")]
    for path in paths:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvarn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t0, t1):
        """Samples taken between host times t0 and t1 (the timed region, widened by one polling
        interval); if the region is shorter than the interval, the sample nearest to it."""
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        if not inside and rows:
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": inside[-1][2] if inside else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# reference arm / cpu baseline: the fp64 oracle on all host cores, whole steps
# ------------------------------------------------------------------------------------------------
# One oracle step is the GPU step's workload done by the oracle: 512 K + 512 V tile encodes (the
# config-1 batch, seed 1) and 16 x 8 (sequence, kv head) decode units of 32768 tokens x 4 query
# heads.  The work is spread over a process pool with one single-threaded worker per host core
# (spawn context: no fork after CUDA is initialised).  The decode units read a packed cache whose
# 256 block-table entries cycle through 16 oracle-encoded blocks of the config-2 data (seed 2):
# the oracle's cost per tile does not depend on the tile's values, and encoding all 65,536 tiles
# of that cache would take longer than every timed step together.
_REF = {}
ORACLE_CACHE_BLOCKS = 16
ORACLE_ENC_CHUNK = 16


def _ref_worker_init():
    import torch

    torch.set_num_threads(1)
    from bit_kv_cache_kvarn_gb300 import synthetic
    from oracle import kvarn_oracle as o

    n = ENC_SEQ * ENC_HKV
    k, v = synthetic.outlier_kv(1, n, 128)
    _REF["xk"] = k.reshape(n, 128, 128).float().double().numpy()
    _REF["xv"] = v.reshape(n, 128, 128).float().double().numpy()
    kk, vv = synthetic.outlier_kv(2, 1, ORACLE_CACHE_BLOCKS * 128)
    kc, kp, ks, _ = o.encode_blocks(kk.reshape(-1, 128, 128).float().double().numpy(), "K", 2)
    vc, vp, vs, _ = o.encode_blocks(vv.reshape(-1, 128, 128).float().double().numpy(), "V", 2)
    _REF["cache"] = (kc, kp, ks, vc, vp, vs)
    _REF["q"] = synthetic.queries(2, DEC_B, DEC_HQ).float().double().numpy()


def _ref_task(task):
    """One piece of an oracle step; returns (its kind, its CPU seconds)."""
    import numpy as np

    from oracle import kvarn_oracle as o

    t0 = time.process_time()
    kind, a, b = task
    if kind == "enc":
        o.encode_blocks(_REF["xk"][a:b], "K", 2)
        o.encode_blocks(_REF["xv"][a:b], "V", 2)
    else:  # decode unit: sequence a, kv head b
        nt = DEC_L // 128
        group = DEC_HQ // DEC_HKV
        table = (np.arange(nt) % ORACLE_CACHE_BLOCKS).reshape(1, 1, nt)
        tails = np.zeros((1, 1, 128, 128))
        q = _REF["q"][a:a + 1, b * group:(b + 1) * group]
        o.decode_attention(q, group, 1, *_REF["cache"], table, [DEC_L], tails, tails, 1 / math.sqrt(128), 2, 2)
    return kind, time.process_time() - t0


def pool_cores(requested=None):
    """Worker count of the oracle pool: every host core this process may run on, or the requested
    number clamped to 1..that."""
    avail = len(os.sched_getaffinity(0))
    return avail if not requested else max(1, min(int(requested), avail))


class OraclePool:
    """The fp64 oracle over every host core; step() runs one whole oracle step."""

    def __init__(self, cores=None):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor

        self.cores = pool_cores(cores)
        # one thread per worker: the cores are the parallelism (children inherit the environment)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.ex = ProcessPoolExecutor(max_workers=self.cores, mp_context=mp.get_context("spawn"),
                                          initializer=_ref_worker_init)
            list(self.ex.map(_noop, range(self.cores)))  # start and initialise every worker
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        n = ENC_SEQ * ENC_HKV
        self.tasks = [("dec", b, h) for b in range(DEC_B) for h in range(DEC_HKV)]
        self.tasks += [("enc", a, min(n, a + ORACLE_ENC_CHUNK)) for a in range(0, n, ORACLE_ENC_CHUNK)]

    def step(self):
        """(wall seconds, summed CPU seconds of the workers) of one whole step; the CPU seconds of
        the encodes and of the decode units are kept apart in self.last_split."""
        t0 = time.perf_counter()
        parts = list(self.ex.map(_ref_task, self.tasks))
        wall = time.perf_counter() - t0
        self.last_split = {k: sum(c for kk, c in parts if kk == k) for k in ("enc", "dec")}
        return wall, sum(c for _, c in parts)

    def close(self):
        self.ex.shutdown()

    def describe(self):
        return (f"whole oracle steps: {ENC_SEQ * ENC_HKV} K + {ENC_SEQ * ENC_HKV} V tile encodes and "
                f"{DEC_B * DEC_HKV} (sequence, kv head) decode units of {DEC_L} tokens x "
                f"{DEC_HQ // DEC_HKV} query heads each, on a pool of {self.cores} single-threaded worker "
                f"processes (one per host core used); the decode cache's block tables cycle through "
                f"{ORACLE_CACHE_BLOCKS} oracle-encoded blocks")


def _noop(_):
    return 0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pool = OraclePool(args.ref_cores)
    try:
        # whole steps: W warm-up and K timed, unless the K steps would take more than about two
        # minutes (then as many as fit, reported in `steps`, so the run ends within a few minutes)
        warm = [pool.step() for _ in range(args.warmup)]
        per = warm[-1][0]
        n_timed = max(1, min(args.steps, int(120.0 / max(per, 1e-3))))
        timed, splits = [], []
        for _ in range(n_timed):
            timed.append(pool.step())
            splits.append(pool.last_split)
    finally:
        pool.close()
    v = statistics.mean(w for w, _ in timed) * 1e6
    cpu = statistics.mean(c for _, c in timed)
    sample = pool.describe() + f"; {n_timed} timed steps after {args.warmup} warm-up"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": args.gpus, "steps": n_timed, "warmup": args.warmup,
        "ms_per_step": round(v / 1000, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "CPU run"},
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": pool.cores, "kind": "oracle",
                         "sample": sample, "cpu_seconds_per_step": round(cpu, 2),
                         # single-threaded workers: the CPU seconds of each part are its one-core time
                         "cpu_seconds_encode_config1": round(statistics.mean(x["enc"] for x in splits), 2),
                         "cpu_seconds_decode_config2": round(statistics.mean(x["dec"] for x in splits), 2)},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_line(n_warm=1, n_timed=2):
    """The oracle as it stands, timed on the host's cores on whole steps of the bench workload."""
    pool = OraclePool()
    try:
        for _ in range(n_warm):
            pool.step()
        timed = [pool.step() for _ in range(n_timed)]
    finally:
        pool.close()
    return {"value": round(statistics.mean(w for w, _ in timed) * 1e6, 1), "unit": "us/step",
            "cores": pool.cores, "kind": "oracle",
            "sample": pool.describe() + f"; {n_timed} timed steps after {n_warm} warm-up",
            "cpu_seconds_per_step": round(statistics.mean(c for _, c in timed), 2)}


def max_over_ranks(values, world, device):
    """Per-rank timings -> their maximum over the ranks (every rank gets the result)."""
    import torch
    import torch.distributed as tdist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_step_rates(step_ms_max, world):
    """(us per step, replica steps per second of the whole job).  Each of the N replicas runs one
    full step of the workload within the max-over-ranks time, so the per-step time stays that of
    one rank (weak scaling, replicas only) while the job completes N steps in that time."""
    us = step_ms_max * 1000.0
    return us, world / (step_ms_max * 1e-3)


def run_diagnostics():
    """E_M / E_D split and token-scale statistics of each preset on the encode workload."""
    import torch

    import bit_kv_cache_kvarn_gb300 as kv
    from bit_kv_cache_kvarn_gb300 import diagnostics

    kv.load()
    n_enc = ENC_SEQ * ENC_HKV
    k, v = kv.synthetic.outlier_kv(1, n_enc, 128, device="cuda")
    res = diagnostics.run(kv, k.reshape(n_enc, 128, 128), v.reshape(n_enc, 128, 128))
    torch.cuda.synchronize()
    print(json.dumps({"impl": "diagnostics", "workload": WORKLOAD.split(" + ")[0], "tiles_per_kind": n_enc,
                      "presets": res}), flush=True)


def graph_us(fn, reps):
    """Per-call device time of fn (one library call) replayed from a CUDA graph: the host enqueues
    nothing per call, so the number excludes the binding's and the launches' host overhead."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    c.record()
    torch.cuda.synchronize()
    return a.elapsed_time(c) / reps * 1000


def run_latency():
    """Decode latency of single calls at serving-like shapes (32q/8kv heads, 2-bit K and V; lengths
    a multiple of 128, or with a 127-token bf16 tail): back-to-back calls timed with CUDA events,
    cache re-read from L2 where it fits (not flushed), so the numbers show the call's own latency,
    not HBM time."""
    import torch

    import bit_kv_cache_kvarn_gb300 as kv

    kv.load()
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    dev = torch.device("cuda", 0)
    res = {}
    for B, ctx in ((1, 4096), (1, 32768), (4, 8192), (16, 32768), (1, 4096 + 127), (16, 32768 + 127)):
        nt = -(-ctx // 128)  # block-table width; the last ctx % 128 tokens are the bf16 tail
        n = B * DEC_HKV * nt
        pool = min(n, 4096)  # distinct tiles; the block table cycles through them
        g = torch.Generator(device="cpu").manual_seed(11)
        x = torch.randn(pool, 128, 128, generator=g).to(torch.bfloat16).to(dev)
        pk = (torch.empty(pool, 4096, dtype=torch.uint8, device=dev),
              torch.empty(pool, 512, dtype=torch.uint8, device=dev), torch.empty(pool, device=dev))
        pv = tuple(torch.empty_like(t) for t in pk)
        kv.kvarn_encode_kv_blocks(cfg, x, x, *pk, *pv)
        table = (torch.arange(n, dtype=torch.int32, device=dev) % pool).reshape(B, DEC_HKV, nt)
        lens = torch.full((B,), ctx, dtype=torch.int32, device=dev)
        tail = (torch.randn(B, DEC_HKV, 128, 128, generator=g) * 0.5).to(torch.bfloat16).to(dev)
        q = torch.randn(B, DEC_HQ, 128, generator=g).to(torch.bfloat16).to(dev)
        ws = torch.empty(kv.kvarn_decode_workspace_size(cfg, B, DEC_HQ, DEC_HKV, nt), dtype=torch.uint8, device=dev)
        out = torch.empty(B, DEC_HQ, 128, device=dev)

        def call():
            kv.kvarn_decode_attention(cfg, q, DEC_HKV, *pk, *pv, table, lens, tail, tail, 1 / math.sqrt(128),
                                      ws, out)

        for _ in range(20):
            call()
        torch.cuda.synchronize()
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 200
        a.record()
        for _ in range(reps):
            call()
        c.record()
        torch.cuda.synchronize()
        res[f"B={B}, ctx={ctx}"] = {"eager_us": round(a.elapsed_time(c) / reps * 1000, 2),
                                    "graph_us": round(graph_us(call, reps), 2)}
    assert kv.kvarn_device_error() == 0
    print(json.dumps({"impl": "latency", "unit": "us per call",
                      "eager": "back-to-back calls from Python (host enqueue cost included when it exceeds the device time)",
                      "graph": "the same call replayed from a CUDA graph (device time)",
                      "heads": f"{DEC_HQ}q/{DEC_HKV}kv", "preset": "kvarn_k2v2_g128", "results": res}), flush=True)


def run_configs():
    """The other workloads, timed as single calls (CUDA events, 256 MiB L2 flush before each):
    the encode of 512 K + 512 V blocks (64 sequences x 8 kv heads, Qwen3-4B shaped, seed 1) under
    both presets, and decode attention over the Phi-4 shaped ragged long-context cache (40q/10kv
    heads, batch 4, lengths U[65536, 131072] from seed 3, 4-bit K / 2-bit V, the last len % 128
    tokens of each sequence in the bf16 tails).  Rates use the algorithmic bytes of each call."""
    import torch

    import bit_kv_cache_kvarn_gb300 as kv

    kv.load()
    dev = torch.device("cuda", 0)
    hbm, src = peaks()
    flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.add_(1.0)
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            c.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(c) * 1000)
        return statistics.mean(ts)

    res = {}
    n_enc = ENC_SEQ * ENC_HKV
    ek, ev = kv.synthetic.outlier_kv(1, n_enc, 128, device=dev)
    ek, ev = ek.reshape(n_enc, 128, 128), ev.reshape(n_enc, 128, 128)
    for preset in ("kvarn_k4v2_g128", "kvarn_k2v2_g128"):
        cfg = kv.kvarn_config_from_preset(preset)
        outs = []
        for bits in (cfg.k_bits, cfg.v_bits):
            outs += [torch.empty(n_enc, 128 * 16 * bits, dtype=torch.uint8, device=dev),
                     torch.empty(n_enc, 512, dtype=torch.uint8, device=dev),
                     torch.empty(n_enc, dtype=torch.float32, device=dev)]
        us = timed(lambda: kv.kvarn_encode_kv_blocks(cfg, ek, ev, *outs), 200)
        e_in, e_out = enc_bytes(n_enc, cfg.k_bits, cfg.v_bits)
        lane_t = 2 * n_enc * 128 * 128 * ENC_FP32_LANE_OPS_PER_ELEMENT / (us * 1e-6) / 1e12
        res[f"encode 512 K + 512 V blocks, {preset}"] = {
            "us": round(us, 2), "bytes": e_in + e_out, "gbs": round((e_in + e_out) / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round((e_in + e_out) / (us * 1e-6) / 1e9 / hbm, 4),
            "alu_frac": round(lane_t / FP32_LANE_PEAK_T, 4)}
    del ek, ev

    cfg = kv.kvarn_config_from_preset("kvarn_k4v2_g128")
    B, Hq, Hkv = 4, 40, 10
    lens = kv.synthetic.ragged_lengths(3, B, 65536, 131072)
    pools, table, (kt, vt), seq_lens, nt = build_ragged_cache(kv, cfg, B, Hkv, lens, 3, dev)
    q = kv.synthetic.queries(3, B, Hq, device=dev)
    ws = torch.empty(kv.kvarn_decode_workspace_size(cfg, B, Hq, Hkv, nt), dtype=torch.uint8, device=dev)
    out = torch.empty(B, Hq, 128, device=dev)
    us = timed(lambda: kv.kvarn_decode_attention(cfg, q, Hkv, *pools["k"], *pools["v"], table, seq_lens, kt, vt,
                                                 1 / math.sqrt(128), ws, out, seq_lens_host=lens), 200)
    nbytes = sum(ragged_dec_bytes(lens, Hq, Hkv, cfg.k_bits, cfg.v_bits))
    res["decode B=4, 40q/10kv heads, ragged 64k-128k context, kvarn_k4v2_g128"] = {
        "us": round(us, 2), "lens": lens, "bytes": nbytes, "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
        "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4),
        "kv_tokens_per_s": round(Hkv * sum(lens) / (us * 1e-6), 1)}
    assert kv.kvarn_device_error() == 0
    print(json.dumps({"impl": "configs", "unit": "us per call", "hbm_peak_gbs": hbm, "peak_source": src,
                      "l2": "flushed (256 MiB read+write) before every call", "results": res}), flush=True)


def build_ragged_cache(kv, cfg, B, Hkv, lens, seed, device):
    """Encode every full 128-token block of each (sequence, kv head) of length lens[b] into pools
    whose tile ids are scattered by a seeded permutation; the last len % 128 tokens go to bf16
    tails.  Returns pools, block table [B, Hkv, nt], (k_tail, v_tail), seq_lens, nt."""
    import torch

    U = B * Hkv
    nt = max(lens) // 128 + 1
    k, v = kv.synthetic.outlier_kv(seed, U, nt * 128, device=device)
    pools = {}
    for kind, name, x in ((kv.KVARN_KIND_K, "k", k), (kv.KVARN_KIND_V, "v", v)):
        bits = cfg.k_bits if name == "k" else cfg.v_bits
        codes = torch.empty(U * nt, 128 * 16 * bits, dtype=torch.uint8, device=device)
        params = torch.empty(U * nt, 512, dtype=torch.uint8, device=device)
        scale = torch.empty(U * nt, dtype=torch.float32, device=device)
        kv.kvarn_encode_blocks(cfg, kind, x.reshape(-1, 128, 128), codes, params, scale)
        pools[name] = (codes, params, scale)
    perm = kv.synthetic.tile_permutation(seed, U * nt, device=device)
    for name in ("k", "v"):
        c, p, s = pools[name]
        c2, p2, s2 = torch.empty_like(c), torch.empty_like(p), torch.empty_like(s)
        c2[perm], p2[perm], s2[perm] = c, p, s
        pools[name] = (c2, p2, s2)
    table = perm.to(torch.int32).reshape(B, Hkv, nt).contiguous()
    tails = []
    for x in (k, v):
        t = torch.zeros(B, Hkv, 128, 128, dtype=torch.bfloat16, device=device)
        xr = x.reshape(B, Hkv, nt * 128, 128)
        for b, L in enumerate(lens):
            full = L // 128 * 128
            t[b, :, :L - full] = xr[b, :, full:L]
        tails.append(t)
    del k, v
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
    torch.cuda.synchronize()
    return pools, table, tuple(tails), seq_lens, nt


def run_append_timing():
    """Time kvarn_append_tokens on the decode workload's shape (B 16 x 8 kv heads): one token per
    sequence per step (1 in 128 steps completes a block), and 128 tokens per sequence (every
    sequence completes one block, as in chunked prefill)."""
    import torch

    import bit_kv_cache_kvarn_gb300 as kv

    kv.load()
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    dev = torch.device("cuda", 0)
    B, H, mt = DEC_B, DEC_HKV, DEC_L // 128 + 2
    n_tiles = B * H * mt
    pools = [torch.zeros(n_tiles, 4096, dtype=torch.uint8, device=dev),
             torch.zeros(n_tiles, 512, dtype=torch.uint8, device=dev), torch.zeros(n_tiles, device=dev),
             torch.zeros(n_tiles, 4096, dtype=torch.uint8, device=dev),
             torch.zeros(n_tiles, 512, dtype=torch.uint8, device=dev), torch.zeros(n_tiles, device=dev)]
    table = torch.arange(n_tiles, dtype=torch.int32, device=dev).reshape(B, H, mt)
    kt = torch.zeros(B, H, 128, 128, dtype=torch.bfloat16, device=dev)
    vt = torch.zeros_like(kt)
    ws = torch.empty(kv.kvarn_append_workspace_size(B, H), dtype=torch.uint8, device=dev)
    res = {}
    for n_new in (1, 128):
        kn = torch.randn(B, H, n_new, 128, device=dev).to(torch.bfloat16)
        lens = torch.zeros(B, dtype=torch.int32, device=dev)
        times = []
        steps = 256 if n_new == 1 else 64
        for i in range(steps):
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if int(lens.max()) + n_new > 128 * mt:
                lens.zero_()
            a.record()
            kv.kvarn_append_tokens(cfg, kn, kn, lens, kt, vt, *pools, table, ws)
            c.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(c) * 1000)
        assert kv.kvarn_device_error() == 0
        lens.zero_()
        reps = 128 if n_new == 1 else 32  # stays inside the block table without a host-side reset
        g_us = graph_us(lambda: kv.kvarn_append_tokens(cfg, kn, kn, lens, kt, vt, *pools, table, ws), reps)
        assert kv.kvarn_device_error() == 0
        res[f"n_new={n_new}"] = {"mean_us": round(statistics.mean(times), 2),
                                 "median_us": round(statistics.median(times), 2),
                                 "max_us": round(max(times), 2), "steps": steps,
                                 "graph_us": round(g_us, 2)}
    print(json.dumps({"impl": "append", "shape": f"B={B}, Hkv={H}, k2v2", "results": res}), flush=True)


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def build_decode_cache(kv, cfg, device):
    import torch

    U = DEC_B * DEC_HKV
    nt = DEC_L // 128
    k, v = kv.synthetic.outlier_kv(2, U, DEC_L, device=device)  # noqa: F841
    pools = {}
    for kind, name, x in ((kv.KVARN_KIND_K, "k", k), (kv.KVARN_KIND_V, "v", v)):
        bits = cfg.k_bits if name == "k" else cfg.v_bits
        codes = torch.empty(U * nt, 128 * 16 * bits, dtype=torch.uint8, device=device)
        params = torch.empty(U * nt, 512, dtype=torch.uint8, device=device)
        scale = torch.empty(U * nt, dtype=torch.float32, device=device)
        kv.kvarn_encode_blocks(cfg, kind, x.reshape(-1, 128, 128), codes, params, scale)
        pools[name] = (codes, params, scale)
    del k, v
    perm = kv.synthetic.tile_permutation(2, U * nt, device=device)
    for name in ("k", "v"):
        c, p, s = pools[name]
        c2, p2, s2 = torch.empty_like(c), torch.empty_like(p), torch.empty_like(s)
        c2[perm], p2[perm], s2[perm] = c, p, s
        pools[name] = (c2, p2, s2)
    table = perm.to(torch.int32).reshape(DEC_B, DEC_HKV, nt).contiguous()
    tail = torch.zeros(DEC_B, DEC_HKV, 128, 128, dtype=torch.bfloat16, device=device)
    lens = torch.full((DEC_B,), DEC_L, dtype=torch.int32, device=device)
    torch.cuda.synchronize()
    return pools, table, tail, lens


def run_gpu(args):
    global DEC_L
    DEC_L = args.ctx
    import torch
    import torch.distributed as dist

    import bit_kv_cache_kvarn_gb300 as kv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")
    kv.load()
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")

    # encode workload (config: Qwen3-4B layer, 64 seq x 8 kv heads x 128 tokens), seed 1
    n_enc = ENC_SEQ * ENC_HKV
    ek, ev = kv.synthetic.outlier_kv(1, n_enc, 128, device=device)
    ek, ev = ek.reshape(n_enc, 128, 128), ev.reshape(n_enc, 128, 128)
    out_k = (torch.empty(n_enc, 4096, dtype=torch.uint8, device=device),
             torch.empty(n_enc, 512, dtype=torch.uint8, device=device),
             torch.empty(n_enc, dtype=torch.float32, device=device))
    out_v = tuple(torch.empty_like(t) for t in out_k)
    # decode workload, seed 2
    pools, table, tail, lens = build_decode_cache(kv, cfg, device)
    q = kv.synthetic.queries(2, DEC_B, DEC_HQ, device=device)
    ws = torch.empty(kv.kvarn_decode_workspace_size(cfg, DEC_B, DEC_HQ, DEC_HKV, DEC_L // 128) // 4,
                     dtype=torch.float32, device=device)
    out = torch.empty(DEC_B, DEC_HQ, 128, dtype=torch.float32, device=device)
    sm_scale = 1 / math.sqrt(128)
    flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def l2_flush():
        # read and write 256 MiB (twice L2): a plain write leaves recently read lines resident
        flush.add_(1.0)

    def enc(xk=ek, xv=ev):
        kv.kvarn_encode_kv_blocks(cfg, xk, xv, *out_k, *out_v)

    def dec(qq=q, o=out):
        kv.kvarn_decode_attention(cfg, qq, DEC_HKV, *pools["k"], *pools["v"], table, lens, tail, tail,
                                  sm_scale, ws, o)

    torch.cuda.empty_cache()
    do_enc = args.only in ("all", "encode")
    do_dec = args.only in ("all", "decode")
    clocks = ClockSampler(local).__enter__()  # polling from before the warm-up on
    for _ in range(args.warmup):
        l2_flush()
        if do_enc:
            enc()
        if do_dec:
            dec()
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0

    ev_ = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    marks = [(ev_(), ev_(), ev_()) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_region0 = time.time()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        l2_flush()
        a, b, c = marks[s]
        a.record()
        if do_enc:
            enc()
        b.record()
        if do_dec:
            dec()
        c.record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    t_region1 = time.time()
    clocks.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    enc_ms = [a.elapsed_time(b) for a, b, _ in marks]
    dec_ms = [b.elapsed_time(c) for _, b, c in marks]
    step_ms = statistics.mean(e + d for e, d in zip(enc_ms, dec_ms))
    step_ms, enc_ms_m, dec_ms_m = max_over_ranks([step_ms, statistics.mean(enc_ms), statistics.mean(dec_ms)],
                                                 world, device)

    # end to end through host buffers: H2D of the new K/V blocks and queries, D2H of the output
    hk = ek.cpu().pin_memory()
    hv = ev.cpu().pin_memory()
    hq = q.cpu().pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    dk, dv, dq = torch.empty_like(ek), torch.empty_like(ev), torch.empty_like(q)
    copy_stream = torch.cuda.Stream(device=device)
    e2e = []
    for s in range(0 if args.no_e2e else args.warmup + args.steps):
        l2_flush()
        a, c = ev_(), ev_()
        kv_ready = torch.cuda.Event()
        a.record()
        # the step's new K/V blocks upload on a copy stream while the decode (which reads the cache
        # already resident) runs; their encode waits for the upload
        copy_stream.wait_event(a)
        with torch.cuda.stream(copy_stream):
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            kv_ready.record()
        dq.copy_(hq, non_blocking=True)
        dec(dq, out)
        hout.copy_(out, non_blocking=True)
        torch.cuda.current_stream().wait_event(kv_ready)
        enc(dk, dv)
        c.record()
        torch.cuda.synchronize()
        if s >= args.warmup:
            e2e.append(a.elapsed_time(c))
    e2e_ms = statistics.mean(e2e) if e2e else float("nan")
    (e2e_ms,) = max_over_ranks([e2e_ms], world, device)

    if rank == 0:
        hbm, src = peaks()
        e_in, e_out = enc_bytes(n_enc)
        d_cache, d_q, d_out = dec_bytes()
        enc_gbs = (e_in + e_out) / (enc_ms_m * 1e-3) / 1e9
        enc_in_gbs = e_in / (enc_ms_m * 1e-3) / 1e9
        enc_lane_t = 2 * n_enc * 128 * 128 * ENC_FP32_LANE_OPS_PER_ELEMENT / (enc_ms_m * 1e-3) / 1e12
        dec_alg = d_cache + d_q + d_out
        dec_gbs = dec_alg / (dec_ms_m * 1e-3) / 1e9
        traffic = ncu_traffic("kvarn_decode_attention")
        value_us, job_steps_per_s = replica_step_rates(step_ms, world)
        line = {
            "metric": METRIC, "value": round(value_us, 2), "unit": "us/step", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "preset": "kvarn_k2v2_g128", "sinkhorn_iters": 8,
                       "l2": "flushed (256 MiB read+write) before every step; decode cache 302 MB > L2",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "job_steps_per_s": round(job_steps_per_s, 1),
            "encode": {"us": round(enc_ms_m * 1000, 2), "gbs_bf16_input": round(enc_in_gbs, 1),
                       "gbs_read_plus_write": round(enc_gbs, 1), "hbm_frac": round(enc_gbs / hbm, 4),
                       "bytes_per_step": e_in + e_out, "launches_per_step": 1,
                       "alu_roofline": {
                           "bound": "alu", "unit": "T FP32 lane-ops/s",
                           "achieved": round(enc_lane_t, 2), "peak": round(FP32_LANE_PEAK_T, 1),
                           "frac": round(enc_lane_t / FP32_LANE_PEAK_T, 4),
                           "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2.07 GHz (a measured FFMA2 "
                                          "loop: 38.3 T lane-ops/s at ~1990 MHz)",
                           "lane_ops_per_element": ENC_FP32_LANE_OPS_PER_ELEMENT}},
            "decode": {"us": round(dec_ms_m * 1000, 2),
                       "tokens_per_s": round(DEC_B / (dec_ms_m * 1e-3), 1),
                       "kv_tokens_per_s": round(DEC_B * DEC_L / (dec_ms_m * 1e-3), 1),
                       "gbs": round(dec_gbs, 1), "hbm_frac": round(dec_gbs / hbm, 4),
                       "bytes_per_step": dec_alg, "launches_per_step": 2},
            "roofline": {"kernel": "kvarn_decode_attention (split + merge launches)", "bound": "hbm",
                         "achieved": round(dec_gbs, 1), "peak": hbm, "peak_source": src,
                         "unit": "GB/s", "frac": round(dec_gbs / hbm, 4),
                         "traffic": traffic},
            "e2e": {"value": round(replica_step_rates(e2e_ms, world)[0], 2), "unit": "us/step",
                    "h2d_bytes_per_step": 2 * ek.numel() * 2 + q.numel() * 2,
                    "d2h_bytes_per_step": out.numel() * 4,
                    "schedule": "K/V upload on a copy stream during the decode; encode after it; "
                                "q upload, decode, output download on the compute stream"},
            "gpu_launches": (do_enc + 2 * do_dec) * args.steps,
            "clocks": clocks.summary(t_region0, t_region1),
            "wall_s_timed_region": round(t_wall, 4),
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_line()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-cores", type=int, default=0,
                    help="reference arm: host cores for the oracle pool (default: all of them)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ctx", type=int, default=32768, help="decode context (profiling runs only)")
    ap.add_argument("--append-timing", action="store_true",
                    help="time kvarn_append_tokens on the decode shape instead of the step")
    ap.add_argument("--configs", action="store_true",
                    help="time the K4/V2 and K2/V2 encodes and the ragged long-context K4/V2 decode")
    ap.add_argument("--latency", action="store_true",
                    help="time single decode calls at small serving shapes instead of the step")
    ap.add_argument("--diagnostics", action="store_true",
                    help="print the codec's error diagnostics on the encode workload instead of timing")
    ap.add_argument("--only", default="all", choices=["all", "encode", "decode"],
                    help="time one part (profiling runs only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.diagnostics:
        run_diagnostics()
    elif args.append_timing:
        run_append_timing()
    elif args.configs:
        run_configs()
    elif args.latency:
        run_latency()
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
