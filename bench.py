"""Benchmark: SnapKV compression + compressed-cache decode on the workloads the metric is quoted on.

Headline (the JSON line's `value`): the full 32-layer Llama-2-7B-shaped prefill compression — B8, H32,
d128 bf16, L_prompt 16384, L_obs 32, K_pool 7, p 0.05 (k = 817 kept prefix slots per head), K with
per-channel scales s_c ~ U(0.5, 2). One step = for every layer, snapkv_compress of that layer's batch
(256 heads in one launch per kernel) followed by one decode step on its compressed cache
(snapkv_append_decode_attend: the new token's row appended, then attention over the cache). All 32
layers' inputs (64 GiB of K/V) are resident in HBM, so every step reads each layer's keys from HBM
(inputs larger than L2; no flush needed). The step is replayed as one CUDA graph.

Decode (`decode_tok_s`): the compressed-decode workload — 64 sequences with ragged prompts
L_prompt ~ U{4096..32768}, 32 layers x 32 heads, d128 bf16, each layer compressed with L_obs 32,
K_pool 7, budget 2048 (one snapkv_compress_varlen call per 16 sequences) into a [64, 32, 2208, 128]
cache per layer (74 GB over the 32 layers), then 128 decode steps x 32 layers of
snapkv_append_decode_attend, timed as a whole (one CUDA graph of 4096 launches).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --case prefill-layer|decode-layer|llama-layer [--steps K]   # small cases for ncu

--impl reference times the CPU oracle (float64 numpy, one head per step on one core) on the headline
workload. Under torchrun every rank runs its own replica (independent sequences: weak scaling, no
data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed prompt tok·head·layer/s and decode tok/s; HBM GB/s vs ~8 TB/s"
UNIT = "tok·head·layer/s"
WORKLOAD_NAME = ("32-layer Llama-2-7B-shaped prefill compression: B8 H32 d128 bf16, L_prompt 16384, L_obs 32, "
                 "K_pool 7, p 0.05 (k 817), K with per-channel scales U(0.5, 2); each layer + 1 decode step "
                 "(append + attend) on its compressed cache")
DECODE_WORKLOAD = ("compressed decode: B64 ragged L_prompt U{4096..32768}, 32 layers x H32 d128 bf16, L_obs 32, "
                   "K_pool 7, budget 2048, cap 2208, 128 decode steps (append + attend) per layer")
STAGES = ["score", "vote", "topk", "gather"]
FALLBACK_HBM_GBS = 6800.0
PROFILE_FILE = "score_vote_prefill_32layer.md"
VOTE_SOURCES = ["vote_tc.cu", "tc_common.cuh", "sm100_ptx.cuh", "snapkv_common.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-decode", action="store_true", help="skip the compressed-decode leg")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the measurements after the timed region (single layer, full-cache decode, hit "
                         "rate, GQA, varlen, long context); used for profiler captures of the step alone")
    ap.add_argument("--case", choices=["prefill-layer", "decode-layer", "llama-layer"], default=None,
                    help="a small profiling case instead of the benchmark: one layer of the headline prefill "
                         "(2 GiB of K/V) compressed --steps times, one layer of the decode workload's cache "
                         "(2.3 GB) decoded --steps times, or the single B1 Llama-2-7B-shaped layer (4 input "
                         "copies, 1 GiB of K/V) compressed and decoded one step --steps times")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------------
# Algorithmic bytes (per head, from the method's definition; intermediates excluded)
# ------------------------------------------------------------------------------------------------

def algorithmic_bytes(wl, ksel, l_prompt=None):
    """Bytes each stage must move per (sequence, layer, head). The vote reads every key once and the
    window queries; the gather reads and writes the R kept + window rows of K and V; the decode step
    reads the R+1 rows of K and V, the query, and writes the output and the appended K/V row."""
    b = 2 if wl.bf16 else 4
    d, L, lo = wl.head_dim, (l_prompt or wl.l_prompt), wl.l_obs
    R = ksel + lo
    return {
        "score+vote": b * d * (L + lo),
        "gather": 2 * 2 * R * d * b,
        "topk": 4 * ksel,
        "compress": b * d * (lo + L + 4 * R) + 4 * ksel,
        "decode": b * d * (2 * (R + 1) + 4),
        "step": b * d * (lo + L + 4 * R) + 4 * ksel + b * d * (2 * (R + 1) + 4),
    }


def decode_pass_bytes(lengths, heads, head_dim, steps, layers, esize=2):
    """Algorithmic bytes of `steps` decode steps over `layers` layers: per (sequence, layer, head) and
    step t the attention reads n = len + t + 1 rows of K and V, the query, writes the output and the
    appended K and V rows: b d (2 n + 4)."""
    total = 0
    for n0 in lengths:
        rows = steps * (2 * n0 + 4) + 2 * (steps * (steps + 1) // 2)    # sum over t of 2 (n0 + t + 1) + 4 - 2
        total += rows
    return total * heads * layers * head_dim * esize


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel_files):
    h = hashlib.sha256()
    for f in kernel_files:
        with open(os.path.join(ROOT, "kv_cache_compression_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_files, profile=PROFILE_FILE):
    """dram bytes per launch recorded in profiles/ for the dominant kernel, if its source is unchanged."""
    digest = source_digest(kernel_files)
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None, digest
    text = open(path).read()
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != digest:
        return None, digest
    return int(m_bytes.group(1)), digest

# ------------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (spawned worker processes, one BLAS thread each)
# ------------------------------------------------------------------------------------------------



# ------------------------------------------------------------------------------------------------
# CPU oracle timing (spawned worker processes, one BLAS thread each)
# ------------------------------------------------------------------------------------------------

def oracle_sample_units(n_units, seed=0x0C0FFEE):
    """A seeded sample of distinct (layer, sequence, head) units of the headline workload."""
    import numpy as np
    rng = np.random.default_rng(seed)
    flat = rng.choice(32 * 8 * 32, size=n_units, replace=False)
    return [(int(u // 256), int((u // 32) % 8), int(u % 32)) for u in flat]


def _oracle_worker(args):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    units, = args
    import synth
    from oracle import snapkv_oracle as orc
    wl = synth.WORKLOADS[2]
    busy, tokens = 0.0, 0
    for layer, seq, head in units:
        hi = synth.host_head(wl, layer, seq, head, threads=1)
        qn, kn, vn = synth.host_decode_token(wl, layer, seq, head, 0)
        t0 = time.perf_counter()
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p)
        kc, vc = orc.append(ref.k_c, ref.v_c, kn, vn)
        orc.decode_attend(qn, kc, vc)
        busy += time.perf_counter() - t0
        tokens += wl.l_prompt
    return busy, tokens


def cpu_baseline(per_core=48):
    import multiprocessing as mp
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    cores = max(1, min(cores, 64))
    units = oracle_sample_units(per_core * cores)
    shards = [units[i::cores] for i in range(cores)]
    env_before = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_before:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(s,) for s in shards if s])
    finally:
        for k, v in env_before.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    busy = [r[0] for r in res]
    tokens = sum(r[1] for r in res)
    return {"value": tokens / max(busy), "unit": UNIT, "cores": len(res), "kind": "oracle",
            "sample": f"{len(units)} seeded (layer, sequence, head) units of the 32-layer prefill workload "
                      f"(compress + append + decode per head), {len(res)} processes with one BLAS thread "
                      f"each; value = tokens*heads*layers / slowest process's compute seconds (extrapolated "
                      f"per head to the workload's 8192 heads); total CPU compute {sum(busy):.1f} s"}


# ------------------------------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ------------------------------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    import synth
    from oracle import snapkv_oracle as orc
    wl = synth.WORKLOADS[2]
    units = oracle_sample_units(8, seed=0x5A17)
    cache = {}

    def inputs(i):
        u = units[i % len(units)]
        if u not in cache:
            cache[u] = (synth.host_head(wl, *u, threads=1), synth.host_decode_token(wl, *u, 0))
        return cache[u]

    def step(i):
        hi, (qn, kn, vn) = inputs(i)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p)
        kc, vc = orc.append(ref.k_c, ref.v_c, kn, vn)
        return orc.decode_attend(qn, kc, vc)

    for i in range(len(units)):   # generate every sampled head's input before timing
        inputs(i)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = wl.l_prompt * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox inputs; no dataset or weights)",
            "config": {"workload": WORKLOAD_NAME, "global_batch": 8, "seq_len": wl.l_prompt, "layers": wl.layers,
                       "sample": "one (layer, sequence, head) per step (compress + append + decode), cycling over "
                                 "8 seeded units; value per head, the unit of the metric"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "one head per step on one core (one BLAS thread)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)



# ------------------------------------------------------------------------------------------------
# Replicas across ranks (weak scaling, no data-path collective)
# ------------------------------------------------------------------------------------------------

def replica_sequence(rank: int) -> int:
    """The sequence a rank compresses in a one-sequence workload: its own, so ranks share no data."""
    return rank


def replica_batch(rank: int, batch: int) -> int:
    """First sequence of a rank's batch: rank r compresses sequences r*batch .. r*batch + batch - 1, so
    the replicas' inputs (and results) are distinct and no data crosses ranks."""
    return rank * batch


def max_over_ranks(elapsed_ms: float, world: int, device) -> float:
    """The slowest rank's timed region (every rank gets it)."""
    if world <= 1:
        return float(elapsed_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, over the slowest rank's step time."""
    return units_per_rank_step * world / (ms_per_step * 1e-3)



def full_cache_decode(torch, snapkv, synth, dev, ksel_budget=1024):
    """Decode attention over the uncompressed prompt cache against the compressed one.

    The synthetic analogue of the SnapKV explainer's decode figures (section 実験結果,
    デコード速度とメモリ効率: 16K-token inputs, batch 2): one layer of B2 H32 d128 bf16, a 16384-row
    uncompressed cache (every prompt row kept) and the cache SnapKV keeps (1024 + 32 rows, + the
    new row). Each decode call is captured as a CUDA graph and replayed; events on the stream
    time 50 replays of each. Attention only (no projections or MLP), so the ratio is of the
    attention's own time and bytes.
    """
    wl = synth.WORKLOADS[1]
    B, H, d, L = 2, wl.heads, wl.head_dim, wl.l_prompt
    _, k, v, _ = synth.device_inputs(wl, 0, 0, B, L, dev)
    qn, _, _ = synth.device_decode_tokens(wl, 0, 0, 0, B, dev)
    r_c = ksel_budget + wl.l_obs
    kc = k[:, :, :r_c].contiguous()
    vc = v[:, :, :r_c].contiguous()
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    res = {}
    for name, (kk, vv, rows) in {"uncompressed": (k, v, L), "compressed": (kc, vc, r_c)}.items():
        length = torch.full((B,), rows, dtype=torch.int32, device=dev)
        ws = snapkv.new_workspace(snapkv.decode_workspace_size(B, H, d, kk.shape[2]), dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                snapkv.decode_attend(qn, kk, vv, length, out=out, workspace=ws, stream=stream)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                snapkv.decode_attend(qn, kk, vv, length, out=out, workspace=ws, stream=stream)
            for _ in range(5):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(50):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / 50
        kv_bytes = 2 * B * H * rows * d * 2
        res[name] = {"ms": ms, "rows": rows, "kv_bytes_per_layer": kv_bytes,
                     "hbm_gbs_algorithmic": (kv_bytes + 2 * B * H * d * 2) / (ms * 1e-3) / 1e9}
    res["decode_speedup"] = res["uncompressed"]["ms"] / res["compressed"]["ms"]
    res["kv_memory_ratio"] = res["uncompressed"]["kv_bytes_per_layer"] / res["compressed"]["kv_bytes_per_layer"]
    res["workload"] = "B2 H32 d128 bf16, 16384-row prompt cache vs 1056-row SnapKV cache (budget 1024 + L_obs 32), one layer"
    del k, v, kc, vc
    return res


def hit_rate_diagnostic(torch, snapkv, synth, dev, theta=0.05):
    """The explainer's Hit Rate (section Hit Rate（適中率）の定式化) of the single-layer workload's
    selection: a decode-step query over the uncompressed cache (prompt + the new row), theta = 0.05,
    summed over the 32 heads; plus the diagnostic kernel's time (mean of 20 calls between events)."""
    wl = synth.WORKLOADS[1]
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, wl.l_prompt, dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget)
    qn, kn, _ = synth.device_decode_tokens(wl, 0, 0, 0, 1, dev)
    cache = torch.cat([k, kn[:, :, None, :]], dim=2).contiguous()
    length = torch.full((1,), wl.l_prompt + 1, dtype=torch.int32, device=dev)
    l_prefix = wl.l_prompt - wl.l_obs
    hits, total = snapkv.hit_rate(qn, cache, length, res["idx"], l_prefix, theta=theta)
    # a finer threshold too: independent random queries spread their weight thinly over 16K keys
    fine = 4.0 / wl.l_prompt
    hf, tf = snapkv.hit_rate(qn, cache, length, res["idx"], l_prefix, theta=fine)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        snapkv.hit_rate(qn, cache, length, res["idx"], l_prefix, theta=theta)
    e1.record()
    torch.cuda.synchronize(dev)
    h, t = int(hits.sum().item()), int(total.sum().item())
    h2, t2 = int(hf.sum().item()), int(tf.sum().item())
    ms = e0.elapsed_time(e1) / 20
    return {"H": (h / t) if t else None, "hits": h, "above_theta": t, "theta": theta,
            "H_fine": (h2 / t2) if t2 else None, "above_fine": t2, "theta_fine": fine,
            "kernel_ms": ms, "kernel_alg_gbs": 32 * (wl.l_prompt + 1) * wl.head_dim * 2 / (ms * 1e-3) / 1e9,
            "note": "synthetic inputs: the value describes these tensors, not a trained model"}


def gqa_compress(torch, snapkv, synth, dev, batch=1, copies=4):
    """SnapKV compression under grouped-query attention on a Llama-3-8B-shaped layer: `batch`
    sequences, 32 query heads sharing 8 KV heads (G = 4), d128 bf16, L_prompt 16384, L_obs 32 (128
    window rows per KV head), K_pool 7, budget 1024. The input copies (more K/V than L2 together) are
    each captured as a CUDA graph and replayed in turn; events time 48 replays."""
    hq, hkv, L, lo = 32, 8, 16384, 32
    wl = synth.WORKLOADS[1].with_(heads=hq, l_prompt=L, l_obs=lo)
    ins = []
    for c in range(copies):
        q, k_all, v_all, _ = synth.device_inputs(wl, c, 0, batch, L, dev)
        ins.append((q, k_all[:, :hkv].contiguous(), v_all[:, :hkv].contiguous()))
        del k_all, v_all
    res = snapkv.compress(*ins[0], pool_kernel=7, budget=1024)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)

    def call(c):
        snapkv.compress(*ins[c], pool_kernel=7, budget=1024, k_out=res["k_out"], v_out=res["v_out"],
                        len_out=res["len"], idx_out=res["idx"], workspace=res["workspace"], stream=stream)
    graphs = []
    with torch.cuda.stream(stream):
        for c in range(copies):
            call(c)
        torch.cuda.synchronize(dev)
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(c)
            graphs.append(g)
        for i in range(8):
            graphs[i % copies].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(48):
            graphs[i % copies].replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / 48
    k_bytes = batch * hkv * L * 128 * 2
    alg = k_bytes + batch * hq * lo * 256 + 4 * batch * hkv * (1024 + lo) * 256
    peak, _ = read_peaks()
    del ins, res, graphs
    torch.cuda.empty_cache()
    return {"workload": f"Llama-3-8B-shaped layer: B{batch}, 32 query heads / 8 KV heads (G 4), d128 bf16, "
                        f"L_prompt 16384, L_obs 32, K_pool 7, budget 1024",
            "ms_per_compress": ms, "tok_head_per_s": batch * L * hkv / (ms * 1e-3), "alg_bytes": alg,
            "compress_alg_gbs": alg / (ms * 1e-3) / 1e9, "frac_of_measured": alg / (ms * 1e-3) / 1e9 / peak,
            "l2": f"{copies} input copies rotated ({copies * 2 * k_bytes / 2**20:.0f} MiB of K/V > L2)"}


def long_context_compress(torch, snapkv, synth, dev, reps=10):
    """The long-context workload: B1 H32 d128 bf16, L_prompt 131072, L_obs 64, K_pool 13, budget
    4096 (planted keys in runs of 8). One input copy (2.1 GB of K/V, far above L2); the compress is
    captured as a CUDA graph and events time `reps` replays."""
    wl = synth.WORKLOADS[3]
    L = wl.l_prompt
    q, k, v, _ = synth.device_inputs(wl, 0, 0, 1, L, dev)
    res = snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)

    def call():
        snapkv.compress(q, k, v, pool_kernel=wl.pool_kernel, budget=wl.budget, k_out=res["k_out"], v_out=res["v_out"],
                        len_out=res["len"], idx_out=res["idx"], workspace=res["workspace"], stream=stream)
    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    H, d, lo, eb, R = wl.heads, wl.head_dim, wl.l_obs, 2, wl.budget + wl.l_obs
    alg = H * (eb * d * (L + lo) + 2 * 2 * R * d * eb + 4 * wl.budget)
    del q, k, v, res, g
    torch.cuda.empty_cache()
    return {"workload": "long context: B1 H32 d128 bf16, L_prompt 131072, L_obs 64, K_pool 13, budget 4096",
            "ms_per_compress": ms, "tok_head_per_s": L * H / (ms * 1e-3), "alg_bytes": alg,
            "alg_gbs": alg / (ms * 1e-3) / 1e9}


def varlen_compress(torch, snapkv, synth, dev, nseq=16, ratio_p=0.125):
    """One snapkv_compress_varlen call over the first 16 prompts of the ragged-prompt decode workload
    (L_prompt drawn from U{4096..32768}, H32 d128 bf16, L_obs 32, K_pool 7) under the ratio rule
    p = 0.125, so that every sequence keeps its own number of rows. Inputs are padded to the longest
    prompt (several GB of K/V, far above L2); the call is captured as a CUDA graph and events time 10
    replays."""
    wl = synth.WORKLOADS[4]
    lengths = wl.prompt_lengths()[:nseq]
    q, k, v = synth.device_inputs_padded(wl, 0, 0, lengths, dev, pad_value=0.0)
    res = snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=ratio_p)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)

    def call():
        snapkv.compress_varlen(q, k, v, lengths, pool_kernel=wl.pool_kernel, ratio_p=ratio_p, out=res, stream=stream)
    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / 10
    H, d, lo, eb = wl.heads, wl.head_dim, wl.l_obs, 2
    alg = sum(H * (eb * d * (L + lo) + 2 * 2 * (kb + lo) * d * eb + 4 * kb) for L, kb in zip(lengths, res["ks"]))
    tok_heads = sum(lengths) * H
    del q, k, v, res, g
    torch.cuda.empty_cache()
    return {"workload": f"ragged prompts: {nseq} sequences, L_prompt U{{4096..32768}} (total {sum(lengths)}), "
                        f"H32 d128 bf16, L_obs 32, K_pool 7, p {ratio_p} (k per sequence)",
            "ms_per_call": ms, "tok_head_per_s": tok_heads / (ms * 1e-3), "alg_bytes": alg,
            "alg_gbs": alg / (ms * 1e-3) / 1e9}

def timing_event(torch):
    """A timing event that, recorded inside a stream capture, becomes an event-record node."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def stage_samples(launch_step, stream, side, n_ev, n_diag, dev, n_rot):
    """Per-stage device times of n_diag calls of launch_step(c, stream, events), c rotating over n_rot
    inputs: graph replays with event nodes, else eager calls."""
    import torch
    names = STAGES + ["decode"]
    samples = {s: [] for s in names}
    try:
        graphs, event_sets = [], []
        for c in range(n_rot):
            evs = [timing_event(torch) for _ in range(n_ev + 2)]
            for e in evs:          # torch creates its events lazily: record once so each has a handle
                e.record(side)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                launch_step(c, side, evs)
            graphs.append(g)
            event_sets.append(evs)
        torch.cuda.synchronize(dev)
        for i in range(n_diag):
            c = i % n_rot
            graphs[c].replay()
            torch.cuda.synchronize(dev)
            evs = event_sets[c]
            for j, s in enumerate(names):
                samples[s].append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
        return samples, ("%d graph replays of the timed work with event-record nodes around each stage's "
                         "kernels (right after the timed region)" % n_diag)
    except RuntimeError:
        samples = {s: [] for s in names}
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev + 2)]
    for e in evs:
        e.record(stream)
    for i in range(n_diag):
        torch.cuda._sleep(2_000_000)   # the GPU never waits for the host inside an event pair
        launch_step(i % n_rot, stream, evs)
        torch.cuda.synchronize(dev)
        for j, s in enumerate(names):
            samples[s].append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
    return samples, "%d eager calls with CUDA events around each stage's kernels" % n_diag



# ------------------------------------------------------------------------------------------------
# Headline workload: the 32-layer prefill compression
# ------------------------------------------------------------------------------------------------

def setup_prefill(torch, snapkv, synth, dev, seq0, layers=None):
    """Device state of the 32-layer prefill: every layer's inputs, decode-step tokens and outputs."""
    wl = synth.WORKLOADS[2]
    B, H, d, L, lo = wl.batch, wl.heads, wl.head_dim, wl.l_prompt, wl.l_obs
    n_layers = wl.layers if layers is None else layers
    params = snapkv.make_params(batch=B, heads=H, head_dim=d, l_obs=lo, l_prompt=L, pool_kernel=wl.pool_kernel,
                                ratio_p=wl.ratio_p, dtype=snapkv.BF16)
    ksel = snapkv.kept(params)
    R = ksel + lo
    cap = R + 1                      # room for the decode step's row
    bf = torch.bfloat16
    per_layer = []
    for layer in range(n_layers):
        q, k, v, _ = synth.device_inputs(wl, layer, seq0, B, L, dev)
        tok = torch.empty((3, B, H, d), dtype=bf, device=dev)
        synth.device_decode_tokens_into(tok, wl, layer, 0, seq0)
        per_layer.append(SimpleNamespace(
            q=q, k=k, v=v, tok=tok,
            k_out=torch.empty((B, H, cap, d), dtype=bf, device=dev),
            v_out=torch.empty((B, H, cap, d), dtype=bf, device=dev),
            idx=torch.empty((B, H, ksel), dtype=torch.int32, device=dev),
            lens=torch.zeros((2, B), dtype=torch.int32, device=dev),
            out=torch.empty((B, H, d), dtype=bf, device=dev)))
    torch.cuda.synchronize(dev)
    return SimpleNamespace(
        wl=wl, B=B, H=H, d=d, L=L, lo=lo, n_layers=n_layers, params=params, ksel=ksel, R=R, cap=cap,
        layers=per_layer, status=torch.zeros((1,), dtype=torch.int32, device=dev),
        ws_c=snapkv.new_workspace(snapkv.compress_workspace_size(params), dev),
        ws_d=snapkv.new_workspace(snapkv.decode_workspace_size(B, H, d, cap), dev))


def launch_layer(m, snapkv, layer, strm, events=None):
    """Enqueue one layer on `strm`: snapkv_compress (stage events recorded inside the library), then one
    decode step on the compressed cache (append + attention in one call). The compression writes the
    cache length into lens[0]; the decode step reads it and writes lens[1]."""
    x = m.layers[layer]
    lib = snapkv.lib()
    P = ctypes.c_void_p
    n_ev = 2 * len(STAGES)
    ev_arr = (ctypes.c_void_p * n_ev)(*[e.cuda_event for e in events[:n_ev]]) if events else None
    st = lib.snapkv_compress_profiled(ctypes.byref(m.params), P(x.q.data_ptr()), P(x.k.data_ptr()),
                                      P(x.v.data_ptr()), P(x.k_out.data_ptr()), P(x.v_out.data_ptr()), m.cap,
                                      P(x.lens[0].data_ptr()), P(x.idx.data_ptr()), None, P(m.ws_c.data_ptr()),
                                      m.ws_c.numel(), P(m.status.data_ptr()), ctypes.c_void_p(strm.cuda_stream),
                                      ev_arr, n_ev if events else 0)
    if st != 0:
        raise RuntimeError(f"snapkv_compress: {snapkv.status_string(st)}")
    if events:
        events[n_ev].record(strm)
    snapkv.append_decode_attend(x.tok[0], x.tok[1], x.tok[2], x.k_out, x.v_out, x.lens[0], x.lens[1], out=x.out,
                                workspace=m.ws_d, dev_status=m.status, stream=strm)
    if events:
        events[n_ev + 1].record(strm)


def check_status(m, snapkv, where):
    st = int(m.status.item())
    if st != 0:
        raise RuntimeError(f"device status {where}: {snapkv.status_string(st)}")


def e2e_prefill(torch, snapkv, m, dev, stream, n_steps, world):
    """The headline step end to end through the public API with host buffers: every layer-call uploads
    its Q, K and decode tokens from pinned host memory, compresses with V left in page-locked host memory
    (only the kept and window rows of V cross the link: the method never reads the rest), runs the decode
    step and reads K_c, V_c, idx and the output back to pinned host memory; copies and kernels of
    neighbouring layer-calls overlap on three streams (two buffer sets). The host link bounds the rate.
    Two host buffer sets hold layers 0 and 1's inputs; layer l of a step uses set l % 2."""
    bf = torch.bfloat16
    host_in, dev_in, dev_out, host_out = [], [], [], []
    for j in range(2):
        x = m.layers[j]
        hs = []
        for t in (x.q, x.k, x.v, x.tok):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            hs.append(h)
        host_in.append(hs)
        dev_in.append([torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.tok)])
        do = [torch.empty_like(x.k_out), torch.empty_like(x.v_out), torch.empty_like(x.idx), torch.empty_like(x.out),
              torch.zeros_like(x.lens)]
        dev_out.append(do)
        host_out.append([torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in do[:4]])
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    wl = m.wl
    torch.cuda.synchronize(dev)

    def run(n_calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_s.wait_stream(stream)
        down_s.wait_stream(stream)
        for i in range(n_calls):
            j = i % 2
            if i >= 2:
                up_s.wait_event(comp_done[j])      # call i-2 is done reading this input set
            with torch.cuda.stream(up_s):
                for dst, src in zip(dev_in[j], (host_in[j][0], host_in[j][1], host_in[j][3])):
                    dst.copy_(src, non_blocking=True)
                up_done[j].record(up_s)
            stream.wait_event(up_done[j])
            if i >= 2:
                stream.wait_event(down_done[j])    # call i-2's outputs have reached the host
            dq, dk, dtok = dev_in[j]
            ko, vo, io, oo, ln = dev_out[j]
            snapkv.compress(dq, dk, host_in[j][2], pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p, cap=m.cap,
                            k_out=ko, v_out=vo, len_out=ln[0], idx_out=io, workspace=m.ws_c, dev_status=m.status,
                            stream=stream)
            snapkv.append_decode_attend(dtok[0], dtok[1], dtok[2], ko, vo, ln[0], ln[1], out=oo, workspace=m.ws_d,
                                        dev_status=m.status, stream=stream)
            comp_done[j].record(stream)
            down_s.wait_event(comp_done[j])
            with torch.cuda.stream(down_s):
                for dst, src in zip(host_out[j], (ko, vo, io, oo)):
                    dst.copy_(src, non_blocking=True)
                down_done[j].record(down_s)
        stream.wait_stream(up_s)
        stream.wait_stream(down_s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    run(2)
    ms = max_over_ranks(run(n_steps * m.n_layers) / n_steps, world, dev)
    check_status(m, snapkv, "after the end-to-end steps")
    esz = 2
    v_rows = m.B * m.H * m.R * m.d * esz                       # kept + window rows of V, per layer
    h2d_layer = sum(t.numel() * t.element_size() for t in (host_in[0][0], host_in[0][1], host_in[0][3])) + v_rows
    d2h_layer = sum(t.numel() * t.element_size() for t in host_out[0])
    units = m.B * m.L * m.H * m.n_layers
    del host_in, dev_in, dev_out, host_out
    return {"value": units * world / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d_layer * m.n_layers,
            "d2h_bytes_per_step": d2h_layer * m.n_layers, "ms_per_step": ms, "steps": n_steps,
            "path": "per layer: pinned host Q, K and decode tokens -> device; V stays in pinned host memory and "
                    "snapkv.compress reads its kept and window rows over the host link (counted in h2d); "
                    "append_decode_attend; K_c, V_c, idx, out -> pinned host. Two host buffer sets (layers 0 "
                    "and 1's inputs; layer l uses set l % 2); uploads, kernels and downloads of neighbouring "
                    "layers overlap on three streams"}


# ------------------------------------------------------------------------------------------------
# Decode workload: B64 ragged prompts, 32 layers, 128 steps
# ------------------------------------------------------------------------------------------------

def setup_decode(torch, snapkv, synth, dev, seq_offset=0, layers=None, chunk=16):
    """Compress every layer's 64 ragged prompts into that layer's cache and generate every step's new
    tokens. Returns the device state and the compression's own time (events around each call)."""
    wl = synth.WORKLOADS[4]
    B, H, d, lo, steps = wl.batch, wl.heads, wl.head_dim, wl.l_obs, wl.decode_steps
    n_layers = wl.layers if layers is None else layers
    lengths = wl.prompt_lengths()
    cap = wl.budget + lo + steps
    bf = torch.bfloat16
    kc = torch.empty((n_layers, B, H, cap, d), dtype=bf, device=dev)
    vc = torch.empty_like(kc)
    lens = torch.zeros((n_layers, 2, B), dtype=torch.int32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    compress_ms, tok_heads = 0.0, 0
    for layer in range(n_layers):
        for c0 in range(0, B, chunk):
            ls = lengths[c0:c0 + chunk]
            q, k, v = synth.device_inputs_padded(wl, layer, seq_offset + c0, ls, dev, pad_value=0.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            snapkv.compress_varlen(q, k, v, ls, pool_kernel=wl.pool_kernel, budget=wl.budget,
                                   k_out=kc[layer, c0:c0 + len(ls)], v_out=vc[layer, c0:c0 + len(ls)],
                                   len_out=lens[layer, 0, c0:c0 + len(ls)], want_idx=False, dev_status=status)
            e1.record()
            torch.cuda.synchronize(dev)
            compress_ms += e0.elapsed_time(e1)
            tok_heads += sum(ls) * H
            del q, k, v
    tok = torch.empty((steps, n_layers, 3, B, H, d), dtype=bf, device=dev)
    for t in range(steps):
        for layer in range(n_layers):
            synth.device_decode_tokens_into(tok[t, layer], wl, layer, t, seq_offset)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status after the decode workload's compression: "
                           f"{snapkv.status_string(int(status.item()))}")
    torch.cuda.empty_cache()
    return SimpleNamespace(wl=wl, B=B, H=H, d=d, cap=cap, steps=steps, n_layers=n_layers, lengths=lengths,
                           kc=kc, vc=vc, lens=lens, len0=lens[:, 0].clone(), tok=tok, status=status,
                           out=torch.empty((n_layers, B, H, d), dtype=bf, device=dev),
                           ws=snapkv.new_workspace(snapkv.decode_workspace_size(B, H, d, cap), dev),
                           compress_ms=compress_ms, compress_tok_heads=tok_heads)


def decode_leg(torch, snapkv, synth, dev, world, rank=0, passes=2, sample_clocks=True, local_rank=0):
    """decode tok/s of the compressed-decode workload: 128 steps x 32 layers of
    snapkv_append_decode_attend over the compressed caches, captured as one CUDA graph; the lengths are
    reset to the compressed lengths before every pass (outside the timed region). Under replicas rank r
    decodes its own 64 sequences (seq_offset = 64 r)."""
    m = setup_decode(torch, snapkv, synth, dev, seq_offset=replica_batch(rank, synth.WORKLOADS[4].batch))
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)

    def calls(strm):
        for t in range(m.steps):
            for layer in range(m.n_layers):
                x = m.tok[t, layer]
                snapkv.append_decode_attend(x[0], x[1], x[2], m.kc[layer], m.vc[layer], m.lens[layer, t % 2],
                                            m.lens[layer, (t + 1) % 2], out=m.out[layer], workspace=m.ws,
                                            dev_status=m.status, stream=strm)

    # one eager pass first (also checks the device status), then the graph
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        calls(side)
    torch.cuda.synchronize(dev)
    if int(m.status.item()) != 0:
        raise RuntimeError(f"device status after an eager decode pass: {snapkv.status_string(int(m.status.item()))}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        calls(side)
    times = []
    sampler = ClockSampler(local_rank) if sample_clocks else None
    for i in range(passes + 1):
        m.lens[:, 0].copy_(m.len0)
        torch.cuda.synchronize(dev)
        if i == 1 and sampler:
            sampler.start()
            time.sleep(0.2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i > 0:                      # pass 0 is the warm-up
            times.append(e0.elapsed_time(e1))
    clocks = sampler.stop() if sampler else None
    if int(m.status.item()) != 0:
        raise RuntimeError(f"device status after the decode passes: {snapkv.status_string(int(m.status.item()))}")
    final_len = m.lens[:, m.steps % 2].cpu()
    assert bool((final_len == m.len0.cpu() + m.steps).all()), "every decode step appended one row"
    pass_ms = max_over_ranks(statistics.fmean(times), world, dev)
    tokens = m.B * m.steps
    alg = decode_pass_bytes([int(x) for x in m.len0[0].cpu().tolist()], m.H, m.d, m.steps, m.n_layers)
    peak, peak_kind = read_peaks()
    launches = m.steps * m.n_layers
    achieved = alg / (pass_ms * 1e-3) / 1e9
    res = {"workload": DECODE_WORKLOAD, "decode_tok_s": tokens * world / (pass_ms * 1e-3), "ms_per_pass": pass_ms,
           "pass_ms_each": times, "tokens_per_pass": tokens,
           "prompt_lengths": {"min": min(m.lengths), "max": max(m.lengths), "sum": sum(m.lengths)},
           "cache_rows_after_compress": int(m.len0[0, 0].item()), "cap": m.cap,
           "launches_per_pass": launches, "avg_launch_ms": pass_ms / launches,
           "roofline": {"bound": "hbm", "kernel": "decode_cluster_kernel (append + attention)", "achieved": achieved,
                        "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                        "alg_bytes_per_pass": alg, "alg_bytes_per_launch": alg / launches,
                        "note": "per (sequence, layer, head) and step: b d (2 n + 4) with n = rows after the append"},
           "ceiling_tok_s_at_peak": tokens / (alg / (peak * 1e9)),
           "clocks": clocks,
           "prefill_compress": {"ms_total": m.compress_ms,
                                "tok_head_layer_per_s": m.compress_tok_heads / (m.compress_ms * 1e-3),
                                "note": "the workload's own compression (snapkv_compress_varlen, 16 sequences per "
                                        "call, 128 calls), events around each call; not part of decode tok/s"},
           "launch": "one CUDA graph of 128 steps x 32 layers of snapkv_append_decode_attend per pass; lengths "
                     "reset to the compressed lengths between passes (outside the timed region)"}
    del m, g
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------------------------
# Single-layer workload (extra): one Llama-2-7B-shaped layer, B1, budget 1024, planted keys
# ------------------------------------------------------------------------------------------------

def setup_single_layer(torch, snapkv, synth, dev, copies=4):
    """The Llama-2-7B-shaped layer (B1 H32 d128 bf16, L_prompt 16384, L_obs 32, K_pool 7, budget 1024, 64
    planted keys per head) in `copies` input copies, with its compressed caches and workspaces."""
    wl = synth.WORKLOADS[1]
    B, H, d, L, lo = 1, wl.heads, wl.head_dim, wl.l_prompt, wl.l_obs
    params = snapkv.make_params(batch=B, heads=H, head_dim=d, l_obs=lo, l_prompt=L, pool_kernel=wl.pool_kernel,
                                budget=wl.budget, dtype=snapkv.BF16)
    ksel = snapkv.kept(params)
    R = ksel + lo
    cap = R + 1
    bf = torch.bfloat16
    layers = []
    for c in range(copies):
        q, k, v, _ = synth.device_inputs(wl, c, 0, 1, L, dev)
        tok = torch.empty((3, B, H, d), dtype=bf, device=dev)
        synth.device_decode_tokens_into(tok, wl, c, 0, 0)
        layers.append(SimpleNamespace(q=q, k=k, v=v, tok=tok,
                                      k_out=torch.empty((B, H, cap, d), dtype=bf, device=dev),
                                      v_out=torch.empty((B, H, cap, d), dtype=bf, device=dev),
                                      idx=torch.empty((B, H, ksel), dtype=torch.int32, device=dev),
                                      lens=torch.zeros((2, B), dtype=torch.int32, device=dev),
                                      out=torch.empty((B, H, d), dtype=bf, device=dev)))
    m = SimpleNamespace(wl=wl, B=B, H=H, d=d, L=L, lo=lo, n_layers=copies, params=params, ksel=ksel, R=R, cap=cap,
                        layers=layers, status=torch.zeros((1,), dtype=torch.int32, device=dev),
                        ws_c=snapkv.new_workspace(snapkv.compress_workspace_size(params), dev),
                        ws_d=snapkv.new_workspace(snapkv.decode_workspace_size(B, H, d, cap), dev))
    return m


def single_layer_extra(torch, snapkv, synth, dev, n_steps=200, copies=4):
    """One layer (setup_single_layer) + one decode step, as CUDA graph replays over 4 input copies (1 GiB
    of K/V > L2), with the score/vote kernel's own time from event nodes."""
    m = setup_single_layer(torch, snapkv, synth, dev, copies)
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for c in range(copies):
            launch_layer(m, snapkv, c, side)
    torch.cuda.synchronize(dev)
    check_status(m, snapkv, "single layer")
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            launch_layer(m, snapkv, c, side)
        graphs.append(g)
    for i in range(8):
        graphs[i % copies].replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n_steps):
        graphs[i % copies].replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n_steps
    samples, _ = stage_samples(lambda c, s, ev: launch_layer(m, snapkv, c, s, ev), stream, side, 2 * len(STAGES),
                               64, dev, copies)
    check_status(m, snapkv, "single layer")
    mean = {s: statistics.fmean(v) for s, v in samples.items()}
    wl, ksel, H, L = m.wl, m.ksel, m.H, m.L
    alg = algorithmic_bytes(wl, ksel)
    peak, _ = read_peaks()
    vote_gbs = alg["score+vote"] * H / (mean["score"] * 1e-3) / 1e9
    del m, graphs
    torch.cuda.empty_cache()
    return {"workload": "Llama-2-7B-shaped layer: B1 H32 d128 bf16, L_prompt 16384, L_obs 32, K_pool 7, budget "
                        "1024 (64 planted keys/head), + 1 decode step",
            "ms_per_step": ms, "tok_head_per_s": L * H / (ms * 1e-3),
            "hbm_gbs_algorithmic_step": alg["step"] * H / (ms * 1e-3) / 1e9,
            "stage_ms_mean": {k: round(v, 5) for k, v in mean.items()},
            "vote_kernel_alg_gbs": vote_gbs, "vote_kernel_frac": vote_gbs / peak,
            "l2": f"{copies} input copies rotated (1 GiB of K/V > L2)"}


# ------------------------------------------------------------------------------------------------
# Small profiling cases (for ncu captures: a few GB on the device)
# ------------------------------------------------------------------------------------------------

def run_case(args, local_rank):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import synth
    from kv_cache_compression_gb300 import snapkv
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    if args.case == "prefill-layer":
        m = setup_prefill(torch, snapkv, synth, dev, 0, layers=1)
        for _ in range(max(1, args.steps)):
            launch_layer(m, snapkv, 0, stream)
        torch.cuda.synchronize(dev)
        check_status(m, snapkv, "prefill-layer case")
        print(json.dumps({"case": args.case, "calls": args.steps, "kept": m.ksel, "heads": m.B * m.H}))
    elif args.case == "llama-layer":
        m = setup_single_layer(torch, snapkv, synth, dev)
        for i in range(max(1, args.steps)):
            launch_layer(m, snapkv, i % m.n_layers, stream)
        torch.cuda.synchronize(dev)
        check_status(m, snapkv, "llama-layer case")
        print(json.dumps({"case": args.case, "calls": args.steps, "kept": m.ksel, "heads": m.B * m.H}))
    else:
        m = setup_decode(torch, snapkv, synth, dev, layers=1)
        for t in range(max(1, args.steps)):
            x = m.tok[t % m.steps, 0]
            snapkv.append_decode_attend(x[0], x[1], x[2], m.kc[0], m.vc[0], m.lens[0, t % 2], m.lens[0, (t + 1) % 2],
                                        out=m.out[0], workspace=m.ws, dev_status=m.status, stream=stream)
        torch.cuda.synchronize(dev)
        if int(m.status.item()) != 0:
            raise RuntimeError(snapkv.status_string(int(m.status.item())))
        print(json.dumps({"case": args.case, "calls": args.steps, "heads": m.B * m.H, "cap": m.cap}))


# ------------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import synth
    from kv_cache_compression_gb300 import snapkv

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    seq0 = replica_batch(rank, synth.WORKLOADS[2].batch)   # each rank compresses its own 8 sequences
    m = setup_prefill(torch, snapkv, synth, dev, seq0)
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)

    # One eager step, then the step captured as one CUDA graph (32 layers x (compress + decode step)).
    with torch.cuda.stream(side):
        for layer in range(m.n_layers):
            launch_layer(m, snapkv, layer, side)
    torch.cuda.synchronize(dev)
    check_status(m, snapkv, "after the eager step")
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=side):
        for layer in range(m.n_layers):
            launch_layer(m, snapkv, layer, side)
    torch.cuda.synchronize(dev)
    for _ in range(max(args.warmup, 3)):
        step_graph.replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)   # let the sampler start before the timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for _ in range(args.steps):
        step_graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    check_status(m, snapkv, "after the timed steps")
    del step_graph

    # Per-kernel durations (right after the timed region): one layer captured with event-record nodes
    # around each stage's kernels, for 4 different layers, replayed in turn.
    n_diag = 32
    samples, stage_method = stage_samples(lambda c, s, ev: launch_layer(m, snapkv, c, s, ev), stream, side,
                                          2 * len(STAGES), n_diag, dev, 4)
    check_status(m, snapkv, "after the stage timing")

    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_per_step = elapsed_ms / args.steps
    heads = m.B * m.H
    units_per_step = m.B * m.L * m.H * m.n_layers
    value = whole_job_rate(units_per_step, world, ms_per_step)
    stage_med = {s: statistics.median(v) for s, v in samples.items()}
    stage_mean = {s: statistics.fmean(v) for s, v in samples.items()}
    alg = algorithmic_bytes(m.wl, m.ksel)
    peak, peak_kind = read_peaks()
    # A stage whose event pair holds no kernel (its work runs inside the previous stage's kernel)
    # reads only the event nodes' overhead: the tensor-core vote runs inside the score kernel, and
    # for prefixes the cluster top-k handles, the gather runs inside the top-k kernel.
    vote_fused = stage_med["vote"] < 0.1 * stage_med["score"]
    gather_fused = stage_med["gather"] < 0.25 * stage_med["topk"]
    sv_ms = stage_mean["score"] + (0.0 if vote_fused else stage_mean["vote"])
    tg_ms = stage_mean["topk"] + (0.0 if gather_fused else stage_mean["gather"])
    traffic, src_hash = profiled_traffic(VOTE_SOURCES)
    vote_bytes = alg["score+vote"] * heads
    achieved = vote_bytes / (sv_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "vote_tc_kernel (score + softmax + vote)", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": traffic, "alg_bytes_per_launch": vote_bytes, "avg_launch_ms": sv_ms,
                "units_per_launch": f"{heads} heads x (L_prompt + L_obs) rows x d x 2 B",
                "timing": "mean over the stage-timing replays (event-record nodes on the launching stream)"}
    compress_bytes = alg["compress"] * heads
    stage_gbs = {
        "score+vote": achieved,
        "topk+gather": alg["gather"] * heads / (tg_ms * 1e-3) / 1e9,
        "compress": compress_bytes / ((sv_ms + tg_ms) * 1e-3) / 1e9,
        "decode": alg["decode"] * heads / (stage_mean["decode"] * 1e-3) / 1e9,
    }

    e2e = e2e_prefill(torch, snapkv, m, dev, stream, 2, world)
    B, L, n_layers, ksel, cap = m.B, m.L, m.n_layers, m.ksel, m.cap
    del m
    torch.cuda.empty_cache()

    decode = None if args.no_decode else decode_leg(torch, snapkv, synth, dev, world, rank=rank,
                                                    local_rank=local_rank)
    if rank != 0:
        return
    extras = world == 1 and not args.no_extras
    single = single_layer_extra(torch, snapkv, synth, dev) if extras else None
    full_cache = full_cache_decode(torch, snapkv, synth, dev) if extras else None
    hit = hit_rate_diagnostic(torch, snapkv, synth, dev) if extras else None
    gqa = {"b1": gqa_compress(torch, snapkv, synth, dev, batch=1, copies=4),
           "b8": gqa_compress(torch, snapkv, synth, dev, batch=8, copies=2)} if extras else None
    varlen = varlen_compress(torch, snapkv, synth, dev) if extras else None
    long_ctx = long_context_compress(torch, snapkv, synth, dev) if extras else None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox inputs, per-channel key scales; no dataset or weights)",
        "config": {"workload": WORKLOAD_NAME, "global_batch": B * world, "seq_len": L, "layers": n_layers,
                   "heads": 32, "head_dim": 128, "l_obs": 32, "pool_kernel": 7, "ratio_p": 0.05, "kept": ksel,
                   "cap": cap, "parallelism": f"replicas x{world}",
                   "launch": "each step replayed as one CUDA graph: 32 x (compress + append/decode)",
                   "l2": "all 32 layers' inputs resident (64 GiB of K/V); each step reads every layer's keys "
                         "once, so no step finds them in L2 (inputs larger than L2, no flush)"},
        "decode_tok_s": decode["decode_tok_s"] if decode else None,
        "decode": decode,
        "compress_alg_gbs": stage_gbs["compress"],
        "hbm_gbs_algorithmic_step": alg["step"] * heads * n_layers / (ms_per_step * 1e-3) / 1e9,
        "stage_ms_mean_per_layer": {k: round(v, 5) for k, v in stage_mean.items()},
        "stage_ms_note": stage_method + ("; the vote runs inside the score kernel" if vote_fused else "") +
                         ("; the gather runs inside the top-k kernel" if gather_fused else ""),
        "stage_alg_gbs": {k: round(v, 1) for k, v in stage_gbs.items()},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * n_layers * 3,   # per layer: vote, top-k (+ gather), decode (+ append)
        "clocks": clocks,
        "wall_s_timed": wall,
        "kernel_source_sha256_16": src_hash,
        "single_layer": single,
        "full_cache_decode": full_cache,
        "hit_rate": hit,
        "gqa": gqa,
        "varlen": varlen,
        "long_context": long_ctx,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.case:
        run_case(args, local_rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
