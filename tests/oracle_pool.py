"""The oracle side of the large GPU parity cases, run in spawned worker processes.

Each job carries what the GPU produced for one (layer, sequence, head) — indices, the compressed
rows as bf16 bit patterns, the vote, and for the decode workload every step's output — and the
worker regenerates that head's inputs on the host, runs the CPU oracle and applies the acceptance
rules of ``tests.parity``. Workers are started with ``spawn`` (never forked from a process that
holds a CUDA context) and use one BLAS thread each.
"""
from __future__ import annotations

import atexit
import multiprocessing as mp
import os
import traceback

import numpy as np

_pool = None


def pool():
    global _pool
    if _pool is None:
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            n = max(1, min(16, os.cpu_count() or 1))
            _pool = mp.get_context("spawn").Pool(n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        atexit.register(_pool.terminate)
    return _pool


def run(fn, jobs):
    """fn over jobs in the workers; returns the results in order."""
    return pool().map(fn, jobs, chunksize=1)


def _bits_to_f32(bits):
    import synth
    return synth.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16))


def check_compress_job(job):
    """One head of a compression call: returns (where, excused, error or None)."""
    import synth
    from oracle import snapkv_oracle as orc
    from tests.parity import check_compress_head
    where = job["where"]
    try:
        wl = job["wl"]
        hi = synth.host_head(wl, job["layer"], job["seq"], job["head"], l_prompt=job["l_prompt"], threads=1)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p,
                                budget=wl.budget, scope=job.get("scope", orc.PROMPT_CAUSAL))
        kc = _bits_to_f32(job["kc_bits"]) if wl.bf16 else job["kc"]
        vc = _bits_to_f32(job["vc_bits"]) if wl.bf16 else job["vc"]
        rep = check_compress_head(gpu_idx=job["idx"], gpu_kc=kc, gpu_vc=vc, gpu_vote=job.get("vote"), ref=ref,
                                  k_in=hi.k, v_in=hi.v, l_prefix=job["l_prompt"] - wl.l_obs, l_obs=wl.l_obs,
                                  where=where)
        return where, rep.excused, None
    except AssertionError as e:
        return where, None, str(e)
    except Exception:
        return where, None, traceback.format_exc()


def check_decode_run_job(job):
    """One (sequence, layer, head) of the decode workload: its compression, then every decode step's
    output against the oracle's decode over the GPU's compressed rows plus the appended tokens."""
    import synth
    from oracle import snapkv_oracle as orc
    from tests.parity import check_compress_head, check_decode
    where = job["where"]
    try:
        wl = job["wl"]
        layer, seq, head, L = job["layer"], job["seq"], job["head"], job["l_prompt"]
        hi = synth.host_head(wl, layer, seq, head, l_prompt=L, threads=1)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, budget=wl.budget)
        l_prefix = L - wl.l_obs
        kc = _bits_to_f32(job["kc_bits"])
        vc = _bits_to_f32(job["vc_bits"])
        rep = check_compress_head(gpu_idx=job["idx"], gpu_kc=kc, gpu_vc=vc, gpu_vote=None, ref=ref, k_in=hi.k,
                                  v_in=hi.v, l_prefix=l_prefix, l_obs=wl.l_obs, where=where)
        # decode over the rows the GPU kept (bit-exact input rows, checked above)
        k_cache = orc.gather_with_window(hi.k, job["idx"], l_prefix)
        v_cache = orc.gather_with_window(hi.v, job["idx"], l_prefix)
        outs = _bits_to_f32(job["out_bits"])
        worst = 0.0
        for t in range(outs.shape[0]):
            qn, kn, vn = synth.host_decode_token(wl, layer, seq, head, t)
            k_cache, v_cache = orc.append(k_cache, v_cache, kn, vn)
            worst = max(worst, check_decode(outs[t], orc.decode_attend(qn, k_cache, v_cache), True,
                                            where=f"{where} step {t}"))
        return where, (rep.excused, worst), None
    except AssertionError as e:
        return where, None, str(e)
    except Exception:
        return where, None, traceback.format_exc()

