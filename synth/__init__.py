"""Seeded synthetic inputs for SnapKV compression and compressed-cache decode.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and benchmark.
It holds none of the method's arithmetic: it only makes the inputs (queries, keys, values,
planted keys, per-channel key scales, ragged prompt lengths, decode-step tokens) from a
counter-based generator (Philox4x32-10) whose host (C) and device (CUDA) copies give
bit-identical values. See ``synth_gen.h`` for the element recipe.

The workloads follow the hyper-parameter presets of the SnapKV explainer ("論文解説: SnapKV",
section 実装のポイント, hyper-parameter table: L_obs 16/32/64, K_pool 5/7/13, 1024-4096 kept
slots per head) and the Llama-2-7B shape of the KV-cache chapter (section 22.4: 32 layers,
32 KV heads, head dimension 128, bf16). They stand in for the datasets and model activations
the pages measure on, which are not used here.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import build as _build

T_Q, T_K, T_V, T_SCALE, T_PLANT, T_LEN, T_QNEW, T_KNEW, T_VNEW = range(1, 10)

_HERE = os.path.dirname(os.path.abspath(__file__))
_host_lib = None
_dev_lib = None


def host_lib():
    global _host_lib
    if _host_lib is None:
        path = _build.host_lib_path()
        if not os.path.exists(path):
            _build.build_host()
        lib = ctypes.CDLL(path)
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.synth_chan_scales.restype = None
        lib.synth_chan_scales.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64]
        lib.synth_u32_stream.restype = None
        lib.synth_u32_stream.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                         ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                         ctypes.c_uint32]
        lib.synth_philox_block.restype = None
        lib.synth_philox_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_floyd.restype = ctypes.c_int
        lib.synth_floyd.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64,
                                    ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.c_uint32, ctypes.c_void_p]
        _host_lib = lib
    return _host_lib


def dev_lib():
    global _dev_lib
    if _dev_lib is None:
        path = _build.dev_lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"device generator library missing: {path} (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        lib.synth_fill_device.restype = ctypes.c_int
        lib.synth_fill_device.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
        _dev_lib = lib
    return _dev_lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox_block(ctr, key):
    """One raw Philox4x32-10 block (known-answer tests)."""
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    host_lib().synth_philox_block(_ptr(c), _ptr(k), _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to the fp32 values they encode (exact)."""
    pair = np.zeros(bits.shape + (2,), dtype=np.uint16)
    pair[..., 1 if np.little_endian else 0] = bits
    return pair.view(np.float32).reshape(bits.shape)


def fill_host(B, H, rows, d, *, row0, seq0, head0, layer, tensor, seed, bf16,
              chan_scale=None, plant_mask=None, plant_vec=None, threads=None):
    """Host copy of a generated [B, H, rows, d] tensor (uint16 bf16 bits or float32)."""
    out = np.empty((B, H, rows, d), dtype=np.uint16 if bf16 else np.float32)
    cs = None if chan_scale is None else np.ascontiguousarray(chan_scale, dtype=np.float32)
    pm = None if plant_mask is None else np.ascontiguousarray(plant_mask, dtype=np.uint8)
    pv = None if plant_vec is None else np.ascontiguousarray(plant_vec, dtype=np.float32)
    if threads is None:
        threads = min(32, os.cpu_count() or 1)
    rc = host_lib().synth_fill(_ptr(out), int(bf16), B, H, rows, d, row0, seq0, head0, layer, tensor,
                               seed, _ptr(cs), _ptr(pm), _ptr(pv), threads)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed ({rc})")
    return out


def fill_device(t, B, H, rows, d, *, row0, seq0, head0, layer, tensor, seed, bf16,
                chan_scale=None, plant_mask=None, plant_vec=None, stream=0):
    """Fill the contiguous torch tensor ``t`` ([B, H, rows, d]) on its GPU with the same values."""
    def p(x):
        return None if x is None else ctypes.c_void_p(x.data_ptr())
    rc = dev_lib().synth_fill_device(ctypes.c_void_p(t.data_ptr()), int(bf16), B, H, rows, d, row0,
                                     seq0, head0, layer, tensor, seed, p(chan_scale), p(plant_mask),
                                     p(plant_vec), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed ({rc})")


def chan_scales(B, H, d, *, seq0, layer, seed) -> np.ndarray:
    out = np.empty((B, H, d), dtype=np.float32)
    host_lib().synth_chan_scales(_ptr(out), B, H, d, seq0, layer, seed)
    return out


def u32_stream(n, *, seed, layer, seq, head, tensor) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    host_lib().synth_u32_stream(_ptr(out), n, seed, layer, seq, head, tensor)
    return out


def floyd_sample(n, m, *, seed, layer, seq, head, tensor=T_PLANT) -> np.ndarray:
    """m distinct integers from [0, n), ascending (Floyd's algorithm)."""
    out = np.empty(m, dtype=np.int32)
    scratch = np.empty(max(n, 1), dtype=np.uint8)
    rc = host_lib().synth_floyd(_ptr(out), n, m, seed, layer, seq, head, tensor, _ptr(scratch))
    if rc != 0:
        raise RuntimeError(f"synth_floyd failed ({rc})")
    return out


# ----------------------------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One synthetic SnapKV workload (shapes, hyper-parameters and input recipe)."""
    name: str
    ident: int
    bf16: bool
    batch: int
    heads: int
    head_dim: int
    layers: int
    l_prompt: int                      # uniform prompt length (0 when ragged)
    l_obs: int
    pool_kernel: int
    ratio_p: float = 0.0
    budget: int = 0                    # > 0: fixed number of kept prefix slots per head
    plants: int = 0                    # planted keys per head
    plant_scale: float = 0.0
    plant_run: int = 1                 # plants come in aligned runs of this many positions
    chan_scale: bool = False           # K = z * s_c with s_c ~ U(0.5, 2) per channel
    l_prompt_range: tuple = ()         # (lo, hi) inclusive, ragged prompts per sequence
    decode_steps: int = 0

    @property
    def seed(self) -> int:
        return 0x5EED0000 + self.ident

    @property
    def ragged(self) -> bool:
        return bool(self.l_prompt_range)

    def prompt_lengths(self) -> list:
        """Prompt length of every sequence (uniform, or drawn from U{lo..hi})."""
        if not self.ragged:
            return [self.l_prompt] * self.batch
        lo, hi = self.l_prompt_range
        draws = u32_stream(self.batch, seed=self.seed, layer=0, seq=0, head=0, tensor=T_LEN)
        span = hi - lo + 1
        return [lo + int((int(u) * span) >> 32) for u in draws]

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    0: Workload("tiny fp32 (1 layer, B1 H4 d64, L_prompt 1024, L_obs 32, K_pool 7, p 0.05)", 0,
                bf16=False, batch=1, heads=4, head_dim=64, layers=1, l_prompt=1024, l_obs=32,
                pool_kernel=7, ratio_p=0.05, plants=16, plant_scale=4.0),
    1: Workload("Llama-2-7B-shaped layer (B1 H32 d128 bf16, L_prompt 16384, L_obs 32, K_pool 7, budget 1024)",
                1, bf16=True, batch=1, heads=32, head_dim=128, layers=1, l_prompt=16384, l_obs=32,
                pool_kernel=7, budget=1024, plants=64, plant_scale=3.0),
    2: Workload("32-layer Llama-2-7B-shaped prefill (B8 H32 d128 bf16, L_prompt 16384, L_obs 32, K_pool 7, p 0.05)",
                2, bf16=True, batch=8, heads=32, head_dim=128, layers=32, l_prompt=16384, l_obs=32,
                pool_kernel=7, ratio_p=0.05, chan_scale=True),
    3: Workload("long context (B1 H32 d128 bf16, L_prompt 131072, L_obs 64, K_pool 13, budget 4096)",
                3, bf16=True, batch=1, heads=32, head_dim=128, layers=1, l_prompt=131072, l_obs=64,
                pool_kernel=13, budget=4096, plants=256, plant_scale=3.0, plant_run=8),
    4: Workload("compressed decode (B64 ragged L_prompt U{4096..32768}, 32 layers, H32 d128 bf16, "
                "L_obs 32, K_pool 7, budget 2048, 128 steps)", 4, bf16=True, batch=64, heads=32,
                head_dim=128, layers=32, l_prompt=0, l_obs=32, pool_kernel=7, budget=2048,
                l_prompt_range=(4096, 32768), decode_steps=128),
}


def _as_f32(raw: np.ndarray, bf16: bool) -> np.ndarray:
    return bf16_bits_to_f32(raw) if bf16 else raw


def plant_positions(wl: Workload, layer: int, seq: int, head: int, l_prefix: int) -> np.ndarray:
    """Planted prefix positions of one head (ascending)."""
    if wl.plants == 0:
        return np.zeros(0, dtype=np.int32)
    if wl.plant_run == 1:
        return floyd_sample(l_prefix, wl.plants, seed=wl.seed, layer=layer, seq=seq, head=head)
    # Runs: distinct aligned blocks of plant_run consecutive positions.
    blocks = floyd_sample(l_prefix // wl.plant_run, wl.plants // wl.plant_run, seed=wl.seed,
                          layer=layer, seq=seq, head=head)
    return (blocks[:, None] * wl.plant_run + np.arange(wl.plant_run)[None, :]).reshape(-1).astype(np.int32)


def plant_vector(wl: Workload, q_obs_f32: np.ndarray) -> np.ndarray:
    """scale * u_hat, u_hat = unit-normalised mean of the head's window queries (double, then fp32)."""
    mean = q_obs_f32.astype(np.float64).mean(axis=0)
    u_hat = mean / np.sqrt(np.dot(mean, mean))
    return (wl.plant_scale * u_hat).astype(np.float32)


@dataclass
class HeadInputs:
    """Host copy of one (layer, sequence, head): storage bits and exact fp32 values."""
    q_obs: np.ndarray      # [L_obs, d] float32 values
    k: np.ndarray          # [L_prompt, d]
    v: np.ndarray          # [L_prompt, d]
    l_prompt: int
    plants: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int32))


def host_head(wl: Workload, layer: int, seq: int, head: int, l_prompt: Optional[int] = None,
              threads: Optional[int] = None) -> HeadInputs:
    """Generate one head's inputs on the host (the oracle's inputs)."""
    L = l_prompt if l_prompt is not None else wl.prompt_lengths()[seq]
    d, lo = wl.head_dim, wl.l_obs
    l_prefix = L - lo
    common = dict(seq0=seq, head0=head, layer=layer, seed=wl.seed, bf16=wl.bf16, threads=threads)
    q_raw = fill_host(1, 1, lo, d, row0=l_prefix, tensor=T_Q, **common)
    q = _as_f32(q_raw, wl.bf16)[0, 0]
    cs = None
    if wl.chan_scale:
        cs = chan_scales(1, wl.heads, d, seq0=seq, layer=layer, seed=wl.seed)[:, head:head + 1]
    mask = vec = None
    plants = plant_positions(wl, layer, seq, head, l_prefix)
    if plants.size:
        mask = np.zeros((1, 1, L), dtype=np.uint8)
        mask[0, 0, plants] = 1
        vec = plant_vector(wl, q)[None, None, :]
    k_raw = fill_host(1, 1, L, d, row0=0, tensor=T_K, chan_scale=cs, plant_mask=mask,
                      plant_vec=vec, **common)
    v_raw = fill_host(1, 1, L, d, row0=0, tensor=T_V, **common)
    return HeadInputs(q_obs=q, k=_as_f32(k_raw, wl.bf16)[0, 0], v=_as_f32(v_raw, wl.bf16)[0, 0],
                      l_prompt=L, plants=plants)


def device_inputs(wl: Workload, layer: int, seq0: int, nseq: int, l_prompt: int, device, stream=0):
    """Generate q_obs [n,H,L_obs,d], k, v [n,H,L_prompt,d] for sequences seq0..seq0+n-1 on the GPU.

    The plant masks and vectors, and the channel scales, are made on the host (small) and copied.
    Returns (q_obs, k, v, plants) with plants a dict (seq, head) -> positions.
    """
    import torch
    H, d, lo = wl.heads, wl.head_dim, wl.l_obs
    l_prefix = l_prompt - lo
    dt = torch.bfloat16 if wl.bf16 else torch.float32
    q = torch.empty((nseq, H, lo, d), dtype=dt, device=device)
    k = torch.empty((nseq, H, l_prompt, d), dtype=dt, device=device)
    v = torch.empty((nseq, H, l_prompt, d), dtype=dt, device=device)
    common = dict(seq0=seq0, head0=0, layer=layer, seed=wl.seed, bf16=wl.bf16, stream=stream)
    fill_device(q, nseq, H, lo, d, row0=l_prefix, tensor=T_Q, **common)
    cs_dev = mask_dev = vec_dev = None
    plants = {}
    if wl.chan_scale:
        cs = chan_scales(nseq, H, d, seq0=seq0, layer=layer, seed=wl.seed)
        cs_dev = torch.from_numpy(cs).to(device)
    if wl.plants:
        q_host = _as_f32(fill_host(nseq, H, lo, d, row0=l_prefix, seq0=seq0, head0=0, layer=layer,
                                   tensor=T_Q, seed=wl.seed, bf16=wl.bf16), wl.bf16)
        mask = np.zeros((nseq, H, l_prompt), dtype=np.uint8)
        vec = np.zeros((nseq, H, d), dtype=np.float32)
        for b in range(nseq):
            for h in range(H):
                pos = plant_positions(wl, layer, seq0 + b, h, l_prefix)
                plants[(seq0 + b, h)] = pos
                mask[b, h, pos] = 1
                vec[b, h] = plant_vector(wl, q_host[b, h])
        mask_dev = torch.from_numpy(mask).to(device)
        vec_dev = torch.from_numpy(vec).to(device)
    fill_device(k, nseq, H, l_prompt, d, row0=0, tensor=T_K, chan_scale=cs_dev, plant_mask=mask_dev,
                plant_vec=vec_dev, **common)
    fill_device(v, nseq, H, l_prompt, d, row0=0, tensor=T_V, **common)
    return q, k, v, plants


def device_inputs_padded(wl: Workload, layer: int, seq0: int, lengths, device, l_pad: Optional[int] = None,
                         pad_value: float = float("nan"), stream=0):
    """Ragged prompts in one padded batch: q_obs [n,H,L_obs,d] and k, v [n,H,L_pad,d] where sequence
    seq0+b holds its own prompt (length lengths[b], identical to ``device_inputs`` of that sequence
    alone) in rows [0, lengths[b]) and ``pad_value`` in the rows after it."""
    import torch
    n = len(lengths)
    L_pad = l_pad if l_pad is not None else max(lengths)
    H, d, lo = wl.heads, wl.head_dim, wl.l_obs
    dt = torch.bfloat16 if wl.bf16 else torch.float32
    q = torch.empty((n, H, lo, d), dtype=dt, device=device)
    k = torch.full((n, H, L_pad, d), pad_value, dtype=dt, device=device)
    v = torch.full((n, H, L_pad, d), pad_value, dtype=dt, device=device)
    for b, L in enumerate(lengths):
        qb, kb, vb, _ = device_inputs(wl, layer, seq0 + b, 1, int(L), device, stream=stream)
        q[b].copy_(qb[0])
        k[b, :, :L].copy_(kb[0])
        v[b, :, :L].copy_(vb[0])
        del qb, kb, vb
    return q, k, v


def host_decode_token(wl: Workload, layer: int, seq: int, head: int, step: int):
    """(q, k, v) of decode step ``step`` for one head, as fp32 values [d]."""
    out = []
    for t in (T_QNEW, T_KNEW, T_VNEW):
        raw = fill_host(1, 1, 1, wl.head_dim, row0=step, seq0=seq, head0=head, layer=layer, tensor=t,
                        seed=wl.seed, bf16=wl.bf16, threads=1)
        out.append(_as_f32(raw, wl.bf16)[0, 0, 0])
    return tuple(out)


def device_decode_tokens(wl: Workload, layer: int, step: int, seq0: int, nseq: int, device, stream=0):
    """(q, k, v) [n, H, d] of decode step ``step`` for sequences seq0..seq0+n-1 on the GPU."""
    import torch
    dt = torch.bfloat16 if wl.bf16 else torch.float32
    outs = []
    for t in (T_QNEW, T_KNEW, T_VNEW):
        x = torch.empty((nseq, wl.heads, wl.head_dim), dtype=dt, device=device)
        fill_device(x, nseq, wl.heads, 1, wl.head_dim, row0=step, seq0=seq0, head0=0, layer=layer,
                    tensor=t, seed=wl.seed, bf16=wl.bf16, stream=stream)
        outs.append(x)
    return tuple(outs)


def device_decode_tokens_into(out, wl: Workload, layer: int, step: int, seq0: int, stream=0):
    """Fill ``out`` ([3, n, H, d], contiguous, on the GPU) with the (q, k, v) of decode step ``step``
    for sequences seq0..seq0+n-1: the values ``device_decode_tokens`` returns, written in place."""
    n = out.shape[1]
    for i, t in enumerate((T_QNEW, T_KNEW, T_VNEW)):
        fill_device(out[i], n, wl.heads, 1, wl.head_dim, row0=step, seq0=seq0, head0=0, layer=layer,
                    tensor=t, seed=wl.seed, bf16=wl.bf16, stream=stream)
