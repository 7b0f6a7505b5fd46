"""Python binding of libsnapkv.so (ctypes). Argument marshalling only.

Every computation runs in the library's CUDA kernels; this module only turns torch tensors into
device pointers and a stream handle, allocates outputs and workspaces with torch when the caller
does not pass them, and raises on a non-OK status. There is no CPU or PyTorch fallback: if the
library is missing the import of the first call fails.

The functions and their arguments mirror include/snapkv.h (see that header for the layouts and
the passages of the pages each operation follows).
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
# SNAPKV_CHECKED=1 selects the bounds-checked build (kv_cache_compression_gb300.build.build(checked=True)).
_LIB_PATH = os.path.join(_HERE, "libsnapkv_checked.so" if os.environ.get("SNAPKV_CHECKED") == "1" else "libsnapkv.so")
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "snapkv.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_INTERNAL = (
    0, 1, 2, 4, 8, 16, 32, 64)
F32, BF16 = 0, 1
SCOPE_PROMPT_CAUSAL, SCOPE_PREFIX_ONLY = 0, 1
ALGO_AUTO, ALGO_SIMT, ALGO_TENSOR_CORE, ALGO_TENSOR_CORE_CLUSTER = 0, 1, 2, 3
_ALGOS = {"auto": ALGO_AUTO, "simt": ALGO_SIMT, "tensor_core": ALGO_TENSOR_CORE,
          "tensor_core_cluster": ALGO_TENSOR_CORE_CLUSTER}
_SCOPES = {"prompt_causal": SCOPE_PROMPT_CAUSAL, "prefix_only": SCOPE_PREFIX_ONLY}


class CompressParams(ctypes.Structure):
    """Mirror of snapkv_compress_params."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("l_obs", ctypes.c_int32), ("l_prompt", ctypes.c_int64), ("pool_kernel", ctypes.c_int32),
        ("softmax_scope", ctypes.c_int32), ("ratio_p", ctypes.c_double), ("budget", ctypes.c_int64),
        ("dtype", ctypes.c_int32), ("algo", ctypes.c_int32),
    ]


class SnapKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libsnapkv.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback path)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        PP = ctypes.POINTER(CompressParams)
        L.snapkv_compress_kept.restype = I64
        L.snapkv_compress_kept.argtypes = [PP]
        L.snapkv_compress_k.restype = I64
        L.snapkv_compress_k.argtypes = [PP]
        L.snapkv_compress_workspace_size.restype = SZ
        L.snapkv_compress_workspace_size.argtypes = [PP]
        L.snapkv_compress.restype = I32
        L.snapkv_compress.argtypes = [PP, P, P, P, P, P, I64, P, P, P, P, SZ, P, P]
        L.snapkv_compress_profiled.restype = I32
        L.snapkv_compress_profiled.argtypes = [PP, P, P, P, P, P, I64, P, P, P, P, SZ, P, P, P, I32]
        L.snapkv_append.restype = I32
        L.snapkv_append.argtypes = [P, P, P, P, I64, P, I32, I32, I32, I32, P, P]
        L.snapkv_decode_workspace_size.restype = SZ
        L.snapkv_decode_workspace_size.argtypes = [I32, I32, I32, I64]
        L.snapkv_decode_attend.restype = I32
        L.snapkv_decode_attend.argtypes = [P, P, P, I64, P, P, I32, I32, I32, I32, P, SZ, P, P]
        L.snapkv_append_decode_attend.restype = I32
        L.snapkv_append_decode_attend.argtypes = [P, P, P, P, P, I64, P, P, P, I32, I32, I32, I32, P, SZ, P, P]
        L.snapkv_decode_attend_noalloc.restype = I32
        L.snapkv_decode_attend_noalloc.argtypes = [P, P, P, I64, P, P, I32, I32, I32, I32, P, P]
        L.snapkv_compress_gqa_workspace_size.restype = SZ
        L.snapkv_compress_gqa_workspace_size.argtypes = [PP, I32]
        L.snapkv_compress_gqa.restype = I32
        L.snapkv_compress_gqa.argtypes = [PP, I32, P, P, P, P, P, I64, P, P, P, P, SZ, P, P]
        L.snapkv_compress_varlen_workspace_size.restype = SZ
        L.snapkv_compress_varlen_workspace_size.argtypes = [PP, P]
        L.snapkv_compress_varlen.restype = I32
        L.snapkv_compress_varlen.argtypes = [PP, P, P, P, P, P, P, I64, P, P, P, P, SZ, P, P]
        L.snapkv_hit_rate.restype = I32
        L.snapkv_hit_rate.argtypes = [P, P, I64, P, I64, P, I64, I32, I32, I32, I32, ctypes.c_double, P, P, P, P]
        L.snapkv_status_string.restype = ctypes.c_char_p
        L.snapkv_status_string.argtypes = [I32]
        L.snapkv_abi_version.restype = I32
        L.snapkv_abi_version.argtypes = []
        _lib = L
    return _lib


def declared_functions() -> list:
    """Names of the functions include/snapkv.h declares."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(snapkv_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib().snapkv_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> Optional[ctypes.c_void_p]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def make_params(*, batch, heads, head_dim, l_obs, l_prompt, pool_kernel, ratio_p=0.0, budget=0,
                scope="prompt_causal", dtype=BF16, algo="auto") -> CompressParams:
    return CompressParams(batch, heads, head_dim, l_obs, l_prompt, pool_kernel, _SCOPES[scope],
                          float(ratio_p), int(budget), dtype, _ALGOS[algo])


def kept(params: CompressParams) -> int:
    return int(lib().snapkv_compress_kept(ctypes.byref(params)))


def compress_k(params: CompressParams) -> int:
    return int(lib().snapkv_compress_k(ctypes.byref(params)))


def compress_workspace_size(params: CompressParams, q_heads=None) -> int:
    if q_heads is None or q_heads == params.heads:
        return int(lib().snapkv_compress_workspace_size(ctypes.byref(params)))
    return int(lib().snapkv_compress_gqa_workspace_size(ctypes.byref(params), int(q_heads)))


def decode_workspace_size(batch, heads, head_dim, cap) -> int:
    return int(lib().snapkv_decode_workspace_size(batch, heads, head_dim, cap))


def new_workspace(nbytes: int, device):
    """A workspace buffer (scratch: the library needs no particular contents on entry)."""
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def compress(q_obs, k, v, *, pool_kernel, ratio_p=0.0, budget=0, scope="prompt_causal", algo="auto", cap=None,
             k_out=None, v_out=None, len_out=None, idx_out=None, vote_out=None, want_idx=True,
             want_vote=False, workspace=None, dev_status=None, stream=None):
    """snapkv_compress on torch tensors q_obs [B,Hq,L_obs,d], k, v [B,H,L_prompt,d].

    Hq > H (a multiple of H) is grouped-query attention (snapkv_compress_gqa): the Hq / H query
    heads of each KV head vote together. ``v`` may be a pinned CPU tensor: only its kept and window
    rows are read, over the host link. Returns a dict with k_out, v_out ([B,H,cap,d]), len_out
    [B], idx [B,H,k] (if wanted) and vote [B,H,L_prefix] (if wanted), plus k (kept slots) and the
    workspace used.
    """
    import torch
    B, H, L, d = k.shape
    l_obs = q_obs.shape[2]
    q_heads = q_obs.shape[1]
    params = make_params(batch=B, heads=H, head_dim=d, l_obs=l_obs, l_prompt=L, pool_kernel=pool_kernel,
                         ratio_p=ratio_p, budget=budget, scope=scope, dtype=_dtype_code(k), algo=algo)
    ksel = kept(params)
    if ksel < 0:
        raise SnapKVError(ERR_INVALID_ARG, "snapkv_compress_kept")
    if cap is None:
        cap = ksel + l_obs
    dev = k.device
    if k_out is None:
        k_out = torch.empty((B, H, cap, d), dtype=k.dtype, device=dev)
    if v_out is None:
        v_out = torch.empty((B, H, cap, d), dtype=k.dtype, device=dev)
    if len_out is None:
        len_out = torch.empty((B,), dtype=torch.int32, device=dev)
    if idx_out is None and want_idx:
        idx_out = torch.empty((B, H, max(ksel, 0)), dtype=torch.int32, device=dev)
    if vote_out is None and want_vote:
        vote_out = torch.empty((B, H, L - l_obs), dtype=torch.float32, device=dev)
    need = compress_workspace_size(params, q_heads)
    if workspace is None:
        workspace = new_workspace(need, dev)
    for t in (q_obs, k, v, k_out, v_out):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    ws_bytes = workspace.numel() * workspace.element_size()
    if q_heads == H:
        st = lib().snapkv_compress(ctypes.byref(params), _ptr(q_obs), _ptr(k), _ptr(v), _ptr(k_out), _ptr(v_out),
                                   int(cap), _ptr(len_out), _ptr(idx_out) if ksel > 0 else None, _ptr(vote_out),
                                   _ptr(workspace), ws_bytes, _ptr(dev_status), _stream_handle(stream))
    else:
        st = lib().snapkv_compress_gqa(ctypes.byref(params), int(q_heads), _ptr(q_obs), _ptr(k), _ptr(v),
                                       _ptr(k_out), _ptr(v_out), int(cap), _ptr(len_out),
                                       _ptr(idx_out) if ksel > 0 else None, _ptr(vote_out), _ptr(workspace),
                                       ws_bytes, _ptr(dev_status), _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_compress" if q_heads == H else "snapkv_compress_gqa")
    return {"k_out": k_out, "v_out": v_out, "len": len_out, "idx": idx_out, "vote": vote_out, "k": ksel,
            "workspace": workspace, "cap": cap}


def compress_varlen(q_obs, k, v, l_prompts, *, pool_kernel, ratio_p=0.0, budget=0, scope="prompt_causal",
                    algo="auto", cap=None, want_idx=True, want_vote=False, workspace=None, dev_status=None,
                    stream=None, out=None, k_out=None, v_out=None, len_out=None):
    """snapkv_compress_varlen: q_obs [B,H,L_obs,d]; k, v [B,H,L_max,d] padded, sequence b using its
    first l_prompts[b] rows (``v`` may be a pinned CPU tensor, as for compress). Returns k_out, v_out
    [B,H,cap,d], len [B], idx [B,H,k_max] (row b, h
    holds k_b indices), vote [B,H,L_max-L_obs] (if wanted), ks (per-sequence k) and the workspace.
    ``out``: a previous call's result whose buffers (outputs and workspace) this call writes again.
    ``k_out``, ``v_out`` (contiguous [B,H,cap,d]) and ``len_out`` [B]: caller-owned outputs, e.g. a
    slice of a larger cache (cap is then their third dimension)."""
    import numpy as np
    import torch
    B, H, L, d = k.shape
    l_obs = q_obs.shape[2]
    lens = np.ascontiguousarray(np.asarray(l_prompts, dtype=np.int64))
    if lens.shape != (B,):
        raise ValueError("one prompt length per sequence")
    params = make_params(batch=B, heads=H, head_dim=d, l_obs=l_obs, l_prompt=L, pool_kernel=pool_kernel,
                         ratio_p=ratio_p, budget=budget, scope=scope, dtype=_dtype_code(k), algo=algo)
    k_max = kept(params)
    ks = []
    for n in lens:
        pb = make_params(batch=1, heads=H, head_dim=d, l_obs=l_obs, l_prompt=int(n), pool_kernel=pool_kernel,
                         ratio_p=ratio_p, budget=budget, scope=scope, dtype=_dtype_code(k), algo=algo)
        ks.append(kept(pb))
    dev = k.device
    if out is not None:
        cap, k_out, v_out, len_out, idx_out, vote_out = (out["cap"], out["k_out"], out["v_out"], out["len"],
                                                        out["idx"], out["vote"])
        workspace = out["workspace"] if workspace is None else workspace
    else:
        if k_out is not None:
            cap = k_out.shape[2]
        if cap is None:
            cap = k_max + l_obs
        if k_out is None:
            k_out = torch.empty((B, H, cap, d), dtype=k.dtype, device=dev)
        if v_out is None:
            v_out = torch.empty_like(k_out)
        if len_out is None:
            len_out = torch.empty((B,), dtype=torch.int32, device=dev)
        for t in (k_out, v_out, len_out):
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
        idx_out = torch.full((B, H, max(k_max, 1)), -1, dtype=torch.int32, device=dev) if want_idx else None
        vote_out = torch.zeros((B, H, L - l_obs), dtype=torch.float32, device=dev) if want_vote else None
    need = int(lib().snapkv_compress_varlen_workspace_size(ctypes.byref(params), lens.ctypes.data_as(ctypes.c_void_p)))
    if need == 0:
        raise SnapKVError(ERR_INVALID_ARG, "snapkv_compress_varlen_workspace_size")
    if workspace is None:
        workspace = new_workspace(need, dev)
    for t in (q_obs, k, v):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    st = lib().snapkv_compress_varlen(ctypes.byref(params), lens.ctypes.data_as(ctypes.c_void_p), _ptr(q_obs),
                                      _ptr(k), _ptr(v), _ptr(k_out), _ptr(v_out), int(cap), _ptr(len_out),
                                      _ptr(idx_out), _ptr(vote_out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                      _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_compress_varlen")
    return {"k_out": k_out, "v_out": v_out, "len": len_out, "idx": idx_out, "vote": vote_out, "ks": ks,
            "k_max": k_max, "workspace": workspace, "cap": cap}


def append(k_new, v_new, k_cache, v_cache, len_, *, dev_status=None, stream=None):
    """snapkv_append: k_new, v_new [B,H,d] into k_cache, v_cache [B,H,cap,d] at row len[b]; len += 1."""
    B, H, cap, d = k_cache.shape
    st = lib().snapkv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), int(cap), _ptr(len_), B, H,
                             d, _dtype_code(k_cache), _ptr(dev_status), _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_append")


def hit_rate(q, k_cache, len_, idx, l_prefix, *, theta=0.05, dev_status=None, stream=None):
    """snapkv_hit_rate: per (sequence, head) counts (hits, total) of the explainer's hit rate, for
    the query q [B,H,d] over the uncompressed cache k_cache [B,H,cap,d] (len rows) and the kept
    prefix positions idx [B,H,k]. H = hits.sum() / total.sum()."""
    import torch
    B, H, cap, d = k_cache.shape
    hits = torch.empty((B, H), dtype=torch.int32, device=k_cache.device)
    total = torch.empty((B, H), dtype=torch.int32, device=k_cache.device)
    k = int(idx.shape[-1])
    st = lib().snapkv_hit_rate(_ptr(q), _ptr(k_cache), int(cap), _ptr(len_), int(l_prefix), _ptr(idx), k, B, H, d,
                               _dtype_code(k_cache), float(theta), _ptr(hits), _ptr(total), _ptr(dev_status),
                               _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_hit_rate")
    return hits, total


def decode_attend(q, k_cache, v_cache, len_, *, out=None, workspace=None, dev_status=None, stream=None):
    """snapkv_decode_attend: q [B,H,d] over rows < len[b] of k_cache, v_cache [B,H,cap,d] -> out [B,H,d]."""
    import torch
    B, H, cap, d = k_cache.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=k_cache.dtype, device=k_cache.device)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(B, H, d, cap), k_cache.device)
    st = lib().snapkv_decode_attend(_ptr(q), _ptr(k_cache), _ptr(v_cache), int(cap), _ptr(len_), _ptr(out), B, H,
                                    d, _dtype_code(k_cache), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                    _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_decode_attend")
    return out


def append_decode_attend(q, k_new, v_new, k_cache, v_cache, len_in, len_out=None, *, out=None, workspace=None,
                         dev_status=None, stream=None):
    """snapkv_append_decode_attend: append k_new, v_new [B,H,d] at row len_in[b], then attend with q [B,H,d]
    over the len_in[b] + 1 rows. Returns (out [B,H,d], len_out [B]); len_out must not be len_in."""
    import torch
    B, H, cap, d = k_cache.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=k_cache.dtype, device=k_cache.device)
    if len_out is None:
        len_out = torch.empty_like(len_in)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(B, H, d, cap), k_cache.device)
    st = lib().snapkv_append_decode_attend(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                           int(cap), _ptr(len_in), _ptr(len_out), _ptr(out), B, H, d,
                                           _dtype_code(k_cache), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                           _stream_handle(stream))
    if st != OK:
        raise SnapKVError(st, "snapkv_append_decode_attend")
    return out, len_out
