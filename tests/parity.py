"""Acceptance rules for comparing the CUDA path with the CPU oracle (shared by the GPU tests).

  * vote C:     |C_gpu - C_ref| <= 1e-4 |C_ref| + 1e-30 (fp32 on the GPU, float64 in the oracle)
  * indices:    equal as sets, except positions whose oracle pooled score lies within 1e-5
                relative of the oracle's k-th value tau (a top-k boundary the fp32 rounding may
                flip); such positions are counted and returned, never silently dropped
  * K_c, V_c:   bit-exact: row r < k equals the input row the GPU says it kept, and the window
                rows equal the input's last L_obs rows
  * decode out: |o_gpu - o_ref| <= 2e-3 + half a bf16 ulp of |o_ref| when the output is bf16
                (the output's own storage rounding), <= 2e-3 when it is fp32
"""
from dataclasses import dataclass

import numpy as np

VOTE_RTOL = 1e-4
VOTE_ATOL = 1e-30
BOUNDARY_RTOL = 1e-5
DECODE_ATOL = 2e-3


@dataclass
class HeadReport:
    excused: int          # indices in the symmetric difference, all within the boundary band
    vote_max_rel: float


def check_compress_head(*, gpu_idx, gpu_kc, gpu_vc, gpu_vote, ref, k_in, v_in, l_prefix, l_obs, where=""):
    """Compare one head; raises AssertionError with a description on failure."""
    ksel = ref.idx.shape[0]
    if gpu_vote is not None:
        err = np.abs(gpu_vote.astype(np.float64) - ref.c)
        bad = err > VOTE_RTOL * np.abs(ref.c) + VOTE_ATOL
        assert not bad.any(), (f"{where}: vote off at {np.nonzero(bad)[0][:8]} "
                               f"(gpu {gpu_vote[bad][:4]}, ref {ref.c[bad][:4]})")
        rel = float((err / np.maximum(np.abs(ref.c), 1e-30)).max()) if err.size else 0.0
    else:
        rel = float("nan")
    gi = np.asarray(gpu_idx, dtype=np.int64)
    assert gi.shape == (ksel,), f"{where}: {gi.shape} indices, expected {ksel}"
    assert ksel == 0 or (np.all(np.diff(gi) > 0) and gi[0] >= 0 and gi[-1] < l_prefix), f"{where}: indices not ascending/in range"
    sym = np.setxor1d(gi, ref.idx)
    if sym.size:
        band = np.abs(ref.p[sym] - ref.tau) <= BOUNDARY_RTOL * abs(ref.tau)
        assert band.all(), (f"{where}: {int((~band).sum())} index differences away from the top-k boundary, "
                            f"e.g. {sym[~band][:6]} (P_ref {ref.p[sym[~band]][:3]}, tau {ref.tau})")
    # gathered rows: bit-exact against the input rows the GPU kept, window appended verbatim
    assert np.array_equal(gpu_kc[:ksel], k_in[gi]), f"{where}: gathered K rows differ"
    assert np.array_equal(gpu_vc[:ksel], v_in[gi]), f"{where}: gathered V rows differ"
    assert np.array_equal(gpu_kc[ksel:ksel + l_obs], k_in[l_prefix:]), f"{where}: window K rows differ"
    assert np.array_equal(gpu_vc[ksel:ksel + l_obs], v_in[l_prefix:]), f"{where}: window V rows differ"
    return HeadReport(excused=int(sym.size), vote_max_rel=rel)


def decode_tolerance(o_ref, bf16: bool):
    o_ref = np.asarray(o_ref, dtype=np.float64)
    if not bf16:
        return np.full(o_ref.shape, DECODE_ATOL)
    return DECODE_ATOL + np.abs(o_ref) * 2.0 ** -8


def check_decode(o_gpu, o_ref, bf16: bool, where=""):
    err = np.abs(np.asarray(o_gpu, dtype=np.float64) - o_ref)
    tol = decode_tolerance(o_ref, bf16)
    assert (err <= tol).all(), f"{where}: decode max err {err.max():.3e} (worst tol {tol[err.argmax()]:.3e})"
    return float(err.max())


def to_numpy_f32(t):
    """A torch tensor (bf16 or fp32, any device) as float32 numpy values."""
    import torch
    return t.detach().to("cpu").to(torch.float32).numpy()


# Canary guard bands: output buffers are pre-filled with a NaN bit pattern that no kernel writes, so
# that every row, index or vote entry the library promises to leave untouched can be checked after
# the call (rows past k + L_obs of the cache, indices past a sequence's own k, votes past its own
# L_prefix).
CANARY_BF16 = 0x7FC1            # bf16 quiet NaN with a payload
CANARY_F32 = 0x7FC00BAD         # fp32 quiet NaN with a payload
CANARY_I32 = -0x5EED


def canary_like(shape, dtype, device):
    """A tensor of `shape` and `dtype` (bf16, fp32 or int32) filled with the canary bit pattern."""
    import torch
    if dtype == torch.bfloat16:
        return torch.full(shape, CANARY_BF16, dtype=torch.int16, device=device).view(torch.bfloat16)
    if dtype == torch.float32:
        return torch.full(shape, CANARY_F32, dtype=torch.int32, device=device).view(torch.float32)
    if dtype == torch.int32:
        return torch.full(shape, CANARY_I32, dtype=torch.int32, device=device)
    raise TypeError(dtype)


def assert_canary(t, where=""):
    """Every element of `t` still holds the canary bit pattern."""
    import torch
    if t.numel() == 0:
        return
    if t.dtype == torch.bfloat16:
        ok = bool((t.view(torch.int16) == CANARY_BF16).all())
    elif t.dtype == torch.float32:
        ok = bool((t.view(torch.int32) == CANARY_F32).all())
    else:
        ok = bool((t == CANARY_I32).all())
    assert ok, f"{where}: an element the call must leave untouched was written"


def bf16_bits(t):
    """A bf16 torch tensor's bit patterns as a uint16 numpy array (host)."""
    import torch
    return t.detach().contiguous().view(torch.int16).to("cpu").numpy().view(np.uint16)
