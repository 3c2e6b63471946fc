"""Shared helpers for the GPU parity tests: device setup, oracle-side
conversions between torch tensors and the oracle's numpy arrays, and the
comparison rules the tests use."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import mx


def cuda_device():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device (run CPU tests with -m 'not gpu')")
    from mxfp8_mixture_experts_gb300 import build
    build.build()
    import mxfp8_mixture_experts_gb300 as m
    m.lib()
    return torch.device("cuda:0")


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (numpy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().astype(np.uint8)


def to_dev_u8(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)


def to_dev_bf16(bits_: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits_, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(dev)


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} of {got.size} bytes differ; first at {bad[:5].tolist()}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def rel_frob(got: np.ndarray, ref: np.ndarray) -> float:
    d = np.linalg.norm(np.asarray(got, np.float64) - ref)
    n = np.linalg.norm(ref)
    return float(d / n) if n > 0 else float(d)


def assert_bf16_within_one_ulp(got_bits: np.ndarray, ref: np.ndarray, what: str, mag=None, K=None):
    """bf16 outputs of an fp32-accumulated product: the result must be the
    fp64 reference rounded to bf16, or one of its two neighbours (the fp32
    accumulation may land on the other side of a rounding midpoint).  With
    `mag` (sum of |a_k b_k| per element, fp64) and the contraction length K,
    an element more than one ulp off still passes when it is within the fp32
    accumulation bound K 2^-24 mag (plus one bf16 ulp of itself) of the
    reference: that bound exceeds a bf16 ulp of the result only where the
    terms nearly cancel, so the result is tiny next to them."""
    want = mx.f64_to_bf16_bits(ref).astype(np.int64)
    got = np.asarray(got_bits).astype(np.int64)
    # ordered integer view of bf16 bit patterns (sign-magnitude -> two's complement)
    def key(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    diff = np.abs(key(got) - key(want))
    bad_mask = diff > 1
    if mag is not None:
        gotv = mx.bf16_to_f64(np.asarray(got_bits))
        bound = K * 2.0 ** -24 * np.asarray(mag, np.float64) + 2.0 ** -8 * np.abs(gotv)
        bad_mask &= np.abs(gotv - np.asarray(ref, np.float64)) > bound
    bad = np.argwhere(bad_mask)
    assert bad.size == 0, f"{what}: {len(bad)} elements more than one bf16 ulp off; first {bad[:3].tolist()}"
    return float(np.mean(diff != 0))


def quant_mismatches_outside_margin(got_q, got_s, values, what, rel_margin=2e-6, max_frac=1e-3, fmt="e4m3"):
    """Row-quantized bytes of values that the GPU computed in fp32 and the
    oracle in fp64: they must match except where the fp64 value lies within
    ``rel_margin`` (relative) of an E4M3 rounding decision or the block amax
    lies that close to a power of two.  ``rel_margin`` is a number or an array
    of per-element bounds of the GPU's relative error (a block then takes the
    largest bound of its elements).  Returns the count of excused elements."""
    q_ref, s_ref = mx.quantize_rows(values, fmt)
    elem_rel, block_rel = mx.quantize_margins(values, fmt)
    rel_margin = np.asarray(rel_margin, np.float64)
    if rel_margin.ndim:
        # the computed amax can reach max_i |v_i| (1 + m_i): a small element
        # with a wide bound matters only if that reaches the block's amax
        av = np.abs(values).reshape(*values.shape[:-1], -1, mx.BLOCK)
        mm = rel_margin.reshape(av.shape)
        with np.errstate(invalid="ignore", over="ignore"):
            top = np.where(av > 0, av * (1 + mm), 0.0).max(axis=-1)
            amax = av.max(axis=-1)
            blk_margin = np.where(amax > 0, top / np.where(amax > 0, amax, 1.0) - 1.0, np.inf)
    else:
        blk_margin = rel_margin
    near_block = np.repeat(block_rel < blk_margin, mx.BLOCK, axis=-1).reshape(values.shape)
    excused = (elem_rel < rel_margin) | near_block
    bad = (np.asarray(got_q) != q_ref) & ~excused
    assert not bad.any(), f"{what}: {int(bad.sum())} bytes differ away from a rounding boundary; " \
                          f"first {np.argwhere(bad)[:3].tolist()}"
    sb = (np.asarray(got_s) != s_ref) & ~(block_rel < blk_margin)
    assert not sb.any(), f"{what}: {int(sb.sum())} scales differ away from a power of two"
    n_exc = int(((np.asarray(got_q) != q_ref) & excused).sum())
    assert n_exc <= max_frac * values.size, f"{what}: {n_exc} boundary mismatches is too many"
    return n_exc


# Bound on the relative error of the kernels' fp32 sigmoid(a) and 1 - sigmoid(a),
# in units of 2^-24, over bf16 a in [-128, 128] (asserted against an exact
# evaluation by test_gpu_swiglu_sweep.test_sigmoid_error_bound).
SIG_ULPS = 4


def swiglu_margins(dh, a, b):
    """Per-element bounds of the relative error of the kernels' fp32 SwiGLU
    values, from the sigmoid bound and the roundings that follow it:
      h  = ((a s) b) back            three roundings after sigma
      db = (dh (a s)) back           three roundings after sigma
      da = (((dh b) s) w) back, w = 1 + a (1 - sigma): the error of
           a (1 - sigma) enters w as an absolute error, relative to w (large
           where w cancels, near a = -1.28)
    plus, for roundings that land among the fp32 subnormals (absolute error
    2^-150 each), 2^-149 times one plus the factor applied after the first of
    them (a tiny a makes a s subnormal before the product with b or dh).
    Returns (m_h, m_da, m_db) as relative bounds."""
    u = 2.0 ** -24
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    dh = np.asarray(dh, np.float64)
    from oracle import moe
    sig = moe.sigmoid(a)
    oms = moe.sigmoid(-a)
    d_sig = SIG_ULPS * u
    h = a * sig * b
    db = dh * a * sig
    uu = a * oms
    w = 1.0 + uu
    da = dh * b * sig * w
    tiny = 2.0 ** -149
    with np.errstate(divide="ignore", invalid="ignore"):
        m_h = d_sig + 3 * u + tiny * (1 + np.abs(b)) / np.abs(h)
        m_db = d_sig + 3 * u + tiny * (1 + np.abs(dh)) / np.abs(db)
        m_da = d_sig + 4 * u + (np.abs(uu) * (d_sig + 2 * u) + u) / np.abs(w) + tiny * (1 + np.abs(w)) / np.abs(da)
    return (np.nan_to_num(m_h, nan=np.inf), np.nan_to_num(m_da, nan=np.inf), np.nan_to_num(m_db, nan=np.inf))
