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


def assert_bf16_within_one_ulp(got_bits: np.ndarray, ref: np.ndarray, what: str):
    """bf16 outputs of an fp32-accumulated product: the result must be the
    fp64 reference rounded to bf16, or one of its two neighbours (the fp32
    accumulation may land on the other side of a rounding midpoint)."""
    want = mx.f64_to_bf16_bits(ref).astype(np.int64)
    got = np.asarray(got_bits).astype(np.int64)
    # ordered integer view of bf16 bit patterns (sign-magnitude -> two's complement)
    def key(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    diff = np.abs(key(got) - key(want))
    bad = np.argwhere(diff > 1)
    assert bad.size == 0, f"{what}: {len(bad)} elements more than one bf16 ulp off; first {bad[:3].tolist()}"
    return float(np.mean(diff != 0))


def quant_mismatches_outside_margin(got_q, got_s, values, what, rel_margin=2e-6, max_frac=1e-3):
    """Row-quantized bytes of values that the GPU computed in fp32 and the
    oracle in fp64: they must match except where the fp64 value lies within
    ``rel_margin`` (relative) of an E4M3 rounding decision or the block amax
    lies that close to a power of two.  Returns the count of excused elements."""
    q_ref, s_ref = mx.quantize_rows(values)
    elem_rel, block_rel = mx.quantize_margins(values)
    near_block = np.repeat(block_rel < rel_margin, mx.BLOCK, axis=-1).reshape(values.shape)
    excused = (elem_rel < rel_margin) | near_block
    bad = (np.asarray(got_q) != q_ref) & ~excused
    assert not bad.any(), f"{what}: {int(bad.sum())} bytes differ away from a rounding boundary; " \
                          f"first {np.argwhere(bad)[:3].tolist()}"
    sb = (np.asarray(got_s) != s_ref) & ~(block_rel < rel_margin)
    assert not sb.any(), f"{what}: {int(sb.sum())} scales differ away from a power of two"
    n_exc = int(((np.asarray(got_q) != q_ref) & excused).sum())
    assert n_exc <= max_frac * values.size, f"{what}: {n_exc} boundary mismatches is too many"
    return n_exc
