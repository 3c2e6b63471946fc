"""MXFP8 quantize on the GPU vs the oracle: bit-exact bytes and scales, every
mode and layout, ragged tiles, special values, and the full-size workload
(bf16 [16384, 7168] with outliers and exact zeros) on sampled rows/columns."""
import numpy as np
import pytest
import torch

import workloads
from oracle import mx
from tests.helpers import assert_bytes_equal, bits, cuda_device, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _oracle(xb, mode, layout):
    x = mx.bf16_to_f64(xb)
    out = {}
    if mode & 1:
        q, s = mx.quantize_rows(x)
        out["row"] = (q, s if layout == 0 else np.concatenate([mx.swizzle_scales(si) for si in s.reshape(-1, *s.shape[-2:])]))
    if mode & 2:
        q, s = mx.quantize_cols(x)
        out["col"] = (q, s if layout == 0 else np.concatenate([mx.swizzle_scales(si) for si in s.reshape(-1, *s.shape[-2:])]))
    return out


def _check(xt, mode, layout):
    import mxfp8_mixture_experts_gb300 as m
    qr, sr, qc, sc = m.mx_quantize(xt, mode, layout)
    torch.cuda.synchronize()
    ref = _oracle(bits(xt), mode, layout)
    if mode & 1:
        assert_bytes_equal(u8(qr), ref["row"][0], "q_row")
        assert_bytes_equal(u8(sr).reshape(ref["row"][1].shape), ref["row"][1], "s_row")
    if mode & 2:
        assert_bytes_equal(u8(qc), ref["col"][0], "q_col")
        assert_bytes_equal(u8(sc).reshape(ref["col"][1].shape), ref["col"][1], "s_col")


@pytest.mark.parametrize("shape", [(32, 32), (64, 96), (160, 224), (160, 256), (96, 384), (256, 512),
                                   (384, 7168)])
@pytest.mark.parametrize("mode", [1, 2, 3])
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_matches_oracle(dev, shape, mode, layout):
    x = workloads.quantize_input(*shape, seed=sum(shape) + mode, device=dev)
    _check(x, mode, layout)


@pytest.mark.parametrize("shape", [(1, 64), (100, 96), (257, 160), (130, 7168)])
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_rows_ragged(dev, shape, layout):
    """ROW mode needs cols % 32 == 0 only: row counts off every tile and
    block boundary (the swizzled array's padding stays zero)."""
    x = workloads.quantize_input(*shape, seed=sum(shape), device=dev)
    _check(x, 1, layout)


@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_batched(dev, layout):
    g = workloads.generator(3, dev)
    x = workloads.randn_bf16((3, 128, 256), 1.0, g, dev)
    _check(x, 3, layout)


def test_quantize_unaligned_scale_pointers(dev):
    """Scale arrays need no alignment: outputs written through C-ABI pointers
    one byte past an aligned address match the oracle."""
    import ctypes
    import mxfp8_mixture_experts_gb300 as m
    R, Cc = 256, 512
    x = workloads.quantize_input(R, Cc, seed=11, device=dev)
    L = m.lib()
    nb = L.mx_scale_bytes(R, Cc, 1)
    nbc = L.mx_scale_bytes(Cc, R, 1)
    qr = torch.empty(R * Cc, dtype=torch.uint8, device=dev)
    qc = torch.empty(R * Cc, dtype=torch.uint8, device=dev)
    sr = torch.zeros(nb + 16, dtype=torch.uint8, device=dev)
    sc = torch.zeros(nbc + 16, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    code = L.mx_quantize(x.data_ptr(), 1, R, Cc, 3, 1, 0, qr.data_ptr(), sr.data_ptr() + 1, qc.data_ptr(),
                         sc.data_ptr() + 1, s)
    assert code == 0
    torch.cuda.synchronize()
    ref = _oracle(bits(x), 3, 1)
    assert_bytes_equal(u8(qr).reshape(ref["row"][0].shape), ref["row"][0], "q_row")
    assert_bytes_equal(u8(sr[1:nb + 1]), ref["row"][1].ravel(), "s_row")
    assert_bytes_equal(u8(qc).reshape(ref["col"][0].shape), ref["col"][0], "q_col")
    assert_bytes_equal(u8(sc[1:nbc + 1]), ref["col"][1].ravel(), "s_col")


def test_quantize_special_values(dev):
    g = np.random.default_rng(0)
    x = g.standard_normal((128, 256)).astype(np.float32)
    x[0, 0:32] = 0.0                      # all-zero block
    x[1, 0:32] = -0.0
    x[2, 5] = np.nan                      # NaN block
    x[3, 40] = np.inf                     # Inf block
    x[4, 70] = -np.inf
    x[5, 96:128] *= 2.0 ** -130           # bf16 subnormals
    x[6, 128:160] = 1.75                  # exactly 448 after scaling
    x[7, 160:192] = 1.9                   # saturates
    x[8, 192:224] *= 2.0 ** 100           # huge
    x[40:72, 300 % 256] = 0.0             # zero column block
    xt = torch.from_numpy(x).to(torch.bfloat16).to(dev)
    for layout in (0, 1):
        _check(xt, 3, layout)


def test_quantize_full_size_sampled(dev):
    """bf16 [16384, 7168], BOTH mode, swizzled scales: 512 sampled rows are
    checked whole (ROW) and 512 sampled columns whole (COL)."""
    import mxfp8_mixture_experts_gb300 as m
    R, Cc = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, Cc, seed=0, device=dev)
    qr, sr, qc, sc = m.mx_quantize(x, 3, 1)
    torch.cuda.synchronize()
    g = np.random.default_rng(1)
    rows = np.sort(g.choice(R, 512, replace=False))
    cols = np.sort(g.choice(Cc, 512, replace=False))
    xr = bits(x[torch.from_numpy(rows).to(dev)])
    q_ref, s_ref = mx.quantize_rows(mx.bf16_to_f64(xr))
    assert_bytes_equal(u8(qr[torch.from_numpy(rows).to(dev)]), q_ref, "q_row sample")
    srf = u8(sr)
    rr, cc = np.meshgrid(rows, np.arange(Cc // 32), indexing="ij")
    assert_bytes_equal(srf[mx.swizzled_offset(rr, cc, Cc // 32)], s_ref, "s_row sample")
    xc = bits(x[:, torch.from_numpy(cols).to(dev)])            # [R, 512]
    qc_ref, sc_ref = mx.quantize_cols(mx.bf16_to_f64(xc))      # [512, R]
    assert_bytes_equal(u8(qc[torch.from_numpy(cols).to(dev)]), qc_ref, "q_col sample")
    scf = u8(sc)
    rr, cc = np.meshgrid(cols, np.arange(R // 32), indexing="ij")
    assert_bytes_equal(scf[mx.swizzled_offset(rr, cc, R // 32)], sc_ref, "s_col sample")
    # every scale byte of the swizzled arrays is defined (no stale padding)
    assert sr.numel() == R * Cc // 32 and sc.numel() == R * Cc // 32
