"""MXFP8 dequantize on the GPU vs the oracle's decode (E4M3 value times the
E8M0 scale 2^(s-127), evaluated exactly in fp64): fp32 output bit-exact, bf16
output equal to the single round-to-nearest-even of the exact value.  Every
E4M3 code and every scale byte (0x00 = 2^-127, 0xFF = NaN), both scale
layouts, ragged shapes, batches, and a quantize -> dequantize round trip on
the full-size quantize workload."""
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


def _layout_scales(s_plain, layout):
    """[batch, rows, cols/32] plain scales -> the device array for `layout`."""
    if layout == 0:
        return s_plain.reshape(-1)
    return np.concatenate([mx.swizzle_scales(si) for si in s_plain])


def _expect(q, s_plain, out_dtype):
    """Exact fp64 values -> the fp32 or bf16 bit patterns the kernel must write."""
    v = mx.dequantize_rows(q, s_plain)
    if out_dtype == 1:
        with np.errstate(over="ignore"):
            return v.astype(np.float32)          # exact in fp32 (overflow -> inf)
    return mx.f64_to_bf16_bits(v)


def _compare(got, want, out_dtype, what):
    if out_dtype == 1:
        g, w = got.view(np.uint32), np.asarray(want, np.float32).view(np.uint32)
        gn, wn = np.isnan(got), np.isnan(want)
    else:
        g, w = got, want
        gn = ((g & 0x7FFF) > 0x7F80)
        wn = ((w & 0x7FFF) > 0x7F80)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    assert_bytes_equal(np.where(gn, 0, g), np.where(wn, 0, w), what)


def _run(dev, q, s_plain, layout, out_dtype):
    import mxfp8_mixture_experts_gb300 as m
    qd = torch.from_numpy(q).to(dev)
    sd = torch.from_numpy(_layout_scales(s_plain, layout)).to(dev)
    out = m.mx_dequantize(qd if q.shape[0] > 1 else qd[0], sd, layout, out_dtype)
    torch.cuda.synchronize()
    if out_dtype == 1:
        return out.cpu().numpy().reshape(q.shape)
    return bits(out).reshape(q.shape)


@pytest.mark.parametrize("shape", [(1, 32, 32), (1, 96, 160), (2, 130, 96), (3, 64, 2080), (1, 257, 4096)])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_dequantize_every_code_and_scale(dev, shape, layout, out_dtype):
    b, r, c = shape
    g = np.random.default_rng(r * 7 + c + b)
    q = g.integers(0, 256, size=shape, dtype=np.uint8)
    q.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)[: q.size]      # every E4M3 code
    s = g.integers(0, 256, size=(b, r, c // 32), dtype=np.uint8)
    s.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)[: s.size]      # every scale byte
    got = _run(dev, q, s, layout, out_dtype)
    _compare(got, _expect(q, s, out_dtype), out_dtype, f"dequantize {shape} layout={layout} out={out_dtype}")


def test_dequantize_extremes(dev):
    """Scale 0x00 (the fp32 subnormal 2^-127) on the smallest E4M3 subnormal
    (2^-9): 2^-136 exactly in fp32, 0 in bf16 (below half its smallest
    subnormal).  Scale 0xFE on 448: 448 * 2^127 overflows to +inf."""
    q = np.zeros((1, 32, 64), np.uint8)
    s = np.zeros((1, 32, 2), np.uint8)
    q[0, 0, 0] = 0x01
    q[0, 1, 32] = 0x7E
    s[0, 1, 1] = 0xFE
    for out_dtype in (0, 1):
        got = _run(dev, q, s, 0, out_dtype)
        _compare(got, _expect(q, s, out_dtype), out_dtype, f"extremes out={out_dtype}")
    got32 = _run(dev, q, s, 0, 1)
    assert got32[0, 0, 0] == np.float32(2.0 ** -136)
    assert np.isposinf(got32[0, 1, 32])


def test_quantize_dequantize_round_trip_full_size(dev):
    """The quantize workload (bf16 [16384, 7168], outliers and exact zeros):
    GPU quantize (ROW, swizzled) then GPU dequantize to bf16 and fp32; 512
    sampled rows against the oracle's decode of the GPU's own bytes, and the
    half-ulp bound of the E4M3 grid against the input."""
    import mxfp8_mixture_experts_gb300 as m
    R, C = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, C, seed=0, device=dev)
    qr, sr, _, _ = m.mx_quantize(x, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    out32 = m.mx_dequantize(qr, sr, m.MX_SCALE_SWIZZLED, m.MX_OUT_F32)
    out16 = m.mx_dequantize(qr, sr, m.MX_SCALE_SWIZZLED, m.MX_OUT_BF16)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(R, 512, replace=False))
    ri = torch.from_numpy(rows).to(dev)
    qh = u8(qr[ri])
    sf = u8(sr)
    rr, cc = np.meshgrid(rows, np.arange(C // 32), indexing="ij")
    s_plain = sf[mx.swizzled_offset(rr, cc, C // 32)]
    _compare(out32[ri].cpu().numpy(), _expect(qh[None], s_plain[None], 1)[0], 1, "fp32 round trip")
    _compare(bits(out16[ri]), _expect(qh[None], s_plain[None], 0)[0], 0, "bf16 round trip")
    # every non-saturated element within half an E4M3 step (times the scale) of the input
    xv = mx.bf16_to_f64(bits(x[ri]))
    v = out32[ri].cpu().numpy().astype(np.float64)
    step = mx.e4m3_ulp(qh) * np.repeat(mx.e8m0_decode(s_plain), 32, axis=1)
    sat = (qh & 0x7F) == 0x7E
    assert np.all(np.abs(v - xv)[~sat] <= 0.5 * step[~sat])
