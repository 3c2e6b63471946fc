"""Row-max-scaled FP8 (fp8_quantize_rowmax) on the GPU vs the oracle: bytes
and fp32 row scales bit for bit, on random rows with outliers and signed
zeros, on special rows (zeros, NaN, Inf, bf16 subnormals, amax exactly 448),
at the largest supported width and on sampled rows of the full quantize
workload (bf16 [16384, 7168])."""
import numpy as np
import pytest
import torch

import workloads
from oracle import mx
from tests.helpers import assert_bytes_equal, bits, cuda_device, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _check(dev, xb, what):
    import mxfp8_mixture_experts_gb300 as m
    q, s = m.fp8_quantize_rowmax(to_dev_bf16(xb, dev))
    torch.cuda.synchronize()
    q_ref, s_ref = mx.quantize_rowmax(mx.bf16_to_f64(xb))
    assert_bytes_equal(u8(q), q_ref, what + " bytes")
    got = s.cpu().numpy()
    nan = np.isnan(s_ref)
    assert np.array_equal(np.isnan(got), nan), what
    assert np.array_equal(got[~nan].view(np.uint32), s_ref[~nan].view(np.uint32)), what + " scales"


@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 48), (64, 1024), (300, 5120)])
def test_rowmax_random_rows(dev, rows, cols):
    g = np.random.default_rng(rows * 131 + cols)
    x = g.standard_normal((rows, cols)) * np.exp(g.uniform(-30, 30, (rows, 1)))
    x[g.random(x.shape) < 0.01] *= 100
    x[:, ::13] = 0.0
    x[0, 1 % cols] = -0.0
    _check(dev, mx.f64_to_bf16_bits(x), f"{rows}x{cols}")


def test_rowmax_special_rows(dev):
    g = np.random.default_rng(5)
    x = g.standard_normal((8, 256))
    x[0] = 0.0                                   # zero row: scale 1
    x[0, 3] = -0.0
    x[1, 7] = np.nan                             # NaN row
    x[2, 9] = np.inf                             # Inf row
    x[3] = x[3] * 2.0 ** -130                    # bf16 subnormals: subnormal fp32 scale
    x[4] = np.clip(x[4], -447, 447)
    x[4, 0] = 448.0                              # amax exactly 448: scale 1
    x[5] = np.exp2(np.linspace(-20, 20, 256))    # wider than E4M3's range
    x[6] = 3.0e38                                # near bf16 max
    x[7, :] = -1.0
    _check(dev, mx.f64_to_bf16_bits(x), "special rows")


def test_rowmax_widest_row(dev):
    """cols = 102400: the row takes 200 KB of shared memory."""
    g = np.random.default_rng(6)
    _check(dev, mx.f64_to_bf16_bits(g.standard_normal((3, 102400))), "widest")


def test_rowmax_empty_and_full_size_sampled(dev):
    import mxfp8_mixture_experts_gb300 as m
    L = m.lib()
    assert L.fp8_quantize_rowmax(None, 0, 64, None, None, None) == 0
    R, C = workloads.QUANTIZE_SHAPE
    x = workloads.quantize_input(R, C, seed=0, device=dev)
    q, s = m.fp8_quantize_rowmax(x)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(7).choice(R, 64, replace=False))
    xr = bits(x[torch.as_tensor(rows, device=dev)])
    q_ref, s_ref = mx.quantize_rowmax(mx.bf16_to_f64(xr))
    assert_bytes_equal(u8(q[torch.as_tensor(rows, device=dev)]), q_ref, "sampled rows")
    assert np.array_equal(s.cpu().numpy()[rows].view(np.uint32), s_ref.view(np.uint32))
