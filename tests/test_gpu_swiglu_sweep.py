"""The SwiGLU arithmetic of the kernels over the whole range of its input.

a is swept over every finite bf16 value in [-128, 128]: where the sigmoid's
exponential is far from 1 (a very negative: silu(a) ~ a e^a, down to the fp32
subnormal range) and where 1 + a (1 - sigmoid(a)) cancels (the zero of the
SwiGLU derivative near a = -1.28).  Three checks:
  * the fp32 sigmoid and 1 - sigmoid the kernels use (through the
    mx_selftest_sigmoid entry point) against an exact evaluation, within
    SIG_ULPS units of 2^-24 relative;
  * moe_swiglu_bwd on the sweep ([da|db] quantized both ways, h quantized by
    columns) against the oracle's fp64 SwiGLU backward;
  * the GLU epilogue of GEMM1 on E4M3-exact operands built so that the fp32
    accumulator holds each swept a exactly (a|b bit-exact, h quantized against
    the oracle).
The quantized bytes must match except where the fp64 value lies within the
kernels' error bound (derived from the sigmoid bound) of an E4M3 rounding
decision."""
import numpy as np
import pytest
import torch

from oracle import moe, mx
from tests.helpers import (SIG_ULPS, assert_bytes_equal, bits, cuda_device, quant_mismatches_outside_margin,
                           swiglu_margins, to_dev_bf16, u8)

pytestmark = pytest.mark.gpu

# Where sigmoid(a) is within 2^-18 of 1/2 (|a| < 2^-16) or within 2^-23 of 1
# (a > 16), h, da and db lie that close to products of bf16 values (and of
# dh): points of the E4M3 rounding lattice (midpoints) and powers of two
# (scale steps), where an fp32 and an fp64 evaluation may legitimately round
# to different sides.  There every mismatch must still fall within the error
# bound, but mismatches are not rare; elsewhere they must be (at most 1e-3 of
# the elements).
def _on_lattice(a):
    return (np.abs(a) < 2.0 ** -16) | (a > 16.0)


def _check(got_q, got_s, values, margins, a_of, what):
    n = quant_mismatches_outside_margin(got_q, got_s, values, what, rel_margin=margins, max_frac=1.0)
    q_ref, _ = mx.quantize_rows(values)
    mis = np.asarray(got_q) != q_ref
    off = ~_on_lattice(a_of)
    print(f"{what}: {int(mis[off].sum())} of {int(off.sum())} off-lattice, {int(mis[~off].sum())} of "
          f"{int((~off).sum())} on-lattice bytes differ (all within the error bound)")
    assert mis[off].sum() <= 1e-3 * off.sum(), f"{what}: {int(mis[off].sum())} mismatches off the lattice"
    return n


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _bf16_sweep(lo=-128.0, hi=128.0, min_abs=0.0, with_neg_zero=True):
    """Every finite bf16 value in [lo, hi] with |v| >= min_abs (and +0; -0
    unless excluded), ascending, as uint16 bit patterns."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = mx.bf16_to_f64(b)
    keep = np.isfinite(v) & (v >= lo) & (v <= hi) & ((np.abs(v) >= min_abs) | (v == 0))
    if not with_neg_zero:
        keep &= b != 0x8000
    b, v = b[keep], v[keep]
    order = np.lexsort((np.signbit(v) == 0, v))
    return b[order]


def test_sigmoid_error_bound(dev):
    """sigma = s * back and 1 - sigma from the kernels' fp32 code, for every
    finite bf16 a: relative error at most SIG_ULPS * 2^-24 against the fp64
    sigmoid, plus the exponential's flush to zero below 2^-126 (which only
    touches 1 - sigma for a > 87 and s for a < -132, where the products the
    kernels form with them are unaffected or below the fp32 range)."""
    import mxfp8_mixture_experts_gb300 as m
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    a = mx.bf16_to_f64(b)
    fin = np.isfinite(a)
    b, a = b[fin], a[fin]
    s, oms, back = m.mx_selftest_sigmoid(to_dev_bf16(b, dev))
    torch.cuda.synchronize()
    s = s.cpu().numpy().astype(np.float64)
    oms = oms.cpu().numpy().astype(np.float64)
    back = back.cpu().numpy().astype(np.float64)
    assert np.array_equal(back, np.where(a < -64, 2.0 ** -64, 1.0))
    sig = moe.sigmoid(a)
    one_minus = moe.sigmoid(-a)
    u = 2.0 ** -24
    err_s = np.abs(s * back - sig)
    err_o = np.abs(oms - one_minus)
    rel_s = err_s / sig
    rel_o = err_o / one_minus
    inside = np.abs(a) <= 128
    print(f"sigmoid: max rel err {rel_s[inside].max() / u:.2f} x 2^-24; 1 - sigmoid: "
          f"{rel_o[inside & (a <= 87)].max() / u:.2f} x 2^-24 (|a| <= 128)")
    assert np.all(err_s <= SIG_ULPS * u * sig + 2.0 ** -126 * back), np.argwhere(err_s > SIG_ULPS * u * sig)[:5]
    assert np.all(err_o <= SIG_ULPS * u * one_minus + 2.0 ** -126)
    # relative bound alone where nothing is flushed
    assert np.all(rel_s[inside] <= SIG_ULPS * u)
    assert np.all(rel_o[inside & (a <= 87)] <= SIG_ULPS * u)


@pytest.mark.parametrize("arrangement", ["sorted", "shuffled"])
def test_swiglu_bwd_sweep(dev, arrangement):
    """moe_swiglu_bwd over every finite bf16 a in [-128, 128] (sorted: each
    32-element block holds neighbouring values, so whole blocks sit among the
    fp32 subnormals or at the derivative's zero; shuffled: every block mixes
    magnitudes), with b cycling over five bf16 values per column and dh over
    four fp32 values per row."""
    import mxfp8_mixture_experts_gb300 as m
    rows, F = 256, 160
    sweep = _bf16_sweep()
    if arrangement == "shuffled":
        sweep = np.random.default_rng(11).permutation(sweep)
    a_bits = np.resize(sweep, rows * F).reshape(rows, F)
    b_vals = mx.f64_to_bf16_bits(np.array([1.0, -0.75, 3.5, -0.0078125, 0.3]))
    b_bits = b_vals[np.arange(F) % 5][None, :].repeat(rows, 0)
    dh = np.array([1.0, -0.37, 2.5e-3, 6.0], np.float32)[np.arange(rows) % 4][:, None].repeat(F, 1)
    ab = to_dev_bf16(np.concatenate([a_bits, b_bits], axis=1), dev)
    dh_t = torch.from_numpy(dh).to(dev)
    dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs = m.moe_swiglu_bwd(dh_t, ab)
    torch.cuda.synchronize()

    a, b = mx.bf16_to_f64(a_bits), mx.bf16_to_f64(b_bits)
    dh64 = dh.astype(np.float64)
    da, db = moe.swiglu_bwd(dh64, a, b)
    h = moe.swiglu(a, b)
    m_h, m_da, m_db = swiglu_margins(dh64, a, b)
    dab = np.concatenate([da, db], axis=1)
    m_dab = np.concatenate([m_da, m_db], axis=1)
    a2 = np.concatenate([a, a], axis=1)
    n = _check(u8(dab_rq), mx.unswizzle_scales(u8(dab_rs), rows, 2 * F // 32), dab, m_dab, a2, "dab rows")
    n += _check(u8(dab_cq), mx.unswizzle_scales(u8(dab_cs), 2 * F, rows // 32), dab.T.copy(), m_dab.T.copy(),
                a2.T, "dab cols")
    n += _check(u8(h_cq), mx.unswizzle_scales(u8(h_cs), F, rows // 32), h.T.copy(), m_h.T.copy(), a.T, "h cols")
    print(f"{arrangement}: {n} bytes differ at excused rounding decisions of {3 * rows * F * 2}")


def test_glu_epilogue_sweep(dev):
    """GEMM1 with the fused SwiGLU epilogue on operands built so that each
    output a is a swept bf16 value, exactly: the weight column of feature j
    holds, in two 32-element blocks of H, the value's top four significant
    bits (hi) and the rest (lo, at most four bits), each beside a power of two
    that sets the block scale so both are E4M3-exact; the activation row picks
    those blocks with ones.  b comes the same way from the W3 half (five bf16
    values, four significant bits each).  The fp32 accumulator then holds
    a = hi + lo exactly, so a|b must come back bit-exact, and h quantized must
    match the oracle under the error bound.  Every bf16 a with
    2^-100 <= |a| <= 128 and +0 (the fp32 products stay normal)."""
    import mxfp8_mixture_experts_gb300 as m
    E, S, F = 2, 16, 1152          # experts, slots per expert, features
    H = 64 * S                     # a slot = two 32-element blocks of H
    rows_e = 128
    M = E * rows_e
    sweep = _bf16_sweep(min_abs=2.0 ** -100, with_neg_zero=False)
    vals = mx.bf16_to_f64(np.resize(sweep, E * S * F)).reshape(E, S, F)

    def split4(v):
        """v = hi + lo with hi rounded to 4 significant bits, lo the rest."""
        v = np.asarray(v, np.float64)
        _, ex = np.frexp(np.where(v == 0, 1.0, v))
        q = np.ldexp(1.0, ex - 4)                    # weight of hi's last bit
        hi = np.where(v == 0, 0.0, np.round(v / q) * q)
        return hi, v - hi

    def scale_partner(v):
        """A power of two 2 to 4 times |v| (0 for v = 0): as the block's amax it
        puts v at 64..128 on the E4M3 grid, where 4 significant bits are exact."""
        _, ex = np.frexp(np.where(v == 0, 1.0, v))
        return np.where(v == 0, 0.0, np.ldexp(1.0, ex + 1))

    hi, lo = split4(vals)
    b_set = np.array([1.0, -0.75, 3.5, -0.0078125, 0.40625])
    b_col = b_set[np.arange(F) % 5]
    W13 = np.zeros((E, H, 2 * F))
    for s in range(S):
        W13[:, 64 * s, :F] = hi[:, s, :]
        W13[:, 64 * s + 1, :F] = scale_partner(hi[:, s, :])
        W13[:, 64 * s + 32, :F] = lo[:, s, :]
        W13[:, 64 * s + 33, :F] = scale_partner(lo[:, s, :])
        W13[:, 64 * s, F:] = b_col
        W13[:, 64 * s + 1, F:] = scale_partner(b_col)
    x = np.zeros((M, H))
    slot = np.arange(M) % rows_e % S
    x[np.arange(M), 64 * slot] = 1.0
    x[np.arange(M), 64 * slot + 32] = 1.0
    W13_bits = mx.f64_to_bf16_bits(W13)
    assert np.array_equal(mx.bf16_to_f64(W13_bits), W13)
    # the operands quantize exactly (checked on the oracle's quantizer)
    cq, cs = mx.quantize_cols(W13)
    assert np.array_equal(mx.dequantize_rows(cq, cs), np.swapaxes(W13, 1, 2))

    W13_t = to_dev_bf16(W13_bits, dev)
    x_t = to_dev_bf16(mx.f64_to_bf16_bits(x), dev)
    _, _, w_cq, w_cs = m.mx_quantize(W13_t, m.MX_MODE_COL, m.MX_SCALE_SWIZZLED)
    xq, xs, _, _ = m.mx_quantize(x_t, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    off = torch.tensor([0, rows_e, M], dtype=torch.int32, device=dev)
    ab, hq, hs = m.moe_gemm1_swiglu(xq, xs, w_cq, w_cs, off, E, M, F, H)
    torch.cuda.synchronize()

    e_of = np.arange(M) // rows_e
    a_want = vals[e_of, slot]                                  # [M, F]
    b_want = np.broadcast_to(b_col, (M, F))
    want_bits = mx.f64_to_bf16_bits(np.concatenate([a_want, b_want], axis=1))
    assert_bytes_equal(bits(ab), want_bits, "a|b")
    h = moe.swiglu(a_want, b_want)
    m_h, _, _ = swiglu_margins(np.ones_like(a_want), a_want, b_want)
    n = _check(u8(hq), mx.unswizzle_scales(u8(hs), M, F // 32), h, m_h, a_want, "h (GLU epilogue)")
    print(f"GLU epilogue: {n} bytes differ at excused rounding decisions of {M * F}")
