"""CPU oracle: the MXFP8 number format and block quantizer (TEST INFRASTRUCTURE).

This file is test infrastructure.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library under
``mxfp8_mixture_experts_gb300/`` never does, and shares no code with it.

Everything here is plain numpy on exact reals (fp64 holds every value that
occurs exactly) or exact integers, written for a reader to check by eye.

Sources
-------
* "1.5x faster MoE training on Blackwell with MXFP8 kernels built from scratch"
  (engineering.fyi), Key Questions Answered ("How does microscaling improve
  training performance?"): the tensor is scaled in fine-grained sub-blocks so a
  low-precision element format covers the dynamic range.
* pytorch/ao PR "[mxfp8 moe training] bench and profile mxfp8 a2a fwd and bwd
  separately", Stacked PRs ("simplify e8m0 -> fp32 calc"): the shared block
  scale is an E8M0 byte that decodes to a power of two in fp32.
* The pages give no formulas.  The block size (32), the element type (E4M3) and
  the scale rule X = 2^(floor(log2 amax) - 8) (8 = the exponent of E4M3's
  largest power of two, 256) follow the OCP Microscaling Formats (MX) v1.0
  specification, section 6.3 (conversion of a vector of scalars to MX).
  Element casts round to nearest, ties to even, and saturate to +-448.

Readings where the sources are silent:
* A block holding a NaN or an infinity gets scale byte 0xFF (NaN) and every
  element byte 0x7F (NaN).
* An all-zero block (amax = 0) gets the smallest scale, byte 0x00 (2^-127);
  its elements encode as signed zeros (+0 -> 0x00, -0 -> 0x80).
* The scale exponent is clamped to [-127, 127]; finite bf16 never exceeds 119,
  bf16 subnormals clamp at -127.
* COL mode quantizes blocks of 32 consecutive rows of one column and stores
  the result transposed: COL(X) is, byte for byte, ROW(X^T).

Parity pins for this file live in tests/test_oracle_mx.py (exhaustive sweep
against torch's float8_e4m3fn cast inside the unsaturated range, hand-worked
blocks in tests/golden/mx_blocks.txt, the half-ulp bound, the swizzle
bijection and a hand-checked swizzle position).
"""
from __future__ import annotations

import numpy as np

BLOCK = 32            # elements that share one scale
E4M3_MAX = 448.0      # largest finite E4M3FN value, 1.75 * 2^8
E4M3_EMAX = 8         # exponent of E4M3's largest power of two
E4M3_NAN = 0x7F
E5M2_MAX = 57344.0    # largest finite E5M2 value, 1.75 * 2^15
E5M2_EMAX = 15        # exponent of E5M2's largest power of two
E5M2_NAN = 0x7F       # S.11111.11
E8M0_NAN = 0xFF
SCALE_EXP_MIN = -127
SCALE_EXP_MAX = 127


# ----------------------------------------------------------------------------
# bf16 <-> real
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values: a bf16 is the top half
    of an IEEE fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16, nearest-even, on the bit pattern.  NaN maps to
    the quiet NaN 0x7FC0 (sign kept)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(nan, ((u >> np.uint64(16)).astype(np.uint16) & np.uint16(0x8000)) | np.uint16(0x7FC0), r)
    return r.astype(np.uint16)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round exact reals (fp64) to bf16 with ONE round-to-nearest-even step
    (no detour through fp32, which would round twice).

    bf16 has 8 significant bits: a normal |x| in [2^p, 2^(p+1)) is a multiple
    of 2^(p-7); below 2^-126 (subnormal) the step is 2^-133.  Results beyond
    the largest finite bf16 become infinities."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                       # a = m * 2^ex, m in [0.5, 1)
    p = np.maximum(ex - 1, -126)              # floor(log2 a), floored at the subnormal binade
    step_exp = p - 7
    n = np.rint(np.ldexp(a, -step_exp))       # nearest, ties to even
    v = np.ldexp(n, step_exp)
    big = v >= 2.0 ** 128
    v = np.where(big, np.inf, v)
    v = np.copysign(v, x)
    v = np.where(np.isnan(x), np.nan, v)
    with np.errstate(over="ignore"):
        bits = v.astype(np.float32).view(np.uint32) >> np.uint32(16)   # exact: v is a bf16 value
    return bits.astype(np.uint16)


# ----------------------------------------------------------------------------
# E4M3 (OCP "E4M3FN": bias 7, no infinities, NaN = S.1111.111, max 448)
# ----------------------------------------------------------------------------
def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """E4M3 byte -> exact value (fp64)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** -9                                   # E == 0: m * 2^-9
    norm = (1.0 + m / 8.0) * np.ldexp(1.0, E - 7)         # E >= 1
    v = sign * np.where(E == 0, sub, norm)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_encode(r: np.ndarray) -> np.ndarray:
    """Exact reals -> E4M3 bytes: saturate |r| > 448 to +-448, otherwise round
    to the nearest E4M3 value with ties to an even mantissa; the sign of zero
    is kept; NaN -> 0x7F.

    E4M3 holds 4 significant bits: in the binade [2^p, 2^(p+1)), p >= -6, the
    values are multiples of 2^(p-3); below 2^-6 (subnormals) multiples of
    2^-9."""
    r = np.asarray(r, dtype=np.float64)
    neg = np.signbit(r)
    a = np.abs(r)
    fin = np.isfinite(a)
    _, ex = np.frexp(np.where(fin, a, 0.0))
    p = np.maximum(ex - 1, -6)
    q_exp = p - 3                                         # exponent of the grid step
    n = np.rint(np.ldexp(np.where(fin, a, 0.0), -q_exp)).astype(np.int64)   # RNE onto the grid
    # n == 16 means rounding carried into the next binade: 16 * 2^q = 8 * 2^(q+1)
    carry = n == 16
    n = np.where(carry, 8, n)
    q_exp = np.where(carry, q_exp + 1, q_exp)
    normal = n >= 8
    biased = q_exp + 3 + 7                                # value = (1 + m/8) * 2^(q_exp+3)
    code = np.where(normal, (biased << 3) | (n - 8), n)   # subnormal: E = 0, m = n
    code = np.where(a > E4M3_MAX, 0x7E, code)
    code = code | np.where(neg, 0x80, 0)
    code = np.where(np.isnan(r), E4M3_NAN, code)
    return code.astype(np.uint8)


def e4m3_ulp(code: np.ndarray) -> np.ndarray:
    """Spacing of the E4M3 grid at the magnitude of ``code`` (fp64)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    E = (c >> 3) & 0xF
    return np.where(E == 0, 2.0 ** -9, np.ldexp(1.0, np.maximum(E, 1) - 7 - 3))


# ----------------------------------------------------------------------------
# E5M2 (OCP: bias 15, infinities S.11111.00, NaN S.11111.xx (xx != 0),
# max 57344) -- the gradient option; the pages name only MXFP8 with E4M3
# ----------------------------------------------------------------------------
def e5m2_decode(code: np.ndarray) -> np.ndarray:
    """E5M2 byte -> exact value (fp64); +-Inf and NaN as such."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 2) & 0x1F
    m = c & 0x3
    sub = m * 2.0 ** -16                                  # E == 0: m * 2^-16
    norm = (1.0 + m / 4.0) * np.ldexp(1.0, E - 15)        # 1 <= E <= 30
    v = sign * np.where(E == 0, sub, norm)
    v = np.where(E == 31, np.where(m == 0, sign * np.inf, np.nan), v)
    return v


def e5m2_encode(r: np.ndarray) -> np.ndarray:
    """Exact reals -> E5M2 bytes: saturate |r| > 57344 (and +-Inf) to
    +-57344, otherwise round to the nearest E5M2 value with ties to an even
    mantissa; the sign of zero is kept; NaN -> 0x7F.

    E5M2 holds 3 significant bits: in the binade [2^p, 2^(p+1)), p >= -14, the
    values are multiples of 2^(p-2); below 2^-14 (subnormals) multiples of
    2^-16."""
    r = np.asarray(r, dtype=np.float64)
    neg = np.signbit(r)
    a = np.abs(r)
    fin = np.isfinite(a)
    _, ex = np.frexp(np.where(fin, a, 0.0))
    p = np.maximum(ex - 1, -14)
    q_exp = p - 2                                         # exponent of the grid step
    n = np.rint(np.ldexp(np.where(fin, a, 0.0), -q_exp)).astype(np.int64)   # RNE onto the grid
    carry = n == 8                                        # rounded into the next binade
    n = np.where(carry, 4, n)
    q_exp = np.where(carry, q_exp + 1, q_exp)
    normal = n >= 4
    biased = q_exp + 2 + 15                               # value = (1 + m/4) * 2^(q_exp+2)
    code = np.where(normal, (biased << 2) | (n - 4), n)   # subnormal: E = 0, m = n
    code = np.where(a > E5M2_MAX, 0x7B, code)             # also +-Inf
    code = code | np.where(neg, 0x80, 0)
    code = np.where(np.isnan(r), E5M2_NAN, code)
    return code.astype(np.uint8)


def e5m2_ulp(code: np.ndarray) -> np.ndarray:
    """Spacing of the E5M2 grid at the magnitude of ``code`` (fp64)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    E = (c >> 2) & 0x1F
    return np.where(E == 0, 2.0 ** -16, np.ldexp(1.0, np.maximum(E, 1) - 15 - 2))


def _fmt(fmt):
    """Element format of an MX block: (encode, decode, exponent of the largest
    power of two, largest finite value)."""
    if fmt == "e4m3":
        return e4m3_encode, e4m3_decode, E4M3_EMAX, E4M3_MAX
    if fmt == "e5m2":
        return e5m2_encode, e5m2_decode, E5M2_EMAX, E5M2_MAX
    raise ValueError(fmt)


# ----------------------------------------------------------------------------
# E8M0 scale
# ----------------------------------------------------------------------------
def e8m0_decode(byte: np.ndarray) -> np.ndarray:
    """E8M0 byte b -> 2^(b - 127); 0xFF is NaN."""
    b = np.asarray(byte, dtype=np.uint8).astype(np.int64)
    return np.where(b == E8M0_NAN, np.nan, np.ldexp(1.0, b - 127))


def floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2 a) for a > 0, exactly, from the binary exponent."""
    _, ex = np.frexp(np.asarray(a, dtype=np.float64))
    return ex - 1


# ----------------------------------------------------------------------------
# Block quantizer
# ----------------------------------------------------------------------------
def quantize_blocks(v: np.ndarray, fmt: str = "e4m3"):
    """Quantize the last axis of ``v`` (length 32, exact reals) as one MX block.

    1. amax = max |v_i|.
    2. Scale exponent e = floor(log2 amax) - emax (amax = 0: e = -127), with
       emax = 8 for E4M3 and 15 for E5M2 (the exponent of the element type's
       largest power of two), clamped to [-127, 127]; the scale byte is
       e + 127.
    3. Each element is cast to the element type from v_i * 2^-e (exact), with
       RNE and saturation.
    A block holding NaN/Inf gets scale 0xFF and element bytes 0x7F.

    Returns (codes uint8 [..., 32], scale bytes uint8 [...])."""
    encode, _, emax, _ = _fmt(fmt)
    v = np.asarray(v, dtype=np.float64)
    assert v.shape[-1] == BLOCK
    bad = ~np.all(np.isfinite(v), axis=-1)
    a = np.abs(np.where(np.isfinite(v), v, 0.0))
    amax = a.max(axis=-1)
    e = np.where(amax > 0, floor_log2(np.where(amax > 0, amax, 1.0)) - emax, SCALE_EXP_MIN)
    e = np.clip(e, SCALE_EXP_MIN, SCALE_EXP_MAX)
    r = np.ldexp(np.where(np.isfinite(v), v, 0.0), -e[..., None])
    codes = encode(r)
    scale = (e + 127).astype(np.uint8)
    codes = np.where(bad[..., None], np.uint8(E4M3_NAN), codes)
    scale = np.where(bad, np.uint8(E8M0_NAN), scale)
    return codes.astype(np.uint8), scale.astype(np.uint8)


def quantize_rows(x: np.ndarray, fmt: str = "e4m3"):
    """ROW mode: blocks of 32 along the last axis of a 2-D (or batched) array.
    Returns (q same shape uint8, s [..., cols/32] uint8)."""
    x = np.asarray(x, dtype=np.float64)
    *lead, cols = x.shape
    assert cols % BLOCK == 0, "ROW mode needs cols % 32 == 0"
    q, s = quantize_blocks(x.reshape(*lead, cols // BLOCK, BLOCK), fmt)
    return q.reshape(*lead, cols), s


def quantize_cols(x: np.ndarray, fmt: str = "e4m3"):
    """COL mode: blocks of 32 consecutive rows of one column, output stored
    transposed, i.e. ROW mode applied to X^T (last two axes swapped)."""
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-2] % BLOCK == 0, "COL mode needs rows % 32 == 0"
    return quantize_rows(np.swapaxes(x, -1, -2), fmt)


def dequantize_rows(q: np.ndarray, s: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """MX bytes -> exact values: element value times its block's scale."""
    _, decode, _, _ = _fmt(fmt)
    q = np.asarray(q, dtype=np.uint8)
    *lead, cols = q.shape
    v = decode(q).reshape(*lead, cols // BLOCK, BLOCK)
    return (v * e8m0_decode(s)[..., None]).reshape(*lead, cols)


def quantize_margins(x: np.ndarray, fmt: str = "e4m3"):
    """How close each element's quantization decision is to flipping, for
    values computed in a different precision (fp32 on a GPU, fp64 here).

    Returns (elem_rel, block_rel):
      elem_rel  [..., cols]    distance of x_i*2^-e from the nearest E4M3
                               rounding midpoint (or from 448 for saturation),
                               relative to |x_i*2^-e|;
      block_rel [..., cols/32] distance of amax from the nearest power of two,
                               relative to amax (the scale flips there).
    Row blocks along the last axis, as in quantize_rows."""
    x = np.asarray(x, dtype=np.float64)
    *lead, cols = x.shape
    xb = x.reshape(*lead, cols // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=-1)
    pos = amax > 0
    safe = np.where(pos, amax, 1.0)
    p = floor_log2(safe)
    lo = np.ldexp(1.0, p)
    block_rel = np.where(pos, np.minimum(safe - lo, 2 * lo - safe) / safe, np.inf)
    _, _, emax, fmax = _fmt(fmt)
    mbits, emin = (3, -6) if fmt == "e4m3" else (2, -14)
    e = np.clip(np.where(pos, p - emax, SCALE_EXP_MIN), SCALE_EXP_MIN, SCALE_EXP_MAX)
    r = np.abs(np.ldexp(xb, -e[..., None]))
    _, ex = np.frexp(r)
    q_exp = np.maximum(ex - 1, emin) - mbits
    t = np.ldexp(r, -q_exp)                  # position on the grid, in steps
    mid_dist = np.abs(t - np.floor(t) - 0.5) * np.ldexp(1.0, q_exp)
    sat_dist = np.abs(r - fmax)
    d = np.minimum(mid_dist, sat_dist)
    elem_rel = np.where(r > 0, d / np.where(r > 0, r, 1.0), np.inf)
    return elem_rel.reshape(*lead, cols), block_rel


# ----------------------------------------------------------------------------
# Row-max-scaled FP8: one scale per row (a comparison to MX block scaling)
# ----------------------------------------------------------------------------
def quantize_rowmax(x: np.ndarray):
    """One fp32 scale per row instead of one E8M0 scale per 32 elements.

    NVIDIA/TransformerEngine issue "FP8 significantly slow down when scaling
    up to 1000+ GPUs" describes casting a row to FP8 after computing its
    row-max and dividing by it, and multiplying the row-max back after the
    GEMM.  Readings (the issue gives no formula):
    * the row-max is max |x| over the row;
    * the scale maps it onto E4M3's largest finite value:
      s = fp32(amax / 448), one IEEE fp32 division;
    * each element is q = E4M3(fp32(x / s)) (IEEE fp32 division, then round to
      nearest even with saturation at +-448); x is bf16, exact in fp32;
    * the decoded value is q * s;
    * a row of zeros gets s = 1 (its elements encode as signed zeros); a row
      holding NaN or Inf gets s = NaN and every byte 0x7F.
    The fp32 steps are the precision in which the GPU takes the same
    decisions (one division each), so bytes and scales compare bit for bit.

    Returns (q uint8 same shape, s float32 [..., rows])."""
    x = np.asarray(x, dtype=np.float64)
    fin = np.isfinite(x)
    bad = ~np.all(fin, axis=-1)
    amax = np.abs(np.where(fin, x, 0.0)).max(axis=-1)
    s = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    r = (np.where(fin, x, 0.0).astype(np.float32) / s[..., None]).astype(np.float32)
    q = e4m3_encode(r.astype(np.float64))
    q = np.where(bad[..., None], np.uint8(E4M3_NAN), q).astype(np.uint8)
    s = np.where(bad, np.float32(np.nan), s).astype(np.float32)
    return q, s


def dequantize_rowmax(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Row-max-scaled FP8 bytes -> values: element value times its row scale."""
    return e4m3_decode(q) * np.asarray(s, np.float64)[..., None]


# ----------------------------------------------------------------------------
# Scale layout for the block-scaled tensor-core MMA
# ----------------------------------------------------------------------------
def swizzled_offset(r, c, cols: int):
    """Byte offset of scale (row r, scale-column c) in the tiled layout the
    block-scaled tcgen05 MMA consumes: tiles of 128 rows x 4 scale columns
    (512 bytes, ordered row-tile-major); inside a tile, row r sits at
    (r % 32) * 16 + ((r % 128) // 32) * 4 and column c at c % 4.
    ``cols`` is the number of scale columns before padding to 4."""
    cols_p = -(-cols // 4) * 4
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tile = (r // 128) * (cols_p // 4) + (c // 4)
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def swizzled_size(rows: int, cols: int) -> int:
    return (-(-rows // 128) * 128) * (-(-cols // 4) * 4)


def swizzle_scales(s: np.ndarray) -> np.ndarray:
    """Plain [rows, cols] scale bytes -> flat tiled layout (padding = 0x00)."""
    s = np.asarray(s, dtype=np.uint8)
    rows, cols = s.shape
    out = np.zeros(swizzled_size(rows, cols), dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    out[swizzled_offset(rr, cc, cols)] = s
    return out


def unswizzle_scales(flat: np.ndarray, rows: int, cols: int) -> np.ndarray:
    flat = np.asarray(flat, dtype=np.uint8).reshape(-1)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    return flat[swizzled_offset(rr, cc, cols)]
