"""CPU oracle: routing, token permute/unpermute, grouped GEMMs, SwiGLU and the
MXFP8 MoE layer forward/backward (TEST INFRASTRUCTURE).

This file is test infrastructure.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library under
``mxfp8_mixture_experts_gb300/`` never does, and shares no code with it.

Plain numpy: fp64 for arithmetic (np.matmul in fp64 is the one library
primitive used, per expert group), exact integers for index work, and fp32
only where a step is defined in fp32 (the unpermute combine).

Sources
-------
* pytorch/ao PR "[mxfp8 moe training] bench and profile mxfp8 a2a fwd and bwd
  separately", Next steps: stay in MXFP8 through the token shuffle and the
  grouped GEMM; an "mxfp8 token shuffle kernel" and a scaled grouped GEMM that
  accepts pre-quantized operands with their scales.
* "1.5x faster MoE training on Blackwell with MXFP8 kernels built from
  scratch", Overview and Key Questions Answered: the whole MoE layer, forward
  and backward, runs on MXFP8 block-scaled tensor-core GEMMs.
* The expert FFN is SwiGLU: h = silu(x W1) * (x W3), y = h W2 (silu(a) =
  a * sigmoid(a)).  The pages name no FFN; SwiGLU is the workload's stated
  expert type.

Readings where the pages are silent:
* Router: top-k of the fp32 logits, ties to the lower expert id; the gate of a
  chosen expert is the softmax over all E logits evaluated at it.
* Each expert's group is padded to a multiple of 128 rows; pad rows hold zero
  data and 0x00 scales; within an expert, routed rows keep the order of the
  flat index t*k + j.
* Combine: out[t] = sum over j of gate[t,j] * y[row(t,j)], products and sums
  in fp32, j in increasing order starting from the j = 0 product, one
  round-to-nearest-even to bf16.
* GEMM outputs: fp32 outputs are compared with the fp64 product of the
  dequantized operands; bf16 outputs (a, b, y, dX) are that product rounded
  once to bf16.
* Backward: dY row = bf16(fp32(gate * dOut[t])), d_gate = <dOut[t], y[row]>;
  the SwiGLU gradient is quantized straight from its fp32/fp64 values.
* Weights W1, W3 [E, H, F] and W2 [E, F, H]; the forward GEMMs use the weights
  quantized along their contraction dim (H for W1/W3, F for W2), dgrad uses
  them quantized along their output dim, and wgrad uses activations and
  gradients quantized along the token dim.
"""
from __future__ import annotations

import numpy as np

from . import mx

ROW_ALIGN = 128


# ----------------------------------------------------------------------------
# Router
# ----------------------------------------------------------------------------
def route(logits: np.ndarray, k: int):
    """Top-k experts per token (ties -> lower id) and softmax gates over all E
    logits, evaluated in fp64 and rounded once to fp32."""
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = l.shape
    order = np.argsort(-l, axis=1, kind="stable")     # stable: equal logits keep id order
    ids = order[:, :k].astype(np.int32)
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    p = z / z.sum(axis=1, keepdims=True)
    gate = np.take_along_axis(p, ids.astype(np.int64), axis=1).astype(np.float32)
    return ids, gate


# ----------------------------------------------------------------------------
# Token permute (group rows by expert, each group padded to 128 rows)
# ----------------------------------------------------------------------------
def permute_map(ids: np.ndarray, E: int, align: int = ROW_ALIGN):
    """counts[e], offsets[E+1] (exclusive prefix of the padded group sizes),
    dst[t*k+j] (destination row of routed pair (t, j)) and src[row]
    (t*k+j, or -1 for a pad row)."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < E)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    padded = -(-counts // align) * align
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    order = np.argsort(flat, kind="stable")            # by expert, then by flat index
    first = np.concatenate([[0], np.cumsum(counts)])[:-1]
    rank = np.arange(flat.size) - first[flat[order]]
    dst = np.empty(flat.size, dtype=np.int64)
    dst[order] = offsets[flat[order]] + rank
    src = np.full(int(offsets[-1]), -1, dtype=np.int64)
    src[dst] = np.arange(flat.size)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            dst.astype(np.int32), src.astype(np.int32))


def permute_rows(x: np.ndarray, src: np.ndarray, k: int) -> np.ndarray:
    """Row gather by the src map: row r holds x[src[r] // k]; pad rows are 0
    (zero bytes for fp8 data and for E8M0 scales, 0 for bf16)."""
    x = np.asarray(x)
    out = np.zeros((src.size,) + x.shape[1:], dtype=x.dtype)
    live = src >= 0
    out[live] = x[src[live] // k]
    return out


def unpermute(y_bits: np.ndarray, dst: np.ndarray, gate, T: int, k: int) -> np.ndarray:
    """Weighted combine, fp32 in j order, one RNE to bf16.  ``y_bits`` are
    bf16 bit patterns [rows, H]; ``gate`` fp32 [T, k] or None (all ones).
    Returns bf16 bit patterns [T, H]."""
    y = mx.bf16_to_f64(y_bits).astype(np.float32)       # exact
    rows = dst.reshape(T, k)
    acc = None
    for j in range(k):
        yj = y[rows[:, j]]
        pj = yj if gate is None else (np.asarray(gate, np.float32)[:, j:j + 1] * yj).astype(np.float32)
        acc = pj if acc is None else (acc + pj).astype(np.float32)
    return mx.f32_to_bf16_bits(acc)


# ----------------------------------------------------------------------------
# Grouped GEMMs over experts (fp64 products of dequantized MX operands)
# ----------------------------------------------------------------------------
def grouped_gemm_rows(A: np.ndarray, B: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Row-grouped GEMM (forward and dgrad): rows off[e]..off[e+1] of A [M, K]
    times B[e]^T ([E, N, K] -> [K, N]).  Rows past off[E] are zero."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    E, N, K2 = B.shape
    assert K == K2
    C = np.zeros((M, N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            C[lo:hi] = A[lo:hi] @ B[e].T
    return C


def grouped_gemm_tokens(X: np.ndarray, Y: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Token-grouped GEMM (wgrad): for each expert e the contraction runs over
    that expert's token columns off[e]..off[e+1] of X [R, M] and Y [S, M]:
    C[e] = X[:, grp] @ Y[:, grp]^T -> [E, R, S].  An empty group gives 0."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    E = len(offsets) - 1
    C = np.zeros((E, X.shape[0], Y.shape[0]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            C[e] = X[:, lo:hi] @ Y[:, lo:hi].T
    return C


# ----------------------------------------------------------------------------
# SwiGLU
# ----------------------------------------------------------------------------
def sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def swiglu(a, b):
    """h = silu(a) * b with silu(a) = a * sigmoid(a) = a / (1 + e^-a)."""
    a = np.asarray(a, np.float64)
    return a * sigmoid(a) * np.asarray(b, np.float64)


def swiglu_bwd(dh, a, b):
    """Gradients of h = silu(a) * b:
    dh/da = b * s * (1 + a * (1 - s)), s = sigmoid(a);  dh/db = silu(a)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    dh = np.asarray(dh, np.float64)
    s = sigmoid(a)
    da = dh * b * s * (1.0 + a * (1.0 - s))
    db = dh * a * s
    return da, db


# ----------------------------------------------------------------------------
# MoE layer (forward and backward)
# ----------------------------------------------------------------------------
def _q_rows(v, quant, fmt="e4m3"):
    """Operand as the GEMM sees it: the dequantized MX values (blocks along the
    last axis, elements of format ``fmt``) when ``quant``, else the values
    themselves."""
    if not quant:
        return np.asarray(v, np.float64)
    q, s = mx.quantize_rows(v, fmt)
    return mx.dequantize_rows(q, s, fmt)


def _q_cols(v, quant, fmt="e4m3"):
    """Transposed operand, quantized along the first axis (blocks of 32 rows)."""
    if not quant:
        return np.swapaxes(np.asarray(v, np.float64), -1, -2)
    q, s = mx.quantize_cols(v, fmt)
    return mx.dequantize_rows(q, s, fmt)


def _vals(v):
    """bf16 bit patterns (uint16) -> exact fp64; any other array -> fp64."""
    v = np.asarray(v)
    return mx.bf16_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64)


def _round_bf16(v, quant):
    return mx.bf16_to_f64(mx.f64_to_bf16_bits(v)) if quant else np.asarray(v, np.float64)


def layer_forward(x_bits, W1_bits, W3_bits, W2_bits, ids, gate, quant: bool = True):
    """MoE SwiGLU layer forward.

    quant=True: the MXFP8 layer (every GEMM operand MX-quantized, GEMM outputs
    a, b, y rounded to bf16, combine in fp32 -> bf16).
    quant=False: the same layer in fp64 on the bf16 inputs with no
    quantization and no intermediate rounding (the reference for SQNR and the
    one the finite-difference pins differentiate).

    Returns a dict with every saved intermediate."""
    x, W1, W3, W2 = _vals(x_bits), _vals(W1_bits), _vals(W3_bits), _vals(W2_bits)
    T, H = x.shape
    E, _, F = W1.shape
    ids = np.asarray(ids)
    k = ids.shape[1]
    if gate is None:
        gate = np.ones((T, k), np.float32)
    gate = np.asarray(gate, np.float32) if quant else np.asarray(gate, np.float64)
    counts, off, dst, src = permute_map(ids, E)

    xp = permute_rows(_q_rows(x, quant), src, k)               # quantize, then permute
    W13 = np.concatenate([W1, W3], axis=2)                      # [E, H, 2F]
    B1 = _q_cols(W13, quant)                                    # [E, 2F, H], blocks along H
    ab = _round_bf16(grouped_gemm_rows(xp, B1, off), quant)     # [P, 2F]
    a, b = ab[:, :F], ab[:, F:]
    h = swiglu(a, b)
    hq = _q_rows(h, quant)                                      # blocks along F
    B2 = _q_cols(W2, quant)                                     # [E, H, F], blocks along F
    y = _round_bf16(grouped_gemm_rows(hq, B2, off), quant)      # [P, H]
    if quant:
        out = mx.bf16_to_f64(unpermute(mx.f64_to_bf16_bits(y), dst, gate, T, k))
    else:
        out = np.zeros((T, H))
        for j in range(k):
            out += gate[:, j:j + 1] * y[dst.reshape(T, k)[:, j]]
    return dict(counts=counts, offsets=off, dst=dst, src=src, xp=xp, a=a, b=b,
                h=h, y=y, out=out, gate=gate, k=k, quant=quant)


def layer_backward(fwd, x_bits, W1_bits, W3_bits, W2_bits, dOut_bits, grad_fmt: str = "e4m3"):
    """MoE SwiGLU layer backward from the saved forward state ``fwd``.

    grad_fmt: element format of the two gradient operands the backward
    quantizes, the routed output gradient dY and [da|db] ("e4m3", or "e5m2",
    the gradient option; the pages name only E4M3); weights, h and the
    permuted input stay E4M3.

    Returns dX [T, H], dW1, dW3 [E, H, F], dW2 [E, F, H], d_gate [T, k], plus
    intermediates (dY, dh, da, db, dxp)."""
    quant = fwd["quant"]
    x, W1, W3, W2 = _vals(x_bits), _vals(W1_bits), _vals(W3_bits), _vals(W2_bits)
    dOut = _vals(dOut_bits)
    T, H = x.shape
    E, _, F = W1.shape
    k, gate, dst, src, off = fwd["k"], fwd["gate"], fwd["dst"], fwd["src"], fwd["offsets"]
    rows = dst.reshape(T, k)

    # upstream gradient per routed row (pad rows stay 0) and the gate gradient
    P = src.size
    dY = np.zeros((P, H))
    d_gate = np.zeros((T, k))
    for j in range(k):
        if quant:
            g = (gate[:, j:j + 1] * dOut.astype(np.float32)).astype(np.float32)
            dY[rows[:, j]] = mx.bf16_to_f64(mx.f32_to_bf16_bits(g))
        else:
            dY[rows[:, j]] = gate[:, j:j + 1] * dOut
        d_gate[:, j] = np.sum(dOut * fwd["y"][rows[:, j]], axis=1)

    # GEMM2 backward: dh = dY W2^T (dgrad), dW2 = h^T dY (wgrad)
    g = grad_fmt
    dh = grouped_gemm_rows(_q_rows(dY, quant, g), _q_rows(W2, quant), off)     # W2[e] [F, H], blocks along H
    dW2 = grouped_gemm_tokens(_q_cols(fwd["h"], quant), _q_cols(dY, quant, g), off)  # [E, F, H]

    # SwiGLU backward
    da, db = swiglu_bwd(dh, fwd["a"], fwd["b"])
    dab = np.concatenate([da, db], axis=1)                                      # [P, 2F]

    # GEMM1 backward: dxp = dab W13^T (dgrad), dW13 = xp^T dab (wgrad)
    W13 = np.concatenate([W1, W3], axis=2)                                      # [E, H, 2F]
    dxp = _round_bf16(grouped_gemm_rows(_q_rows(dab, quant, g), _q_rows(W13, quant), off), quant)
    xp_hi = permute_rows(x, src, k)                                             # bf16 values, permuted
    dW13 = grouped_gemm_tokens(_q_cols(xp_hi, quant), _q_cols(dab, quant, g), off)  # [E, H, 2F]

    # combine the routed-row gradients back to tokens (unit weights)
    if quant:
        dX = mx.bf16_to_f64(unpermute(mx.f64_to_bf16_bits(dxp), dst, None, T, k))
    else:
        dX = np.zeros((T, H))
        for j in range(k):
            dX += dxp[rows[:, j]]
    return dict(dX=dX, dW1=dW13[:, :, :F], dW3=dW13[:, :, F:], dW2=dW2,
                d_gate=d_gate, dY=dY, dh=dh, da=da, db=db, dxp=dxp)


def layer_flops(T_routed: int, H: int, F: int) -> dict:
    """Algorithmic GEMM FLOPs of one layer step over ``T_routed`` real routed
    rows (pad rows are overhead, not work): GEMM1 2*T*H*2F, GEMM2 2*T*F*H,
    and backward twice the forward (dgrad + wgrad of each GEMM)."""
    fwd = 2 * T_routed * H * 2 * F + 2 * T_routed * F * H
    return {"fwd": fwd, "bwd": 2 * fwd, "total": 3 * fwd}
