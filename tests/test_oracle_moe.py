"""Pins for the oracle's router, permute/unpermute, grouped GEMMs, SwiGLU and
layer forward/backward: brute force on tiny inputs in plain Python, closed
forms, invariants and finite differences of the unquantized layer.  CPU only."""
import itertools
import math

import numpy as np
import pytest

from oracle import moe, mx


# ----------------------------------------------------------------------------
# router
# ----------------------------------------------------------------------------
def test_route_brute_force_with_ties():
    g = np.random.default_rng(0)
    T, E, k = 40, 6, 2
    l = g.standard_normal((T, E)).astype(np.float32)
    l[3, 1] = l[3, 4] = 5.0          # tie for first place: lower id wins
    l[7, :] = 0.5                     # all equal
    ids, gate = moe.route(l, k)
    for t in range(T):
        row = [float(v) for v in l[t]]
        want = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        assert list(ids[t]) == want
        z = [math.exp(v - max(row)) for v in row]
        for j in range(k):
            assert abs(gate[t, j] - z[want[j]] / sum(z)) <= 1e-7 * abs(gate[t, j]) + 1e-12
    assert list(ids[3]) == [1, 4] and list(ids[7]) == [0, 1]


# ----------------------------------------------------------------------------
# permute / unpermute
# ----------------------------------------------------------------------------
def _brute_map(ids, E, align=128):
    T, k = ids.shape
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[ids[t, j]] += 1
    padded = [-(-c // align) * align for c in counts]
    off = [0]
    for p in padded:
        off.append(off[-1] + p)
    nxt = list(off[:-1])
    dst = []
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            dst.append(nxt[e])
            nxt[e] += 1
    return counts, off, dst


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 5, 2), (300, 16, 4), (130, 3, 3)])
def test_permute_map_brute_force(T, E, k):
    g = np.random.default_rng(T * 7 + E)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if k <= E else None
    counts, off, dst, src = moe.permute_map(ids, E)
    c2, o2, d2 = _brute_map(ids, E)
    assert list(counts) == c2 and list(off) == o2 and list(dst) == d2
    # invariants: every routed pair once, offsets multiples of 128, pad = -1
    assert sorted(src[src >= 0].tolist()) == list(range(T * k))
    assert all(o % 128 == 0 for o in off) and all(np.diff(off) >= 0)
    assert np.sum(src < 0) == off[-1] - T * k
    for e in range(E):
        live = src[off[e]:off[e] + counts[e]]
        assert np.all(live >= 0) and np.all(np.diff(live) > 0)         # stable by t*k+j
        assert np.all(ids.reshape(-1)[live] == e)
        assert np.all(src[off[e] + counts[e]:off[e + 1]] == -1)


def test_permute_empty_experts_and_quant_commutes():
    g = np.random.default_rng(5)
    T, E, k, H = 200, 8, 2, 64
    ids = np.stack([g.choice([1, 4, 6], 2, replace=False) for _ in range(T)]).astype(np.int32)
    counts, off, dst, src = moe.permute_map(ids, E)
    assert counts[0] == 0 and off[0] == off[1] == 0
    x = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((T, H))))
    q, s = mx.quantize_rows(x)
    qp, sp = moe.permute_rows(q, src, k), moe.permute_rows(s, src, k)
    q2, s2 = mx.quantize_rows(moe.permute_rows(x, src, k))
    assert np.array_equal(qp, q2) and np.array_equal(sp, s2)           # pad rows: Q(0) = (0x00, 0x00)
    assert np.all(qp[src < 0] == 0) and np.all(sp[src < 0] == 0)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_unpermute_of_permute_is_k_times_x(k):
    g = np.random.default_rng(k)
    T, E, H = 64, 6, 32
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, off, dst, src = moe.permute_map(ids, E)
    xb = mx.f64_to_bf16_bits(g.standard_normal((T, H)))
    yb = moe.permute_rows(xb, src, k)
    out = mx.bf16_to_f64(moe.unpermute(yb, dst, None, T, k))
    assert np.array_equal(out, k * mx.bf16_to_f64(xb))


def test_unpermute_fp32_order():
    # gate * y products and left-to-right fp32 sums, by hand for one element
    y = mx.f64_to_bf16_bits(np.array([[1.0], [2.0 ** -24], [2.0 ** -24]]))
    dst = np.array([0, 1, 2], np.int32)
    gate = np.array([[1.0, 1.0, 1.0]], np.float32)
    out = mx.bf16_to_f64(moe.unpermute(y, dst, gate, 1, 3))
    # (1 + 2^-24) rounds to 1 in fp32, and again: left-to-right gives exactly 1
    assert out[0, 0] == 1.0
    gate = np.array([[0.5, 3.0, -1.0]], np.float32)
    y = mx.f64_to_bf16_bits(np.array([[3.0], [0.25], [1.0]]))
    out = mx.bf16_to_f64(moe.unpermute(y, dst, gate, 1, 3))
    assert out[0, 0] == 1.5 + 0.75 - 1.0


# ----------------------------------------------------------------------------
# grouped GEMMs
# ----------------------------------------------------------------------------
def test_grouped_gemm_rows_brute_force():
    g = np.random.default_rng(11)
    E, K, N = 3, 8, 5
    offsets = [0, 4, 4, 9]                          # expert 1 empty
    A = g.standard_normal((9, K))
    B = g.standard_normal((E, N, K))
    C = moe.grouped_gemm_rows(A, B, np.array(offsets))
    for e in range(E):
        for m in range(offsets[e], offsets[e + 1]):
            for n in range(N):
                s = 0.0
                for kk in range(K):
                    s += A[m, kk] * B[e, n, kk]
                assert abs(C[m, n] - s) < 1e-12


def test_grouped_gemm_tokens_brute_force():
    g = np.random.default_rng(12)
    R, S = 4, 6
    offsets = [0, 3, 3, 7]
    X = g.standard_normal((R, 7))
    Y = g.standard_normal((S, 7))
    C = moe.grouped_gemm_tokens(X, Y, np.array(offsets))
    assert np.all(C[1] == 0)
    for e in range(3):
        for r, s_ in itertools.product(range(R), range(S)):
            ref = sum(X[r, t] * Y[s_, t] for t in range(offsets[e], offsets[e + 1]))
            assert abs(C[e, r, s_] - ref) < 1e-12


def test_gemm_closed_form_all_ones():
    # all-ones data at scales 2^a and 2^b: every output is K * 2^(a+b)
    K, a, b = 256, -3, 5
    qa = np.full((128, K), 0x38, np.uint8)          # 0x38 = 1.0 in E4M3
    qb = np.full((1, 64, K), 0x38, np.uint8)
    sa = np.full((128, K // 32), 127 + a, np.uint8)
    sb = np.full((1, 64, K // 32), 127 + b, np.uint8)
    C = moe.grouped_gemm_rows(mx.dequantize_rows(qa, sa), mx.dequantize_rows(qb, sb), np.array([0, 128]))
    assert np.all(C == K * 2.0 ** (a + b))


# ----------------------------------------------------------------------------
# SwiGLU
# ----------------------------------------------------------------------------
def test_swiglu_special_values_and_fd():
    assert moe.swiglu(0.0, 3.0) == 0.0
    da, db = moe.swiglu_bwd(1.0, 0.0, 2.0)
    assert da == 2.0 * 0.25 * 2 and db == 0.0       # sigma(0) = 1/2, sigma'(0) = 1/4 -> silu'(0) = 1/2
    g = np.random.default_rng(4)
    a, b = g.standard_normal(50) * 3, g.standard_normal(50)
    da, db = moe.swiglu_bwd(np.ones(50), a, b)
    h = 1e-6
    assert np.allclose(da, (moe.swiglu(a + h, b) - moe.swiglu(a - h, b)) / (2 * h), rtol=1e-7, atol=1e-9)
    assert np.allclose(db, (moe.swiglu(a, b + h) - moe.swiglu(a, b - h)) / (2 * h), rtol=1e-7, atol=1e-9)


# ----------------------------------------------------------------------------
# layer: finite differences of the unquantized fp64 layer
# ----------------------------------------------------------------------------
def _tiny_layer(seed=0, T=24, H=64, E=3, F=64, k=2):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    gate = g.random((T, k))
    x = g.standard_normal((T, H))
    W1 = g.standard_normal((E, H, F)) * 0.1
    W3 = g.standard_normal((E, H, F)) * 0.1
    W2 = g.standard_normal((E, F, H)) * 0.1
    dOut = g.standard_normal((T, H))
    return ids, gate, x, W1, W3, W2, dOut


def _loss(x, W1, W3, W2, ids, gate, dOut):
    f = moe.layer_forward(x, W1, W3, W2, ids, gate, quant=False)
    return float(np.sum(f["out"] * dOut))


def test_layer_backward_finite_differences():
    ids, gate, x, W1, W3, W2, dOut = _tiny_layer()
    fwd = moe.layer_forward(x, W1, W3, W2, ids, gate, quant=False)
    bwd = moe.layer_backward(fwd, x, W1, W3, W2, dOut)
    g = np.random.default_rng(9)
    eps = 1e-6

    def check(name, arr, grad, n=6):
        flat = arr.reshape(-1)
        gflat = grad.reshape(-1)
        for i in g.choice(flat.size, n, replace=False):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(x, W1, W3, W2, ids, gate, dOut)
            flat[i] = old - eps
            lm = _loss(x, W1, W3, W2, ids, gate, dOut)
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - gflat[i]) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, gflat[i])

    check("x", x, bwd["dX"])
    check("W1", W1, bwd["dW1"])
    check("W3", W3, bwd["dW3"])
    check("W2", W2, bwd["dW2"])
    check("gate", gate, bwd["d_gate"])


def test_layer_with_unused_expert_has_zero_weight_grad():
    ids, gate, x, W1, W3, W2, dOut = _tiny_layer(seed=1, E=4, k=1)
    ids[:] = np.where(ids == 3, 1, ids)
    fwd = moe.layer_forward(x, W1, W3, W2, ids, gate, quant=False)
    bwd = moe.layer_backward(fwd, x, W1, W3, W2, dOut)
    assert np.all(bwd["dW1"][3] == 0) and np.all(bwd["dW2"][3] == 0)


def test_quantized_layer_is_close_to_unquantized():
    """The MXFP8 layer tracks the fp64 layer to MXFP8 accuracy (E4M3 keeps 4
    significant bits): relative Frobenius error of a few percent, not more."""
    ids, gate, x, W1, W3, W2, dOut = _tiny_layer(seed=2, T=64, H=128, E=3, F=128, k=2)
    bits = [mx.f64_to_bf16_bits(v) for v in (x, W1, W3, W2, dOut)]
    fq = moe.layer_forward(*bits[:4], ids, gate.astype(np.float32), quant=True)
    fr = moe.layer_forward(*bits[:4], ids, gate.astype(np.float32), quant=False)
    rel = np.linalg.norm(fq["out"] - fr["out"]) / np.linalg.norm(fr["out"])
    assert 1e-3 < rel < 0.1
    bq = moe.layer_backward(fq, *bits[:4], bits[4])
    br = moe.layer_backward(fr, *bits[:4], bits[4])
    for key in ("dX", "dW1", "dW3", "dW2"):
        rel = np.linalg.norm(bq[key] - br[key]) / np.linalg.norm(br[key])
        assert rel < 0.1, key


def test_layer_flops_formula():
    f = moe.layer_flops(16384, 5120, 8192)
    assert abs(f["fwd"] / 1e12 - 4.123) < 1e-3 and abs(f["total"] / 1e12 - 12.37) < 1e-2


def test_e5m2_gradient_option():
    """With E5M2 gradients (dY and [da|db]: 3 significant bits instead of 4)
    the backward still tracks the fp64 layer, less closely than with E4M3;
    the forward is untouched.  Each gradient operand quantized in E5M2
    decodes to the same values as quantizing it directly (the option changes
    only the element format of those two operands)."""
    ids, gate, x, W1, W3, W2, dOut = _tiny_layer(seed=2, T=64, H=128, E=3, F=128, k=2)
    bits = [mx.f64_to_bf16_bits(v) for v in (x, W1, W3, W2, dOut)]
    fq = moe.layer_forward(*bits[:4], ids, gate.astype(np.float32), quant=True)
    fr = moe.layer_forward(*bits[:4], ids, gate.astype(np.float32), quant=False)
    b4 = moe.layer_backward(fq, *bits[:4], bits[4])
    b5 = moe.layer_backward(fq, *bits[:4], bits[4], grad_fmt="e5m2")
    br = moe.layer_backward(fr, *bits[:4], bits[4])
    assert np.array_equal(b4["dY"], b5["dY"])          # dY itself is formed the same way
    for key in ("dX", "dW1", "dW3", "dW2"):
        e4 = np.linalg.norm(b4[key] - br[key]) / np.linalg.norm(br[key])
        e5 = np.linalg.norm(b5[key] - br[key]) / np.linalg.norm(br[key])
        assert e4 < e5 < 0.2, (key, e4, e5)
    # dW2 = h^T dY with dY blocked along tokens in E5M2
    off = fq["offsets"]
    q, s = mx.quantize_cols(b5["dY"], "e5m2")
    dY5 = mx.dequantize_rows(q, s, "e5m2")
    qh, sh = mx.quantize_cols(fq["h"])
    ref = moe.grouped_gemm_tokens(mx.dequantize_rows(qh, sh), dY5, off)
    assert np.allclose(b5["dW2"], ref, rtol=0, atol=0)
