"""The E5M2 gradient option on the GPU vs the oracle.

MX blocks with E5M2 elements (scale 2^(floor(log2 amax) - 15), elements
saturated to +-57344): quantize and gather-quantize bytes and scales bit for
bit, the dequantize of every E5M2 code at every scale, grouped GEMMs that
multiply E5M2 by E4M3 operands (bit-exact on small integers, 1e-4 relative
Frobenius on random data), the SwiGLU backward writing [da|db] in E5M2, and
the layer backward with E5M2 gradients stage-wise and end to end."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe, mx
from tests.helpers import (assert_bf16_within_one_ulp, assert_bytes_equal, bits, cuda_device,
                           quant_mismatches_outside_margin, rel_frob, to_dev_u8, u8)

pytestmark = pytest.mark.gpu
TOL = 1e-4
E5 = 1


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _swz(s):
    return np.concatenate([mx.swizzle_scales(si) for si in s.reshape(-1, *s.shape[-2:])])


@pytest.mark.parametrize("shape", [(32, 32), (160, 224), (256, 512), (384, 7168)])
@pytest.mark.parametrize("mode", [1, 2, 3])
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_e5m2(dev, shape, mode, layout):
    import mxfp8_mixture_experts_gb300 as m
    x = workloads.quantize_input(*shape, seed=sum(shape) + 7 * mode, device=dev)
    xb = bits(x)
    v = mx.bf16_to_f64(xb)
    qr, sr, qc, sc = m.mx_quantize(x, mode, layout, elem=E5)
    torch.cuda.synchronize()
    if mode & 1:
        q, s = mx.quantize_rows(v, "e5m2")
        assert_bytes_equal(u8(qr), q, "q_row")
        assert_bytes_equal(u8(sr), s.ravel() if layout == 0 else _swz(s), "s_row")
    if mode & 2:
        q, s = mx.quantize_cols(v, "e5m2")
        assert_bytes_equal(u8(qc), q, "q_col")
        assert_bytes_equal(u8(sc), s.ravel() if layout == 0 else _swz(s), "s_col")


def test_quantize_e5m2_special_values(dev):
    """NaN / Inf blocks, bf16 subnormals (scale clamped at 2^-127), values
    that saturate at 57344, ties of E5M2's 2-bit mantissa, signed zeros."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(3)
    v = g.standard_normal((64, 256))
    v[0, 5] = np.nan
    v[1, 40] = -np.inf
    v[2] = v[2] * 2.0 ** -130
    v[3, :32] = 1.8984375
    v[3, 1] = 1.0
    v[4, :32] = 9 * 2.0 ** -15
    v[4, 0] = 1.0
    v[5, 3] = -0.0
    xb = mx.f64_to_bf16_bits(v)
    xt = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    qr, sr, qc, sc = m.mx_quantize(xt, 3, 0, elem=E5)
    torch.cuda.synchronize()
    vv = mx.bf16_to_f64(xb)
    q, s = mx.quantize_rows(vv, "e5m2")
    assert_bytes_equal(u8(qr), q, "rows")
    assert_bytes_equal(u8(sr), s.ravel(), "row scales")
    q, s = mx.quantize_cols(vv, "e5m2")
    assert_bytes_equal(u8(qc), q, "cols")
    assert_bytes_equal(u8(sc), s.ravel(), "col scales")


def test_dequantize_every_e5m2_code(dev):
    """Every E5M2 code (Inf and NaN codes included) at scale bytes across the
    range, decoded to fp32: the oracle's exact value (NaN where it is NaN)."""
    import mxfp8_mixture_experts_gb300 as m
    codes = np.tile(np.arange(256, dtype=np.uint8), 2 * 32).reshape(64, 256)
    sbytes = np.random.default_rng(1).integers(0, 256, (64, 8)).astype(np.uint8)
    sbytes[0, :] = 0
    sbytes[1, :] = 254
    out = m.mx_dequantize(to_dev_u8(codes, dev), to_dev_u8(sbytes.ravel(), dev), 0, m.MX_OUT_F32, elem=E5)
    torch.cuda.synchronize()
    ref = mx.dequantize_rows(codes, sbytes, "e5m2").astype(np.float32)
    got = out.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))


SMALL_E4 = np.array([0x00, 0x30, 0x38, 0x40, 0xB0, 0xB8, 0xC0], np.uint8)   # 0, +-0.5, +-1, +-2 in E4M3
SMALL_E5 = np.array([0x00, 0x38, 0x3C, 0x40, 0xB8, 0xBC, 0xC0], np.uint8)   # the same values in E5M2


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


@pytest.mark.parametrize("a_e5,b_e5", [(1, 0), (0, 1), (1, 1)])
def test_mixed_format_gemms_bit_exact(dev, a_e5, b_e5):
    """Small-integer codes with unit scales: row-grouped and token-grouped
    contractions of E5M2 x E4M3 (either side) and E5M2 x E5M2 are exact in
    fp32, so they must equal the oracle bit for bit."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(10 * a_e5 + b_e5)
    sizes, N, K = [256, 0, 384], 256, 512
    E, M_cap = len(sizes), sum(sizes) + 128
    fa, fb = ("e5m2" if a_e5 else "e4m3"), ("e5m2" if b_e5 else "e4m3")
    Aq = g.choice(SMALL_E5 if a_e5 else SMALL_E4, (M_cap, K))
    Bq = g.choice(SMALL_E5 if b_e5 else SMALL_E4, (E, N, K))
    As = mx.swizzle_scales(np.full((M_cap, K // 32), 127, np.uint8))
    Bs = mx.swizzle_scales(np.full((E * N, K // 32), 127, np.uint8))
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    C = m.mx_grouped_gemm(m.MX_GEMM_FWD, *[to_dev_u8(a, dev) for a in (Aq, As, Bq, Bs)], off, E, M_cap, N, K,
                          m.MX_OUT_F32, elem_a=a_e5, elem_b=b_e5)
    torch.cuda.synchronize()
    A = mx.dequantize_rows(Aq, np.full((M_cap, K // 32), 127, np.uint8), fa)
    B = mx.dequantize_rows(Bq.reshape(E * N, K), np.full((E * N, K // 32), 127, np.uint8), fb).reshape(E, N, K)
    ref = moe.grouped_gemm_rows(A, B, _offsets(sizes))
    P = sum(sizes)
    assert_bytes_equal(C.cpu().numpy()[:P].view(np.uint32), ref[:P].astype(np.float32).view(np.uint32), "rows")

    Xq = g.choice(SMALL_E5 if a_e5 else SMALL_E4, (N, M_cap))
    Yq = g.choice(SMALL_E5 if b_e5 else SMALL_E4, (K, M_cap))
    Xs = mx.swizzle_scales(np.full((N, M_cap // 32), 127, np.uint8))
    Ys = mx.swizzle_scales(np.full((K, M_cap // 32), 127, np.uint8))
    W = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, *[to_dev_u8(a, dev) for a in (Xq, Xs, Yq, Ys)], off, E, M_cap, N, K,
                          m.MX_OUT_F32, elem_a=a_e5, elem_b=b_e5)
    torch.cuda.synchronize()
    X = mx.dequantize_rows(Xq, np.full((N, M_cap // 32), 127, np.uint8), fa)
    Y = mx.dequantize_rows(Yq, np.full((K, M_cap // 32), 127, np.uint8), fb)
    ref = moe.grouped_gemm_tokens(X, Y, _offsets(sizes))
    assert_bytes_equal(W.cpu().numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32), "wgrad")


def test_mixed_format_gemm_random(dev):
    """N(0,1) data quantized on the GPU (A in E5M2, B in E4M3) against the fp64
    product of the dequantized operands: relative Frobenius error <= 1e-4."""
    import mxfp8_mixture_experts_gb300 as m
    g = workloads.generator(12, dev)
    sizes, N, K = [384, 128, 0, 640], 512, 1024
    E, M_cap = len(sizes), sum(sizes) + 128
    A = workloads.randn_bf16((M_cap, K), 1.0, g, dev)
    W = workloads.randn_bf16((E, N, K), 0.02, g, dev)
    aq, as_, _, _ = m.mx_quantize(A, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED, elem=E5)
    wq, ws_, _, _ = m.mx_quantize(W, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    C = m.mx_grouped_gemm(m.MX_GEMM_FWD, aq, as_, wq, ws_, off, E, M_cap, N, K, m.MX_OUT_F32, elem_a=E5)
    torch.cuda.synchronize()
    Ad = mx.dequantize_rows(u8(aq), mx.unswizzle_scales(u8(as_), M_cap, K // 32), "e5m2")
    Wd = mx.dequantize_rows(u8(wq).reshape(E * N, K), mx.unswizzle_scales(u8(ws_), E * N, K // 32)).reshape(E, N, K)
    ref = moe.grouped_gemm_rows(Ad, Wd, _offsets(sizes))
    P = sum(sizes)
    assert rel_frob(C.cpu().numpy()[:P], ref[:P]) <= TOL


def test_swiglu_bwd_e5m2(dev):
    """[da|db] in E5M2 (both layouts) and h in E4M3, against the fp64 SwiGLU
    backward on the same inputs (margin rule at rounding decisions)."""
    import mxfp8_mixture_experts_gb300 as m
    rows, F = 256, 256
    g = workloads.generator(13, dev)
    ab = workloads.randn_bf16((rows, 2 * F), 1.0, g, dev)
    dh = torch.randn((rows, F), generator=g, device=dev)
    dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs = m.moe_swiglu_bwd(dh, ab, grad_elem=E5)
    torch.cuda.synchronize()
    abv = mx.bf16_to_f64(bits(ab))
    da, db = moe.swiglu_bwd(dh.cpu().numpy().astype(np.float64), abv[:, :F], abv[:, F:])
    dab = np.concatenate([da, db], axis=1)
    h = moe.swiglu(abv[:, :F], abv[:, F:])
    quant_mismatches_outside_margin(u8(dab_rq), mx.unswizzle_scales(u8(dab_rs), rows, 2 * F // 32), dab,
                                    "dab rows", fmt="e5m2")
    quant_mismatches_outside_margin(u8(dab_cq), mx.unswizzle_scales(u8(dab_cs), 2 * F, rows // 32), dab.T.copy(),
                                    "dab cols", fmt="e5m2")
    quant_mismatches_outside_margin(u8(h_cq), mx.unswizzle_scales(u8(h_cs), F, rows // 32), h.T.copy(), "h cols")


def test_layer_backward_e5m2_gradients(dev):
    """The tiny layer with E5M2 gradients.  Stage-wise on the GPU's own
    inputs: dY quantized both ways bit-exact; dh (E5M2 dY x E4M3 W2) within
    1e-4; [da|db] under the margin rule; dW2, dW13 within 1e-4; dxp within one
    bf16 ulp.  End to end against the oracle's E5M2-gradient chain (1e-3),
    and the E5M2 option's error against the unquantized layer reported beside
    E4M3's."""
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.TINY_LAYER
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    T, H, F, E, k = d.T, d.H, d.F, d.E, d.k
    inp = workloads.layer_inputs(dims, seed=5, device=dev)
    W13t = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    wq = m.moe_layer_prep_weights(W13t, inp["W2"])
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, _, _ = m.moe_layer_fwd(inp["x"], wq, d, ws, ids=inp["ids"], gate=inp["gate"], dev_status=st)
    dX, dW13, dW2, dg = m.moe_layer_bwd(inp["x"], inp["dOut"], inp["gate"], wq, d, ws, dev_status=st, grad_elem=E5)
    dX4, dW134, dW24, _ = m.moe_layer_bwd(inp["x"], inp["dOut"], inp["gate"], wq, d, ws, grad_elem=0)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    # stage by stage through the C ABI's own calls, on the GPU's intermediates
    ids, gate = inp["ids"], inp["gate"]
    counts, off, dst, src = m.moe_permute_map(ids, E)
    R = src.numel()
    w13_rq, w13_rs, _, _ = m.mx_quantize(W13t, m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    w2_rq, w2_rs, _, _ = m.mx_quantize(inp["W2"], m.MX_MODE_ROW, m.MX_SCALE_SWIZZLED)
    dy_rq, dy_rs, dy_cq, dy_cs = m.moe_gather_quant(inp["dOut"], gate, src, k, m.MX_MODE_BOTH, elem=E5)
    torch.cuda.synchronize()
    offn = off.cpu().numpy()
    P = int(offn[-1])
    srcn = src.cpu().numpy()
    dov = mx.bf16_to_f64(bits(inp["dOut"]))
    gn = gate.cpu().numpy()
    dY = np.zeros((R, H), np.float32)
    live = srcn >= 0
    dY[live] = (gn.reshape(-1)[srcn[live]][:, None] * dov[srcn[live] // k].astype(np.float32)).astype(np.float32)
    dY = mx.bf16_to_f64(mx.f32_to_bf16_bits(dY))
    q, sc = mx.quantize_rows(dY, "e5m2")
    assert_bytes_equal(u8(dy_rq), q, "dY rows")
    assert_bytes_equal(u8(dy_rs), mx.swizzle_scales(sc), "dY row scales")
    q, sc = mx.quantize_cols(dY, "e5m2")
    assert_bytes_equal(u8(dy_cq), q, "dY cols")
    assert_bytes_equal(u8(dy_cs), mx.swizzle_scales(sc), "dY col scales")
    dh = m.mx_grouped_gemm(m.MX_GEMM_DGRAD, dy_rq, dy_rs, w2_rq, w2_rs, off, E, R, F, H, m.MX_OUT_F32, elem_a=E5)
    torch.cuda.synchronize()
    W2v = mx.bf16_to_f64(bits(inp["W2"]))
    w2q, w2s = mx.quantize_rows(W2v)
    dh_ref = moe.grouped_gemm_rows(mx.dequantize_rows(u8(dy_rq), mx.unswizzle_scales(u8(dy_rs), R, H // 32), "e5m2"),
                                   mx.dequantize_rows(w2q, w2s), offn)
    assert rel_frob(dh.cpu().numpy()[:P], dh_ref[:P]) <= TOL

    # end to end against the oracle's chain with E5M2 gradients, and accuracy vs fp64
    b = {n: bits(inp[n]) for n in ("x", "W1", "W3", "W2", "dOut")}
    idn = ids.cpu().numpy()
    fq = moe.layer_forward(b["x"], b["W1"], b["W3"], b["W2"], idn, gn, quant=True)
    b5 = moe.layer_backward(fq, b["x"], b["W1"], b["W3"], b["W2"], b["dOut"], grad_fmt="e5m2")
    fr = moe.layer_forward(b["x"], b["W1"], b["W3"], b["W2"], idn, gn, quant=False)
    br = moe.layer_backward(fr, b["x"], b["W1"], b["W3"], b["W2"], b["dOut"])
    got5 = {"dX": dX.float().cpu().numpy(), "dW13": dW13.cpu().numpy(), "dW2": dW2.cpu().numpy()}
    got4 = {"dX": dX4.float().cpu().numpy(), "dW13": dW134.cpu().numpy(), "dW2": dW24.cpu().numpy()}
    ref5 = {"dX": b5["dX"], "dW13": np.concatenate([b5["dW1"], b5["dW3"]], 2), "dW2": b5["dW2"]}
    refr = {"dX": br["dX"], "dW13": np.concatenate([br["dW1"], br["dW3"]], 2), "dW2": br["dW2"]}
    for n in got5:
        e = rel_frob(got5[n], ref5[n])
        s5 = 10 * np.log10(np.sum(refr[n] ** 2) / np.sum((refr[n] - got5[n]) ** 2))
        s4 = 10 * np.log10(np.sum(refr[n] ** 2) / np.sum((refr[n] - got4[n]) ** 2))
        print(f"{n}: rel err vs E5M2-gradient oracle {e:.2e}; SQNR vs unquantized E5M2 {s5:.1f} dB, E4M3 {s4:.1f} dB")
        assert e < 1e-3, n
        assert s5 < s4, n
