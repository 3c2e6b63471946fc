"""The MXFP8 MoE SwiGLU layer on the GPU vs the oracle.

Stage-wise teacher forcing: each GPU stage is checked against the oracle run
on the GPU's own inputs to that stage (an independent fp64 chain would flip
E4M3 roundings wherever fp32 and fp64 land on different sides of a rounding
boundary).  Integer/byte stages are bit-exact, GEMM stages meet the 1e-4
relative Frobenius bound (fp32 outputs) or one bf16 ulp (bf16 outputs), and
quantized SwiGLU values match except at elements within a few fp32 ulps of a
rounding decision.  The layer entry points must reproduce the staged pipeline
bit for bit, and the end-to-end result is reported against the independent
oracle and as SQNR against the unquantized layer."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe, mx
from tests.helpers import (assert_bf16_within_one_ulp, assert_bytes_equal, bits, cuda_device,
                           quant_mismatches_outside_margin, rel_frob, u8)

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _deq_swz(q, s, rows, cols):
    qh = u8(q).reshape(rows, cols)
    return mx.dequantize_rows(qh, mx.unswizzle_scales(u8(s), rows, cols // 32))


def _staged(dev, inp, d, logits):
    """Run the layer op by op (the same calls moe_layer_fwd/bwd make) and
    keep every intermediate."""
    import mxfp8_mixture_experts_gb300 as m
    T, H, F, E, k = d.T, d.H, d.F, d.E, d.k
    W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    w13_rq, w13_rs, w13_cq, w13_cs = m.mx_quantize(W13, m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    w2_rq, w2_rs, w2_cq, w2_cs = m.mx_quantize(inp["W2"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    if logits is not None:
        ids, gate = m.moe_route(logits, k)
    else:
        ids, gate = inp["ids"], inp["gate"]
    counts, off, dst, src = m.moe_permute_map(ids, E)
    R = src.numel()
    xq, xs = m.moe_permute(m.MX_PERMUTE_BF16_QUANT, inp["x"], dst, src, k, scale_layout=m.MX_SCALE_SWIZZLED)
    ab, hq, hs = m.moe_gemm1_swiglu(xq, xs, w13_cq, w13_cs, off, E, R, F, H)
    y = m.mx_grouped_gemm(m.MX_GEMM_FWD, hq, hs, w2_cq, w2_cs, off, E, R, H, F, m.MX_OUT_BF16)
    out = m.moe_unpermute(y, dst, gate, T, k)
    d_gate = m.moe_gate_grad(inp["dOut"], y, dst, k)
    dy_rq, dy_rs, dy_cq, dy_cs = m.moe_gather_quant(inp["dOut"], gate, src, k, m.MX_MODE_BOTH)
    dh = m.mx_grouped_gemm(m.MX_GEMM_DGRAD, dy_rq, dy_rs, w2_rq, w2_rs, off, E, R, F, H, m.MX_OUT_F32)
    dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs = m.moe_swiglu_bwd(dh, ab)
    dW2 = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, h_cq, h_cs, dy_cq, dy_cs, off, E, R, F, H, m.MX_OUT_F32)
    dxp = m.mx_grouped_gemm(m.MX_GEMM_DGRAD, dab_rq, dab_rs, w13_rq, w13_rs, off, E, R, H, 2 * F, m.MX_OUT_BF16)
    _, _, xp_cq, xp_cs = m.moe_gather_quant(inp["x"], None, src, k, m.MX_MODE_COL)
    dW13 = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, xp_cq, xp_cs, dab_cq, dab_cs, off, E, R, H, 2 * F, m.MX_OUT_F32)
    dX = m.moe_unpermute(dxp, dst, None, T, k)
    torch.cuda.synchronize()
    return {k_: v for k_, v in locals().items() if isinstance(v, torch.Tensor)} | {"R": R}


CASES = {
    # the tiny layer workload: T=512, H=256, E=4, F=512, top-1 uniform ids, gate 1
    "tiny": (workloads.TINY_LAYER, "uniform"),
    # top-2 with a softmax router over N(0,1) logits
    "top2_router": (workloads.LayerDims(T=384, H=256, E=4, F=256, k=2), "logits"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_layer_stagewise(dev, case):
    import mxfp8_mixture_experts_gb300 as m
    dims, router = CASES[case]
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    inp = workloads.layer_inputs(dims, seed=3, device=dev, router=router)
    s = _staged(dev, inp, d, inp["logits"])
    T, H, F, E, k, R = d.T, d.H, d.F, d.E, d.k, s["R"]
    xb, W1b, W3b, W2b, dOb = (bits(inp[n]) for n in ("x", "W1", "W3", "W2", "dOut"))

    # router + map (bit-exact ids; fp32 softmax gate to a few ulps)
    if router == "logits":
        ids_ref, gate_ref = moe.route(inp["logits"].cpu().numpy(), k)
        assert_bytes_equal(s["ids"].cpu().numpy(), ids_ref, "ids")
        np.testing.assert_allclose(s["gate"].cpu().numpy(), gate_ref, rtol=2e-6)
    ids_np = s["ids"].cpu().numpy()
    gate_np = s["gate"].cpu().numpy()
    counts, off, dst, src = moe.permute_map(ids_np, E)
    assert_bytes_equal(s["off"].cpu().numpy(), off, "offsets")
    assert_bytes_equal(s["dst"].cpu().numpy(), dst, "dst")
    src_full = np.concatenate([src, -np.ones(R - len(src), np.int32)])
    P = int(off[-1])

    # permute + quantize x
    xq_ref, xs_ref = mx.quantize_rows(mx.bf16_to_f64(xb))
    assert_bytes_equal(u8(s["xq"]), moe.permute_rows(xq_ref, src_full, k), "xq")
    assert_bytes_equal(u8(s["xs"]), mx.swizzle_scales(moe.permute_rows(xs_ref, src_full, k)), "xs")

    # GEMM1 (+ SwiGLU): a|b within one bf16 ulp of fp64 on the GPU's own operands
    W13 = np.concatenate([mx.bf16_to_f64(W1b), mx.bf16_to_f64(W3b)], axis=2)
    w13c_q, w13c_s = mx.quantize_cols(W13)                       # [E, 2F, H]
    xp = _deq_swz(s["xq"], s["xs"], R, H)
    w13c = mx.dequantize_rows(w13c_q, w13c_s)
    ab_ref = moe.grouped_gemm_rows(xp, w13c, off)
    ab_mag = moe.grouped_gemm_rows(np.abs(xp), np.abs(w13c), off)
    ab_b = bits(s["ab"])
    assert_bf16_within_one_ulp(ab_b[:P], ab_ref[:P], "a|b", mag=ab_mag[:P], K=H)
    abv = mx.bf16_to_f64(ab_b[:P])
    h = moe.swiglu(abv[:, :F], abv[:, F:])
    quant_mismatches_outside_margin(u8(s["hq"])[:P], mx.unswizzle_scales(u8(s["hs"]), R, F // 32)[:P], h, "hq")

    # GEMM2
    w2c_q, w2c_s = mx.quantize_cols(mx.bf16_to_f64(W2b))          # [E, H, F]
    hp = _deq_swz(s["hq"], s["hs"], R, F)
    w2c = mx.dequantize_rows(w2c_q, w2c_s)
    y_ref = moe.grouped_gemm_rows(hp, w2c, off)
    y_mag = moe.grouped_gemm_rows(np.abs(hp), np.abs(w2c), off)
    assert_bf16_within_one_ulp(bits(s["y"])[:P], y_ref[:P], "y", mag=y_mag[:P], K=F)

    # combine
    assert_bytes_equal(bits(s["out"]), moe.unpermute(bits(s["y"]), dst, gate_np, T, k), "out")

    # backward: gate gradient (fp32 dot products of H terms)
    yv = mx.bf16_to_f64(bits(s["y"]))
    dov = mx.bf16_to_f64(dOb)
    rows = dst.reshape(T, k)
    dg_ref = np.stack([np.sum(dov * yv[rows[:, j]], axis=1) for j in range(k)], axis=1)
    dg_bound = H * 2.0 ** -24 * np.stack([np.sum(np.abs(dov * yv[rows[:, j]]), axis=1) for j in range(k)], axis=1)
    assert np.all(np.abs(s["d_gate"].cpu().numpy() - dg_ref) <= dg_bound + 1e-30)

    # dY = bf16(gate * dOut) permuted, quantized both ways (bit-exact)
    dY = np.zeros((R, H), np.float32)
    for j in range(k):
        dY[rows[:, j]] = (gate_np[:, j:j + 1] * dov.astype(np.float32)).astype(np.float32)
    dY = mx.bf16_to_f64(mx.f32_to_bf16_bits(dY))
    q, sc = mx.quantize_rows(dY)
    assert_bytes_equal(u8(s["dy_rq"]), q, "dY row q")
    assert_bytes_equal(u8(s["dy_rs"]), mx.swizzle_scales(sc), "dY row s")
    q, sc = mx.quantize_cols(dY)
    assert_bytes_equal(u8(s["dy_cq"]), q, "dY col q")
    assert_bytes_equal(u8(s["dy_cs"]), mx.swizzle_scales(sc), "dY col s")

    # dgrad2: dh (fp32) on the GPU's quantized dY
    w2r_q, w2r_s = mx.quantize_rows(mx.bf16_to_f64(W2b))          # [E, F, H]
    dh_ref = moe.grouped_gemm_rows(_deq_swz(s["dy_rq"], s["dy_rs"], R, H), mx.dequantize_rows(w2r_q, w2r_s), off)
    dh = s["dh"].cpu().numpy()
    assert rel_frob(dh[:P], dh_ref[:P]) <= TOL

    # SwiGLU backward on the GPU's dh, a, b
    da, db = moe.swiglu_bwd(dh[:P].astype(np.float64), abv[:, :F], abv[:, F:])
    dab = np.concatenate([da, db], axis=1)
    quant_mismatches_outside_margin(u8(s["dab_rq"])[:P], mx.unswizzle_scales(u8(s["dab_rs"]), R, 2 * F // 32)[:P],
                                    dab, "dab rows")
    dab_cq_plain = u8(s["dab_cq"])[:, :P]
    dab_cs_plain = mx.unswizzle_scales(u8(s["dab_cs"]), 2 * F, R // 32)[:, :P // 32]
    quant_mismatches_outside_margin(dab_cq_plain, dab_cs_plain, dab.T.copy(), "dab cols")
    quant_mismatches_outside_margin(u8(s["h_cq"])[:, :P], mx.unswizzle_scales(u8(s["h_cs"]), F, R // 32)[:, :P // 32],
                                    h.T.copy(), "h cols")

    # wgrad2 on the GPU's column-quantized h and dY
    dW2_ref = moe.grouped_gemm_tokens(_deq_swz(s["h_cq"], s["h_cs"], F, R), _deq_swz(s["dy_cq"], s["dy_cs"], H, R), off)
    dW2 = s["dW2"].cpu().numpy()
    for e in range(E):
        assert rel_frob(dW2[e], dW2_ref[e]) <= TOL if counts[e] else np.all(dW2[e] == 0)

    # dgrad1
    w13r_q, w13r_s = mx.quantize_rows(W13)                       # [E, H, 2F]
    dab_r = _deq_swz(s["dab_rq"], s["dab_rs"], R, 2 * F)
    w13r = mx.dequantize_rows(w13r_q, w13r_s)
    dxp_ref = moe.grouped_gemm_rows(dab_r, w13r, off)
    dxp_mag = moe.grouped_gemm_rows(np.abs(dab_r), np.abs(w13r), off)
    assert_bf16_within_one_ulp(bits(s["dxp"])[:P], dxp_ref[:P], "dxp", mag=dxp_mag[:P], K=2 * F)

    # x permuted, column-quantized (bit-exact)
    q, sc = mx.quantize_cols(moe.permute_rows(mx.bf16_to_f64(xb), src_full, k))
    assert_bytes_equal(u8(s["xp_cq"]), q, "xp col q")
    assert_bytes_equal(u8(s["xp_cs"]), mx.swizzle_scales(sc), "xp col s")

    # wgrad1
    dW13_ref = moe.grouped_gemm_tokens(_deq_swz(s["xp_cq"], s["xp_cs"], H, R),
                                       _deq_swz(s["dab_cq"], s["dab_cs"], 2 * F, R), off)
    dW13 = s["dW13"].cpu().numpy()
    for e in range(E):
        assert rel_frob(dW13[e], dW13_ref[e]) <= TOL if counts[e] else np.all(dW13[e] == 0)

    # combine of the routed input gradients
    assert_bytes_equal(bits(s["dX"]), moe.unpermute(bits(s["dxp"]), dst, None, T, k), "dX")

    # the layer entry points reproduce the staged pipeline bit for bit
    W13t = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    wq = m.moe_layer_prep_weights(W13t, inp["W2"])
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if router == "logits":
        out, ids2, gate2 = m.moe_layer_fwd(inp["x"], wq, d, ws, logits=inp["logits"], dev_status=st)
    else:
        out, ids2, gate2 = m.moe_layer_fwd(inp["x"], wq, d, ws, ids=inp["ids"], gate=inp["gate"], dev_status=st)
    dX, dW13l, dW2l, dgl = m.moe_layer_bwd(inp["x"], inp["dOut"], gate2, wq, d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, s["out"]) and torch.equal(dX, s["dX"])
    assert torch.equal(dW13l, s["dW13"]) and torch.equal(dW2l, s["dW2"]) and torch.equal(dgl, s["d_gate"])


def test_layer_end_to_end_vs_independent_oracle(dev):
    """No teacher forcing: the GPU layer against the oracle's own MXFP8 chain
    (relative error reported, bounded by the rare E4M3 rounding flips), and the
    MXFP8 error against the unquantized fp64 layer, as SQNR."""
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.TINY_LAYER
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    inp = workloads.layer_inputs(dims, seed=0, device=dev)
    W13t = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    wq = m.moe_layer_prep_weights(W13t, inp["W2"])
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    out, _, _ = m.moe_layer_fwd(inp["x"], wq, d, ws, ids=inp["ids"], gate=inp["gate"])
    dX, dW13, dW2, dg = m.moe_layer_bwd(inp["x"], inp["dOut"], inp["gate"], wq, d, ws)
    torch.cuda.synchronize()
    b = {n: bits(inp[n]) for n in ("x", "W1", "W3", "W2", "dOut")}
    ids = inp["ids"].cpu().numpy()
    gate = inp["gate"].cpu().numpy()
    fq = moe.layer_forward(b["x"], b["W1"], b["W3"], b["W2"], ids, gate, quant=True)
    bq = moe.layer_backward(fq, b["x"], b["W1"], b["W3"], b["W2"], b["dOut"])
    fr = moe.layer_forward(b["x"], b["W1"], b["W3"], b["W2"], ids, gate, quant=False)
    br = moe.layer_backward(fr, b["x"], b["W1"], b["W3"], b["W2"], b["dOut"])
    got = {"out": out.float().cpu().numpy(), "dX": dX.float().cpu().numpy(),
           "dW13": dW13.cpu().numpy(), "dW2": dW2.cpu().numpy()}
    refq = {"out": fq["out"], "dX": bq["dX"], "dW13": np.concatenate([bq["dW1"], bq["dW3"]], 2), "dW2": bq["dW2"]}
    refr = {"out": fr["out"], "dX": br["dX"], "dW13": np.concatenate([br["dW1"], br["dW3"]], 2), "dW2": br["dW2"]}
    for n in got:
        e = rel_frob(got[n], refq[n])
        sqnr = 10 * np.log10(np.sum(refr[n] ** 2) / np.sum((refr[n] - got[n]) ** 2))
        print(f"{n}: rel err vs MXFP8 oracle {e:.2e}, SQNR vs unquantized layer {sqnr:.1f} dB")
        assert e < 1e-3, n
        assert sqnr > 20, n


def test_layer_with_empty_experts(dev):
    """Experts 1, 4 and 5 of 6 receive no token (ids drawn from {0, 2, 3}),
    gates U(0.5, 1): their weight gradients are exactly zero, and the layer
    matches the independent MXFP8 oracle chain as in the end-to-end test."""
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.LayerDims(T=256, H=256, E=6, F=256, k=1)
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    inp = workloads.layer_inputs(dims, seed=4, device=dev)
    g = np.random.default_rng(4)
    ids_np = np.array([0, 2, 3], np.int32)[g.integers(0, 3, (dims.T, 1))]
    gate_np = g.uniform(0.5, 1.0, (dims.T, 1)).astype(np.float32)
    ids = torch.from_numpy(ids_np).to(dev)
    gate = torch.from_numpy(gate_np).to(dev)
    W13t = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    wq = m.moe_layer_prep_weights(W13t, inp["W2"])
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    out, _, _ = m.moe_layer_fwd(inp["x"], wq, d, ws, ids=ids, gate=gate)
    dX, dW13, dW2, dg = m.moe_layer_bwd(inp["x"], inp["dOut"], gate, wq, d, ws)
    torch.cuda.synchronize()
    for e in (1, 4, 5):
        assert torch.all(dW13[e] == 0) and torch.all(dW2[e] == 0), e
    b = {n: bits(inp[n]) for n in ("x", "W1", "W3", "W2", "dOut")}
    fq = moe.layer_forward(b["x"], b["W1"], b["W3"], b["W2"], ids_np, gate_np, quant=True)
    bq = moe.layer_backward(fq, b["x"], b["W1"], b["W3"], b["W2"], b["dOut"])
    got = {"out": out.float().cpu().numpy(), "dX": dX.float().cpu().numpy(),
           "dW13": dW13.cpu().numpy()[[0, 2, 3]], "dW2": dW2.cpu().numpy()[[0, 2, 3]]}
    ref = {"out": fq["out"], "dX": bq["dX"], "dW13": np.concatenate([bq["dW1"], bq["dW3"]], 2)[[0, 2, 3]],
           "dW2": bq["dW2"][[0, 2, 3]]}
    for n in got:
        assert rel_frob(got[n], ref[n]) < 1e-3, n


@pytest.mark.parametrize("rows,F", [(128, 96), (384, 32), (256, 160)])
def test_swiglu_bwd_standalone(dev, rows, F):
    """moe_swiglu_bwd on widths the layer never uses (F a multiple of 32 but
    not of 256) with N(0,1) a, b and dh: [da|db] and h quantized both ways
    against the fp64 SwiGLU backward of the same bf16 a, b and fp32 dh
    (margin rule at E4M3 rounding boundaries)."""
    import mxfp8_mixture_experts_gb300 as m
    g = workloads.generator(rows + F, dev)
    ab = workloads.randn_bf16((rows, 2 * F), 1.0, g, dev)
    dh = torch.randn((rows, F), generator=g, device=dev)
    dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs = m.moe_swiglu_bwd(dh, ab)
    torch.cuda.synchronize()
    abv = mx.bf16_to_f64(bits(ab))
    da, db = moe.swiglu_bwd(dh.cpu().numpy().astype(np.float64), abv[:, :F], abv[:, F:])
    dab = np.concatenate([da, db], axis=1)
    h = moe.swiglu(abv[:, :F], abv[:, F:])
    quant_mismatches_outside_margin(u8(dab_rq), mx.unswizzle_scales(u8(dab_rs), rows, 2 * F // 32), dab, "dab rows")
    quant_mismatches_outside_margin(u8(dab_cq), mx.unswizzle_scales(u8(dab_cs), 2 * F, rows // 32), dab.T.copy(),
                                    "dab cols")
    quant_mismatches_outside_margin(u8(h_cq), mx.unswizzle_scales(u8(h_cs), F, rows // 32), h.T.copy(), "h cols")


def test_swiglu_bwd_scales_at_any_byte(dev):
    """moe_swiglu_bwd writes every scale byte on its own, so its three scale
    arrays may start at any byte: with dab_rs, dab_cs and h_cs placed 1, 2
    and 3 bytes past a 16-byte boundary, every output is bit-identical to
    the call with aligned scale arrays, and the bytes before each array are
    untouched."""
    import mxfp8_mixture_experts_gb300 as m
    L = m.lib()
    s = torch.cuda.current_stream(dev).cuda_stream
    R, F = 256, 96
    g = workloads.generator(33, dev)
    ab = workloads.randn_bf16((R, 2 * F), 1.0, g, dev)
    dh = torch.randn((R, F), generator=g, device=dev)
    sb = lambda r, c: m.mx_scale_bytes(r, c, m.MX_SCALE_SWIZZLED)
    sizes = {"dab_rq": R * 2 * F, "dab_rs": sb(R, 2 * F), "dab_cq": 2 * F * R, "dab_cs": sb(2 * F, R),
             "h_cq": F * R, "h_cs": sb(F, R)}
    shift = {"dab_rq": 0, "dab_rs": 1, "dab_cq": 0, "dab_cs": 2, "h_cq": 0, "h_cs": 3}

    def run(offsets):
        bufs = {n: torch.full((k + 16,), 0xAB, dtype=torch.uint8, device=dev) for n, k in sizes.items()}
        assert L.moe_swiglu_bwd(dh.data_ptr(), ab.data_ptr(), R, F, 0,
                                *(bufs[n].data_ptr() + offsets[n] for n in sizes), None, s) == 0
        return bufs

    ref, shifted = run({n: 0 for n in sizes}), run(shift)
    torch.cuda.synchronize()
    for n, k in sizes.items():
        o = shift[n]
        assert np.array_equal(u8(shifted[n])[o:o + k], u8(ref[n])[:k]), n
        assert np.all(u8(shifted[n])[:o] == 0xAB), n


def test_row_limit_skips_rows_past_the_groups(dev):
    """moe_swiglu_bwd and moe_gather_quant with a device row limit (the layer
    passes offsets[E], where the routed rows end): every output of a row
    below the limit is bit-identical to the unlimited call, and nothing at or
    past it is written (buffers pre-filled with 0xAB keep that byte)."""
    import mxfp8_mixture_experts_gb300 as m
    L = m.lib()
    s = torch.cuda.current_stream(dev).cuda_stream
    R, F, P = 512, 256, 256
    g = workloads.generator(21, dev)
    ab = workloads.randn_bf16((R, 2 * F), 1.0, g, dev)
    dh = torch.randn((R, F), generator=g, device=dev)
    lim = torch.tensor([P], dtype=torch.int32, device=dev)
    sb = lambda r, c: m.mx_scale_bytes(r, c, m.MX_SCALE_SWIZZLED)
    shapes = {"dab_rq": R * 2 * F, "dab_rs": sb(R, 2 * F), "dab_cq": 2 * F * R, "dab_cs": sb(2 * F, R),
              "h_cq": F * R, "h_cs": sb(F, R)}

    def run(limit):
        o = {n: torch.full((k,), 0xAB, dtype=torch.uint8, device=dev) for n, k in shapes.items()}
        assert L.moe_swiglu_bwd(dh.data_ptr(), ab.data_ptr(), R, F, 0, *(o[n].data_ptr() for n in shapes),
                                None if limit is None else limit.data_ptr(), s) == 0
        return o

    full, part = run(None), run(lim)
    torch.cuda.synchronize()

    def col_scale_mask(rows, cols_blocks):
        rr, cc = np.meshgrid(np.arange(rows), np.arange(cols_blocks), indexing="ij")
        mask = np.zeros(sb(rows, cols_blocks * 32), bool)
        mask[mx.swizzled_offset(rr, cc, cols_blocks)[cc < P // 32]] = True
        return mask

    f, p_ = {n: u8(t) for n, t in full.items()}, {n: u8(t) for n, t in part.items()}
    below = {"dab_rq": np.arange(R * 2 * F) < P * 2 * F,
             "dab_rs": np.arange(sb(R, 2 * F)) < sb(P, 2 * F),
             "dab_cq": (np.arange(2 * F * R) % R) < P, "dab_cs": col_scale_mask(2 * F, R // 32),
             "h_cq": (np.arange(F * R) % R) < P, "h_cs": col_scale_mask(F, R // 32)}
    for n in shapes:
        assert np.array_equal(p_[n][below[n]], f[n][below[n]]), n
        assert np.all(p_[n][~below[n]] == 0xAB), n

    # gather + quantize, both layouts
    T, H, k = 300, 256, 1
    x = workloads.randn_bf16((T, H), 1.0, g, dev)
    src = torch.full((R,), -1, dtype=torch.int32, device=dev)
    src[:T] = torch.arange(T, dtype=torch.int32, device=dev)
    shapes = {"q_row": R * H, "s_row": sb(R, H), "q_col": H * R, "s_col": sb(H, R)}

    def gq(limit):
        o = {n: torch.full((k_,), 0xAB, dtype=torch.uint8, device=dev) for n, k_ in shapes.items()}
        assert L.moe_gather_quant(x.data_ptr(), None, src.data_ptr(), T, H, k, R, m.MX_MODE_BOTH, 0,
                                  *(o[n].data_ptr() for n in shapes), None if limit is None else limit.data_ptr(),
                                  s) == 0
        return o

    full, part = gq(None), gq(lim)
    torch.cuda.synchronize()
    f, p_ = {n: u8(t) for n, t in full.items()}, {n: u8(t) for n, t in part.items()}
    below = {"q_row": np.arange(R * H) < P * H, "s_row": np.arange(sb(R, H)) < sb(P, H),
             "q_col": (np.arange(H * R) % R) < P, "s_col": col_scale_mask(H, R // 32)}
    for n in shapes:
        assert np.array_equal(p_[n][below[n]], f[n][below[n]]), n
        assert np.all(p_[n][~below[n]] == 0xAB), n


def test_layer_empty_batch(dev):
    """T = 0 through moe_layer_fwd/bwd: no error, zero weight gradients."""
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.LayerDims(T=0, H=256, E=4, F=256, k=1)
    d = m.MoELayerDims(T=0, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    g = workloads.generator(2, dev)
    W13 = workloads.randn_bf16((dims.E, dims.H, 2 * dims.F), 0.02, g, dev)
    W2 = workloads.randn_bf16((dims.E, dims.F, dims.H), 0.02, g, dev)
    wq = m.moe_layer_prep_weights(W13, W2)
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    x = torch.empty((0, dims.H), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, ids, gate = m.moe_layer_fwd(x, wq, d, ws, logits=torch.empty((0, dims.E), device=dev), dev_status=st)
    dX, dW13, dW2, dg = m.moe_layer_bwd(x, x, gate, wq, d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert out.shape == (0, dims.H) and dX.shape == (0, dims.H)
    assert bool(torch.all(dW13 == 0)) and bool(torch.all(dW2 == 0))


def test_bounded_wait_reports_timeout_and_context_survives():
    """The device failure path: a bounded wait on an mbarrier that nothing
    arrives on expires after 20 ms and reports MX_ERR_TIMEOUT; the context
    stays usable (a quantize right after it is still bit-exact)."""
    import mxfp8_mixture_experts_gb300 as m
    from mxfp8_mixture_experts_gb300 import _lib
    from oracle import mx as omx
    dev = torch.device("cuda", 0)
    L = m.lib()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    assert L.mx_selftest_wait_timeout(20_000_000, st.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.MX_ERR_TIMEOUT
    assert L.mx_selftest_wait_timeout(0, st.data_ptr(), s) == _lib.MX_ERR_INVALID_ARG
    assert L.mx_selftest_wait_timeout(10**9, st.data_ptr(), s) == _lib.MX_ERR_INVALID_ARG
    x = workloads.quantize_input(64, 128, seed=4, device=dev)
    q, sc, _, _ = m.mx_quantize(x, m.MX_MODE_ROW, m.MX_SCALE_PLAIN)
    torch.cuda.synchronize()
    qr, sr = omx.quantize_rows(omx.bf16_to_f64(workloads.bf16_bits(x)))
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(sc.cpu().numpy().reshape(sr.shape), sr)


def test_layer_is_deterministic():
    """Two runs of the layer forward and backward on the same inputs give
    bit-identical outputs (no atomics and fixed reduction orders)."""
    import mxfp8_mixture_experts_gb300 as m
    dev = torch.device("cuda", 0)
    d = m.MoELayerDims(T=512, H=256, F=512, E=4, k=2)
    inp = workloads.layer_inputs(workloads.LayerDims(T=d.T, H=d.H, E=d.E, F=d.F, k=d.k), seed=9, device=dev,
                                 router="logits")
    W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()

    def run():
        wq = m.moe_layer_prep_weights(W13, inp["W2"])
        ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
        out, ids, gate = m.moe_layer_fwd(inp["x"], wq, d, ws, logits=inp["logits"])
        dX, dW13, dW2, dg = m.moe_layer_bwd(inp["x"], inp["dOut"], gate, wq, d, ws)
        torch.cuda.synchronize()
        return [t.clone() for t in (out, ids, gate, dX, dW13, dW2, dg)]

    a, b = run(), run()
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.uint8) if u.dtype != torch.int32 else u,
                           v.view(torch.uint8) if v.dtype != torch.int32 else v)


def test_layer_bf16_weight_gradients():
    """wgrad_dtype = MX_OUT_BF16: the weight gradients are the fp32 ones of
    the default run rounded once to bf16 (round to nearest even), bit for
    bit, since both runs accumulate the same products in the same order and
    only the epilogue rounds; dX and d_gate are unchanged."""
    import mxfp8_mixture_experts_gb300 as m
    dev = torch.device("cuda", 0)
    d = m.MoELayerDims(T=512, H=256, F=512, E=4, k=2)
    inp = workloads.layer_inputs(workloads.LayerDims(T=d.T, H=d.H, E=d.E, F=d.F, k=d.k), seed=17, device=dev,
                                 router="logits")
    W13 = torch.cat([inp["W1"], inp["W3"]], dim=2).contiguous()
    wq = m.moe_layer_prep_weights(W13, inp["W2"])
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _, _, gate = m.moe_layer_fwd(inp["x"], wq, d, ws, logits=inp["logits"], dev_status=st)
    f32 = m.moe_layer_bwd(inp["x"], inp["dOut"], gate, wq, d, ws, dev_status=st)
    f32 = [t.clone() for t in f32]
    b16 = m.moe_layer_bwd(inp["x"], inp["dOut"], gate, wq, d, ws, dev_status=st, wgrad_dtype=m.MX_OUT_BF16)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert b16[1].dtype == torch.bfloat16 and b16[2].dtype == torch.bfloat16
    for got, ref, what in ((b16[1], f32[1], "dW13"), (b16[2], f32[2], "dW2")):
        assert torch.equal(got.view(torch.int16), ref.to(torch.bfloat16).view(torch.int16)), what
    assert torch.equal(b16[0].view(torch.int16), f32[0].view(torch.int16))
    assert torch.equal(b16[3], f32[3])


def test_layer_replays_from_a_cuda_graph():
    """The layer API makes no host synchronisation and keeps the group sizes
    on the device, so weight prep, forward and backward can be captured into
    one CUDA graph.  Replays match eager calls bit for bit, and a replay after
    new inputs are copied into the captured buffers computes on those inputs
    (nothing is frozen at capture time but the buffers' addresses)."""
    import mxfp8_mixture_experts_gb300 as m
    dev = torch.device("cuda", 0)
    d = m.MoELayerDims(T=512, H=256, F=512, E=4, k=2)
    dims = workloads.LayerDims(T=d.T, H=d.H, E=d.E, F=d.F, k=d.k)
    inputs = [workloads.layer_inputs(dims, seed=s, device=dev, router="logits") for s in (13, 14)]
    W13 = [torch.cat([i["W1"], i["W3"]], dim=2).contiguous() for i in inputs]

    def eager(i):
        wq = m.moe_layer_prep_weights(W13[i], inputs[i]["W2"])
        ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
        out, ids, gate = m.moe_layer_fwd(inputs[i]["x"], wq, d, ws, logits=inputs[i]["logits"])
        dX, dW13, dW2, dg = m.moe_layer_bwd(inputs[i]["x"], inputs[i]["dOut"], gate, wq, d, ws)
        torch.cuda.synchronize()
        return [t.clone() for t in (out, ids, gate, dX, dW13, dW2, dg)]

    ref = [eager(0), eager(1)]
    # static buffers, filled with the first inputs
    sx, slog, sdo = inputs[0]["x"].clone(), inputs[0]["logits"].clone(), inputs[0]["dOut"].clone()
    sW13, sW2 = W13[0].clone(), inputs[0]["W2"].clone()
    wq = torch.empty(m.moe_layer_weights_size(d.H, d.F, d.E), dtype=torch.uint8, device=dev)
    ws = torch.empty(m.moe_layer_workspace_size(d), dtype=torch.uint8, device=dev)
    out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((d.T, d.k), dtype=torch.int32, device=dev)
    gate = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
    dX = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
    dW13 = torch.empty((d.E, d.H, 2 * d.F), dtype=torch.float32, device=dev)
    dW2 = torch.empty((d.E, d.F, d.H), dtype=torch.float32, device=dev)
    dg = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        m.moe_layer_prep_weights(sW13, sW2, wq)
        m.moe_layer_fwd(sx, wq, d, ws, logits=slog, ids=ids, gate=gate, out=out, dev_status=st)
        m.moe_layer_bwd(sx, sdo, gate, wq, d, ws, dX=dX, dW13=dW13, dW2=dW2, d_gate=dg, dev_status=st)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()  # warm-up on the capture stream's side (one-time set-up happens here)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for i in (0, 1, 0):
        sx.copy_(inputs[i]["x"]); slog.copy_(inputs[i]["logits"]); sdo.copy_(inputs[i]["dOut"])
        sW13.copy_(W13[i]); sW2.copy_(inputs[i]["W2"])
        for t in (out, dX, dW13, dW2, dg):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for u, v in zip((out, ids, gate, dX, dW13, dW2, dg), ref[i]):
            assert torch.equal(u.view(torch.uint8) if u.dtype != torch.int32 else u,
                               v.view(torch.uint8) if v.dtype != torch.int32 else v)


# ---------------------------------------------------------------------------
# full-size layer (T=16384, H=5120, E=16, F=8192, top-1 softmax router): every
# stage checked on sampled outputs that the oracle computes one at a time, on
# the GPU's own inputs to that stage
# ---------------------------------------------------------------------------
def _rows_u8(t, rows):
    return t[torch.as_tensor(np.asarray(rows), device=t.device)].cpu().numpy().astype(np.uint8)


def _deq_sampled(q_rows, s_flat, rows, ncols):
    """Dequantize sampled rows of an MXFP8 matrix with ncols columns whose
    scales are in the swizzled layout (flat numpy array)."""
    cb = ncols // 32
    rr, cc = np.meshgrid(np.asarray(rows), np.arange(cb), indexing="ij")
    sc = s_flat[mx.swizzled_offset(rr, cc, cb)]
    return mx.dequantize_rows(q_rows, sc)


def _sampled_scales(s_flat, rows, ncols):
    cb = ncols // 32
    rr, cc = np.meshgrid(np.asarray(rows), np.arange(cb), indexing="ij")
    return s_flat[mx.swizzled_offset(rr, cc, cb)]


def _frob_check(got, ref, what, min_entries=64):
    """fp32 GEMM outputs on sampled entries against the fp64 products of the
    same dequantized operands: relative Frobenius error over the sample at
    most TOL, the bound the full matrices are held to."""
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape and got.size >= min_entries, (what, got.shape, ref.shape)
    e = rel_frob(got, ref)
    print(f"{what}: rel Frobenius {e:.2e} over {got.size} sampled entries")
    assert e <= TOL, f"{what}: rel Frobenius {e:.3e} > {TOL}"


def test_layer_full_size_sampled(dev):
    import mxfp8_mixture_experts_gb300 as m
    dims = workloads.FULL_LAYER
    d = m.MoELayerDims(T=dims.T, H=dims.H, F=dims.F, E=dims.E, k=dims.k)
    T, H, F, E, k = d.T, d.H, d.F, d.E, d.k
    inp = workloads.layer_inputs(dims, seed=0, device=dev, router="logits")
    s = _staged(dev, inp, d, inp["logits"])
    R = s["R"]
    g = np.random.default_rng(123)

    # router and grouping map: exact over all tokens
    ids_ref, gate_ref = moe.route(inp["logits"].cpu().numpy(), k)
    assert np.array_equal(s["ids"].cpu().numpy(), ids_ref)
    gate = s["gate"].cpu().numpy()
    np.testing.assert_allclose(gate, gate_ref, rtol=2e-6, atol=1e-9)
    counts, off, dst, src = moe.permute_map(ids_ref, E)
    assert np.array_equal(s["off"].cpu().numpy(), off)
    assert np.array_equal(s["dst"].cpu().numpy(), dst)
    P = int(off[E])
    assert np.array_equal(s["src"].cpu().numpy()[:P], src[:P])
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1       # expert of each padded row
    real = np.flatnonzero(src[:P] >= 0)

    x_bits = workloads.bf16_bits(inp["x"])
    W1b, W3b, W2b = (inp[n] for n in ("W1", "W3", "W2"))

    # permuted, quantized x: sampled rows bit-exact
    rows = np.sort(g.choice(real, 48, replace=False))
    xr = mx.bf16_to_f64(x_bits[src[rows] // k])
    q_ref, s_ref = mx.quantize_rows(xr)
    assert_bytes_equal(_rows_u8(s["xq"], rows), q_ref, "xq rows")
    xs_flat = u8(s["xs"])
    assert_bytes_equal(_sampled_scales(xs_flat, rows, H), s_ref, "xs rows")

    # GEMM1: a|b entries on the GPU's quantized x and the column-quantized W13 row
    xhat = _deq_sampled(_rows_u8(s["xq"], rows), xs_flat, rows, H)                 # [48, H]
    cols = g.choice(2 * F, 16, replace=False)
    ab_rows = bits(s["ab"][torch.as_tensor(rows, device=dev)])                      # [48, 2F]
    for c in cols:
        ex = e_of[rows]
        wcol = np.stack([mx.bf16_to_f64(workloads.bf16_bits(
            (W1b if c < F else W3b)[e, :, c % F].contiguous())) for e in ex])         # [48, H]
        wq, ws_ = mx.quantize_rows(wcol)                                               # blocks along H
        terms = xhat * mx.dequantize_rows(wq, ws_)
        assert_bf16_within_one_ulp(ab_rows[:, c], terms.sum(axis=1), f"a|b col {c}", mag=np.abs(terms).sum(axis=1),
                                   K=H)

    # fused SwiGLU -> h, quantized (teacher forced on the GPU's a, b)
    abv = mx.bf16_to_f64(ab_rows)
    h = moe.swiglu(abv[:, :F], abv[:, F:])
    hs_flat = u8(s["hs"])
    quant_mismatches_outside_margin(_rows_u8(s["hq"], rows), _sampled_scales(hs_flat, rows, F), h, "hq rows")

    # GEMM2: y entries on the GPU's h and the column-quantized W2 row
    hhat = _deq_sampled(_rows_u8(s["hq"], rows), hs_flat, rows, F)
    y_rows = bits(s["y"][torch.as_tensor(rows, device=dev)])
    for c in g.choice(H, 8, replace=False):
        wcol = np.stack([mx.bf16_to_f64(workloads.bf16_bits(W2b[e, :, c].contiguous())) for e in e_of[rows]])
        wq, ws_ = mx.quantize_rows(wcol)
        terms = hhat * mx.dequantize_rows(wq, ws_)
        assert_bf16_within_one_ulp(y_rows[:, c], terms.sum(axis=1), f"y col {c}", mag=np.abs(terms).sum(axis=1), K=F)

    # combine (top-1): out[t] = bf16(fp32(gate * y[dst[t]])), exact
    toks = g.choice(T, 64, replace=False)
    yv = mx.bf16_to_f64(bits(s["y"][torch.as_tensor(dst[toks], device=dev)])).astype(np.float32)
    want = mx.f32_to_bf16_bits((gate[toks, 0:1] * yv).astype(np.float32))
    assert_bytes_equal(bits(s["out"][torch.as_tensor(toks, device=dev)]).view(np.uint8),
                       want.view(np.uint8), "out")

    # gradient shuffle: dY rows = bf16(fp32(gate * dOut)), quantized both ways, exact
    dO_bits = workloads.bf16_bits(inp["dOut"])
    tok = src[rows] // k
    dY = mx.bf16_to_f64(mx.f32_to_bf16_bits((gate[tok, 0:1] * mx.bf16_to_f64(dO_bits[tok]).astype(np.float32))
                                            .astype(np.float32)))
    q_ref, s_ref = mx.quantize_rows(dY)
    assert_bytes_equal(_rows_u8(s["dy_rq"], rows), q_ref, "dY row q")
    dys_flat = u8(s["dy_rs"])
    assert_bytes_equal(_sampled_scales(dys_flat, rows, H), s_ref, "dY row s")
    # a column block of dY: 32 routed rows x one column
    blk = int(g.choice(P // 32)) * 32
    col = int(g.integers(H))
    brows = np.arange(blk, blk + 32)
    btok = src[brows]
    colvals = np.zeros(32)
    live = btok >= 0
    colvals[live] = mx.bf16_to_f64(mx.f32_to_bf16_bits(
        (gate[btok[live] // k, 0] * mx.bf16_to_f64(dO_bits[btok[live] // k, col]).astype(np.float32)).astype(np.float32)))
    q_ref, s_ref = mx.quantize_blocks(colvals)
    assert_bytes_equal(u8(s["dy_cq"][col, blk:blk + 32]), q_ref, "dY col block")
    assert int(u8(s["dy_cs"])[mx.swizzled_offset(col, blk // 32, R // 32)]) == int(s_ref)

    # dgrad2: dh entries on the GPU's dY and the row-quantized W2 row
    dyhat = _deq_sampled(_rows_u8(s["dy_rq"], rows), dys_flat, rows, H)
    dh_rows = s["dh"][torch.as_tensor(rows, device=dev)].cpu().numpy()
    fsel = g.choice(F, 8, replace=False)
    dh_ref = np.zeros((len(rows), len(fsel)))
    for i, f in enumerate(fsel):
        wrow = np.stack([mx.bf16_to_f64(workloads.bf16_bits(W2b[e, f, :].contiguous())) for e in e_of[rows]])
        wq, ws_ = mx.quantize_rows(wrow)
        dh_ref[:, i] = (dyhat * mx.dequantize_rows(wq, ws_)).sum(axis=1)
    _frob_check(dh_rows[:, fsel], dh_ref, "dh")

    # SwiGLU backward on the GPU's dh, a, b: row-quantized [da|db] (teacher forced)
    da, db = moe.swiglu_bwd(dh_rows.astype(np.float64), abv[:, :F], abv[:, F:])
    dab = np.concatenate([da, db], axis=1)
    quant_mismatches_outside_margin(_rows_u8(s["dab_rq"], rows), _sampled_scales(u8(s["dab_rs"]), rows, 2 * F),
                                    dab, "dab rows")

    # wgrad2 / wgrad1 on the GPU's column-quantized operands, for the expert
    # with the most routed rows and the one with the fewest (non-empty), 8 x 8
    # sampled entries of each weight gradient per expert:
    # dW2[e, f, c] = sum over its tokens of h[t, f] dY[t, c];
    # dW13[e, c, j] = sum over its tokens of xp[t, c] [da|db][t, j]
    sizes = np.diff(off)
    live = np.flatnonzero(sizes > 0)
    for e in sorted({int(live[np.argmax(sizes[live])]), int(live[np.argmin(sizes[live])])}):
        lo, hi = int(off[e]), int(off[e + 1])
        fs, cs, js = g.choice(F, 8, replace=False), g.choice(H, 8, replace=False), g.choice(2 * F, 8, replace=False)

        def col_rows(qname, sname, which):
            q = _rows_u8(s[qname], which)                                  # [n, R] transposed rows
            return _deq_sampled(q, u8(s[sname]), which, R)[:, lo:hi]

        hT, dyT = col_rows("h_cq", "h_cs", fs), col_rows("dy_cq", "dy_cs", cs)
        got = s["dW2"][e][torch.as_tensor(fs, device=dev)][:, torch.as_tensor(cs, device=dev)].cpu().numpy()
        _frob_check(got, hT @ dyT.T, f"dW2[{e}] ({hi - lo} rows)")
        xT, dabT = col_rows("xp_cq", "xp_cs", cs), col_rows("dab_cq", "dab_cs", js)
        got = s["dW13"][e][torch.as_tensor(cs, device=dev)][:, torch.as_tensor(js, device=dev)].cpu().numpy()
        _frob_check(got, xT @ dabT.T, f"dW13[{e}] ({hi - lo} rows)")

    # dgrad1: dxp entries on the GPU's row-quantized [da|db] and the row-quantized W13 row
    dabhat = _deq_sampled(_rows_u8(s["dab_rq"], rows), u8(s["dab_rs"]), rows, 2 * F)
    dxp_rows = bits(s["dxp"][torch.as_tensor(rows, device=dev)])
    for c in g.choice(H, 4, replace=False):
        wrow = np.stack([np.concatenate([mx.bf16_to_f64(workloads.bf16_bits(W1b[e_, c, :].contiguous())),
                                         mx.bf16_to_f64(workloads.bf16_bits(W3b[e_, c, :].contiguous()))])
                         for e_ in e_of[rows]])
        wq, ws_ = mx.quantize_rows(wrow)
        terms = dabhat * mx.dequantize_rows(wq, ws_)
        assert_bf16_within_one_ulp(dxp_rows[:, c], terms.sum(axis=1), f"dxp col {c}", mag=np.abs(terms).sum(axis=1),
                                   K=2 * F)

    # combine of dX (unit gates, top-1): dX[t] = dxp[dst[t]] exactly
    assert_bytes_equal(bits(s["dX"][torch.as_tensor(toks, device=dev)]).view(np.uint8),
                       bits(s["dxp"][torch.as_tensor(dst[toks], device=dev)]).view(np.uint8), "dX")
