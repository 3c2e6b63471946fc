"""Router, grouping map, token permute/unpermute, gather+quantize and the gate
gradient on the GPU vs the oracle.  Index, byte and bf16 results must be
bit-exact; fp32 reductions (softmax gate, gate gradient) within a stated
tolerance."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe, mx
from tests.helpers import assert_bytes_equal, bits, cuda_device, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def test_route(dev):
    import mxfp8_mixture_experts_gb300 as m
    g = workloads.generator(5, dev)
    for T, E, k in [(1, 1, 1), (1000, 16, 1), (777, 16, 4), (64, 256, 8)]:
        logits = torch.randn((T, E), generator=g, device=dev)
        if T > 10:
            logits[3, :] = 0.25                   # all tied: ids 0..k-1
            logits[7, 1] = logits[7, 0]           # tie for a top slot
        ids, gate = m.moe_route(logits, k)
        torch.cuda.synchronize()
        ids_ref, gate_ref = moe.route(logits.cpu().numpy(), k)
        assert_bytes_equal(ids.cpu().numpy(), ids_ref, "ids")
        np.testing.assert_allclose(gate.cpu().numpy(), gate_ref, rtol=2e-6, atol=1e-9)


def _map_check(dev, ids_np, E):
    import mxfp8_mixture_experts_gb300 as m
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(dev)
    counts, offsets, dst, src = m.moe_permute_map(ids, E)
    torch.cuda.synchronize()
    c, o, d, s = moe.permute_map(ids_np, E)
    assert_bytes_equal(counts.cpu().numpy(), c, "counts")
    assert_bytes_equal(offsets.cpu().numpy(), o, "offsets")
    assert_bytes_equal(dst.cpu().numpy(), d, "dst")
    src_h = src.cpu().numpy()
    assert_bytes_equal(src_h[: len(s)], s, "src")
    assert np.all(src_h[len(s):] == -1)
    return ids, counts, offsets, dst, src


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 3, 2), (1000, 16, 1), (3000, 16, 4), (4097, 7, 3)])
def test_permute_map(dev, T, E, k):
    g = np.random.default_rng(T + E + k)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)])
    _map_check(dev, ids, E)


def test_permute_map_full_size_zipf(dev):
    d = workloads.PERMUTE_DIMS
    g = workloads.generator(0, dev)
    ids = workloads.zipf_topk_ids(d["T"], d["E"], d["k"], d["E"] - 2, 1.1, g, dev)
    _, counts, _, _, _ = _map_check(dev, ids.cpu().numpy(), d["E"])
    assert int((counts == 0).sum()) == 2          # two experts stay empty


def test_permute_map_bad_id_sets_status(dev):
    import mxfp8_mixture_experts_gb300 as m
    ids = torch.tensor([[0], [5], [1]], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _, _, dst, _ = m.moe_permute_map(ids, 4, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == m._lib.MX_ERR_DEVICE
    assert dst.cpu().tolist()[1] == -1


@pytest.mark.parametrize("kind", ["fp8", "bf16", "bf16_quant"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("H", [256, 96])
def test_permute_rows(dev, kind, layout, H):
    """H = 256: scales move as 32-bit words (four blocks); H = 96 (three
    blocks a row, plain layout only): byte by byte."""
    import mxfp8_mixture_experts_gb300 as m
    if kind == "bf16" and layout == 1:
        pytest.skip("bf16 rows carry no scales")
    if H % 128 and layout == 1:
        pytest.skip("swizzled fp8 outputs need H % 128 == 0")
    T, E, k = 300, 6, 2
    inp = workloads.permute_inputs(T, H, E, k, seed=4, device=dev, live=5)
    ids_np = inp["ids"].cpu().numpy()
    _, _, _, dst, src = _map_check(dev, ids_np, E)
    c, o, d, s = moe.permute_map(ids_np, E)
    R = src.numel()
    xb = bits(inp["x"])
    xq, xs = mx.quantize_rows(mx.bf16_to_f64(xb))
    src_full = np.concatenate([s, -np.ones(R - len(s), np.int32)])
    if kind == "fp8":
        qr, sr, _, _ = m.mx_quantize(inp["x"], 1, 0)
        out, out_s = m.moe_permute(m.MX_PERMUTE_FP8, qr, dst, src, k, x_scales=sr, scale_layout=layout)
    elif kind == "bf16":
        out, out_s = m.moe_permute(m.MX_PERMUTE_BF16, inp["x"], dst, src, k)
    else:
        out, out_s = m.moe_permute(m.MX_PERMUTE_BF16_QUANT, inp["x"], dst, src, k, scale_layout=layout)
    torch.cuda.synchronize()
    if kind == "bf16":
        assert_bytes_equal(bits(out), moe.permute_rows(xb, src_full, k), "bf16 rows")
        return
    assert_bytes_equal(u8(out), moe.permute_rows(xq, src_full, k), "fp8 rows")
    sp = moe.permute_rows(xs, src_full, k)
    want_s = sp if layout == 0 else mx.swizzle_scales(sp)
    assert_bytes_equal(u8(out_s).reshape(want_s.shape), want_s, "scales")


def test_permute_full_size_sampled(dev):
    """T=32768, H=5120, E=16, top-4 Zipf: fused quantize+permute; 256 sampled
    tokens (all k destinations) and every pad row are checked."""
    import mxfp8_mixture_experts_gb300 as m
    d = workloads.PERMUTE_DIMS
    inp = workloads.permute_inputs(d["T"], d["H"], d["E"], d["k"], seed=0, device=dev)
    counts, offsets, dst, src = m.moe_permute_map(inp["ids"], d["E"])
    out, out_s = m.moe_permute(m.MX_PERMUTE_BF16_QUANT, inp["x"], dst, src, d["k"], scale_layout=1)
    torch.cuda.synchronize()
    g = np.random.default_rng(0)
    toks = np.sort(g.choice(d["T"], 256, replace=False))
    xq, xs = mx.quantize_rows(mx.bf16_to_f64(bits(inp["x"][torch.from_numpy(toks).to(dev)])))
    dst_h = dst.cpu().numpy().reshape(d["T"], d["k"])
    out_h = u8(out)
    sf = u8(out_s)
    nb = d["H"] // 32
    for j in range(d["k"]):
        rows = dst_h[toks, j]
        assert_bytes_equal(out_h[rows], xq, f"rows j={j}")
        rr, cc = np.meshgrid(rows, np.arange(nb), indexing="ij")
        assert_bytes_equal(sf[mx.swizzled_offset(rr, cc, nb)], xs, f"scales j={j}")
    pad = np.flatnonzero(src.cpu().numpy() < 0)
    assert np.all(out_h[pad] == 0)
    rr, cc = np.meshgrid(pad, np.arange(nb), indexing="ij")
    assert np.all(sf[mx.swizzled_offset(rr, cc, nb)] == 0)


@pytest.mark.parametrize("k", [1, 2, 4])
@pytest.mark.parametrize("with_gate", [True, False])
def test_unpermute(dev, k, with_gate):
    import mxfp8_mixture_experts_gb300 as m
    T, H, E = 500, 512, 8
    inp = workloads.permute_inputs(T, H, E, k, seed=k, device=dev, live=6)
    _, _, dst, src = m.moe_permute_map(inp["ids"], E)
    R = src.numel()
    y = workloads.randn_bf16((R, H), 1.0, workloads.generator(9, dev), dev)
    gate = inp["gate"] if with_gate else None
    out = m.moe_unpermute(y, dst, gate, T, k)
    torch.cuda.synchronize()
    ref = moe.unpermute(bits(y), dst.cpu().numpy(), None if gate is None else gate.cpu().numpy(), T, k)
    assert_bytes_equal(bits(out), ref, "combine")


@pytest.mark.parametrize("with_gate", [True, False])
def test_gather_quant(dev, with_gate):
    import mxfp8_mixture_experts_gb300 as m
    T, H, E, k = 400, 256, 5, 2
    inp = workloads.permute_inputs(T, H, E, k, seed=11, device=dev, live=5)
    _, _, dst, src = m.moe_permute_map(inp["ids"], E)
    gate = inp["gate"] if with_gate else None
    qr, sr, qc, sc = m.moe_gather_quant(inp["x"], gate, src, k, m.MX_MODE_BOTH)
    torch.cuda.synchronize()
    src_h = src.cpu().numpy()
    xb = bits(inp["x"])
    # the gathered matrix, built by the oracle's definitions: gate * x rounded to bf16
    Z = moe.permute_rows(mx.bf16_to_f64(xb).astype(np.float32), src_h, k)
    if with_gate:
        gsel = np.where(src_h >= 0, gate.cpu().numpy().reshape(-1)[np.maximum(src_h, 0)], 0).astype(np.float32)
        Z = (gsel[:, None] * Z).astype(np.float32)
    Z = mx.bf16_to_f64(mx.f32_to_bf16_bits(Z))
    q_ref, s_ref = mx.quantize_rows(Z)
    assert_bytes_equal(u8(qr), q_ref, "gather q_row")
    assert_bytes_equal(u8(sr), mx.swizzle_scales(s_ref), "gather s_row")
    qc_ref, sc_ref = mx.quantize_cols(Z)
    assert_bytes_equal(u8(qc), qc_ref, "gather q_col")
    assert_bytes_equal(u8(sc), mx.swizzle_scales(sc_ref), "gather s_col")


def test_gate_grad(dev):
    import mxfp8_mixture_experts_gb300 as m
    T, H, E, k = 300, 1024, 6, 3
    inp = workloads.permute_inputs(T, H, E, k, seed=2, device=dev)
    _, _, dst, src = m.moe_permute_map(inp["ids"], E)
    g = workloads.generator(3, dev)
    y = workloads.randn_bf16((src.numel(), H), 1.0, g, dev)
    dOut = workloads.randn_bf16((T, H), 1.0, g, dev)
    dg = m.moe_gate_grad(dOut, y, dst, k)
    torch.cuda.synchronize()
    yv = mx.bf16_to_f64(bits(y))
    dv = mx.bf16_to_f64(bits(dOut))
    rows = dst.cpu().numpy().reshape(T, k)
    ref = np.stack([np.sum(dv * yv[rows[:, j]], axis=1) for j in range(k)], axis=1)
    # fp32 accumulation of H = 1024 products: |err| <= ~H * 2^-24 * sum|terms|
    bound = 1024 * 2.0 ** -24 * np.stack([np.sum(np.abs(dv * yv[rows[:, j]]), axis=1) for j in range(k)], axis=1)
    assert np.all(np.abs(dg.cpu().numpy() - ref) <= bound)


def test_empty_batch(dev):
    """T = 0 through the token-indexed entry points: no error; the map marks
    every row a pad row, the permute and gather outputs are zero rows with
    zero scales, and the combine and gate gradient have nothing to do."""
    import mxfp8_mixture_experts_gb300 as m
    E, k, H = 4, 2, 256
    ids, gate = m.moe_route(torch.empty((0, E), device=dev), k)
    assert ids.shape == (0, k) and gate.shape == (0, k)
    counts, off, dst, src = m.moe_permute_map(ids, E)
    x = torch.empty((0, H), dtype=torch.bfloat16, device=dev)
    out, out_s = m.moe_permute(m.MX_PERMUTE_BF16_QUANT, x, dst, src, k, scale_layout=m.MX_SCALE_SWIZZLED)
    qr, sr, qc, sc = m.moe_gather_quant(x, gate, src, k, m.MX_MODE_BOTH)
    y = torch.zeros((src.numel(), H), dtype=torch.bfloat16, device=dev)
    comb = m.moe_unpermute(y, dst, gate, 0, k)
    dg = m.moe_gate_grad(x, y, dst, k)
    torch.cuda.synchronize()
    assert int(counts.sum()) == 0 and off.cpu().tolist() == [0] * (E + 1)
    assert src.numel() == m.moe_rows_cap(0, k, E) and bool(torch.all(src == -1))
    for t in (out, out_s, qr, sr, qc, sc):
        assert bool(torch.all(t == 0))
    assert comb.shape == (0, H) and dg.shape == (0, k)
