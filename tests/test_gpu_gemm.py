"""Block-scaled grouped GEMM (tcgen05) on the GPU vs the oracle.

* small-integer operands with unit scales and all-ones data with varied
  scales: every product and sum is exact in fp32, so the GPU must be
  bit-exact (pins operand and scale layouts, group boundaries, K steps);
* random MXFP8 operands: relative Frobenius error <= 1e-4 against the fp64
  product of the dequantized operands (fp32 outputs); bf16 outputs within
  one bf16 ulp of the fp64 result;
* wgrad with an empty group (exact zeros) and the fused SwiGLU epilogue;
* the full-size grouped GEMM workload (E=8, 32768 rows, K=7168, N=2048) on
  sampled outputs, in the launch configuration the bench times."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe, mx
from tests.helpers import (assert_bf16_within_one_ulp, assert_bytes_equal, bits, cuda_device, quant_mismatches_outside_margin,
                           rel_frob, to_dev_u8, u8)

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _quant_operand(vals):
    """[..., R, K] values -> (codes [.., R, K], swizzled scales of (prod lead * R, K)), via the oracle."""
    v = np.asarray(vals, np.float64)
    R, K = v.shape[-2:]
    q, s = mx.quantize_rows(v.reshape(-1, K))
    return q.reshape(v.shape), mx.swizzle_scales(s)


def _deq(q, s_swz):
    q2 = q.reshape(-1, q.shape[-1])
    s = mx.unswizzle_scales(s_swz, q2.shape[0], q2.shape[1] // 32)
    return mx.dequantize_rows(q2, s).reshape(q.shape)


def _run_rows(dev, op, Aq, As, Bq, Bs, sizes, M_cap, N, K, out_dtype):
    import mxfp8_mixture_experts_gb300 as m
    E = len(sizes)
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    C = m.mx_grouped_gemm(op, to_dev_u8(Aq, dev), to_dev_u8(As, dev), to_dev_u8(Bq, dev), to_dev_u8(Bs, dev), off,
                          E, M_cap, N, K, out_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return C


def _ref_rows(Aq, As, Bq, Bs, sizes, M_cap):
    off = _offsets(sizes)
    return moe.grouped_gemm_rows(_deq(Aq, As), _deq(Bq, Bs), off)


SMALL_CODES = np.array([0x00, 0x30, 0x38, 0x40, 0xB0, 0xB8, 0xC0], np.uint8)   # 0, +-0.5, +-1, +-2


@pytest.mark.parametrize("sizes,N,K", [([128], 256, 128), ([128, 0, 256], 256, 256), ([256, 384, 128], 512, 640)])
def test_small_integer_operands_bit_exact(dev, sizes, N, K):
    g = np.random.default_rng(sum(sizes) + N + K)
    E = len(sizes)
    M_cap = sum(sizes) + 128
    Aq = g.choice(SMALL_CODES, (M_cap, K))
    Bq = g.choice(SMALL_CODES, (E, N, K))
    As = mx.swizzle_scales(np.full((M_cap, K // 32), 127, np.uint8))
    Bs = mx.swizzle_scales(np.full((E * N, K // 32), 127, np.uint8))
    C = _run_rows(dev, 0, Aq, As, Bq, Bs, sizes, M_cap, N, K, 1).cpu().numpy()
    ref = _ref_rows(Aq, As, Bq, Bs, sizes, M_cap)
    P = sum(sizes)
    assert_bytes_equal(C[:P].view(np.uint32), ref[:P].astype(np.float32).view(np.uint32), "C")


def _run_wgrad(dev, Xq, Xs, Yq, Ys, sizes, M_cap, N, K):
    import mxfp8_mixture_experts_gb300 as m
    E = len(sizes)
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    C = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, to_dev_u8(Xq, dev), to_dev_u8(Xs, dev), to_dev_u8(Yq, dev),
                          to_dev_u8(Ys, dev), off, E, M_cap, N, K, m.MX_OUT_F32, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return C.cpu().numpy()


# K = 256: the 256-wide part alone; 512: 256 + 128, then a 128-wide part in
# the first accumulator; 1280: three full 384-column super-tiles and a 128 rest
WGRAD_SHAPES = [([256, 0, 384], 256, 256), ([128, 256], 512, 512), ([384, 128, 0, 256], 256, 1280)]


@pytest.mark.parametrize("sizes,N,K", WGRAD_SHAPES)
def test_wgrad_small_integer_operands_bit_exact(dev, sizes, N, K):
    """Token-grouped contraction on codes {0, +-1/2, +-1, +-2} with unit
    scales: every product and partial sum is exact in fp32."""
    g = np.random.default_rng(sum(sizes) + N + K + 1)
    E = len(sizes)
    M_cap = sum(sizes) + 128
    Xq = g.choice(SMALL_CODES, (N, M_cap))
    Yq = g.choice(SMALL_CODES, (K, M_cap))
    Xs = mx.swizzle_scales(np.full((N, M_cap // 32), 127, np.uint8))
    Ys = mx.swizzle_scales(np.full((K, M_cap // 32), 127, np.uint8))
    C = _run_wgrad(dev, Xq, Xs, Yq, Ys, sizes, M_cap, N, K)
    ref = moe.grouped_gemm_tokens(_deq(Xq, Xs), _deq(Yq, Ys), _offsets(sizes))
    assert_bytes_equal(C.view(np.uint32), ref.astype(np.float32).view(np.uint32), "dW")


@pytest.mark.parametrize("sizes,N,K", WGRAD_SHAPES)
def test_wgrad_scale_layout_bit_exact(dev, sizes, N, K):
    """All-ones codes with every (row, 32-token block) scale drawn from
    2^-3..2^3 on both operands: each output is a sum of powers of two, exact
    in fp32, so a scale chunk fetched for the wrong rows or tokens shows."""
    g = np.random.default_rng(sum(sizes) + N + K + 2)
    E = len(sizes)
    M_cap = sum(sizes) + 128
    Xq = np.full((N, M_cap), 0x38, np.uint8)
    Yq = np.full((K, M_cap), 0x38, np.uint8)
    Xs = mx.swizzle_scales(g.integers(124, 131, (N, M_cap // 32)).astype(np.uint8))
    Ys = mx.swizzle_scales(g.integers(124, 131, (K, M_cap // 32)).astype(np.uint8))
    C = _run_wgrad(dev, Xq, Xs, Yq, Ys, sizes, M_cap, N, K)
    ref = moe.grouped_gemm_tokens(_deq(Xq, Xs), _deq(Yq, Ys), _offsets(sizes))
    assert_bytes_equal(C.view(np.uint32), ref.astype(np.float32).view(np.uint32), "dW")


def test_scale_layout_bit_exact(dev):
    """All-ones data, every (row, 32-block) scale drawn from 2^-3..2^3: C is a
    sum of K/32 powers of two, exact in fp32; a misplaced scale shows."""
    g = np.random.default_rng(2)
    sizes, N, K = [256, 128], 512, 512
    E, M_cap = 2, 384
    Aq = np.full((M_cap, K), 0x38, np.uint8)
    Bq = np.full((E, N, K), 0x38, np.uint8)
    As = mx.swizzle_scales(g.integers(124, 131, (M_cap, K // 32)).astype(np.uint8))
    Bs = mx.swizzle_scales(g.integers(124, 131, (E * N, K // 32)).astype(np.uint8))
    C = _run_rows(dev, 0, Aq, As, Bq, Bs, sizes, M_cap, N, K, 1).cpu().numpy()
    ref = _ref_rows(Aq, As, Bq, Bs, sizes, M_cap)
    assert_bytes_equal(C[:384].view(np.uint32), ref[:384].astype(np.float32).view(np.uint32), "C")


@pytest.mark.parametrize("out_dtype", [1, 0])
@pytest.mark.parametrize("sizes,N,K", [([384, 0, 128, 256], 256, 1024), ([128, 512], 768, 384),
                                       ([384, 0, 640], 1024, 256)])
def test_random_operands(dev, out_dtype, sizes, N, K):
    g = np.random.default_rng(7)
    E = len(sizes)
    M_cap = sum(sizes) + 256
    A = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, K))))
    W = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((E, N, K)) * 0.02))
    Aq, As = _quant_operand(A)
    Bq, Bs = _quant_operand(W)
    C = _run_rows(dev, 0, Aq, As, Bq, Bs, sizes, M_cap, N, K, out_dtype)
    ref = _ref_rows(Aq, As, Bq, Bs, sizes, M_cap)
    P = sum(sizes)
    if out_dtype == 1:
        assert rel_frob(C.cpu().numpy()[:P], ref[:P]) <= TOL
    else:
        mag = moe.grouped_gemm_rows(np.abs(_deq(Aq, As)), np.abs(_deq(Bq, Bs)), _offsets(sizes))
        assert_bf16_within_one_ulp(bits(C)[:P], ref[:P], "C bf16", mag=mag[:P], K=K)


@pytest.mark.parametrize("N,K", [(256, 512), (512, 768)])
def test_wgrad_with_empty_group(dev, N, K):
    """An even (K = 512) and an odd (K = 768) number of 256-wide column
    tiles, with an empty group in the middle."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(3)
    sizes = [256, 0, 128, 384]
    E = 4
    M_cap = sum(sizes) + 128
    X = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, N))))
    Y = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, K))))
    Xq, Xs = _quant_operand(X.T.copy())     # [N, M_cap], blocks along tokens
    Yq, Ys = _quant_operand(Y.T.copy())     # [K, M_cap]
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    C = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, to_dev_u8(Xq, dev), to_dev_u8(Xs, dev), to_dev_u8(Yq, dev),
                          to_dev_u8(Ys, dev), off, E, M_cap, N, K, m.MX_OUT_F32)
    torch.cuda.synchronize()
    ref = moe.grouped_gemm_tokens(_deq(Xq, Xs), _deq(Yq, Ys), _offsets(sizes))
    Ch = C.cpu().numpy()
    assert np.all(Ch[1] == 0)
    for e in (0, 2, 3):
        assert rel_frob(Ch[e], ref[e]) <= TOL


def test_all_groups_empty(dev):
    """offsets all zero: the row-grouped GEMM touches no output row (rows past
    offsets[E] are never written) and wgrad writes exact zeros for every
    expert; no device error either way."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(11)
    E, M_cap, N, K = 3, 256, 256, 256
    A = g.integers(0, 126, (M_cap, K), dtype=np.uint8)
    B = g.integers(0, 126, (E, N, K), dtype=np.uint8)
    As = mx.swizzle_scales(np.full((M_cap, K // 32), 127, np.uint8))
    Bs = mx.swizzle_scales(np.full((E * N, K // 32), 127, np.uint8))
    off = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    C = torch.full((M_cap, N), 7.0, device=dev)
    m.mx_grouped_gemm(m.MX_GEMM_FWD, to_dev_u8(A, dev), to_dev_u8(As, dev), to_dev_u8(B, dev), to_dev_u8(Bs, dev),
                      off, E, M_cap, N, K, m.MX_OUT_F32, out=C, dev_status=st)
    X = g.integers(0, 126, (N, M_cap), dtype=np.uint8)
    Y = g.integers(0, 126, (K, M_cap), dtype=np.uint8)
    Xs = mx.swizzle_scales(np.full((N, M_cap // 32), 127, np.uint8))
    Ys = mx.swizzle_scales(np.full((K, M_cap // 32), 127, np.uint8))
    W = torch.full((E, N, K), 7.0, device=dev)
    m.mx_grouped_gemm(m.MX_GEMM_WGRAD, to_dev_u8(X, dev), to_dev_u8(Xs, dev), to_dev_u8(Y, dev), to_dev_u8(Ys, dev),
                      off, E, M_cap, N, K, m.MX_OUT_F32, out=W, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.all(C == 7.0)
    assert torch.all(W == 0.0)


def test_bad_offsets_set_device_status(dev):
    import mxfp8_mixture_experts_gb300 as m
    A = torch.zeros((256, 128), dtype=torch.uint8, device=dev)
    As = torch.zeros(256 * 4, dtype=torch.uint8, device=dev)
    B = torch.zeros((1, 256, 128), dtype=torch.uint8, device=dev)
    Bs = torch.zeros(256 * 4, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    off = torch.tensor([0, 100], dtype=torch.int32, device=dev)      # not a multiple of 128
    C = torch.full((256, 256), 7.0, device=dev)
    m.mx_grouped_gemm(0, A, As, B, Bs, off, 1, 256, 256, 128, m.MX_OUT_F32, out=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == m._lib.MX_ERR_DEVICE
    assert torch.all(C == 7.0)


@pytest.mark.parametrize("F,sizes", [(256, [256, 0, 128]), (384, [256, 0, 128]), (512, [128] * 12 + [384])])
def test_gemm1_swiglu_fused(dev, F, sizes):
    """GEMM1 with the fused SwiGLU epilogue.  A group with an odd number of
    128-row tiles ends in a lone tile, which the CTA pair computes transposed
    with a and b in different CTAs; the last case makes almost every tile a
    lone tile, so each pair hands b across several lone tiles in a row."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(5)
    H = 512
    E = len(sizes)
    M_cap = sum(sizes) + 128
    x = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, H))))
    W13 = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((E, H, 2 * F)) * 0.05))
    Aq, As = _quant_operand(x)
    Bq, Bs = _quant_operand(np.swapaxes(W13, 1, 2).copy())     # [E, 2F, H], blocks along H
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    ab, hq, hs = m.moe_gemm1_swiglu(to_dev_u8(Aq, dev), to_dev_u8(As, dev), to_dev_u8(Bq, dev), to_dev_u8(Bs, dev),
                                    off, E, M_cap, F, H)
    torch.cuda.synchronize()
    P = sum(sizes)
    ref = moe.grouped_gemm_rows(_deq(Aq, As), _deq(Bq, Bs), _offsets(sizes))[:P]
    mag = moe.grouped_gemm_rows(np.abs(_deq(Aq, As)), np.abs(_deq(Bq, Bs)), _offsets(sizes))[:P]
    abb = bits(ab)[:P]
    assert_bf16_within_one_ulp(abb, ref, "a|b", mag=mag, K=H)
    # h from the GPU's own a, b (teacher forcing), fp64 SwiGLU, then the quantizer
    abv = mx.bf16_to_f64(abb)
    h = moe.swiglu(abv[:, :F], abv[:, F:])
    hs_plain = mx.unswizzle_scales(u8(hs), M_cap, F // 32)[:P]
    quant_mismatches_outside_margin(u8(hq)[:P], hs_plain, h, "h")


def _full_gemm_case(dev):
    d = workloads.GEMM_DIMS
    sizes = workloads.gemm_group_sizes(d["E"], d["M"], seed=0)
    inp = workloads.gemm_inputs(d["E"], d["M"], d["K"], d["N"], sizes, seed=0, device=dev)
    return d, sizes, inp


def test_full_size_grouped_gemm_sampled(dev):
    """E=8, 32768 routed rows in Zipf-sized groups (one empty), K=7168,
    N=2048: forward, dgrad and wgrad on the GPU-quantized operands; 256 x 256
    sampled outputs of each (all groups covered) against fp64."""
    import mxfp8_mixture_experts_gb300 as m
    d, sizes, inp = _full_gemm_case(dev)
    E, M, K, N = d["E"], d["M"], d["K"], d["N"]
    off_np = _offsets(sizes)
    off = torch.from_numpy(off_np).to(dev)
    g = np.random.default_rng(0)
    # forward: A [M, K] rows quantized along K; B = W^T [E, N, K] along K
    a_rq, a_rs, a_cq, a_cs = m.mx_quantize(inp["A"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    w_rq, w_rs, w_cq, w_cs = m.mx_quantize(inp["W"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)   # [E,K,N] / [E,N,K]
    c_rq, c_rs, c_cq, c_cs = m.mx_quantize(inp["dC"], m.MX_MODE_BOTH, m.MX_SCALE_SWIZZLED)
    C = m.mx_grouped_gemm(m.MX_GEMM_FWD, a_rq, a_rs, w_cq, w_cs, off, E, M, N, K, m.MX_OUT_F32)
    dA = m.mx_grouped_gemm(m.MX_GEMM_DGRAD, c_rq, c_rs, w_rq, w_rs, off, E, M, K, N, m.MX_OUT_F32)
    dW = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, c_cq, c_cs, a_cq, a_cs, off, E, M, N, K, m.MX_OUT_F32)
    torch.cuda.synchronize()

    def deq_rows(q, s, rows, inner):
        """dequantize selected rows of a row-quantized [R, inner] operand (swizzled scales)"""
        qh = u8(q.reshape(-1, inner)[torch.from_numpy(rows).to(dev)])
        sf = u8(s)
        rr, cc = np.meshgrid(rows, np.arange(inner // 32), indexing="ij")
        return mx.dequantize_rows(qh, sf[mx.swizzled_offset(rr, cc, inner // 32)])

    rows = np.sort(g.choice(M, 256, replace=False))
    grp = np.searchsorted(off_np, rows, side="right") - 1
    cols_n = np.sort(g.choice(N, 256, replace=False))
    cols_k = np.sort(g.choice(K, 256, replace=False))
    # forward
    Ar = deq_rows(a_rq, a_rs, rows, K)
    ref = np.empty((256, 256))
    for i, (r, e) in enumerate(zip(rows, grp)):
        Bsel = deq_rows(w_cq, w_cs, e * N + cols_n, K)
        ref[i] = Bsel @ Ar[i]
    rt = torch.from_numpy(rows).to(dev)
    got = C[rt][:, torch.from_numpy(cols_n).to(dev)].cpu().numpy()
    assert rel_frob(got, ref) <= TOL
    # dgrad: dA[r, k] = sum_n dC[r, n] W[e, k, n]
    Cr = deq_rows(c_rq, c_rs, rows, N)
    ref = np.empty((256, 256))
    for i, (r, e) in enumerate(zip(rows, grp)):
        Wsel = deq_rows(w_rq, w_rs, e * K + cols_k, N)
        ref[i] = Wsel @ Cr[i]
    got = dA[rt][:, torch.from_numpy(cols_k).to(dev)].cpu().numpy()
    assert rel_frob(got, ref) <= TOL
    # wgrad: dW[e, n, k] = sum over tokens of group e of dC[t, n] A[t, k]
    dWh = dW.cpu().numpy()
    for e in range(E):
        lo, hi = off_np[e], off_np[e + 1]
        if hi == lo:
            assert np.all(dWh[e] == 0)
            continue
        n_s = cols_n[:32]
        k_s = cols_k[:32]
        X = deq_rows(c_cq, c_cs, n_s, M)[:, lo:hi]
        Y = deq_rows(a_cq, a_cs, k_s, M)[:, lo:hi]
        assert rel_frob(dWh[e][np.ix_(n_s, k_s)], X @ Y.T) <= TOL


def test_one_cta_kernel_variant():
    """The one-CTA kernel (128 x 256 tiles, selected by MXMOE_GEMM_CTAS=1 at
    process start) passes the same GEMM tests in a child process."""
    import os
    import subprocess
    import sys
    if os.environ.get("MXMOE_GEMM_CTAS") == "1":
        pytest.skip("already running the one-CTA variant")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MXMOE_GEMM_CTAS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(root, "tests", "test_gpu_gemm.py"), "-q", "-x",
                        "-m", "gpu", "-k", "not one_cta and not full_size", "-p", "no:cacheprovider"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]



@pytest.mark.parametrize("splits", [1, 2, 3, 5])
def test_wgrad_splitk(dev, splits):
    """Deterministic split-K wgrad: groups of 128 tokens (fewer 128-token
    blocks than splits: some chunks empty), 0 and 1152 tokens; within 1e-4
    of the oracle, zeros for the empty group, bit-identical across two runs,
    and bit-identical to the unsplit GEMM when splits = 1; small-integer
    operands give exact sums in any order, so there every split is
    bit-exact."""
    import mxfp8_mixture_experts_gb300 as m
    g = np.random.default_rng(40 + splits)
    sizes, N, K = [1152, 0, 128, 640], 256, 768
    E, M_cap = len(sizes), sum(sizes) + 128
    off = torch.from_numpy(_offsets(sizes)).to(dev)
    X = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, N))))
    Y = mx.bf16_to_f64(mx.f64_to_bf16_bits(g.standard_normal((M_cap, K))))
    Xq, Xs = _quant_operand(X.T.copy())
    Yq, Ys = _quant_operand(Y.T.copy())
    args = [to_dev_u8(a, dev) for a in (Xq, Xs, Yq, Ys)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    C1 = m.mx_grouped_gemm_wgrad_splitk(*args, off, E, M_cap, N, K, splits, dev_status=st)
    C2 = m.mx_grouped_gemm_wgrad_splitk(*args, off, E, M_cap, N, K, splits, dev_status=st)
    ref_gpu = m.mx_grouped_gemm(m.MX_GEMM_WGRAD, *args, off, E, M_cap, N, K, m.MX_OUT_F32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    if splits == 1:
        assert torch.equal(C1.view(torch.int32), ref_gpu.view(torch.int32))
    ref = moe.grouped_gemm_tokens(_deq(Xq, Xs), _deq(Yq, Ys), _offsets(sizes))
    C = C1.cpu().numpy()
    assert np.all(C[1] == 0)
    for e in (0, 2, 3):
        assert rel_frob(C[e], ref[e]) <= TOL, e

    Xq = g.choice(SMALL_CODES, (N, M_cap))
    Yq = g.choice(SMALL_CODES, (K, M_cap))
    Xs = mx.swizzle_scales(np.full((N, M_cap // 32), 127, np.uint8))
    Ys = mx.swizzle_scales(np.full((K, M_cap // 32), 127, np.uint8))
    C = m.mx_grouped_gemm_wgrad_splitk(*[to_dev_u8(a, dev) for a in (Xq, Xs, Yq, Ys)], off, E, M_cap, N, K, splits)
    torch.cuda.synchronize()
    ref = moe.grouped_gemm_tokens(_deq(Xq, Xs), _deq(Yq, Ys), _offsets(sizes))
    assert_bytes_equal(C.cpu().numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32), "split-K exact")
