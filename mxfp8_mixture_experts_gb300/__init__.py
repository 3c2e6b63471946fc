"""GB300-native MXFP8 Mixture-of-Experts training hot path.

A thin Python binding over libmxmoe.so (C ABI: include/mxmoe.h).  Each
function here only marshals arguments: it allocates the output tensors with
torch on the inputs' device, passes raw pointers and the current CUDA stream
to the C entry point of the same name, and raises ``MxError`` on a non-zero
status.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and nothing here works without the
built library and an sm_103 GPU.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (MX_GEMM_DGRAD, MX_GEMM_FWD, MX_GEMM_WGRAD, MX_MODE_BOTH, MX_MODE_COL,  # noqa: F401
                   MX_MODE_ROW, MX_OUT_BF16, MX_OUT_F32, MX_PERMUTE_BF16, MX_PERMUTE_BF16_QUANT,
                   MX_PERMUTE_FP8, MX_SCALE_PLAIN, MX_SCALE_SWIZZLED, MX_ELEM_E4M3, MX_ELEM_E5M2, MxError)

__all__ = [
    "lib", "MxError", "mx_quantize", "mx_dequantize", "mx_scale_bytes", "moe_route", "moe_rows_cap", "moe_permute_map",
    "moe_permute", "moe_unpermute", "mx_grouped_gemm", "mx_grouped_gemm_wgrad_splitk", "moe_gemm1_swiglu", "moe_swiglu_bwd",
    "moe_gather_quant", "moe_gate_grad", "mx_selftest_sigmoid", "fp8_quantize_rowmax", "MoELayerDims", "moe_layer_prep_weights", "moe_layer_fwd",
    "moe_layer_bwd", "moe_layer_workspace_size", "moe_layer_weights_size",
]


def lib():
    return _lib.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(dev: torch.device):
    return torch.cuda.current_stream(dev).cuda_stream


def _req(t: torch.Tensor, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _u8(n, dev):
    return torch.empty(int(n), dtype=torch.uint8, device=dev)


def mx_scale_bytes(rows: int, cols: int, layout: int) -> int:
    return int(lib().mx_scale_bytes(rows, cols, layout))


def mx_quantize(x: torch.Tensor, mode: int = MX_MODE_ROW, scale_layout: int = MX_SCALE_PLAIN,
                elem: int = MX_ELEM_E4M3):
    """x bf16 [rows, cols] or [batch, rows, cols] -> (q_row, s_row, q_col, s_col);
    unused outputs are None.  q_col is [.., cols, rows].  elem: element format
    (MX_ELEM_E4M3 or MX_ELEM_E5M2)."""
    _req(x, torch.bfloat16, "x")
    batched = x.dim() == 3
    b, r, c = (x.shape if batched else (1, *x.shape))
    dev = x.device
    q_row = s_row = q_col = s_col = None
    lead = (b,) if batched else ()
    if mode & MX_MODE_ROW:
        q_row = torch.empty((*lead, r, c), dtype=torch.uint8, device=dev)
        s_row = _u8(b * mx_scale_bytes(r, c, scale_layout), dev)
    if mode & MX_MODE_COL:
        q_col = torch.empty((*lead, c, r), dtype=torch.uint8, device=dev)
        s_col = _u8(b * mx_scale_bytes(c, r, scale_layout), dev)
    _lib.check(lib().mx_quantize(_ptr(x), b, r, c, mode, scale_layout, elem, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                 _ptr(s_col), _stream(dev)), "mx_quantize")
    return q_row, s_row, q_col, s_col


def mx_dequantize(q: torch.Tensor, s: torch.Tensor, scale_layout: int = MX_SCALE_PLAIN,
                  out_dtype: int = MX_OUT_F32, elem: int = MX_ELEM_E4M3):
    """q uint8 [rows, cols] or [batch, rows, cols] with its scales -> fp32 or
    bf16 of the same shape."""
    _req(q, torch.uint8, "q")
    batched = q.dim() == 3
    b, r, c = (q.shape if batched else (1, *q.shape))
    out = torch.empty(q.shape, dtype=torch.float32 if out_dtype == MX_OUT_F32 else torch.bfloat16, device=q.device)
    _lib.check(lib().mx_dequantize(_ptr(q), _ptr(s), b, r, c, scale_layout, elem, out_dtype, _ptr(out),
                                   _stream(q.device)), "mx_dequantize")
    return out


def moe_route(logits: torch.Tensor, k: int):
    _req(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    gate = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _lib.check(lib().moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(gate), _stream(logits.device)), "moe_route")
    return ids, gate


def moe_rows_cap(T: int, k: int, E: int) -> int:
    return int(lib().moe_rows_cap(T, k, E))


def moe_permute_map(ids: torch.Tensor, E: int, rows_cap: int | None = None, dev_status: torch.Tensor | None = None):
    """ids int32 [T, k] -> (counts [E], offsets [E+1], dst [T*k], src [rows_cap])."""
    _req(ids, torch.int32, "ids")
    T, k = ids.shape
    dev = ids.device
    rows_cap = moe_rows_cap(T, k, E) if rows_cap is None else rows_cap
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    dst = torch.empty(T * k, dtype=torch.int32, device=dev)
    src = torch.empty(rows_cap, dtype=torch.int32, device=dev)
    wsb = int(lib().moe_permute_map_workspace_size(T, k, E))
    ws = _u8(max(wsb, 16), dev)
    _lib.check(lib().moe_permute_map(_ptr(ids), T, k, E, rows_cap, _ptr(counts), _ptr(offsets), _ptr(dst), _ptr(src),
                                     _ptr(ws), ws.numel(), _ptr(dev_status), _stream(dev)), "moe_permute_map")
    return counts, offsets, dst, src


def moe_permute(kind: int, x: torch.Tensor, dst: torch.Tensor, src: torch.Tensor, k: int,
                x_scales: torch.Tensor | None = None, scale_layout: int = MX_SCALE_SWIZZLED):
    """-> (out [rows_cap, H], out_scales or None)."""
    T, H = x.shape
    rows_cap = src.numel()
    dev = x.device
    if kind == MX_PERMUTE_BF16:
        out = torch.empty((rows_cap, H), dtype=torch.bfloat16, device=dev)
        out_s = None
    else:
        out = torch.empty((rows_cap, H), dtype=torch.uint8, device=dev)
        out_s = _u8(mx_scale_bytes(rows_cap, H, scale_layout), dev)
    _lib.check(lib().moe_permute(kind, _ptr(x), _ptr(x_scales), T, H, k, _ptr(dst), _ptr(src), rows_cap, _ptr(out),
                                 _ptr(out_s), scale_layout, _stream(dev)), "moe_permute")
    return out, out_s


def moe_unpermute(y: torch.Tensor, dst: torch.Tensor, gate: torch.Tensor | None, T: int, k: int,
                  out: torch.Tensor | None = None):
    _req(y, torch.bfloat16, "y")
    H = y.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device) if out is None else out
    _lib.check(lib().moe_unpermute(_ptr(y), _ptr(dst), _ptr(gate), T, H, k, _ptr(out), _stream(y.device)),
               "moe_unpermute")
    return out


def mx_grouped_gemm(op: int, A, sA, B, sB, offsets, E: int, M_cap: int, N: int, K: int,
                    out_dtype: int = MX_OUT_F32, out: torch.Tensor | None = None,
                    dev_status: torch.Tensor | None = None, elem_a: int = MX_ELEM_E4M3, elem_b: int = MX_ELEM_E4M3):
    """FWD/DGRAD: C [M_cap, N]; WGRAD: C [E, N, K] (see include/mxmoe.h)."""
    dev = A.device
    dt = torch.float32 if out_dtype == MX_OUT_F32 else torch.bfloat16
    if out is None:
        shape = (E, N, K) if op == MX_GEMM_WGRAD else (M_cap, N)
        out = torch.empty(shape, dtype=dt, device=dev)
    _lib.check(lib().mx_grouped_gemm(op, _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offsets), E, M_cap, N, K,
                                     _ptr(out), out_dtype, elem_a, elem_b, _ptr(dev_status), _stream(dev)),
               "mx_grouped_gemm")
    return out


def mx_grouped_gemm_wgrad_splitk(A, sA, B, sB, offsets, E: int, M_cap: int, N: int, K: int, splits: int,
                                 out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                                 dev_status: torch.Tensor | None = None, elem_a: int = MX_ELEM_E4M3,
                                 elem_b: int = MX_ELEM_E4M3):
    """Deterministic split-K wgrad: C fp32 [E, N, K] (see include/mxmoe.h)."""
    dev = A.device
    need = int(lib().mx_wgrad_splitk_workspace_size(E, N, K, splits))
    if need < 0:
        raise ValueError("bad split-K sizes")
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.float32, device=dev)
    _lib.check(lib().mx_grouped_gemm_wgrad_splitk(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offsets), E, M_cap, N,
                                                  K, splits, elem_a, elem_b, _ptr(ws), ws.numel(), _ptr(out),
                                                  _ptr(dev_status), _stream(dev)), "mx_grouped_gemm_wgrad_splitk")
    return out


def moe_gemm1_swiglu(A, sA, B, sB, offsets, E: int, M_cap: int, F: int, H: int,
                     dev_status: torch.Tensor | None = None):
    """-> (ab bf16 [M_cap, 2F], hq uint8 [M_cap, F], hs swizzled scales)."""
    dev = A.device
    ab = torch.empty((M_cap, 2 * F), dtype=torch.bfloat16, device=dev)
    hq = torch.empty((M_cap, F), dtype=torch.uint8, device=dev)
    hs = _u8(mx_scale_bytes(M_cap, F, MX_SCALE_SWIZZLED), dev)
    _lib.check(lib().moe_gemm1_swiglu(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offsets), E, M_cap, F, H, _ptr(ab),
                                      _ptr(hq), _ptr(hs), _ptr(dev_status), _stream(dev)), "moe_gemm1_swiglu")
    return ab, hq, hs


def moe_swiglu_bwd(dh: torch.Tensor, ab: torch.Tensor, row_limit: torch.Tensor | None = None,
                   grad_elem: int = MX_ELEM_E4M3):
    """-> (dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs), scales swizzled.
    row_limit: optional device int32 tensor whose first element bounds the
    rows processed (128-row bands at or past it are left unwritten)."""
    _req(dh, torch.float32, "dh")
    _req(ab, torch.bfloat16, "ab")
    rows, F = dh.shape
    dev = dh.device
    dab_rq = torch.empty((rows, 2 * F), dtype=torch.uint8, device=dev)
    dab_rs = _u8(mx_scale_bytes(rows, 2 * F, MX_SCALE_SWIZZLED), dev)
    dab_cq = torch.empty((2 * F, rows), dtype=torch.uint8, device=dev)
    dab_cs = _u8(mx_scale_bytes(2 * F, rows, MX_SCALE_SWIZZLED), dev)
    h_cq = torch.empty((F, rows), dtype=torch.uint8, device=dev)
    h_cs = _u8(mx_scale_bytes(F, rows, MX_SCALE_SWIZZLED), dev)
    _lib.check(lib().moe_swiglu_bwd(_ptr(dh), _ptr(ab), rows, F, grad_elem, _ptr(dab_rq), _ptr(dab_rs), _ptr(dab_cq),
                                    _ptr(dab_cs), _ptr(h_cq), _ptr(h_cs), _ptr(row_limit), _stream(dev)),
               "moe_swiglu_bwd")
    return dab_rq, dab_rs, dab_cq, dab_cs, h_cq, h_cs


def moe_gather_quant(x: torch.Tensor, gate, src: torch.Tensor, k: int, mode: int = MX_MODE_BOTH,
                     row_limit: torch.Tensor | None = None, elem: int = MX_ELEM_E4M3):
    """-> (q_row, s_row, q_col, s_col) of the gathered [rows_cap, H] matrix.
    row_limit: as in moe_swiglu_bwd."""
    _req(x, torch.bfloat16, "x")
    T, H = x.shape
    R = src.numel()
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if mode & MX_MODE_ROW:
        q_row = torch.empty((R, H), dtype=torch.uint8, device=dev)
        s_row = _u8(mx_scale_bytes(R, H, MX_SCALE_SWIZZLED), dev)
    if mode & MX_MODE_COL:
        q_col = torch.empty((H, R), dtype=torch.uint8, device=dev)
        s_col = _u8(mx_scale_bytes(H, R, MX_SCALE_SWIZZLED), dev)
    _lib.check(lib().moe_gather_quant(_ptr(x), _ptr(gate), _ptr(src), T, H, k, R, mode, elem, _ptr(q_row), _ptr(s_row),
                                      _ptr(q_col), _ptr(s_col), _ptr(row_limit), _stream(dev)), "moe_gather_quant")
    return q_row, s_row, q_col, s_col


def fp8_quantize_rowmax(x: torch.Tensor):
    """bf16 [rows, cols] -> (q uint8 [rows, cols] E4M3, row_scale fp32 [rows]):
    one scale per row, amax / 448 (see fp8_quantize_rowmax in mxmoe.h)."""
    _req(x, torch.bfloat16, "x")
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    s = torch.empty(rows, dtype=torch.float32, device=x.device)
    _lib.check(lib().fp8_quantize_rowmax(_ptr(x), rows, cols, _ptr(q), _ptr(s), _stream(x.device)),
               "fp8_quantize_rowmax")
    return q, s


def mx_selftest_sigmoid(a: torch.Tensor):
    """The SwiGLU kernels' fp32 sigmoid pieces on bf16 values a (any shape):
    -> (s, one_minus_sigma, back) fp32 tensors of a's shape, sigma = s * back."""
    _req(a, torch.bfloat16, "a")
    a = a.contiguous()
    out = torch.empty(a.shape + (3,), dtype=torch.float32, device=a.device)
    _lib.check(lib().mx_selftest_sigmoid(_ptr(a), a.numel(), _ptr(out), _stream(a.device)), "mx_selftest_sigmoid")
    return out[..., 0], out[..., 1], out[..., 2]


def moe_gate_grad(dOut: torch.Tensor, y: torch.Tensor, dst: torch.Tensor, k: int):
    T, H = dOut.shape
    d_gate = torch.empty((T, k), dtype=torch.float32, device=dOut.device)
    _lib.check(lib().moe_gate_grad(_ptr(dOut), _ptr(y), _ptr(dst), T, H, k, _ptr(d_gate), _stream(dOut.device)),
               "moe_gate_grad")
    return d_gate


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class MoELayerDims:
    T: int
    H: int
    F: int
    E: int
    k: int


def moe_layer_weights_size(H: int, F: int, E: int) -> int:
    return int(lib().moe_layer_weights_size(H, F, E))


def moe_layer_workspace_size(d: MoELayerDims) -> int:
    return int(lib().moe_layer_workspace_size(d.T, d.H, d.F, d.E, d.k))


def moe_layer_prep_weights(W13: torch.Tensor, W2: torch.Tensor, wq: torch.Tensor | None = None):
    """W13 bf16 [E, H, 2F], W2 bf16 [E, F, H] -> the quantized weight buffer."""
    _req(W13, torch.bfloat16, "W13")
    _req(W2, torch.bfloat16, "W2")
    E, H, F2 = W13.shape
    F = F2 // 2
    n = moe_layer_weights_size(H, F, E)
    wq = _u8(n, W13.device) if wq is None else wq
    _lib.check(lib().moe_layer_prep_weights(_ptr(W13), _ptr(W2), H, F, E, _ptr(wq), wq.numel(),
                                            _stream(W13.device)), "moe_layer_prep_weights")
    return wq


def moe_layer_fwd(x: torch.Tensor, wq: torch.Tensor, d: MoELayerDims, ws: torch.Tensor, *,
                  logits: torch.Tensor | None = None, ids: torch.Tensor | None = None,
                  gate: torch.Tensor | None = None, out: torch.Tensor | None = None,
                  dev_status: torch.Tensor | None = None):
    """Forward; with ``logits`` the router fills ``ids``/``gate`` (allocated here
    when not given).  Returns (out, ids, gate)."""
    _req(x, torch.bfloat16, "x")
    dev = x.device
    if logits is not None:
        ids = torch.empty((d.T, d.k), dtype=torch.int32, device=dev) if ids is None else ids
        gate = torch.empty((d.T, d.k), dtype=torch.float32, device=dev) if gate is None else gate
    out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) if out is None else out
    _lib.check(lib().moe_layer_fwd(_ptr(x), _ptr(logits), _ptr(ids), _ptr(gate), _ptr(wq), d.T, d.H, d.F, d.E, d.k,
                                   _ptr(ws), ws.numel(), _ptr(out), _ptr(dev_status), _stream(dev)), "moe_layer_fwd")
    return out, ids, gate


def moe_layer_bwd(x: torch.Tensor, dOut: torch.Tensor, gate, wq: torch.Tensor, d: MoELayerDims,
                  ws: torch.Tensor, *, dX=None, dW13=None, dW2=None, d_gate=None, want_d_gate: bool = True,
                  dev_status: torch.Tensor | None = None, grad_elem: int = MX_ELEM_E4M3,
                  wgrad_dtype: int = MX_OUT_F32):
    """Backward -> (dX bf16 [T,H], dW13 [E,H,2F], dW2 [E,F,H], d_gate fp32 [T,k] or None); the
    weight gradients are fp32 (wgrad_dtype MX_OUT_F32) or bf16 (MX_OUT_BF16)."""
    dev = x.device
    wdt = torch.float32 if wgrad_dtype == MX_OUT_F32 else torch.bfloat16
    dX = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) if dX is None else dX
    dW13 = torch.empty((d.E, d.H, 2 * d.F), dtype=wdt, device=dev) if dW13 is None else dW13
    dW2 = torch.empty((d.E, d.F, d.H), dtype=wdt, device=dev) if dW2 is None else dW2
    _req(dW13, wdt, "dW13")
    _req(dW2, wdt, "dW2")
    if want_d_gate and d_gate is None:
        d_gate = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
    _lib.check(lib().moe_layer_bwd(_ptr(x), _ptr(dOut), _ptr(gate), _ptr(wq), d.T, d.H, d.F, d.E, d.k, grad_elem,
                                   wgrad_dtype, _ptr(ws),
                                   ws.numel(), _ptr(dX), _ptr(dW13), _ptr(dW2), _ptr(d_gate), _ptr(dev_status),
                                   _stream(dev)), "moe_layer_bwd")
    return dX, dW13, dW2, d_gate
