"""The C ABI library loads, exports every function include/mxmoe.h declares,
and rejects bad arguments on the host before touching a device.  CPU only:
no call here launches work."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxmoe.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?(?:mx_status|int64_t|int32_t|char)\s*\*?\s*(\w+)\s*\(", text, re.M))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_mixture_experts_gb300 import _lib, build
    build.build()
    return _lib.load()


def test_header_declares_the_scope_entry_points():
    names = _declared()
    for n in ("mx_quantize", "moe_route", "moe_permute_map", "moe_permute", "moe_unpermute", "mx_grouped_gemm",
              "moe_gemm1_swiglu", "moe_swiglu_bwd", "moe_layer_fwd", "moe_layer_bwd", "moe_layer_prep_weights"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    from mxfp8_mixture_experts_gb300 import _lib
    names = _declared()
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, 10):
        s = lib.mx_status_string(code).decode()
        assert s.startswith("MX_")
    assert lib.mx_abi_version() == 4


def test_size_queries(lib):
    assert lib.mx_scale_bytes(256, 7168, 0) == 256 * 224
    assert lib.mx_scale_bytes(130, 96, 1) == 256 * 4
    assert lib.mx_scale_bytes(10, 33, 0) == -1
    assert lib.moe_rows_cap(32768, 4, 16) == (32768 * 4 + 16 * 127 + 127) // 128 * 128
    assert lib.moe_layer_workspace_size(512, 256, 512, 4, 1) > 0
    assert lib.moe_layer_weights_size(256, 512, 4) >= 4 * 256 * 512 * 3


def test_host_side_argument_errors(lib):
    from mxfp8_mixture_experts_gb300 import _lib
    fake = C.c_void_p(1 << 20)        # never dereferenced: the checks fail first
    odd = C.c_void_p((1 << 20) + 4)
    # null input
    assert lib.mx_quantize(None, 1, 64, 64, 1, 0, 0, fake, fake, None, None, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_dequantize(None, fake, 1, 64, 64, 0, 0, 1, fake, None) == _lib.MX_ERR_INVALID_ARG
    # T = 0: the token arrays may be NULL (the argument checks pass; without a
    # GPU the device check then fails)
    assert lib.moe_route(None, 0, 4, 1, None, None, None) != _lib.MX_ERR_INVALID_ARG
    assert lib.moe_route(None, 5, 4, 1, None, None, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.moe_unpermute(None, None, None, 0, 64, 1, None, None) != _lib.MX_ERR_INVALID_ARG
    assert lib.mx_dequantize(fake, fake, 1, 64, 64, 2, 0, 1, fake, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_dequantize(fake, fake, 1, 64, 64, 0, 0, 5, fake, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_dequantize(fake, fake, 1, 64, 48, 0, 0, 1, fake, None) == _lib.MX_ERR_SHAPE
    assert lib.mx_dequantize(C.c_void_p((1 << 20) + 8), fake, 1, 64, 64, 0, 0, 1, fake, None) == _lib.MX_ERR_ALIGNMENT
    # unknown mode / layout
    assert lib.mx_quantize(fake, 1, 64, 64, 7, 0, 0, fake, fake, None, None, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_quantize(fake, 1, 64, 64, 1, 5, 0, fake, fake, None, None, None) == _lib.MX_ERR_INVALID_ARG
    # cols not a multiple of 32
    assert lib.mx_quantize(fake, 1, 64, 48, 1, 0, 0, fake, fake, None, None, None) == _lib.MX_ERR_SHAPE
    # misaligned
    assert lib.mx_quantize(odd, 1, 64, 64, 1, 0, 0, fake, fake, None, None, None) == _lib.MX_ERR_ALIGNMENT
    # GEMM shape rules
    assert lib.mx_grouped_gemm(0, fake, fake, fake, fake, fake, 4, 256, 200, 256, fake, 1, 0, 0, None, None) == \
        _lib.MX_ERR_SHAPE
    assert lib.mx_grouped_gemm(0, fake, fake, fake, fake, fake, 4, 100, 256, 256, fake, 1, 0, 0, None, None) == \
        _lib.MX_ERR_SHAPE
    assert lib.mx_grouped_gemm(9, fake, fake, fake, fake, fake, 4, 256, 256, 256, fake, 1, 0, 0, None, None) == \
        _lib.MX_ERR_INVALID_ARG
    assert lib.mx_grouped_gemm(0, fake, fake, fake, fake, fake, 0, 256, 256, 256, fake, 1, 0, 0, None, None) == \
        _lib.MX_ERR_INVALID_ARG
    # permute map: rows_cap too small, workspace too small
    assert lib.moe_permute_map(fake, 100, 2, 4, 128, fake, fake, fake, fake, fake, 1 << 20, None, None) == \
        _lib.MX_ERR_SHAPE
    assert lib.moe_permute_map(fake, 100, 2, 4, 1024, fake, fake, fake, fake, fake, 0, None, None) == \
        _lib.MX_ERR_WORKSPACE
    # layer: H must be a multiple of 256
    assert lib.moe_layer_fwd(fake, None, fake, None, fake, 16, 128, 256, 4, 1, fake, 1 << 40, fake, None, None) == \
        _lib.MX_ERR_SHAPE
    # route: k > E
    assert lib.moe_route(fake, 16, 4, 5, fake, fake, None) == _lib.MX_ERR_INVALID_ARG
    # row-max FP8: cols not a multiple of 16, too wide, misaligned scale
    assert lib.fp8_quantize_rowmax(fake, 4, 40, fake, fake, None) == _lib.MX_ERR_SHAPE
    assert lib.fp8_quantize_rowmax(fake, 4, 102416, fake, fake, None) == _lib.MX_ERR_SHAPE
    assert lib.fp8_quantize_rowmax(fake, 4, 64, fake, C.c_void_p((1 << 20) + 2), None) == _lib.MX_ERR_ALIGNMENT
    assert lib.fp8_quantize_rowmax(None, 4, 64, fake, fake, None) == _lib.MX_ERR_INVALID_ARG
    # split-K wgrad: splits out of range, E * splits > 1024, workspace too small
    big = lib.mx_wgrad_splitk_workspace_size(4, 256, 256, 2)
    assert big == 256 + 4 * 2 * 256 * 256 * 4
    assert lib.mx_wgrad_splitk_workspace_size(4, 256, 256, 17) == -1
    assert lib.mx_grouped_gemm_wgrad_splitk(fake, fake, fake, fake, fake, 4, 256, 256, 256, 0, 0, 0, fake, big, fake, None,
                                            None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_grouped_gemm_wgrad_splitk(fake, fake, fake, fake, fake, 512, 256, 256, 256, 4, 0, 0, fake, 1 << 40, fake,
                                            None, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_grouped_gemm_wgrad_splitk(fake, fake, fake, fake, fake, 4, 256, 256, 256, 2, 0, 0, fake, big - 1, fake,
                                            None, None) == _lib.MX_ERR_WORKSPACE
    assert lib.mx_grouped_gemm_wgrad_splitk(fake, fake, fake, fake, fake, 4, 256, 256, 384, 2, 0, 0, fake, 1 << 40, fake,
                                            None, None) == _lib.MX_ERR_SHAPE
    # element formats: only E4M3 (0) and E5M2 (1)
    assert lib.mx_quantize(fake, 1, 64, 64, 1, 0, 2, fake, fake, None, None, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_dequantize(fake, fake, 1, 64, 64, 0, 7, 1, fake, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_grouped_gemm(0, fake, fake, fake, fake, fake, 4, 256, 256, 256, fake, 1, 0, 3, None, None) == \
        _lib.MX_ERR_INVALID_ARG
    # sigmoid self-test: negative count, null buffers
    assert lib.mx_selftest_sigmoid(fake, -1, fake, None) == _lib.MX_ERR_INVALID_ARG
    assert lib.mx_selftest_sigmoid(None, 4, fake, None) == _lib.MX_ERR_INVALID_ARG


def test_swiglu_bwd_alignment_rules(lib):
    """moe_swiglu_bwd writes every scale byte by byte, so dab_rs, dab_cs and
    h_cs may sit at any offset: such calls get past every argument check and
    stop only at the device check of this GPU-less machine.  Its data
    pointers (dh, ab, dab_rq, dab_cq, h_cq) take 16-byte vector accesses: one
    off a 16-byte boundary is refused on the host with MX_ERR_ALIGNMENT before
    anything is launched."""
    from mxfp8_mixture_experts_gb300 import _lib
    base = 1 << 20
    f = C.c_void_p(base)
    ok = {_lib.MX_ERR_UNSUPPORTED_DEVICE, _lib.MX_ERR_CUDA}
    args = lambda dab_rs, dab_cs, h_cs: (f, f, 256, 64, 0, f, dab_rs, f, dab_cs, f, h_cs, None, None)
    for off in (1, 2, 3):
        o = C.c_void_p(base + off)
        assert lib.moe_swiglu_bwd(*args(o, f, f)) in ok
        assert lib.moe_swiglu_bwd(*args(f, o, f)) in ok
        assert lib.moe_swiglu_bwd(*args(f, f, o)) in ok
    for pos in (0, 1, 5, 7, 9):  # dh, ab, dab_rq, dab_cq, h_cq
        for off in (4, 8):
            a = list(args(f, f, f))
            a[pos] = C.c_void_p(base + off)
            assert lib.moe_swiglu_bwd(*a) == _lib.MX_ERR_ALIGNMENT


def test_package_imports_and_fails_loudly_without_library(tmp_path):
    from mxfp8_mixture_experts_gb300 import _lib
    with pytest.raises(ImportError):
        _lib.load.__wrapped__(str(tmp_path / "nope.so")) if hasattr(_lib.load, "__wrapped__") else \
            _load_fresh(str(tmp_path / "nope.so"))


def _load_fresh(path):
    from mxfp8_mixture_experts_gb300 import _lib
    saved = _lib._lib
    try:
        _lib._lib = None
        return _lib.load(path)
    finally:
        _lib._lib = saved
