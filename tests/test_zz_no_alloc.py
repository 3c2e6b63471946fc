"""The allocation-free grouping map (moe_permute_map_noalloc) against the
regular one (moe_permute_map, which takes a caller workspace).

Callers that only own their input and output buffers -- plugins or callbacks
inside another framework whose allocator they may not call, runtimes with a
memory budget fixed up front -- cannot hand the library the map's scratch
workspace; the allocation-free entry point keeps that scratch in a fixed
array of the library's own device memory instead.  Its results must equal the
regular entry point's bit for bit (integer index work), on consecutive calls
that reuse the shared array.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.helpers import cuda_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_device()


def _map(lib, fn_name, ids, E, dev, stream):
    T, k = ids.shape
    R = int(lib.moe_rows_cap(T, k, E))
    out = {
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "dst": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        "src": torch.full((R,), -7, dtype=torch.int32, device=dev),
    }
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    if fn_name == "moe_permute_map":
        ws_bytes = int(lib.moe_permute_map_workspace_size(T, k, E))
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        code = lib.moe_permute_map(p(ids), T, k, E, R, p(out["counts"]), p(out["offsets"]), p(out["dst"]),
                                   p(out["src"]), p(ws), ws.numel(), p(st), stream)
    else:
        code = lib.moe_permute_map_noalloc(p(ids), T, k, E, R, p(out["counts"]), p(out["offsets"]), p(out["dst"]),
                                           p(out["src"]), p(st), stream)
    assert code == 0, lib.mx_status_string(code).decode()
    return out, st


def test_noalloc_map_matches_workspace_map_on_consecutive_calls(dev):
    from mxfp8_mixture_experts_gb300 import _lib
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    cases = [(32768, 16, 4, 0), (3000, 7, 2, 1)]      # two different problems, back to back
    for T, E, k, seed in cases:
        g = workloads.generator(seed, dev)
        ids = workloads.zipf_topk_ids(T, E, k, max(E - 2, k), 1.1, g, dev)
        ref, st_ref = _map(lib, "moe_permute_map", ids, E, dev, stream)
        got, st_got = _map(lib, "moe_permute_map_noalloc", ids, E, dev, stream)
        torch.cuda.synchronize()
        assert int(st_ref.item()) == 0 and int(st_got.item()) == 0
        for name in ("counts", "offsets", "dst", "src"):
            assert torch.equal(ref[name], got[name]), (T, E, k, name)
        # the map is complete: every routed pair has a row
        assert int((got["dst"] < 0).sum()) == 0


def test_noalloc_map_rejects_problems_beyond_its_scratch(dev):
    from mxfp8_mixture_experts_gb300 import _lib
    lib = _lib.load()
    T, k, E = 1 << 20, 8, 256          # 2 * 8192 chunks * 256 experts * 4 bytes >> the fixed array
    assert lib.moe_permute_map_workspace_size(T, k, E) > 256 * 1024
    fake = ctypes.c_void_p(1 << 20)   # never touched: the size check fails first
    code = lib.moe_permute_map_noalloc(fake, T, k, E, lib.moe_rows_cap(T, k, E), fake, fake, fake, fake, None, None)
    assert code == _lib.MX_ERR_SCRATCH_LIMIT
