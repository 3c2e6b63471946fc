"""CPU oracle for the MXFP8 MoE hot path (TEST INFRASTRUCTURE).

A plain, slow, obviously correct numpy implementation of what the path
computes: the MX block quantizer (``oracle.mx``) and the router, token
permute/unpermute, grouped GEMMs, SwiGLU and layer forward/backward
(``oracle.moe``).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library and never imports it; the two meet only through the seeded
inputs of ``workloads``.

Parity status: every function is pinned by tests/test_oracle_*.py except the
end-to-end MXFP8-vs-bf16 layer accuracy, which is reported as SQNR only
(parity unpinned: the pages give no expected value for it).
"""
from . import mx, moe  # noqa: F401
