"""CPU oracle for the NVFP4 MoE expert FFN — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the forward pass computes,
written from the debug log and commit messages of the NVFP4 MegaMoE kernel
("NVFP4 MegaMoE Debug Log": Architecture Notes / NVFP4 MoE Pipeline,
Hypotheses §3, §5, §6; the commit messages on ``src`` about the E2M1 quantiser,
the FP8 view-vs-convert fix, the SF remap, and the plain [gate; up] concat).

Rules this package keeps:

* Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
  ``bench.py`` may import it.  The library (``nvfp4_block_scaled_route_gb300``)
  never does, and has no CPU fallback.
* It shares no code with the CUDA path: no kernels, headers, tables, layouts
  or helpers.  Inputs come from the seeded generator module, which holds none
  of the method's arithmetic.
* Floating point: quantisation decisions are taken in IEEE fp32 with
  round-to-nearest-even, in the order the pages give (the pages' quantiser is
  fp32 torch code); every accumulation (GEMM, SiLU, reduction) is fp64.
* Codecs decode by bit pattern through explicit tables and encode by nearest
  search over the representable values; no library float8/float4 conversion is
  used inside the oracle (those are used only as pins in the tests).

Pinning status of each function is listed in its docstring.  Every function is
pinned by a ``-m "not gpu"`` test (tests/test_oracle_pins.py) against values
the pages print, closed forms, library routines for special cases, or
pure-Python brute force on tiny inputs.
"""
from . import nvfp4, moe  # noqa: F401
