"""CPU oracle for the NVFP4 routed-expert MoE stage -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the MoE
layer computes, written from the nvfp4-megamoe-kernel commit pages (the commit
logs of ``src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py``, of ``src``, of
``vllm/nvfp4_cutedsl.py`` and of ``tests``).  It exists to check the CUDA
library, never to serve it:

* only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
  ``bench.py`` may import it;
* it shares no code with the CUDA path (no kernels, tables, headers or
  helpers); the only thing both sides use is the seeded input generator in
  ``workloads``, which holds none of the method's arithmetic.

Precision: every step the pages fix in fp32 (global scale, block scales, the
scaled value that picks an E2M1 code, the epilogue alpha, SiLU, the weighted
combine) is done in IEEE fp32 with round-to-nearest-even and no fused
multiply-add; the GEMM contraction is done in fp64 on exactly-dequantised
operands and rounded once to fp32.

Parity pins (what ties this oracle to something other than itself) live in
``tests/test_oracle_*.py``.  Functions whose result no pin fixes say
"parity unpinned" in their docstring.  Modules:

* ``nvfp4``  -- E2M1 / UE4M3 codecs, nibble packing, tensor quantisation,
  the block-scale swizzle.
* ``route``  -- token -> slot routing.
* ``moe``    -- grouped GEMMs, SiLU*up, requantisation, weighted combine and
  the whole layer.
"""

from . import nvfp4, route, moe  # noqa: F401
