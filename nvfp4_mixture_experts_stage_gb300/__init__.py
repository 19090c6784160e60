"""NVFP4 routed-expert MoE stage for GB300 (sm_103a).

The compute lives in ``libmoe_stage.so`` (CUDA kernels behind the C ABI of
``include/moe_stage.h``); ``binding`` is its thin ctypes wrapper and ``build``
compiles it in-tree.  Import ``nvfp4_mixture_experts_stage_gb300.binding`` to
use the library (importing fails loudly if the library was not built).
"""

__all__ = ["build", "binding"]
