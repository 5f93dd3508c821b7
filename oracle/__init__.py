"""CPU oracle for single-query paged-attention decode (test infrastructure).

This package is test infrastructure, not part of the product. Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
or run it. It shares no code with the CUDA library and imports nothing from it.

Every function computes from the contiguous, pre-paging K/V in float64, never
from the paged cache, as the page "vLLM's custom ROCm paged-attention kernel
wins all sixty cells" (gqa-gate-costs-nothing, §1) does for its reference.
"""
from .decode_ref import decode_ref, decode_ref_one, decode_ref_rows, rel_linf_error
from .fp8 import dequant, e4m3_to_float64

__all__ = ["decode_ref", "decode_ref_one", "decode_ref_rows", "rel_linf_error", "dequant",
           "e4m3_to_float64"]
