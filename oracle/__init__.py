"""CPU oracle for the W4A16 GEMM pipeline (test infrastructure only).

This package is the plain, slow, obviously-correct definition of what the GPU
path computes.  It is test infrastructure: only the test-suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product path (the CUDA library and its Python binding) never
calls into it, and it never calls into them: the two share no code.

Every function cites the passage of the source pages it follows, as
"<page title>, <figure/section>".  The pages are the TurboMind/LMDeploy
paper pages ("Efficient Mixed-Precision Large Language Model Inference with
TurboMind", arXiv 2508.15601, its abstract page and its pith.science review
with figure captions).
"""

from .w4a16 import (  # noqa: F401
    ATOM_K,
    ATOM_N,
    TILE_N,
    NIBBLE_POS,
    f16_bits_to_f64,
    bf16_bits_to_f64,
    rne_f16_bits,
    rne_bf16_bits,
    act_bits_to_f64,
    dequant_bits,
    dequant_f64,
    gemm_ref,
    pack_ref,
    unpack_ref,
    pack_scales_ref,
    unpack_scales_ref,
    pack_zeros_ref,
    unpack_zeros_ref,
    rms,
    tolerance_ok,
    max_err_ratio,
)
