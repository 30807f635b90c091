"""GB300-native W4A16 GEMM: int4 group-quantized weights x fp16/bf16 activations.

The compute path is the C-ABI library ``libtmw4.so`` (CUDA for sm_103a, built
in-tree by ``w4a16_gemm_gb300.build``); :mod:`w4a16_gemm_gb300.binding` is a
thin ctypes layer over it that marshals torch tensors into device pointers.
:mod:`w4a16_gemm_gb300.synth` holds the seeded synthetic inputs.  The binding
is imported lazily so that the input generators work on machines without the
library.
"""

__all__ = ["binding", "synth", "build"]


def __getattr__(name):
    if name in ("pack", "gemm", "dequant", "tune", "PackedW4", "TmError", "lib"):
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
