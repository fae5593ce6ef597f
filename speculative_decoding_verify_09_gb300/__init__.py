"""GB300-native (sm_103a) batched speculative-decoding verify step.

The verify step of speculative sampling over a padding-free batch: ragged
split-KV verify attention, modified rejection sampling (temperature, nucleus,
Philox uniforms, residual and bonus draws) and the append of accepted K/V
rows, as CUDA kernels behind the C ABI in include/spec_verify.h.  This package
is the thin Python face of that library: `build` compiles it, `api` passes
torch CUDA tensors to it.
"""
from .build import build, LIB as LIB_PATH  # noqa: F401


def load():
    """Import the binding (fails loudly if the CUDA library is not built)."""
    from . import api  # noqa: F401
    return api
