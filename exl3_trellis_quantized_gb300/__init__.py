"""EXL3 trellis-quantized linear layer for GB300 (sm_103a).

The compute lives in ``libexl3.so`` (hand-written CUDA behind a C ABI, see
``include/exl3.h``).  This package is a thin binding: it marshals torch
tensors into pointers and sizes and calls the library.  There is no CPU or
PyTorch fallback; if the library is missing every call raises.
"""
from .binding import (  # noqa: F401
    CODEBOOKS,
    Exl3Error,
    autotune_entries,
    clear_autotune,
    device_status,
    gemm,
    gemm_splitk,
    input_transform,
    input_transform_swiglu,
    lib,
    linear,
    set_autotune,
    moe_combine,
    moe_gemm,
    moe_input_transform,
    splitk_parts,
    splitk_workspace_bytes,
    status_string,
    test_codebook,
    test_unpack,
)
