"""Hadamard-folded 1-bit GEMV for NVIDIA GB300 (sm_103a).

A thin Python binding of the C-ABI library ``libbitlin.so`` (declared in
``include/bitlin.h``).  The binding only marshals arguments: every step of the
computation (permutation, signs, 1024-block Walsh-Hadamard transform, one-bit
product) runs in the library's CUDA kernels.  PyTorch provides device memory
and streams.  There is no CPU fallback: if the library is missing the first
use raises.

    >>> import torch, hadamard_rotated_binary_gb300 as hrb
    >>> lin = hrb.BitLinear(bits, scales, signs, perm=0)   # device tensors
    >>> y = lin(x)                                           # x: cuda f32 [M][K]
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    BITLIN_EDEVICE,
    BITLIN_EINDEX,
    BITLIN_ESCRATCH,
    BITLIN_EINVAL,
    BITLIN_ENOMEM,
    BITLIN_ECUDA,
    BITLIN_ETIMEOUT,
    BITLIN_OK,
    PATH_AUTO,
    PATH_DECODE,
    PATH_PREFILL,
    PATH_TC_EXACT,
    PERM_NONE,
    PERM_SSM_TILED_TO_GROUPED,
    BitlinError,
    BitLinear,
    header_functions,
    lib,
    library_path,
    load_q1g128,
    mlp_forward,
    q1g128_words,
)

__all__ = [
    "BitLinear",
    "BitlinError",
    "mlp_forward",
    "load_q1g128",
    "q1g128_words",
    "lib",
    "library_path",
    "header_functions",
    "PATH_AUTO",
    "PATH_DECODE",
    "PATH_PREFILL",
    "PATH_TC_EXACT",
    "PERM_NONE",
    "PERM_SSM_TILED_TO_GROUPED",
]
