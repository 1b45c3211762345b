"""Host-side checks of the C-ABI library (no GPU needed).

The library must load and export every function include/bitlin.h declares,
and argument validation must answer before any device work.
"""
import ctypes

import pytest

import hadamard_rotated_binary_gb300 as hrb
from hadamard_rotated_binary_gb300 import build as hbuild


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return hrb.lib()


def test_every_header_function_is_exported(L):
    names = hrb.header_functions()
    assert "bitlin_create" in names and "bitlin_forward" in names and "bitlin_destroy" in names
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    for st in range(8):
        assert L.bitlin_status_string(st) != b"unknown status"
    assert L.bitlin_status_string(99) == b"unknown status"
    assert L.bitlin_version() >= 100


def test_argument_validation_without_device(L):
    h = ctypes.c_void_p()
    p = 256  # any 16-byte aligned non-NULL value; validation fails before it is used
    assert L.bitlin_create(None, 8, 1024, p, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create(ctypes.byref(h), 0, 1024, p, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create(ctypes.byref(h), 8, 1000, p, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create(ctypes.byref(h), 8, 0, p, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create(ctypes.byref(h), 8, 1024, None, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create(ctypes.byref(h), 8, 1024, p, p, p, 7) == hrb.BITLIN_EINVAL
    # the ssm_out permutation is defined for K = 6144 only
    assert L.bitlin_create(ctypes.byref(h), 8, 5120, p, p, p, 1) == hrb.BITLIN_EINVAL
    # misaligned pointers
    assert L.bitlin_create(ctypes.byref(h), 8, 1024, p + 4, p, p, 0) == hrb.BITLIN_EINVAL
    assert h.value is None
    assert L.bitlin_forward(None, p, 1, p, None) == hrb.BITLIN_EINVAL
    assert L.bitlin_forward_host(None, p, 1, p, None) == hrb.BITLIN_EINVAL
    assert L.bitlin_embed(None, p, 1, p, None) == hrb.BITLIN_EINVAL
    assert L.bitlin_argmax(None, p, 1, None, p, None) == hrb.BITLIN_EINVAL
    assert L.bitlin_mlp_forward(None, None, p, 1, p, None) == hrb.BITLIN_EINVAL
    assert L.bitlin_set_path(None, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create_q1g128(None, 8, 1024, p, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create_q1g128(ctypes.byref(h), 8, 1024, None, p, 0) == hrb.BITLIN_EINVAL
    assert L.bitlin_create_q1g128(ctypes.byref(h), 8, 1000, p, p, 0) == hrb.BITLIN_EINVAL
    assert h.value is None
    a, b = ctypes.c_int32(), ctypes.c_int32()
    assert L.bitlin_plan(None, 1, ctypes.byref(a), ctypes.byref(b)) == hrb.BITLIN_EINVAL
    assert L.bitlin_get_error(None) == hrb.BITLIN_EINVAL
    assert L.bitlin_destroy(None) == hrb.BITLIN_OK
    assert L.bitlin_cuda_error(None) == 0
