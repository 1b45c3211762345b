"""bitlin_forward_noalloc, the entry point for callers that may not allocate
device memory on their call path (a runtime that owns every device
allocation, or a loop that must never enter the allocator because cudaMalloc
can synchronize the device).

Called through the C-ABI on the ffn_gate-shaped matrix, two calls in a row
with different inputs, each compared with bitlin_forward on the same input
within the decode tolerance.  Kept in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DECODE_TOL = 1e-5


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float((np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1)).max())


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hadamard_rotated_binary_gb300 import build as hbuild

    hbuild.build()
    import hadamard_rotated_binary_gb300 as hrb

    L = hrb.lib()
    w = synth.workload("ffn_gate")
    bits, scales, signs, _ = synth.make_inputs(w)
    layer = hrb.BitLinear(torch.from_numpy(bits.view(np.int32)).cuda(),
                          torch.from_numpy(scales.view(np.int16)).cuda(),
                          torch.from_numpy(signs).cuda(), w.perm)
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((101, 202)):
        x = torch.from_numpy(synth.random_x(seed, 1, w.K)).cuda()
        ref = layer(x)
        y = torch.full((1, w.N), float("nan"), device="cuda")
        st = L.bitlin_forward_noalloc(layer.handle, ctypes.c_void_p(x.data_ptr()), 1,
                                      ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == hrb.BITLIN_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert layer.get_error() == hrb.BITLIN_OK
        assert torch.isfinite(y).all()
        assert _rel(y, ref) <= DECODE_TOL, f"call {call}"

    # Sizes beyond the fixed scratch are refused before any launch.
    cap = L.bitlin_noalloc_scratch_bytes()
    too_many = cap // (w.K // 512 * ((w.N + 31) // 32) * 128) + 1
    xb = torch.zeros((too_many, w.K), device="cuda")
    yb = torch.zeros((too_many, w.N), device="cuda")
    st = L.bitlin_forward_noalloc(layer.handle, ctypes.c_void_p(xb.data_ptr()), too_many,
                                  ctypes.c_void_p(yb.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert st == hrb.BITLIN_ESCRATCH
    layer.close()
