"""bitlin_forward_noalloc, the entry point for callers that may not allocate
device memory on their call path (a runtime that owns every device
allocation, or a loop that must never enter the allocator because cudaMalloc
can synchronize the device).

Called through the C-ABI, two calls in a row with different inputs, on the
ffn_gate shape at M = 1, 2 and 4 (the one-token and the two-tokens-per-pass
kernels, both writing their partial sums into the fixed array), on the
permuted ssm_out shape and on ffn_down (34 slices).  Each call is compared
with the oracle within the decode tolerance and with bitlin_forward on the
same input.  A fresh handle's first call must leave the device's free memory
unchanged.  Kept in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DECODE_TOL = 1e-5


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float((np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1)).max())


@pytest.fixture(scope="module")
def hrb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hadamard_rotated_binary_gb300 import build as hbuild

    hbuild.build()
    oracle.build()
    import hadamard_rotated_binary_gb300 as m

    return m


def _layer(hrb, w):
    bits, scales, signs, _ = synth.make_inputs(w)
    layer = hrb.BitLinear(torch.from_numpy(bits.view(np.int32)).cuda(),
                          torch.from_numpy(scales.view(np.int16)).cuda(),
                          torch.from_numpy(signs).cuda(), w.perm)
    return layer, (bits, scales, signs)


def _noalloc(hrb, layer, x, M, N):
    L = hrb.lib()
    stream = torch.cuda.current_stream()
    y = torch.full((M, N), float("nan"), device="cuda")
    st = L.bitlin_forward_noalloc(layer.handle, ctypes.c_void_p(x.data_ptr()), M,
                                  ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    return st, y


@pytest.mark.parametrize("name,M", [("ffn_gate", 1), ("ffn_gate", 2), ("ffn_gate", 4), ("ssm_out", 1),
                                    ("ffn_down", 1), ("ffn_down", 4)])
def test_noalloc_matches_oracle_on_two_calls_in_a_row(hrb, name, M):
    w = synth.workload(name, M)
    layer, (bits, scales, signs) = _layer(hrb, w)
    for call, seed in enumerate((101, 202)):
        xh = synth.random_x(seed, M, w.K)
        x = torch.from_numpy(xh).cuda()
        st, y = _noalloc(hrb, layer, x, M, w.N)
        assert st == hrb.BITLIN_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert layer.get_error() == hrb.BITLIN_OK
        got = y.cpu().numpy()
        assert np.isfinite(got).all()
        ref = oracle.forward(bits, scales, signs, w.perm, xh)
        assert _rel(got, ref) <= DECODE_TOL, f"call {call} against the oracle"
        assert _rel(got, layer(x).cpu().numpy()) <= DECODE_TOL, f"call {call} against bitlin_forward"
    layer.close()


def test_noalloc_allocates_nothing_and_refuses_oversize(hrb):
    L = hrb.lib()
    w = synth.workload("ffn_gate", 4)
    # A first call on another handle loads the library's kernels and its fixed
    # array on this device; after that, a fresh handle's first call (which on
    # bitlin_forward would allocate its split-K scratch) must allocate nothing.
    # The warm-up runs both kernel instances (one token, two tokens per pass).
    warm, _ = _layer(hrb, synth.workload("tiny"))
    for m in (1, 4):
        xw = torch.from_numpy(synth.random_x(7, m, 1024)).cuda()
        assert _noalloc(hrb, warm, xw, m, 256)[0] == hrb.BITLIN_OK
    torch.cuda.synchronize()
    layer, (bits, scales, signs) = _layer(hrb, w)
    xh = synth.random_x(303, 4, w.K)
    x = torch.from_numpy(xh).cuda()
    y = torch.empty((4, w.N), device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    st = L.bitlin_forward_noalloc(layer.handle, ctypes.c_void_p(x.data_ptr()), 4,
                                  ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert st == hrb.BITLIN_OK
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert _rel(y.cpu().numpy(), oracle.forward(bits, scales, signs, w.perm, xh)) <= DECODE_TOL

    # Sizes beyond the fixed scratch are refused before any launch.
    cap = L.bitlin_noalloc_scratch_bytes()
    too_many = cap // (w.K // 512 * ((w.N + 31) // 32) * 128) + 1
    xb = torch.zeros((too_many, w.K), device="cuda")
    yb = torch.zeros((too_many, w.N), device="cuda")
    st = L.bitlin_forward_noalloc(layer.handle, ctypes.c_void_p(xb.data_ptr()), too_many,
                                  ctypes.c_void_p(yb.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert st == hrb.BITLIN_ESCRATCH
    layer.close()
    warm.close()
