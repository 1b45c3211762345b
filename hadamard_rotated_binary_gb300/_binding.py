"""ctypes binding of libbitlin.so: same names as the C-ABI, argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "bitlin.h")

BITLIN_OK = 0
BITLIN_EINVAL = 1
BITLIN_ENOMEM = 2
BITLIN_ECUDA = 3
BITLIN_ETIMEOUT = 4
BITLIN_EDEVICE = 5
BITLIN_ESCRATCH = 6
BITLIN_EINDEX = 7

PERM_NONE = 0
PERM_SSM_TILED_TO_GROUPED = 1
PATH_AUTO = 0
PATH_DECODE = 1
PATH_PREFILL = 2
PATH_TC_EXACT = 3

_lib = None


def library_path() -> str:
    return os.path.join(PKG, "libbitlin.so")


def header_functions() -> list[str]:
    """Names of every function declared in include/bitlin.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bitlin_[a-z_]+)\s*\(", text)))


class BitlinError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        msg = f"{what}: {lib().bitlin_status_string(status).decode()} (status {status})"
        if cuda_error:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load libbitlin.so (built by build()).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with hadamard_rotated_binary_gb300.build.build()")
    L = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    L.bitlin_create.argtypes = [ctypes.POINTER(P), i32, i32, P, P, P, i32]
    L.bitlin_create_q1g128.argtypes = [ctypes.POINTER(P), i32, i32, P, P, i32]
    L.bitlin_forward.argtypes = [P, P, i32, P, P]
    L.bitlin_forward_host.argtypes = [P, P, i32, P, P]
    L.bitlin_forward_noalloc.argtypes = [P, P, i32, P, P]
    L.bitlin_forward_noalloc.restype = i32
    L.bitlin_noalloc_scratch_bytes.restype = ctypes.c_size_t
    L.bitlin_embed.argtypes = [P, P, i32, P, P]
    L.bitlin_mlp_forward.argtypes = [P, P, P, i32, P, P]
    L.bitlin_argmax.argtypes = [P, P, i32, P, P, P]
    L.bitlin_set_path.argtypes = [P, i32]
    L.bitlin_plan.argtypes = [P, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.bitlin_set_wait_budget.argtypes = [P, i64]
    L.bitlin_test_stall.argtypes = [P, i32]
    L.bitlin_destroy.argtypes = [P]
    L.bitlin_get_error.argtypes = [P]
    L.bitlin_cuda_error.argtypes = [P]
    L.bitlin_status_string.argtypes = [i32]
    L.bitlin_status_string.restype = ctypes.c_char_p
    for name in ("bitlin_create", "bitlin_create_q1g128", "bitlin_forward", "bitlin_forward_host", "bitlin_embed", "bitlin_mlp_forward",
                 "bitlin_argmax", "bitlin_set_path", "bitlin_plan", "bitlin_set_wait_budget", "bitlin_test_stall", "bitlin_destroy", "bitlin_get_error",
                 "bitlin_cuda_error", "bitlin_version"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def _stream_handle(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def mlp_forward(gate_up: "BitLinear", down: "BitLinear", x, out=None, stream=None):
    """bitlin_mlp_forward: down(silu(gate) * up) with [gate | up] = gate_up(x)."""
    import torch

    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous float32 CUDA tensor [M][K]")
    M = int(x.shape[0])
    if out is None:
        out = torch.empty((M, down.N), dtype=torch.float32, device=x.device)
    st = lib().bitlin_mlp_forward(gate_up.handle, down.handle, x.data_ptr(), M, out.data_ptr(),
                                  _stream_handle(stream))
    if st != BITLIN_OK:
        raise BitlinError(st, "bitlin_mlp_forward", lib().bitlin_cuda_error(down.handle))
    return out


def q1g128_words(N: int, K: int) -> int:
    """32-bit words of one stored Q1G128 tensor: N*K/256 of scales, then N*K/32 of bits."""
    if N < 1 or K < 1024 or K % 1024:
        raise ValueError("N >= 1 and K a positive multiple of 1024")
    return N * K // 256 + N * K // 32


def load_q1g128(path: str, N: int, K: int, offset: int = 0, device="cuda"):
    """Read one stored Q1G128 tensor (q1g128_words(N, K) little-endian words starting at byte
    `offset` of the file) into a CUDA int32 tensor for BitLinear.from_q1g128."""
    import numpy as np
    import torch

    n = q1g128_words(N, K)
    words = np.fromfile(path, dtype="<u4", count=n, offset=offset)
    if words.size != n:
        raise ValueError(f"{path}: {4 * words.size} bytes at offset {offset}, need {4 * n}")
    return torch.from_numpy(words.view(np.int32)).to(device)


class BitLinear:
    """One folded 1-bit matrix on the GPU (a bitlin handle).

    bits    torch int32/uint32 cuda tensor [N][K/32] (LSB-first packed signs, 1 -> +1)
    scales  torch int16/uint16/float16 cuda tensor [N][K/128] (IEEE fp16)
    signs   torch float32 cuda tensor [K] of exact +-1
    perm    PERM_NONE or PERM_SSM_TILED_TO_GROUPED (K == 6144)
    """

    def __init__(self, bits, scales, signs, perm: int = PERM_NONE):
        import torch

        N = int(bits.shape[0])
        K = int(bits.shape[1]) * 32
        for t in (bits, scales, signs):
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("bits, scales and signs must be contiguous CUDA tensors")
        if signs.dtype != torch.float32:
            raise ValueError("signs must be float32")
        h = ctypes.c_void_p()
        with torch.cuda.device(bits.device):
            st = lib().bitlin_create(ctypes.byref(h), N, K, bits.data_ptr(), scales.data_ptr(),
                                     signs.data_ptr(), int(perm))
        if st != BITLIN_OK:
            raise BitlinError(st, "bitlin_create")
        self._adopt(h, N, K, perm, bits.device)

    def _adopt(self, h, N: int, K: int, perm: int, device):
        self._h = h
        self.N, self.K, self.perm = N, K, perm
        self.device = device

    @classmethod
    def from_q1g128(cls, qdata, N: int, K: int, signs, perm: int = PERM_NONE) -> "BitLinear":
        """bitlin_create_q1g128: a handle from one Q1G128 tensor in its stored form (fp16 scales
        two per word, then the sign bits; q1g128_words(N, K) words in a CUDA tensor)."""
        import torch

        for t in (qdata, signs):
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("qdata and signs must be contiguous CUDA tensors")
        if qdata.numel() * qdata.element_size() != 4 * q1g128_words(N, K):
            raise ValueError(f"qdata must hold {4 * q1g128_words(N, K)} bytes for N={N}, K={K}")
        if signs.dtype != torch.float32:
            raise ValueError("signs must be float32")
        h = ctypes.c_void_p()
        with torch.cuda.device(qdata.device):
            st = lib().bitlin_create_q1g128(ctypes.byref(h), int(N), int(K), qdata.data_ptr(), signs.data_ptr(),
                                            int(perm))
        if st != BITLIN_OK:
            raise BitlinError(st, "bitlin_create_q1g128")
        self = cls.__new__(cls)
        self._adopt(h, int(N), int(K), perm, qdata.device)
        return self

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def _check(self, st: int, what: str):
        if st != BITLIN_OK:
            raise BitlinError(st, what, lib().bitlin_cuda_error(self._h))

    def forward(self, x, out=None, stream=None):
        """y[M][N] for x a contiguous float32 CUDA tensor [M][K] (or [K])."""
        import torch

        squeeze = x.dim() == 1
        x2 = x.reshape(1, -1) if squeeze else x
        if x2.dtype != torch.float32 or not x2.is_cuda or not x2.is_contiguous() or x2.shape[1] != self.K:
            raise ValueError("x must be a contiguous float32 CUDA tensor [M][K]")
        M = int(x2.shape[0])
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32, device=x2.device)
        self._check(lib().bitlin_forward(self._h, x2.data_ptr(), M, out.data_ptr(), _stream_handle(stream)),
                    "bitlin_forward")
        return out.reshape(-1) if squeeze else out

    __call__ = forward

    def forward_host(self, x_host, y_host, stream=None):
        """numpy float32 [M][K] -> numpy float32 [M][N] through host buffers (synchronous)."""
        M = int(x_host.shape[0])
        assert x_host.flags["C_CONTIGUOUS"] and y_host.flags["C_CONTIGUOUS"]
        assert x_host.shape == (M, self.K) and y_host.shape == (M, self.N)
        self._check(lib().bitlin_forward_host(self._h, x_host.ctypes.data, M, y_host.ctypes.data,
                                              _stream_handle(stream)), "bitlin_forward_host")
        return y_host

    def forward_noalloc(self, x, out, stream=None):
        """bitlin_forward_noalloc: y into `out` with the library's fixed scratch (no allocation)."""
        M = int(x.shape[0])
        self._check(lib().bitlin_forward_noalloc(self._h, x.data_ptr(), M, out.data_ptr(),
                                                 _stream_handle(stream)), "bitlin_forward_noalloc")
        return out

    def argmax(self, x, logits=None, ids=None, stream=None):
        """bitlin_argmax: int32 [M] ids of the largest score per token (smallest index on ties);
        the scores go to `logits` ([M][N] float32) when given."""
        import torch

        if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
            raise ValueError("x must be a contiguous float32 CUDA tensor [M][K]")
        M = int(x.shape[0])
        if ids is None:
            ids = torch.empty((M,), dtype=torch.int32, device=x.device)
        self._check(lib().bitlin_argmax(self._h, x.data_ptr(), M, logits.data_ptr() if logits is not None else None,
                                        ids.data_ptr(), _stream_handle(stream)), "bitlin_argmax")
        return ids

    def embed(self, ids, out=None, stream=None):
        """bitlin_embed: rows ids (int32 CUDA tensor [M]) of the matrix, dequantized and
        inverse-rotated, as float32 [M][K]."""
        import torch

        if ids.dtype != torch.int32 or not ids.is_cuda or not ids.is_contiguous() or ids.dim() != 1:
            raise ValueError("ids must be a contiguous int32 CUDA tensor [M]")
        M = int(ids.shape[0])
        if out is None:
            out = torch.empty((M, self.K), dtype=torch.float32, device=ids.device)
        self._check(lib().bitlin_embed(self._h, ids.data_ptr(), M, out.data_ptr(), _stream_handle(stream)),
                    "bitlin_embed")
        return out

    def set_path(self, path: int):
        self._check(lib().bitlin_set_path(self._h, int(path)), "bitlin_set_path")

    def plan(self, M: int) -> tuple[int, int]:
        """bitlin_plan: (path, kernels launched) of a forward call with M tokens."""
        path, kernels = ctypes.c_int32(), ctypes.c_int32()
        self._check(lib().bitlin_plan(self._h, int(M), ctypes.byref(path), ctypes.byref(kernels)), "bitlin_plan")
        return path.value, kernels.value

    def set_wait_budget(self, ns: int):
        self._check(lib().bitlin_set_wait_budget(self._h, int(ns)), "bitlin_set_wait_budget")

    def test_stall(self, on: bool):
        self._check(lib().bitlin_test_stall(self._h, 1 if on else 0), "bitlin_test_stall")

    def get_error(self) -> int:
        return lib().bitlin_get_error(self._h)

    def close(self):
        if getattr(self, "_h", None):
            lib().bitlin_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
