"""CPU oracle of the Hadamard-folded 1-bit GEMV (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this module.  It wraps ``bitlin_oracle.c`` (plain C, double precision,
built with gcc) through ctypes.  It shares no code with the CUDA library and
never imports it.

Functions and the passages they follow are documented in the C source.  One
reading stays unpinned and is marked so here as well: the Walsh-Hadamard
ordering ("normalized Sylvester-Walsh" is read as the natural Sylvester order,
H[i][j] = (-1)^popcount(i & j)) - parity unpinned, because only real folded
weights could distinguish it from the sequency order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlin_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available); returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    d, i32, i64 = ctypes.c_double, ctypes.c_int, ctypes.c_int64
    P = ctypes.c_void_p
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = d
    lib.oracle_round_bf16.argtypes = [d]
    lib.oracle_round_bf16.restype = d
    lib.oracle_wht_block.argtypes = [P, P]
    lib.oracle_permute_tiled_to_grouped.argtypes = [P, P]
    lib.oracle_rotate.argtypes = [P, i32, P, i32, P]
    lib.oracle_rotate.restype = i32
    lib.oracle_rotate_f64.argtypes = [P, i32, P, i32, P]
    lib.oracle_rotate_f64.restype = i32
    lib.oracle_inverse_rotate.argtypes = [P, i32, P, P]
    lib.oracle_rotate_tokens.argtypes = [P, i32, i32, P, i32, i32, P]
    lib.oracle_rotate_tokens.restype = i32
    lib.oracle_product.argtypes = [P, P, P, i32, i32, i32, P, i32, P]
    lib.oracle_dequant_row.argtypes = [P, P, i32, i32, P]
    lib.oracle_max_threads.restype = i32
    lib.oracle_set_threads.argtypes = [i32]
    _ = i64
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def f16_to_f64(h: int) -> float:
    return _load().oracle_f16_to_f64(int(h))


def round_bf16(v: float) -> float:
    return _load().oracle_round_bf16(float(v))


def wht_block(v: np.ndarray) -> np.ndarray:
    """Normalized 1024-point transform of one block, by the O(1024^2) definition."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert v.shape == (1024,)
    out = np.empty(1024, dtype=np.float64)
    _load().oracle_wht_block(_ptr(v), _ptr(out))
    return out


def permute_tiled_to_grouped(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert v.shape == (6144,)
    out = np.empty(6144, dtype=np.float64)
    _load().oracle_permute_tiled_to_grouped(_ptr(v), _ptr(out))
    return out


def rotate(x: np.ndarray, signs: np.ndarray, perm: int, round_bf16: bool = False) -> np.ndarray:
    """x f32 [M][K] -> rotated activations f64 [M][K] (perm -> signs -> WHT blocks)."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    signs = np.ascontiguousarray(signs, dtype=np.float32)
    M, K = x.shape
    assert K % 1024 == 0 and signs.shape == (K,)
    assert not perm or K == 6144
    out = np.empty((M, K), dtype=np.float64)
    rc = _load().oracle_rotate_tokens(_ptr(x), M, K, _ptr(signs), int(perm), int(round_bf16), _ptr(out))
    if rc != 0:
        raise MemoryError("oracle rotate: allocation failed")
    return out


def inverse_rotate(z: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """The embedding order h = signs * WHT(z), one vector of width K."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    signs = np.ascontiguousarray(signs, dtype=np.float32)
    K = z.shape[0]
    out = np.empty(K, dtype=np.float64)
    _load().oracle_inverse_rotate(_ptr(z), K, _ptr(signs), _ptr(out))
    return out


def product(bits: np.ndarray, scales: np.ndarray, xt: np.ndarray, rows=None) -> np.ndarray:
    """y[M][len(rows)] = one-bit matrix rows times rotated activations, f64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    xt = np.ascontiguousarray(np.atleast_2d(xt), dtype=np.float64)
    N = bits.shape[0]
    M, K = xt.shape
    assert bits.shape == (N, K // 32) and scales.shape == (N, K // 128)
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((M, rows.size), dtype=np.float64)
    _load().oracle_product(_ptr(bits), _ptr(scales), _ptr(xt), M, N, K, _ptr(rows), rows.size, _ptr(out))
    return out


def forward(bits, scales, signs, perm, x, rows=None, round_bf16: bool = False) -> np.ndarray:
    """The whole method in f64: rotate each token, then the folded one-bit product."""
    xt = rotate(x, signs, perm, round_bf16=round_bf16)
    return product(bits, scales, xt, rows)


def dequant_row(bits: np.ndarray, scales: np.ndarray, n: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    K = bits.shape[1] * 32
    out = np.empty(K, dtype=np.float64)
    _load().oracle_dequant_row(_ptr(bits), _ptr(scales), K, int(n), _ptr(out))
    return out


def q1g128_weight(qdata: np.ndarray, N: int, K: int, n: int, k: int) -> float:
    """Weight (n, k) read from one stored Q1G128 tensor by the engine page's indexing
    ("Inside the One-Bit Engine", embedding-lookup and weight-format stations): scale index
    sidx = n*(K/128) + (k >> 7) selects half (sidx & 1) of word sidx >> 1 (two binary16 per
    word, the first in the low 16 bits); the bit words start after the scale words (N*K/256
    of them), row n at n*(K/32), weight k at bit k & 31 of word k >> 5; w = (2*bit - 1) * scale."""
    G = K // 128
    scale_words = N * G // 2
    sidx = n * G + (k >> 7)
    half = (int(qdata[sidx >> 1]) >> (16 * (sidx & 1))) & 0xFFFF
    word = int(qdata[scale_words + n * (K >> 5) + (k >> 5)])
    bit = (word >> (k & 31)) & 1
    return (2.0 * bit - 1.0) * f16_to_f64(half)


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g / (1 + e^-g), f64 ("Inside the One-Bit Engine", MLP station)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def rotate_f64(x: np.ndarray, signs: np.ndarray, perm: int) -> np.ndarray:
    """As rotate, for f64 activations (no rounding of the input to f32)."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    signs = np.ascontiguousarray(signs, dtype=np.float32)
    M, K = x.shape
    out = np.empty((M, K), dtype=np.float64)
    L = _load()
    for m in range(M):
        if L.oracle_rotate_f64(_ptr(x[m]), K, _ptr(signs), int(perm), _ptr(out[m])) != 0:
            raise MemoryError("oracle rotate: allocation failed")
    return out


def mlp(gu, down, x, rows=None) -> np.ndarray:
    """The MLP block in f64: [g | u] = forward(gate_up, x) (first F rows gate, next F up),
    mid = silu(g) * u, y = the folded product of down on mid (kept in f64).  gu and down are
    (bits, scales, signs, perm)."""
    F = gu[0].shape[0] // 2
    h = forward(*gu, x)
    mid = silu(h[:, :F]) * h[:, F:]
    bits, scales, signs, perm = down
    return product(bits, scales, rotate_f64(mid, signs, perm), rows)


def embed(bits: np.ndarray, scales: np.ndarray, signs: np.ndarray, ids) -> np.ndarray:
    """Embedding lookup with the inverse rotation, f64: row ids[m] dequantized, then
    h = signs * WHT(z) (Pulse "ARCHITECTURE-SPEC", Hadamard-fold section, embedding order)."""
    return np.stack([inverse_rotate(dequant_row(bits, scales, int(t)), signs) for t in ids])


def max_threads() -> int:
    return _load().oracle_max_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def timed_forward(bits, scales, signs, perm, x, rows) -> tuple[np.ndarray, float]:
    """forward() on a row sample, with its wall time in seconds."""
    t0 = time.perf_counter()
    y = forward(bits, scales, signs, perm, x, rows)
    return y, time.perf_counter() - t0
