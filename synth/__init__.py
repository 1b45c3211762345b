"""Seeded synthetic inputs for the Hadamard-folded 1-bit GEMV.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds no part of the method's arithmetic: it only draws random
numbers and arranges them in the storage layout the method consumes
(packed sign bits, IEEE fp16 scale bit patterns, a +-1 sign vector, f32
activations).

Generator: SplitMix64 in counter mode.  Element ``i`` of stream ``sid`` under
seed ``seed`` is ``mix64(base + (i + 1) * GOLDEN)`` with
``base = mix64(seed ^ (sid * 0xD1B54A32D192ED03))``, where ``mix64`` is the
SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Counter mode lets any slice of
a stream be drawn without drawing what precedes it.

Workload shapes follow the Bonsai-27B (qwen35 hybrid) matrices described on
the "Inside the One-Bit Engine" page (station on the MLP: hidden 5120, ffn
17408; the attention station's projection table: q [12288, 5120] holding
queries and the output gate, k and v [1024, 5120], o [5120, 6144]) and the
Pulse architecture spec (ssm inner 6144; the folded-weights table: attn_qkv,
ssm_out, attn_output; sign widths 5120/6144/17408).  The gated-delta qkv
(16 key heads x 128 x 2 + 48 value heads x 128 = 10240 rows) and its output
gate (48 x 128 = 6144 rows) follow from the head counts on the same pages.  Distributions: sign bits are fair coins (the engine page's
weight forensics measured per-group popcount variance 31.985 against the
fair-coin 32.0); scales are uniform on a stated interval and rounded to fp16;
activations are standard normal.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_SID_MUL = np.uint64(0xD1B54A32D192ED03)

# Stream identifiers (one independent stream per kind of input).
SID_BITS = 1
SID_SCALES = 2
SID_SIGNS = 3
SID_X = 4


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream(seed: int, sid: int, count: int, start: int = 0) -> np.ndarray:
    """Elements [start, start+count) of stream ``sid`` as uint64."""
    with np.errstate(over="ignore"):
        base = mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(sid) * _SID_MUL))
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return mix64(base + idx * GOLDEN)


def uniform01(u64: np.ndarray) -> np.ndarray:
    """53-bit uniform doubles in [0, 1)."""
    return (u64 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def random_bits(seed: int, N: int, K: int) -> np.ndarray:
    """Packed sign bits, uint32 [N][K/32]; every bit an independent fair coin."""
    assert K % 32 == 0
    words = N * (K // 32)
    raw = stream(seed, SID_BITS, (words + 1) // 2)
    out = raw.view(np.uint32)[:words]
    return np.ascontiguousarray(out.reshape(N, K // 32))


def random_scales(seed: int, N: int, K: int, lo: float, hi: float) -> np.ndarray:
    """fp16 scale bit patterns, uint16 [N][K/128]; U[lo, hi] drawn in f64, rounded to nearest-even fp16."""
    assert K % 128 == 0
    G = K // 128
    u = uniform01(stream(seed, SID_SCALES, N * G))
    vals = (lo + (hi - lo) * u).astype(np.float16)
    return np.ascontiguousarray(vals.view(np.uint16).reshape(N, G))


def random_signs(seed: int, K: int) -> np.ndarray:
    """Sign vector, f32 [K], each entry exactly +1.0 or -1.0 with probability 1/2."""
    b = stream(seed, SID_SIGNS, K) & np.uint64(1)
    return np.where(b == 1, np.float32(1.0), np.float32(-1.0)).astype(np.float32)


def random_x(seed: int, M: int, K: int) -> np.ndarray:
    """Activations, f32 [M][K], standard normal by Box-Muller on two uniforms."""
    n = M * K
    raw = stream(seed, SID_X, 2 * n)
    u1 = 1.0 - uniform01(raw[0::2])  # (0, 1]
    u2 = uniform01(raw[1::2])
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return np.ascontiguousarray(z.astype(np.float32).reshape(M, K))


@dataclass(frozen=True)
class Workload:
    """One synthetic GEMV problem: y[M][N] from x[M][K] and an N x K one-bit matrix."""

    name: str
    M: int
    K: int
    N: int
    scale_lo: float
    scale_hi: float
    perm: int  # 0 = none, 1 = ssm_out tiled->grouped head permutation (K == 6144)
    seed: int
    extra: dict = field(default_factory=dict, compare=False)

    def weight_bytes(self) -> int:
        return self.K * self.N // 8 + 2 * self.N * (self.K // 128)

    def algorithmic_bytes(self) -> int:
        """Bits + fp16 scales + f32 x + f32 y + f32 signs for one call."""
        return self.weight_bytes() + 4 * self.M * self.K + 4 * self.M * self.N + 4 * self.K


_BASE_SEED = 0xB1711A00


def workload(name: str, M: int | None = None) -> Workload:
    """The named workloads (sizes of the Bonsai-27B folded matrices)."""
    table = {
        "tiny": (1, 1024, 256, 0.01, 0.05, 0, 1),
        "ffn_gate": (1, 5120, 17408, 0.005, 0.03, 0, 2),
        "ffn_down": (1, 17408, 5120, 0.005, 0.03, 0, 3),
        "ssm_out": (1, 6144, 5120, 0.005, 0.03, 1, 4),
        "gate_up": (1, 5120, 34816, 0.005, 0.03, 0, 5),
        "prefill": (1024, 5120, 17408, 0.005, 0.03, 0, 6),
        "attn_output": (1, 6144, 5120, 0.005, 0.03, 0, 7),
        # attention-side folded matrices (gated-delta qkv and output gate, full
        # attention's q-with-gate and k/v projections)
        "attn_qkv": (1, 5120, 10240, 0.005, 0.03, 0, 8),
        "attn_gate": (1, 5120, 6144, 0.005, 0.03, 0, 9),
        "attn_q": (1, 5120, 12288, 0.005, 0.03, 0, 10),
        "attn_kv": (1, 5120, 1024, 0.005, 0.03, 0, 11),
        # the folded vocabulary matrix (LM head, output.weight)
        "lm_head": (1, 5120, 248320, 0.005, 0.03, 0, 12),
    }
    m, K, N, lo, hi, perm, cid = table[name]
    if M is not None:
        m = M
    return Workload(name, m, K, N, lo, hi, perm, _BASE_SEED + cid)


def make_inputs(w: Workload):
    """(bits u32[N][K/32], scales u16[N][K/128], signs f32[K], x f32[M][K]) for a workload."""
    bits = random_bits(w.seed, w.N, w.K)
    scales = random_scales(w.seed, w.N, w.K, w.scale_lo, w.scale_hi)
    signs = random_signs(w.seed, w.K)
    x = random_x(w.seed, w.M, w.K)
    return bits, scales, signs, x


def sample_rows(seed: int, N: int, count: int) -> np.ndarray:
    """A sorted, duplicate-free sample of at most ``count`` output rows that always holds row 0 and row N-1."""
    count = max(2, min(count, N))
    r = np.unique((stream(seed, 99, 4 * count) % np.uint64(N)).astype(np.int64))
    r = r[(r != 0) & (r != N - 1)][: count - 2]
    return np.unique(np.concatenate([[0, N - 1], r]).astype(np.int64))


def q1g128_blob(bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The same weights in the stored Q1G128 form of the "Inside the One-Bit Engine" page
    (embedding-lookup station): one uint32 array holding first the fp16 scales, two per word
    (scale index n*(K/128) + g; the even index in the low 16 bits), then the bit words
    [N][K/32].  Layout only; N*K/256 + N*K/32 words."""
    s = np.ascontiguousarray(scales, dtype=np.uint16).reshape(-1).astype(np.uint32)
    if s.size % 2:
        raise ValueError("an even number of scales (K is a multiple of 1024)")
    words = s[0::2] | (s[1::2] << np.uint32(16))
    return np.concatenate([words, np.ascontiguousarray(bits, dtype=np.uint32).reshape(-1)])

