"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (scipy's Sylvester Hadamard matrix, numpy's float16 decoder, torch's
bfloat16 cast, numpy's unpackbits), a closed form, an invariant, a value the
pages print, or a brute-force dense product built independently.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _page_facts():
    facts = {}
    with open(os.path.join(GOLDEN, "page_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                facts[k] = v
    return facts


# ---------------------------------------------------------------- format decoders

def test_f16_decoder_matches_numpy_on_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(p)) for p in pats])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    # subnormals exist in real scale data (5.96e-08 on the engine page): 2^-24
    assert oracle_lib.f16_to_f64(1) == 2.0 ** -24


def test_bf16_rounding_matches_torch(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-3).astype(np.float32),
        np.array([1.0, -1.0, 1.00390625, 1.01171875, 3.0e38, 1e-39, -2.5e-41], dtype=np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_lib.round_bf16(float(a)) for a in v])
    assert np.array_equal(ref, got)


# ---------------------------------------------------------------- the transform

def test_wht_equals_scipy_sylvester_matrix(oracle_lib):
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    rng = np.random.default_rng(1)
    v = rng.standard_normal(1024)
    np.testing.assert_allclose(oracle_lib.wht_block(v), H @ v / 32.0, rtol=0, atol=1e-12)
    for j in (0, 1, 2, 511, 512, 777, 1023):
        e = np.zeros(1024)
        e[j] = 1.0
        np.testing.assert_array_equal(oracle_lib.wht_block(e), H[:, j] / 32.0)


def test_wht_is_an_involution_and_preserves_length(oracle_lib):
    rng = np.random.default_rng(2)
    v = rng.standard_normal(1024)
    w = oracle_lib.wht_block(v)
    np.testing.assert_allclose(oracle_lib.wht_block(w), v, rtol=0, atol=1e-12)
    assert math.isclose(np.linalg.norm(w), np.linalg.norm(v), rel_tol=1e-13)


def test_wht_of_constant_block(oracle_lib):
    c = 0.37
    w = oracle_lib.wht_block(np.full(1024, c))
    expect = np.zeros(1024)
    expect[0] = 32.0 * c
    np.testing.assert_allclose(w, expect, rtol=0, atol=1e-12)


def test_inverse_order_round_trips(oracle_lib):
    """Embedding order h = signs * WHT(z) undoes z = WHT(signs * x) (Pulse spec, fold section)."""
    K = 2048
    signs = synth.random_signs(11, K)
    x = synth.random_x(11, 1, K)
    z = oracle_lib.rotate(x, signs, 0)[0]
    h = oracle_lib.inverse_rotate(z, signs)
    np.testing.assert_allclose(h, x[0].astype(np.float64), rtol=0, atol=1e-12)
    # negative control: the forward order applied twice does not come back
    twice = oracle_lib.rotate(z.astype(np.float32)[None, :], signs, 0)[0]
    assert np.linalg.norm(twice - x[0]) > 0.5 * np.linalg.norm(x[0])


# ---------------------------------------------------------------- the permutation

def test_permutation_is_a_bijection(oracle_lib):
    v = np.arange(6144, dtype=np.float64)
    p = oracle_lib.permute_tiled_to_grouped(v)
    assert sorted(p.tolist()) == v.tolist()


def test_permutation_moves_heads_to_their_parent(oracle_lib):
    """Tiled value head h belongs to key head h % 16 (Pulse head-mapping table); after
    tiled->grouped, the grouped value head j must belong to key head j // 3, the blocked
    order attention already uses (h = kv*rep + r)."""
    f = _page_facts()
    hd, nk, rep = (int(s) for s in f["perm_tiled"].split(","))
    assert int(f["gdn_value_heads"]) == nk * rep and int(f["gdn_key_heads"]) == nk
    tiled = np.repeat(np.arange(nk * rep) % nk, hd).astype(np.float64)
    grouped = oracle_lib.permute_tiled_to_grouped(tiled)
    expect = np.repeat(np.arange(nk * rep) // rep, hd).astype(np.float64)
    np.testing.assert_array_equal(grouped, expect)
    # within a head the 128 lanes stay in order
    lanes = np.tile(np.arange(hd), nk * rep).astype(np.float64)
    np.testing.assert_array_equal(oracle_lib.permute_tiled_to_grouped(lanes), lanes)


# ---------------------------------------------------------------- the one-bit product

def _small_problem(N, K, seed):
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.01, 0.05)
    rng = np.random.default_rng(seed)
    xt = rng.standard_normal((1, K))
    return bits, scales, xt


def test_all_ones_and_all_zeros_rows(oracle_lib):
    N, K = 3, 1024
    _, scales, xt = _small_problem(N, K, 5)
    s = scales.view(np.float16).astype(np.float64)
    group_sums = xt[0].reshape(K // 128, 128).sum(axis=1)
    ones = np.full((N, K // 32), 0xFFFFFFFF, dtype=np.uint32)
    zeros = np.zeros((N, K // 32), dtype=np.uint32)
    np.testing.assert_allclose(oracle_lib.product(ones, scales, xt)[0], s @ group_sums, rtol=1e-13)
    np.testing.assert_allclose(oracle_lib.product(zeros, scales, xt)[0], -(s @ group_sums), rtol=1e-13)


def test_single_bit_flip_changes_output_by_twice_scaled_input(oracle_lib):
    """First station of the engine page: flipping one bit moves the sum by 2*s*x_k."""
    N, K = 4, 2048
    bits, scales, xt = _small_problem(N, K, 6)
    base = oracle_lib.product(bits, scales, xt)[0]
    for n, k in ((0, 0), (1, 31), (2, 777), (3, 2047)):
        flipped = bits.copy()
        flipped[n, k >> 5] ^= np.uint32(1 << (k & 31))
        now = oracle_lib.product(flipped, scales, xt)[0]
        new_bit = (int(flipped[n, k >> 5]) >> (k & 31)) & 1
        s = float(scales[n, k >> 7:(k >> 7) + 1].view(np.float16)[0])
        delta = (2.0 if new_bit else -2.0) * s * xt[0, k]
        assert math.isclose(now[n] - base[n], delta, rel_tol=1e-9, abs_tol=1e-14)
        others = [i for i in range(N) if i != n]
        np.testing.assert_array_equal(now[others], base[others])


def test_dequantized_group_length(oracle_lib):
    f = _page_facts()
    N, K = 2, 1024
    bits, scales, _ = _small_problem(N, K, 8)
    w = oracle_lib.dequant_row(bits, scales, 1)
    for g in range(K // 128):
        s = float(scales[1, g:g + 1].view(np.float16)[0])
        length = np.linalg.norm(w[g * 128:(g + 1) * 128])
        assert math.isclose(length / s, math.sqrt(128), rel_tol=1e-13)
        assert round(length / s, 3) == float(f["group_length_over_scale"])


def _dense_reference(bits, scales, signs, perm, x):
    """y = Wd @ blockdiag(H/32) @ diag(signs) @ P @ x, with every factor built from
    library routines (unpackbits, float16 view, scipy's Hadamard, numpy transpose)."""
    N = bits.shape[0]
    K = bits.shape[1] * 32
    pm = np.unpackbits(bits.view(np.uint8), bitorder="little").reshape(N, K).astype(np.float64)
    s = np.repeat(scales.view(np.float16).astype(np.float64), 128, axis=1)
    Wd = (2.0 * pm - 1.0) * s
    H = scipy.linalg.hadamard(1024).astype(np.float64) / 32.0
    Hb = np.kron(np.eye(K // 1024), H)
    xs = x.astype(np.float64)
    if perm:
        # tiled [hd=128, nk=16, rep=3] (innermost first) is C-order (3, 16, 128);
        # grouped [hd, rep, nk] is C-order (16, 3, 128)
        xs = xs.reshape(-1, 3, 16, 128).transpose(0, 2, 1, 3).reshape(-1, K)
    xs = xs * signs.astype(np.float64)[None, :]
    return (Wd @ (Hb @ xs.T)).T


@pytest.mark.parametrize("N,K,perm", [(8, 1024, 0), (5, 2048, 0), (4, 6144, 1), (3, 6144, 0)])
def test_whole_method_against_dense_brute_force(oracle_lib, N, K, perm):
    seed = 100 + N + K + perm
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, 2, K)
    got = oracle_lib.forward(bits, scales, signs, perm, x)
    ref = _dense_reference(bits, scales, signs, perm, x)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_row_subset_equals_full_rows(oracle_lib):
    w = synth.workload("tiny")
    bits, scales, signs, x = synth.make_inputs(w)
    full = oracle_lib.forward(bits, scales, signs, 0, x)
    rows = np.array([0, 17, 100, 255])
    np.testing.assert_array_equal(oracle_lib.forward(bits, scales, signs, 0, x, rows), full[:, rows])


def test_bf16_variant_stays_within_prefill_tolerance(oracle_lib):
    N, K = 64, 2048
    bits = synth.random_bits(3, N, K)
    scales = synth.random_scales(3, N, K, 0.005, 0.03)
    signs = synth.random_signs(3, K)
    x = synth.random_x(3, 4, K)
    exact = oracle_lib.forward(bits, scales, signs, 0, x)
    approx = oracle_lib.forward(bits, scales, signs, 0, x, round_bf16=True)
    rel = np.linalg.norm(approx - exact, axis=1) / np.linalg.norm(exact, axis=1)
    assert 1e-5 < rel.max() < 1e-2


def test_tiny_workload_regression_fixture(oracle_lib):
    """Known answer on the 256-row probe (the engine page's subgroup probe checks 256 rows)."""
    ref = np.loadtxt(os.path.join(GOLDEN, "tiny_oracle.txt"))
    w = synth.workload("tiny")
    bits, scales, signs, x = synth.make_inputs(w)
    y = oracle_lib.forward(bits, scales, signs, 0, x)[0]
    assert y.shape == (256,)
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- sizes and inputs

def test_storage_accounting_matches_page_figures():
    f = _page_facts()
    K = 5120
    row = K // 8 + 2 * (K // 128)
    assert row == int(f["row_bytes_k5120"])
    assert row * int(f["token_embd_rows"]) == int(f["token_embd_bytes"])
    widths = [int(v) for v in f["sign_widths"].split(",")]
    assert sum(widths) == int(f["sign_values"])
    assert all(wd % int(f["wht_block"]) == 0 for wd in widths)
    w = synth.Workload("embd", 1, K, int(f["token_embd_rows"]), 0.01, 0.02, 0, 1)
    assert w.weight_bytes() == int(f["token_embd_bytes"])


def test_generator_bits_are_fair_coins():
    f = _page_facts()
    bits = synth.random_bits(42, 512, 5120)
    pm = np.unpackbits(bits.view(np.uint8), bitorder="little").reshape(512, 40, 128)
    var = pm.sum(axis=2).var()
    assert abs(var - float(f["fair_coin_popcount_variance"])) < 1.5
    signs = synth.random_signs(42, 17408)
    assert set(np.unique(signs).tolist()) == {-1.0, 1.0}
    x = synth.random_x(42, 4, 4096)
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1.0) < 0.05
    s = synth.random_scales(42, 100, 1024, 0.005, 0.03).view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 - 1e-5 and s.max() <= 0.03 + 1e-5


def test_generator_counter_mode_slices_agree():
    a = synth.stream(5, 1, 1000)
    b = synth.stream(5, 1, 300, start=700)
    np.testing.assert_array_equal(a[700:], b)


# ------------------------------------------------------------------ NEXT rows: SiLU, MLP block, embedding

def test_silu_against_scipy_expit_and_identities(oracle_lib):
    """SiLU(g) = g / (1 + e^-g) ("Inside the One-Bit Engine", MLP station) against
    scipy.special.expit (the logistic function, a library routine) times g, and the
    identities silu(0) = 0, silu(g) - silu(-g) = g, silu(g) -> g for large g."""
    import scipy.special

    g = np.concatenate([np.linspace(-30, 30, 1201), [-700.0, 700.0, 0.0]])
    got = oracle_lib.silu(g)
    np.testing.assert_allclose(got, g * scipy.special.expit(g), rtol=1e-14, atol=1e-300)
    assert oracle_lib.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(got - oracle_lib.silu(-g), g, rtol=1e-13, atol=1e-13)
    assert oracle_lib.silu(np.array([700.0]))[0] == 700.0
    assert abs(oracle_lib.silu(np.array([-700.0]))[0]) < 1e-300
    # the small dip below zero: minimum near g = -1.278, value -0.2785
    assert abs(oracle_lib.silu(np.array([-1.2784645]))[0] + 0.2784645) < 1e-6


def test_mlp_block_against_dense_brute_force(oracle_lib):
    """down(silu(gate x) * (up x)) with the first F rows of gate_up as gate, built from
    the dense brute-force product and scipy's logistic function."""
    import scipy.special

    F, Hd = 1024, 2048
    sgu, sd = 321, 654
    gu = (synth.random_bits(sgu, 2 * F, Hd), synth.random_scales(sgu, 2 * F, Hd, 0.005, 0.03),
          synth.random_signs(sgu, Hd), 0)
    dn = (synth.random_bits(sd, 6, F), synth.random_scales(sd, 6, F, 0.005, 0.03), synth.random_signs(sd, F), 0)
    x = synth.random_x(7, 2, Hd)
    got = oracle_lib.mlp(gu, dn, x)
    h = _dense_reference(*gu, x)
    mid = h[:, :F] * scipy.special.expit(h[:, :F]) * h[:, F:]
    ref = _dense_reference(*dn, mid)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)
    # swapping the roles of gate and up changes the answer (the order is pinned)
    swapped = (np.concatenate([gu[0][F:], gu[0][:F]]), np.concatenate([gu[1][F:], gu[1][:F]]), gu[2], 0)
    assert np.linalg.norm(oracle_lib.mlp(swapped, dn, x) - got) > 0.1 * np.linalg.norm(got)


def test_embedding_closed_form_and_brute_force(oracle_lib):
    """h = signs * WHT(z) / 32 per block (Pulse spec, embedding order).  Closed form: an
    all-ones row with one scale s per block gives 32 s at each block's first position
    (times its sign) and 0 elsewhere; and against the dense Hadamard matrix product."""
    import scipy.linalg

    K, N = 2048, 4
    bits = synth.random_bits(77, N, K)
    scales = synth.random_scales(77, N, K, 0.01, 0.05)
    signs = synth.random_signs(77, K)
    bits[2, :] = 0xFFFFFFFF
    scales[2, :] = np.float16(0.03125).view(np.uint16)  # one scale for the whole row
    h = oracle_lib.embed(bits, scales, signs, [2])[0]
    expect = np.zeros(K)
    expect[0::1024] = 32 * 0.03125
    np.testing.assert_allclose(h, expect * signs, rtol=0, atol=1e-15)
    H = scipy.linalg.hadamard(1024).astype(np.float64) / 32.0
    Hb = np.kron(np.eye(K // 1024), H)
    pm = np.unpackbits(bits.view(np.uint8), bitorder="little").reshape(N, K).astype(np.float64)
    Wd = (2 * pm - 1) * np.repeat(scales.view(np.float16).astype(np.float64), 128, axis=1)
    got = oracle_lib.embed(bits, scales, signs, [0, 3, 1])
    ref = (Hb @ Wd[[0, 3, 1]].T).T * signs.astype(np.float64)[None, :]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ NEXT row: the stored Q1G128 form

def _dense_weights(bits, scales):
    """w[n][k] = (2 bit - 1) * scale through numpy's own bit unpacking and fp16 decoding."""
    N, W = bits.shape
    pm = np.unpackbits(np.ascontiguousarray(bits).view(np.uint8), bitorder="little").reshape(N, 32 * W)
    sc = np.repeat(np.ascontiguousarray(scales).view(np.float16).astype(np.float64), 128, axis=1)
    return (2.0 * pm - 1.0) * sc


def test_q1g128_stored_form_size_matches_page_figures():
    """One row is 720 bytes at K = 5120 and the vocabulary tensor 178,790,400 bytes."""
    from hadamard_rotated_binary_gb300 import q1g128_words

    f = _page_facts()
    K, N = 5120, 3
    blob = synth.q1g128_blob(synth.random_bits(5, N, K), synth.random_scales(5, N, K, 0.01, 0.02))
    assert blob.dtype == np.uint32 and 4 * blob.size == N * int(f["row_bytes_k5120"])
    assert 4 * q1g128_words(int(f["token_embd_rows"]), K) == int(f["token_embd_bytes"])
    assert 4 * q1g128_words(N, K) == 4 * blob.size


def test_q1g128_reader_follows_the_page_indexing(oracle_lib):
    """A hand-made tensor: scales 1..8 (one row, K = 1024), bit word 0 = 0b101.  Scale index 0
    sits in the low half of word 0 (unpack2x16float's first component is bits 0..15), and the bit
    words start right after the N*K/256 scale words."""
    K, N = 1024, 1
    scales = np.array([[np.float16(v).view(np.uint16) for v in range(1, 9)]], dtype=np.uint16)
    bits = np.zeros((N, K // 32), dtype=np.uint32)
    bits[0, 0] = 0b101
    bits[0, 31] = 0x80000000  # the last weight of the row
    blob = synth.q1g128_blob(bits, scales)
    assert blob[0] == 0x40003C00 and blob.size == 4 + 32  # 2.0 high, 1.0 low; 4 scale words
    got = [oracle_lib.q1g128_weight(blob, N, K, 0, k) for k in (0, 1, 2, 127, 128, 1023)]
    assert got == [1.0, -1.0, 1.0, -1.0, -2.0, 8.0]


def test_q1g128_reader_against_numpy_dequantization(oracle_lib):
    """Every weight of a random 3 x 2048 tensor read from the stored form equals numpy's own
    unpacking; a packer with the two halves of each scale word swapped fails (negative control)."""
    N, K = 3, 2048
    bits = synth.random_bits(11, N, K)
    scales = synth.random_scales(11, N, K, 0.01, 0.05)
    dense = _dense_weights(bits, scales)
    blob = synth.q1g128_blob(bits, scales)
    got = np.array([[oracle_lib.q1g128_weight(blob, N, K, n, k) for k in range(K)] for n in range(N)])
    np.testing.assert_array_equal(got, dense)
    s = scales.reshape(-1).astype(np.uint32)
    swapped = np.concatenate([s[1::2] | (s[0::2] << np.uint32(16)), bits.reshape(-1)])
    bad = np.array([oracle_lib.q1g128_weight(swapped, N, K, 0, k) for k in range(0, K, 128)])
    assert not np.array_equal(bad, dense[0, ::128])

