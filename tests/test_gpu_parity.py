"""GPU parity of the CUDA path (through the C-ABI) against the CPU oracle.

Every case draws its inputs from the seeded generator, runs the library on
cuda:0, and compares with the oracle's f64 evaluation of the same inputs:
max relative L2 error per token row <= 1e-5 on the decode path and <= 1e-2
on the tensor-core path.  Full-size cases of the five workloads compare every
output (the prefill case takes the OpenMP oracle some seconds); the other
shapes and the largest widths compare a seeded sample of rows (always
including the first and last).
"""
import os

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

DECODE_TOL = 1e-5
PREFILL_TOL = 1e-2
BF16_DIAG_TOL = 1e-3


@pytest.fixture(scope="module")
def hrb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hadamard_rotated_binary_gb300 import build as hbuild

    hbuild.build()
    oracle.build()
    import hadamard_rotated_binary_gb300 as m

    return m


def make_layer(hrb, bits, scales, signs, perm):
    tb = torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).cuda()
    ts = torch.from_numpy(np.ascontiguousarray(scales).view(np.int16)).cuda()
    tg = torch.from_numpy(np.ascontiguousarray(signs)).cuda()
    return hrb.BitLinear(tb, ts, tg, perm)


def run(layer, x, path=None):
    if path is not None:
        layer.set_path(path)
    y = layer(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    return y.cpu().numpy().astype(np.float64)


def max_rel_l2(y, ref):
    num = np.linalg.norm(y - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    return float((num / den).max())


def rel_err(y, ref):
    """max_rel_l2 per token row; with fewer than 32 outputs per token that norm is the error of a
    handful of dot products, any of which can be near zero by cancellation, so there the norm is
    taken over the tokens of each output instead (the transpose)."""
    if y.shape[1] >= 32:
        return max_rel_l2(y, ref)
    return max_rel_l2(np.ascontiguousarray(y.T), np.ascontiguousarray(ref.T))


def inputs(name, M=None):
    w = synth.workload(name, M)
    return (w,) + synth.make_inputs(w)


# ------------------------------------------------------------------ decode

def test_tiny_probe(hrb):
    w, bits, scales, signs, x = inputs("tiny")
    y = run(make_layer(hrb, bits, scales, signs, w.perm), x)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL
    # known-answer probe of 256 rows: no output off by more than 0.5
    assert int((np.abs(y - ref) > 0.5).sum()) == 0
    golden = np.loadtxt(os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.txt"))
    assert max_rel_l2(y, golden[None, :]) <= DECODE_TOL


@pytest.mark.parametrize("name", ["ffn_gate", "ffn_down", "ssm_out", "attn_output", "attn_qkv", "attn_gate",
                                  "attn_q", "attn_kv"])
def test_decode_full_size_every_output(hrb, name):
    w, bits, scales, signs, x = inputs(name)
    y = run(make_layer(hrb, bits, scales, signs, w.perm), x)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL


def test_ssm_out_permutation_matters(hrb):
    """The same ssm_out weights without the permutation must not match (Pulse spec:
    skipping the permutation gives an unrelated answer)."""
    w, bits, scales, signs, x = inputs("ssm_out")
    y = run(make_layer(hrb, bits, scales, signs, 0), x)
    ref = oracle.forward(bits, scales, signs, 1, x)
    assert max_rel_l2(y, ref) > 0.5


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gate_up_decode_sweep(hrb, M):
    """Config 4 below M = 64, every output: the decode GEMV at M = 1 and 4 (two tokens per
    pass), the exact three-digit tensor path at M = 16."""
    w, bits, scales, signs, x = inputs("gate_up", M)
    y = run(make_layer(hrb, bits, scales, signs, w.perm), x)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL


@pytest.mark.parametrize("name,M", [("attn_qkv", 4), ("attn_qkv", 16), ("attn_gate", 16), ("attn_q", 8),
                                    ("attn_kv", 3), ("attn_output", 5)])
def test_attention_shapes_small_batch(hrb, name, M):
    """The attention-side folded shapes at small M (decode GEMV to M = 6, exact tensor path above), sampled rows.
    On 152 SMs the exact cases run split-K over clusters: attn_qkv at M = 16 two CTAs per SM split 3,
    attn_q at M = 8 two per SM split 2, attn_gate at M = 16 one per SM split 2 (the resident-cluster
    limit cuts 3 to 2)."""
    w, bits, scales, signs, x = inputs(name, M)
    y = run(make_layer(hrb, bits, scales, signs, w.perm), x)
    rows = synth.sample_rows(w.seed, w.N, 768)
    ref = oracle.forward(bits, scales, signs, w.perm, x, rows)
    assert max_rel_l2(y[:, rows], ref) <= DECODE_TOL


def test_gate_up_m64_both_paths(hrb):
    """Config 4 at M = 64, every output: the bf16 tensor path (the automatic choice) within
    1e-2 and the decode GEMV (forced) within 1e-5."""
    w, bits, scales, signs, x = inputs("gate_up", 64)
    layer = make_layer(hrb, bits, scales, signs, w.perm)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    y_auto = run(layer, x)  # M = 64 selects the tensor-core path
    assert max_rel_l2(y_auto, ref) <= PREFILL_TOL
    y_dec = run(layer, x, path=hrb.PATH_DECODE)
    assert max_rel_l2(y_dec, ref) <= DECODE_TOL


# ------------------------------------------------------------------ prefill

def test_prefill_full_size_every_output(hrb):
    """Config 5 (1024 tokens through the 17,408 x 5,120 matrix), every output against the
    oracle within 1e-2."""
    w, bits, scales, signs, x = inputs("prefill")
    y = run(make_layer(hrb, bits, scales, signs, w.perm), x)
    assert np.all(np.isfinite(y))
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y, ref) <= PREFILL_TOL
    # Against the oracle with bf16-rounded activations what remains is the f32
    # accumulation and the few elements whose rounding to bf16 flips because
    # the kernel rounds its f32 value and the oracle its f64 value (one bf16
    # ulp, 2^-8 relative, each): well under 1e-3.  A seeded sample of rows.
    rows = synth.sample_rows(w.seed, w.N, 1024)
    ref16 = oracle.forward(bits, scales, signs, w.perm, x, rows, round_bf16=True)
    assert max_rel_l2(y[:, rows], ref16) <= BF16_DIAG_TOL


@pytest.mark.parametrize("N,K,M,perm", [(300, 2048, 65, 0), (129, 1024, 130, 0), (256, 6144, 128, 1),
                                        (1000, 3072, 200, 0), (1000, 2048, 2600, 0), (5000, 6144, 520, 1),
                                        (2048, 1024, 1900, 0), (1, 1024, 65, 0), (100, 2048, 300, 0)])
def test_prefill_ragged(hrb, N, K, M, perm):
    """Ragged N and M on the bf16 tensor path, every output.  Three cases have more tiles than
    SMs (1000 x 2600: 8 x 21 tiles, 5000 x 520: 40 x 5, 2048 x 1900: 16 x 15), so they run on
    the persistent grid with ragged edge tiles.  On 152 SMs the first two leave 16 and 48 tiles
    past the last full wave, which run as a second, split-K launch; the third leaves 88 (more
    than half the SMs), which stay in the persistent grid.  N = 1 and 100: fewer rows than one
    128-row tile (the bits copy reads past N, the epilogue writes the rows that exist)."""
    seed = 7 + N + K + M
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    y = run(make_layer(hrb, bits, scales, signs, perm), x)
    ref = oracle.forward(bits, scales, signs, perm, x)
    assert rel_err(y, ref) <= PREFILL_TOL
    ref16 = oracle.forward(bits, scales, signs, perm, x, round_bf16=True)
    assert rel_err(y, ref16) <= BF16_DIAG_TOL


def test_prefill_whole_waves_no_tail(hrb):
    """Tiles an exact multiple of the SMs (2 waves of 128-token tiles): the persistent grid with
    no split tail launch.  Sampled rows within 1e-2 and the bf16 diagnostic."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K, M = sms * 128, 1024, 256
    seed = 17
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    layer = make_layer(hrb, bits, scales, signs, 0)
    assert layer.plan(M) == (hrb.PATH_PREFILL, 2)
    y = run(layer, x)
    rows = synth.sample_rows(seed, N, 512)
    ref = oracle.forward(bits, scales, signs, 0, x, rows)
    assert max_rel_l2(y[:, rows], ref) <= PREFILL_TOL
    ref16 = oracle.forward(bits, scales, signs, 0, x, rows, round_bf16=True)
    assert max_rel_l2(y[:, rows], ref16) <= BF16_DIAG_TOL


@pytest.mark.parametrize("N,K,M", [(1000, 2048, 33), (20000, 1024, 50), (5120, 17408, 64), (300, 1024, 1),
                                   (1, 2048, 64), (7, 1024, 20)])
def test_prefill_narrow_tiles(hrb, N, K, M):
    """The bf16 path at most 64 tokens runs 64-token tiles: one CTA per SM with split-K for
    few tiles (8 tiles split 2; 40 tiles split 3 at K = 17,408), two per SM when the tiles fill
    every SM (157 tiles on 152 SMs), ragged N and M; the path is forced where M alone would
    pick the decode GEMV; N = 1 and 7, fewer rows than one tile.  Every output (a sample of rows
    at K = 17,408) within 1e-2, and within the bf16 diagnostic."""
    seed = 13 + N + K + M
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    layer = make_layer(hrb, bits, scales, signs, 0)
    layer.set_path(hrb.PATH_PREFILL)
    assert layer.plan(M) == (hrb.PATH_PREFILL, 2)  # the rotation and one GEMM launch
    y = run(layer, x)
    rows = synth.sample_rows(seed, N, 320) if K > 8192 else None
    ref = oracle.forward(bits, scales, signs, 0, x, rows)
    yy = y[:, rows] if rows is not None else y
    assert rel_err(yy, ref) <= PREFILL_TOL
    ref16 = oracle.forward(bits, scales, signs, 0, x, rows, round_bf16=True)
    assert rel_err(yy, ref16) <= BF16_DIAG_TOL


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("N,K,M", [(1, 1024, 1), (100, 1024, 1), (31, 2048, 3), (1000, 3072, 5),
                                   (4097, 1024, 2), (33, 17408, 1)])
def test_decode_ragged(hrb, N, K, M):
    seed = 11 + N + K + M
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    y = run(make_layer(hrb, bits, scales, signs, 0), x)
    ref = oracle.forward(bits, scales, signs, 0, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL


@pytest.mark.parametrize("N,K,M,path", [(300, 65536, 1, "decode"), (257, 65536, 3, "exact"),
                                         (129, 81920, 1, "decode")])
def test_maximum_widths(hrb, N, K, M, path):
    """Wide K: 128 and 160 slices of 512 (more slices than SMs: the decode GEMV splits the units
    over the grid with the global-scratch split-K), and the exact tensor path over 512 K-groups."""
    seed = 19 + N + K + M
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    layer = make_layer(hrb, bits, scales, signs, 0)
    y = run(layer, x, path=hrb.PATH_DECODE if path == "decode" else hrb.PATH_TC_EXACT)
    ref = oracle.forward(bits, scales, signs, 0, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL


def test_prefill_many_tokens(hrb):
    """M = 4096 tokens (32 token tiles per weight-row tile) on the bf16 tensor path, sampled rows."""
    N, K, M = 384, 2048, 4096
    seed = 91
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    y = run(make_layer(hrb, bits, scales, signs, 0), x)
    ref = oracle.forward(bits, scales, signs, 0, x)
    assert max_rel_l2(y, ref) <= PREFILL_TOL


def test_prefill_path_forced_at_one_token(hrb):
    w, bits, scales, signs, x = inputs("tiny")
    y = run(make_layer(hrb, bits, scales, signs, 0), x, path=hrb.PATH_PREFILL)
    ref = oracle.forward(bits, scales, signs, 0, x)
    assert max_rel_l2(y, ref) <= PREFILL_TOL


def test_degenerate_all_ones_and_zero_input(hrb):
    N, K = 64, 2048
    scales = synth.random_scales(3, N, K, 0.005, 0.03)
    signs = synth.random_signs(3, K)
    x = synth.random_x(3, 2, K)
    ones = np.full((N, K // 32), 0xFFFFFFFF, dtype=np.uint32)
    layer = make_layer(hrb, ones, scales, signs, 0)
    y = run(layer, x)
    ref = oracle.forward(ones, scales, signs, 0, x)
    assert max_rel_l2(y, ref) <= DECODE_TOL
    z = run(layer, np.zeros_like(x))
    assert np.all(z == 0.0)


def test_repeat_calls_are_bitwise_identical(hrb):
    w, bits, scales, signs, x = inputs("ffn_down")
    layer = make_layer(hrb, bits, scales, signs, 0)
    xd = torch.from_numpy(x).cuda()
    a = layer(xd).clone()
    b = layer(xd).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_alternating_token_counts_reuse_scratch(hrb):
    w, bits, scales, signs, x = inputs("ffn_gate", 8)
    layer = make_layer(hrb, bits, scales, signs, 0)
    rows = synth.sample_rows(w.seed, w.N, 512)
    ref = oracle.forward(bits, scales, signs, 0, x, rows)
    for m in (8, 1, 3, 8):
        y = run(layer, x[:m].copy())
        assert max_rel_l2(y[:, rows], ref[:m]) <= DECODE_TOL


def test_cuda_graph_replay_matches(hrb):
    w, bits, scales, signs, x = inputs("ffn_gate")
    layer = make_layer(hrb, bits, scales, signs, 0)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty((1, w.N), device="cuda")
    layer(xd, out=yd)  # warm-up allocates the scratch
    torch.cuda.synchronize()
    eager = yd.clone()
    yd.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                layer(xd, out=yd, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yd, eager)


@pytest.mark.parametrize("name,M", [("ssm_out", 1), ("ffn_down", 2), ("attn_kv", 70)])
def test_forward_host_buffers(hrb, name, M):
    """Host buffers, pageable (numpy) and page-locked (torch pin_memory): the same y, bit for
    bit, as the device-buffer call, within tolerance of the oracle; on the decode, scratch
    split-K and bf16 tensor paths."""
    w, bits, scales, signs, x = inputs(name, M)
    layer = make_layer(hrb, bits, scales, signs, w.perm)
    y_dev = layer(torch.from_numpy(x).cuda()).cpu().numpy()
    y = np.full((M, w.N), np.nan, dtype=np.float32)
    layer.forward_host(x, y)
    xp = torch.from_numpy(x).pin_memory()
    yp = torch.full((M, w.N), float("nan")).pin_memory()
    layer.forward_host(xp.numpy(), yp.numpy())
    assert layer.get_error() == 0
    np.testing.assert_array_equal(y, y_dev)
    np.testing.assert_array_equal(yp.numpy(), y_dev)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y.astype(np.float64), ref) <= (DECODE_TOL if M < 64 else PREFILL_TOL)


# ------------------------------------------------------------------ exact tensor path (7 <= M < 64; any M forced)

@pytest.mark.parametrize("M,perm", [(70, 0), (9, 0), (9, 1)])
def test_rotation_with_unaligned_activations(hrb, M, perm):
    """x at an address that is not 16-byte aligned (a view one float into a buffer) takes the
    rotation's scalar loads: the same y, bit for bit, as from an aligned copy, on the bf16
    (M = 70) and the exact (M = 9) tensor paths, with and without the permutation."""
    K, N = 6144, 320
    seed = 71 + M + perm
    bits, scales = synth.random_bits(seed, N, K), synth.random_scales(seed, N, K, 0.005, 0.03)
    signs, x = synth.random_signs(seed, K), synth.random_x(seed, M, K)
    layer = make_layer(hrb, bits, scales, signs, perm)
    aligned = torch.from_numpy(x).cuda()
    buf = torch.empty(M * K + 1, dtype=torch.float32, device="cuda")
    shifted = buf[1:].view(M, K)
    shifted.copy_(aligned)
    assert shifted.data_ptr() % 16 != 0
    y1, y2 = layer(aligned), layer(shifted)
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    assert torch.equal(y1, y2)
    ref = oracle.forward(bits, scales, signs, perm, x)
    assert max_rel_l2(y1.cpu().numpy().astype(np.float64), ref) <= (PREFILL_TOL if M >= 64 else DECODE_TOL)


@pytest.mark.parametrize("M,N,K,perm", [(2, 256, 1024, 0), (16, 1000, 2048, 0), (17, 384, 6144, 1),
                                        (40, 300, 3072, 0), (63, 129, 1024, 0), (100, 200, 1024, 0),
                                        (9, 1, 1024, 0), (16, 7, 2048, 0), (33, 100, 4096, 0)])
def test_tc_exact_path_every_tile_width(hrb, M, N, K, perm):
    """Activations split into three bf16 digits: f32-level results at both tile widths (64, 128),
    with the tokens spread over several tiles (M = 40, 63, 100), and with fewer rows than one
    128-row tile (N = 1, 7, 100: the bits copy reads past N, the epilogue writes the rows that
    exist; split-K over 2 and 4 K-group ranges at K = 2048 and 4096)."""
    seed = 23 + M + N + K
    bits = synth.random_bits(seed, N, K)
    scales = synth.random_scales(seed, N, K, 0.005, 0.03)
    signs = synth.random_signs(seed, K)
    x = synth.random_x(seed, M, K)
    layer = make_layer(hrb, bits, scales, signs, perm)
    y = run(layer, x, path=hrb.PATH_TC_EXACT)
    ref = oracle.forward(bits, scales, signs, perm, x)
    assert rel_err(y, ref) <= DECODE_TOL
    y_dec = run(layer, x, path=hrb.PATH_DECODE)
    assert rel_err(y_dec, ref) <= DECODE_TOL


def test_auto_path_choice(hrb):
    """M <= 6 -> table GEMV, 7..63 -> exact tensor path, >= 64 -> bf16 tensor path; all in tolerance."""
    w, bits, scales, signs, x = inputs("ffn_gate", 70)
    layer = make_layer(hrb, bits, scales, signs, 0)
    rows = synth.sample_rows(w.seed, w.N, 256)
    ref = oracle.forward(bits, scales, signs, 0, x, rows)
    for m, tol in ((1, DECODE_TOL), (2, DECODE_TOL), (5, DECODE_TOL), (6, DECODE_TOL), (7, DECODE_TOL),
                   (63, DECODE_TOL), (64, PREFILL_TOL), (70, PREFILL_TOL)):
        y = run(layer, np.ascontiguousarray(x[:m]))
        assert max_rel_l2(y[:, rows], ref[:m]) <= tol, m


def test_plan_reports_path_and_kernels(hrb):
    """bitlin_plan: the path of each M range, one kernel for the cluster split-K (10 slices at
    K = 5120), two (GEMV + sum) for 34 slices at K = 17408 and for 128 at K = 65536, two
    (rotation + GEMM) on the tensor paths, three on the bf16 path when the GEMM's tiles past its
    last full wave (fewer than half the SMs) run as a split-K launch of their own; a forced path
    is reported as forced."""
    gate = make_layer(hrb, *inputs("ffn_gate", 1)[1:4], 0)
    down = make_layer(hrb, *inputs("ffn_down", 1)[1:4], 0)
    assert [gate.plan(m) for m in (1, 2, 6, 7, 63, 64)] == [(1, 1), (1, 1), (1, 1), (3, 2), (3, 2), (2, 2)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for m in (256, 1024, 1900):
        tiles = 136 * -(-m // 128)  # 17408 rows / 128 per tile, 128 tokens per tile
        tail = tiles > sms and 0 < 2 * (tiles % sms) < sms
        assert gate.plan(m) == (2, 3 if tail else 2), (m, sms)
    assert down.plan(1) == (1, 2)
    wide = make_layer(hrb, synth.random_bits(3, 64, 65536), synth.random_scales(3, 64, 65536, 0.005, 0.03),
                      synth.random_signs(3, 65536), 0)
    assert wide.plan(1) == (1, 2)
    gate.set_path(1)
    assert gate.plan(200) == (1, 2)  # 200 tokens' partials do not fit shared memory: scratch + sum


# ------------------------------------------------------------------ MLP block (gate|up -> SiLU -> down)

def _mlp_pair(hrb, F, H, seed):
    gu = (synth.random_bits(seed, 2 * F, H), synth.random_scales(seed, 2 * F, H, 0.005, 0.03),
          synth.random_signs(seed, H), 0)
    dn = (synth.random_bits(seed + 1, H, F), synth.random_scales(seed + 1, H, F, 0.005, 0.03),
          synth.random_signs(seed + 1, F), 0)
    return gu, dn, make_layer(hrb, *gu), make_layer(hrb, *dn)


@pytest.mark.parametrize("M", [1, 4])
def test_mlp_block_full_size(hrb, M):
    """Bonsai-27B MLP shapes (5120 -> 2 x 17408 -> 5120) on the decode GEMVs (M = 1: one token
    per pass; M = 4: two), every output, <= 1e-5."""
    gu, dn, lgu, ldn = _mlp_pair(hrb, 17408, 5120, 0xB1711A00 + 5)
    x = synth.random_x(0xB1711A00 + 5, M, 5120)
    y = hrb.mlp_forward(lgu, ldn, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert lgu.get_error() == 0 and ldn.get_error() == 0
    ref = oracle.mlp(gu, dn, x)
    assert max_rel_l2(y.cpu().numpy().astype(np.float64), ref) <= DECODE_TOL


def test_mlp_block_bf16_path_and_forced_paths(hrb):
    """M = 64 runs both products on the bf16 tensor path (<= 1e-2); forcing the f32 decode
    GEMV on both handles gives <= 1e-5 at the same M."""
    gu, dn, lgu, ldn = _mlp_pair(hrb, 2048, 1024, 31)
    x = synth.random_x(32, 64, 1024)
    ref = oracle.mlp(gu, dn, x)
    y = hrb.mlp_forward(lgu, ldn, torch.from_numpy(x).cuda())
    assert max_rel_l2(y.cpu().numpy().astype(np.float64), ref) <= PREFILL_TOL
    lgu.set_path(hrb.PATH_DECODE)
    ldn.set_path(hrb.PATH_DECODE)
    y = hrb.mlp_forward(lgu, ldn, torch.from_numpy(x).cuda())
    assert max_rel_l2(y.cpu().numpy().astype(np.float64), ref) <= DECODE_TOL


def test_mlp_block_bf16_path_persistent_grids(hrb):
    """1280 tokens through a 2048 -> 2 x 1024 -> 2048 block on the bf16 tensor path: both
    products run persistent grids of more than one wave (gate_up 16 x 10 tiles, down 16 x 10),
    the down projection's rotation with SiLU(gate) * up; within 1e-2 of the oracle on sampled
    rows, and the same bits from a second call."""
    F, H, M = 1024, 2048, 1280
    gu, dn, lgu, ldn = _mlp_pair(hrb, F, H, 77)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert -(-2 * F // 128) * -(-M // 128) > sms and -(-H // 128) * -(-M // 128) > sms
    assert lgu.plan(M)[0] == ldn.plan(M)[0] == hrb.PATH_PREFILL
    x = synth.random_x(78, M, H)
    xd = torch.from_numpy(x).cuda()
    y1 = hrb.mlp_forward(lgu, ldn, xd)
    y2 = hrb.mlp_forward(lgu, ldn, xd)
    torch.cuda.synchronize()
    assert lgu.get_error() == 0 and ldn.get_error() == 0
    assert torch.equal(y1, y2)
    rows = synth.sample_rows(79, H, 192)
    ref = oracle.mlp(gu, dn, x, rows)
    assert max_rel_l2(y1.cpu().numpy()[:, rows].astype(np.float64), ref) <= PREFILL_TOL


def test_mlp_block_rejects_mismatched_pair(hrb):
    gu, dn, lgu, ldn = _mlp_pair(hrb, 1024, 1024, 41)
    w, bits, scales, signs, _ = inputs("tiny")
    other = make_layer(hrb, bits, scales, signs, 0)
    x = torch.zeros((1, 1024), dtype=torch.float32, device="cuda")
    with pytest.raises(hrb.BitlinError) as e:
        hrb.mlp_forward(other, ldn, x)  # other has N = 256, not 2 * 1024
    assert e.value.status == hrb.BITLIN_EINVAL


# ------------------------------------------------------------------ LM head + argmax

def _lm_head():
    N, K, seed = 248320, 5120, 0xB1711A00 + 12
    return (synth.random_bits(seed, N, K), synth.random_scales(seed, N, K, 0.005, 0.03),
            synth.random_signs(seed, K), seed)


@pytest.mark.parametrize("M", [1, 3])
def test_lm_head_argmax_full_size(hrb, M):
    """The folded vocabulary matrix (248,320 x 5,120): scores within 1e-5 of the oracle; the
    id is the argmax of the scores the GPU computed (same precision decides), and its oracle
    score is the oracle's maximum up to that tolerance."""
    bits, scales, signs, seed = _lm_head()
    x = synth.random_x(seed, M, 5120)
    layer = make_layer(hrb, bits, scales, signs, 0)
    logits = torch.empty((M, bits.shape[0]), dtype=torch.float32, device="cuda")
    ids = layer.argmax(torch.from_numpy(x).cuda(), logits=logits).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    lg = logits.cpu().numpy()
    ref = oracle.forward(bits, scales, signs, 0, x)
    assert max_rel_l2(lg.astype(np.float64), ref) <= DECODE_TOL
    for m in range(M):
        assert ids[m] == int(np.argmax(lg[m]))
        assert ref[m, ids[m]] >= ref[m].max() - DECODE_TOL * np.linalg.norm(ref[m])
    # without a caller buffer: same ids
    assert np.array_equal(layer.argmax(torch.from_numpy(x).cuda()).cpu().numpy(), ids)


def test_argmax_ties_take_the_smallest_index(hrb):
    """Rows 100 and 132 (same lane, so the same summation order) are identical and carry the
    largest scores; zero input makes every score exactly 0."""
    w, bits, scales, signs, x = inputs("tiny")
    bits = bits.copy()
    scales = scales.copy()
    scales[:] = np.float16(1e-4).view(np.uint16)
    bits[132] = bits[100]
    scales[100] = scales[132] = np.float16(0.05).view(np.uint16)
    if oracle.forward(bits, scales, signs, 0, x, [100])[0, 0] < 0:
        bits[100] = ~bits[100]
        bits[132] = bits[100]
    layer = make_layer(hrb, bits, scales, signs, 0)
    assert layer.argmax(torch.from_numpy(x).cuda()).cpu().numpy()[0] == 100
    z = torch.zeros((2, w.K), dtype=torch.float32, device="cuda")
    assert layer.argmax(z).cpu().numpy().tolist() == [0, 0]


def test_argmax_consecutive_calls_and_nan(hrb):
    """Several calls in a row on one handle (the pick's ticket is re-armed by each call):
    each id is the argmax of that call's scores, at one token (the pick fused into the
    product's finish) and at two; a NaN input makes every score NaN, and a NaN counts as the
    largest value, so the smallest index wins."""
    N, K = 20000, 5120
    bits = synth.random_bits(21, N, K)
    scales = synth.random_scales(21, N, K, 0.005, 0.03)
    signs = synth.random_signs(21, K)
    layer = make_layer(hrb, bits, scales, signs, 0)
    for M in (1, 2):
        for seed in (1, 2, 3):
            x = torch.from_numpy(synth.random_x(seed, M, K)).cuda()
            lg = torch.empty((M, N), dtype=torch.float32, device="cuda")
            ids = layer.argmax(x, logits=lg).cpu().numpy()
            assert ids.tolist() == np.argmax(lg.cpu().numpy(), axis=1).tolist()
    x = torch.from_numpy(synth.random_x(4, 1, K)).cuda()
    x[0, 77] = float("nan")
    assert layer.argmax(x).cpu().numpy().tolist() == [0]
    torch.cuda.synchronize()
    assert layer.get_error() == 0


def test_lm_head_bf16_narrow_tiles_m64(hrb):
    """The vocabulary matrix at M = 64 on the bf16 path: 1940 tiles of 64 tokens, two CTAs per
    SM over several waves; a seeded sample of rows within 1e-2 and the bf16 diagnostic, and the
    ids picked by the separate argmax kernel equal to the argmax of the scores."""
    bits, scales, signs, seed = _lm_head()
    x = synth.random_x(seed + 1, 64, 5120)
    layer = make_layer(hrb, bits, scales, signs, 0)
    assert layer.plan(64) == (hrb.PATH_PREFILL, 2)
    logits = torch.empty((64, bits.shape[0]), dtype=torch.float32, device="cuda")
    ids = layer.argmax(torch.from_numpy(x).cuda(), logits=logits).cpu().numpy()
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    lg = logits.cpu().numpy()
    rows = synth.sample_rows(seed, bits.shape[0], 512)
    ref = oracle.forward(bits, scales, signs, 0, x, rows)
    assert max_rel_l2(lg[:, rows].astype(np.float64), ref) <= PREFILL_TOL
    ref16 = oracle.forward(bits, scales, signs, 0, x, rows, round_bf16=True)
    assert max_rel_l2(lg[:, rows].astype(np.float64), ref16) <= BF16_DIAG_TOL
    assert np.array_equal(ids, np.argmax(lg, axis=1))


# ------------------------------------------------------------------ embedding (inverse rotation)

@pytest.mark.parametrize("name,ids", [("tiny", [0, 255, 17, 17, 128]), ("ffn_down", [0, 5119, 1234]),
                                      ("attn_kv", list(range(0, 1024, 97)) + [1023])])
def test_embedding_inverse_rotation(hrb, name, ids):
    """out[m] = signs * WHT(dequantized row ids[m]) against the oracle (f64), <= 1e-5."""
    w, bits, scales, signs, _ = inputs(name)
    layer = make_layer(hrb, bits, scales, signs, 0)
    tid = torch.tensor(ids, dtype=torch.int32, device="cuda")
    out = layer.embed(tid)
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    ref = oracle.embed(bits, scales, signs, ids)
    assert max_rel_l2(out.cpu().numpy().astype(np.float64), ref) <= DECODE_TOL


def test_embedding_round_trips_through_the_activation_rotation(hrb):
    """Reading an embedded row back through the activation rotation (signs, then the
    transform) gives the dequantized row again: the fold's two orders are inverses."""
    w, bits, scales, signs, _ = inputs("ffn_gate")
    layer = make_layer(hrb, bits, scales, signs, 0)
    ids = [3, 17000]
    h = layer.embed(torch.tensor(ids, dtype=torch.int32, device="cuda")).cpu().numpy().astype(np.float64)
    for m, t in enumerate(ids):
        back = oracle.rotate(h[m:m + 1], signs, 0)[0]
        z = oracle.dequant_row(bits, scales, t)
        assert np.linalg.norm(back - z) <= 1e-5 * np.linalg.norm(z)


def test_embedding_bad_id_reports_once(hrb):
    w, bits, scales, signs, _ = inputs("tiny")
    layer = make_layer(hrb, bits, scales, signs, 0)
    out = layer.embed(torch.tensor([1, 256, -1, 2], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert layer.get_error() == hrb.BITLIN_EINDEX
    assert layer.get_error() == 0  # reported once, not sticky
    o = out.cpu().numpy()
    assert not o[1].any() and not o[2].any()
    ref = oracle.embed(bits, scales, signs, [1, 2])
    assert max_rel_l2(o[[0, 3]].astype(np.float64), ref) <= DECODE_TOL
    # the handle still works
    x = synth.random_x(5, 1, w.K)
    assert max_rel_l2(run(layer, x), oracle.forward(bits, scales, signs, 0, x)) <= DECODE_TOL


# ------------------------------------------------------------------ errors

def test_empty_and_mismatched_inputs_are_rejected(hrb):
    """M = 0 (an empty batch) and wrong shapes are argument errors, reported before any launch."""
    w, bits, scales, signs, x = inputs("tiny")
    layer = make_layer(hrb, bits, scales, signs, 0)
    empty = torch.empty((0, w.K), dtype=torch.float32, device="cuda")
    with pytest.raises(hrb.BitlinError) as e:
        layer(empty, out=torch.empty((0, w.N), dtype=torch.float32, device="cuda"))
    assert e.value.status == hrb.BITLIN_EINVAL
    with pytest.raises(hrb.BitlinError) as e:
        layer.embed(torch.empty((0,), dtype=torch.int32, device="cuda"), out=torch.empty((0, w.K), device="cuda"))
    assert e.value.status == hrb.BITLIN_EINVAL
    with pytest.raises(ValueError):
        layer(torch.zeros((1, w.K + 32), dtype=torch.float32, device="cuda"))
    # the handle is unaffected
    assert max_rel_l2(run(layer, x), oracle.forward(bits, scales, signs, 0, x)) <= DECODE_TOL


def test_signs_must_be_plus_minus_one(hrb):
    w, bits, scales, signs, x = inputs("tiny")
    bad = signs.copy()
    bad[5] = 0.5
    with pytest.raises(hrb.BitlinError) as e:
        make_layer(hrb, bits, scales, bad, 0)
    assert e.value.status == hrb.BITLIN_EINVAL


def test_bounded_wait_times_out_without_hanging(hrb):
    """A barrier nobody arrives at: the kernel gives up after its budget,
    releases its resources and reports a timeout; the context stays usable."""
    w, bits, scales, signs, x = inputs("tiny")
    layer = make_layer(hrb, bits, scales, signs, 0)
    layer.set_path(hrb.PATH_PREFILL)
    layer.set_wait_budget(200_000_000)  # 0.2 s
    layer.test_stall(True)
    layer(torch.from_numpy(x).cuda())
    assert layer.get_error() == hrb.BITLIN_ETIMEOUT
    with pytest.raises(hrb.BitlinError):
        layer(torch.from_numpy(x).cuda())
    layer.close()
    # The host-buffer entry point reports the timeout of its own call.
    stalled = make_layer(hrb, bits, scales, signs, 0)
    stalled.set_path(hrb.PATH_PREFILL)
    stalled.set_wait_budget(200_000_000)
    stalled.test_stall(True)
    with pytest.raises(hrb.BitlinError) as e:
        stalled.forward_host(x, np.empty((1, w.N), dtype=np.float32))
    assert e.value.status == hrb.BITLIN_ETIMEOUT
    stalled.close()
    fresh = make_layer(hrb, bits, scales, signs, 0)
    y = run(fresh, x)
    assert max_rel_l2(y, oracle.forward(bits, scales, signs, 0, x)) <= DECODE_TOL


# ------------------------------------------------------------------ the stored Q1G128 form

@pytest.mark.parametrize("name", ["attn_kv", "ssm_out"])
def test_q1g128_stored_form_handle(hrb, tmp_path, name):
    """A handle made from the stored Q1G128 tensor (read from a file at a byte offset) gives
    the same y, bit for bit, as one made from separate bits and scales, within 1e-5 of the
    oracle; its embedding rows match the oracle's."""
    w, bits, scales, signs, x = inputs(name, 3)
    blob = synth.q1g128_blob(bits, scales)
    path = tmp_path / "tensor.bin"
    with open(path, "wb") as f:
        f.write(b"\0" * 64)  # something in front of the tensor, as in a checkpoint file
        f.write(blob.astype("<u4").tobytes())
    qd = hrb.load_q1g128(str(path), w.N, w.K, offset=64)
    tg = torch.from_numpy(signs).cuda()
    from_blob = hrb.BitLinear.from_q1g128(qd, w.N, w.K, tg, w.perm)
    del qd  # the handle owns its copy
    plain = make_layer(hrb, bits, scales, signs, w.perm)
    xd = torch.from_numpy(x).cuda()
    y1, y2 = from_blob(xd), plain(xd)
    torch.cuda.synchronize()
    assert from_blob.get_error() == 0
    assert torch.equal(y1, y2)
    ref = oracle.forward(bits, scales, signs, w.perm, x)
    assert max_rel_l2(y1.cpu().numpy().astype(np.float64), ref) <= DECODE_TOL
    ids = [0, w.N // 2, w.N - 1]
    h = from_blob.embed(torch.tensor(ids, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    # (the permutation flag does not apply to embedding rows)
    assert max_rel_l2(h.cpu().numpy().astype(np.float64), oracle.embed(bits, scales, signs, ids)) <= DECODE_TOL
    with pytest.raises(ValueError):
        hrb.BitLinear.from_q1g128(torch.zeros(5, dtype=torch.int32, device="cuda"), w.N, w.K, tg, w.perm)

