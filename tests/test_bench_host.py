"""Host-side reporting logic of bench.py (no GPU): the roofline arithmetic and
the rule that a kernel's DRAM traffic is reported only from an ncu capture of
the source it was taken on."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

PEAKS = {"hbm_gbs": 6785.2, "bf16_tflops": 1904.4, "bf16_tflops_sustained": 1699.9}


def _fake_tree(tmp_path, source_text: bytes, recorded_text: bytes, bytes_per_launch: int):
    """A repository layout with one kernel source and a traffic record taken on recorded_text."""
    csrc = tmp_path / "hadamard_rotated_binary_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "decode.cu").write_bytes(source_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"bitlin_decode_gemv:ffn_gate": {"bytes_per_launch": bytes_per_launch, "source": "decode.cu",
                                           "sha256": hashlib.sha256(recorded_text).hexdigest(), "from": "test"}}
    (prof / "traffic.json").write_text(json.dumps(rec))


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = b"// kernel as profiled\n"
    _fake_tree(tmp_path, src, src, 12_615_509)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("bitlin_decode_gemv", "ffn_gate") == 12_615_509
    # another workload, or a kernel with no record: nothing to report
    assert bench.traffic_record("bitlin_decode_gemv", "lm_head") is None
    assert bench.traffic_record("bitlin_tc_gemm", "prefill") is None


def test_traffic_prefers_the_record_at_the_same_token_count(tmp_path, monkeypatch):
    csrc = tmp_path / "hadamard_rotated_binary_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = b"// kernel as profiled\n"
    (csrc / "decode.cu").write_bytes(src)
    (tmp_path / "profiles").mkdir()
    digest = hashlib.sha256(src).hexdigest()
    rec = {"bitlin_decode_gemv:gate_up:4": {"bytes_per_launch": 25_225_472, "source": "decode.cu", "sha256": digest},
           "bitlin_decode_gemv:gate_up": {"bytes_per_launch": 25_200_000, "source": "decode.cu", "sha256": digest}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("bitlin_decode_gemv", "gate_up", 4) == 25_225_472
    assert bench.traffic_record("bitlin_decode_gemv", "gate_up", 1) == 25_200_000
    assert bench.traffic_record("bitlin_decode_gemv", "gate_up") == 25_200_000


def test_traffic_is_null_once_the_source_changed(tmp_path, monkeypatch):
    _fake_tree(tmp_path, b"// kernel as it is now\n", b"// kernel as profiled\n", 12_615_509)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("bitlin_decode_gemv", "ffn_gate") is None


def test_traffic_is_null_without_a_record(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("bitlin_decode_gemv", "ffn_gate") is None


def test_decode_roofline_is_algorithmic_bytes_over_step_time(monkeypatch):
    monkeypatch.setattr(bench, "traffic_record", lambda kernel, workload, M=None: None)
    w = synth.workload("ffn_gate")
    s_per_step = 5.7e-6
    r = bench.roofline(w, s_per_step, PEAKS, "measured", path=1, kernels=1)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"] == "bitlin_decode_gemv"
    assert r["bytes_per_launch"] == w.algorithmic_bytes() == 12_644_352
    assert r["achieved"] == pytest.approx(12_644_352 / 5.7e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6785.2)
    # the scratch split-K path names its summing kernel too
    assert bench.roofline(w, s_per_step, PEAKS, "measured", path=1, kernels=2)["kernel"] == (
        "bitlin_decode_gemv + bitlin_decode_reduce")


@pytest.mark.parametrize("path,digits", [(2, 1), (3, 3)])
def test_tensor_roofline_counts_digit_columns(monkeypatch, path, digits):
    monkeypatch.setattr(bench, "traffic_record", lambda kernel, workload, M=None: None)
    w = synth.workload("gate_up", 16)
    s_per_step = 38.3e-6
    r = bench.roofline(w, s_per_step, PEAKS, "measured", path=path, kernels=2)
    flops = 2.0 * 16 * digits * w.N * w.K
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["flops_per_launch"] == flops
    assert r["achieved"] == pytest.approx(flops / s_per_step / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1904.4)
