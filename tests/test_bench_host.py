"""Host-side arithmetic of bench.py: algorithmic bytes, the integer-pipe bound,
host information and the kernel-source hash.  No GPU needed."""
import os

import pytest

import bench


def test_layer_bytes_match_the_shapes():
    # 2-bit: 3 matrices of 17408 x 5120 codes at 4 per byte + fp16 per 128-block scales
    assert bench.layer_bytes(5120, 17408, 0) == 3 * (17408 * 5120 // 4 + 2 * 17408 * 40)
    assert bench.layer_bytes(5120, 17408, 0) == 71_024_640
    # 1-bit: 8 per byte, the same scales
    assert bench.layer_bytes(5120, 17408, 1) == 37_601_280
    assert 64 * bench.layer_bytes(5120, 17408, 0) == 4_545_576_960
    assert 64 * bench.layer_bytes(5120, 17408, 1) == 2_406_481_920


def test_gemv_shapes_bytes():
    for name, n, k in bench.GEMV_SHAPES:
        assert k % 128 == 0 and n > 0, name
    # the tiny config: 512 x 256 codes at 4 per byte + scales
    assert 512 * 256 // 4 + 2 * 512 * 2 == 34_816


def test_integer_ops_per_weight():
    # 2-bit: 7 decode ops per 16 weights, one dp4a per 4 weights and row
    assert bench.int_ops_per_weight(0, 1) == pytest.approx(11 / 16)
    assert bench.int_ops_per_weight(0, 4) == pytest.approx(23 / 16)
    # 1-bit: a shift and a mask per 4 weights, one dp4a per 4 weights and row
    assert bench.int_ops_per_weight(1, 1) == pytest.approx(3 / 4)
    assert bench.int_ops_per_weight(1, 4) == pytest.approx(6 / 4)


def test_alu_bound_counts_passes_of_four_rows():
    w = 3 * 5120 * 17408
    one = bench.alu_bound_us(0, 1, w, 2070.0)
    # 267,386,880 weights x 11/16 ops / (152 SMs x 64 lanes x 2.07e9 /s)
    assert one == pytest.approx(w * 11 / 16 / (152 * 64 * 2.07e9) * 1e6)
    assert 9.0 < one < 9.3
    # 8 rows = two passes of 4; 9 rows = two passes of 4 and one of 1
    assert bench.alu_bound_us(0, 8, w, 2070.0) == pytest.approx(2 * bench.alu_bound_us(0, 4, w, 2070.0))
    assert bench.alu_bound_us(0, 9, w, 2070.0) == pytest.approx(
        2 * bench.alu_bound_us(0, 4, w, 2070.0) + one)
    # halving the clock doubles the bound
    assert bench.alu_bound_us(1, 1, w, 1035.0) == pytest.approx(2 * bench.alu_bound_us(1, 1, w, 2070.0))


def test_host_info():
    h = bench.host_info()
    assert h["nproc"] == os.cpu_count()
    assert isinstance(h["cpu_model"], str) and h["cpu_model"]


def test_source_hash_leaves_out_host_only_sources(monkeypatch, tmp_path):
    csrc = tmp_path / "ternary_weight_dp4a_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash()
    (csrc / bench.HOST_ONLY_SOURCES[0]).write_text("host policy")
    assert bench.source_hash() == h0                 # host-only file: same hash
    (csrc / "k.cu").write_text("kernel, changed")
    assert bench.source_hash() != h0                 # kernel file: new hash


def test_reference_arm_runs_the_requested_steps(monkeypatch):
    """The reference arm times exactly --warmup untimed and --steps timed
    oracle steps: whole layer steps when they fit the budget, else the same
    fraction of every matrix's rows (bytes counted from the rows read)."""
    monkeypatch.setattr(bench, "HIDDEN", 256)
    monkeypatch.setattr(bench, "INTER", 512)
    full = bench.reference_arm(2, 1, budget_s=30.0)
    assert full["sample"].startswith("2 timed steps after 1 untimed: full FFN layer steps")
    assert full["bytes_per_step"] == bench.layer_bytes(256, 512, 0)
    assert full["kind"] == "oracle" and full["value"] > 0 and full["cores"] >= 1
    part = bench.reference_arm(50, 3, budget_s=1e-6)
    assert part["sample"].startswith("50 timed steps after 3 untimed: 1 of 512 gate/up rows and 1 of 256 down rows")
    assert part["bytes_per_step"] == 2 * (256 // 4 + 2 * 256 // 128) + (512 // 4 + 2 * 512 // 128)
    assert part["value"] > 0
