"""Host-side logic of bench.py (no GPU): byte and roofline accounting, recorded traffic."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_alu_peak_is_32_updates_per_sm_clock():
    # 152 SMs at 2070 MHz, 32 updates per SM clock
    assert bench.alu_peak_updates(152, 2070.0) == pytest.approx(152 * 2070e6 * 32)
    # the exponential unit and the FP32 lanes give the same cap for this update
    assert bench.EX2_PER_CLK_SM == bench.FP32_LANES_PER_CLK_SM / bench.FP32_OPS_PER_UPDATE


def test_m1_bytes_130m_layer():
    # x, delta, z in and y out (bf16) per (b, d, t); B and C per (b, t, n); A, D, bias
    b = bench.m1_bytes(8, 1536, 16, 2048)
    assert b == 8 * 1536 * 2048 * 8 + 2 * 8 * 16 * 2048 * 2 + 1536 * 16 * 4 + 1536 * 8


def test_step_bytes_780m():
    b = bench.step_bytes(64, 48, 64, 128, 1)
    assert b == 2 * 64 * 48 * 64 * 128 * 4 + 64 * 48 * 64 * 2 * 3 + 64 * 48 * 2 + 2 * 64 * 128 * 2


def test_recorded_traffic_needs_matching_digest(tmp_path, monkeypatch):
    digest = bench._source_digest("m1_scan_tmem")
    assert len(digest) == 16
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(f"# header\nm1_scan_tmem 123456 {digest}\n"
                                      "m1_scan_tmem 999 0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the digest is taken from the sources under ROOT: point it back at the repo for them
    monkeypatch.setattr(bench, "_source_digest", lambda kernel="m1_scan_tmem": digest)
    assert bench.recorded_traffic("m1_scan_tmem") == 123456.0
    (prof / "traffic.txt").write_text("m1_scan_tmem 999 0000000000000000\n")
    assert bench.recorded_traffic("m1_scan_tmem") is None


def test_bwd_bytes_130m_layer():
    # 4 bf16 reads and 3 float32 writes per (b, d, t); B, C bf16 in and dB, dC float32 out
    b = bench.bwd_bytes(8, 1536, 16, 2048)
    assert b == 8 * 1536 * 2048 * 20 + 8 * 16 * 2048 * 12 + 1536 * 16 * 8 + 1536 * 16


def test_ssd_bwd_macs_130m():
    # per 64-step chunk: 4 Q^2 N + 3 Q^2 P + 6 Q N P with Q 64, N 128, P 64; 4 x 24 x 64 chunks
    per_chunk = 4 * 64 * 64 * 128 + 3 * 64 * 64 * 64 + 6 * 64 * 128 * 64
    assert per_chunk == 6029312
    assert bench.ssd_bwd_macs(4, 4096, 24, 64, 128) == 4 * 24 * 64 * per_chunk
    assert bench.ssd_bwd_macs(1, 65, 1, 64, 128) == 2 * per_chunk  # a ragged chunk counts whole
    assert bench.fp32_fma_peak(152, 2070.0) == pytest.approx(152 * 2070e6 * 128)


def test_percentile_interpolates_order_statistics():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 0) == 1.0
    assert bench.percentile(xs, 50) == 3.0
    assert bench.percentile(xs, 100) == 5.0
    assert bench.percentile(xs, 95) == pytest.approx(4.8)
    assert bench.percentile([], 95) is None


def test_path_rooflines_carry_every_measured_path():
    paths = {"ssd_130m_chunk64": {"roofline_bound": "hbm", "roofline_frac": 0.2, "ms": 0.08},
             "decode_780m": {"hbm_frac": 0.75, "us_per_step": 40.0},
             "m1_790m_long": {"4096": {"hbm_frac": 0.3, "ms": 0.05, "alu_frac": 0.5}},
             "ssd_130m_bwd": {"ms": 2.8, "fma_frac": 0.33, "multiply_adds": 37e9}}
    r = bench.path_rooflines(paths)
    assert r["ssd_130m_bwd"] == {"bound": "alu", "frac": 0.33, "ms": 2.8}
    assert r["ssd_130m_chunk64"] == {"bound": "hbm", "frac": 0.2, "ms": 0.08}
    assert r["decode_780m"]["frac"] == 0.75 and r["decode_780m"]["bound"] == "hbm"
    assert r["m1_790m_L4096"]["frac"] == 0.3 and r["m1_790m_L4096"]["alu_frac"] == 0.5
    assert bench.path_rooflines({}) == {}
    assert bench.path_rooflines({"error": "RuntimeError: x"}) == {}


def test_sources_digest_is_stable():
    d = bench.sources_digest()
    assert len(d) == 16 and d == bench.sources_digest()
