"""Host logic of bench.py, no GPU: the per-stage work model the roofline
fractions divide by, the ncu traffic lookup that goes stale with the CUDA
sources, and the peaks file with its fallback."""
import json
import os

import pytest

import bench
from expert_moe_route_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_stage_work_counts_each_contraction_once():
    wl = synth.workload("train")
    T, d, R, f = wl.T, wl.d, wl.R, wl.f
    N = T * R
    w = bench.stage_work(wl)
    assert w["gateup"] == ("tflop", 4.0 * N * d * f)     # a and b
    assert w["down"] == ("tflop", 2.0 * N * d * f)
    gemms = ("gateup", "down", "bwd_dh", "bwd_dx", "bwd_wg2", "bwd_wg13")
    # forward 6 N d f, backward twice that: dgrad (DH, DX) and wgrad (WG2, WG13)
    assert sum(w[k][1] for k in gemms) == 18.0 * N * d * f
    assert sum(w[k][1] for k in ("bwd_dh", "bwd_dx")) == sum(w[k][1] for k in ("bwd_wg2", "bwd_wg13"))
    # dispatch: read x, write x_perm, 12 B of maps per row; combine: gather + write y
    assert w["dispatch"] == ("gb", 2.0 * T * d + 2.0 * N * d + 12.0 * N)
    assert w["combine"] == ("gb", 2.0 * N * d + 8.0 * N + 2.0 * T * d)
    assert "shared_fwd" not in w


def test_stage_work_fp8_dispatch_bytes():
    q8 = lambda N, d: N * d + 4.0 * N * d / 128           # E4M3 codes + one fp32 scale per 128
    wl = synth.workload("large")                           # layer: codes out, back in, bf16 rows out
    T, d, N = wl.T, wl.d, wl.T * wl.R
    assert bench.stage_work(wl, fp8=True)["dispatch"][1] == (2.0 * T * d + 2 * q8(N, d)
                                                             + 2.0 * N * d + 12.0 * N)
    wl = synth.workload("dispatch", T=1024)                # identity experts: codes out only
    T, d, N = wl.T, wl.d, wl.T * wl.R
    assert wl.f == 0
    assert bench.stage_work(wl, fp8=True)["dispatch"][1] == 2.0 * T * d + q8(N, d) + 12.0 * N


def test_stage_work_shared_expert_is_reported_beside():
    wl = synth.workload("mid")
    w = bench.stage_work(wl, shared_fs=512)
    assert w["shared_fwd"] == ("side", 6.0 * wl.T * wl.d * 512)
    assert w["shared_bwd"] == ("side", 12.0 * wl.T * wl.d * 512)


def test_profiled_traffic_goes_stale_with_the_sources(monkeypatch, tmp_path):
    table = {"kernel_sources_sha256": "abc",
             "workloads": {"train": {"bwd_wg13": {"bytes_per_launch": 123}}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(table))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(path))
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "abc")
    assert bench.profiled_traffic("train", "bwd_wg13") == 123
    assert bench.profiled_traffic("train", "gateup") is None
    assert bench.profiled_traffic("large", "bwd_wg13") is None
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "def")   # a source changed
    assert bench.profiled_traffic("train", "bwd_wg13") is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.json"))
    assert bench.profiled_traffic("train", "bwd_wg13") is None


def test_kernel_sources_digest_covers_every_source_file(monkeypatch, tmp_path):
    csrc = tmp_path / "expert_moe_route_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("one")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d1 = bench.kernel_sources_digest()
    (csrc / "b.cuh").write_text("two")
    d2 = bench.kernel_sources_digest()
    (csrc / "b.cuh").write_text("two ")
    assert len({d1, d2, bench.kernel_sources_digest()}) == 3


def test_committed_traffic_entries_against_their_algorithmic_bytes():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        table = json.load(fh)
    e = table["workloads"]["train"]["bwd_wg13"]
    wl = synth.workload("train")
    N, d, f, E = wl.T * wl.R, wl.d, wl.f, wl.E
    # WG13 reads [da | db] (N x 2f bf16) and x_perm (N x d bf16) once and writes
    # dW1 and dW3 (2 E f d fp32) once
    assert e["algorithmic_bytes_per_launch"] == N * 2 * f * 2 + N * d * 2 + 2 * E * f * d * 4
    # the measured DRAM bytes are that, give or take what stays in L2
    assert 0.9 <= e["bytes_per_launch"] / e["algorithmic_bytes_per_launch"] <= 1.1
    assert os.path.exists(os.path.join(ROOT, e["profile"]))


def test_peaks_file_or_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "missing.json"))
    pk, source = bench.load_peaks()
    assert source == "fallback" and pk == dict(bench.FALLBACK_PEAKS)
    path = tmp_path / "peaks.json"
    path.write_text(json.dumps({"hbm_gbs": 6778.0, "bf16_tflops": 1934.0}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(path))
    pk, source = bench.load_peaks()
    assert source == "measured" and pk["hbm_gbs"] == pytest.approx(6778.0)


def test_alu_peak_uses_the_sampled_clock():
    assert bench.alu_peak_tflops(2070.0) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    assert bench.alu_peak_tflops(None) == bench.alu_peak_tflops(2070.0)
