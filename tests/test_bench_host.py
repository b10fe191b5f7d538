"""Host logic of bench.py, no GPU: the per-stage work model the roofline
fractions divide by, the ncu traffic lookup that goes stale with the CUDA
sources, and the peaks file with its fallback."""
import json
import os

import pytest

import bench
from workloads import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_stage_work_counts_each_contraction_once():
    wl = synth.workload("train")
    T, d, E, R, f = wl.T, wl.d, wl.E, wl.R, wl.f
    N = T * R
    w = bench.stage_work(wl)
    assert w["gateup"]["kind"] == "tensor" and w["gateup"]["flops"] == 4.0 * N * d * f  # a and b
    assert w["down"]["flops"] == 2.0 * N * d * f
    gemms = ("gateup", "down", "bwd_dh", "bwd_dx", "bwd_wg2", "bwd_wg13")
    # forward 6 N d f, backward twice that: dgrad (DH, DX) and wgrad (WG2, WG13)
    assert sum(w[k]["flops"] for k in gemms) == 18.0 * N * d * f
    assert (sum(w[k]["flops"] for k in ("bwd_dh", "bwd_dx"))
            == sum(w[k]["flops"] for k in ("bwd_wg2", "bwd_wg13")))
    # dispatch: read x, write x_perm, 12 B of maps per row; combine: gather + write y
    assert w["dispatch"] == {"kind": "hbm", "flops": 0.0, "bytes": 2.0 * T * d + 2.0 * N * d + 12.0 * N}
    assert w["combine"]["bytes"] == 2.0 * N * d + 8.0 * N + 2.0 * T * d
    # gate-up reads x_perm and W1, W3 once, writes h and (training) the saved a, b
    assert w["gateup"]["bytes"] == 2.0 * N * d + 4.0 * E * f * d + 2.0 * N * f + 4.0 * N * f
    # WG13 reads [da | db] and x_perm once, writes dW1 and dW3 (fp32) once
    assert w["bwd_wg13"]["bytes"] == N * 2 * f * 2 + N * d * 2 + 2 * E * f * d * 4
    assert "shared_fwd" not in w


def test_stage_work_reads_only_the_weights_of_experts_with_rows():
    wl = synth.workload("mid")
    N, d, f = wl.T * wl.R, wl.d, wl.f
    full, part = bench.stage_work(wl), bench.stage_work(wl, active_experts=wl.E - 8)
    assert full["gateup"]["bytes"] - part["gateup"]["bytes"] == 4.0 * 8 * f * d
    assert full["down"]["bytes"] - part["down"]["bytes"] == 2.0 * 8 * f * d
    assert "save" not in wl.name and full["gateup"]["bytes"] == 2.0 * N * d + 4.0 * wl.E * f * d + 2.0 * N * f


def test_stage_work_fp8_dispatch_bytes():
    q8 = lambda N, d: N * d + 4.0 * N * d / 128           # E4M3 codes + one fp32 scale per 128
    wl = synth.workload("large")                           # layer: codes out, back in, bf16 rows out
    T, d, N = wl.T, wl.d, wl.T * wl.R
    assert bench.stage_work(wl, fp8=True)["dispatch"]["bytes"] == (2.0 * T * d + 2 * q8(N, d)
                                                                   + 2.0 * N * d + 12.0 * N)
    wl = synth.workload("dispatch", T=1024)                # identity experts: codes out only
    T, d, N = wl.T, wl.d, wl.T * wl.R
    assert wl.f == 0
    assert bench.stage_work(wl, fp8=True)["dispatch"]["bytes"] == 2.0 * T * d + q8(N, d) + 12.0 * N


def test_stage_work_shared_expert_is_reported_beside():
    wl = synth.workload("mid")
    w = bench.stage_work(wl, shared_fs=512)
    assert w["shared_fwd"] == {"kind": "side", "flops": 6.0 * wl.T * wl.d * 512, "bytes": 0.0}
    assert w["shared_bwd"]["flops"] == 12.0 * wl.T * wl.d * 512


PK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def test_roofline_of_the_large_forward_is_the_weight_stream():
    """large: 22.5 GB of W1/W3 at 6.8 TB/s outlast 3.85 TFLOP at 1.9 PFLOP/s."""
    wl = synth.workload("large")
    w = bench.stage_work(wl)["gateup"]
    t_mem, t_tc = w["bytes"] / 6.8e12, w["flops"] / 1.9e15
    assert t_mem > t_tc
    st = bench.stage_roofline(w, 4.0, 1900.0, PK)
    assert st["bound"] == "hbm"
    assert st["frac"] == pytest.approx(t_mem / 4e-3, abs=1e-4)
    assert st["frac_burst"] == pytest.approx(w["flops"] / 4e-3 / 1.9e15, abs=1e-4)
    roof = bench.dominant_roofline({"gateup": st}, {"gateup": w}, "gateup", 1900.0, "burst", PK,
                                   "measured", None)
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] == 6800.0
    assert roof["achieved"] == pytest.approx(w["bytes"] / 4e-3 / 1e9, rel=1e-4)


def test_roofline_of_the_training_weight_gradient_is_the_tensor_pipe():
    wl = synth.workload("train")
    w = bench.stage_work(wl)["bwd_wg13"]
    assert w["flops"] / 1.9e15 > w["bytes"] / 6.8e12
    st = bench.stage_roofline(w, 2.5, 1900.0, PK)
    assert st["bound"] == "tensor"
    assert st["frac"] == st["frac_burst"] == pytest.approx(w["flops"] / 2.5e-3 / 1.9e15, abs=1e-4)
    assert st["frac_sustained"] == pytest.approx(w["flops"] / 2.5e-3 / 1.7e15, abs=1e-4)
    roof = bench.dominant_roofline({"bwd_wg13": st}, {"bwd_wg13": w}, "bwd_wg13", 1900.0, "burst",
                                   PK, "measured", 123)
    assert roof["bound"] == "tensor" and roof["frac_burst"] == st["frac_burst"]
    assert roof["traffic"] == 123 and roof["algorithmic_bytes"] == w["bytes"]


def test_gate_on_the_tensor_cores_executes_three_products():
    wl = synth.workload("train")
    w = bench.stage_work(wl)["gate"]
    assert w["kind"] == "tensor3"
    st = bench.stage_roofline(w, 0.1, 1900.0, PK)
    assert st["tensor_tflops"] == pytest.approx(3 * st["tflops"], rel=1e-3)


def test_tensor_peak_follows_the_clock_regime():
    assert bench.tensor_peak(PK, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}) == (1900.0, "burst")
    assert bench.tensor_peak(PK, {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0}) == (1900.0, "burst")
    assert bench.tensor_peak(PK, {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0}) == (1700.0, "sustained")
    assert bench.tensor_peak(PK, {"sm_mhz": None, "sm_max_mhz": None}) == (1900.0, "burst")


def test_clock_samples_median_and_reasons():
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2000, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage"]
    c = bench.parse_clock_samples(rows)
    assert c["sm_mhz"] == 2000.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_oracle_full_step_estimate_separates_fixed_and_per_token_cost():
    wl = synth.workload("train")
    fixed, per_tok = 4.0, 0.03
    samples = [(n, fixed + per_tok * n, wl.E) for n in (64, 128, 64, 128)]
    est = bench.full_step_estimate(wl, samples)
    assert est["per_token_s"] == pytest.approx(per_tok)
    assert est["fixed_s"] == pytest.approx(fixed)
    assert est["full_step_s"] == pytest.approx(fixed + per_tok * wl.T)
    line = bench.cpu_baseline_line(wl, est, 16, "test")
    assert line["value"] == pytest.approx(wl.T / (fixed + per_tok * wl.T), rel=1e-3)
    assert line["cores"] == 16 and line["kind"] == "oracle" and str(wl.T) in line["sample"]
    one = bench.full_step_estimate(wl, [(64, 2.0, 100)])
    assert one["full_step_s"] == pytest.approx(2.0 / 64 * wl.T)


def test_extra_workloads_only_with_the_default_headline():
    assert bench.want_extras(bench.parse([]))
    assert not bench.want_extras(bench.parse(["--workload", "large"]))
    assert not bench.want_extras(bench.parse(["--tokens", "4096"]))
    assert not bench.want_extras(bench.parse(["--extra-workloads", "off"]))
    assert bench.want_extras(bench.parse(["--workload", "mid", "--extra-workloads", "on"]))
    names = [(n, mx) for n, _, _, mx in bench.EXTRA_WORKLOADS]
    assert names == [("large", False), ("large", True), ("large_hot", False), ("mid", False),
                     ("dispatch", False), ("dispatch", False)]
    assert [o.get("T") for n, o, fl, _ in bench.EXTRA_WORKLOADS if n == "dispatch"] == [8192, 65536]
    assert all(fl for n, _, fl, _ in bench.EXTRA_WORKLOADS if n == "dispatch")
    assert not bench.want_extras(bench.parse(["--mx"]))


def test_microscaled_fp8_gemm_stages_count_bytes_and_the_fp8_peak():
    wl = synth.workload("large")
    T, d, E, R, f = wl.T, wl.d, wl.E, wl.R, wl.f
    N = T * R
    w = bench.stage_work(wl, mx=True)
    q = 1 + 1 / 32
    assert w["gateup"]["kind"] == "tensor_fp8" and w["gateup"]["flops"] == 4.0 * N * d * f
    # codes and scales of x, W1, W3 and h: half the bf16 weight bytes and a little
    assert w["gateup"]["bytes"] == q * N * d + 2 * q * E * f * d + q * N * f
    assert w["down"]["bytes"] == q * N * f + q * E * d * f + 2.0 * N * d
    st = bench.stage_roofline(w["gateup"], 2.0, 1900.0, PK)
    assert st["frac_burst"] == pytest.approx(w["gateup"]["flops"] / 2e-3 / 3.8e15, abs=1e-4)
    assert st["bound"] == "hbm"           # 12.3 GB at 6.8 TB/s outlast 3.85 TFLOP at 3.8 PF
    roof = bench.dominant_roofline({"gateup": st}, w, "gateup", 1900.0, "burst", PK, "m", None)
    assert roof["bound"] == "hbm"


def test_profiled_traffic_goes_stale_with_the_sources(monkeypatch, tmp_path):
    csrc = tmp_path / "expert_moe_route_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (csrc / "other.cu").write_text("other v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    table = {"workloads": {"train": {"bwd_wg13": {
        "bytes_per_launch": 123, "sources": ["k.cu"],
        "sources_sha256": bench.kernel_sources_digest(["k.cu"])}}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(table))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(path))
    assert bench.profiled_traffic("train", "bwd_wg13") == 123
    assert bench.profiled_traffic("train", "gateup") is None
    assert bench.profiled_traffic("large", "bwd_wg13") is None
    (csrc / "other.cu").write_text("other v2")            # another kernel's source changed
    assert bench.profiled_traffic("train", "bwd_wg13") == 123
    (csrc / "k.cu").write_text("kernel v2")               # this kernel's source changed
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
    assert bench.kernel_sources_digest(["a.cu"]) == d1 != d2   # only the named files count


def test_traffic_keys_name_a_non_default_token_count():
    assert bench.traffic_key(synth.workload("train")) == "train"
    assert bench.traffic_key(synth.workload("dispatch", T=8192)) == "dispatch"
    assert bench.traffic_key(synth.workload("dispatch", T=65536)) == "dispatch@T=65536"
    assert bench.traffic_key(synth.workload("large"), mx=True) == "large+mx"


def test_committed_traffic_entries_against_their_algorithmic_bytes():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        table = json.load(fh)
    assert table["workloads"], "no entries"
    for key, stages in table["workloads"].items():
        base, mx = (key[:-3], True) if key.endswith("+mx") else (key, False)
        name, _, t = base.partition("@T=")
        wl = synth.workload(name, **({"T": int(t)} if t else {}))
        work = bench.stage_work(wl, mx=mx)
        for stage, e in stages.items():
            # the algorithmic bytes of the entry are the work model's
            assert e["algorithmic_bytes_per_launch"] == work[stage]["bytes"], (key, stage)
            # the measured DRAM bytes are that, give or take what stays in L2;
            # more than 1.1x is waste, and the entry must say where it comes from
            ratio = e["bytes_per_launch"] / e["algorithmic_bytes_per_launch"]
            assert 0.85 <= ratio <= 1.1 or (ratio <= 1.25 and e.get("waste")), (key, stage)
            assert os.path.exists(os.path.join(ROOT, e["profile"]))
            assert e["sources"] and len(e["sources_sha256"]) == 64


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
