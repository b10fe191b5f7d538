"""Benchmark of the MoE layer hot path on GB300 (one JSON line on rank 0).

Headline workload: the MoE layer training step (forward + backward) with
T=16384 tokens, d=4096, E=128 experts, top-8 routing, SwiGLU width f=1536 --
one pass of every step of the path (route, dispatch, grouped SwiGLU FFN,
combine, and their backward).  Other workloads: --workload large | large_hot |
mid | tiny (forward only) and dispatch (dispatch + combine with identity
experts, --tokens T).  With the default headline the same run also times, each
on its own clock and with its own stages and roofline, the forward of large,
large_hot and mid and dispatch + combine at T=8192 and T=65536 (L2 flushed
between steps), under the "workloads" key.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

value = tokens per second of the whole job (all ranks); each rank runs an
independent replica of the workload (the path has no cross-GPU exchange), so
scaling is weak.  The timed region is K back-to-back steps between CUDA events
on the launching stream, after W warm-up steps, bracketed by a barrier and a
device synchronisation; the max over ranks is reported.  Each layer step
streams more than L2 (5 GB of expert weights for the headline), so no flush is
needed between its steps.

Roofline: every stage is timed by CUDA events the library records around it.
A stage's roofline time is max(FLOPs / tensor peak, bytes / HBM bandwidth),
with the FLOPs of real rows only and the bytes it must move to or from HBM at
least once; its fraction is that time over the measured one.  The tensor peak
is the measured burst bf16 rate when the SM clock stayed within 5% of its
maximum during the timed region, else the sustained (power-capped) rate; both
fractions are printed.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s on 1 GB300; grouped-GEMM % BF16 TC peak; dispatch/combine GB/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
BURST_CLOCK_FRACTION = 0.95

# the other workloads the default run times after the headline:
# (name, overrides, flush L2 between steps, expert FFN in microscaled fp8)
EXTRA_WORKLOADS = (("large", {}, False, False), ("large", {}, False, True),
                   ("large_hot", {}, False, False), ("mid", {}, False, False),
                   ("dispatch", {"T": 8192}, True, False), ("dispatch", {"T": 65536}, True, False))
FP8_PER_BF16 = 2.0   # dense fp8 tensor rate per bf16 rate (nominal 4.5 / 2.25 PFLOP/s)

# two token counts of the oracle sample per workload (full-step estimate: a
# straight line through the two timings).  The smaller one already routes to
# (nearly) every expert; the larger one adds enough rows that the per-token
# cost stands well above the timing noise of the per-expert part.
CPU_SAMPLE_TOKENS = {"train": (256, 2048), "mid": (512, 2048), "large": (512, 1024),
                     "large_hot": (512, 1024), "tiny": (128, 256), "dispatch": (2048, 8192),
                     "dispatch_zipf": (2048, 8192)}


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="train",
                   choices=["train", "large", "large_hot", "mid", "tiny", "dispatch",
                            "dispatch_zipf"])
    p.add_argument("--tokens", type=int, default=None, help="override T")
    p.add_argument("--experts", type=int, default=None, help="override E (smaller profiling cases)")
    p.add_argument("--cpu-tokens", type=int, nargs=2, default=None, metavar=("N1", "N2"),
                   help="token counts of the two CPU oracle samples (default per workload)")
    p.add_argument("--fp8", action="store_true",
                   help="block-scaled fp8 dispatch (E4M3 + per-128 scales), bf16 combine: "
                        "dispatch workloads dequantise in identity experts; layer workloads "
                        "pass MOE_FP8_DISPATCH (the GEMMs read the dequantised rows)")
    p.add_argument("--mx", action="store_true",
                   help="forward-only layer workloads: the expert FFN on the fp8 tensor cores in "
                        "microscaled fp8 (MOE_FP8_MX; weights quantised once before timing)")
    p.add_argument("--no-prepack", action="store_true",
                   help="forward-only workloads: stream the plain weight layout instead of the "
                        "tiles moe_prepack_weights writes once before timing")
    p.add_argument("--single-cta", action="store_true",
                   help="expert GEMMs on single-CTA 128-row tiles instead of 256-row tiles on "
                        "CTA pairs")
    p.add_argument("--shared-expert", type=int, default=0, metavar="FS",
                   help="layer workloads: add one shared expert of hidden size FS (0: none), run "
                        "on the library's side stream beside route, dispatch and the routed FFN")
    p.add_argument("--shared-serial", action="store_true",
                   help="run the shared expert on the caller's stream after the routed path "
                        "(MOE_SHARED_SERIAL), for comparison")
    p.add_argument("--flush-l2", action="store_true",
                   help="write a 512 MB buffer (4x L2) between timed steps, so small workloads "
                        "read HBM; each step is then timed by its own events, the flush outside them")
    p.add_argument("--extra-workloads", default="auto", choices=["auto", "on", "off"],
                   help="also time large, large_hot, mid and dispatch + combine (auto: only "
                        "with the default headline workload)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args(argv)


def load_peaks():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(pk, clk):
    """(peak TFLOP/s, regime): the burst bf16 peak when the median SM clock under
    load stayed within 5% of its maximum, else the sustained (power-capped) one."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    burst = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sust = pk.get("bf16_tflops_sustained", burst)
    if sm and smax and sm < BURST_CLOCK_FRACTION * smax:
        return sust, "sustained"
    return burst, "burst"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            out = parse_clock_samples(fh)
        os.unlink(self.path)
        return out


def parse_clock_samples(lines):
    """Median SM clock, max clock and the throttle reasons seen in nvidia-smi CSV rows."""
    sms, maxs, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [c.strip() for c in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sms.append(float(f[1]))
            maxs.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(sms) if sms else None,
            "sm_max_mhz": max(maxs) if maxs else None, "reasons": sorted(reasons),
            "samples": len(sms)}


# ---------------------------------------------------------------- work model
def stage_work(wl, fp8=False, shared_fs=0, active_experts=None, mx=False):
    """Algorithmic work of one launch of each traced stage.

    Returns {stage: {"kind": K, "flops": F, "bytes": B}}.  F counts the
    FLOPs of real rows only (no padding); B the bytes the stage must move to or
    from HBM at least once (inputs read, outputs written).  Kinds: "tensor" (a
    grouped GEMM on the tensor cores), "tensor3" (the gate projection x W_g on
    the tensor cores as three bf16 products, W_g split into hi + mid + lo, so
    the pipe executes 3 F), "alu" (the FP32 FMA gate, d % 64 != 0), "hbm"
    (data movement only), "side" (the shared expert's GEMMs, overlapping
    other stages) and "tensor_fp8" (a grouped GEMM on microscaled fp8
    operands, ``mx``: one byte per element plus a scale byte per 32).
    ``active_experts``: experts with at least one row, whose weights the
    forward and data-gradient GEMMs read (default: all E).
    """
    T, d, E, R, f = wl.T, wl.d, wl.E, wl.R, wl.f
    Ea = E if active_experts is None else active_experts
    N = T * R
    q8 = N * d + 4.0 * N * d / 128          # fp8 codes and their scales
    # fp8 in a layer: the codes and scales are written, read back and the bf16
    # rows the GEMMs read are written, all inside the dispatch stage
    disp = (2.0 * N * d if not fp8 else q8 if not f else 2.0 * q8 + 2.0 * N * d)

    def k(kind, flops=0.0, nbytes=0.0):
        return {"kind": kind, "flops": float(flops), "bytes": float(nbytes)}

    w = {
        "gate": k("tensor3" if d % 64 == 0 else "alu", 2.0 * T * d * E,
                  2.0 * T * d + 4.0 * d * E + 4.0 * T * E),
        "topk": k("hbm", 0, 4.0 * T * E + 8.0 * N),
        "dispatch": k("hbm", 0, 2.0 * T * d + disp + 4.0 * N * 3),
        "combine": k("hbm", 0, 2.0 * N * d + 8.0 * N + 2.0 * T * d),
    }
    if f:
        save_ab = 4.0 * N * f if wl.train else 0.0    # the saved a and b (training)
        w.update({
            "gateup": k("tensor", 4.0 * N * d * f, 2.0 * N * d + 4.0 * Ea * f * d + 2.0 * N * f
                        + save_ab),
            "down": k("tensor", 2.0 * N * d * f, 2.0 * N * f + 2.0 * Ea * d * f + 2.0 * N * d),
            "bwd_route": k("hbm", 0, 2.0 * T * d + 2.0 * N * d + 2.0 * N * d + 12.0 * N),
            # dh = do W2: reads do, W2, the saved a and b; writes [da | db]
            "bwd_dh": k("tensor", 2.0 * N * d * f, 2.0 * N * d + 2.0 * Ea * d * f + 4.0 * N * f
                        + 4.0 * N * f),
            "bwd_dx": k("tensor", 4.0 * N * d * f, 4.0 * N * f + 4.0 * Ea * f * d + 2.0 * N * d),
            # weight gradients: every expert's fp32 gradient is written
            "bwd_wg2": k("tensor", 2.0 * N * d * f, 2.0 * N * d + 2.0 * N * f + 4.0 * E * d * f),
            "bwd_wg13": k("tensor", 4.0 * N * d * f, 4.0 * N * f + 2.0 * N * d + 8.0 * E * f * d),
            # x once (its rows are gathered through row_slot, the R reads of a
            # row mostly from L2), row_slot and dsel per row, dW_g written
            "bwd_dwg": k("hbm", 0, 2.0 * T * d + 8.0 * N + 4.0 * d * E),
            "bwd_dxc": k("hbm", 0, 2.0 * N * d + 2.0 * T * d + 8.0 * E * d),
        })
    if f and mx:
        q = 1.0 + 1.0 / 32                    # a code byte per element, a scale byte per 32
        w.update({
            "dispatch": k("hbm", 0, 2.0 * T * d + q * N * d + 12.0 * N),
            "gateup": k("tensor_fp8", 4.0 * N * d * f, q * N * d + 2.0 * q * Ea * f * d
                        + q * N * f),
            "down": k("tensor_fp8", 2.0 * N * d * f, q * N * f + q * Ea * d * f + 2.0 * N * d),
        })
    if f and shared_fs:
        # the shared expert on the side stream: reported, but its time overlaps
        # other stages, so it stays out of the GEMM summary and the dominant kernel
        w.update({"shared_fwd": k("side", 6.0 * T * d * shared_fs),
                  "shared_bwd": k("side", 12.0 * T * d * shared_fs)})
    return w


def stage_roofline(work, ms, tc_peak, pk, sm_mhz=None):
    """One stage's figures: achieved rates, its roofline bound and fractions.

    tc_peak: the tensor peak the fractions divide by (TFLOP/s); the burst and
    sustained fractions are printed beside it for tensor stages.
    """
    kind, fl, nb = work["kind"], work["flops"], work["bytes"]
    s = ms / 1e3
    out = {"ms": round(ms, 4)}
    hbm = pk["hbm_gbs"] * 1e9
    if kind in ("tensor", "tensor3", "side", "tensor_fp8"):
        ex = 3.0 * fl if kind == "tensor3" else fl     # FLOPs the tensor pipe executes
        rate = FP8_PER_BF16 if kind == "tensor_fp8" else 1.0
        tc_peak = tc_peak * rate
        out["tflops"] = round(fl / s / 1e12, 1)
        if kind == "tensor3":
            out["tensor_tflops"] = round(ex / s / 1e12, 1)
        out["frac_burst"] = round(ex / s / 1e12 / (rate * pk.get("bf16_tflops", tc_peak)), 4)
        out["frac_sustained"] = round(
            ex / s / 1e12 / (rate * pk.get("bf16_tflops_sustained", tc_peak)), 4)
        if kind == "side":
            out["frac"] = round(ex / s / 1e12 / tc_peak, 4)
            return out
        t_tc = ex / (tc_peak * 1e12)
        t_mem = nb / hbm
        if nb:
            out["gbs"] = round(nb / s / 1e9, 1)
        out["bound"] = "tensor" if t_tc >= t_mem else "hbm"
        out["roofline_ms"] = round(max(t_tc, t_mem) * 1e3, 4)
        out["frac"] = round(max(t_tc, t_mem) / s, 4)
    elif kind == "hbm":
        out["gbs"] = round(nb / s / 1e9, 1)
        out["bound"] = "hbm"
        out["roofline_ms"] = round(nb / hbm * 1e3, 4)
        out["frac"] = round(nb / hbm / s, 4)
    else:   # FP32 FMA gate
        peak = alu_peak_tflops(sm_mhz)
        out["tflops"] = round(fl / s / 1e12, 2)
        out["bound"] = "alu"
        out["roofline_ms"] = round(fl / (peak * 1e12) * 1e3, 4)
        out["frac"] = round(fl / (peak * 1e12) / s, 4)
    return out


def dominant_roofline(stages, work, dom, tc_peak, regime, pk, pk_src, traffic, sm_mhz=None):
    """The roofline object of the bench line for the dominant stage ``dom``."""
    st, w = stages[dom], work[dom]
    r = {"kernel": dom, "traffic": traffic,
         "algorithmic_bytes": w["bytes"] or None}
    fp8 = w["kind"] == "tensor_fp8"
    if st["bound"] == "tensor":
        r.update(bound="tensor", unit="TFLOP/s",
                 achieved=st.get("tensor_tflops", st["tflops"]),
                 peak=tc_peak * (FP8_PER_BF16 if fp8 else 1.0),
                 frac=st["frac"], frac_burst=st["frac_burst"],
                 frac_sustained=st["frac_sustained"],
                 peak_source=(f"{pk_src} bf16 {regime} (median SM clock "
                              f"{'within' if regime == 'burst' else 'below'} 5% of max)"
                              + (", x2 for fp8 (derived: nominal dense fp8 / bf16 rate)"
                                 if fp8 else "")))
    elif st["bound"] == "hbm":
        r.update(bound="hbm", unit="GB/s", achieved=st["gbs"], peak=pk["hbm_gbs"],
                 frac=st["frac"], peak_source=f"{pk_src} HBM copy")
        if "frac_burst" in st:   # a GEMM bound by its operand bytes
            r.update(tensor_frac_burst=st["frac_burst"],
                     tensor_frac_sustained=st["frac_sustained"])
    else:
        r.update(bound="alu", unit="TFLOP/s", achieved=st["tflops"],
                 peak=round(alu_peak_tflops(sm_mhz), 1), frac=st["frac"],
                 peak_source="FP32 FMA: 152 SMs x 128 lanes x 2 x median SM clock")
    return r


def kernel_sources_digest(files=None):
    """sha256 over CUDA sources (all of them, or the named files of csrc/); an ncu
    traffic figure is void once the sources of its kernel change."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "expert_moe_route_gb300", "csrc")
    for name in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()


def traffic_key(wl, mx=False):
    """The traffic table's key of a workload: its name, plus T when not the default
    one, plus "+mx" for the microscaled fp8 expert FFN."""
    from workloads import synth
    default_T = synth.WORKLOADS[wl.name].T
    key = wl.name if wl.T == default_T else f"{wl.name}@T={wl.T}"
    return key + ("+mx" if mx else "")


def profiled_traffic(workload, stage):
    """DRAM bytes per launch of a stage's kernels from the committed ncu summary, or
    None when there is none for this workload or the stage's kernel sources changed
    since it was taken."""
    try:
        with open(PROFILE_TRAFFIC) as fh:
            table = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = table.get("workloads", {}).get(workload, {}).get(stage)
    if not entry:
        return None
    try:
        if entry.get("sources_sha256") != kernel_sources_digest(entry.get("sources", [])):
            return None
    except OSError:
        return None
    return entry.get("bytes_per_launch")


def alu_peak_tflops(sm_mhz):
    """FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOP per cycle."""
    return 152 * 128 * 2 * (sm_mhz or 2070.0) * 1e6 / 1e12


# ---------------------------------------------------------------- our arm
class Opts:
    """What one measured workload runs with."""

    def __init__(self, args, name=None, over=None, flush_l2=None, e2e=None, mx=None):
        self.name = name or args.workload
        self.over = overrides(args) if over is None else over
        self.flush_l2 = args.flush_l2 if flush_l2 is None else flush_l2
        self.e2e = (not args.no_e2e) if e2e is None else e2e
        self.steps, self.warmup = args.steps, args.warmup
        self.fp8 = args.fp8
        self.mx = args.mx if mx is None else mx
        self.single_cta = args.single_cta
        self.no_prepack = args.no_prepack
        self.shared_expert = args.shared_expert
        self.shared_serial = args.shared_serial


def run_ours(o, rank, world, device):
    import torch

    from expert_moe_route_gb300 import binding as B
    from workloads import synth

    wl = synth.workload(o.name, **o.over)
    identity = wl.f == 0
    stream = torch.cuda.current_stream()
    mxw = None

    # ---- inputs, resident in HBM before timing
    if identity:
        r = synth.drawn_routing(wl, device=device)
        x, idx, w = r["x"], r["topk_idx"], r["topk_w"]
        N = wl.T * wl.R
        counts = torch.empty(wl.E, dtype=torch.int32, device=device)
        offsets = torch.empty(wl.E + 1, dtype=torch.int32, device=device)
        row_slot = torch.empty(N, dtype=torch.int32, device=device)
        slot_row = torch.empty(N, dtype=torch.int32, device=device)
        x_perm = torch.empty((N, wl.d), dtype=torch.bfloat16, device=device)
        y = torch.empty_like(x)
        ws = B.workspace(B.dispatch_ws_bytes(wl.T, wl.d, wl.E, wl.R), device)
        if o.fp8:
            xq = torch.empty((N, wl.d), dtype=torch.uint8, device=device)
            xs = torch.empty((N, wl.d // 128), dtype=torch.float32, device=device)

        def step(xin=None, yout=None):
            if o.fp8:   # fp8 dispatch, identity experts dequantise to bf16, bf16 combine
                B.moe_dispatch_fp8(x if xin is None else xin, idx, wl.E, counts, offsets,
                                   row_slot, slot_row, xq, xs, ws)
                B.moe_dequant_fp8(xq, xs, x_perm)
            else:
                B.moe_dispatch(x if xin is None else xin, idx, wl.E, counts, offsets, row_slot,
                               slot_row, x_perm, ws)
            B.moe_combine(x_perm, slot_row, w, y if yout is None else yout, wl.R)
        train = False
        host_in = [("x", x)]
        host_out = [("y", y)]
    else:
        big = wl.E * wl.f * wl.d > (1 << 28)
        inp = synth.layer_inputs(wl, device=device, weight_device=device if big else "cpu")
        train = wl.train
        gemm_flags = B.MOE_SINGLE_CTA_TILES if o.single_cta else 0
        fwd_flags = gemm_flags | (B.MOE_FP8_DISPATCH if o.fp8 else 0)
        weights_note = "plain [E, out, in]"
        mxw = None
        if o.mx and not train:
            # inference in microscaled fp8: the weights are quantised once, outside the timing
            mxw = B.MxWeights(inp["W1"], inp["W3"], inp["W2"])
            torch.cuda.synchronize()
            fwd_flags |= B.MOE_FP8_MX
            weights_note = ("microscaled fp8 (E4M3 codes + a power-of-two scale per 32 along K; "
                            "moe_quantize_mx once, before timing)")
        elif (not train and not o.no_prepack and wl.d % 256 == 0 and wl.f % 128 == 0):
            # inference: the weights are laid out once (like loading a model), outside the timing
            packed = [torch.empty_like(inp[k]) for k in ("W1", "W3", "W2")]
            B.moe_prepack_weights(inp["W1"], inp["W3"], inp["W2"], *packed)
            torch.cuda.synchronize()
            for k, t in zip(("W1", "W3", "W2"), packed):
                inp[k] = t
            del packed
            fwd_flags |= B.MOE_WEIGHTS_PREPACKED
            weights_note = "prepacked tiles (moe_prepack_weights once, before timing)"
        shared = None
        if o.shared_expert:
            fs = o.shared_expert
            sw = {k: v.to(device) for k, v in synth.shared_expert_inputs(wl, fs).items()}
            sg = {}
            if train:
                sg = dict(dW1=torch.empty((fs, wl.d), dtype=torch.float32, device=device),
                          dW3=torch.empty((fs, wl.d), dtype=torch.float32, device=device),
                          dW2=torch.empty((wl.d, fs), dtype=torch.float32, device=device))
            shared = B.Shared(sw["W1"], sw["W3"], sw["W2"], **sg)
            if o.shared_serial:
                gemm_flags |= B.MOE_SHARED_SERIAL
                fwd_flags |= B.MOE_SHARED_SERIAL
        layer = B.Layer(inp["w_gate"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], wl.R, wl.T,
                        shared=shared, mx=mxw)
        saved = B.Saved(layer, device, train=train)
        x = inp["x"]
        y = torch.empty_like(x)
        fws = B.workspace(B.layer_fwd_ws_bytes(layer, fwd_flags), device)
        if train:
            g = inp["g"]
            dx = torch.empty_like(x)
            dWg = torch.empty((wl.d, wl.E), dtype=torch.float32, device=device)
            dW1 = torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device=device)
            dW3 = torch.empty_like(dW1)
            dW2 = torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device=device)
            bws = B.workspace(B.layer_bwd_ws_bytes(layer), device)

        def step(xin=None, yout=None, gin=None, dxout=None):
            xx = x if xin is None else xin
            B.moe_layer_fwd(layer, xx, y if yout is None else yout, saved, fws, flags=fwd_flags)
            if train:
                B.moe_layer_bwd(layer, xx, saved, g if gin is None else gin,
                                dx if dxout is None else dxout, dWg, dW1, dW3, dW2, bws,
                                flags=gemm_flags)
        host_in = [("x", x)] + ([("g", inp["g"])] if train else [])
        host_out = [("y", y)] + ([("dx", dx)] if train else [])
    if identity:
        weights_note = "identity experts"

    # ---- one checked step (device error word) before timing
    if identity:
        step()
        active = wl.E
    else:
        B.moe_layer_fwd(layer, x, y, saved, fws, flags=B.MOE_CHECK | fwd_flags)
        if train:
            B.moe_layer_bwd(layer, x, saved, g, dx, dWg, dW1, dW3, dW2, bws,
                            flags=B.MOE_CHECK | gemm_flags)
        active = int((saved.counts > 0).sum().item())   # experts whose weights are read
    torch.cuda.synchronize()
    for _ in range(o.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region
    traces = [B.StageTrace() for _ in range(o.steps)]
    world_barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    launches0 = B.kernel_launches()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    flush = (torch.empty(512 << 20, dtype=torch.uint8, device=device) if o.flush_l2
             else None)
    # with an L2 flush between steps, each step is timed on its own (the flush
    # between two steps' events is not part of either)
    marks = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(o.steps)] if flush is not None else None)
    t0.record(stream)
    for k in range(o.steps):
        if flush is not None:
            flush.fill_(k & 0xff)
            marks[k][0].record(stream)
        traces[k].arm()
        step()
        if flush is not None:
            marks[k][1].record(stream)
    B.StageTrace.disarm()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = B.kernel_launches() - launches0
    clk = clocks.stop()
    world_barrier(world)
    ms_total = (t0.elapsed_time(t1) if flush is None
                else sum(a.elapsed_time(b) for a, b in marks))
    ms_total = world_max(ms_total, world, device)
    ms_step = ms_total / o.steps
    tokens_per_step = wl.T
    value = job_tokens_per_s(tokens_per_step, world, o.steps, ms_total)

    # ---- per-stage device time, averaged over the timed steps
    stage_ms = {}
    for tr in traces:
        for name, ms in tr.elapsed_ms().items():
            stage_ms[name] = stage_ms.get(name, 0.0) + ms / o.steps
    pk, pk_src = load_peaks()
    tc_peak, regime = tensor_peak(pk, clk)
    work = stage_work(wl, fp8=o.fp8, shared_fs=o.shared_expert, active_experts=active,
                      mx=o.mx and not train)
    if identity:
        ran = ("dispatch", "combine")
    elif train:
        ran = tuple(work)
    else:
        ran = ("gate", "topk", "dispatch", "gateup", "down", "combine", "shared_fwd")
    stages = {}
    for name, ms in stage_ms.items():
        if name not in ran or name not in work or ms <= 0:
            continue
        stages[name] = stage_roofline(work[name], ms, tc_peak, pk, clk.get("sm_mhz"))
    dom = max((n for n in stages if work[n]["kind"] != "side"), key=lambda n: stages[n]["ms"])
    roof = dominant_roofline(stages, work, dom, tc_peak, regime, pk, pk_src,
                             profiled_traffic(traffic_key(wl, mxw is not None), dom),
                             clk.get("sm_mhz"))
    # the whole step: its FLOPs against the tensor peak, and the sum of the
    # stages' roofline times against the measured step
    step_fl = sum(3.0 * w["flops"] if w["kind"] == "tensor3" else w["flops"]
                  for n, w in work.items() if n in ran and w["kind"] != "side")
    step_fp8 = any(w["kind"] == "tensor_fp8" for n, w in work.items() if n in ran)
    step_roof_ms = sum(stages[n]["roofline_ms"] for n in stages if "roofline_ms" in stages[n])
    summary = {"tensor_peak_regime": regime, "tensor_peak_tflops": tc_peak,
               "active_experts": active}
    if step_fl:
        step_tf = step_fl / (ms_step / 1e3) / 1e12
        summary["step_tflops"] = round(step_tf, 1)
        roof["frac_step"] = round(step_tf / tc_peak, 4)   # against the bf16 peak
        if step_fp8:
            roof["frac_step_note"] = "the step's FLOPs against the bf16 peak; its GEMMs run in fp8"
    summary["step_roofline_ms"] = round(step_roof_ms, 4)
    summary["step_frac_of_roofline"] = round(step_roof_ms / ms_step, 4)
    roof["step_frac_of_roofline"] = summary["step_frac_of_roofline"]
    gemm = [n for n in stages if work[n]["kind"] in ("tensor", "tensor_fp8")]
    gemm_ms = sum(stages[n]["ms"] for n in gemm)
    if gemm_ms > 0:
        fl = sum(work[n]["flops"] for n in gemm)
        tf = fl / (gemm_ms / 1e3) / 1e12
        rate = FP8_PER_BF16 if step_fp8 else 1.0
        summary["grouped_gemm_tflops"] = round(tf, 1)
        summary["grouped_gemm_dtype"] = "fp8 (microscaled)" if step_fp8 else "bf16"
        summary["grouped_gemm_frac_burst"] = round(tf / (rate * pk.get("bf16_tflops", tc_peak)), 4)
        summary["grouped_gemm_frac_sustained"] = round(
            tf / (rate * pk.get("bf16_tflops_sustained", tc_peak)), 4)
        summary["grouped_gemm_frac_of_roofline"] = round(
            sum(stages[n]["roofline_ms"] for n in gemm) / gemm_ms, 4)
        summary["grouped_gemm_bound"] = (
            "hbm" if sum(work[n]["bytes"] for n in gemm) / (pk["hbm_gbs"] * 1e9)
            > fl / (rate * tc_peak * 1e12) else "tensor")
    for n in ("dispatch", "combine"):
        if n in stages:
            summary[f"{n}_gbs"] = stages[n]["gbs"]
            summary[f"{n}_frac_of_hbm"] = stages[n]["frac"]

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs in from pinned host memory and its results
    # out to pinned host memory, all inside the timed region.  As a caller
    # would, the copies run on two copy streams with double-buffered device
    # copies, so step k+1's inputs upload and step k's results download while
    # the layer computes.
    e2e = None
    if o.e2e:
        pin_in = {n: t.detach().cpu().pin_memory() for n, t in host_in}
        pin_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in host_out}
        dev_in = [{n: torch.empty_like(t) for n, t in host_in} for _ in range(2)]
        dev_out = [{n: torch.empty_like(t) for n, t in host_out} for _ in range(2)]
        bi = sum(t.numel() * t.element_size() for t in pin_in.values())
        bo = sum(t.numel() * t.element_size() for t in pin_out.values())
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

        def ev():
            return torch.cuda.Event()

        def run_e2e(n_steps):
            in_ready, comp_done, out_done = [None, None], [None, None], [None, None]

            def upload(k):
                b = k % 2
                with torch.cuda.stream(h2d_s):
                    if comp_done[b] is not None:      # step k-2 has finished reading it
                        h2d_s.wait_event(comp_done[b])
                    for n, t in pin_in.items():
                        dev_in[b][n].copy_(t, non_blocking=True)
                    in_ready[b] = ev()
                    in_ready[b].record(h2d_s)

            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            h2d_s.wait_event(t0)
            d2h_s.wait_event(t0)
            upload(0)
            for k in range(n_steps):
                b = k % 2
                if k + 1 < n_steps:
                    upload(k + 1)
                stream.wait_event(in_ready[b])
                if out_done[b] is not None:           # step k-2's results are downloaded
                    stream.wait_event(out_done[b])
                di, do = dev_in[b], dev_out[b]
                if identity or not train:
                    step(xin=di["x"], yout=do["y"])
                else:
                    step(xin=di["x"], yout=do["y"], gin=di["g"], dxout=do["dx"])
                comp_done[b] = ev()
                comp_done[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(comp_done[b])
                    for n, t in pin_out.items():
                        t.copy_(do[n], non_blocking=True)
                    out_done[b] = ev()
                    out_done[b].record(d2h_s)
            for e in out_done:
                if e is not None:
                    stream.wait_event(e)
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        run_e2e(max(1, o.warmup))
        world_barrier(world)
        ems = world_max(run_e2e(o.steps), world, device)
        e2e = {"value": round(job_tokens_per_s(tokens_per_step, world, o.steps, ems), 1),
               "unit": "tokens/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": round(ems / o.steps, 4),
               "copies": "pinned host <-> device on two copy streams, double-buffered, "
                         "overlapping the layer's compute"}

    config = {"workload": synth.describe(wl) + (" fwd+bwd" if train else " fwd")
              + (" fp8-dispatch" if o.fp8 else "") + (" mx-fp8" if mxw is not None else ""),
              "parallelism": f"replicas x{world} (no cross-GPU exchange)",
              "global_batch_tokens": wl.T * world,
              "l2": ("512 MB written between steps (flushes L2); each step timed by its own "
                     "events, the flush outside them" if o.flush_l2 else
                     "inputs larger than L2 every step (no flush)"),
              "weights": weights_note,
              "gemm_tiles": None if identity else
              ("128-row, one CTA" if o.single_cta else "256-row, CTA pairs"),
              "shared_expert": (None if not o.shared_expert else
                                {"fs": o.shared_expert,
                                 "stream": "caller's, after the routed path"
                                 if o.shared_serial else "side stream, overlapped"})}
    result = {"value": round(value, 1), "ms_per_step": round(ms_step, 4), "config": config,
              "roofline": roof, "summary": summary, "stages": stages, "clocks": clk,
              "gpu_launches": launches, "e2e": e2e}
    return result, wl


class LazyExperts:
    """[E, ...] weight tensor whose expert slices are copied to the host on access."""

    def __init__(self, t, bits):
        self.t, self.bits, self.shape = t, bits, tuple(t.shape)

    def __getitem__(self, e):
        return self.bits(self.t[e])


_ORACLE_INPUTS = {}


def _oracle_inputs(wl, device):
    """The workload's seeded inputs for the oracle samples, drawn once per process."""
    import torch

    from workloads import synth
    key = (repr(wl), device)
    if key not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        if wl.f == 0:
            _ORACLE_INPUTS[key] = synth.drawn_routing(wl)
        else:
            big = wl.E * wl.f * wl.d > (1 << 28)
            use_dev = device if (big and torch.cuda.is_available()) else "cpu"
            _ORACLE_INPUTS[key] = synth.layer_inputs(wl, device=use_dev)
    return _ORACLE_INPUTS[key]


def cpu_oracle_sample(wl, device, n_tokens, steps=1, shared_fs=0):
    """Times the CPU oracle (fwd, and bwd for training) on the first n_tokens tokens.

    Returns (tokens/s of the sample, seconds, tokens, experts the sample routes to)."""
    import numpy as np
    import torch

    from oracle import moe_oracle as O
    from workloads import synth

    def bits(t):
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    n = min(n_tokens, wl.T)
    if wl.f == 0:
        r = _oracle_inputs(wl, device)
        x = bits(r["x"])[:n]
        idx = r["topk_idx"].numpy()[:n]
        w = r["topk_w"].numpy()[:n]
        t0 = time.perf_counter()
        for _ in range(steps):
            _, _, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
            xp = O.permute_rows(x, row_slot, wl.R)
            O.combine(O.bf16_to_f64(xp), slot_row, w, n, wl.R)
        dt = time.perf_counter() - t0
        touched = len(np.unique(idx))
    else:
        inp = _oracle_inputs(wl, device)
        x = bits(inp["x"])[:n]
        # expert weights stay where they were drawn; the oracle reads one expert at a time
        W1, W3, W2 = (LazyExperts(inp[k], bits) for k in ("W1", "W3", "W2"))
        wg = inp["w_gate"].cpu().numpy()
        bias = None if inp["bias"] is None else inp["bias"].cpu().numpy()
        g = bits(inp["g"])[:n] if wl.train else None
        shared = None
        if shared_fs:
            sw = synth.shared_expert_inputs(wl, shared_fs)
            shared = tuple(bits(sw[k]) for k in ("W1", "W3", "W2"))
        t0 = time.perf_counter()
        for _ in range(steps):
            fw = O.layer_fwd(x, wg, bias, W1, W3, W2, wl.R, shared=shared)
            if wl.train:
                O.layer_bwd(fw, x, wg, W1, W3, W2, g, wl.R, shared=shared)
        dt = time.perf_counter() - t0
        touched = int((fw["counts"] > 0).sum())
        del fw, W1, W3, W2
        gc.collect()
    return n * steps / dt, dt, n, touched


def full_step_estimate(wl, samples):
    """The oracle's time for the whole workload from timed samples.

    samples: [(tokens, seconds, experts routed to)] at two or more token counts.
    The oracle's cost has a part that grows with the tokens (routing, dispatch,
    the FFN rows, combine) and a part per expert the sample routes to (decoding
    that expert's weights, and in training writing its dense weight gradients);
    the samples are sized so that they route to (nearly) every expert, so a
    straight line through (tokens, mean seconds) separates the two: the slope is
    the per-token cost, the intercept the per-expert part.  Returns a dict with
    the line and the extrapolated time for wl.T tokens.
    """
    by_n = {}
    for n, s, touched in samples:
        by_n.setdefault(n, []).append((s, touched))
    ns = sorted(by_n)
    if len(ns) < 2:
        n = ns[0]
        sec = statistics.mean(s for s, _ in by_n[n])
        return {"per_token_s": sec / n, "fixed_s": 0.0, "full_step_s": sec / n * wl.T,
                "tokens": ns, "experts_routed": [min(t for _, t in by_n[n])],
                "method": "one sample size: proportional"}
    xs = [float(n) for n in ns]
    ys = [statistics.mean(s for s, _ in by_n[n]) for n in ns]
    mx, my = statistics.mean(xs), statistics.mean(ys)
    slope = sum((a - mx) * (b - my) for a, b in zip(xs, ys)) / sum((a - mx) ** 2 for a in xs)
    slope = max(slope, 1e-12)
    fixed = max(0.0, my - slope * mx)
    return {"per_token_s": slope, "fixed_s": fixed, "full_step_s": fixed + slope * wl.T,
            "tokens": ns, "experts_routed": [min(t for _, t in by_n[n]) for n in ns],
            "mean_s": [round(y, 3) for y in ys],
            "method": "straight line through (tokens, seconds), extrapolated to T"}


def cpu_baseline_line(wl, est, cores, runs):
    """The cpu_baseline object: the oracle's extrapolated full-step throughput."""
    value = wl.T / est["full_step_s"]
    return {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "full_step_s": round(est["full_step_s"], 1),
            "sample": (f"the oracle ({'fwd+bwd' if wl.train else 'fwd'}, full d, E, R, f and "
                       f"weights) timed on the first {est['tokens']} tokens of the workload "
                       f"({runs}; they route to {est['experts_routed']} of {wl.E} experts); "
                       f"per-token cost {est['per_token_s'] * 1e3:.2f} ms and fixed per-expert "
                       f"cost {est['fixed_s']:.2f} s from a straight line through the timings, "
                       f"extrapolated to all {wl.T} tokens: {est['full_step_s']:.1f} s per step")}


def overrides(args):
    over = {}
    if args.tokens is not None:
        over["T"] = args.tokens
    if args.experts is not None:
        over["E"] = args.experts
    return over


def world_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def world_max(v, world, device):
    """The maximum of v over all ranks (NCCL on GPUs, gloo on the host)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step, world, steps, ms_total):
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return tokens_per_step * world * steps / (ms_total / 1e3)


def cpu_sample_tokens(wl, args):
    if args.cpu_tokens:
        return tuple(args.cpu_tokens)
    return CPU_SAMPLE_TOKENS.get(wl.name, (64, 128))


def want_extras(args):
    if args.extra_workloads == "on":
        return True
    if args.extra_workloads == "off":
        return False
    return (args.workload == "train" and not overrides(args) and not args.fp8 and not args.mx
            and not args.single_cta and not args.shared_expert and not args.flush_l2)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    from workloads import synth
    wl = synth.workload(args.workload, **overrides(args))
    n1, n2 = cpu_sample_tokens(wl, args)
    device = "cuda:0"
    try:
        import torch
        if not torch.cuda.is_available():
            device = "cpu"
    except ImportError:
        device = "cpu"
    for _ in range(args.warmup):       # warm-up: a few tokens (the oracle's code paths, cached inputs)
        cpu_oracle_sample(wl, device, min(8, n1), shared_fs=args.shared_expert)
    samples, t_all = [], 0.0
    for k in range(args.steps):        # steps alternate between the two sample sizes
        n = n1 if k % 2 == 0 else n2
        _, dt, n, touched = cpu_oracle_sample(wl, device, n, shared_fs=args.shared_expert)
        samples.append((n, dt, touched))
        t_all += dt
    est = full_step_estimate(wl, samples)
    cb = cpu_baseline_line(wl, est, os.cpu_count(),
                           f"{args.steps} timed samples alternating between the two sizes")
    value = cb["value"]
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_all / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (bf16 storage points)",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": synth.describe(wl) + (" fwd+bwd" if wl.train else " fwd"),
                       "parallelism": "host cores"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "note": "value is the oracle's full-workload throughput extrapolated from the "
                    "timed samples; ms_per_step is the mean time of one sample"}
    print(json.dumps(line))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = f"cuda:{torch.cuda.current_device()}"
    res, wl = run_ours(Opts(args), rank, world, device)
    result = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
              "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "bf16 (fp32 accumulation)",
              "data": "synthetic (seeded, shapes and distributions of the workload)"}
    result.update({k: res[k] for k in ("config", "roofline", "summary", "stages", "clocks",
                                       "gpu_launches", "e2e")})
    del res
    gc.collect()
    torch.cuda.empty_cache()
    if want_extras(args):
        extras = []
        for name, over, flush, mx in EXTRA_WORKLOADS:
            r, _ = run_ours(Opts(args, name, over, flush, e2e=False, mx=mx), rank, world, device)
            extras.append({"workload": r["config"]["workload"], "value": r["value"],
                           "unit": "tokens/s", "ms_per_step": r["ms_per_step"],
                           "l2": r["config"]["l2"], "weights": r["config"]["weights"],
                           "roofline": r["roofline"], "summary": r["summary"],
                           "stages": r["stages"], "clocks": r["clocks"],
                           "gpu_launches": r["gpu_launches"]})
            del r
            gc.collect()
            torch.cuda.empty_cache()
        result["workloads"] = extras
    if rank == 0 and not args.no_cpu_baseline:
        n1, n2 = cpu_sample_tokens(wl, args)
        samples = []
        for n in (n1, n2):
            _, dt, n, touched = cpu_oracle_sample(wl, device, n, shared_fs=args.shared_expert)
            samples.append((n, dt, touched))
        result["cpu_baseline"] = cpu_baseline_line(wl, full_step_estimate(wl, samples),
                                                   os.cpu_count(), "one timed sample of each")
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
