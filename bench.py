"""Benchmark of the MoE layer hot path on GB300 (one JSON line on rank 0).

Default workload: the MoE layer training step (forward + backward) with
T=16384 tokens, d=4096, E=128 experts, top-8 routing, SwiGLU width f=1536 --
one pass of every step of the path (route, dispatch, grouped SwiGLU FFN,
combine, and their backward).  Other workloads: --workload large | large_hot |
mid | tiny (forward only) and dispatch (dispatch + combine with identity
experts, --tokens T).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

value = tokens per second of the whole job (all ranks); each rank runs an
independent replica of the workload (the path has no cross-GPU exchange), so
scaling is weak.  The timed region is K back-to-back steps between CUDA events
on the launching stream, after W warm-up steps, bracketed by a barrier and a
device synchronisation; the max over ranks is reported.  Each step streams
more than L2 (5 GB of expert weights for the default workload), so no flush
is needed between steps.
"""
from __future__ import annotations

import argparse
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


def parse():
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
    p.add_argument("--cpu-tokens", type=int, default=None,
                   help="tokens in the CPU oracle sample (default per workload)")
    p.add_argument("--fp8", action="store_true",
                   help="block-scaled fp8 dispatch (E4M3 + per-128 scales), bf16 combine: "
                        "dispatch workloads dequantise in identity experts; layer workloads "
                        "pass MOE_FP8_DISPATCH (the GEMMs read the dequantised rows)")
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
                   help="write a 512 MB buffer (4x L2) between timed steps, outside the stage "
                        "events, so small workloads read HBM; ms_per_step then includes it")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def load_peaks():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


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
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
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
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxs) if maxs else None, "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------- work model
def stage_work(wl, fp8=False, shared_fs=0):
    """Algorithmic work of one launch of each traced stage: (kind, amount).

    kind "tflop": FLOPs of real rows only (no padding); "side": the same for the
    shared expert's GEMMs (overlapping other stages); "gb": bytes that must
    move to or from HBM at least once (reads of inputs + writes of outputs);
    "tflop3": the gate projection x W_g on the tensor cores as three bf16
    products (W_g split into hi + mid + lo), so the pipe executes 3x the
    algorithmic FLOPs counted here; "alu": the FP32 FMA gate (d % 64 != 0).
    """
    T, d, E, R, f = wl.T, wl.d, wl.E, wl.R, wl.f
    N = T * R
    q8 = N * d + 4.0 * N * d / 128          # fp8 codes and their scales
    # fp8 in a layer: the codes and scales are written, read back and the bf16
    # rows the GEMMs read are written, all inside the dispatch stage
    disp = (2.0 * N * d if not fp8 else q8 if not f else 2.0 * q8 + 2.0 * N * d)
    w = {
        "gate": ("tflop3" if d % 64 == 0 else "alu", 2.0 * T * d * E),
        "topk": ("gb", 4.0 * T * E + 8.0 * N),
        "dispatch": ("gb", 2.0 * T * d + disp + 4.0 * N * 3),
        "combine": ("gb", 2.0 * N * d + 8.0 * N + 2.0 * T * d),
    }
    if f:
        w.update({
            "gateup": ("tflop", 4.0 * N * d * f),
            "down": ("tflop", 2.0 * N * d * f),
            "bwd_route": ("gb", 2.0 * T * d + 2.0 * N * d + 2.0 * N * d + 12.0 * N),
            "bwd_dh": ("tflop", 2.0 * N * d * f),
            "bwd_dx": ("tflop", 4.0 * N * d * f),
            "bwd_wg2": ("tflop", 2.0 * N * d * f),
            "bwd_wg13": ("tflop", 4.0 * N * d * f),
            # x once (its rows are gathered through row_slot, the R reads of a
            # row mostly from L2), row_slot and dsel per row, dW_g written
            "bwd_dwg": ("gb", 2.0 * T * d + 8.0 * N + 4.0 * d * E),
            "bwd_dxc": ("gb", 2.0 * N * d + 2.0 * T * d + 8.0 * E * d),
        })
    if f and shared_fs:
        # the shared expert on the side stream: reported, but its time overlaps
        # other stages, so it stays out of the GEMM summary and the dominant kernel
        w.update({"shared_fwd": ("side", 6.0 * T * d * shared_fs),
                  "shared_bwd": ("side", 12.0 * T * d * shared_fs)})
    return w


def kernel_sources_digest():
    """sha256 over the CUDA sources; ncu traffic is void once they change."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "expert_moe_route_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload, stage):
    """DRAM bytes per launch of a stage's kernel from the committed ncu summary, or None
    when there is none for this workload or the kernels changed since it was taken."""
    try:
        with open(PROFILE_TRAFFIC) as fh:
            table = json.load(fh)
    except (OSError, ValueError):
        return None
    if table.get("kernel_sources_sha256") != kernel_sources_digest():
        return None
    entry = table.get("workloads", {}).get(workload, {}).get(stage)
    return entry.get("bytes_per_launch") if entry else None


def alu_peak_tflops(sm_mhz):
    """FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOP per cycle."""
    return 152 * 128 * 2 * (sm_mhz or 2070.0) * 1e6 / 1e12


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, device):
    import torch

    from expert_moe_route_gb300 import binding as B
    from expert_moe_route_gb300 import synth

    wl = synth.workload(args.workload, **overrides(args))
    identity = wl.f == 0
    stream = torch.cuda.current_stream()

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
        if args.fp8:
            xq = torch.empty((N, wl.d), dtype=torch.uint8, device=device)
            xs = torch.empty((N, wl.d // 128), dtype=torch.float32, device=device)

        def step(xin=None, yout=None):
            if args.fp8:   # fp8 dispatch, identity experts dequantise to bf16, bf16 combine
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
        gemm_flags = B.MOE_SINGLE_CTA_TILES if args.single_cta else 0
        fwd_flags = gemm_flags | (B.MOE_FP8_DISPATCH if args.fp8 else 0)
        weights_note = "plain [E, out, in]"
        if (not train and not args.no_prepack and wl.d % 256 == 0 and wl.f % 128 == 0):
            # inference: the weights are laid out once (like loading a model), outside the timing
            packed = [torch.empty_like(inp[k]) for k in ("W1", "W3", "W2")]
            B.moe_prepack_weights(inp["W1"], inp["W3"], inp["W2"], *packed)
            torch.cuda.synchronize()
            for k, t in zip(("W1", "W3", "W2"), packed):
                inp[k] = t
            fwd_flags |= B.MOE_WEIGHTS_PREPACKED
            weights_note = "prepacked tiles (moe_prepack_weights once, before timing)"
        shared = None
        if args.shared_expert:
            fs = args.shared_expert
            sw = {k: v.to(device) for k, v in synth.shared_expert_inputs(wl, fs).items()}
            sg = {}
            if train:
                sg = dict(dW1=torch.empty((fs, wl.d), dtype=torch.float32, device=device),
                          dW3=torch.empty((fs, wl.d), dtype=torch.float32, device=device),
                          dW2=torch.empty((wl.d, fs), dtype=torch.float32, device=device))
            shared = B.Shared(sw["W1"], sw["W3"], sw["W2"], **sg)
            if args.shared_serial:
                gemm_flags |= B.MOE_SHARED_SERIAL
                fwd_flags |= B.MOE_SHARED_SERIAL
        layer = B.Layer(inp["w_gate"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], wl.R, wl.T,
                        shared=shared)
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
    else:
        B.moe_layer_fwd(layer, x, y, saved, fws, flags=B.MOE_CHECK | fwd_flags)
        if train:
            B.moe_layer_bwd(layer, x, saved, g, dx, dWg, dW1, dW3, dW2, bws,
                            flags=B.MOE_CHECK | gemm_flags)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region
    traces = [B.StageTrace() for _ in range(args.steps)]
    world_barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    launches0 = B.kernel_launches()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    flush = (torch.empty(512 << 20, dtype=torch.uint8, device=device) if args.flush_l2
             else None)
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(k & 0xff)
        traces[k].arm()
        step()
    B.StageTrace.disarm()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = B.kernel_launches() - launches0
    clk = clocks.stop()
    world_barrier(world)
    ms_total = t0.elapsed_time(t1)
    ms_total = world_max(ms_total, world, device)
    ms_step = ms_total / args.steps
    tokens_per_step = wl.T
    value = job_tokens_per_s(tokens_per_step, world, args.steps, ms_total)

    # ---- per-stage device time, averaged over the timed steps
    stage_ms = {}
    for tr in traces:
        for name, ms in tr.elapsed_ms().items():
            stage_ms[name] = stage_ms.get(name, 0.0) + ms / args.steps
    pk, pk_src = load_peaks()
    work = stage_work(wl, fp8=args.fp8, shared_fs=args.shared_expert)
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
        kind, amount = work[name]
        if kind == "tflop":
            ach = amount / (ms / 1e3) / 1e12
            stages[name] = {"ms": round(ms, 4), "tflops": round(ach, 1),
                            "frac": round(ach / pk["bf16_tflops_sustained"], 4)}
        elif kind == "gb":
            ach = amount / (ms / 1e3) / 1e9
            stages[name] = {"ms": round(ms, 4), "gbs": round(ach, 1),
                            "frac": round(ach / pk["hbm_gbs"], 4)}
        elif kind == "side":
            ach = amount / (ms / 1e3) / 1e12
            stages[name] = {"ms": round(ms, 4), "tflops": round(ach, 1),
                            "frac": round(ach / pk["bf16_tflops_sustained"], 4),
                            "overlaps_other_stages": not args.shared_serial}
        elif kind == "tflop3":
            ach = amount / (ms / 1e3) / 1e12
            stages[name] = {"ms": round(ms, 4), "tflops": round(ach, 1),
                            "tensor_tflops": round(3 * ach, 1),
                            "frac": round(3 * ach / pk["bf16_tflops_sustained"], 4)}
        else:
            ach = amount / (ms / 1e3) / 1e12
            stages[name] = {"ms": round(ms, 4), "tflops": round(ach, 2),
                            "frac": round(ach / alu_peak_tflops(clk.get("sm_mhz")), 4)}
    dom = max((n for n in stages if work[n][0] != "side"), key=lambda n: stages[n]["ms"])
    kind, amount = work[dom]
    traffic = profiled_traffic(wl.name, dom)
    if kind in ("tflop", "tflop3"):
        roof = {"bound": "tensor", "kernel": dom,
                "achieved": stages[dom].get("tensor_tflops", stages[dom]["tflops"]),
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": stages[dom]["frac"], "traffic": traffic,
                "peak_source": f"{pk_src} bf16 sustained (kernel timed inside a long step)"}
    elif kind == "gb":
        roof = {"bound": "hbm", "kernel": dom, "achieved": stages[dom]["gbs"],
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": stages[dom]["frac"],
                "traffic": traffic, "peak_source": f"{pk_src} HBM copy"}
    else:
        roof = {"bound": "alu", "kernel": dom, "achieved": stages[dom]["tflops"],
                "peak": round(alu_peak_tflops(clk.get("sm_mhz")), 1), "unit": "TFLOP/s",
                "frac": stages[dom]["frac"], "traffic": traffic,
                "peak_source": "FP32 FMA: 152 SMs x 128 lanes x 2 x median SM clock"}
    gemm = [n for n in stages if work[n][0] == "tflop"]
    gemm_ms = sum(stages[n]["ms"] for n in gemm)
    gemm_fl = sum(work[n][1] for n in gemm)
    summary = {}
    if gemm_ms > 0:
        tf = gemm_fl / (gemm_ms / 1e3) / 1e12
        summary["grouped_gemm_tflops"] = round(tf, 1)
        summary["grouped_gemm_frac_of_bf16_peak"] = round(tf / pk["bf16_tflops_sustained"], 4)
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
    if not args.no_e2e:
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

        run_e2e(max(1, args.warmup))
        world_barrier(world)
        ems = world_max(run_e2e(args.steps), world, device)
        e2e = {"value": round(job_tokens_per_s(tokens_per_step, world, args.steps, ems), 1),
               "unit": "tokens/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": round(ems / args.steps, 4),
               "copies": "pinned host <-> device on two copy streams, double-buffered, "
                         "overlapping the layer's compute"}

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (fp32 accumulation)",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": synth.describe(wl) + (" fwd+bwd" if train else " fwd")
                   + (" fp8-dispatch" if args.fp8 else ""),
                   "parallelism": f"replicas x{world} (no cross-GPU exchange)",
                   "global_batch_tokens": wl.T * world,
                   "l2": ("512 MB written between steps (flushes L2; outside the stage events, "
                          "inside ms_per_step)" if args.flush_l2 else
                          "inputs larger than L2 every step (no flush)"),
                   "weights": weights_note,
                   "gemm_tiles": None if identity else
                   ("128-row, one CTA" if args.single_cta else "256-row, CTA pairs"),
                   "shared_expert": (None if not args.shared_expert else
                                     {"fs": args.shared_expert,
                                      "stream": "caller's, after the routed path"
                                      if args.shared_serial else "side stream, overlapped"})},
        "roofline": roof,
        "summary": summary,
        "stages": stages,
        "clocks": clk,
        "gpu_launches": launches,
        "e2e": e2e,
    }
    return result, wl


class LazyExperts:
    """[E, ...] weight tensor whose expert slices are copied to the host on access."""

    def __init__(self, t, bits):
        self.t, self.bits, self.shape = t, bits, tuple(t.shape)

    def __getitem__(self, e):
        return self.bits(self.t[e])


def cpu_oracle_sample(wl, device, n_tokens, steps=1, shared_fs=0):
    """Times the CPU oracle (fwd, and bwd for training) on the first n_tokens tokens."""
    import numpy as np
    import torch

    from expert_moe_route_gb300 import synth
    from oracle import moe_oracle as O

    def bits(t):
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    n = min(n_tokens, wl.T)
    if wl.f == 0:
        r = synth.drawn_routing(wl)
        x = bits(r["x"])[:n]
        idx = r["topk_idx"].numpy()[:n]
        w = r["topk_w"].numpy()[:n]
        t0 = time.perf_counter()
        for _ in range(steps):
            _, _, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
            xp = O.permute_rows(x, row_slot, wl.R)
            O.combine(O.bf16_to_f64(xp), slot_row, w, n, wl.R)
        dt = time.perf_counter() - t0
    else:
        big = wl.E * wl.f * wl.d > (1 << 28)
        use_dev = device if (big and torch.cuda.is_available()) else "cpu"
        inp = synth.layer_inputs(wl, device=use_dev)
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
    return n * steps / dt, dt, n


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


def default_cpu_tokens(wl):
    if wl.f == 0:
        return 4096
    return {"train": 192, "large": 16, "large_hot": 16, "mid": 512, "tiny": 256}.get(wl.name, 128)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

    if args.impl == "reference":
        if rank != 0:
            return
        from expert_moe_route_gb300 import synth
        wl = synth.workload(args.workload, **overrides(args))
        n = args.cpu_tokens or (8 if wl.f else 1024)
        device = "cuda:0"
        try:
            import torch
            if not torch.cuda.is_available():
                device = "cpu"
        except ImportError:
            device = "cpu"
        for _ in range(args.warmup):
            cpu_oracle_sample(wl, device, n, shared_fs=args.shared_expert)
        rates = []
        t_all = 0.0
        for _ in range(args.steps):
            rate, dt, _ = cpu_oracle_sample(wl, device, n, shared_fs=args.shared_expert)
            rates.append(rate)
            t_all += dt
        value = n * args.steps / t_all
        line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * t_all / args.steps, 2), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64 (bf16 storage points)",
                "data": "synthetic (seeded)", "impl": "reference",
                "config": {"workload": synth.describe(wl) + (" fwd+bwd" if wl.train else " fwd"),
                           "parallelism": "host cores"},
                "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                                 "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": f"each step: the oracle on the first {n} of {wl.T} tokens "
                                           f"of the workload (full d, E, R, f and weights)"},
                "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = f"cuda:{torch.cuda.current_device()}"
    result, wl = run_ours(args, rank, world, device)
    if rank == 0 and not args.no_cpu_baseline:
        n = args.cpu_tokens or default_cpu_tokens(wl)
        rate, dt, n = cpu_oracle_sample(wl, device, n, shared_fs=args.shared_expert)
        result["cpu_baseline"] = {
            "value": round(rate, 2), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"the oracle ({'fwd+bwd' if wl.train else 'fwd'}) on the first {n} of "
                      f"{wl.T} tokens (full d, E, R, f and weights), {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
