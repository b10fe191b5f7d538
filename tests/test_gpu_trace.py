"""GPU: per-stage trace events and the library's kernel-launch counter."""
import pytest
import torch

from workloads import synth

pytestmark = pytest.mark.gpu


def test_trace_events_and_launch_count(lib):
    wl = synth.workload("tiny", T=300)
    inp = synth.layer_inputs(wl, with_grad=True)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T)
    saved = lib.Saved(layer, "cuda", train=True)
    y = torch.empty_like(dev["x"])
    fws = lib.workspace(lib.layer_fwd_ws_bytes(layer))
    bws = lib.workspace(lib.layer_bwd_ws_bytes(layer))
    dx = torch.empty_like(dev["x"])
    dWg = torch.empty((wl.d, wl.E), dtype=torch.float32, device="cuda")
    dW1 = torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda")
    dW3 = torch.empty_like(dW1)
    dW2 = torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device="cuda")
    tr = lib.StageTrace()
    n0 = lib.kernel_launches()
    tr.arm()
    lib.moe_layer_fwd(layer, dev["x"], y, saved, fws)
    lib.moe_layer_bwd(layer, dev["x"], saved, dev["g"], dx, dWg, dW1, dW3, dW2, bws)
    lib.StageTrace.disarm()
    torch.cuda.synchronize()
    # fwd: W_g split, gate GEMM (K over four CTAs at this size) and the partials'
    #      sum, topk, 4 dispatch, tile list, gate-up (pairs, then one CTA for the
    #      experts' last tiles of at most 128 rows), down (same), combine
    # bwd: route, tile list, DH (2), DX (2), per-expert weight-gradient maps, WG2, WG13,
    #      dW_g (operand S, per-chunk maps, GEMM, sum), W_g^T, dx
    assert lib.kernel_launches() - n0 == 14 + 15
    ms = tr.elapsed_ms()
    for name in lib.STAGES:
        assert ms[name] > 0.0, name
    # a traced call still reports no error afterwards
    lib.moe_layer_fwd(layer, dev["x"], y, saved, fws, flags=lib.MOE_CHECK)
