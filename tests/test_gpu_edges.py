"""GPU: whole-layer determinism and degenerate inputs."""
import numpy as np
import pytest
import torch

from workloads import synth

pytestmark = pytest.mark.gpu


def _run(B, wl, inp):
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    layer = B.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T)
    saved = B.Saved(layer, "cuda", train=True)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device="cuda")
    B.moe_layer_fwd(layer, dev["x"], y, saved, B.workspace(B.layer_fwd_ws_bytes(layer)),
                    flags=B.MOE_CHECK)
    g = {"dx": torch.empty_like(dev["x"]),
         "dWg": torch.empty((wl.d, wl.E), dtype=torch.float32, device="cuda"),
         "dW1": torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda"),
         "dW3": torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda"),
         "dW2": torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device="cuda")}
    B.moe_layer_bwd(layer, dev["x"], saved, dev["g"], g["dx"], g["dWg"], g["dW1"], g["dW3"],
                    g["dW2"], B.workspace(B.layer_bwd_ws_bytes(layer)), flags=B.MOE_CHECK)
    torch.cuda.synchronize()
    return y, g, saved


def test_layer_forward_and_backward_are_bitwise_reproducible(lib):
    wl = synth.workload("mid", T=1024, f=448)
    inp = synth.layer_inputs(wl, with_grad=True)
    y1, g1, s1 = _run(lib, wl, inp)
    y2, g2, s2 = _run(lib, wl, inp)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(s1.logits.view(torch.int32), s2.logits.view(torch.int32))
    assert torch.equal(s1.slot_row, s2.slot_row)
    for k in g1:
        assert torch.equal(g1[k].view(torch.int16 if g1[k].dtype == torch.bfloat16 else torch.int32),
                           g2[k].view(torch.int16 if g2[k].dtype == torch.bfloat16 else torch.int32)), k


def test_zero_tokens(lib):
    wl = synth.workload("tiny", T=0)
    inp = synth.layer_inputs(synth.workload("tiny", T=8), with_grad=True)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    layer = lib.Layer(dev["w_gate"], None, dev["W1"], dev["W3"], dev["W2"], wl.R, 0)
    saved = lib.Saved(layer, "cuda", train=True)
    x0 = torch.empty((0, wl.d), dtype=torch.bfloat16, device="cuda")
    y0 = torch.empty_like(x0)
    # tensors of size 0 have no storage; the library must accept T = 0 and do nothing
    ws = lib.workspace(lib.layer_fwd_ws_bytes(layer))
    import ctypes
    n = ctypes.c_size_t(ws.numel())
    st = lib.lib().moe_layer_fwd(ctypes.byref(layer.c), ctypes.c_void_p(ws.data_ptr()),
                                 ctypes.c_void_p(ws.data_ptr()), ctypes.byref(saved.c),
                                 ctypes.c_void_p(ws.data_ptr()), ctypes.byref(n), lib.MOE_CHECK,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0
    dW = [torch.full(sh, 7.0, device="cuda") for sh in ((wl.d, wl.E), (wl.E, wl.f, wl.d),
                                                        (wl.E, wl.f, wl.d), (wl.E, wl.d, wl.f))]
    bws = lib.workspace(lib.layer_bwd_ws_bytes(layer))
    st = lib.lib().moe_layer_bwd(ctypes.byref(layer.c), None, ctypes.byref(saved.c), None, None,
                                 *[t.data_ptr() for t in dW], bws.data_ptr(),
                                 ctypes.byref(ctypes.c_size_t(bws.numel())), lib.MOE_CHECK,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0 and not any(t.any() for t in dW)       # no tokens: zero gradients
    counts = torch.full((wl.E,), 5, dtype=torch.int32, device="cuda")
    offsets = torch.full((wl.E + 1,), 5, dtype=torch.int32, device="cuda")
    dws = lib.workspace(lib.dispatch_ws_bytes(0, wl.d, wl.E, wl.R))
    st = lib.lib().moe_dispatch_fp8(None, None, 0, wl.d, wl.E, wl.R, counts.data_ptr(),
                                    offsets.data_ptr(), None, None, None, None, dws.data_ptr(),
                                    ctypes.byref(ctypes.c_size_t(dws.numel())), lib.MOE_CHECK,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert not counts.any() and not offsets.any()


def test_fp8_dispatch_reports_bad_routing(lib):
    T, d, E, R = 32, 128, 4, 2
    x = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    idx = torch.tensor(np.tile([0, 1], (T, 1)), dtype=torch.int32, device="cuda")
    idx[7, 0] = -1
    N = T * R
    bufs = [torch.empty(E, dtype=torch.int32, device="cuda"),
            torch.empty(E + 1, dtype=torch.int32, device="cuda"),
            torch.empty(N, dtype=torch.int32, device="cuda"),
            torch.empty(N, dtype=torch.int32, device="cuda"),
            torch.empty((N, d), dtype=torch.uint8, device="cuda"),
            torch.empty((N, 1), dtype=torch.float32, device="cuda")]
    ws = lib.workspace(lib.dispatch_ws_bytes(T, d, E, R))
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_dispatch_fp8(x, idx, E, *bufs, ws, flags=lib.MOE_CHECK)
    assert ei.value.status == 4
