"""GPU: the layer's forward and backward captured in a CUDA graph and
replayed (the library enqueues everything on the caller's stream, allocates
nothing and does not synchronise; the shared expert's side stream becomes a
fork and join inside the graph).  Replays on new inputs give the eager results
bit for bit."""
import pytest
import torch

from workloads import synth

pytestmark = pytest.mark.gpu


def _same(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("shared_fs", [0, 512])
def test_layer_fwd_bwd_in_a_cuda_graph(lib, shared_fs):
    wl = synth.workload("train", T=512)
    inp = synth.layer_inputs(wl, with_grad=True)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    shared = None
    if shared_fs:
        sw = {k: v.cuda() for k, v in synth.shared_expert_inputs(wl, shared_fs).items()}
        shared = lib.Shared(sw["W1"], sw["W3"], sw["W2"],
                            torch.empty((shared_fs, wl.d), device="cuda"),
                            torch.empty((shared_fs, wl.d), device="cuda"),
                            torch.empty((wl.d, shared_fs), device="cuda"))
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T,
                      shared=shared)
    saved = lib.Saved(layer, "cuda", train=True)
    fws = lib.workspace(lib.layer_fwd_ws_bytes(layer))
    bws = lib.workspace(lib.layer_bwd_ws_bytes(layer))
    x = dev["x"].clone()
    g = dev["g"].clone()
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dWg = torch.empty((wl.d, wl.E), device="cuda")
    dW1 = torch.empty((wl.E, wl.f, wl.d), device="cuda")
    dW3 = torch.empty_like(dW1)
    dW2 = torch.empty((wl.E, wl.d, wl.f), device="cuda")

    def step():
        lib.moe_layer_fwd(layer, x, y, saved, fws)
        lib.moe_layer_bwd(layer, x, saved, g, dx, dWg, dW1, dW3, dW2, bws)

    def results():
        out = [y.clone(), dx.clone(), dWg.clone(), dW1.clone(), dW3.clone(), dW2.clone()]
        if shared is not None:
            out += [shared.dW1.clone(), shared.dW3.clone(), shared.dW2.clone()]
        return out

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                       # first call outside the capture (per-device set-up)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    gen = torch.Generator().manual_seed(7)
    for rep in range(3):
        x.copy_(torch.randn(x.shape, generator=gen).to(torch.bfloat16))
        g.copy_(torch.randn(g.shape, generator=gen).to(torch.bfloat16))
        torch.cuda.synchronize()
        step()                       # eager on the same inputs
        torch.cuda.synchronize()
        want = results()
        graph.replay()
        torch.cuda.synchronize()
        got = results()
        for i, (a, b) in enumerate(zip(got, want)):
            assert _same(a, b), (rep, i)
