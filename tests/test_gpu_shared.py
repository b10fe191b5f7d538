"""GPU parity: the shared expert (a SwiGLU FFN every token passes through,
added to the routed experts' weighted sum with weight 1), run on the
library's side stream beside route / dispatch / the routed FFN, and on the
caller's stream (MOE_SHARED_SERIAL): the same bits either way, and the oracle's
values."""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64, near_tie_tokens

pytestmark = pytest.mark.gpu


def _run(B, wl, inp, sw, fs, flags, train=True):
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sdev = {k: v.cuda() for k, v in sw.items()}
    grads = dict(dW1=torch.full((fs, wl.d), 7.0, device="cuda"),
                 dW3=torch.full((fs, wl.d), 7.0, device="cuda"),
                 dW2=torch.full((wl.d, fs), 7.0, device="cuda"))
    shared = B.Shared(sdev["W1"], sdev["W3"], sdev["W2"], **grads)
    layer = B.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T,
                    shared=shared)
    saved = B.Saved(layer, "cuda", train=train)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device="cuda")
    B.moe_layer_fwd(layer, dev["x"], y, saved, B.workspace(B.layer_fwd_ws_bytes(layer)),
                    flags=flags | B.MOE_CHECK)
    out = dict(y=y, saved=saved)
    if train:
        dx = torch.empty_like(dev["x"])
        dWg = torch.empty((wl.d, wl.E), dtype=torch.float32, device="cuda")
        dW1 = torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda")
        dW3 = torch.empty_like(dW1)
        dW2 = torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device="cuda")
        B.moe_layer_bwd(layer, dev["x"], saved, dev["g"], dx, dWg, dW1, dW3, dW2,
                        B.workspace(B.layer_bwd_ws_bytes(layer)), flags=flags | B.MOE_CHECK)
        out.update(dx=dx, dWg=dWg, dW1=dW1, dW3=dW3, dW2=dW2, **{"s" + k: v for k, v in grads.items()})
    torch.cuda.synchronize()
    return out


def _same(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("name,over,fs", [("tiny", {}, 512), ("train", dict(T=512), 1536),
                                          ("mid", dict(T=1024, f=448), 256)])
def test_shared_expert_forward_backward_against_oracle(lib, name, over, fs):
    wl = synth.workload(name, **over)
    inp = synth.layer_inputs(wl, with_grad=True)
    sw = synth.shared_expert_inputs(wl, fs)
    got = _run(lib, wl, inp, sw, fs, 0)
    Ws = (bits(sw["W1"]), bits(sw["W3"]), bits(sw["W2"]))
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    ref = O.layer_fwd(bits(inp["x"]), inp["w_gate"].numpy(), bias, bits(inp["W1"]),
                      bits(inp["W3"]), bits(inp["W2"]), wl.R, shared=Ws)
    sv = got["saved"]
    # the shared expert does not depend on the routing
    assert_close(f64(sv.sh), ref["sh"], "sh")
    assert_close(f64(sv.sa), O.bf16_round(ref["sa"]), "sa")
    assert_close(f64(sv.sb), O.bf16_round(ref["sb"]), "sb")
    tie = near_tie_tokens(ref["logits"], wl.R)
    same = (sv.topk_idx.cpu().numpy() == ref["idx"]).all(axis=1)
    assert (same | tie).all(), "routing differs on a token without a near tie"
    assert_close(f64(got["y"])[same], ref["y"][same], "y")
    rb = O.layer_bwd(ref, bits(inp["x"]), inp["w_gate"].numpy(), bits(inp["W1"]),
                     bits(inp["W3"]), bits(inp["W2"]), bits(inp["g"]), wl.R, shared=Ws)
    # the shared expert's weight gradients sum over every token; a near-tie
    # token changes only its own dx and routed gradients
    assert_close(f64(got["sdW1"]), rb["dWs1"], "dWs1")
    assert_close(f64(got["sdW3"]), rb["dWs3"], "dWs3")
    assert_close(f64(got["sdW2"]), rb["dWs2"], "dWs2")
    assert_close(f64(got["dx"])[same], rb["dx"][same], "dx")


@pytest.mark.parametrize("name,over,fs", [("train", dict(T=512), 1536), ("mid", dict(T=1024), 640)])
def test_side_stream_and_serial_give_the_same_bits(lib, name, over, fs):
    wl = synth.workload(name, **over)
    inp = synth.layer_inputs(wl, with_grad=True)
    sw = synth.shared_expert_inputs(wl, fs)
    a = _run(lib, wl, inp, sw, fs, 0)
    b = _run(lib, wl, inp, sw, fs, lib.MOE_SHARED_SERIAL)
    for k in ("y", "dx", "dWg", "dW1", "dW3", "dW2", "sdW1", "sdW3", "sdW2"):
        assert _same(a[k], b[k]), k
    for k in ("sa", "sb", "sh", "h", "o", "x_perm"):
        assert _same(getattr(a["saved"], k), getattr(b["saved"], k)), k


def test_shared_expert_leaves_the_routed_path_alone_and_inference_matches(lib):
    wl = synth.workload("train", T=512)
    inp = synth.layer_inputs(wl, with_grad=True)
    fs = 1024
    sw = synth.shared_expert_inputs(wl, fs)
    with_shared = _run(lib, wl, inp, sw, fs, 0)
    infer = _run(lib, wl, inp, sw, fs, 0, train=False)
    assert _same(with_shared["y"], infer["y"])
    # no shared expert: the routed intermediates are bit-identical
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T)
    saved = lib.Saved(layer, "cuda", train=True)
    y = torch.empty_like(dev["x"])
    lib.moe_layer_fwd(layer, dev["x"], y, saved, lib.workspace(lib.layer_fwd_ws_bytes(layer)),
                      flags=lib.MOE_CHECK)
    torch.cuda.synchronize()
    for k in ("logits", "topk_idx", "x_perm", "h", "o"):
        assert _same(getattr(saved, k), getattr(with_shared["saved"], k)), k
    # y - (routed-only y) is the shared expert's output, to within two bf16 roundings
    s_ref = O.shared_expert_fwd(bits(inp["x"]), bits(sw["W1"]), bits(sw["W3"]), bits(sw["W2"]))[3]
    diff = f64(with_shared["y"]) - f64(y)
    assert np.abs(diff - s_ref).max() <= 4 * 2.0 ** -8 * (np.abs(f64(y)).max() + np.abs(s_ref).max())


def test_shared_expert_argument_checks(lib):
    wl = synth.workload("tiny")
    inp = synth.layer_inputs(wl)
    d = wl.d
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    W = torch.zeros((60, d), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((d, 60), dtype=torch.bfloat16, device="cuda")
    sh = lib.Shared(W, W, W2)
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T,
                      shared=sh)
    with pytest.raises(lib.MoeError) as ei:            # fs % 8 != 0
        lib.layer_fwd_ws_bytes(layer)
    assert ei.value.status == 2
    W = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((d, 64), dtype=torch.bfloat16, device="cuda")
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T,
                      shared=lib.Shared(W, W, W2))
    saved = lib.Saved(layer, "cuda", train=True)
    z = torch.empty(1, device="cuda")
    with pytest.raises(lib.MoeError) as ei:            # backward without shared gradient buffers
        lib.moe_layer_bwd(layer, dev["x"], saved, dev["x"], dev["x"], z, z, z, z,
                          lib.workspace(lib.layer_bwd_ws_bytes(layer)))
    assert ei.value.status == 1
