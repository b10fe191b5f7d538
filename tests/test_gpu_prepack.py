"""GPU: prepacked forward weight tiles give the same results bit for bit."""
import pytest
import torch

from workloads import synth

pytestmark = pytest.mark.gpu


def _prepack(B, W1, W3, W2):
    P = [torch.empty_like(W1), torch.empty_like(W3), torch.empty_like(W2)]
    B.moe_prepack_weights(W1, W3, W2, *P)
    torch.cuda.synchronize()
    return P


def test_prepack_layout(lib):
    E, d, f = 3, 512, 384
    g = torch.Generator(device="cuda").manual_seed(1)
    W1, W3 = (torch.randn((E, f, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    W2 = torch.randn((E, d, f), generator=g, device="cuda").to(torch.bfloat16)
    P1, P3, P2 = _prepack(lib, W1, W3, W2)
    for W, P in ((W1, P1), (W3, P3)):
        want = W.view(E, f // 128, 128, d // 64, 64).permute(0, 1, 3, 2, 4).contiguous()
        assert torch.equal(P.view(E, f // 128, d // 64, 128, 64), want)
    want = W2.view(E, d // 256, 256, f // 64, 64).permute(0, 1, 3, 2, 4).contiguous()
    assert torch.equal(P2.view(E, d // 256, f // 64, 256, 64), want)


@pytest.mark.parametrize("name,T", [("tiny", None), ("mid", None), ("large", 1024)])
def test_layer_forward_prepacked_is_bitwise_equal(lib, name, T):
    wl = synth.workload(name) if T is None else synth.workload(name, T=T)
    inp = synth.layer_inputs(wl, device="cuda")
    layer = lib.Layer(inp["w_gate"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], wl.R, wl.T)
    P = _prepack(lib, inp["W1"], inp["W3"], inp["W2"])
    packed = lib.Layer(inp["w_gate"], inp["bias"], *P, wl.R, wl.T)
    outs = []
    for lay, flags in ((layer, 0), (packed, lib.MOE_WEIGHTS_PREPACKED)):
        saved = lib.Saved(lay, "cuda", train=False)
        y = torch.empty_like(inp["x"])
        lib.moe_layer_fwd(lay, inp["x"], y, saved, lib.workspace(lib.layer_fwd_ws_bytes(lay)),
                          flags=flags | lib.MOE_CHECK)
        outs.append((y, saved.h, saved.o))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # the backward takes the plain layout only
    with pytest.raises(lib.MoeError) as ei:
        z = torch.empty(1, device="cuda")
        lib.moe_layer_bwd(packed, inp["x"], lib.Saved(packed, "cuda"), inp["x"], inp["x"], z, z, z,
                          z, lib.workspace(1024), flags=lib.MOE_WEIGHTS_PREPACKED)
    assert ei.value.status == 2
