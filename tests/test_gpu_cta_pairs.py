"""GPU: the expert GEMMs on 256-row tiles shared by CTA pairs (tcgen05
.cta_group::2, the default) against single-CTA 128-row tiles
(MOE_SINGLE_CTA_TILES) and the oracle: forward, backward, ragged and empty
experts, tails of fewer than 128 rows in a 256-row tile."""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64

pytestmark = pytest.mark.gpu


def _ffn(B, x_perm, offsets, W, flags):
    N, d = x_perm.shape
    E, f, _ = W[0].shape
    h = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    a = torch.empty_like(h)
    b = torch.empty_like(h)
    ws = B.workspace(B.grouped_ffn_ws_bytes(N, d, f, E))
    B.moe_grouped_ffn(x_perm, offsets, *W, h, out, ws, a_save=a, b_save=b,
                      flags=flags | B.MOE_CHECK)
    return h, out, a, b


@pytest.mark.parametrize("counts,d,f", [
    ([64, 100, 0, 300, 37, 1, 0, 10], 512, 1024),    # tails of 1..127 rows, empty experts
    ([256, 257, 511, 129], 1024, 384),               # 256-row tiles, 1-row and 129-row tails
    ([300, 0, 7], 200, 136),                         # d, f not multiples of 64 / 128
    ([1000], 256, 64),
])
def test_ffn_pairs_match_single_cta_and_oracle(lib, counts, d, f):
    E = len(counts)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    N = int(offsets[-1])
    g = torch.Generator().manual_seed(N + d + f)
    x_perm = torch.randn((N, d), generator=g).to(torch.bfloat16)
    W = [(torch.randn(s, generator=g) * 0.02).to(torch.bfloat16)
         for s in ((E, f, d), (E, f, d), (E, d, f))]
    dev = [t.cuda() for t in W]
    off = torch.from_numpy(offsets).cuda()
    pairs = _ffn(lib, x_perm.cuda(), off, dev, 0)
    single = _ffn(lib, x_perm.cuda(), off, dev, lib.MOE_SINGLE_CTA_TILES)
    torch.cuda.synchronize()
    ra, rb, rh, ro = O.expert_ffn(bits(x_perm), offsets, *(bits(w) for w in W))
    assert_close(f64(pairs[0]), rh, "h")
    assert_close(f64(pairs[1]), ro, "o")
    assert_close(f64(pairs[2]), O.bf16_round(ra), "a")
    assert_close(f64(pairs[3]), O.bf16_round(rb), "b")
    for p, s in zip(pairs, single):
        assert torch.equal(p.view(torch.int16), s.view(torch.int16))


def _fwd_bwd(B, wl, dev, flags):
    layer = B.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T)
    saved = B.Saved(layer, "cuda", train=True)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device="cuda")
    B.moe_layer_fwd(layer, dev["x"], y, saved, B.workspace(B.layer_fwd_ws_bytes(layer)),
                    flags=flags | B.MOE_CHECK)
    dx = torch.empty_like(dev["x"])
    dWg = torch.empty((wl.d, wl.E), dtype=torch.float32, device="cuda")
    dW1 = torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda")
    dW3 = torch.empty_like(dW1)
    dW2 = torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device="cuda")
    B.moe_layer_bwd(layer, dev["x"], saved, dev["g"], dx, dWg, dW1, dW3, dW2,
                    B.workspace(B.layer_bwd_ws_bytes(layer)), flags=flags | B.MOE_CHECK)
    torch.cuda.synchronize()
    return dict(y=y, h=saved.h, a=saved.a, b=saved.b, dx=dx, dWg=dWg, dW1=dW1, dW3=dW3, dW2=dW2)


@pytest.mark.parametrize("name,over", [("train", dict(T=512)), ("mid", dict(T=1024, f=448)),
                                       ("tiny", {})])
def test_layer_pairs_match_single_cta(lib, name, over):
    wl = synth.workload(name, **over)
    dev = {k: (v.cuda() if v is not None else None)
           for k, v in synth.layer_inputs(wl, with_grad=True).items()}
    p = _fwd_bwd(lib, wl, dev, 0)
    s = _fwd_bwd(lib, wl, dev, lib.MOE_SINGLE_CTA_TILES)
    for k in p:
        a, b = p[k], s[k]
        if a.dtype == torch.bfloat16:
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), k
        else:
            assert torch.equal(a, b), k
