"""GPU: the weight-gradient GEMMs (dW1, dW3, dW2) at every kind of ragged end.

The weight gradients contract over each expert's rows, so an expert whose
rows end inside a 64-row k-block loads that last block through tensor maps
cut at its last row, and the rows of the next expert arrive as zeros.  Here
the router is built so that each expert gets a chosen number of rows (one-hot
logits, top-1), covering ends inside and on the 16-row groups the tensor core
consumes, single rows, empty experts between full ones and long experts, and
the gradients are compared with the oracle and between CTA pairs and single
CTAs bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64

pytestmark = pytest.mark.gpu

COUNTS = [1, 15, 16, 17, 0, 63, 64, 65, 127, 0, 0, 128, 129, 300, 2, 33]


def _inputs(counts, d, f, seed):
    E = len(counts)
    T = int(sum(counts))
    expert = np.repeat(np.arange(E), counts)
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(T, generator=g).numpy()
    expert = expert[perm]                       # tokens of an expert spread over the batch
    x = torch.randn((T, d), generator=g)
    x[:, :E] = 0.0
    x[np.arange(T), expert] = 8.0               # logits: 8 for the token's expert, 0 elsewhere
    w_gate = torch.zeros((d, E), dtype=torch.float32)
    w_gate[np.arange(E), np.arange(E)] = 1.0
    W = [(torch.randn(s, generator=g) * 0.02).to(torch.bfloat16)
         for s in ((E, f, d), (E, f, d), (E, d, f))]
    dy = torch.randn((T, d), generator=g).to(torch.bfloat16)
    return dict(x=x.to(torch.bfloat16), w_gate=w_gate, W1=W[0], W3=W[1], W2=W[2], g=dy), expert


def _run(B, inp, R, flags):
    dev = {k: v.cuda() for k, v in inp.items()}
    T, d = inp["x"].shape
    E, f, _ = inp["W1"].shape
    layer = B.Layer(dev["w_gate"], None, dev["W1"], dev["W3"], dev["W2"], R, T)
    saved = B.Saved(layer, "cuda", train=True)
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    B.moe_layer_fwd(layer, dev["x"], y, saved, B.workspace(B.layer_fwd_ws_bytes(layer)),
                    flags=flags | B.MOE_CHECK)
    dx = torch.empty_like(dev["x"])
    dWg = torch.empty((d, E), dtype=torch.float32, device="cuda")
    dW1 = torch.full((E, f, d), float("nan"), dtype=torch.float32, device="cuda")
    dW3 = torch.full_like(dW1, float("nan"))
    dW2 = torch.full((E, d, f), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_layer_bwd(layer, dev["x"], saved, dev["g"], dx, dWg, dW1, dW3, dW2,
                    B.workspace(B.layer_bwd_ws_bytes(layer)), flags=flags | B.MOE_CHECK)
    torch.cuda.synchronize()
    return saved, dict(dx=dx, dW1=dW1, dW3=dW3, dW2=dW2)


@pytest.mark.parametrize("d,f", [(256, 128), (512, 192)])
def test_weight_gradients_at_ragged_expert_ends(lib, d, f):
    inp, expert = _inputs(COUNTS, d, f, seed=d + f)
    saved, got = _run(lib, inp, 1, 0)
    assert np.array_equal(saved.topk_idx.cpu().numpy()[:, 0], expert)
    assert np.array_equal(saved.counts.cpu().numpy(), np.asarray(COUNTS))
    ref = O.layer_fwd(bits(inp["x"]), inp["w_gate"].numpy(), None, bits(inp["W1"]),
                      bits(inp["W3"]), bits(inp["W2"]), 1)
    rb = O.layer_bwd(ref, bits(inp["x"]), inp["w_gate"].numpy(), bits(inp["W1"]),
                     bits(inp["W3"]), bits(inp["W2"]), bits(inp["g"]), 1)
    for k in ("dW1", "dW3", "dW2"):
        assert torch.isfinite(got[k]).all(), k   # every expert's gradient was written
        for e, c in enumerate(COUNTS):           # per expert, so a wrong tail cannot hide
            if c == 0:
                assert not got[k][e].any(), (k, e)
            else:
                assert_close(f64(got[k][e]), rb[k][e], f"{k}[{e}] ({c} rows)")
    assert_close(f64(got["dx"]), rb["dx"], "dx")
    _, single = _run(lib, inp, 1, lib.MOE_SINGLE_CTA_TILES)
    for k in got:
        a, b = got[k], single[k]
        if a.dtype == torch.bfloat16:
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), k
        else:
            assert torch.equal(a, b), k
