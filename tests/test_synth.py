"""CPU tests of the seeded input recipe (expert_moe_route_gb300/synth.py) that
both the CUDA path and the oracle are fed from: the workload sizes, seeding,
the value distributions and the router variants as stated in its docstring."""
import json
import math
import os

import numpy as np
import pytest
import torch

from workloads import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_workload_sizes():
    sizes = {n: (w.T, w.d, w.E, w.R, w.f) for n, w in synth.WORKLOADS.items()}
    assert sizes["tiny"] == (256, 512, 8, 2, 1024)
    assert sizes["mid"] == (4096, 2048, 64, 6, 1408)
    assert sizes["large"] == sizes["large_hot"] == (8192, 7168, 384, 8, 2048)
    assert sizes["dispatch"] == sizes["dispatch_zipf"] == (8192, 7168, 256, 8, 0)
    assert sizes["train"] == (16384, 4096, 128, 8, 1536)
    assert synth.WORKLOADS["train"].train and not synth.WORKLOADS["large"].train
    assert synth.DISPATCH_T_SWEEP[0] == 128 and synth.DISPATCH_T_SWEEP[-1] == 65536
    assert synth.workload("train", T=512).T == 512 and synth.WORKLOADS["train"].T == 16384


def test_inputs_are_reproducible_and_independent_per_tensor():
    wl = synth.workload("tiny")
    a, b = synth.layer_inputs(wl, with_grad=True), synth.layer_inputs(wl, with_grad=True)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k
    # each tensor has its own seed: a smaller T leaves the weights unchanged
    c = synth.layer_inputs(synth.workload("tiny", T=16))
    assert torch.equal(c["W1"], a["W1"]) and torch.equal(c["x"], a["x"][:16])
    assert not torch.equal(a["W1"], a["W3"])
    # another workload index gives other values
    m = synth.router_inputs(synth.workload("mid", T=16, d=512))[0]
    assert not torch.equal(m, a["x"][:16])


def test_value_distributions():
    wl = synth.workload("tiny")
    inp = synth.layer_inputs(wl, with_grad=True)
    for k, std in (("x", 1.0), ("g", 1.0), ("W1", 0.02), ("W3", 0.02), ("W2", 0.02)):
        v = inp[k].double()
        assert inp[k].dtype == torch.bfloat16
        assert abs(v.mean().item()) < 0.05 * std, k
        assert v.std().item() == pytest.approx(std, rel=0.01), k
    assert inp["w_gate"].dtype == torch.float32
    assert inp["w_gate"].std().item() == pytest.approx(0.02, rel=0.05)
    assert inp["bias"] is None
    sw = synth.shared_expert_inputs(wl, 256)
    assert sw["W1"].shape == (256, wl.d) and sw["W2"].shape == (wl.d, 256)
    assert sw["W1"].double().std().item() == pytest.approx(0.02, rel=0.02)
    assert not torch.equal(sw["W1"][:8], inp["W1"][0, :8])


def test_zipf_router_bias():
    wl = synth.workload("mid")
    b = synth.router_bias(wl).double()
    off = b == -30.0
    assert off.sum().item() == wl.E // 8
    ranks = torch.exp(-b[~off] / wl.zipf_s)            # k_e = exp(-b_e / s)
    assert torch.allclose(torch.sort(ranks).values,
                          torch.arange(1, wl.E - wl.E // 8 + 1, dtype=torch.float64), rtol=1e-6)


def test_hot_router_bias():
    wl = synth.workload("large_hot")
    b = synth.router_bias(wl)
    with open(os.path.join(ROOT, "tests", "golden", "hot_bias.json")) as fh:
        beta = json.load(fh)["large_hot"]["beta"]
    hot = torch.nonzero(b).flatten()
    assert len(hot) == wl.hot_experts
    assert torch.equal(torch.sort(hot).values, torch.sort(synth.hot_experts(wl)).values)
    assert (b[hot] == np.float32(beta)).all()
    assert synth.router_bias(synth.workload("large")) is None


def test_hot_bias_gives_a_quarter_of_the_assignments():
    # the share the stored bias was bisected for, on the seeded x and W_g
    wl = synth.workload("large_hot")
    x, wg, b = synth.router_inputs(wl)
    logits = x.float() @ wg + b
    idx = torch.topk(logits, wl.R, dim=1).indices
    share = torch.isin(idx, synth.hot_experts(wl)).float().mean().item()
    assert share == pytest.approx(0.25, abs=0.005)


@pytest.mark.parametrize("name", ["dispatch", "dispatch_zipf"])
def test_drawn_routing(name):
    wl = synth.workload(name, T=4096)
    r = synth.drawn_routing(wl)
    idx, w = r["topk_idx"], r["topk_w"]
    assert idx.dtype == torch.int32 and idx.shape == (wl.T, wl.R)
    assert ((idx >= 0) & (idx < wl.E)).all()
    srt = torch.sort(idx, dim=1).values
    assert (srt[:, 1:] != srt[:, :-1]).all()                 # R distinct experts per token
    assert (w > 0).all() and torch.allclose(w.double().sum(1), torch.ones(wl.T, dtype=torch.float64),
                                            atol=1e-6)
    counts = torch.bincount(idx.flatten().long(), minlength=wl.E).double()
    mean = wl.T * wl.R / wl.E
    if wl.zipf_s == 0:
        # uniform: every expert near T*R/E (multinomial spread, a few sigma)
        assert (counts - mean).abs().max().item() < 6 * math.sqrt(mean)
    else:
        # Zipf: the counts fall with the seeded rank k
        g = synth._gen("cpu", wl.index * 1000 + synth._ROUTE)   # the routing tensor's seed
        k = torch.randperm(wl.E, generator=g) + 1
        top, bottom = counts[k <= 8].mean().item(), counts[k > wl.E - 64].mean().item()
        assert top > 4 * bottom
