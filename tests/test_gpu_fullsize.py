"""GPU parity at full workload sizes, in the launch configuration bench.py times.

The GPU runs the whole layer (forward, and backward for training) on the full
workload; the oracle then recomputes, on its own routing, outputs it can afford
one by one: a sample of tokens (their y, and dx for training) and every row of
a few experts (their weight gradients).  A token's outputs depend only on its
own routing and an expert's weight gradients only on the tokens routed to it,
so running the oracle's layer on that subset of tokens gives exact references.
"""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import LazyExperts, assert_close, bits, f64, near_tie_tokens

pytestmark = pytest.mark.gpu


def _gpu_layer(B, wl, train, prepacked=False):
    inp = synth.layer_inputs(wl, device="cuda")          # as bench.py: weights drawn on the GPU
    layer = B.Layer(inp["w_gate"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], wl.R, wl.T)
    packed_y = None
    if prepacked:   # bench.py streams prepacked tiles in forward-only workloads: same bits
        P = [torch.empty_like(inp[k]) for k in ("W1", "W3", "W2")]
        B.moe_prepack_weights(inp["W1"], inp["W3"], inp["W2"], *P)
        pl = B.Layer(inp["w_gate"], inp["bias"], *P, wl.R, wl.T)
        packed_y = torch.empty_like(inp["x"])
        B.moe_layer_fwd(pl, inp["x"], packed_y, B.Saved(pl, "cuda", train=False),
                        B.workspace(B.layer_fwd_ws_bytes(pl)),
                        flags=B.MOE_CHECK | B.MOE_WEIGHTS_PREPACKED)
        del P, pl
    saved = B.Saved(layer, "cuda", train=train)
    y = torch.empty_like(inp["x"])
    B.moe_layer_fwd(layer, inp["x"], y, saved, B.workspace(B.layer_fwd_ws_bytes(layer)),
                    flags=B.MOE_CHECK)
    out = {"inp": inp, "saved": saved, "y": y, "packed_y": packed_y}
    if train:
        dx = torch.empty_like(inp["x"])
        dWg = torch.empty((wl.d, wl.E), dtype=torch.float32, device="cuda")
        dW1 = torch.empty((wl.E, wl.f, wl.d), dtype=torch.float32, device="cuda")
        dW3 = torch.empty_like(dW1)
        dW2 = torch.empty((wl.E, wl.d, wl.f), dtype=torch.float32, device="cuda")
        B.moe_layer_bwd(layer, inp["x"], saved, inp["g"], dx, dWg, dW1, dW3, dW2,
                        B.workspace(B.layer_bwd_ws_bytes(layer)), flags=B.MOE_CHECK)
        out.update(dx=dx, dWg=dWg, dW1=dW1, dW3=dW3, dW2=dW2)
    torch.cuda.synchronize()
    return out


def _oracle_routing(inp, wl):
    bias = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    logits = O.gate_logits(bits(inp["x"]), inp["w_gate"].cpu().numpy(), bias)
    idx, w = O.route_topk(logits, wl.R)
    return logits, idx, w, bias


def _oracle_subset(inp, wl, toks, bias, train):
    x = bits(inp["x"])[toks]
    W = [LazyExperts(inp[k]) for k in ("W1", "W3", "W2")]
    wg = inp["w_gate"].cpu().numpy()
    fw = O.layer_fwd(x, wg, bias, *W, wl.R)
    bw = O.layer_bwd(fw, x, wg, *W, bits(inp["g"])[toks], wl.R) if train else None
    return fw, bw


def _tokens_covering_every_expert(gidx, same, E, seed):
    """Tokens routed alike on both sides such that every expert with rows has at
    least one of them (greedy: for each expert not yet covered, a random token
    routed to it), plus a few random ones."""
    rng = np.random.default_rng(seed)
    covered = np.zeros(E, dtype=bool)
    toks = set(rng.choice(np.nonzero(same)[0], 8, replace=False).tolist())
    for t in toks:
        covered[gidx[t]] = True
    for e in np.unique(gidx):
        if covered[e]:
            continue
        cand = np.nonzero(same & (gidx == e).any(axis=1))[0]
        if cand.size == 0:
            continue                                  # every row of e has a near tie
        t = int(rng.choice(cand))
        toks.add(t)
        covered[gidx[t]] = True
    return np.array(sorted(toks)), covered


@pytest.mark.parametrize("name", ["large", "large_hot", "train"])
def test_forward_full_size_sampled_tokens(lib, name):
    wl = synth.workload(name)
    run = _gpu_layer(lib, wl, train=False, prepacked=name != "train")
    if run["packed_y"] is not None:
        assert torch.equal(run["packed_y"].view(torch.int16), run["y"].view(torch.int16))
    logits, idx, w, bias = _oracle_routing(run["inp"], wl)
    gidx = run["saved"].topk_idx.cpu().numpy()
    same = (gidx == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, wl.R)).all()
    toks, covered = _tokens_covering_every_expert(gidx, same, wl.E, seed=1)
    counts = run["saved"].counts.cpu().numpy()
    assert covered[counts > 0].mean() > 0.99           # (only an all-tie expert may be missed)
    fw, _ = _oracle_subset(run["inp"], wl, toks, bias, train=False)
    assert np.array_equal(fw["idx"], gidx[toks])
    assert_close(f64(run["y"][torch.from_numpy(toks).cuda()]), fw["y"], "y (sampled tokens)")
    rows = run["saved"].slot_row.cpu().numpy().reshape(wl.T, wl.R)[toks].reshape(-1)
    ref_rows = fw["slot_row"]                       # oracle's rows for the subset, same slot order
    sel = torch.from_numpy(rows).long().cuda()
    # every expert with rows contributes at least one row to each comparison (the
    # tensor-wide bar: max and mean), and each expert's rows are held to the
    # max bar on their own (a mean over one or two rows of one expert is a
    # noisier statistic than the bar is stated for)
    assert_close(f64(run["saved"].h[sel]), fw["h"][ref_rows], "h (sampled rows)")
    assert_close(f64(run["saved"].o[sel]), fw["o"][ref_rows], "o (sampled rows)")
    ex = gidx[toks].reshape(-1)
    gh, go = f64(run["saved"].h[sel]), f64(run["saved"].o[sel])
    for e in np.unique(ex):
        m = ex == e
        assert_close(gh[m], fw["h"][ref_rows][m], f"h rows of expert {e}", mean_rel=1.0)
        assert_close(go[m], fw["o"][ref_rows][m], f"o rows of expert {e}", mean_rel=1.0)


def test_train_backward_full_size_sampled(lib):
    wl = synth.workload("train")
    run = _gpu_layer(lib, wl, train=True)
    logits, idx, w, bias = _oracle_routing(run["inp"], wl)
    gidx = run["saved"].topk_idx.cpu().numpy()
    same = (gidx == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, wl.R)).all()
    # dx of sampled tokens
    toks = np.sort(np.random.default_rng(2).choice(np.nonzero(same)[0], 6, replace=False))
    _, bw = _oracle_subset(run["inp"], wl, toks, bias, train=True)
    assert_close(f64(run["dx"][torch.from_numpy(toks).cuda()]), bw["dx"], "dx (sampled tokens)")
    # every weight gradient of the experts with the fewest and the most rows
    counts = np.bincount(idx.reshape(-1), minlength=wl.E)
    for e in (int(np.argmin(counts)), int(np.argmax(counts))):
        toks_e = np.nonzero((idx == e).any(axis=1))[0]
        if not same[toks_e].all():
            continue                                  # a near tie moved a row of this expert
        _, bw = _oracle_subset(run["inp"], wl, toks_e, bias, train=True)
        assert_close(f64(run["dW1"][e]), bw["dW1"][e], f"dW1[{e}]")
        assert_close(f64(run["dW3"][e]), bw["dW3"][e], f"dW3[{e}]")
        assert_close(f64(run["dW2"][e]), bw["dW2"][e], f"dW2[{e}]")
        assert_close(f64(run["dWg"][:, e]), bw["dW_gate"][:, e], f"dW_gate[:, {e}]")
