"""GPU parity: router, dispatch and combine against the CPU oracle."""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64, near_tie_tokens, random_routing

pytestmark = pytest.mark.gpu


def _route(B, x, wg, bias, T, E, R, logits_in=None):
    logits = (logits_in.clone() if logits_in is not None
              else torch.empty((T, E), dtype=torch.float32, device="cuda"))
    idx = torch.empty((T, R), dtype=torch.int32, device="cuda")
    w = torch.empty((T, R), dtype=torch.float32, device="cuda")
    if logits_in is not None:
        B.moe_route(None, None, None, logits, idx, w, flags=B.MOE_LOGITS_IN)
    else:
        ws = B.workspace(B.route_ws_bytes(T, x.shape[1], E, R))
        B.moe_route(x, wg, bias, logits, idx, w, ws=ws, flags=B.MOE_CHECK)
    torch.cuda.synchronize()
    return logits, idx, w


@pytest.mark.parametrize("name", ["tiny", "mid", "large", "train"])
def test_route_end_to_end(lib, name):
    wl = synth.workload(name)
    x, wg, bias = synth.router_inputs(wl)
    ref_l = O.gate_logits(bits(x), wg.numpy(), None if bias is None else bias.numpy())
    logits, idx, w = _route(lib, x.cuda(), wg.cuda(), None if bias is None else bias.cuda(),
                            wl.T, wl.E, wl.R)
    # fp32 sums of d products against float64 sums: ~sqrt(d) * 2^-24 relative
    assert_close(f64(logits), ref_l, "logits", max_rel=3e-5, mean_rel=1e-5)
    ridx, rw = O.route_topk(ref_l, wl.R)
    tie = near_tie_tokens(ref_l, wl.R)
    mism = (idx.cpu().numpy() != ridx).any(axis=1)
    assert not (mism & ~tie).any(), f"{(mism & ~tie).sum()} tokens routed differently"
    ok = ~mism
    # the weights inherit the ~1e-6 relative differences of the two logit sums
    np.testing.assert_allclose(f64(w)[ok], rw[ok], rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("name", ["tiny", "mid", "large"])
def test_route_logits_in_is_bit_exact(lib, name):
    wl = synth.workload(name)
    x, wg, bias = synth.router_inputs(wl)
    ref_l = O.gate_logits(bits(x), wg.numpy(), None if bias is None else bias.numpy())
    _, idx, w = _route(lib, None, None, None, wl.T, wl.E, wl.R,
                       logits_in=torch.from_numpy(ref_l).cuda())
    ridx, rw = O.route_topk(ref_l, wl.R)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(f64(w), rw, rtol=2e-6, atol=2e-7)


@pytest.mark.parametrize("T,E,R", [(1000, 8, 2), (777, 64, 6), (300, 384, 8), (64, 1024, 32),
                                   (50, 33, 32), (5, 1, 1)])
def test_route_ties_and_edge_shapes(lib, T, E, R):
    g = np.random.default_rng(T + E + R)
    ref_l = g.integers(-2, 3, (T, E)).astype(np.float32)       # dense exact ties
    _, idx, w = _route(lib, None, None, None, T, E, R, logits_in=torch.from_numpy(ref_l).cuda())
    ridx, rw = O.route_topk(ref_l, R)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(f64(w), rw, rtol=2e-6, atol=2e-7)


def _dispatch(B, x, idx, E):
    T, R = idx.shape
    d = x.shape[1]
    N = T * R
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               row_slot=torch.empty(N, dtype=torch.int32, device="cuda"),
               slot_row=torch.empty(N, dtype=torch.int32, device="cuda"),
               x_perm=torch.empty((N, d), dtype=torch.bfloat16, device="cuda"))
    ws = B.workspace(B.dispatch_ws_bytes(T, d, E, R))
    B.moe_dispatch(x, idx, E, out["counts"], out["offsets"], out["row_slot"], out["slot_row"],
                   out["x_perm"], ws, flags=B.MOE_CHECK)
    return out


@pytest.mark.parametrize("T,d,E,R,skew", [(256, 512, 8, 2, 0.0), (1000, 136, 64, 6, 1.0),
                                          (4096, 2048, 64, 6, 1.0), (1, 64, 4, 4, 0.0),
                                          (3000, 64, 1024, 32, 1.2), (513, 64, 256, 8, 1.2)])
def test_dispatch_bit_exact(lib, T, d, E, R, skew):
    idx, _ = random_routing(T, E, R, seed=T * 7 + E, skew=skew)
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    out = _dispatch(lib, x.cuda(), torch.from_numpy(idx).cuda(), E)
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx, E)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["row_slot"].cpu().numpy(), row_slot)
    assert np.array_equal(out["slot_row"].cpu().numpy(), slot_row)
    assert np.array_equal(bits(out["x_perm"]), O.permute_rows(bits(x), row_slot, R))


@pytest.mark.parametrize("name,T", [("dispatch", 128), ("dispatch", 8192), ("dispatch_zipf", 8192),
                                    ("dispatch_zipf", 65536), ("dispatch", 65536)])
def test_dispatch_full_size_and_roundtrip(lib, name, T):
    wl = synth.workload(name, T=T)
    r = synth.drawn_routing(wl)
    idx = r["topk_idx"].numpy()
    x = r["x"].cuda()
    out = _dispatch(lib, x, r["topk_idx"].cuda(), wl.E)
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["row_slot"].cpu().numpy(), row_slot)
    assert np.array_equal(out["slot_row"].cpu().numpy(), slot_row)
    assert int(out["counts"].sum()) == T * wl.R
    # x_perm[row] == x[row_slot[row] / R] at any size (checked on the device, exact)
    src = torch.from_numpy(row_slot // wl.R).long().cuda()
    assert torch.equal(out["x_perm"].view(torch.int16), x.view(torch.int16)[src])
    # identity experts: combine(dispatch(x)) == x exactly (the gate weights sum to 1)
    y = torch.empty_like(x)
    lib.moe_combine(out["x_perm"], out["slot_row"], r["topk_w"].cuda(), y, wl.R)
    torch.cuda.synchronize()
    assert torch.equal(y.float(), x.float())


def test_dispatch_rejects_bad_routing(lib):
    T, E, R, d = 64, 8, 2, 64
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor(np.tile([0, 1], (T, 1)), dtype=torch.int32, device="cuda")
    idx[5, 1] = E           # out of range
    with pytest.raises(lib.MoeError) as ei:
        _dispatch(lib, x, idx, E)
    assert ei.value.status == 4
    idx[5, 1] = 0           # repeated within a token
    with pytest.raises(lib.MoeError) as ei:
        _dispatch(lib, x, idx, E)
    assert ei.value.status == 4
    idx[5, 1] = 1
    _dispatch(lib, x, idx, E)   # valid again: no error left over


@pytest.mark.parametrize("T,d,R,weighted", [(300, 512, 2, True), (77, 7168, 8, True),
                                            (1000, 64, 32, True), (64, 128, 3, False)])
def test_combine_matches_oracle(lib, T, d, R, weighted):
    g = np.random.default_rng(T + d)
    N = T * R
    o = torch.randn((N, d), generator=torch.Generator().manual_seed(d)).to(torch.bfloat16)
    slot_row = g.permutation(N).astype(np.int32)
    u = g.random((T, R)) + 0.5
    w = (u / u.sum(1, keepdims=True)).astype(np.float32)
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    wt = torch.from_numpy(w).cuda() if weighted else None
    lib.moe_combine(o.cuda(), torch.from_numpy(slot_row).cuda(), wt, y, R)
    ref = O.combine(f64(o), slot_row, w if weighted else None, T, R)
    assert_close(f64(y), ref, "y")
    y2 = torch.empty_like(y)
    lib.moe_combine(o.cuda(), torch.from_numpy(slot_row).cuda(), wt, y2, R)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))     # bitwise reproducible


@pytest.mark.parametrize("T,d,E,R", [(500, 200, 64, 6), (129, 8, 3, 2), (300, 1024, 1000, 8)])
def test_route_gate_paths(lib, T, d, E, R):
    # d % 64 != 0 runs the fp32 FMA projection; d % 64 == 0 the split-bf16 tensor-core one
    g = torch.Generator().manual_seed(T + d)
    x = torch.randn((T, d), generator=g).to(torch.bfloat16)
    wg = torch.randn((d, E), generator=g) * 0.05
    bias = torch.randn((E,), generator=g)
    ref_l = O.gate_logits(bits(x), wg.numpy(), bias.numpy())
    logits, idx, w = _route(lib, x.cuda(), wg.cuda(), bias.cuda(), T, E, R)
    assert_close(f64(logits), ref_l, "logits", max_rel=3e-5, mean_rel=1e-5)
    ridx, _ = O.route_topk(ref_l, R)
    same = (idx.cpu().numpy() == ridx).all(axis=1)
    assert (same | near_tie_tokens(ref_l, R)).all()


@pytest.mark.parametrize("d,E", [(2048, 64), (512, 200)])
def test_gate_split_over_ctas_same_bits(lib, d, E):
    """With few 128-token tiles the gate splits each tile's K over four CTAs (one
    per partial accumulator) and adds the partials in a second kernel; a token's
    logits must be the same bits as when its tile runs on one CTA (a larger T)."""
    g = torch.Generator().manual_seed(d + E)
    x = torch.randn((8192, d), generator=g).to(torch.bfloat16)
    wg = torch.randn((d, E), generator=g) * 0.02
    bias = torch.randn(E, generator=g)
    small, _, _ = _route(lib, x[:1024].cuda(), wg.cuda(), bias.cuda(), 1024, E, 2)   # split
    big, _, _ = _route(lib, x.cuda(), wg.cuda(), bias.cuda(), 8192, E, 2)            # one CTA
    assert torch.equal(small, big[:1024])
    ref = O.gate_logits(bits(x[:1024]), wg.numpy(), bias.numpy())
    assert_close(f64(small), ref, "logits", max_rel=3e-5, mean_rel=1e-5)
