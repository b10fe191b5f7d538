"""GPU parity: microscaled fp8 operands and the fp8 tensor-core grouped FFN.

Quantisation (moe_quantize_mx, moe_dispatch_mx) is compared with the oracle bit
for bit: codes and scales are exact functions of the bf16 inputs.  The grouped
FFN (moe_grouped_ffn_mx) is compared with the oracle's expert_ffn_mx on the
same codes and scales: h within the bar after dequantisation (the GPU decides
h's codes from fp32 accumulators, the oracle from float64 sums, so a code can
differ by one step where the two straddle a rounding boundary), o within the
bf16 bar.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64, near_tie_tokens, random_routing

pytestmark = pytest.mark.gpu


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _quantize(B, W):
    K = W.shape[-1]
    codes = torch.empty(W.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(W.shape[:-1] + (B.mx_scale_row_bytes(K),), dtype=torch.uint8, device="cuda")
    B.moe_quantize_mx(W, codes, scales)
    return codes, scales


@pytest.mark.parametrize("rows,K", [(7, 128), (300, 512), (64, 7168), (129, 1408)])
def test_quantize_mx_bit_exact(lib, rows, K):
    x = _bf16((rows, K), 1.0, rows + K)
    x = (x.float() * torch.exp(torch.linspace(-20, 20, rows))[:, None]).to(torch.bfloat16)
    x[rows // 2, 32:64] = 0                                # an all-zero block
    x[0, :32] = 0
    codes, scales = _quantize(lib, x.cuda())
    torch.cuda.synchronize()
    want_c, want_s = O.quantize_mx(bits(x))
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy()[:, : K // 32], want_s)


def test_dispatch_mx_bit_exact(lib):
    T, d, E, R = 1000, 1024, 64, 6
    idx_np, _ = random_routing(T, E, R, seed=3, skew=1.0)
    x = _bf16((T, d), 1.0, 4)
    N = T * R
    sk = lib.mx_scale_row_bytes(d)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               row_slot=torch.empty(N, dtype=torch.int32, device="cuda"),
               slot_row=torch.empty(N, dtype=torch.int32, device="cuda"))
    xq = torch.empty((N, d), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((N, sk), dtype=torch.uint8, device="cuda")
    ws = lib.workspace(lib.dispatch_ws_bytes(T, d, E, R))
    lib.moe_dispatch_mx(x.cuda(), torch.from_numpy(idx_np).cuda(), E, out["counts"], out["offsets"],
                        out["row_slot"], out["slot_row"], xq, xs, ws, flags=lib.MOE_CHECK)
    torch.cuda.synchronize()
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx_np, E)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["row_slot"].cpu().numpy(), row_slot)
    assert np.array_equal(out["slot_row"].cpu().numpy(), slot_row)
    qc, qs = O.quantize_mx(bits(x))
    tok = row_slot // R
    assert np.array_equal(xq.cpu().numpy(), qc[tok])
    assert np.array_equal(xs.cpu().numpy()[:, : d // 32], qs[tok])


def _host_mx(w):
    """The oracle's codes and scales of a bf16 tensor [..., K], quantised along K."""
    K = w.shape[-1]
    c, s = O.quantize_mx(bits(w).reshape(-1, K))
    return c.reshape(w.shape), s.reshape(w.shape[:-1] + (K // 32,))


def _assert_codes(dev, host, what):
    """The device's codes and (unpadded) scales equal the oracle's, bit for bit."""
    (dc, ds), (hc, hs) = dev, host
    assert np.array_equal(dc.cpu().numpy(), hc), f"{what}: codes"
    assert np.array_equal(ds.cpu().numpy()[..., : hs.shape[-1]], hs), f"{what}: scales"


def _ffn_mx_case(B, counts, d, f, seed, row_scale=False, flags=0):
    E = len(counts)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    N = int(offsets[-1])
    x = _bf16((N, d), 1.0, seed)
    W1, W3 = _bf16((E, f, d), 0.02, seed + 1), _bf16((E, f, d), 0.02, seed + 2)
    W2 = _bf16((E, d, f), 0.02, seed + 3)
    xq, xs = _quantize(B, x.cuda())
    q1, q3, q2 = (_quantize(B, w.cuda()) for w in (W1, W3, W2))
    out = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    hq = torch.empty((N, f), dtype=torch.uint8, device="cuda")
    hs = torch.zeros((N, B.mx_scale_row_bytes(f)), dtype=torch.uint8, device="cuda")
    rs = None
    if row_scale:
        rs = torch.rand(N, generator=torch.Generator().manual_seed(seed + 4)) + 0.25
    ws = B.workspace(B.grouped_ffn_mx_ws_bytes(N, d, f, E))
    B.moe_grouped_ffn_mx(xq, xs, torch.from_numpy(offsets).cuda(), *q1, *q3, *q2, out, ws,
                         hq=hq, hs=hs, row_scale=None if rs is None else rs.cuda(),
                         flags=flags | B.MOE_CHECK)
    torch.cuda.synchronize()
    # the oracle quantises the same bf16 inputs itself; the device's codes and
    # scales must equal its own, bit for bit
    hx, h1, h3, h2 = _host_mx(x), _host_mx(W1), _host_mx(W3), _host_mx(W2)
    for dev, host, what in (((xq, xs), hx, "x"), (q1, h1, "W1"), (q3, h3, "W3"), (q2, h2, "W2")):
        _assert_codes(dev, host, what)
    a, b, hv, rq, rsc, h, o = O.expert_ffn_mx(*hx, offsets, *h1, *h3, *h2,
                                              row_scale=None if rs is None else rs.numpy())
    npc = lambda t: t.cpu().numpy()
    got_h = O.dequantize_mx(npc(hq), npc(hs)[:, : f // 32])
    assert_close(got_h, h, "h (dequantised)")
    same = np.mean(npc(hq) == rq)
    assert same > 0.99, f"only {same:.4%} of h codes agree"
    assert_close(f64(out), o, "o")
    return out, hq, hs


@pytest.mark.parametrize("counts,d,f", [
    ([64, 100, 0, 300, 37, 1, 0, 10], 512, 1024),     # ragged, empty experts, tails
    ([128, 128], 256, 256),                            # exact tiles
    ([1000], 128, 128),                                # one expert, one k-block
    ([3, 130, 257, 129], 1024, 384),                   # partial groups of k-blocks
    ([200, 50], 2048, 1408),                           # mid's widths: f = 11 k-blocks
])
def test_grouped_ffn_mx_matches_oracle(lib, counts, d, f):
    _ffn_mx_case(lib, counts, d, f, seed=sum(counts) + d + f)


def test_grouped_ffn_mx_row_scale_and_repeatability(lib):
    o1 = _ffn_mx_case(lib, [70, 0, 250, 5], 512, 256, seed=9, row_scale=True)[0]
    o2 = _ffn_mx_case(lib, [70, 0, 250, 5], 512, 256, seed=9, row_scale=True)[0]
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_grouped_ffn_mx_large_shape_sampled_experts(lib):
    """The large workload's widths (d=7168, f=2048) on three experts' rows."""
    # (the quantiser itself is checked bit for bit at d = 7168 above)
    _ffn_mx_case(lib, [21, 0, 300, 133], 7168, 2048, seed=77)


@pytest.mark.parametrize("name,over", [("tiny", {}), ("mid", dict(T=1024)), ("large", dict(T=128, E=8))])
def test_layer_forward_mx(lib, name, over):
    """moe_layer_fwd with MOE_FP8_MX against the oracle's whole MX forward: its
    own routing, dispatch, quantisation of x and of the weights (the device's
    weight codes must equal its own), microscaled fp8 expert FFN and combine.
    Rows and tokens are compared where the two routings agree (near ties aside)."""
    from workloads import synth
    wl = synth.workload(name, **over)
    inp = synth.layer_inputs(wl)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    mxw = lib.MxWeights(dev["W1"], dev["W3"], dev["W2"])
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T, mx=mxw)
    saved = lib.Saved(layer, "cuda", train=False)
    y = torch.empty_like(dev["x"])
    flags = lib.MOE_FP8_MX
    lib.moe_layer_fwd(layer, dev["x"], y, saved, lib.workspace(lib.layer_fwd_ws_bytes(layer, flags)),
                      flags=flags | lib.MOE_CHECK)
    torch.cuda.synchronize()
    h1, h3, h2 = _host_mx(inp["W1"]), _host_mx(inp["W3"]), _host_mx(inp["W2"])
    for dev_q, host, what in (((mxw.W1q, mxw.W1s), h1, "W1"), ((mxw.W3q, mxw.W3s), h3, "W3"),
                              ((mxw.W2q, mxw.W2s), h2, "W2")):
        _assert_codes(dev_q, host, what)
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    logits = O.gate_logits(bits(inp["x"]), inp["w_gate"].numpy(), bias)
    idx, w = O.route_topk(logits, wl.R)
    gidx = saved.topk_idx.cpu().numpy()
    same = (gidx == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, wl.R)).all(), "routing differs without a near tie"
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
    xq, xs = O.quantize_mx(bits(inp["x"]))
    tok = row_slot // wl.R
    *_, o = O.expert_ffn_mx(xq[tok], xs[tok], offsets, *h1, *h3, *h2)
    yr = O.combine(o, slot_row, w, wl.T, wl.R)
    # a row's o depends only on its token and expert: every row of every token routed alike
    gsr = saved.slot_row.cpu().numpy().reshape(wl.T, wl.R)[same].reshape(-1)
    rsr = slot_row.reshape(wl.T, wl.R)[same].reshape(-1)
    assert_close(f64(saved.o)[gsr], o[rsr], "o (rows of tokens routed alike)")
    assert_close(f64(y)[same], yr[same], "y (tokens routed alike)")


def test_layer_forward_mx_full_size_sampled_experts(lib):
    """The large workload (T=8192, d=7168, E=384, R=8, f=2048) as bench.py times it
    with the microscaled fp8 FFN: weights quantised once on the device, then
    moe_layer_fwd with MOE_FP8_MX.  The oracle recomputes every row of three
    experts (the fewest rows, the most, one drawn at random) from its own
    routing and its own quantisation of x and of those experts' weights."""
    from workloads import synth
    wl = synth.workload("large")
    inp = synth.layer_inputs(wl, device="cuda")
    mxw = lib.MxWeights(inp["W1"], inp["W3"], inp["W2"])
    layer = lib.Layer(inp["w_gate"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], wl.R, wl.T,
                      mx=mxw)
    saved = lib.Saved(layer, "cuda", train=False)
    y = torch.empty_like(inp["x"])
    flags = lib.MOE_FP8_MX
    lib.moe_layer_fwd(layer, inp["x"], y, saved, lib.workspace(lib.layer_fwd_ws_bytes(layer, flags)),
                      flags=flags | lib.MOE_CHECK)
    torch.cuda.synchronize()
    xb = bits(inp["x"])
    logits = O.gate_logits(xb, inp["w_gate"].cpu().numpy(), None)
    idx, _ = O.route_topk(logits, wl.R)
    gidx = saved.topk_idx.cpu().numpy()
    same = (gidx == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, wl.R)).all()
    counts = np.bincount(idx[same].reshape(-1), minlength=wl.E)
    live = np.nonzero(counts)[0]
    rng = np.random.default_rng(5)
    experts = sorted({int(live[np.argmin(counts[live])]), int(np.argmax(counts)),
                      int(rng.choice(live))})
    dev_slot_row = saved.slot_row.cpu().numpy().reshape(wl.T, wl.R)
    for e in experts:
        t_e, r_e = np.nonzero((idx == e) & same[:, None])       # the expert's tokens, ascending
        host = [O.quantize_mx(bits(inp[k][e])) for k in ("W1", "W3", "W2")]
        for (c, sc), (dq, ds), what in zip(host, ((mxw.W1q, mxw.W1s), (mxw.W3q, mxw.W3s),
                                                  (mxw.W2q, mxw.W2s)), ("W1", "W3", "W2")):
            _assert_codes((dq[e], ds[e]), (c, sc), f"{what}[{e}]")
        xq, xs = O.quantize_mx(xb[t_e])
        *_, o = O.expert_ffn_mx(xq, xs, np.array([0, len(t_e)]),
                                *(a[None] for pair in host for a in pair))
        rows = torch.from_numpy(dev_slot_row[t_e, r_e]).long().cuda()
        assert_close(f64(saved.o[rows]), o, f"o rows of expert {e} ({len(t_e)} rows)")


@pytest.mark.parametrize("serial", [False, True])
def test_layer_forward_mx_with_shared_expert(lib, serial):
    """MOE_FP8_MX with a shared expert: the routed experts on the fp8 tensor cores,
    the shared one in bf16 (on the side stream, or serially), added with weight 1
    before y's rounding -- against the oracle's shared expert plus its MX routed
    path, on the tokens routed alike; side stream and serial give the same bits."""
    from workloads import synth
    wl = synth.workload("tiny", T=200)
    fs = 256
    inp = synth.layer_inputs(wl)
    sw = synth.shared_expert_inputs(wl, fs)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    shared = lib.Shared(*(sw[k].cuda() for k in ("W1", "W3", "W2")))
    mxw = lib.MxWeights(dev["W1"], dev["W3"], dev["W2"])
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], wl.R, wl.T,
                      shared=shared, mx=mxw)
    flags = lib.MOE_FP8_MX | (lib.MOE_SHARED_SERIAL if serial else 0)
    ys = []
    for fl in (flags, flags ^ lib.MOE_SHARED_SERIAL):
        saved = lib.Saved(layer, "cuda", train=False)
        y = torch.empty_like(dev["x"])
        lib.moe_layer_fwd(layer, dev["x"], y, saved,
                          lib.workspace(lib.layer_fwd_ws_bytes(layer, fl)), flags=fl | lib.MOE_CHECK)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    y = ys[0]
    h1, h3, h2 = _host_mx(inp["W1"]), _host_mx(inp["W3"]), _host_mx(inp["W2"])
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    logits = O.gate_logits(bits(inp["x"]), inp["w_gate"].numpy(), bias)
    idx, w = O.route_topk(logits, wl.R)
    same = (saved.topk_idx.cpu().numpy() == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, wl.R)).all(), "routing differs without a near tie"
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
    xq, xs = O.quantize_mx(bits(inp["x"]))
    tok = row_slot // wl.R
    *_, o = O.expert_ffn_mx(xq[tok], xs[tok], offsets, *h1, *h3, *h2)
    s_out = O.shared_expert_fwd(bits(inp["x"]), bits(sw["W1"]), bits(sw["W3"]), bits(sw["W2"]))[3]
    yr = O.combine(o, slot_row, w, wl.T, wl.R, add=s_out)
    assert_close(f64(y)[same], yr[same], "y (routed MX + shared bf16, tokens routed alike)")
