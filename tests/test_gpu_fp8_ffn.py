"""GPU parity: the grouped SwiGLU FFN on block-scaled fp8 rows
(moe_grouped_ffn_fp8, which dequantises the rows once into its workspace and
runs the bf16 grouped FFN).  Every output must equal, bit for bit,
moe_dequant_fp8 followed by moe_grouped_ffn with caller buffers, and match the
oracle's FFN on the oracle's dequantised rows within the layer's tolerance."""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64, near_tie_tokens, random_routing

pytestmark = pytest.mark.gpu


def _bf16(shape, std, seed):
    return (torch.randn(shape, generator=torch.Generator().manual_seed(seed)) * std).to(torch.bfloat16)


def _fp8_rows(N, d, seed):
    """Block-scaled fp8 rows as the fp8 dispatch writes them: the oracle's
    quantiser applied to seeded bf16 rows whose magnitudes span 2^4."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((N, d), generator=g) * torch.exp(torch.rand((N, 1), generator=g) * 4.0 - 2.0)
    if N > 0:
        x[0, :128] = 0.0                     # an all-zero block: scale 0
    codes, scales = O.quantize_fp8_blocks(bits(x.to(torch.bfloat16)))
    return codes, scales


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _both_paths(B, xq, xs, offsets, W1, W3, W2, flags, row_scale=None, save=True):
    """(fp8 GEMM outputs, dequantise-then-bf16 GEMM outputs), each h, out, a, b."""
    N, d = xq.shape
    E, f, _ = W1.shape
    ws = B.workspace(B.grouped_ffn_fp8_ws_bytes(N, d, f, E))

    def bufs():
        a = torch.empty((N, f), dtype=torch.bfloat16, device="cuda") if save else None
        b = torch.empty((N, f), dtype=torch.bfloat16, device="cuda") if save else None
        return dict(h=torch.empty((N, f), dtype=torch.bfloat16, device="cuda"),
                    out=torch.empty((N, d), dtype=torch.bfloat16, device="cuda"), a=a, b=b)

    got = bufs()
    B.moe_grouped_ffn_fp8(xq, xs, offsets, W1, W3, W2, got["h"], got["out"], ws, a_save=got["a"],
                          b_save=got["b"], flags=flags | B.MOE_CHECK, row_scale=row_scale)
    xd = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    B.moe_dequant_fp8(xq, xs, xd)
    want = bufs()
    B.moe_grouped_ffn(xd, offsets, W1, W3, W2, want["h"], want["out"], ws, a_save=want["a"],
                      b_save=want["b"], flags=flags | B.MOE_CHECK, row_scale=row_scale)
    torch.cuda.synchronize()
    return got, want


@pytest.mark.parametrize("counts,d,f", [
    ([64, 100, 0, 300, 37, 1, 0, 10], 512, 1024),      # ragged, empty experts
    ([5], 512, 1024),                                   # one partial tile
    ([128, 128], 256, 256),                             # exact tiles
    ([3, 130, 257, 129], 1024, 384),                    # several row tiles per expert
    ([1000], 128, 64),                                  # one k-block pair (d = 128)
])
@pytest.mark.parametrize("single_cta", [False, True])
def test_fp8_ffn_equals_dequantised_bf16_ffn_and_oracle(lib, counts, d, f, single_cta):
    E = len(counts)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    N = int(offsets[-1])
    seed = N + d + f
    codes, scales = _fp8_rows(N, d, seed)
    W1 = _bf16((E, f, d), 0.02, seed + 1)
    W3 = _bf16((E, f, d), 0.02, seed + 2)
    W2 = _bf16((E, d, f), 0.02, seed + 3)
    flags = lib.MOE_SINGLE_CTA_TILES if single_cta else 0
    got, want = _both_paths(lib, torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                            torch.from_numpy(offsets).cuda(), W1.cuda(), W3.cuda(), W2.cuda(),
                            flags)
    for k in ("h", "out", "a", "b"):
        assert _same(got[k], want[k]), k
    # the oracle on its own dequantised rows (bf16 storage of code * scale)
    xd = O.bf16_round(O.dequantize_fp8_blocks(codes, scales))
    ra, rb, rh, ro = O.expert_ffn(xd, offsets, bits(W1), bits(W3), bits(W2))
    assert_close(f64(got["h"]), rh, "h")
    assert_close(f64(got["out"]), ro, "o")
    assert_close(f64(got["a"]), O.bf16_round(ra), "a")


def test_fp8_ffn_row_scale_prepacked_and_without_saves(lib):
    counts = [40, 90, 0, 200, 129]
    E, d, f = len(counts), 512, 256
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    N = int(offsets[-1])
    codes, scales = _fp8_rows(N, d, 21)
    W1, W3, W2 = (_bf16((E, f, d), 0.02, 22).cuda(), _bf16((E, f, d), 0.02, 23).cuda(),
                  _bf16((E, d, f), 0.02, 24).cuda())
    rs = torch.rand(N, generator=torch.Generator().manual_seed(25)).cuda()
    xq, xs = torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()
    offs = torch.from_numpy(offsets).cuda()
    got, want = _both_paths(lib, xq, xs, offs, W1, W3, W2, 0, row_scale=rs, save=False)
    assert _same(got["h"], want["h"]) and _same(got["out"], want["out"])
    # prepacked weights give the same bits
    W1p, W3p, W2p = torch.empty_like(W1), torch.empty_like(W3), torch.empty_like(W2)
    lib.moe_prepack_weights(W1, W3, W2, W1p, W3p, W2p)
    h = torch.empty_like(got["h"])
    out = torch.empty_like(got["out"])
    lib.moe_grouped_ffn_fp8(xq, xs, offs, W1p, W3p, W2p, h, out,
                            lib.workspace(lib.grouped_ffn_fp8_ws_bytes(N, d, f, E)),
                            flags=lib.MOE_WEIGHTS_PREPACKED | lib.MOE_CHECK, row_scale=rs)
    torch.cuda.synchronize()
    assert _same(h, got["h"]) and _same(out, got["out"])


def test_fp8_ffn_argument_checks(lib):
    xq = torch.zeros((8, 192), dtype=torch.uint8, device="cuda")      # d % 128 != 0
    xs = torch.zeros((8, 1), dtype=torch.float32, device="cuda")
    W = torch.zeros((2, 64, 192), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((2, 192, 64), dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([0, 4, 8], dtype=torch.int32, device="cuda")
    h = torch.empty((8, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((8, 192), dtype=torch.bfloat16, device="cuda")
    ws = lib.workspace(1 << 16)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_grouped_ffn_fp8(xq, xs, offs, W, W, W2, h, out, ws)
    assert ei.value.status == 2


def _device_bf16(shape, std, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * std).to(torch.bfloat16)


@pytest.mark.parametrize("T,d,E,R,f,skew", [(16384, 4096, 128, 8, 1536, 0.0),    # training shape
                                            (2048, 7168, 384, 8, 2048, 0.0)])   # large: tails
def test_fp8_ffn_full_size_equals_dequantised_path(lib, T, d, E, R, f, skew):
    idx, _ = random_routing(T, E, R, seed=T + E, skew=skew)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    N = T * R
    # codes: every finite E4M3 pattern but the NaNs (0x7f, 0xff), scales in [2^-6, 2^-2]
    g = torch.Generator(device="cuda").manual_seed(N)
    xq = torch.randint(0, 254, (N, d), generator=g, device="cuda", dtype=torch.int32)
    xq = torch.where(xq >= 127, xq + 1, xq).to(torch.uint8)
    xs = torch.exp2(torch.rand((N, d // 128), generator=g, device="cuda") * 4.0 - 6.0)
    W1 = _device_bf16((E, f, d), 0.02, 1)
    W3 = _device_bf16((E, f, d), 0.02, 2)
    W2 = _device_bf16((E, d, f), 0.02, 3)
    got, want = _both_paths(lib, xq, xs, torch.from_numpy(offsets).cuda(), W1, W3, W2, 0,
                            save=False)
    assert _same(got["h"], want["h"]) and _same(got["out"], want["out"])
    del W1, W3, W2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,over", [("mid", dict(T=1024)), ("train", dict(T=512))])
def test_layer_forward_with_fp8_dispatch(lib, name, over):
    """MOE_FP8_DISPATCH: the layer's rows travel as fp8 and the GEMMs read them
    dequantised -- the same bits as the separate calls on the layer's routing,
    and the oracle's layer on fp8-quantised rows."""
    wl = synth.workload(name, **over)
    inp = synth.layer_inputs(wl)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    T, d, E, R, f = wl.T, wl.d, wl.E, wl.R, wl.f
    N = T * R
    layer = lib.Layer(dev["w_gate"], dev["bias"], dev["W1"], dev["W3"], dev["W2"], R, T)
    saved = lib.Saved(layer, "cuda", train=False)
    y = torch.empty_like(dev["x"])
    flags = lib.MOE_FP8_DISPATCH
    assert lib.layer_fwd_ws_bytes(layer, flags) > lib.layer_fwd_ws_bytes(layer)
    lib.moe_layer_fwd(layer, dev["x"], y, saved, lib.workspace(lib.layer_fwd_ws_bytes(layer, flags)),
                      flags=flags | lib.MOE_CHECK)
    torch.cuda.synchronize()
    # the separate calls on the layer's routing
    i32 = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    row_slot, slot_row = torch.empty(N, **i32), torch.empty(N, **i32)
    xq = torch.empty((N, d), dtype=torch.uint8, device="cuda")
    xs = torch.empty((N, d // 128), dtype=torch.float32, device="cuda")
    lib.moe_dispatch_fp8(dev["x"], saved.topk_idx, E, counts, offsets, row_slot, slot_row, xq, xs,
                         lib.workspace(lib.dispatch_ws_bytes(T, d, E, R)), flags=lib.MOE_CHECK)
    xd = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    lib.moe_dequant_fp8(xq, xs, xd)
    h = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    lib.moe_grouped_ffn(xd, offsets, dev["W1"], dev["W3"], dev["W2"], h, o,
                        lib.workspace(lib.grouped_ffn_ws_bytes(N, d, f, E)), flags=lib.MOE_CHECK)
    y2 = torch.empty_like(y)
    lib.moe_combine(o, slot_row, saved.topk_w, y2, R)
    torch.cuda.synchronize()
    assert _same(saved.x_perm, xd)
    assert _same(y, y2)
    # the oracle's own layer on fp8-quantised rows: its routing, its quantiser,
    # its FFN and combine; compared on the tokens routed alike (near ties aside)
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    logits = O.gate_logits(bits(inp["x"]), inp["w_gate"].numpy(), bias)
    idx, w = O.route_topk(logits, R)
    same = (saved.topk_idx.cpu().numpy() == idx).all(axis=1)
    assert (same | near_tie_tokens(logits, R)).all(), "routing differs without a near tie"
    _, offs, rs, sr = O.dispatch_plan(idx, E)
    codes, scales = O.quantize_fp8_blocks(bits(inp["x"]))
    xp = O.bf16_round(O.dequantize_fp8_blocks(codes, scales))[rs // R]
    o_ref = O.expert_ffn(xp, offs, bits(inp["W1"]), bits(inp["W3"]), bits(inp["W2"]))[3]
    y_ref = O.combine(o_ref, sr, w, T, R)
    assert_close(f64(y)[same], y_ref[same], "y (fp8 dispatch, tokens routed alike)")
