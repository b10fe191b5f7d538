"""GPU parity: block-scaled fp8 dispatch (E4M3 codes + per-128-channel fp32
scales) and the bf16 identity expert + combine behind it."""
import numpy as np
import pytest
import torch

from workloads import synth
from oracle import moe_oracle as O
from tests.helpers import assert_close, bits, f64, random_routing

pytestmark = pytest.mark.gpu


def _dispatch_fp8(B, x, idx, E):
    T, R = idx.shape
    d = x.shape[1]
    N = T * R
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               row_slot=torch.empty(N, dtype=torch.int32, device="cuda"),
               slot_row=torch.empty(N, dtype=torch.int32, device="cuda"),
               xq=torch.empty((N, d), dtype=torch.uint8, device="cuda"),
               xs=torch.empty((N, d // 128), dtype=torch.float32, device="cuda"))
    ws = B.workspace(B.dispatch_ws_bytes(T, d, E, R))
    B.moe_dispatch_fp8(x, idx, E, out["counts"], out["offsets"], out["row_slot"], out["slot_row"],
                       out["xq"], out["xs"], ws, flags=B.MOE_CHECK)
    torch.cuda.synchronize()
    return out


def _x(T, d, seed, spread=4.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, d), generator=g) * torch.exp(torch.rand((T, 1), generator=g) * spread - spread / 2)
    x[0, :128] = 0.0                                  # an all-zero block
    if T > 1:
        x[1, 5] = -0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,d,E,R", [(256, 512, 8, 2), (1000, 2048, 64, 6), (77, 7168, 256, 8),
                                     (3, 128, 4, 4)])
def test_dispatch_fp8_bit_exact(lib, T, d, E, R):
    idx, _ = random_routing(T, E, R, seed=T + d)
    x = _x(T, d, seed=T * d)
    out = _dispatch_fp8(lib, x.cuda(), torch.from_numpy(idx).cuda(), E)
    counts, offsets, row_slot, slot_row = O.dispatch_plan(idx, E)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["row_slot"].cpu().numpy(), row_slot)
    codes, scales = O.quantize_fp8_blocks(bits(x))
    tok = row_slot // R
    assert np.array_equal(out["xq"].cpu().numpy(), codes[tok])
    assert np.array_equal(out["xs"].cpu().numpy(), scales[tok])


@pytest.mark.parametrize("name,T", [("dispatch", 4096), ("dispatch_zipf", 65536)])
def test_dispatch_fp8_full_size_sampled_and_roundtrip(lib, name, T):
    wl = synth.workload(name, T=T)
    r = synth.drawn_routing(wl)
    x = r["x"].cuda()
    out = _dispatch_fp8(lib, x, r["topk_idx"].cuda(), wl.E)
    idx = r["topk_idx"].numpy()
    _, _, row_slot, slot_row = O.dispatch_plan(idx, wl.E)
    assert np.array_equal(out["slot_row"].cpu().numpy(), slot_row)
    toks = np.sort(np.random.default_rng(3).choice(T, 64, replace=False))
    codes, scales = O.quantize_fp8_blocks(bits(r["x"])[toks])
    rows = torch.from_numpy(slot_row.reshape(T, wl.R)[toks]).long().cuda()   # [64, R]
    for q in range(wl.R):
        assert np.array_equal(out["xq"][rows[:, q]].cpu().numpy(), codes)
        assert np.array_equal(out["xs"][rows[:, q]].cpu().numpy(), scales)
    # identity experts in fp8: dequantise, combine in bf16, compare with the oracle
    o = torch.empty((T * wl.R, wl.d), dtype=torch.bfloat16, device="cuda")
    lib.moe_dequant_fp8(out["xq"], out["xs"], o)
    y = torch.empty_like(x)
    lib.moe_combine(o, out["slot_row"], r["topk_w"].cuda(), y, wl.R)
    torch.cuda.synchronize()
    deq = O.dequantize_fp8_blocks(codes, scales)                    # sampled tokens' rows
    ref = O.combine(np.repeat(deq, wl.R, axis=0), np.arange(64 * wl.R), r["topk_w"].numpy()[toks],
                    64, wl.R)
    assert_close(f64(y[torch.from_numpy(toks).cuda()]), ref, "y (fp8 dispatch, identity experts)")
    # and the fp8 round trip stays within the E4M3 step of x
    assert_close(f64(y[torch.from_numpy(toks).cuda()]), O.bf16_to_f64(bits(r["x"])[toks]),
                 "y vs x", max_rel=2.0 ** -4, mean_rel=2.0 ** -5)
