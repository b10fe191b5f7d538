"""GPU: moe_dispatch_noalloc, the dispatch entry point that allocates nothing.

It serves callers that cannot call cudaMalloc or pass a workspace -- code inside
a host application or framework whose allocator owns all device memory, and
latency-critical loops that cannot take cudaMalloc's implicit synchronisation.
Its scratch is a fixed array the library reserves on each GPU.  These tests call
it through the C ABI and check it against moe_dispatch (which takes a
caller-provided workspace) on consecutive calls, since every call reuses the
same array.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import random_routing

pytestmark = pytest.mark.gpu


def _buffers(T, d, E, R):
    N = T * R
    return dict(counts=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                row_slot=torch.full((N,), -7, dtype=torch.int32, device="cuda"),
                slot_row=torch.full((N,), -7, dtype=torch.int32, device="cuda"),
                x_perm=torch.zeros((N, d), dtype=torch.bfloat16, device="cuda"))


def _noalloc(B, x, idx, E, out, flags):
    T, R = idx.shape
    stream = torch.cuda.current_stream().cuda_stream
    return B.lib().moe_dispatch_noalloc(
        x.data_ptr(), idx.data_ptr(), T, x.shape[1], E, R, out["counts"].data_ptr(),
        out["offsets"].data_ptr(), out["row_slot"].data_ptr(), out["slot_row"].data_ptr(),
        out["x_perm"].data_ptr(), flags, stream)


def _with_workspace(B, x, idx, E, out):
    T, R = idx.shape
    d = x.shape[1]
    ws = B.workspace(B.dispatch_ws_bytes(T, d, E, R))
    n = ctypes.c_size_t(ws.numel())
    st = B.lib().moe_dispatch(x.data_ptr(), idx.data_ptr(), T, d, E, R, out["counts"].data_ptr(),
                              out["offsets"].data_ptr(), out["row_slot"].data_ptr(),
                              out["slot_row"].data_ptr(), out["x_perm"].data_ptr(), ws.data_ptr(),
                              ctypes.byref(n), B.MOE_CHECK,
                              torch.cuda.current_stream().cuda_stream)
    assert st == B.MOE_OK, B.STATUS[st]


@pytest.mark.parametrize("cases", [[(4096, 256, 64, 6, 1.0), (1000, 136, 256, 8, 0.0)],
                                   [(65536, 64, 256, 8, 1.2), (3, 64, 8, 2, 0.0)]])
def test_noalloc_dispatch_matches_workspace_dispatch(lib, cases):
    for T, d, E, R, skew in cases:          # two calls in a row share the static scratch
        idx_np, _ = random_routing(T, E, R, seed=T + E, skew=skew)
        idx = torch.from_numpy(idx_np).cuda()
        x = torch.randn((T, d), generator=torch.Generator().manual_seed(T)).to(torch.bfloat16).cuda()
        got = _buffers(T, d, E, R)
        st = _noalloc(lib, x, idx, E, got, lib.MOE_CHECK)
        assert st == lib.MOE_OK, lib.STATUS[st]
        want = _buffers(T, d, E, R)
        _with_workspace(lib, x, idx, E, want)
        torch.cuda.synchronize()
        for k in ("counts", "offsets", "row_slot", "slot_row"):
            assert torch.equal(got[k], want[k]), k
        assert torch.equal(got["x_perm"].view(torch.int16), want["x_perm"].view(torch.int16))


def test_noalloc_dispatch_clears_its_error_word_and_rejects_oversize(lib):
    T, d, E, R = 64, 64, 8, 2
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor(np.tile([0, 1], (T, 1)), dtype=torch.int32, device="cuda")
    idx[3, 1] = E                                            # out of range
    code = {name: value for value, name in lib.STATUS.items()}
    assert _noalloc(lib, x, idx, E, _buffers(T, d, E, R), lib.MOE_CHECK) == code["MOE_ERR_BAD_ROUTING"]
    idx[3, 1] = 1                                            # the next call starts clean
    assert _noalloc(lib, x, idx, E, _buffers(T, d, E, R), lib.MOE_CHECK) == lib.MOE_OK
    # 1024 experts x 1025 token blocks of histograms exceed the 4 MiB array
    big_T = 1025 * 256
    st = lib.lib().moe_dispatch_noalloc(None, None, big_T, 64, 1024, 8, None, None, None, None,
                                        None, 0, None)
    assert st == code["MOE_ERR_WORKSPACE"]          # before anything is enqueued
