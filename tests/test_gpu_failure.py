"""GPU: failure detection without a GPU fault.

A pipeline wait that can never be satisfied must give up after its limit,
report MOE_ERR_TIMEOUT through the device error word, and leave the context
usable.  The self-test kernel waits on an mbarrier that nothing arrives on,
through the same bounded-wait routine the GEMM pipelines use.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    ws = lib.workspace(256)
    stream = torch.cuda.current_stream().cuda_stream
    t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t[0].record()
    st = lib.lib().moe_selftest_wait_timeout(50000, ws.data_ptr(), stream)   # 50 ms limit
    t[1].record()
    torch.cuda.synchronize()
    assert st == 5, lib.STATUS.get(st, st)               # MOE_ERR_TIMEOUT
    assert 40.0 <= t[0].elapsed_time(t[1]) < 5000.0       # it waited about the limit, then left
    # the context is intact: ordinary work runs and reports no error
    x = torch.randn((64, 64), device="cuda").to(torch.bfloat16)
    idx = torch.stack([torch.arange(64) % 4, (torch.arange(64) + 1) % 4], 1).int().cuda()
    w = torch.full((64, 2), 0.5, device="cuda")
    N = 128
    outs = [torch.empty(4, dtype=torch.int32, device="cuda"),
            torch.empty(5, dtype=torch.int32, device="cuda"),
            torch.empty(N, dtype=torch.int32, device="cuda"),
            torch.empty(N, dtype=torch.int32, device="cuda"),
            torch.empty((N, 64), dtype=torch.bfloat16, device="cuda")]
    lib.moe_dispatch(x, idx, 4, *outs, lib.workspace(lib.dispatch_ws_bytes(64, 64, 4, 2)),
                     flags=lib.MOE_CHECK)
    y = torch.empty_like(x)
    lib.moe_combine(outs[4], outs[3], w, y, 2)
    torch.cuda.synchronize()
    assert torch.equal(y.float(), x.float())
