"""The C ABI library builds, loads and exports what include/moe.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from expert_moe_route_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")


def declared_functions():
    with open(HEADER) as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_six_entry_points():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_grouped_ffn", "moe_combine", "moe_layer_fwd",
              "moe_layer_bwd"):
        assert n in names
    assert set(names) == set(B.SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert lib.moe_version() == 100
    assert B.status_string(0) == "MOE_OK" and B.status_string(4) == "MOE_ERR_BAD_ROUTING"


def test_library_is_in_tree():
    assert os.path.realpath(B.library_path()).startswith(
        os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def _st(fn, *args):
    return fn(*args)


def test_host_argument_checks():
    lib = B.lib()
    n = ctypes.c_size_t(0)
    # workspace queries need no device
    assert lib.moe_dispatch(None, None, 100, 64, 8, 2, None, None, None, None, None, None,
                            ctypes.byref(n), 0, None) == 0 and n.value > 0
    # bad shapes
    assert lib.moe_dispatch(None, None, 100, 64, 8, 9, None, None, None, None, None, None,
                            ctypes.byref(n), 0, None) == 1          # R > E
    assert lib.moe_dispatch(None, None, 100, 60, 8, 2, None, None, None, None, None, None,
                            ctypes.byref(n), 0, None) == 2          # d % 8 != 0
    assert lib.moe_dispatch(None, None, 100, 64, 2000, 2, None, None, None, None, None, None,
                            ctypes.byref(n), 0, None) == 2          # E > 1024
    assert lib.moe_dispatch(None, None, -1, 64, 8, 2, None, None, None, None, None, None,
                            ctypes.byref(n), 0, None) == 1
    # too-small or misaligned workspace
    small = ctypes.c_size_t(16)
    assert lib.moe_dispatch(None, None, 100, 64, 8, 2, None, None, None, None, None,
                            ctypes.c_void_p(4096), ctypes.byref(small), 0, None) == 3
    big = ctypes.c_size_t(1 << 20)
    assert lib.moe_dispatch(None, None, 100, 64, 8, 2, None, None, None, None, None,
                            ctypes.c_void_p(4096 + 16), ctypes.byref(big), 0, None) == 3
    # route: R > 32 unsupported, R > E invalid
    assert lib.moe_route(None, None, None, 4, 64, 64, 33, None, None, None, None,
                         ctypes.byref(n), 0, None) == 2
    assert lib.moe_route(None, None, None, 4, 64, 4, 5, None, None, None, None,
                         ctypes.byref(n), 0, None) == 1
    # route workspace: split gate weights when d % 64 == 0, error word only otherwise
    assert lib.moe_route(None, None, None, 4, 128, 8, 2, None, None, None, None,
                         ctypes.byref(n), 0, None) == 0 and n.value >= 6 * 8 * 128
    assert lib.moe_route(None, None, None, 4, 72, 8, 2, None, None, None, None,
                         ctypes.byref(n), 0, None) == 0 and n.value == 256
    # combine: misaligned output
    assert lib.moe_combine(ctypes.c_void_p(4096), ctypes.c_void_p(8192), None, 4, 64, 2,
                           ctypes.c_void_p(4098), None) == 2
    # grouped ffn: f % 8
    assert lib.moe_grouped_ffn(None, None, 10, 64, 60, 4, None, None, None, None, None, None,
                               None, None, None, ctypes.byref(n), 0, None) == 2
    # fp8 grouped ffn: d % 128 (scale blocks), then a size query
    assert lib.moe_grouped_ffn_fp8(None, None, None, 10, 192, 64, 4, None, None, None, None, None,
                                   None, None, None, None, ctypes.byref(n), 0, None) == 2
    assert lib.moe_grouped_ffn_fp8(None, None, None, 10, 256, 64, 4, None, None, None, None, None,
                                   None, None, None, None, ctypes.byref(n), 0, None) == 0
    m = ctypes.c_size_t(0)
    assert lib.moe_grouped_ffn(None, None, 10, 256, 64, 4, None, None, None, None, None, None,
                               None, None, None, ctypes.byref(m), 0, None) == 0
    assert n.value == m.value + 10 * 256 * 2    # + the dequantised bf16 rows (5120 B)


def test_layer_ws_query_and_bwd_shape_limits():
    lib = B.lib()
    L = B.moe_layer_t(256, 512, 8, 2, 1024, 8, 0, 16, 32, 48)
    n = ctypes.c_size_t(0)
    assert lib.moe_layer_fwd(ctypes.byref(L), None, None, None, None, ctypes.byref(n), 0, None) == 0
    assert n.value > 0
    assert lib.moe_layer_bwd(ctypes.byref(L), None, None, None, None, None, None, None, None,
                             None, ctypes.byref(n), 0, None) == 0
    L2 = B.moe_layer_t(256, 520, 8, 2, 1024, 8, 0, 16, 32, 48)   # d % 64 != 0: no backward
    assert lib.moe_layer_bwd(ctypes.byref(L2), None, None, None, None, None, None, None, None,
                             None, ctypes.byref(n), 0, None) == 2
    # fp8 dispatch in the forward: its workspace adds the codes (N*d B) and
    # scales (4*N*d/128 B) of N = 512 rows; d % 128 != 0 is refused
    plain, fp8 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.moe_layer_fwd(ctypes.byref(L), None, None, None, None, ctypes.byref(plain), 0,
                             None) == 0
    assert lib.moe_layer_fwd(ctypes.byref(L), None, None, None, None, ctypes.byref(fp8),
                             B.MOE_FP8_DISPATCH, None) == 0
    assert fp8.value - plain.value == 512 * 512 + 512 * 4 * 4
    assert lib.moe_layer_fwd(ctypes.byref(L2), None, None, None, None, ctypes.byref(fp8),
                             B.MOE_FP8_DISPATCH, None) == 2


def test_no_cpu_fallback_without_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    # with no device the library reports a CUDA error instead of computing on the host
    lib = B.lib()
    n = ctypes.c_size_t(1 << 20)
    st = lib.moe_combine(ctypes.c_void_p(4096), ctypes.c_void_p(8192), None, 4, 64, 2,
                         ctypes.c_void_p(1 << 20), None)
    assert st == 6


def test_selftest_argument_checks():
    lib = B.lib()
    assert lib.moe_selftest_wait_timeout(0, ctypes.c_void_p(4096), None) == 1
    assert lib.moe_selftest_wait_timeout(2000000, ctypes.c_void_p(4096), None) == 1
    assert lib.moe_selftest_wait_timeout(100, None, None) == 1
    assert lib.moe_selftest_wait_timeout(100, ctypes.c_void_p(4096 + 8), None) == 3


def test_noalloc_dispatch_argument_checks_match_moe_dispatch():
    """moe_dispatch_noalloc rejects the shapes and arguments moe_dispatch rejects,
    with the same status, before it touches a device."""
    lib = B.lib()
    code = {name: value for value, name in B.STATUS.items()}
    n = ctypes.c_size_t(0)
    P = 1 << 20                       # a 16-byte-aligned stand-in pointer; never dereferenced

    def noalloc(T, d, E, R, x=None, idx=P, counts=P, offsets=P, row_slot=P, slot_row=P,
                x_perm=None):
        return lib.moe_dispatch_noalloc(x, idx, T, d, E, R, counts, offsets, row_slot, slot_row,
                                        x_perm, 0, None)

    def query(T, d, E, R):
        return lib.moe_dispatch(None, None, T, d, E, R, None, None, None, None, None, None,
                                ctypes.byref(n), 0, None)

    for shape, want in [((100, 64, 8, 9), "MOE_ERR_INVALID_ARG"),      # R > E
                        ((-1, 64, 8, 2), "MOE_ERR_INVALID_ARG"),       # T < 0
                        ((100, 0, 8, 2), "MOE_ERR_INVALID_ARG"),       # d <= 0
                        ((100, 60, 8, 2), "MOE_ERR_UNSUPPORTED"),      # d % 8 != 0
                        ((100, 64, 2000, 2), "MOE_ERR_UNSUPPORTED"),   # E > 1024
                        ((100, 64, 64, 33), "MOE_ERR_UNSUPPORTED"),    # R > 32
                        ((1 << 28, 4096, 8, 1), "MOE_ERR_UNSUPPORTED")]:  # T*d >= 2^40
        assert noalloc(*shape) == code[want], shape
        assert query(*shape) == code[want], shape
    # the static 4 MiB scratch: 1024 experts x 1025 blocks of 256 tokens do not fit
    assert noalloc(1025 * 256, 64, 1024, 8) == code["MOE_ERR_WORKSPACE"]
    shape = (64, 64, 8, 2)
    assert noalloc(*shape, counts=None) == code["MOE_ERR_INVALID_ARG"]
    assert noalloc(*shape, offsets=None) == code["MOE_ERR_INVALID_ARG"]
    assert noalloc(*shape, idx=None) == code["MOE_ERR_INVALID_ARG"]
    assert noalloc(*shape, row_slot=None) == code["MOE_ERR_INVALID_ARG"]
    assert noalloc(*shape, x=P, x_perm=None) == code["MOE_ERR_INVALID_ARG"]  # x without x_perm
    assert noalloc(*shape, x=P + 8, x_perm=P) == code["MOE_ERR_UNSUPPORTED"]  # x not 16-B aligned
    assert noalloc(*shape, x=P, x_perm=P + 4) == code["MOE_ERR_UNSUPPORTED"]


def test_microscaled_fp8_host_checks():
    """moe_quantize_mx, moe_dispatch_mx and moe_grouped_ffn_mx check their shapes
    and answer workspace queries on the host."""
    lib = B.lib()
    st = {v: k for k, v in B.STATUS.items()}
    n = ctypes.c_size_t(0)
    # quantise: K a multiple of 32; no rows is a no-op
    assert lib.moe_quantize_mx(None, ctypes.c_longlong(4), 48, None, None, None) == \
        st["MOE_ERR_UNSUPPORTED"]
    assert lib.moe_quantize_mx(None, ctypes.c_longlong(-1), 64, None, None, None) == \
        st["MOE_ERR_INVALID_ARG"]
    assert lib.moe_quantize_mx(None, ctypes.c_longlong(0), 64, None, None, None) == st["MOE_OK"]
    assert lib.moe_quantize_mx(None, ctypes.c_longlong(4), 64, None, None, None) == \
        st["MOE_ERR_INVALID_ARG"]
    # dispatch: d a multiple of 128, the same shape rules as moe_dispatch, a workspace query
    args = (None, None, 100, 256, 8, 2) + (None,) * 6
    assert lib.moe_dispatch_mx(*args, None, ctypes.byref(n), 0, None) == st["MOE_OK"]
    assert n.value > 0
    bad_d = (None, None, 100, 192, 8, 2) + (None,) * 6
    assert lib.moe_dispatch_mx(*bad_d, None, ctypes.byref(n), 0, None) == st["MOE_ERR_UNSUPPORTED"]
    bad_r = (None, None, 100, 256, 8, 9) + (None,) * 6
    assert lib.moe_dispatch_mx(*bad_r, None, ctypes.byref(n), 0, None) == st["MOE_ERR_INVALID_ARG"]
    small = ctypes.c_size_t(16)
    assert lib.moe_dispatch_mx(*args, ctypes.c_void_p(4096), ctypes.byref(small), 0, None) == \
        st["MOE_ERR_WORKSPACE"]
    # grouped FFN: d and f multiples of 128, E up to 1024, a workspace query
    def ffn(N, d, f, E, ws=None, nb=None):
        return lib.moe_grouped_ffn_mx(*(None,) * 3, N, d, f, E, *(None,) * 10, ws,
                                      ctypes.byref(nb if nb is not None else n), 0, None)
    assert ffn(1000, 256, 384, 8) == st["MOE_OK"] and n.value > 0
    assert ffn(1000, 256, 320, 8) == st["MOE_ERR_UNSUPPORTED"]
    assert ffn(1000, 192, 384, 8) == st["MOE_ERR_UNSUPPORTED"]
    assert ffn(1000, 256, 384, 2000) == st["MOE_ERR_UNSUPPORTED"]
    assert ffn(-1, 256, 384, 8) == st["MOE_ERR_INVALID_ARG"]
    assert ffn(1000, 256, 384, 8, ctypes.c_void_p(4096), ctypes.c_size_t(16)) == \
        st["MOE_ERR_WORKSPACE"]
    # workspace present but no weights
    big = ctypes.c_size_t(1 << 30)
    assert ffn(1000, 256, 384, 8, ctypes.c_void_p(1 << 20), big) == st["MOE_ERR_INVALID_ARG"]
