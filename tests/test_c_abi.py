"""The boundary is a C ABI: include/moe.h compiles as C99 and as C++, and a
plain C program links libmoe.so and calls it.  Only calls that touch no GPU run
here: the version, status strings, host argument checks and workspace size
queries (the same answers the Python binding gets)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from expert_moe_route_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  size_t n = 0, n8 = 0;
  moe_layer_t L;
  moe_status_t st;
  memset(&L, 0, sizeof L);
  L.T = 256; L.d = 512; L.E = 8; L.R = 2; L.f = 1024;
  /* host checks only look at these for non-NULL and 16-byte alignment */
  L.w_gate = (const float*)(size_t)4096;
  L.W1 = (const uint16_t*)(size_t)8192;
  L.W3 = (const uint16_t*)(size_t)12288;
  L.W2 = (const uint16_t*)(size_t)16384;
  printf("version %d\n", moe_version());
  printf("status %s\n", moe_status_string(MOE_ERR_BAD_ROUTING));
  st = moe_layer_fwd(&L, NULL, NULL, NULL, NULL, &n, 0, NULL);
  printf("fwd %d %zu\n", (int)st, n);
  st = moe_layer_fwd(&L, NULL, NULL, NULL, NULL, &n8, MOE_FP8_DISPATCH, NULL);
  printf("fwd_fp8 %d %zu\n", (int)st, n8);
  st = moe_layer_bwd(&L, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, &n, 0, NULL);
  printf("bwd %d %zu\n", (int)st, n);
  st = moe_grouped_ffn(NULL, NULL, 10, 64, 60, 4, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                       NULL, &n, 0, NULL);
  printf("ffn_f60 %d\n", (int)st);
  return 0;
}
"""


def _compile_and_run(tmp_path, compiler, std, lang):
    src = tmp_path / ("prog.c" if lang == "c" else "prog.cpp")
    src.write_text(C_PROGRAM)
    exe = tmp_path / f"prog_{lang}"
    libdir = os.path.dirname(B.library_path())
    subprocess.run([compiler, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
                    str(src), "-o", str(exe), "-L", libdir, "-lmoe", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True, text=True, timeout=300)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    return dict(line.split(" ", 1) for line in out.stdout.splitlines())


@pytest.mark.parametrize("compiler,std,lang", [("gcc", "c99", "c"), ("g++", "c++17", "cpp")])
def test_plain_program_calls_the_c_abi(tmp_path, compiler, std, lang):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    B.lib()                                     # builds libmoe.so in-tree if needed
    got = _compile_and_run(tmp_path, compiler, std, lang)
    assert got["version"] == "100"
    assert got["status"] == "MOE_ERR_BAD_ROUTING"
    # the same workspace sizes the binding queries through ctypes
    layer = B.moe_layer_t(256, 512, 8, 2, 1024, 4096, 0, 8192, 12288, 16384)
    n = ctypes.c_size_t(0)
    assert B.lib().moe_layer_fwd(ctypes.byref(layer), None, None, None, None, ctypes.byref(n), 0,
                                 None) == 0
    assert got["fwd"] == f"0 {n.value}"
    st8, n8 = got["fwd_fp8"].split()
    assert st8 == "0" and int(n8) == n.value + 512 * 512 + 512 * 4 * 4
    assert got["bwd"].split()[0] == "0" and int(got["bwd"].split()[1]) > 0
    assert got["ffn_f60"] == "2"                # f % 8 != 0: MOE_ERR_UNSUPPORTED
