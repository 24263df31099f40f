"""The C ABI from plain C and from C++ (no GPU needed): include/moe_route.h
compiles as strict C99 and as C++17 with every warning an error, a client
links against libmoe_route.so, and the host-side calls it makes behave as
the header says (the ABI version, a call refused on the host before any CUDA
call, its status string, no kernel launched, the normal library's
debug-bounds query)."""
import os
import shutil
import subprocess

import pytest

from moe_routing_precision_gb300 import _build

CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "moe_route.h"

int main(void) {
  if (moe_abi_version() != MOE_ROUTE_ABI_VERSION) return 1;
  /* k = 0 is refused on the host before any CUDA call */
  moe_status_t s = moe_topk_gate((const float *)0x10000, 4, 16, 0, (int32_t *)0x10000,
                                 (float *)0x10000, MOE_WEIGHTS_SOFTMAX_TOPK, NULL);
  if (s != MOE_ERR_INVALID_ARG) return 2;
  if (strncmp(moe_status_string(s), "MOE_ERR_INVALID_ARG", 19) != 0) return 3;
  if (moe_kernel_launch_count() != 0) return 4;
  if (moe_debug_bounds_enabled() != 0) return 5;
  if (moe_debug_bounds_selftest(NULL) != MOE_ERR_UNSUPPORTED) return 6;
  printf("OK\n");
  return 0;
}
"""


@pytest.mark.parametrize("compiler,std,suffix", [("gcc", "-std=c99", ".c"),
                                                 ("g++", "-std=c++17", ".cpp")])
def test_header_compiles_links_and_runs(tmp_path, compiler, std, suffix):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    lib = _build.build()
    src = tmp_path / f"client{suffix}"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib)
    cmd = [compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{_build.INCLUDE}",
           str(src), f"-L{libdir}", "-lmoe_route", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "OK", (r.returncode, r.stdout, r.stderr)
