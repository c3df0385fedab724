"""The public header is plain C: a C99 program that includes it compiles with
-pedantic -Werror, links against the library and calls its host-side entry
points, getting the same sizes and layouts as the Python binding (no GPU,
no Python or torch types across the boundary)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from moe_expert_layer_05_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stddef.h>
#include <stdio.h>
#include "moe_gb300.h"

int main(void) {
  moe_config c = {4096, 4096, 8, 2, 14336, 0, MOE_SCORE_SOFTMAX, MOE_GEMM_BF16};
  moe_act_layout L;
  if (moe_activation_layout(&c, 1, &L) != MOE_OK) return 1;
  moe_config n = c;
  n.dtype = MOE_GEMM_NVFP4;
  moe_config bad = c;
  bad.H = 100;
  printf("%d %d %zu %zu %zu %zu %d %zu %zu %s\n", (int)moe_version(), (int)moe_capacity_rows(&c), L.total,
         moe_workspace_bytes(&c), moe_nvfp4_weights_bytes(&n), moe_mxfp8_weights_bytes(&c),
         (int)moe_capacity_rows(&bad), sizeof(moe_gemm_args), offsetof(moe_gemm_args, b_scale_group),
         moe_status_string(MOE_ERR_WORKSPACE));
  return 0;
}
"""


def test_header_is_plain_c_and_links():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = api.library_path()
    api.load()                                    # builds the library if it is missing
    out_dir = os.path.dirname(lib)                # the library's own (git-ignored) build folder
    src = os.path.join(out_dir, "c_abi_check.c")
    exe = os.path.join(out_dir, "c_abi_check")
    with open(src, "w") as fh:
        fh.write(C_SRC)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-o", exe, lib, "-Wl,-rpath," + out_dir], check=True)
    res = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    cfg = api.make_config(4096, 4096, 8, 2, 14336)
    nv = api.make_config(4096, 4096, 8, 2, 14336, dtype="nvfp4")
    assert int(res[0]) == api.moe_version()
    assert int(res[1]) == api.moe_capacity_rows(cfg)
    assert int(res[2]) == api.moe_activation_layout(cfg, True).total
    assert int(res[3]) == api.moe_workspace_bytes(cfg)
    assert int(res[4]) == api.moe_nvfp4_weights_bytes(nv) > 0
    assert int(res[5]) == api.moe_mxfp8_weights_bytes(cfg) > 0
    assert int(res[6]) == -1
    assert int(res[7]) == ctypes.sizeof(api.MoeGemmArgs)             # the binding's struct matches the header's
    assert int(res[8]) == api.MoeGemmArgs.b_scale_group.offset
    assert " ".join(res[9:]) == api.moe_status_string(-4)
