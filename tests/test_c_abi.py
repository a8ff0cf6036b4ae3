"""The boundary is a C ABI: a plain C99 program includes include/mhc.h
(compiled with -pedantic), links libmhc.so and calls the entry points that
need no GPU -- defaults, error strings, workspace sizes and host-side
argument checks.  No CUDA call is reached."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mhc.h"

int main(void) {
    mhc_params p;
    mhc_default_params(&p);
    if (p.sinkhorn_iters != 20 || p.post_mult != 2.0f || p.norm_eps != 1e-6f) return 1;
    if (strcmp(mhc_strerror(MHC_OK), "ok") != 0) return 2;
    if (mhc_pre_workspace_bytes(0) != 0 || mhc_pre_workspace_bytes(1000) == 0) return 3;
    if (mhc_swizzle_scales_128x4_bytes(200, 160) != (size_t)256 * 160) return 4;
    /* host-side checks answer before any launch */
    if (mhc_post(NULL, NULL, NULL, NULL, 4, 4, NULL, NULL) != MHC_ERR_NULL) return 5;
    if (mhc_post(NULL, NULL, NULL, NULL, -1, 4, NULL, NULL) != MHC_ERR_SHAPE) return 6;
    if (mhc_post(NULL, NULL, NULL, NULL, 0, 0, NULL, NULL) != MHC_OK) return 7;
    if (mhc_quantize_mxfp8(NULL, 4, 48, 4, NULL, NULL, NULL) != MHC_ERR_SHAPE) return 8;
    if (mhc_release_weights(NULL) != MHC_OK) return 9;
    puts("c-abi ok");
    return 0;
}
"""


def test_c_program_links_and_calls_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from hyper_connection_residual_mhc_gb300 import build
    build.build()
    libdir = os.path.join(ROOT, "hyper_connection_residual_mhc_gb300", "_build")
    src = tmp_path / "use_mhc.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_mhc"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                           "-L", libdir, "-lmhc", "-Wl,-rpath," + libdir])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == "c-abi ok"
