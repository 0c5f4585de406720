"""include/qmm.h is a C header: a strict C11 program includes it, links
libqmm.so and calls the host-only entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import gemv_dequant_gemm_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include "qmm.h"
#include <stdio.h>
#include <string.h>

int main(void) {
    if (qmm_block_weights(QMM_Q4_K) != 256 || qmm_block_bytes(QMM_Q4_K) != 144) return 1;
    if (qmm_row_bytes(QMM_Q4_0, 4608) != 4608 / 32 * 18) return 2;
    if (qmm_row_bytes(QMM_NVFP4, 4096) != 2304 || qmm_row_bytes(QMM_NVFP4_V2, 4096) != 2304) return 3;
    if (qmm_row_bytes(QMM_Q8_0, 33) != 0) return 4;
    if (qmm_gemm_workspace_bytes(QMM_Q4_0, 4608, 1024, 512) != (size_t)512 * 1024 * 2) return 5;
    if (qmm_moe_down_workspace_bytes(4096, 8, 1) != (size_t)8 * 4096 * 4) return 6;
    const char *msg = qmm_strerror(QMM_ERR_SHAPE);
    if (msg == NULL || strlen(msg) == 0) return 7;
    if (qmm_gemm(NULL, QMM_Q4_0, NULL, NULL, NULL, 1, 32, 1, NULL, 0, NULL) != QMM_ERR_INVALID_ARG) return 8;
    printf("c-abi ok\n");
    return 0;
}
"""


def test_header_compiles_as_c11_and_links():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = q.load()  # builds libqmm.so if needed
    pkg = os.path.dirname(q.LIB_PATH)
    out_dir = os.path.join(pkg, "_build")
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "c_abi_check.c")
    exe = os.path.join(out_dir, "c_abi_check")
    with open(src, "w") as f:
        f.write(C_SRC)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), src,
           "-L", pkg, "-lqmm", "-Wl,-rpath," + pkg, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "c-abi ok" in r.stdout
    del lib
