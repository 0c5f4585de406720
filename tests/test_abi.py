"""The C-ABI library builds, loads and exports every declared symbol; its
host-only helpers agree with the format definitions (no GPU needed)."""
import os
import re

import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in ("qmm.h", "qmm_testing.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(qmm_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    lib = q.load()
    declared = _declared()
    assert len(declared) >= 14
    assert declared == set(q.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_row_bytes_agree_with_the_oracle():
    for fmt in ("f32", "q4_0", "q8_0", "q4_k", "q6_k", "nvfp4", "nvfp4_v2"):
        assert q.qmm_block_weights(fmt) == oracle.block_weights(fmt)
        assert q.qmm_block_bytes(fmt) == oracle.block_bytes(fmt)
        for k in (1, 32, 64, 96, 256, 1000, 1024, 4096, 4608):
            assert q.qmm_row_bytes(fmt, k) == oracle.row_bytes(fmt, k), (fmt, k)
    assert q.qmm_row_bytes("q4_0", 0) == 0
    assert q.qmm_row_bytes(99, 32) == 0


def test_workspace_bytes():
    assert q.qmm_gemm_workspace_bytes("q4_0", 4608, 1024, 512) == 512 * 1024 * 2
    assert q.qmm_gemm_workspace_bytes("q4_k", 1024, 4608, 512) == 512 * 4608 * 2
    assert q.qmm_gemm_workspace_bytes("q4_0", 64, 32, 9) == 768  # 576 rounded up to 256
    assert q.qmm_gemm_workspace_bytes("q8_0", 64, 64, 8) == 0    # GEMV regime
    assert q.qmm_gemm_workspace_bytes("f32", 64, 64, 512) == 0   # tf32 path reads X directly
    assert q.qmm_gemm_workspace_bytes("nvfp4_v2", 64, 64, 512) == 0  # no tensor-core path for V2
    assert q.qmm_moe_down_workspace_bytes(4096, 8, 1) == 8 * 4096 * 4
    assert q.qmm_moe_down_workspace_bytes(101, 3, 2) == 2560     # 2424 rounded up to 256
    assert q.qmm_moe_down_workspace_bytes(4096, 1, 5) == 0       # one expert: products go straight to y
    assert q.qmm_moe_down_workspace_bytes(0, 8, 1) == 0


def test_strerror_covers_every_status():
    for s in range(10):
        msg = q.qmm_strerror(s)
        assert msg and msg != "unknown status"
    assert q.qmm_strerror(1234) == "unknown status"


def test_null_handle_and_arguments_are_rejected_without_a_device():
    lib = q.load()
    assert lib.qmm_gemm(None, 1, 16, 16, 16, 32, 32, 32, None, 0, None) == 1
    assert lib.qmm_gemv(None, 1, 16, 16, 16, 32, 32, 1, None) == 1
    assert lib.qmm_dequant(None, 1, 16, 16, 32, 32, 1.0, None) == 1
    assert lib.qmm_moe_gemv(None, 5, 16, 16, 16, 16, 64, 16, 1, 1, None) == 1
    assert lib.qmm_moe_down(None, 5, 16, 16, 16, 16, 64, 16, 2, 1, 16, 256, None) == 1
    assert lib.qmm_nvfp4_repack_v2(None, 16, 16, 1, 64, None) == 1
    assert lib.qmm_gemm_noalloc(7, 16, 16, 16, 16, 64, 16, None) == 1  # unknown dtype
    assert lib.qmm_sync_status(None, None) == 1
    assert lib.qmm_destroy(None) == 0
    assert lib.qmm_create(0, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure mode")
def test_create_fails_loudly_without_a_gpu():
    with pytest.raises(q.QmmError):
        q.qmm_create(0)
    assert q.load().qmm_gemm_noalloc_status(None) == 6  # QMM_ERR_CUDA: no device to set up
