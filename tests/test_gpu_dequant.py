"""qmm_dequant is bit-exact with the oracle (signed zeros compare equal)."""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
from qmm_cases import FORMATS, assert_bitexact, dev, nan_filled, weights

pytestmark = pytest.mark.gpu

SHAPES = [(256, 256), (4608, 1024), (1024, 4608), (3, 768), (1, 256)]


def _run(h, fmt, w, m, k, ts):
    out = nan_filled(m, k)
    q.qmm_dequant(h, fmt, dev(w), out, m, k, ts)
    assert q.qmm_sync_status(h) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("m,k", SHAPES)
@pytest.mark.parametrize("fmt", FORMATS)
def test_dequant_bitexact(h, fmt, m, k):
    w = weights(fmt, m, k)
    ts = 0.7 if fmt == "nvfp4" else 1.0
    assert_bitexact(_run(h, fmt, w, m, k, ts), oracle.dequant(fmt, w, m, k, ts), f"{fmt} {m}x{k}")


def test_dequant_nvfp4_moe_matrix(h):
    # one 2048 x 4096 expert matrix of the MoE workload
    w = weights("nvfp4", 2048, 4096, seed=0x8181)
    assert_bitexact(_run(h, "nvfp4", w, 2048, 4096, 1.0), oracle.dequant("nvfp4", w, 2048, 4096), "nvfp4 moe")


@pytest.mark.parametrize("fmt,k", [("q4_0", 32), ("q8_0", 64), ("q4_k", 256), ("q6_k", 512), ("nvfp4", 64)])
def test_dequant_every_subnormal_and_negative_scale(h, fmt, k):
    # scale codes swept over every f16 subnormal and sign (the low two bytes of
    # each block are the d field of Q4_0 / Q8_0 / Q4_K; Q6_K keeps d last)
    m = 1024
    w = weights(fmt, m, k).copy().reshape(m, -1)
    bb = oracle.block_bytes(fmt)
    codes = np.arange(m * (k // oracle.block_weights(fmt)), dtype=np.uint32)
    codes = (codes % 1024) | ((codes & 1024) << 5)  # 0..1023 subnormals, both signs
    blocks = w.reshape(-1, bb)
    if fmt in ("q4_0", "q8_0", "q4_k"):
        blocks[:, 0] = codes & 0xFF
        blocks[:, 1] = codes >> 8
    elif fmt == "q6_k":
        blocks[:, 208] = codes & 0xFF
        blocks[:, 209] = codes >> 8
    else:  # nvfp4: every E4M3 scale code except the NaN ones
        c = (codes[:, None] + np.arange(4)) & 0xFF
        blocks[:, 0:4] = np.where((c & 0x7F) == 0x7F, 0x38, c)
    w = blocks.reshape(-1)
    assert_bitexact(_run(h, fmt, w, m, k, 1.0), oracle.dequant(fmt, w, m, k), fmt)
