"""A seeded sweep of random shapes through the public calls, against the oracle.

The fixed cases elsewhere pin the workload shapes, the edges and exact
arithmetic.  This sweep adds breadth: ragged m, n and k of every format,
drawn from one seeded stream, so that a tile, tail or plan combination that
no fixed case names still has to match the oracle -- the GEMM within its
tensor-core tolerance, the GEMV and the MoE calls within 1e-5 * sum|W*X|,
the dequant bit for bit.  Half of the down-projection cases are drawn where
the grouped kernel applies (rows of 2048 or 4096, 2, 4 or 8 pairs a token).
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, FORMATS, TC_ABS, TC_REL, assert_bitexact, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu

# k granularity per format (f32: the GEMM's TMA pitch wants k % 4 == 0)
QK = {"f32": 4, "q4_0": 32, "q8_0": 32, "q4_k": 256, "q6_k": 256, "nvfp4": 64, "nvfp4_v2": 64}
V2_FORMATS = FORMATS + ["nvfp4_v2"]


def _k(rng, fmt, kmax):
    return QK[fmt] * int(rng.integers(1, max(2, kmax // QK[fmt]) + 1))


def _w(fmt, m, k, seed):
    """Packed weights; V2 rows made from 36-byte groups by the oracle's repack."""
    if fmt == "nvfp4_v2":
        return oracle.nvfp4_repack_v2(weights("nvfp4", m, k, seed=seed), m, k)
    return weights(fmt, m, k, seed=seed)


def _cases(count, seed, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng, i) for i in range(count)]


def _gemm_case(rng, i):
    fmt = FORMATS[int(rng.integers(len(FORMATS)))]
    return fmt, int(rng.integers(1, 600)), _k(rng, fmt, 2304), int(rng.integers(9, 600))


@pytest.mark.parametrize("fmt,m,k,n", _cases(16, 2026, _gemm_case))
def test_sweep_gemm(h, fmt, m, k, n):
    w, x = _w(fmt, m, k, seed=m + 7 * k), synth.activations(n, k, seed=n)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    wsb = q.qmm_gemm_workspace_bytes(fmt, m, k, n)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    d = nan_filled(n, m)
    q.qmm_gemm(h, fmt, dev(w), dev(x), d, m, k, n, ws if wsb else None, wsb)
    assert q.qmm_sync_status(h) == 0
    assert_close(d.cpu().numpy(), ref, am, TC_REL, TC_ABS, what=f"gemm {fmt} {m}x{k}x{n}")


def _gemv_case(rng, i):
    fmt = V2_FORMATS[int(rng.integers(len(V2_FORMATS)))]
    k = int(rng.integers(1, 3000)) if fmt == "f32" else _k(rng, fmt, 6144)
    return fmt, int(rng.integers(1, 2500)), k, int(rng.integers(1, 9))


@pytest.mark.parametrize("fmt,m,k,n", _cases(24, 2027, _gemv_case))
def test_sweep_gemv(h, fmt, m, k, n):
    w, x = _w(fmt, m, k, seed=m + 3 * k), synth.activations(n, k, seed=n + 1)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    d = nan_filled(n, m)
    q.qmm_gemv(h, fmt, dev(w), dev(x), d, m, k, n)
    assert q.qmm_sync_status(h) == 0
    assert_close(d.cpu().numpy(), ref, am, FMA_REL, what=f"gemv {fmt} {m}x{k} n={n}")


def _dequant_case(rng, i):
    fmt = V2_FORMATS[i % len(V2_FORMATS)]
    return fmt, int(rng.integers(1, 700)), _k(rng, fmt, 4096)


@pytest.mark.parametrize("fmt,m,k", _cases(14, 2028, _dequant_case))
def test_sweep_dequant(h, fmt, m, k):
    w = _w(fmt, m, k, seed=m + k)
    ts = 0.37 if fmt.startswith("nvfp4") else 1.0
    out = nan_filled(m, k)
    q.qmm_dequant(h, fmt, dev(w), out, m, k, ts)
    assert q.qmm_sync_status(h) == 0
    assert_bitexact(out.cpu().numpy(), oracle.dequant(fmt, w, m, k, ts), what=f"dequant {fmt} {m}x{k}")


def _moe_case(rng, i):
    fmt = V2_FORMATS[int(rng.integers(len(V2_FORMATS)))]
    return fmt, _k(rng, fmt, 4096), int(rng.integers(1, 500)), int(rng.integers(1, 9)), int(rng.integers(1, 4))


def _scales(count):
    return np.array([0.5 + 0.01 * p for p in range(count)], np.float32)


@pytest.mark.parametrize("fmt,in_f,n_ff,n_used,t", _cases(8, 2029, _moe_case))
def test_sweep_moe_gate_up(h, fmt, in_f, n_ff, n_used, t):
    n_pairs = n_used * t
    mats = [_w(fmt, n_ff, in_f, seed=synth.nvfp4_matrix_seed(20, j, p)) for p in range(2) for j in range(n_pairs)]
    dm = [dev(a) for a in mats]
    table = torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f, seed=in_f)
    y = nan_filled(2, n_pairs, n_ff)
    q.qmm_moe_gemv(h, fmt, table, dev(scales), dev(x), y, in_f, n_ff, n_used, t)
    assert q.qmm_sync_status(h) == 0
    ref, am = oracle.moe_gate_up(fmt, mats, scales, x, in_f, n_ff, n_used, t)
    assert_close(y.cpu().numpy(), ref, am, FMA_REL, what=f"moe {fmt} {in_f}->{n_ff} {n_used}x{t}")


def _down_case(rng, i):
    fmt = V2_FORMATS[int(rng.integers(len(V2_FORMATS)))]
    if i % 2 == 0:  # where the grouped kernel applies
        return fmt, int(rng.choice([2048, 4096])), int(rng.integers(1, 300)), int(rng.choice([2, 4, 8])), \
            int(rng.integers(1, 3))
    return fmt, _k(rng, fmt, 2048), int(rng.integers(1, 500)), int(rng.integers(1, 9)), int(rng.integers(1, 4))


@pytest.mark.parametrize("fmt,n_ff,gin,n_used,t", _cases(12, 2030, _down_case))
def test_sweep_moe_down(h, fmt, n_ff, gin, n_used, t):
    n_pairs = n_used * t
    mats = [_w(fmt, gin, n_ff, seed=synth.nvfp4_matrix_seed(21, j, 2)) for j in range(n_pairs)]
    dm = [dev(a) for a in mats]
    table = torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=n_ff + gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    y = nan_filled(t, gin)
    q.qmm_moe_down(h, fmt, table, dev(scales), dev(hact), y, n_ff, gin, n_used, t, ws if wsb else None, wsb)
    assert q.qmm_sync_status(h) == 0
    ref, am = oracle.moe_down(fmt, mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y.cpu().numpy(), ref, am, FMA_REL, what=f"down {fmt} {n_ff}->{gin} {n_used}x{t}")
