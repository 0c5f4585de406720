"""NVFP4 V2 rows (codes, then the scale stream): the repack against the
oracle's, and every call that takes V2 weights against the oracle and, bit
for bit, against the same call on the 36-byte-group rows (the V2 arms of
memra-engine moe_rows_ceiling_bench.rs assert that bit-identity)."""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, assert_bitexact, assert_close, dev, nan_filled

pytestmark = pytest.mark.gpu


def _v1_v2(m, k, seed):
    v1 = synth.nvfp4_rows(seed, m, k)
    return v1, oracle.nvfp4_repack_v2(v1, m, k)


# k % 256 == 0 takes the chunked kernel (bulk stores of each chunk's row
# segments): 4 groups a row (64 rows a chunk), 20 a row (rows straddling
# chunks), a last chunk of a few groups; the others take the per-thread kernel
@pytest.mark.parametrize("m,k", [(1, 64), (37, 320), (2048, 4096), (5, 256), (53, 256), (37, 1280), (3, 2304),
                                 (1000, 2048)])
def test_repack_matches_the_oracle(h, m, k):
    v1, want = _v1_v2(m, k, 0x7001 + m)
    out = torch.full((want.size,), 0xA5, dtype=torch.uint8, device="cuda")
    q.qmm_nvfp4_repack_v2(h, dev(v1), out, m, k)
    assert q.qmm_sync_status(h) == 0
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("ts", [1.0, 0.75])
def test_dequant_v2_bit_exact(h, ts):
    m, k = 70, 576
    v1, v2 = _v1_v2(m, k, 0x7101)
    out = torch.full((m, k), float("nan"), device="cuda")
    q.qmm_dequant(h, "nvfp4_v2", dev(v2), out, m, k, ts)
    assert q.qmm_sync_status(h) == 0
    want = oracle.dequant("nvfp4_v2", v2, m, k, ts)
    assert_bitexact(out.cpu().numpy(), want, what="dequant v2")
    assert np.array_equal(want, oracle.dequant("nvfp4", v1, m, k, ts))


# The plain GEMV reads 36-byte-group rows through the split-K kernel and V2
# rows through the shared-memory X / register-X kernels, whose summation
# orders differ: both are held to the oracle's tolerance and to each other's
# within it (the MoE calls below, one kernel for both layouts, stay
# bit-identical).
@pytest.mark.parametrize("m,k", [(300, 512), (1024, 4096)])  # shared-memory X kernel, register-X kernel
def test_gemv_v2_matches_oracle_and_v1(h, m, k):
    v1, v2 = _v1_v2(m, k, 0x7201 + k)
    d1, d2 = dev(v1), dev(v2)
    for n in range(1, 9):
        x = synth.activations(n, k)
        xd = dev(x)
        y1, y2 = nan_filled(n, m), nan_filled(n, m)
        q.qmm_gemv(h, "nvfp4", d1, xd, y1, m, k, n)
        q.qmm_gemv(h, "nvfp4_v2", d2, xd, y2, m, k, n)
        assert q.qmm_sync_status(h) == 0
        ref, am = oracle.matmul("nvfp4_v2", v2, x, m, k, n)
        g1, g2 = y1.cpu().numpy(), y2.cpu().numpy()
        assert_close(g2, ref, am, FMA_REL, what=f"v2 n={n}")
        assert_close(g1, ref, am, FMA_REL, what=f"v1 n={n}")
        assert_close(g2, g1.astype(np.float64), am, 2 * FMA_REL, what=f"v2 vs v1 n={n}")


def test_moe_gate_up_v2_workload(h):
    in_f, n_ff, n_used, t = 4096, 2048, 8, 1
    n_pairs = n_used * t
    v1s = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    v2s = [oracle.nvfp4_repack_v2(a, n_ff, in_f) for a in v1s]
    scales = np.array([0.5 + 0.01 * p for p in range(2 * n_pairs)], np.float32)
    x = synth.activations(t, in_f)
    outs = []
    for fmt, mats in (("nvfp4", v1s), ("nvfp4_v2", v2s)):
        dm = [dev(a) for a in mats]
        table = torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")
        y = nan_filled(2, n_pairs, n_ff)
        q.qmm_moe_gemv(h, fmt, table, dev(scales), dev(x), y, in_f, n_ff, n_used, t)
        assert q.qmm_sync_status(h) == 0
        outs.append(y.cpu().numpy())
    ref, am = oracle.moe_gate_up("nvfp4_v2", v2s, scales, x, in_f, n_ff, n_used, t)
    assert_close(outs[1], ref, am, FMA_REL, what="moe v2")
    assert np.array_equal(outs[1].view(np.uint32), outs[0].view(np.uint32))


def test_moe_down_v2(h):
    n_ff, gin, n_used, t = 2048, 512, 8, 2
    n_pairs = n_used * t
    v1s = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(1, j, 2), gin, n_ff) for j in range(n_pairs)]
    v2s = [oracle.nvfp4_repack_v2(a, gin, n_ff) for a in v1s]
    scales = np.array([0.5 + 0.01 * p for p in range(n_pairs)], np.float32)
    hact = synth.activations(n_pairs, n_ff, seed=1234)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    outs = []
    for fmt, mats in (("nvfp4", v1s), ("nvfp4_v2", v2s)):
        dm = [dev(a) for a in mats]
        table = torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")
        y = nan_filled(t, gin)
        q.qmm_moe_down(h, fmt, table, dev(scales), dev(hact), y, n_ff, gin, n_used, t, ws, wsb)
        assert q.qmm_sync_status(h) == 0
        outs.append(y.cpu().numpy())
    ref, am = oracle.moe_down("nvfp4_v2", v2s, scales, hact, n_ff, gin, n_used, t)
    assert_close(outs[1], ref, am, FMA_REL, what="moe down v2")
    assert np.array_equal(outs[1].view(np.uint32), outs[0].view(np.uint32))


def test_v2_argument_errors(h):
    m, k = 64, 128
    v1, v2 = _v1_v2(m, k, 0x7301)
    d2 = dev(v2)
    x = dev(synth.activations(16, k))
    y = nan_filled(16, m)
    ws = torch.empty(16 * k * 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError) as e:  # no tensor-core path for V2 rows
        q.qmm_gemm(h, "nvfp4_v2", d2, x, y, m, k, 16, ws)
    assert e.value.status == 2
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_noalloc("nvfp4_v2", d2, x, y, m, k, 16)
    assert e.value.status == 2
    with pytest.raises(q.QmmError) as e:  # V2 needs k % 64 == 0
        q.qmm_gemv(h, "nvfp4_v2", d2, x, y, m, 96, 1)
    assert e.value.status == 3
    buf = torch.empty(2 * v1.size, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError) as e:  # repack into an overlapping buffer
        q.qmm_nvfp4_repack_v2(h, buf, buf[16:], m, k)
    assert e.value.status == 9
    with pytest.raises(q.QmmError) as e:
        q.qmm_nvfp4_repack_v2(h, dev(v1), buf, m, 96)
    assert e.value.status == 3
    assert np.all(np.isnan(y.cpu().numpy()))  # nothing was launched
