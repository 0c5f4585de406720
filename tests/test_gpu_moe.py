"""qmm_moe_gemv against the oracle (NVFP4 gate/up over a routed pointer table)."""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, FORMATS, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu


def _table(ptrs, extra_null=0):
    return torch.tensor(list(ptrs) + [0] * extra_null, dtype=torch.int64, device="cuda")


def _scales(count):
    # per-matrix scale 0.5 + 0.01 * pair index (memra moe_rows_ceiling_bench.rs, scl)
    return np.array([0.5 + 0.01 * p for p in range(count)], np.float32)


def _run_moe(h, fmt, mats_np, scales, x, in_f, n_ff, n_used, t, extra_null=0):
    mats = [dev(mm) for mm in mats_np]
    table = _table([mm.data_ptr() for mm in mats], extra_null)
    y = nan_filled(2, t * n_used, n_ff)
    q.qmm_moe_gemv(h, fmt, table, dev(scales), dev(x), y, in_f, n_ff, n_used, t)
    st = q.qmm_sync_status(h)
    return st, y.cpu().numpy()


def test_moe_gate_up_workload(h):
    # in_f 4096, n_ff 2048, 8 experts, 1 token; the page's 3*n_pairs table with
    # its down plane left empty; every matrix from its own seeded stream
    in_f, n_ff, n_used, t = 4096, 2048, 8, 1
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    scales = _scales(3 * n_pairs)
    x = synth.activations(t, in_f)
    st, y = _run_moe(h, "nvfp4", mats, scales, x, in_f, n_ff, n_used, t, extra_null=n_pairs)
    assert st == 0
    ref, am = oracle.moe_gate_up("nvfp4", mats, scales, x, in_f, n_ff, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="moe")


@pytest.mark.parametrize("fmt", FORMATS)
def test_moe_multi_token_every_format(h, fmt):
    in_f, n_ff, n_used, t = 512, 101, 3, 2
    n_pairs = n_used * t
    mats = [weights(fmt, n_ff, in_f, seed=synth.nvfp4_matrix_seed(1, j, p)) for p in range(2) for j in range(n_pairs)]
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f)
    st, y = _run_moe(h, fmt, mats, scales, x, in_f, n_ff, n_used, t)
    assert st == 0
    ref, am = oracle.moe_gate_up(fmt, mats, scales, x, in_f, n_ff, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=fmt)


def test_moe_bad_table_entry_is_reported(h):
    # a misaligned matrix pointer is caught by the kernel before any access:
    # the call reports QMM_ERR_ALIGN and that matrix's rows come back NaN
    in_f, n_ff, n_used, t = 256, 16, 2, 1
    n_pairs = 2
    mats_np = [weights("nvfp4", n_ff, in_f, seed=synth.nvfp4_matrix_seed(2, j, p)) for p in range(2) for j in range(n_pairs)]
    mats = [dev(mm) for mm in mats_np]
    ptrs = [mm.data_ptr() for mm in mats]
    ptrs[1] += 4
    y = nan_filled(2, n_pairs, n_ff)
    scales, x = _scales(2 * n_pairs), synth.activations(t, in_f)
    q.qmm_moe_gemv(h, "nvfp4", _table(ptrs), dev(scales), dev(x), y, in_f, n_ff, n_used, t)
    assert q.qmm_sync_status(h) == 4
    yh = y.cpu().numpy()
    assert np.all(np.isnan(yh[0, 1]))
    ref, am = oracle.moe_gate_up("nvfp4", mats_np, scales, x, in_f, n_ff, n_used, t)
    for p, j in [(0, 0), (1, 0), (1, 1)]:
        assert_close(yh[p, j], ref[p, j], am[p, j], FMA_REL, what=f"{p},{j}")
    assert q.qmm_sync_status(h) == 0  # the status was cleared by the read
