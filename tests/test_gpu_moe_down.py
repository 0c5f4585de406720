"""qmm_moe_down against the oracle (per-token sum over routed experts of the
scaled down-projection products, memra-engine moe_rows_ceiling_bench.rs)."""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, FORMATS, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu

H_SEED = 1234  # the page's seed of the synthetic per-pair down activations


def _scales(count):
    return np.array([0.5 + 0.01 * p for p in range(count)], np.float32)


def _run_down(h, fmt, mats_np, scales, hact, n_ff, gin, n_used, t, ptr_fix=None):
    mats = [dev(mm) for mm in mats_np]
    ptrs = [mm.data_ptr() for mm in mats]
    if ptr_fix:
        ptrs = ptr_fix(ptrs)
    table = torch.tensor(ptrs, dtype=torch.int64, device="cuda")
    y = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    q.qmm_moe_down(h, fmt, table, dev(scales), dev(hact), y, n_ff, gin, n_used, t, ws, wsb)
    st = q.qmm_sync_status(h)
    return st, y.cpu().numpy()


def test_moe_down_workload(h):
    # n_ff 2048 -> gin 4096, 8 experts, 1 token; each down matrix from its own
    # seeded stream (plane 2 of the page's gate/up/down table)
    n_ff, gin, n_used, t = 2048, 4096, 8, 1
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="moe_down")


def test_moe_down_register_x_path_multi_token(h):
    # n_ff >= 2048 takes the register-X kernel; 3 tokens exercise the combine
    n_ff, gin, n_used, t = 2048, 260, 4, 3
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(1, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="rx")


@pytest.mark.parametrize("fmt", FORMATS)
def test_moe_down_multi_token_every_format(h, fmt):
    n_ff, gin, n_used, t = 512, 101, 3, 2  # ragged gin, the shared-memory X kernel
    n_pairs = n_used * t
    mats = [weights(fmt, gin, n_ff, seed=synth.nvfp4_matrix_seed(2, j, 2)) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    st, y = _run_down(h, fmt, mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down(fmt, mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=fmt)


def test_moe_down_single_expert_needs_no_workspace(h):
    n_ff, gin, n_used, t = 256, 70, 1, 3
    assert q.qmm_moe_down_workspace_bytes(gin, n_used, t) == 0
    mats = [weights("q4_0", gin, n_ff, seed=synth.nvfp4_matrix_seed(3, j, 2)) for j in range(t)]
    scales = _scales(t)
    hact = synth.activations(t, n_ff, seed=H_SEED)
    st, y = _run_down(h, "q4_0", mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down("q4_0", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="n_used=1")


def test_moe_down_table_larger_than_shared_memory_copy(h):
    # 1040 pairs: the kernel reads pointers and scales from the device table
    # instead of its shared-memory copy (which holds up to 1024)
    n_ff, gin, n_used, t = 64, 64, 8, 130
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(4, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="big table")


def test_moe_down_is_deterministic(h):
    n_ff, gin, n_used, t = 2048, 512, 8, 2
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(5, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    _, y1 = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    _, y2 = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_moe_down_bad_table_entry_is_reported(h):
    # a misaligned pointer of pair 1 (token 0): the kernel skips that matrix,
    # token 0's rows come back NaN, token 1 is exact, the status reads ALIGN
    n_ff, gin, n_used, t = 256, 16, 2, 2
    n_pairs = n_used * t
    mats = [weights("nvfp4", gin, n_ff, seed=synth.nvfp4_matrix_seed(6, j, 2)) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)

    def fix(p):
        p[1] += 4
        return p

    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t, ptr_fix=fix)
    assert st == 4
    assert np.all(np.isnan(y[0]))
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y[1], ref[1], am[1], FMA_REL, what="token 1")
    assert q.qmm_sync_status(h) == 0


def test_moe_down_argument_errors(h):
    n_ff, gin, n_used, t = 64, 32, 2, 1
    mats = [dev(weights("nvfp4", gin, n_ff, seed=synth.nvfp4_matrix_seed(7, j, 2))) for j in range(2)]
    table = torch.tensor([m.data_ptr() for m in mats], dtype=torch.int64, device="cuda")
    scales = dev(_scales(2))
    hact = dev(synth.activations(2, n_ff, seed=H_SEED))
    y = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    assert wsb == 256  # 2 * 32 * 4 bytes rounded up to 256
    with pytest.raises(q.QmmError) as e:  # workspace missing
        q.qmm_moe_down(h, "nvfp4", table, scales, hact, y, n_ff, gin, n_used, t)
    assert e.value.status == 8
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError) as e:  # too small
        q.qmm_moe_down(h, "nvfp4", table, scales, hact, y, n_ff, gin, n_used, t, ws, wsb - 16)
    assert e.value.status == 8
    with pytest.raises(q.QmmError) as e:  # n_ff not a multiple of the block
        q.qmm_moe_down(h, "nvfp4", table, scales, hact, y, 96, gin, n_used, t, ws, wsb)
    assert e.value.status == 3
    with pytest.raises(q.QmmError) as e:  # workspace overlapping y
        yb = torch.empty(wsb + t * gin * 4, dtype=torch.uint8, device="cuda")
        q.qmm_moe_down(h, "nvfp4", table, scales, hact, yb[: t * gin * 4].view(torch.float32), n_ff, gin, n_used, t,
                       yb, wsb)
    assert e.value.status == 9
    assert np.all(np.isnan(y.cpu().numpy()))  # nothing was launched


# ---- the grouped register-X kernel (rows of 2048, 4 or 8 pairs per token):
# a stage holds the same rows of all of a token's pair matrices and the
# kernel sums the pairs itself, with no workspace round trip ----------------

@pytest.mark.parametrize("fmt,n_used", [(f, 4) for f in FORMATS] + [("q8_0", 2), ("f32", 8), ("nvfp4", 8)])
def test_moe_down_grouped_every_format(h, fmt, n_used):
    # teams of 128 threads (4 pairs), 256 (2 pairs: 8-weight blocks only) and 64 (8 pairs)
    n_ff, gin, t = 2048, 261, 2  # 261 rows: a partial last stage
    n_pairs = n_used * t
    mats = [weights(fmt, gin, n_ff, seed=synth.nvfp4_matrix_seed(8, j, 2)) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED + 2)
    st, y = _run_down(h, fmt, mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down(fmt, mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"grouped {fmt} n_used={n_used}")


def test_moe_down_grouped_device_table(h):
    # 8 pairs x 40 tokens = 320 pairs: pointers and scales come from the
    # device table, not the kernel's shared-memory copy of the first 256
    n_ff, gin, n_used, t = 2048, 24, 8, 40
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(9, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED + 3)
    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert st == 0
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what="grouped, device table")


def test_moe_down_grouped_bad_table_entry_is_reported(h):
    # pair 5 (token 1) misaligned: token 1's rows NaN, token 0 exact
    n_ff, gin, n_used, t = 2048, 40, 4, 2
    n_pairs = n_used * t
    mats = [weights("nvfp4", gin, n_ff, seed=synth.nvfp4_matrix_seed(10, j, 2)) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)

    def fix(p):
        p[5] += 4
        return p

    st, y = _run_down(h, "nvfp4", mats, scales, hact, n_ff, gin, n_used, t, ptr_fix=fix)
    assert st == 4
    assert np.all(np.isnan(y[1]))
    ref, am = oracle.moe_down("nvfp4", mats, scales, hact, n_ff, gin, n_used, t)
    assert_close(y[0], ref[0], am[0], FMA_REL, what="token 0")
    assert q.qmm_sync_status(h) == 0
