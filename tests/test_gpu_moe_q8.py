"""The int8-activation (Q8_1) MoE path against the oracle.

qmm_quantize_q8_1 must reproduce the oracle's integer codes and block scales
bit for bit (both decide them in float32 by the same steps).  qmm_moe_gemv_q8
and qmm_moe_down_q8 must be within 1e-5 * sum|W * q*d| of the exact products
on the quantized activation (oracle.moe_gate_up_q8 / moe_down_q8), for the
36-byte NVFP4 groups and the V2 rows.  The fused calls, which quantize inside
the product kernel, must equal the two-call path bit for bit.
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, assert_close, dev, nan_filled

pytestmark = pytest.mark.gpu

H_SEED = 1234


def _scales(count):
    return np.array([0.5 + 0.01 * p for p in range(count)], np.float32)


def _quantize(h, x, rows, k):
    xd = dev(np.ascontiguousarray(x, np.float32).reshape(rows, k))
    qd = torch.full((rows, k), 77, dtype=torch.int8, device="cuda")
    dd = torch.full((rows, k // 32), float("nan"), dtype=torch.float32, device="cuda")
    q.qmm_quantize_q8_1(h, xd, qd, dd, rows, k)
    assert q.qmm_sync_status(h) == 0
    return qd, dd


def _as_fmt(fmt, mats, rows, k):
    return [oracle.nvfp4_repack_v2(a, rows, k) for a in mats] if fmt == "nvfp4_v2" else mats


# ---- the quantizer ---------------------------------------------------------------

@pytest.mark.parametrize("rows,k", [(1, 4096), (8, 2048), (3, 96), (130, 64)])
def test_quantize_q8_1_is_bitexact(h, rows, k):
    x = synth.activations(rows, k, seed=H_SEED)
    qd, dd = _quantize(h, x, rows, k)
    qo, do = oracle.quantize_q8_1(x, rows, k)
    assert np.array_equal(qd.cpu().numpy(), qo)
    assert np.array_equal(dd.cpu().numpy().view(np.uint32), do.view(np.uint32))


def test_quantize_q8_1_special_blocks(h):
    # block 0: amax 127 -> d = 1 exactly, so x = +-2.5 and +-0.5 are ties that
    # round away from zero; block 1: all zeros (d = 0, q = 0); block 2: one
    # tiny value; block 3: mixed magnitudes with a negative maximum
    x = np.zeros((1, 128), np.float32)
    x[0, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.4999999, -126.5, 63.5]
    x[0, 64] = 1e-30
    x[0, 96:100] = [-3.0, 1.0, 0.25, -0.75]
    qd, dd = _quantize(h, x, 1, 128)
    qo, do = oracle.quantize_q8_1(x, 1, 128)
    assert np.array_equal(qd.cpu().numpy(), qo)
    assert np.array_equal(dd.cpu().numpy().view(np.uint32), do.view(np.uint32))
    assert list(qo[0, :8]) == [127, 3, -3, 1, -1, 1, -127, 64]
    assert do[0, 1] == 0.0 and not np.any(qo[0, 32:64])


# ---- gate/up ---------------------------------------------------------------------

def _run_gate_up(h, fmt, mats, scales, qd, dd, in_f, n_ff, n_used, t, ptr_fix=None):
    dm = [dev(a) for a in mats]
    ptrs = [a.data_ptr() for a in dm]
    if ptr_fix:
        ptrs = ptr_fix(ptrs)
    table = torch.tensor(ptrs, dtype=torch.int64, device="cuda")
    y = nan_filled(2, t * n_used, n_ff)
    q.qmm_moe_gemv_q8(h, fmt, table, dev(scales), qd, dd, y, in_f, n_ff, n_used, t)
    return q.qmm_sync_status(h), y.cpu().numpy()


@pytest.mark.parametrize("fmt", ["nvfp4", "nvfp4_v2"])
def test_moe_gate_up_q8_workload(h, fmt):
    # in_f 4096, n_ff 2048, 8 experts, 1 token: the served gate/up shape
    in_f, n_ff, n_used, t = 4096, 2048, 8, 1
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    mats = _as_fmt(fmt, mats, n_ff, in_f)
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f)
    qd, dd = _quantize(h, x, t, in_f)
    st, y = _run_gate_up(h, fmt, mats, scales, qd, dd, in_f, n_ff, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(x, t, in_f)
    ref, am = oracle.moe_gate_up_q8(fmt, mats, scales, qo, do, in_f, n_ff, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"moe q8 {fmt}")


@pytest.mark.parametrize("in_f", [64, 192, 2048, 6144, 8192])
@pytest.mark.parametrize("fmt", ["nvfp4", "nvfp4_v2"])
def test_moe_gate_up_q8_row_lengths_and_tokens(h, fmt, in_f):
    # 1, 3, 32, 96 and 128 groups of 64 per row (idle lanes, one to four
    # groups per lane); ragged n_ff (a partial 16-row stage); two tokens
    n_ff, n_used, t = 37, 3, 2
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(1, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    mats = _as_fmt(fmt, mats, n_ff, in_f)
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f, seed=9)
    qd, dd = _quantize(h, x, t, in_f)
    st, y = _run_gate_up(h, fmt, mats, scales, qd, dd, in_f, n_ff, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(x, t, in_f)
    ref, am = oracle.moe_gate_up_q8(fmt, mats, scales, qo, do, in_f, n_ff, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"{fmt} in_f={in_f}")


def test_moe_gate_up_q8_exact_products(h):
    # E4M3 scales 1.0 and activation blocks with d = 1 (amax 127, integer x):
    # every region sum and every partial sum is an integer below 2^24, so the
    # result equals the oracle's exactly, whatever the summation order
    in_f, n_ff, n_used, t = 512, 64, 2, 1
    n_pairs = n_used * t
    rng = np.random.default_rng(3)
    mats = []
    for _ in range(2 * n_pairs):
        g = rng.integers(0, 256, (n_ff * in_f // 64, 36)).astype(np.uint8)
        g[:, 0:4] = 0x38
        mats.append(g.reshape(-1))
    x = rng.integers(-127, 128, (t, in_f)).astype(np.float32)
    x[:, ::32] = 127.0
    scales = np.ones(2 * n_pairs, np.float32)
    qd, dd = _quantize(h, x, t, in_f)
    st, y = _run_gate_up(h, "nvfp4", mats, scales, qd, dd, in_f, n_ff, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(x, t, in_f)
    assert np.all(do == 1.0)
    ref, _ = oracle.moe_gate_up_q8("nvfp4", mats, scales, qo, do, in_f, n_ff, n_used, t)
    assert np.array_equal(y.astype(np.float64), ref)


def test_moe_gate_up_q8_is_deterministic_and_reports_bad_entries(h):
    in_f, n_ff, n_used, t = 1024, 48, 2, 1
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(2, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f)
    qd, dd = _quantize(h, x, t, in_f)
    _, y1 = _run_gate_up(h, "nvfp4", mats, scales, qd, dd, in_f, n_ff, n_used, t)
    _, y2 = _run_gate_up(h, "nvfp4", mats, scales, qd, dd, in_f, n_ff, n_used, t)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))

    def fix(p):
        p[1] += 4  # misaligned: gate plane, pair 1
        return p

    st, y = _run_gate_up(h, "nvfp4", mats, scales, qd, dd, in_f, n_ff, n_used, t, ptr_fix=fix)
    assert st == 4  # QMM_ERR_ALIGN
    assert np.all(np.isnan(y[0, 1]))
    assert np.array_equal(y[1].view(np.uint32), y1[1].view(np.uint32))
    assert q.qmm_sync_status(h) == 0


def test_q8_argument_errors(h):
    in_f, n_ff = 128, 16
    mats = [dev(synth.nvfp4_rows(synth.nvfp4_matrix_seed(3, j, 0), n_ff, in_f)) for j in range(2)]
    table = torch.tensor([a.data_ptr() for a in mats], dtype=torch.int64, device="cuda")
    scales = dev(_scales(2))
    qd = torch.zeros(1, 16384, dtype=torch.int8, device="cuda")
    dd = torch.zeros(1, 512, dtype=torch.float32, device="cuda")
    y = nan_filled(2, 1, n_ff)
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8(h, "q4_0", table, scales, qd, dd, y, in_f, n_ff, 1, 1)
    assert e.value.status == 2  # NVFP4 only
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8(h, "nvfp4", table, scales, qd, dd, y, 96, n_ff, 1, 1)
    assert e.value.status == 3  # in_f % 64
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8(h, "nvfp4", table, scales, qd, dd, y, q.Q8_MAX_K + 64, n_ff, 1, 1)
    assert e.value.status == 3  # longer than the register plan covers
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8(h, "nvfp4", table, scales, qd.data_ptr() + 4, dd, y, in_f, n_ff, 1, 1)
    assert e.value.status == 4
    x = dev(synth.activations(1, 64))
    with pytest.raises(q.QmmError) as e:
        q.qmm_quantize_q8_1(h, x, qd, dd, 1, 48)
    assert e.value.status == 3  # k % 32
    with pytest.raises(q.QmmError) as e:
        q.qmm_quantize_q8_1(h, x, x.view(torch.int8), dd, 1, 64)
    assert e.value.status == 9  # q overlaps x
    assert np.all(np.isnan(y.cpu().numpy()))


# ---- down projection ------------------------------------------------------------

def _run_down(h, fmt, mats, scales, qd, dd, n_ff, gin, n_used, t):
    dm = [dev(a) for a in mats]
    table = torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")
    y = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda") if wsb else None
    q.qmm_moe_down_q8(h, fmt, table, dev(scales), qd, dd, y, n_ff, gin, n_used, t, ws, wsb)
    return q.qmm_sync_status(h), y.cpu().numpy()


@pytest.mark.parametrize("fmt", ["nvfp4", "nvfp4_v2"])
def test_moe_down_q8_workload(h, fmt):
    # gin 4096, n_ff 2048, 8 experts of one token summed into y
    n_ff, gin, n_used, t = 2048, 4096, 8, 1
    n_pairs = n_used * t
    mats = _as_fmt(fmt, [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, 2), gin, n_ff) for j in range(n_pairs)],
                   gin, n_ff)
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    qd, dd = _quantize(h, hact, n_pairs, n_ff)
    st, y = _run_down(h, fmt, mats, scales, qd, dd, n_ff, gin, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(hact, n_pairs, n_ff)
    ref, am = oracle.moe_down_q8(fmt, mats, scales, qo, do, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"down q8 {fmt}")


@pytest.mark.parametrize("n_used,t", [(1, 3), (3, 2)])
def test_moe_down_q8_tokens(h, n_used, t):
    n_ff, gin = 320, 53
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(4, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED)
    qd, dd = _quantize(h, hact, n_pairs, n_ff)
    st, y = _run_down(h, "nvfp4", mats, scales, qd, dd, n_ff, gin, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(hact, n_pairs, n_ff)
    ref, am = oracle.moe_down_q8("nvfp4", mats, scales, qo, do, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"n_used={n_used} t={t}")


# ---- the fused calls (quantization inside the product kernel) --------------------

def _table(mats):
    dm = [dev(a) for a in mats]
    return dm, torch.tensor([a.data_ptr() for a in dm], dtype=torch.int64, device="cuda")


@pytest.mark.parametrize("fmt,in_f,n_ff,n_used,t", [("nvfp4", 4096, 2048, 8, 1), ("nvfp4_v2", 4096, 2048, 8, 1),
                                                     ("nvfp4", 192, 37, 3, 2), ("nvfp4_v2", 8192, 21, 1, 3),
                                                     ("nvfp4", 64, 16, 2, 1)])
def test_moe_gate_up_q8_fused_equals_quantize_then_product(h, fmt, in_f, n_ff, n_used, t):
    # the served shape and ragged ones (idle lanes, one to four groups per
    # lane, several tokens): bit-identical to the two calls, and within the
    # tolerance of the oracle on the oracle's own quantization
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(5, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    mats = _as_fmt(fmt, mats, n_ff, in_f)
    scales = _scales(2 * n_pairs)
    x = synth.activations(t, in_f, seed=21)
    x[0, :32] *= 40.0  # one block with a large scale
    x[-1, 64:96] = 0.0  # one all-zero block (d = 0)
    qd, dd = _quantize(h, x, t, in_f)
    st, y2 = _run_gate_up(h, fmt, mats, scales, qd, dd, in_f, n_ff, n_used, t)
    assert st == 0
    _, table = _table(mats)
    y1 = nan_filled(2, n_pairs, n_ff)
    q.qmm_moe_gemv_q8_fused(h, fmt, table, dev(scales), dev(x), y1, in_f, n_ff, n_used, t)
    assert q.qmm_sync_status(h) == 0
    y1 = y1.cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    qo, do = oracle.quantize_q8_1(x, t, in_f)
    ref, am = oracle.moe_gate_up_q8(fmt, mats, scales, qo, do, in_f, n_ff, n_used, t)
    assert_close(y1, ref, am, FMA_REL, what=f"fused {fmt} in_f={in_f}")


@pytest.mark.parametrize("fmt,n_ff,gin,n_used,t", [("nvfp4", 2048, 4096, 8, 1), ("nvfp4_v2", 2048, 4096, 8, 1),
                                                    ("nvfp4", 320, 53, 3, 2), ("nvfp4", 128, 40, 1, 3)])
def test_moe_down_q8_fused_equals_quantize_then_product(h, fmt, n_ff, gin, n_used, t):
    n_pairs = n_used * t
    mats = _as_fmt(fmt, [synth.nvfp4_rows(synth.nvfp4_matrix_seed(6, j, 2), gin, n_ff) for j in range(n_pairs)],
                   gin, n_ff)
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED + 1)
    qd, dd = _quantize(h, hact, n_pairs, n_ff)
    st, y2 = _run_down(h, fmt, mats, scales, qd, dd, n_ff, gin, n_used, t)
    assert st == 0
    _, table = _table(mats)
    y1 = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda") if wsb else None
    q.qmm_moe_down_q8_fused(h, fmt, table, dev(scales), dev(hact), y1, n_ff, gin, n_used, t, ws, wsb)
    assert q.qmm_sync_status(h) == 0
    y1 = y1.cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    qo, do = oracle.quantize_q8_1(hact, n_pairs, n_ff)
    ref, am = oracle.moe_down_q8(fmt, mats, scales, qo, do, n_ff, gin, n_used, t)
    assert_close(y1, ref, am, FMA_REL, what=f"fused down {fmt} n_used={n_used} t={t}")


def test_q8_fused_argument_errors(h):
    in_f, n_ff = 128, 16
    mats = [dev(synth.nvfp4_rows(synth.nvfp4_matrix_seed(3, j, 0), n_ff, in_f)) for j in range(2)]
    table = torch.tensor([a.data_ptr() for a in mats], dtype=torch.int64, device="cuda")
    scales = dev(_scales(2))
    x = dev(synth.activations(1, in_f))
    y = nan_filled(2, 1, n_ff)
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8_fused(h, "q8_0", table, scales, x, y, in_f, n_ff, 1, 1)
    assert e.value.status == 2  # NVFP4 only
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8_fused(h, "nvfp4", table, scales, x, y, 96, n_ff, 1, 1)
    assert e.value.status == 3  # in_f % 64
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8_fused(h, "nvfp4", table, scales, x.data_ptr() + 4, y, in_f, n_ff, 1, 1)
    assert e.value.status == 4  # x not 16-byte aligned
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_gemv_q8_fused(h, "nvfp4", table, scales, y, y, in_f, n_ff, 1, 1)
    assert e.value.status == 9  # y overlaps x
    yd = nan_filled(1, 40)
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_down_q8_fused(h, "nvfp4", table, scales, x, yd, 96, 40, 1, 1)
    assert e.value.status == 3  # n_ff % 64
    with pytest.raises(q.QmmError) as e:
        q.qmm_moe_down_q8_fused(h, "nvfp4", table, scales, 0, yd, in_f, 40, 1, 1)
    assert e.value.status == 1  # no activation
    assert np.all(np.isnan(y.cpu().numpy())) and np.all(np.isnan(yd.cpu().numpy()))


# ---- more down-projection shapes: 2 to 16 pairs per token, ragged row
# counts, the longest rows, both layouts ------------------------------------

@pytest.mark.parametrize("fmt,n_ff,gin,n_used,t", [("nvfp4", 2048, 261, 2, 3), ("nvfp4_v2", 1024, 261, 4, 2),
                                                    ("nvfp4", 128, 37, 16, 2), ("nvfp4_v2", 8192, 19, 8, 1)])
def test_moe_down_q8_pair_counts(h, fmt, n_ff, gin, n_used, t):
    n_pairs = n_used * t
    mats = _as_fmt(fmt, [synth.nvfp4_rows(synth.nvfp4_matrix_seed(11, j, 2), gin, n_ff) for j in range(n_pairs)],
                   gin, n_ff)
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED + 4)
    qd, dd = _quantize(h, hact, n_pairs, n_ff)
    st, y = _run_down(h, fmt, mats, scales, qd, dd, n_ff, gin, n_used, t)
    assert st == 0
    qo, do = oracle.quantize_q8_1(hact, n_pairs, n_ff)
    ref, am = oracle.moe_down_q8(fmt, mats, scales, qo, do, n_ff, gin, n_used, t)
    assert_close(y, ref, am, FMA_REL, what=f"down q8 {fmt} n_used={n_used}")
    # the fused call (quantizing inside the kernel) writes the same bits
    _, table = _table(mats)
    y1 = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    q.qmm_moe_down_q8_fused(h, fmt, table, dev(scales), dev(hact), y1, n_ff, gin, n_used, t, ws, wsb)
    assert q.qmm_sync_status(h) == 0
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), y.view(np.uint32))


def test_moe_down_q8_device_table_and_bad_entry(h):
    # 8 pairs x 70 tokens = 560 pairs: pointers and scales from the device
    # table (the kernel copies up to 512); pair 13 (token 1) misaligned:
    # token 1's rows NaN, the other tokens exact
    n_ff, gin, n_used, t = 128, 16, 8, 70
    n_pairs = n_used * t
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(12, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = _scales(n_pairs)
    hact = synth.activations(n_pairs, n_ff, seed=H_SEED + 5)
    qd, dd = _quantize(h, hact, n_pairs, n_ff)
    dm, table = _table(mats)
    ptrs = [a.data_ptr() for a in dm]
    ptrs[13] += 4
    table = torch.tensor(ptrs, dtype=torch.int64, device="cuda")
    y = nan_filled(t, gin)
    wsb = q.qmm_moe_down_workspace_bytes(gin, n_used, t)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    q.qmm_moe_down_q8(h, "nvfp4", table, dev(scales), qd, dd, y, n_ff, gin, n_used, t, ws, wsb)
    assert q.qmm_sync_status(h) == 4
    y = y.cpu().numpy()
    assert np.all(np.isnan(y[1]))
    qo, do = oracle.quantize_q8_1(hact, n_pairs, n_ff)
    ref, am = oracle.moe_down_q8("nvfp4", mats, scales, qo, do, n_ff, gin, n_used, t)
    keep = [i for i in range(t) if i != 1]
    assert_close(y[keep], ref[keep], am[keep], FMA_REL, what="down q8, other tokens")
    assert q.qmm_sync_status(h) == 0
