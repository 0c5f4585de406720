"""Pins of the CPU oracle to values fixed outside it (no GPU needed).

Each check would fail on a plausible mistake in the oracle: a wrong field
offset or nibble order (hand-derived golden blocks), a dropped sign (negative
scales), a wrong exponent bias or subnormal rule (exhaustive code tables
against numpy / torch), a dropped or extra term or a transposed operand in the
product (one-hot permutation, exact integer matmul, library matmul).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _same(a, b):
    """Equal values with the same sign of zero, or both NaN."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


# ---- scalar codes ------------------------------------------------------------

def test_fp16_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    got = oracle.fp16(codes)
    want = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_fp16_subnormal_and_specials():
    # exponent field 0 is mantissa * 2^-24 (hrx-rs patch_bench.rs, fn float)
    assert oracle.fp16([0x0001])[0] == 2.0 ** -24
    assert oracle.fp16([0x03FF])[0] == 1023 * 2.0 ** -24
    assert oracle.fp16([0x7BFF])[0] == 65504.0
    assert oracle.fp16([0xFC00])[0] == -math.inf


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(got[c], want[c]), (c, got[c], want[c])


def test_e4m3_scale_bytes_of_the_moe_workload():
    # (r & 7) | 0x38 gives 1.0, 1.125, ..., 1.875 (memra synth_rows)
    got = oracle.e4m3([0x38 | r for r in range(8)])
    assert list(got) == [1.0 + r / 8 for r in range(8)]


def test_e2m1_all_codes_match_ocp_table():
    table = read_golden("e2m1_ocp.txt")
    assert len(table) == 16
    got = oracle.e2m1([c for c, _ in table])
    for (c, v), g in zip(table, got):
        assert _same(g, v), (c, g, v)


# ---- block decoders ----------------------------------------------------------

@pytest.mark.parametrize("fname,fmt", [("q4_0_blocks.txt", "q4_0"), ("q8_0_blocks.txt", "q8_0")])
def test_whole_blocks_match_hand_values(fname, fmt):
    blocks = read_golden(fname)
    assert blocks
    for blk in blocks:
        got = oracle.decode(fmt, np.frombuffer(blk["bytes"], np.uint8), 1, 32)[0]
        for e, (g, w) in enumerate(zip(got, blk["values"])):
            assert _same(g, w), (fname, e, g, w)


@pytest.mark.parametrize("fname,fmt,k", [("q4_k_block.txt", "q4_k", 256), ("q6_k_block.txt", "q6_k", 256),
                                         ("nvfp4_group.txt", "nvfp4", 64)])
def test_block_spot_values_match_hand_values(fname, fmt, k):
    (blk,) = read_golden(fname)
    assert len(blk["bytes"]) == oracle.block_bytes(fmt)
    got = oracle.decode(fmt, np.frombuffer(blk["bytes"], np.uint8), 1, k)[0]
    assert len(blk["at"]) >= 8
    for e, w in blk["at"].items():
        assert got[e] == w, (fname, e, got[e], w)


def _pack_q4k_scales(sc, mn):
    """Independent packer for the 12 Q4_K scale bytes (the inverse direction of
    the oracle's unpacking, written bit field by bit field)."""
    out = [0] * 12
    for j in range(4):
        out[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        out[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        out[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return out


def test_q4k_every_scale_and_min_round_trips():
    # For each sub-block and each 6-bit value, a block whose nibbles are all 1
    # and d = 1, dmin = 0 decodes to the sub-block's scale; with nibbles 0 and
    # dmin = -1 it decodes to its min.  Other sub-blocks get a different value.
    rng = np.random.default_rng(7)
    for trial in range(64):
        sc = list(rng.integers(0, 64, 8))
        mn = list(rng.integers(0, 64, 8))
        scales = _pack_q4k_scales(sc, mn)
        ones = bytes([0x00, 0x3C, 0x00, 0x00] + scales + [0x11] * 128)
        got = oracle.decode("q4_k", np.frombuffer(ones, np.uint8), 1, 256)[0]
        for j in range(8):
            assert np.all(got[32 * j:32 * j + 32] == sc[j]), (trial, j)
        zeros = bytes([0x00, 0x3C, 0x00, 0xBC] + scales + [0x00] * 128)
        got = oracle.decode("q4_k", np.frombuffer(zeros, np.uint8), 1, 256)[0]
        for j in range(8):
            assert np.all(got[32 * j:32 * j + 32] == mn[j]), (trial, j)


def test_q4k_nibble_positions():
    # A single nonzero nibble anywhere lands on exactly one element: byte i of
    # the nibble area feeds element 64*(i//32) + i%32 (low) and +32 (high).
    for i in range(128):
        for high in (0, 1):
            qs = [0] * 128
            qs[i] = 0x50 if high else 0x05
            sc = _pack_q4k_scales([1] * 8, [0] * 8)
            b = bytes([0x00, 0x3C, 0x00, 0x00] + sc + qs)
            got = oracle.decode("q4_k", np.frombuffer(b, np.uint8), 1, 256)[0]
            e = 64 * (i // 32) + i % 32 + 32 * high
            want = np.zeros(256)
            want[e] = 5.0
            assert np.array_equal(got, want), (i, high)


def test_q6k_bit_positions():
    # Setting one low nibble or one high 2-bit pair moves exactly one element
    # away from -32 (all-zero codes, scales 1, d = 1).
    base_ql, base_qh = [0] * 128, [0] * 64
    sc = [1] * 16

    def decode(ql, qh):
        b = bytes(ql + qh + sc + [0x00, 0x3C])
        return oracle.decode("q6_k", np.frombuffer(b, np.uint8), 1, 256)[0]

    for i in range(128):
        for hi_nib in (0, 1):
            ql = list(base_ql)
            ql[i] = 0x30 if hi_nib else 0x03
            got = decode(ql, base_qh)
            h, rem = divmod(i, 64)
            s = (rem >= 32) + 2 * hi_nib
            e = 128 * h + 32 * s + rem % 32
            want = np.full(256, -32.0)
            want[e] = -29.0
            assert np.array_equal(got, want), (i, hi_nib)
    for i in range(64):
        for s in range(4):
            qh = list(base_qh)
            qh[i] = 1 << (2 * s)
            got = decode(base_ql, qh)
            h, l = divmod(i, 32)
            e = 128 * h + 32 * s + l
            want = np.full(256, -32.0)
            want[e] = -16.0
            assert np.array_equal(got, want), (i, s)


def test_q6k_scale_index_and_sign():
    # Scale number i covers the 16 elements the reading assigns to it.
    for i in range(16):
        sc = [0] * 16
        sc[i] = -2
        b = bytes([0] * 128 + [0] * 64 + [s & 0xFF for s in sc] + [0x00, 0x3C])
        got = oracle.decode("q6_k", np.frombuffer(b, np.uint8), 1, 256)[0]
        h, rest = divmod(i, 8)
        s, half = divmod(rest, 2)
        idx = [128 * h + 32 * s + 16 * half + t for t in range(16)]
        want = np.zeros(256)
        want[idx] = 64.0  # -2 * (0 - 32)
        assert np.array_equal(np.abs(got), np.abs(want)), i
        assert np.all(got[idx] == 64.0)


def test_nvfp4_every_code_and_scale_slot():
    for slot in range(4):
        for code in range(16):
            scales = [0x38] * 4
            scales[slot] = 0x3F  # 1.875
            nib = bytes([code | (code << 4)] * 32)
            got = oracle.decode("nvfp4", np.frombuffer(bytes(scales) + nib, np.uint8), 1, 64)[0]
            e2m1 = oracle.e2m1([code])[0]
            want = np.full(64, e2m1)
            want[16 * slot:16 * slot + 16] *= 1.875
            assert np.array_equal(got, want)


def test_row_bytes_match_the_packed_sizes():
    # cera VARIANTS src0_bytes and memra synth_rows (in_f/64 * 36)
    assert oracle.row_bytes("f32", 1024) == 4096
    assert oracle.row_bytes("q4_0", 1024) == 1024 // 32 * 18
    assert oracle.row_bytes("q8_0", 4608) == 4608 // 32 * 34
    assert oracle.row_bytes("q4_k", 4608) == 4608 // 256 * 144
    assert oracle.row_bytes("q6_k", 1024) == 840
    assert oracle.row_bytes("nvfp4", 4096) == 2304
    assert oracle.row_bytes("q4_k", 1000) == 0


# ---- dequant -----------------------------------------------------------------

def test_dequant_is_the_decoded_value_rounded_once():
    import synth
    for fmt, k in [("q4_0", 64), ("q8_0", 64), ("q4_k", 256), ("q6_k", 256), ("nvfp4", 128)]:
        m = 8
        w = synth.weights(fmt, m, k, m * oracle.row_bytes(fmt, k))
        exact = oracle.decode(fmt, w, m, k)
        got = oracle.dequant(fmt, w, m, k)
        assert np.array_equal(got, exact.astype(np.float32)), fmt
        # decoded values are exact in f32 except Q4_K's d*sc*q - dmin*min,
        # a difference of two products that can need more than 24 bits
        if fmt != "q4_k":
            assert np.array_equal(got.astype(np.float64), exact), fmt
    w = synth.weights("nvfp4", 2, 64, 72)
    got = oracle.dequant("nvfp4", w, 2, 64, tensor_scale=0.3)
    want = (oracle.decode("nvfp4", w, 2, 64) * float(np.float32(0.3))).astype(np.float32)
    assert np.array_equal(got, want)


# ---- the product -------------------------------------------------------------

def _q8_0_matrix(q, d_code=0x3C00):
    """Pack an int8 matrix [m][k] as Q8_0 with every scale = d_code."""
    m, k = q.shape
    out = bytearray()
    for r in range(m):
        for b in range(k // 32):
            out += bytes([d_code & 0xFF, d_code >> 8]) + q[r, 32 * b:32 * b + 32].astype(np.int8).tobytes()
    return np.frombuffer(bytes(out), np.uint8)


def test_one_hot_permutation_recovers_x():
    # W[j][c] = [c == perm(j)] with m < k: dst[i][j] must be X[i][perm(j)];
    # a transposed operand or an off-by-one index fails.
    m, k, n = 24, 64, 3
    rng = np.random.default_rng(3)
    perm = rng.permutation(k)[:m]
    q = np.zeros((m, k), np.int64)
    q[np.arange(m), perm] = 1
    x = rng.uniform(-1, 1, (n, k)).astype(np.float32)
    dst, am = oracle.matmul("q8_0", _q8_0_matrix(q), x, m, k, n)
    assert np.array_equal(dst, x[:, perm].astype(np.float64))
    assert np.array_equal(am, np.abs(x[:, perm]).astype(np.float64))


def test_q8_0_unit_scale_equals_integer_matmul():
    m, k, n = 16, 96, 5
    rng = np.random.default_rng(11)
    q = rng.integers(-128, 128, (m, k))
    x = rng.integers(-8, 9, (n, k)).astype(np.float32)
    dst, am = oracle.matmul("q8_0", _q8_0_matrix(q), x, m, k, n)
    want = x.astype(np.int64) @ q.T
    assert np.array_equal(dst, want.astype(np.float64))
    assert np.array_equal(am, (np.abs(x.astype(np.int64)) @ np.abs(q).T).astype(np.float64))


@pytest.mark.parametrize("fmt,k", [("f32", 32), ("q4_0", 32), ("q8_0", 32), ("q4_k", 256), ("q6_k", 256),
                                   ("nvfp4", 64)])
def test_tiny_brute_force_against_library_matmul(fmt, k):
    import synth
    m, n = 8, 2
    w = synth.weights(fmt, m, k, m * oracle.row_bytes(fmt, k))
    x = synth.activations(n, k)
    dst, am = oracle.matmul(fmt, w, x, m, k, n)
    wd = oracle.decode(fmt, w, m, k)
    want = x.astype(np.float64) @ wd.T
    assert np.allclose(dst, want, rtol=1e-13, atol=1e-13 * np.abs(want).max())
    assert np.allclose(am, np.abs(x.astype(np.float64)) @ np.abs(wd).T, rtol=1e-13)
    ent, ament = oracle.matmul_entries(fmt, w, x, m, k, n, [0, 1, 1], [7, 0, 3])
    assert np.array_equal(ent, dst[[0, 1, 1], [7, 0, 3]])
    assert np.array_equal(ament, am[[0, 1, 1], [7, 0, 3]])


def test_moe_all_ones_weights_sum_x():
    # Every scale byte 0x38 (1.0) and every code 2 (1.0): W is all ones, so
    # y[p][j][r] = scale[p*n_pairs + j] * sum(x[token(j)]).
    in_f, n_ff, n_used, t = 128, 4, 2, 2
    n_pairs = t * n_used
    grp = bytes([0x38] * 4 + [0x22] * 32)
    mat = np.frombuffer(grp * (n_ff * in_f // 64), np.uint8)
    mats = [mat] * (2 * n_pairs)
    scales = np.array([0.5 + 0.01 * p for p in range(2 * n_pairs)], np.float32)
    x = np.arange(t * in_f, dtype=np.float32).reshape(t, in_f) / 64
    y, am = oracle.moe_gate_up("nvfp4", mats, scales, x, in_f, n_ff, n_used, t)
    for p in range(2):
        for j in range(n_pairs):
            want = float(scales[p * n_pairs + j]) * float(x[j // n_used].astype(np.float64).sum())
            assert np.all(y[p, j] == want)


def test_moe_matches_per_matrix_products():
    import synth
    in_f, n_ff, n_used, t = 128, 16, 3, 1
    n_pairs = t * n_used
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, p), n_ff, in_f)
            for p in range(2) for j in range(n_pairs)]
    scales = np.array([0.5 + 0.01 * p for p in range(2 * n_pairs)], np.float32)
    x = synth.activations(t, in_f)
    y, am = oracle.moe_gate_up("nvfp4", mats, scales, x, in_f, n_ff, n_used, t)
    for p in range(2):
        for j in range(n_pairs):
            wd = oracle.decode("nvfp4", mats[p * n_pairs + j], n_ff, in_f)
            want = float(scales[p * n_pairs + j]) * (wd @ x[0].astype(np.float64))
            assert np.allclose(y[p, j], want, rtol=1e-13, atol=1e-12)
    # distinct matrices give distinct outputs (each pair reads its own matrix)
    assert not np.allclose(y[0, 0], y[0, 1])


# ---- MoE down projection -----------------------------------------------------

_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP E2M1 magnitudes, codes 0-7; code | 8 negates


def test_moe_down_all_ones_weights_sum_h():
    # Every scale byte 0x38 (1.0) and every code 2 (1.0): W_j is all ones, so
    # y[i][r] = sum_u scales[j] * sum(h[j]) with j = i*n_used + u.
    n_ff, gin, n_used, t = 128, 4, 3, 2
    n_pairs = t * n_used
    grp = bytes([0x38] * 4 + [0x22] * 32)
    mat = np.frombuffer(grp * (gin * n_ff // 64), np.uint8)
    scales = np.array([0.5 + 0.01 * j for j in range(n_pairs)], np.float32)
    h = (np.arange(n_pairs * n_ff, dtype=np.float32).reshape(n_pairs, n_ff) - 300) / 64
    y, am = oracle.moe_down("nvfp4", [mat] * n_pairs, scales, h, n_ff, gin, n_used, t)
    hs = h.astype(np.float64).sum(axis=1)
    for i in range(t):
        want = sum(float(scales[i * n_used + u]) * hs[i * n_used + u] for u in range(n_used))
        assert np.allclose(y[i], want, rtol=1e-15, atol=0)
        want_am = sum(abs(float(scales[i * n_used + u])) * np.abs(h[i * n_used + u].astype(np.float64)).sum()
                      for u in range(n_used))
        assert np.allclose(am[i], want_am, rtol=1e-15, atol=0)


def test_moe_down_matches_hand_decoded_codes():
    # Rows whose 64-weight groups cycle through all 16 E2M1 codes with E4M3
    # scales 1.0 / 2.0 (0x38 / 0x40): the expected product comes from the OCP
    # table above, not from the oracle's decoder.
    n_ff, gin, n_used, t = 64, 3, 2, 1
    rng = np.random.default_rng(9)
    mats, wvals = [], []
    for j in range(n_used):
        rows = []
        wj = np.zeros((gin, n_ff))
        for r in range(gin):
            sc = [0x38, 0x40, 0x38, 0x40]
            codes = rng.integers(0, 16, n_ff)
            packed = bytes(int(codes[2 * b]) | (int(codes[2 * b + 1]) << 4) for b in range(32))
            rows.append(bytes(sc) + packed)
            for c in range(n_ff):
                mag = _E2M1[codes[c] & 7] * (-1.0 if codes[c] & 8 else 1.0)
                wj[r, c] = mag * (1.0 if sc[c // 16] == 0x38 else 2.0)
        mats.append(np.frombuffer(b"".join(rows), np.uint8))
        wvals.append(wj)
    scales = np.array([0.75, -1.25], np.float32)
    h = rng.integers(-16, 17, (n_used, n_ff)).astype(np.float32) / 8
    y, _ = oracle.moe_down("nvfp4", mats, scales, h, n_ff, gin, n_used, t)
    want = sum(float(scales[u]) * (wvals[u] @ h[u].astype(np.float64)) for u in range(n_used))
    assert np.array_equal(y[0], want)  # every product and partial sum is exact in f64


def test_moe_down_pair_order_linearity_and_token_separation():
    import synth
    n_ff, gin, n_used, t = 128, 8, 3, 2
    n_pairs = t * n_used
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(0, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = np.array([0.5 + 0.01 * j for j in range(n_pairs)], np.float32)
    h = synth.activations(n_pairs, n_ff)
    y, _ = oracle.moe_down("nvfp4", mats, scales, h, n_ff, gin, n_used, t)
    # reversing the pairs of token 1 (matrix, scale and activation together) leaves y unchanged
    perm = [0, 1, 2, 5, 4, 3]
    y2, _ = oracle.moe_down("nvfp4", [mats[p] for p in perm], scales[perm], h[perm], n_ff, gin, n_used, t)
    assert np.allclose(y2, y, rtol=1e-13, atol=1e-12)
    # y is linear in the pair scales
    y3, _ = oracle.moe_down("nvfp4", mats, 2 * scales, h, n_ff, gin, n_used, t)
    assert np.allclose(y3, 2 * y, rtol=1e-13, atol=1e-12)
    # token 1's activations do not reach token 0's output
    h4 = h.copy()
    h4[n_used:] = 0
    y4, _ = oracle.moe_down("nvfp4", mats, scales, h4, n_ff, gin, n_used, t)
    assert np.array_equal(y4[0], y[0]) and np.all(y4[1] == 0)
    # each pair uses its own matrix: swapping two matrices of token 0 changes y[0]
    y5, _ = oracle.moe_down("nvfp4", [mats[1], mats[0]] + mats[2:], scales, h, n_ff, gin, n_used, t)
    assert not np.allclose(y5[0], y[0])


# ---- NVFP4 V2 rows (codes, then the scale stream) ----------------------------

_E4M3_BY_HAND = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0xB8: -1.0}  # sign | 4-bit exponent (bias 7) | 3-bit mantissa


def test_nvfp4_v2_hand_decoded_row():
    # k = 64: 32 code bytes, then 4 scale bytes; expected values from the OCP
    # E2M1 table and the four E4M3 bytes decoded by hand above
    k = 64
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 16, k)
    code_bytes = bytes(int(codes[2 * j]) | (int(codes[2 * j + 1]) << 4) for j in range(k // 2))
    scale_bytes = bytes([0x38, 0x40, 0x30, 0xB8])
    row = np.frombuffer(code_bytes + scale_bytes, np.uint8)
    assert row.size == oracle.row_bytes("nvfp4_v2", k) == 36
    got = oracle.decode("nvfp4_v2", row, 1, k)[0]
    want = [(_E2M1[c & 7] * (-1.0 if c & 8 else 1.0)) * _E4M3_BY_HAND[scale_bytes[e // 16]]
            for e, c in enumerate(codes)]
    assert np.array_equal(got, np.array(want))


def test_nvfp4_v2_row_sizes():
    assert oracle.block_weights("nvfp4_v2") == 32 and oracle.block_bytes("nvfp4_v2") == 18
    assert oracle.row_bytes("nvfp4_v2", 32) == 18
    assert oracle.row_bytes("nvfp4_v2", 4096) == oracle.row_bytes("nvfp4", 4096) == 2304
    assert oracle.row_bytes("nvfp4_v2", 48) == 0


def test_nvfp4_repack_v2_is_the_split_of_the_groups():
    import synth
    m, k = 5, 256
    v1 = synth.nvfp4_rows(0x5151, m, k)
    v2 = oracle.nvfp4_repack_v2(v1, m, k)
    # the same split restated with numpy reshapes: per row, every group's 32
    # code bytes in group order, then every group's 4 scale bytes
    grp = v1.reshape(m, k // 64, 36)
    want = np.concatenate([grp[:, :, 4:].reshape(m, -1), grp[:, :, :4].reshape(m, -1)], axis=1).reshape(-1)
    assert np.array_equal(v2, want)
    # the V2 rows hold the same values
    assert np.array_equal(oracle.decode("nvfp4_v2", v2, m, k), oracle.decode("nvfp4", v1, m, k))
    x = synth.activations(3, k)
    a, am = oracle.matmul("nvfp4", v1, x, m, k, 3)
    b, bm = oracle.matmul("nvfp4_v2", v2, x, m, k, 3)
    assert np.array_equal(a, b) and np.array_equal(am, bm)
    with pytest.raises(ValueError):
        oracle.nvfp4_repack_v2(v1[:36], 1, 32)  # k must be a multiple of 64


# ---- Q8_1 activation blocks (int8 codes, one float32 scale per 32 values) ----


def test_q8_1_hand_block():
    # amax 127 gives d = 1, so every code is its value rounded, halves away from zero
    x = np.zeros((1, 64), np.float32)
    x[0, :8] = [127.0, -63.5, 0.5, -0.5, 1.49, -2.5, 126.6, 0.0]
    q, d = oracle.quantize_q8_1(x, 1, 64)
    assert q[0, :8].tolist() == [127, -64, 1, -1, 1, -3, 127, 0]
    assert np.all(q[0, 8:] == 0)
    assert d.tolist() == [[1.0, 0.0]]  # the all-zero second block has scale 0


def test_q8_1_block_boundaries_and_scales():
    # block 0 peaks at 127/8 (d = 1/8), block 1 at 127*4 (d = 4): both exact
    # in binary, so x/d is exact and only the half-away rounding acts; index 40
    # lies in block 1
    x = np.zeros((1, 64), np.float32)
    x[0, 3] = 127 / 8
    x[0, 5] = 0.0625      # x/d = 0.5  -> 1
    x[0, 6] = -0.1875     # x/d = -1.5 -> -2
    x[0, 40] = -127 * 4
    x[0, 41] = 6.0        # x/d = 1.5  -> 2
    x[0, 42] = -10.0      # x/d = -2.5 -> -3
    q, d = oracle.quantize_q8_1(x, 1, 64)
    assert d.tolist() == [[0.125, 4.0]]
    assert (q[0, 3], q[0, 5], q[0, 6]) == (127, 1, -2)
    assert (q[0, 40], q[0, 41], q[0, 42]) == (-127, 2, -3)


def test_q8_1_invariants_on_random_rows():
    import synth
    rows, k = 4, 4096
    x = synth.activations(rows, k)
    q, d = oracle.quantize_q8_1(x, rows, k)
    xb = x.reshape(rows, k // 32, 32).astype(np.float64)
    qb = q.reshape(rows, k // 32, 32).astype(np.float64)
    db = d.astype(np.float64)[:, :, None]
    assert np.all(np.abs(qb) <= 127)
    assert np.all(np.abs(qb).max(axis=2) == 127)  # the block's largest value maps to +-127
    assert np.all(np.abs(xb - qb * db) <= 0.5 * db * (1 + 1e-6))


def test_moe_gate_up_q8_equals_the_float_path_on_exact_activations():
    import synth
    # integer activations with +-127 in every block: d = 1 and q = x, so the
    # Q8_1 product must equal the pinned float product exactly
    in_f, n_ff, n_used, t = 128, 16, 2, 2
    n_pairs = n_used * t
    rng = np.random.default_rng(5)
    x = rng.integers(-127, 128, (t, in_f)).astype(np.float32)
    x[:, ::32] = 127.0
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(3, j, p), n_ff, in_f) for p in range(2) for j in range(n_pairs)]
    scales = np.array([0.5 + 0.01 * p for p in range(2 * n_pairs)], np.float32)
    q, d = oracle.quantize_q8_1(x, t, in_f)
    assert np.all(d == 1.0) and np.array_equal(q.astype(np.float32), x)
    y8, a8 = oracle.moe_gate_up_q8("nvfp4", mats, scales, q, d, in_f, n_ff, n_used, t)
    yf, af = oracle.moe_gate_up("nvfp4", mats, scales, x, in_f, n_ff, n_used, t)
    assert np.array_equal(y8, yf) and np.array_equal(a8, af)


def test_moe_gate_up_q8_all_ones_weights():
    # W all ones: y = scale * sum_c q[c] * d[c // 32]
    in_f, n_ff, n_used, t = 128, 4, 1, 1
    grp = bytes([0x38] * 4 + [0x22] * 32)
    mat = np.frombuffer(grp * (n_ff * in_f // 64), np.uint8)
    x = ((np.arange(in_f, dtype=np.float32) - 50) / 7).reshape(1, in_f)
    q, d = oracle.quantize_q8_1(x, 1, in_f)
    scales = np.array([0.75, -1.5], np.float32)
    y, _ = oracle.moe_gate_up_q8("nvfp4", [mat, mat], scales, q, d, in_f, n_ff, n_used, t)
    s = sum(float(q[0, c]) * float(d[0, c // 32]) for c in range(in_f))
    assert np.allclose(y[0, 0], 0.75 * s, rtol=1e-15, atol=0) and np.allclose(y[1, 0], -1.5 * s, rtol=1e-15, atol=0)


def test_moe_down_q8_equals_the_float_path_on_exact_activations():
    import synth
    # integer activations with +-127 in every block: d = 1 and q = h, so the
    # Q8_1 down projection must equal the pinned float one exactly
    n_ff, gin, n_used, t = 128, 8, 3, 2
    n_pairs = n_used * t
    rng = np.random.default_rng(6)
    h = rng.integers(-127, 128, (n_pairs, n_ff)).astype(np.float32)
    h[:, ::32] = -127.0
    mats = [synth.nvfp4_rows(synth.nvfp4_matrix_seed(4, j, 2), gin, n_ff) for j in range(n_pairs)]
    scales = np.array([0.5 + 0.01 * j for j in range(n_pairs)], np.float32)
    q, d = oracle.quantize_q8_1(h, n_pairs, n_ff)
    assert np.all(d == 1.0) and np.array_equal(q.astype(np.float32), h)
    y8, a8 = oracle.moe_down_q8("nvfp4", mats, scales, q, d, n_ff, gin, n_used, t)
    yf, af = oracle.moe_down("nvfp4", mats, scales, h, n_ff, gin, n_used, t)
    assert np.array_equal(y8, yf) and np.array_equal(a8, af)
    # a scale of 2 on one pair's blocks doubles that pair's share exactly
    d2 = d.copy()
    d2[1] = 2.0
    y9, _ = oracle.moe_down_q8("nvfp4", mats, scales, q, d2, n_ff, gin, n_used, t)
    h2 = h.copy()
    h2[1] *= 2
    yg, _ = oracle.moe_down("nvfp4", mats, scales, h2, n_ff, gin, n_used, t)
    assert np.array_equal(y9, yg)


# ---- NVFP4 activations for the block-scaled tensor-core product -------------

def _e2m1v(c):
    return float(oracle.e2m1([c])[0])


def _e4m3v(c):
    return float(oracle.e4m3([c])[0])


def _e2m1_rounding_cases():
    cases = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_rounding.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                v, c = line.split()
                cases.append((float(v), int(c)))
    return cases


def test_e2m1_rn_hand_rounded_values():
    cases = _e2m1_rounding_cases()
    assert len(cases) >= 20
    for v, code in cases:
        assert oracle.e2m1_rn(v) == code, (v, code)


def test_e2m1_rn_is_the_identity_on_the_grid():
    for c in range(16):
        v = _e2m1v(c)
        got = oracle.e2m1_rn(v)
        assert got == c or (c in (0, 8) and got in (0, 8) and math.copysign(1, v) == (-1 if got == 8 else 1)), c


def test_e4m3_rn_identity_midpoints_and_saturation():
    # every finite positive E4M3 value maps to its own code; the midpoint of
    # two neighbours (exact in float32) maps to the code with mantissa bit 0,
    # and a hair above or below it to the nearer one
    vals = [_e4m3v(c) for c in range(0x7F)]
    for c in range(0x7F):
        assert oracle.e4m3_rn(vals[c]) == c, c
    for c in range(0x7E):
        mid = np.float32((vals[c] + vals[c + 1]) / 2)
        assert float(mid) == (vals[c] + vals[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_rn(float(mid)) == even, hex(c)
        up, down = np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))
        assert oracle.e4m3_rn(float(up)) == c + 1 and oracle.e4m3_rn(float(down)) == c, hex(c)
    assert oracle.e4m3_rn(448.0) == 0x7E and oracle.e4m3_rn(1e30) == 0x7E and oracle.e4m3_rn(0.0) == 0


def _v2_block(row, k, b):
    """(scale code, 16 codes) of block b of one V2 row."""
    codes = [(row[(16 * b + j) // 2] >> (4 * ((16 * b + j) % 2))) & 15 for j in range(16)]
    return int(row[k // 2 + b]), codes


def test_quantize_nvfp4_hand_blocks():
    k = 64
    x = np.zeros((1, k), np.float32)
    # block 0: amax 6 -> amax/6 = 1.0 exactly, E4M3 0x38; the values are on the grid
    x[0, :6] = [6.0, -3.0, 1.5, 0.5, 0.0, -0.25]
    # block 1: the same values doubled -> scale 2.0 (0x40), the same codes
    x[0, 16:22] = [12.0, -6.0, 3.0, 1.0, 0.0, -0.5]
    # block 2: all zeros -> scale 0 and zero codes
    # block 3: amax 1 -> 1/6 rounds to 1.375 * 2^-3 = 0.171875 (0x23); 1/0.171875
    # = 5.818... rounds to 6 (code 7), 0.5/0.171875 = 2.909... to 3 (code 5)
    x[0, 48:51] = [1.0, 0.5, -0.1]
    row = oracle.quantize_nvfp4_v2(x, 1, k)
    assert row.size == k // 32 * 18
    assert _v2_block(row, k, 0) == (0x38, [7, 13, 3, 1, 0, 8] + [0] * 10)
    assert _v2_block(row, k, 1) == (0x40, [7, 13, 3, 1, 0, 8] + [0] * 10)
    assert _v2_block(row, k, 2) == (0x00, [0] * 16)
    # -0.1 / 0.171875 = -0.58 -> -0.5 (code 9)
    assert _v2_block(row, k, 3) == (0x23, [7, 5, 9] + [0] * 13)


def test_quantize_nvfp4_round_trip_and_error_bound_on_random_rows():
    rng = np.random.default_rng(11)
    rows, k = 5, 256
    x = rng.uniform(-1, 1, (rows, k)).astype(np.float32)
    x[1] *= 40.0
    x[2, :16] = 0.0
    q = oracle.quantize_nvfp4_v2(x, rows, k)
    xq = oracle.dequant("nvfp4_v2", q, rows, k)
    rb = k // 32 * 18
    for r in range(rows):
        row = q[r * rb:(r + 1) * rb]
        for b in range(k // 16):
            sc, codes = _v2_block(row, k, b)
            s = _e4m3v(sc)
            blk = x[r, 16 * b:16 * b + 16].astype(np.float64)
            amax = np.abs(blk).max()
            # the scale is the E4M3 value nearest amax/6: no code is nearer
            t = float(np.float32(amax) / np.float32(6))
            assert all(abs(_e4m3v(c) - t) >= abs(s - t) for c in range(0x7F))
            for j in range(16):
                v = blk[j]
                got = xq[r, 16 * b + j]
                assert got == _e2m1v(codes[j]) * s
                if s == 0:
                    assert got == 0
                    continue
                a = abs(v) / s
                # E2M1 gap at this magnitude (0.5 below 2, 1 below 4, 2 above);
                # past 6 the value saturates
                gap = 0.5 if a < 2 else (1.0 if a < 4 else 2.0)
                assert abs(v - got) <= (gap / 2) * s * (1 + 1e-6) or (a > 6 and abs(got) == 6 * s)
    # values already on the grid with scale 1 come back exactly
    g = np.array([[6, -4, 3, -2, 1.5, -1, 0.5, 0, 6, 4, -3, 2, -1.5, 1, -0.5, 0]], np.float32)
    assert np.array_equal(oracle.dequant("nvfp4_v2", oracle.quantize_nvfp4_v2(g.repeat(2, 1), 1, 32), 1, 32),
                          g.repeat(2, 1))
