"""The tensor-core GEMM (qmm_gemm, n > 8) against the oracle.

Tolerance |gpu - exact| <= 2e-3 * sum|W*X| + 1e-6 per element (f16 / tf32
operands, fp32 accumulation).  The exact-arithmetic cases build W and X whose
products and partial sums are all exactly representable, so the GPU result
must equal the oracle bit for bit whatever the summation order: a wrong tile
mapping, swizzle or transposition cannot hide inside the tolerance.
"""
import math

import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FORMATS, TC_ABS, TC_REL, assert_bitexact, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu

LFM2_SHAPES = {"ffn_gate": (4608, 1024), "ffn_down": (1024, 4608), "conv_in": (3072, 1024), "attn_out": (1024, 1024)}
BM, BN = 128, 256


def _gemm(h, fmt, w, x, m, k, n, dst=None):
    wd, xd = (w if torch.is_tensor(w) else dev(w)), (x if torch.is_tensor(x) else dev(x))
    if dst is None:
        dst = nan_filled(n, m)
    ws_bytes = q.qmm_gemm_workspace_bytes(fmt, m, k, n)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    q.qmm_gemm(h, fmt, wd, xd, dst, m, k, n, ws if ws_bytes else None, ws_bytes)
    assert q.qmm_sync_status(h) == 0
    return dst


def tile_samples(m, n, per_tile=6, seed=5):
    """Entries covering every 128 x 256 output tile: its corners plus random ones."""
    rng = np.random.default_rng(seed)
    ni, mj = [], []
    for mt in range(math.ceil(m / BM)):
        for nt in range(math.ceil(n / BN)):
            m_lo, m_hi = mt * BM, min(m, mt * BM + BM)
            n_lo, n_hi = nt * BN, min(n, nt * BN + BN)
            for a, b in [(n_lo, m_lo), (n_hi - 1, m_hi - 1), (n_lo, m_hi - 1), (n_hi - 1, m_lo)]:
                ni.append(a)
                mj.append(b)
            ni += list(rng.integers(n_lo, n_hi, per_tile))
            mj += list(rng.integers(m_lo, m_hi, per_tile))
    return np.array(ni), np.array(mj)


@pytest.mark.parametrize("fmt", ["f32", "q4_0", "q8_0"])
def test_correctness_workload_256x256x16(h, fmt):
    m, k, n = 256, 256, 16
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert_close(got, ref, am, TC_REL, TC_ABS, what=fmt)


@pytest.mark.parametrize("m,k,n", [(300, 512, 300), (129, 768, 257), (1, 256, 600), (128, 256, 9), (77, 1280, 513), (100, 2048, 100)])
@pytest.mark.parametrize("fmt", FORMATS)
def test_ragged_tiles(h, fmt, m, k, n):
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert_close(got, ref, am, TC_REL, TC_ABS, what=f"{fmt} {m}x{k}x{n}")


@pytest.mark.parametrize("fmt", ["f32", "q4_0", "q8_0"])
def test_k_not_a_multiple_of_the_stage(h, fmt):
    m, k, n = 200, 96, 100
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(_gemm(h, fmt, w, x, m, k, n).cpu().numpy(), ref, am, TC_REL, TC_ABS, what=fmt)


@pytest.mark.parametrize("shape", list(LFM2_SHAPES))
@pytest.mark.parametrize("fmt", ["f32", "q4_0", "q8_0", "q4_k", "q6_k"])
def test_prefill_workload_sampled(h, fmt, shape):
    m, k = LFM2_SHAPES[shape]
    n = 512
    w, x = weights(fmt, m, k), synth.activations(n, k)
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    ni, mj = tile_samples(m, n)
    ref, am = oracle.matmul_entries(fmt, w, x, m, k, n, ni, mj)
    assert_close(got[ni, mj], ref, am, TC_REL, TC_ABS, what=f"{fmt} {shape}")


# ---- exact arithmetic --------------------------------------------------------

def _exact_weights(fmt, m, k, rng):
    """Packed weights whose decoded values are small multiples of powers of two."""
    nb = k // oracle.block_weights(fmt)
    if fmt == "f32":
        return (rng.integers(-16, 17, (m, k)) / 8).astype(np.float32).view(np.uint8).reshape(-1)
    if fmt == "q8_0":
        blk = np.zeros((m * nb, 34), np.uint8)
        blk[:, 0], blk[:, 1] = 0x00, 0x30  # d = 0.125
        blk[:, 2:] = rng.integers(-16, 17, (m * nb, 32)).astype(np.int8).view(np.uint8)
        return blk.reshape(-1)
    if fmt == "q4_0":
        blk = rng.integers(0, 256, (m * nb, 18)).astype(np.uint8)
        blk[:, 0], blk[:, 1] = 0x00, 0x34  # d = 0.25
        return blk.reshape(-1)
    if fmt == "q4_k":
        blk = rng.integers(0, 256, (m * nb, 144)).astype(np.uint8)
        blk[:, 0:4] = [0x00, 0x38, 0x00, 0x34]  # d = 0.5, dmin = 0.25
        # every 6-bit scale and minimum at most 15 (fields of sub-blocks 0..3
        # below 16, the high bits of sub-blocks 4..7 zero, their low nibbles
        # as drawn): |W| <= 0.5*15*15, so sums over k = 4608 of products with
        # X (multiples of 1/8) stay exact in f32
        blk[:, 4:12] &= 0x0F
        return blk.reshape(-1)
    if fmt == "q6_k":
        blk = rng.integers(0, 256, (m * nb, 210)).astype(np.uint8)
        blk[:, 192:208] = rng.integers(-8, 9, (m * nb, 16)).astype(np.int8).view(np.uint8)
        blk[:, 208], blk[:, 209] = 0x00, 0x2C  # d = 1/16
        return blk.reshape(-1)
    if fmt == "nvfp4":
        blk = rng.integers(0, 256, (m * nb, 36)).astype(np.uint8)
        blk[:, 0:4] = 0x38 | (blk[:, 0:4] & 7)  # scales 1.0 .. 1.875
        return blk.reshape(-1)
    raise ValueError(fmt)


@pytest.mark.parametrize("m,k,n", [(256, 512, 512), (129, 768, 300)])
@pytest.mark.parametrize("fmt", FORMATS)
def test_exact_arithmetic_is_bit_identical(h, fmt, m, k, n):
    rng = np.random.default_rng(17)
    w = _exact_weights(fmt, m, k, rng)
    x = (rng.integers(-8, 9, (n, k)) / 8).astype(np.float32)
    ref, _ = oracle.matmul(fmt, w, x, m, k, n)
    assert np.array_equal(ref, ref.astype(np.float32).astype(np.float64)), "case is not exact in f32"
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert_bitexact(got, ref.astype(np.float32), f"{fmt} {m}x{k}x{n}")


# Full-size exact-arithmetic cases, every output element compared bit for
# bit with the oracle: ffn_gate at n = 512 (one 128-row tile per CTA, no
# split-K), ffn_down at n = 512 (split-K over a cluster of four), and
# 4864 x 512 x 1024, where 38 row tiles x 8 token tiles exceed the 152 SMs
# while 19 two-subtile CTAs x 8 cover them exactly: the launcher takes the
# two-subtile (256-row) CTAs there.
FULL_EXACT = {"ffn_gate": (4608, 1024, 512), "ffn_down": (1024, 4608, 512), "two_subtiles": (4864, 512, 1024)}


@pytest.mark.parametrize("case", list(FULL_EXACT))
@pytest.mark.parametrize("fmt", FORMATS)
def test_exact_arithmetic_full_size_every_element(h, fmt, case):
    m, k, n = FULL_EXACT[case]
    if fmt == "f32" and case == "two_subtiles":
        pytest.skip("f32 weights have no two-subtile variant")
    rng = np.random.default_rng(23)
    w = _exact_weights(fmt, m, k, rng)
    x = (rng.integers(-8, 9, (n, k)) / 8).astype(np.float32)
    ref, _ = oracle.matmul(fmt, w, x, m, k, n)
    assert np.array_equal(ref, ref.astype(np.float32).astype(np.float64)), "case is not exact in f32"
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert_bitexact(got, ref.astype(np.float32), f"{fmt} {case} {m}x{k}x{n}")


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k", "nvfp4"])
def test_prefill_ffn_down_every_element(h, fmt):
    # the split-K path on random packed bytes, every element within tolerance
    m, k = LFM2_SHAPES["ffn_down"]
    n = 512
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    got = _gemm(h, fmt, w, x, m, k, n).cpu().numpy()
    assert_close(got, ref, am, TC_REL, TC_ABS, what=f"{fmt} ffn_down")


def test_gemm_is_deterministic(h):
    m, k, n = 1024, 4608, 512
    w, x = dev(weights("q4_k", m, k)), dev(synth.activations(n, k))
    a = _gemm(h, "q4_k", w, x, m, k, n)
    b = _gemm(h, "q4_k", w, x, m, k, n)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gemm_argument_errors(h):
    m, k, n = 256, 256, 64
    w, x, d = dev(weights("q8_0", m, k)), dev(synth.activations(n, k)), nan_filled(n, m)
    need = q.qmm_gemm_workspace_bytes("q8_0", m, k, n)
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm(h, "q8_0", w, x, d, m, k, n, None, 0)
    assert e.value.status == 8
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm(h, "q8_0", w, x, d, m, k, n, ws, need - 1)
    assert e.value.status == 8
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm(h, "q8_0", w, x, d, m, k, n, ws.data_ptr() + 8, need)
    assert e.value.status == 4
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm(h, "q8_0", w, x, d, m, k, n, x, need)
    assert e.value.status == 9
    wf, xf = dev(weights("f32", m, 30)), dev(synth.activations(n, 30))
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm(h, "f32", wf, xf, d, m, 30, n)
    assert e.value.status == 3  # tf32 path needs k % 4 == 0
