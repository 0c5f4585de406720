"""The block-scaled FP4 prefill path against the oracle.

qmm_quantize_nvfp4 must reproduce the oracle's NVFP4 activation bytes bit for
bit (codes and scales are decided in float32 on both sides).  qmm_gemm_fp4
must equal the oracle bit for bit where every product and partial sum is
exact (E2M1 codes with power-of-two E4M3 scales that differ per row and per
block, so a wrong lane, column or byte of the scale layout cannot hide), and
stay within the tensor-core tolerance 2e-3 * sum|W*Xq| + 1e-6 of the exact
product on the quantized activation elsewhere.
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import TC_ABS, TC_REL, assert_bitexact, assert_close, dev, nan_filled

pytestmark = pytest.mark.gpu

LFM2_SHAPES = {"ffn_gate": (4608, 1024), "ffn_down": (1024, 4608), "conv_in": (3072, 1024), "attn_out": (1024, 1024)}


def _v2_bytes(rows, k):
    return rows * q.qmm_row_bytes("nvfp4_v2", k)


def _quantize_gpu(h, x, rows, k):
    xq = torch.full((_v2_bytes(rows, k),), 0xA5, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_nvfp4(h, dev(np.ascontiguousarray(x, np.float32)), xq, rows, k)
    assert q.qmm_sync_status(h) == 0
    return xq


def _gemm_fp4(h, w, xq, m, k, n):
    wd = w if torch.is_tensor(w) else dev(w)
    xd = xq if torch.is_tensor(xq) else dev(xq)
    d = nan_filled(n, m)
    q.qmm_gemm_fp4(h, wd, xd, d, m, k, n)
    assert q.qmm_sync_status(h) == 0
    return d.cpu().numpy()


def _v2_weights(m, k, seed):
    v1 = synth.nvfp4_rows(seed, m, k)
    return oracle.nvfp4_repack_v2(v1, m, k)


# ---- the activation quantizer ----------------------------------------------------

@pytest.mark.parametrize("rows,k", [(1, 256), (512, 1024), (37, 4608)])
def test_quantize_nvfp4_is_bitexact(h, rows, k):
    x = synth.activations(rows, k, seed=3)
    x[0, :16] *= 30.0  # one block with a large scale
    got = _quantize_gpu(h, x, rows, k).cpu().numpy()
    assert np.array_equal(got, oracle.quantize_nvfp4_v2(x, rows, k))


def test_quantize_nvfp4_ties_saturation_and_zero_blocks(h):
    k = 256
    x = np.zeros((2, k), np.float32)
    # block 0: amax 6 (scale exactly 1): every E2M1 midpoint, both signs
    x[0, :16] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -0.1]
    # block 1: amax/6 = 1.0625, an E4M3 midpoint (goes to 1.0, the even code)
    x[0, 16:20] = [6.375, 1.0, -2.0, 0.3]
    # block 2: amax 3000 -> 500, saturates to 448
    x[0, 32:34] = [3000.0, -1.0]
    # block 3: tiny values -> scale rounds to 0, zero codes
    x[0, 48:50] = [1e-6, -2e-6]
    # row 1: a ramp over several magnitudes
    x[1] = np.linspace(-40, 40, k, dtype=np.float32)
    got = _quantize_gpu(h, x, 2, k).cpu().numpy()
    want = oracle.quantize_nvfp4_v2(x, 2, k)
    assert np.array_equal(got, want), np.nonzero(got != want)[0][:16]


# ---- the tensor-core product -------------------------------------------------------

def _exact_v2(rows, k, rng):
    """V2 rows with random E2M1 codes and power-of-two scales (0.5 .. 2) that
    differ from row to row and block to block."""
    rb = k // 32 * 18
    out = np.zeros((rows, rb), np.uint8)
    out[:, : k // 2] = rng.integers(0, 256, (rows, k // 2))
    exps = rng.integers(-1, 2, (rows, k // 16))        # 2^-1 .. 2^1: partial sums stay exact
    out[:, k // 2:] = ((exps + 7) << 3).astype(np.uint8)  # E4M3 with zero mantissa
    return out.reshape(-1)


# one tile; split-K over clusters of 2 and 4 with ragged tiles; 144 tiles with
# m % 4 != 0 (no split, stores without the TMA store map); ffn_down's k
@pytest.mark.parametrize("m,k,n", [(128, 256, 128), (256, 1024, 384), (300, 512, 200), (129, 768, 257),
                                   (1027, 256, 2048), (256, 4608, 256)])
def test_fp4_exact_arithmetic_is_bit_identical(h, m, k, n):
    rng = np.random.default_rng(m + k + n)
    w = _exact_v2(m, k, rng)
    xq = _exact_v2(n, k, rng)
    xdq = oracle.dequant("nvfp4_v2", xq, n, k)
    ref, _ = oracle.matmul("nvfp4_v2", w, xdq, m, k, n)
    assert np.array_equal(ref, ref.astype(np.float32).astype(np.float64)), "case is not exact in f32"
    got = _gemm_fp4(h, w, xq, m, k, n)
    assert_bitexact(got, ref.astype(np.float32), f"fp4 exact {m}x{k}x{n}")


@pytest.mark.parametrize("shape", list(LFM2_SHAPES))
def test_fp4_prefill_workload_every_element(h, shape):
    # the 512-token shapes: weights from the NVFP4 stream repacked to V2,
    # activations quantized on the GPU (bit-exact with the oracle, checked above)
    m, k = LFM2_SHAPES[shape]
    n = 512
    w = _v2_weights(m, k, 0x4F00 + m)
    x = synth.activations(n, k)
    xq = _quantize_gpu(h, x, n, k)
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_nvfp4_v2(x, n, k))
    got = _gemm_fp4(h, w, xq, m, k, n)
    xdq = oracle.dequant("nvfp4_v2", xq.cpu().numpy(), n, k)
    ref, am = oracle.matmul("nvfp4_v2", w, xdq, m, k, n)
    assert_close(got, ref, am, TC_REL, TC_ABS, what=f"fp4 {shape}")


def test_fp4_is_deterministic(h):
    m, k, n = 512, 1024, 256
    w = dev(_v2_weights(m, k, 0x4F77))
    xq = _quantize_gpu(h, synth.activations(n, k), n, k)
    a, b = _gemm_fp4(h, w, xq, m, k, n), _gemm_fp4(h, w, xq, m, k, n)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_fp4_argument_errors(h):
    m, k, n = 128, 256, 128
    w = dev(_v2_weights(m, k, 1))
    x = dev(synth.activations(n, k))
    xq = torch.zeros(_v2_bytes(n, k), dtype=torch.uint8, device="cuda")
    d = nan_filled(n, m)
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_fp4(h, w, xq, d, m, 192, n)
    assert e.value.status == 3  # k % 256
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_fp4(h, w.data_ptr() + 4, xq, d, m, k, n)
    assert e.value.status == 4
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_fp4(h, w, xq, w, m, k, n)
    assert e.value.status == 9  # dst overlaps W
    with pytest.raises(q.QmmError) as e:
        q.qmm_quantize_nvfp4(h, x, x, n, k)
    assert e.value.status == 9
    with pytest.raises(q.QmmError) as e:
        q.qmm_quantize_nvfp4(h, x, xq, n, 96)
    assert e.value.status == 3
    assert torch.isnan(d).all()
