"""qmm_gemv (and qmm_gemm at n <= 8) against the oracle: |gpu - exact| <= 1e-5 * sum|W*X|."""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, FORMATS, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu


def _gemv(h, fmt, w, x, m, k, n):
    dst = nan_filled(n, m)
    q.qmm_gemv(h, fmt, dev(w), dev(x), dst, m, k, n)
    assert q.qmm_sync_status(h) == 0
    return dst.cpu().numpy()


@pytest.mark.parametrize("n", range(1, 9))
@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_every_n(h, fmt, n):
    m, k = 67, 512  # ragged row count (not a multiple of the rows per CTA)
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(_gemv(h, fmt, w, x, m, k, n), ref, am, FMA_REL, what=f"{fmt} n={n}")


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("m,k", [(4608, 1024), (1024, 4608)])
@pytest.mark.parametrize("fmt", ["q4_k", "q8_0"])
def test_gemv_decode_workload(h, fmt, m, k, n):
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(_gemv(h, fmt, w, x, m, k, n), ref, am, FMA_REL, what=f"{fmt} {m}x{k} n={n}")


# shapes whose plans split k over clusters of 1 to 8 CTAs, with a ragged last
# row block, and every n class of the register layout
@pytest.mark.parametrize("n", [1, 3, 5, 8])
@pytest.mark.parametrize("fmt,m,k", [("q6_k", 1001, 4608), ("q4_0", 333, 6144), ("nvfp4", 517, 2560),
                                     ("q8_0", 2050, 1536), ("q4_k", 97, 9216), ("q8_0", 5, 512)])
def test_gemv_split_k_plans(h, fmt, m, k, n):
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(_gemv(h, fmt, w, x, m, k, n), ref, am, FMA_REL, what=f"{fmt} {m}x{k} n={n}")


@pytest.mark.parametrize("fmt", ["q4_0", "q6_k", "nvfp4", "f32"])
def test_gemv_other_formats_full_shape(h, fmt):
    m, k, n = 1024, 4608, 3
    w, x = weights(fmt, m, k), synth.activations(n, k)
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(_gemv(h, fmt, w, x, m, k, n), ref, am, FMA_REL, what=fmt)


@pytest.mark.parametrize("k", [1, 7, 37, 100])
def test_gemv_f32_ragged_k(h, k):
    m, n = 33, 5
    w, x = weights("f32", m, k), synth.activations(n, k)
    ref, am = oracle.matmul("f32", w, x, m, k, n)
    assert_close(_gemv(h, "f32", w, x, m, k, n), ref, am, FMA_REL, what=f"k={k}")


def test_gemm_small_n_is_the_gemv(h):
    m, k, n = 300, 1024, 6
    w, x = dev(weights("q4_k", m, k)), dev(synth.activations(n, k))
    a, b = nan_filled(n, m), nan_filled(n, m)
    q.qmm_gemv(h, "q4_k", w, x, a, m, k, n)
    q.qmm_gemm(h, "q4_k", w, x, b, m, k, n)
    assert q.qmm_sync_status(h) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gemv_is_deterministic(h):
    m, k, n = 4608, 1024, 8
    w, x = dev(weights("q8_0", m, k)), dev(synth.activations(n, k))
    outs = []
    for _ in range(3):
        d = nan_filled(n, m)
        q.qmm_gemv(h, "q8_0", w, x, d, m, k, n)
        outs.append(d)
    assert q.qmm_sync_status(h) == 0
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))


def test_gemv_rejects_bad_arguments(h):
    m, k = 64, 64
    w, x, d = dev(weights("q8_0", m, k)), dev(synth.activations(9, k)), nan_filled(9, m)
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemv(h, "q8_0", w, x, d, m, k, 9)
    assert e.value.status == 3  # n > 8
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemv(h, "q8_0", w, x, d, m, 48, 1)
    assert e.value.status == 3  # k not a whole block
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemv(h, "q8_0", w.data_ptr() + 2, x, d, m, k, 1)
    assert e.value.status == 4  # misaligned
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemv(h, "q8_0", w, x, x, m, k, 1)
    assert e.value.status == 9  # output overlaps input
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemv(h, 17, w, x, d, m, k, 1)
    assert e.value.status == 1
