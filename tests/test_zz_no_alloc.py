"""qmm_gemm_noalloc: the GEMM entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc at the point where they need a matmul: a
custom device allocator or memory-pool callback (allocating there would
re-enter the allocator), a process whose device memory already belongs to
another framework's pool, or code that runs under a no-allocation-after-start
rule.  Such callers can create neither a handle (qmm_create allocates a status
word) nor a workspace.  qmm_gemm_noalloc keeps its scratch in a static device
array inside the library instead.  This file checks, on two calls in a row,
that it returns what the handle-and-workspace entry point returns, and that
it refuses problems whose scratch would not fit.  It is named to run last.
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import TC_ABS, TC_REL, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu


def _with_workspace(h, fmt, wd, xd, m, k, n):
    d = nan_filled(n, m)
    wsb = q.qmm_gemm_workspace_bytes(fmt, m, k, n)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    q.qmm_gemm(h, fmt, wd, xd, d, m, k, n, ws, wsb)
    assert q.qmm_sync_status(h) == 0
    return d


def test_noalloc_matches_qmm_gemm_on_two_calls_in_a_row(h):
    cases = [("q4_0", 1024, 1024, 512, 2), ("q8_0", 1024, 2048, 300, 3)]
    for fmt, m, k, n, xseed in cases:
        w, x = weights(fmt, m, k), synth.activations(n, k, seed=xseed)
        wd, xd = dev(w), dev(x)
        ref = _with_workspace(h, fmt, wd, xd, m, k, n).cpu().numpy()
        got = nan_filled(n, m)
        q.qmm_gemm_noalloc(fmt, wd, xd, got, m, k, n)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        _, am = oracle.matmul(fmt, w, x, m, k, n)
        # within the tensor-core tolerance of the handle-based result ...
        assert_close(got, ref.astype(np.float64), am, TC_REL, TC_ABS, what=f"noalloc vs qmm_gemm {fmt}")
        # ... and in fact identical: the same kernels on the same inputs
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), fmt


def test_noalloc_rejects_problems_larger_than_its_scratch():
    m, k, n = 64, 4096, 1024  # the f16 copy of X needs 8 MiB, more than the scratch holds
    assert n * k * 2 > q.NOALLOC_SCRATCH_BYTES - 256
    w = dev(weights("q8_0", m, k))
    x = torch.zeros(n, k, dtype=torch.float32, device="cuda")
    d = torch.empty(n, m, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_noalloc("q8_0", w, x, d, m, k, n)
    assert e.value.status == 8  # QMM_ERR_WORKSPACE
