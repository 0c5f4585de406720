"""qmm_gemm_noalloc: the GEMM entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc at the point where they need a matmul: a
custom device allocator or memory-pool callback (allocating there would
re-enter the allocator), a process whose device memory already belongs to
another framework's pool, or code that runs under a no-allocation-after-start
rule.  Such callers can create neither a handle (qmm_create allocates a status
word) nor a workspace.  qmm_gemm_noalloc keeps its scratch in a static device
array inside the library instead.  This file checks, on two calls in a row,
that it returns what the handle-and-workspace entry point returns and what the
oracle computes (tensor-core path for packed and f32 weights, GEMV path for
n <= 8), that device memory does not change around a repeated call in a fresh
process that never created a handle, that its status read works, and that it
refuses problems whose scratch would not fit.  It is named to run last.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import FMA_REL, TC_ABS, TC_REL, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _with_workspace(h, fmt, wd, xd, m, k, n):
    d = nan_filled(n, m)
    wsb = q.qmm_gemm_workspace_bytes(fmt, m, k, n)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    q.qmm_gemm(h, fmt, wd, xd, d, m, k, n, ws if wsb else None, wsb)
    assert q.qmm_sync_status(h) == 0
    return d


# (fmt, m, k, n, x seed): tensor-core path with packed and f32 weights, and
# the GEMV path at both ends of its n range
CASES = [("q4_0", 1024, 1024, 512, 2), ("q8_0", 1024, 2048, 300, 3), ("f32", 640, 512, 200, 4),
         ("q4_k", 1000, 1024, 1, 5), ("q6_k", 777, 512, 8, 6)]


@pytest.mark.parametrize("fmt,m,k,n,xseed", CASES)
def test_noalloc_matches_qmm_gemm_and_the_oracle_on_two_calls_in_a_row(h, fmt, m, k, n, xseed):
    w, x = weights(fmt, m, k), synth.activations(n, k, seed=xseed)
    wd, xd = dev(w), dev(x)
    ref_gpu = _with_workspace(h, fmt, wd, xd, m, k, n).cpu().numpy()
    exact, am = oracle.matmul(fmt, w, x, m, k, n)
    rel, abs_ = (FMA_REL, 0.0) if n <= q.GEMV_MAX_N else (TC_REL, TC_ABS)
    for call in range(2):
        got = nan_filled(n, m)
        q.qmm_gemm_noalloc(fmt, wd, xd, got, m, k, n)
        assert q.qmm_gemm_noalloc_status() == 0
        got = got.cpu().numpy()
        # within the stated tolerance of the exact product ...
        assert_close(got, exact, am, rel, abs_, what=f"noalloc vs oracle {fmt} call {call}")
        # ... and identical to the handle-and-workspace entry point: the same kernels on the same inputs
        assert np.array_equal(got.view(np.uint32), ref_gpu.view(np.uint32)), (fmt, call)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    m, k, n = 64, 4096, 1024  # the f16 copy of X needs 8 MiB, more than the scratch holds
    assert n * k * 2 > q.NOALLOC_SCRATCH_BYTES - 256
    w = dev(weights("q8_0", m, k))
    x = torch.zeros(n, k, dtype=torch.float32, device="cuda")
    d = torch.empty(n, m, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.qmm_gemm_noalloc("q8_0", w, x, d, m, k, n)
    assert e.value.status == 8  # QMM_ERR_WORKSPACE


_FRESH = textwrap.dedent(r"""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np
    import torch
    import gemv_dequant_gemm_gb300 as q
    import oracle
    import synth

    torch.cuda.set_device(0)
    out = []
    for fmt, m, k, n in (("q4_0", 512, 1024, 256), ("q8_0", 300, 512, 4)):
        w = synth.weights(fmt, m, k, m * q.qmm_row_bytes(fmt, k))
        x = synth.activations(n, k, seed=7)
        wd, xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
        d1 = torch.full((n, m), float("nan"), device="cuda")
        d2 = torch.full((n, m), float("nan"), device="cuda")
        torch.cuda.synchronize()
        # first call in this process: sets the device up and loads what it runs
        q.qmm_gemm_noalloc(fmt, wd, xd, d1, m, k, n)
        assert q.qmm_gemm_noalloc_status() == 0
        free0 = torch.cuda.mem_get_info()[0]
        q.qmm_gemm_noalloc(fmt, wd, xd, d2, m, k, n)
        assert q.qmm_gemm_noalloc_status() == 0
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, ("device memory changed around the second call", fmt, free0, free1)
        ref, am = oracle.matmul(fmt, w, x, m, k, n)
        rel, abs_ = (1e-5, 0.0) if n <= 8 else (2e-3, 1e-6)
        for d in (d1, d2):
            err = np.abs(d.cpu().numpy().astype(np.float64) - ref)
            assert np.all(err <= rel * am + abs_), (fmt, float(err.max()))
        out.append(fmt)
    print("fresh-process ok", *out)
""")


def test_noalloc_in_a_fresh_process_without_a_handle_allocates_nothing_on_repeat():
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT)], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert "fresh-process ok q4_0 q8_0" in r.stdout
