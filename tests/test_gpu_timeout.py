"""Failure detection without a GPU fault: a device-side wait that runs out.

The test hook leaves the first k stage of the tensor-core GEMM unloaded, so
the MMA issuer's bounded wait expires (after 20 ms here).  The kernel then
latches the timeout bit, waits for its own copies and MMAs in flight, frees
its tensor memory and returns; the host reads QMM_ERR_TIMEOUT and the same
handle keeps working afterwards.
"""
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import TC_ABS, TC_REL, assert_close, dev, nan_filled, weights

pytestmark = pytest.mark.gpu


# (256, 512, 256): split-K clusters; (512, 256, 128): one CTA per tile;
# (38912, 256, 128): two 128-row subtiles per CTA; f32: tf32 with split-K
@pytest.mark.parametrize("fmt,m,k,n", [("q8_0", 256, 512, 256), ("q4_0", 512, 256, 128), ("q4_0", 38912, 256, 128),
                                       ("f32", 256, 512, 256)])
def test_expired_wait_is_reported_and_the_context_survives(h, fmt, m, k, n):
    w, x = weights(fmt, m, k), synth.activations(n, k)
    wd, xd = dev(w), dev(x)
    ws_bytes = q.qmm_gemm_workspace_bytes(fmt, m, k, n)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    d = nan_filled(n, m)
    q.qmm_testing_set_wait_limit_ns(h, 20_000_000)
    q.qmm_testing_skip_first_stage_load(h, True)
    try:
        q.qmm_gemm(h, fmt, wd, xd, d, m, k, n, ws if ws_bytes else None, ws_bytes)
        assert q.qmm_sync_status(h) == 7  # QMM_ERR_TIMEOUT
    finally:
        q.qmm_testing_skip_first_stage_load(h, False)
        q.qmm_testing_set_wait_limit_ns(h, 2_000_000_000)
    assert torch.isnan(d).all()  # the aborted call wrote nothing
    q.qmm_gemm(h, fmt, wd, xd, d, m, k, n, ws if ws_bytes else None, ws_bytes)
    assert q.qmm_sync_status(h) == 0
    ref, am = oracle.matmul(fmt, w, x, m, k, n)
    assert_close(d.cpu().numpy(), ref, am, TC_REL, TC_ABS, what="after the timeout")
