"""The library's calls captured in a CUDA graph and replayed.

The calls allocate nothing and make no host round trip, so a stream that
issues them can be captured: a tensor-core GEMM (with the f16 copy of X in
its workspace), a small-n GEMV, the fused int8 MoE gate/up and the FP4
prefill (quantizer and block-scaled GEMM), captured once and replayed, must
write exactly what the same calls write when issued directly, and a replay
after the inputs change in place must follow the new inputs.  (The
allocation-free entry point is not part of this.)
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import oracle
import synth
from qmm_cases import dev, nan_filled, weights

pytestmark = pytest.mark.gpu


class _Calls:
    def __init__(self, h):
        self.h = h
        # tensor-core GEMM, Q4_0, two tiles along n
        self.m, self.k, self.n = 384, 1024, 200
        self.w = dev(weights("q4_0", self.m, self.k))
        self.x = dev(synth.activations(self.n, self.k, seed=31))
        self.wsb = q.qmm_gemm_workspace_bytes("q4_0", self.m, self.k, self.n)
        self.ws = torch.empty(max(self.wsb, 256), dtype=torch.uint8, device="cuda")
        # GEMV, Q8_0, n = 4
        self.gm, self.gk, self.gn = 1000, 2048, 4
        self.gw = dev(weights("q8_0", self.gm, self.gk))
        self.gx = dev(synth.activations(self.gn, self.gk, seed=32))
        # fused int8 MoE gate/up: 3 experts of one token
        self.in_f, self.n_ff, self.n_used = 1024, 96, 3
        self.mats = [dev(synth.nvfp4_rows(synth.nvfp4_matrix_seed(7, j, p), self.n_ff, self.in_f))
                     for p in range(2) for j in range(self.n_used)]
        self.table = torch.tensor([a.data_ptr() for a in self.mats], dtype=torch.int64, device="cuda")
        self.scales = dev(np.array([0.5 + 0.01 * i for i in range(2 * self.n_used)], np.float32))
        self.mx = dev(synth.activations(1, self.in_f, seed=33))
        # FP4 prefill: 256 x 512 weights (V2 rows), 130 activation rows
        self.fm, self.fk, self.fn = 256, 512, 130
        v1 = synth.nvfp4_rows(synth.nvfp4_matrix_seed(8, 0, 0), self.fm, self.fk)
        self.fw = dev(oracle.nvfp4_repack_v2(v1, self.fm, self.fk))
        self.fx = dev(synth.activations(self.fn, self.fk, seed=34))
        self.fxq = torch.zeros(self.fn * q.qmm_row_bytes("nvfp4_v2", self.fk), dtype=torch.uint8, device="cuda")

    def outputs(self):
        return [nan_filled(self.n, self.m), nan_filled(self.gn, self.gm), nan_filled(2, self.n_used, self.n_ff),
                nan_filled(self.fn, self.fm)]

    def issue(self, outs):
        """Every call on the current stream."""
        d, gd, y, fd = outs
        q.qmm_gemm(self.h, "q4_0", self.w, self.x, d, self.m, self.k, self.n, self.ws, self.wsb)
        q.qmm_gemv(self.h, "q8_0", self.gw, self.gx, gd, self.gm, self.gk, self.gn)
        q.qmm_moe_gemv_q8_fused(self.h, "nvfp4", self.table, self.scales, self.mx, y, self.in_f, self.n_ff,
                                self.n_used, 1)
        q.qmm_quantize_nvfp4(self.h, self.fx, self.fxq, self.fn, self.fk)
        q.qmm_gemm_fp4(self.h, self.fw, self.fxq, fd, self.fm, self.fk, self.fn)


def _bits(ts):
    return [t.cpu().numpy().view(np.uint32).copy() for t in ts]


def test_calls_replay_in_a_cuda_graph(h):
    c = _Calls(h)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    direct = c.outputs()
    with torch.cuda.stream(s):  # issued directly (this also sets every kernel up before the capture)
        c.issue(direct)
    s.synchronize()
    assert q.qmm_sync_status(h) == 0
    want = _bits(direct)
    assert all(np.all(np.isfinite(w.view(np.float32))) for w in want)

    captured = c.outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.issue(captured)
    for t in captured:  # capture ran nothing: refill, so only the replay can write them
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert q.qmm_sync_status(h) == 0
    for name, got, exp in zip(("gemm", "gemv", "moe_q8_fused", "fp4"), _bits(captured), want):
        assert np.array_equal(got, exp), name

    # new inputs in place: the replay follows them, bit for bit as direct calls
    c.x.copy_(dev(synth.activations(c.n, c.k, seed=41)))
    c.gx.copy_(dev(synth.activations(c.gn, c.gk, seed=42)))
    c.mx.copy_(dev(synth.activations(1, c.in_f, seed=43)))
    c.fx.copy_(dev(synth.activations(c.fn, c.fk, seed=44)))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert q.qmm_sync_status(h) == 0
    replayed = _bits(captured)
    direct2 = c.outputs()
    with torch.cuda.stream(s):
        c.issue(direct2)
    s.synchronize()
    for name, got, exp in zip(("gemm", "gemv", "moe_q8_fused", "fp4"), replayed, _bits(direct2)):
        assert np.array_equal(got, exp), name
    assert not np.array_equal(replayed[0], want[0])  # the inputs did change
