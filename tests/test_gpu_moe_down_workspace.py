"""The down projection's workspace, reused call after call.

qmm_moe_down, qmm_moe_down_q8 and qmm_moe_down_q8_fused sum each token's
pairs in a fixed order, either inside the product kernel (the grouped
register-X kernel: rows of 2048, 4 pairs per token) or from the pair products
they write into the caller's workspace.  The workspace may hold anything
before a call, so one buffer filled with random bytes must serve any sequence
of calls, whatever their token counts and whichever path they take (grouped
f32, f32 shared-memory X kernel, int8, int8 with in-kernel quantization),
CUDA-graph replays included: every result bit for bit the result of the same
call on a fresh workspace of its own size.
"""
import numpy as np
import pytest
import torch

import gemv_dequant_gemm_gb300 as q
import synth
from qmm_cases import dev, nan_filled

pytestmark = pytest.mark.gpu

GIN, N_USED, T_MAX = 260, 4, 3  # 260 rows: row blocks with a ragged last one


class _Down:
    """Matrices, factors and activations for up to T_MAX tokens of one path."""

    def __init__(self, h, kind, n_ff, seed):
        self.h, self.kind, self.n_ff = h, kind, n_ff
        pairs = N_USED * T_MAX
        self.mats = [dev(synth.nvfp4_rows(synth.nvfp4_matrix_seed(seed, j, 2), GIN, n_ff)) for j in range(pairs)]
        self.table = torch.tensor([a.data_ptr() for a in self.mats], dtype=torch.int64, device="cuda")
        self.scales = dev(np.array([0.5 + 0.01 * p for p in range(pairs)], np.float32))
        self.hact = dev(synth.activations(pairs, n_ff, seed=seed + 100))
        self.qd = torch.zeros((pairs, n_ff), dtype=torch.int8, device="cuda")
        self.dd = torch.zeros((pairs, n_ff // 32), dtype=torch.float32, device="cuda")
        self.requantize()

    def requantize(self):
        q.qmm_quantize_q8_1(self.h, self.hact, self.qd, self.dd, N_USED * T_MAX, self.n_ff)

    def call(self, t, y, ws, wsb):
        args = (self.h, "nvfp4", self.table, self.scales)
        if self.kind == "q8":
            q.qmm_moe_down_q8(*args, self.qd, self.dd, y, self.n_ff, GIN, N_USED, t, ws, wsb)
        elif self.kind == "q8_fused":
            q.qmm_moe_down_q8_fused(*args, self.hact, y, self.n_ff, GIN, N_USED, t, ws, wsb)
        else:
            q.qmm_moe_down(*args, self.hact, y, self.n_ff, GIN, N_USED, t, ws, wsb)

    def fresh(self, t):
        """The call on a fresh workspace of exactly its own size."""
        wsb = q.qmm_moe_down_workspace_bytes(GIN, N_USED, t)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        y = nan_filled(t, GIN)
        self.call(t, y, ws, wsb)
        torch.cuda.synchronize()
        assert q.qmm_sync_status(self.h) == 0
        return y.cpu().numpy().view(np.uint32).copy()


def _paths(h):
    # n_ff 2048 takes the grouped register-X kernel, 512 the shared-memory X kernel
    return {"f32_rx": _Down(h, "f32", 2048, 11), "f32_smem": _Down(h, "f32", 512, 12),
            "q8": _Down(h, "q8", 1024, 13), "q8_fused": _Down(h, "q8_fused", 1024, 14)}


def _random_workspace(wsb, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(0, 256, (wsb,), dtype=torch.uint8, generator=g).cuda()


def test_one_workspace_serves_every_path_and_token_count(h):
    paths = _paths(h)
    wsb = q.qmm_moe_down_workspace_bytes(GIN, N_USED, T_MAX)
    ws = _random_workspace(wsb, 1)
    want = {(name, t): d.fresh(t) for name, d in paths.items() for t in range(1, T_MAX + 1)}
    order = [(name, t) for t in (3, 1, 2) for name in paths] + [(name, t) for name in paths for t in (2, 3, 1)]
    for name, t in order:
        y = nan_filled(t, GIN)
        paths[name].call(t, y, ws, wsb)
        torch.cuda.synchronize()
        assert q.qmm_sync_status(h) == 0
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want[(name, t)]), (name, t)


def test_graph_replays_share_the_workspace_with_direct_calls(h):
    paths = _paths(h)
    wsb = q.qmm_moe_down_workspace_bytes(GIN, N_USED, T_MAX)
    ws = _random_workspace(wsb, 2)
    captured = [("f32_rx", 3), ("q8_fused", 2), ("f32_smem", 1)]
    ys = [nan_filled(t, GIN) for _, t in captured]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # issued directly once, which also sets every kernel up
        for (name, t), y in zip(captured, ys):
            paths[name].call(t, y, ws, wsb)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (name, t), y in zip(captured, ys):
            paths[name].call(t, y, ws, wsb)
    for rnd in range(3):
        # direct calls of other token counts on the same workspace in between
        for name, t in (("q8", 2), ("f32_rx", 1)):
            y = nan_filled(t, GIN)
            paths[name].call(t, y, ws, wsb)
        for y in ys:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert q.qmm_sync_status(h) == 0
        for (name, t), y in zip(captured, ys):
            assert np.array_equal(y.cpu().numpy().view(np.uint32), paths[name].fresh(t)), (rnd, name, t)
        # new activations in place for the next round
        for d in paths.values():
            d.hact.copy_(dev(synth.activations(N_USED * T_MAX, d.n_ff, seed=500 + rnd)))
            d.requantize()
        torch.cuda.synchronize()
