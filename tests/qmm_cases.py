"""Shared helpers of the GPU parity tests: seeded inputs, uploads, comparisons.

Inputs come from ``synth`` (the seeded generators); expected values come only
from ``oracle`` (the f64 CPU oracle).  Nothing here computes the method.
"""
import numpy as np
import torch

import oracle
import synth

FORMATS = ["f32", "q4_0", "q8_0", "q4_k", "q6_k", "nvfp4"]
QK = {"f32": 1, "q4_0": 32, "q8_0": 32, "q4_k": 256, "q6_k": 256, "nvfp4": 64}

# Tolerances stated for the method: tensor-core (f16 / tf32 inputs, fp32
# accumulate) and fp32-FMA paths, relative to sum_k |W*X| per element.
TC_REL, TC_ABS = 2e-3, 1e-6
FMA_REL = 1e-5


def weights(fmt, m, k, seed=None):
    return synth.weights(fmt, m, k, m * oracle.row_bytes(fmt, k), seed)


def dev(a):
    """numpy -> CUDA tensor with the same bytes (uint8 / float32)."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda()


def nan_filled(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def assert_close(got, ref, absmag, rel, abs_=0.0, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = rel * absmag + abs_
    bad = err > bound
    if np.any(bad):
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {idx}: "
                             f"got {got[idx]!r} want {ref[idx]!r} err {err[idx]:.3e} bound {bound[idx]:.3e}")


def assert_bitexact(got, want, what=""):
    """float32 arrays equal bit for bit, except that +0 and -0 compare equal."""
    g = np.ascontiguousarray(got, dtype=np.float32)
    w = np.ascontiguousarray(want, dtype=np.float32)
    same = (g.view(np.uint32) == w.view(np.uint32)) | ((g == 0) & (w == 0))
    if not np.all(same):
        idx = np.argwhere(~same)[0]
        raise AssertionError(f"{what}: {int((~same).sum())} mismatches; first at {tuple(idx)}: "
                             f"got {g[tuple(idx)]!r} want {w[tuple(idx)]!r}")
