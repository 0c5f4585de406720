"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle checks.

This module only produces byte and float streams; it holds none of the
method's arithmetic (no decode, no product).  Sizes are passed in by the
caller.  The streams follow the generators printed on the pages:

* ``lcg_bytes`` -- cera 0.4.0 examples/wgpu_gemm_bench.rs, ``fill_quant_bytes``
  (LCG, byte = bits 16..23 of the state, bit 6 cleared at odd offsets so every
  f16 scale's exponent stays below the Inf/NaN code; the sign is kept).
* ``vecf`` -- memra-engine 0.128.0 moe_rows_ceiling_bench.rs, ``vecf``
  (xorshift64, uniform in [-1, 1)).
* ``nvfp4_rows`` -- the same page's ``synth_rows`` (36-byte groups, scale bytes
  ``(r & 7) | 0x38``, raw code bytes).

Seeds of the workloads: packed weight bytes use LCG seed 1, f32 weights use
``vecf`` seed 1, activations use ``vecf`` seed 2; NVFP4 matrix (copy c, expert
j, plane p) uses LCG seed ``0x8181 + 16*c + 2*j + p``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

WEIGHT_BYTE_SEED = 1
WEIGHT_F32_SEED = 1
X_SEED = 2


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC], check=True,
                   capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_lcg_bytes.restype = None
        lib.synth_lcg_bytes.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        lib.synth_vecf.restype = None
        lib.synth_vecf.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_nvfp4_rows.restype = None
        lib.synth_nvfp4_rows.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int64]
        _lib = lib
    return _lib


def lcg_bytes(seed: int, nbytes: int, clear_bit6_odd: bool = True) -> np.ndarray:
    out = np.empty(nbytes, np.uint8)
    _load().synth_lcg_bytes(seed & 0xFFFFFFFF, out.ctypes.data, nbytes, int(clear_bit6_odd))
    return out


def vecf(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_vecf(seed & 0xFFFFFFFFFFFFFFFF, out.ctypes.data, n)
    return out


def nvfp4_rows(seed: int, rows: int, in_f: int) -> np.ndarray:
    """rows x in_f NVFP4 weights as rows*in_f/64 groups of 36 bytes."""
    if in_f % 64:
        raise ValueError("in_f must be a multiple of 64")
    groups = rows * (in_f // 64)
    out = np.empty(groups * 36, np.uint8)
    _load().synth_nvfp4_rows(seed & 0xFFFFFFFF, out.ctypes.data, groups)
    return out


def nvfp4_matrix_seed(copy: int, expert: int, plane: int) -> int:
    return 0x8181 + 16 * copy + 2 * expert + plane


def weights(fmt: str, m: int, k: int, nbytes: int, seed: int | None = None) -> np.ndarray:
    """Packed weight bytes of an m x k matrix in format ``fmt`` whose size in
    bytes (``nbytes``) the caller computed.  f32 weights are ``vecf`` floats."""
    if fmt == "f32":
        if nbytes != 4 * m * k:
            raise ValueError("f32 weights take 4 bytes each")
        return vecf(WEIGHT_F32_SEED if seed is None else seed, m * k).view(np.uint8)
    if fmt == "nvfp4":
        return nvfp4_rows(0x8181 if seed is None else seed, m, k)
    return lcg_bytes(WEIGHT_BYTE_SEED if seed is None else seed, nbytes)


def activations(n: int, k: int, seed: int = X_SEED) -> np.ndarray:
    return vecf(seed, n * k).reshape(n, k)
