"""Plain f64 CPU oracle for the quantized-weight projection matmul.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / ``--impl reference`` leg may import this
package.  The CUDA library never imports or links it, and it shares no code
with the CUDA library: the arithmetic is in ``qmm_oracle.c`` (plain C, double
precision, one loop per definition), this module only marshals numpy arrays.

Format names: ``f32``, ``q4_0``, ``q8_0``, ``q4_k``, ``q6_k``, ``nvfp4``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# The oracle's own format numbering (qmm_oracle.c, enum ORC_*).
FORMATS = {"f32": 0, "q4_0": 1, "q8_0": 2, "q4_k": 3, "q6_k": 4, "nvfp4": 5, "nvfp4_v2": 6}

_lib = None


def build(force: bool = False) -> str:
    """Compile qmm_oracle.c into liboracle.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_fp16.restype = ctypes.c_double
    lib.oracle_fp16.argtypes = [ctypes.c_uint32]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_e4m3.argtypes = [ctypes.c_uint32]
    lib.oracle_e2m1.restype = ctypes.c_double
    lib.oracle_e2m1.argtypes = [ctypes.c_uint32]
    for f in ("oracle_fp16_array", "oracle_e4m3_array", "oracle_e2m1_array"):
        getattr(lib, f).restype = None
        getattr(lib, f).argtypes = [P, P, I64]
    lib.oracle_block_weights.restype = I64
    lib.oracle_block_weights.argtypes = [ctypes.c_int]
    lib.oracle_block_bytes.restype = I64
    lib.oracle_block_bytes.argtypes = [ctypes.c_int]
    lib.oracle_row_bytes.restype = I64
    lib.oracle_row_bytes.argtypes = [ctypes.c_int, I64]
    lib.oracle_decode_row.restype = ctypes.c_int
    lib.oracle_decode_row.argtypes = [ctypes.c_int, P, I64, P]
    lib.oracle_dequant.restype = ctypes.c_int
    lib.oracle_dequant.argtypes = [ctypes.c_int, P, I64, I64, ctypes.c_double, P]
    lib.oracle_matmul.restype = ctypes.c_int
    lib.oracle_matmul.argtypes = [ctypes.c_int, P, P, I64, I64, I64, P, P, ctypes.c_int]
    lib.oracle_matmul_entries.restype = ctypes.c_int
    lib.oracle_matmul_entries.argtypes = [ctypes.c_int, P, P, I64, I64, I64, I64, P, P, P, P, ctypes.c_int]
    lib.oracle_moe_gate_up.restype = ctypes.c_int
    lib.oracle_moe_gate_up.argtypes = [ctypes.c_int, P, P, P, I64, I64, ctypes.c_int, ctypes.c_int,
                                       I64, I64, P, P, ctypes.c_int]
    lib.oracle_moe_down.restype = ctypes.c_int
    lib.oracle_moe_down.argtypes = [ctypes.c_int, P, P, P, I64, I64, ctypes.c_int, ctypes.c_int,
                                    I64, I64, P, P, ctypes.c_int]
    lib.oracle_nvfp4_repack_v2.restype = ctypes.c_int
    lib.oracle_nvfp4_repack_v2.argtypes = [P, P, I64, I64]
    lib.oracle_quantize_q8_1.restype = ctypes.c_int
    lib.oracle_quantize_q8_1.argtypes = [P, I64, I64, P, P]
    lib.oracle_moe_gate_up_q8.restype = ctypes.c_int
    lib.oracle_moe_gate_up_q8.argtypes = [ctypes.c_int, P, P, P, P, I64, I64, ctypes.c_int, ctypes.c_int,
                                          I64, I64, P, P, ctypes.c_int]
    lib.oracle_moe_down_q8.restype = ctypes.c_int
    lib.oracle_moe_down_q8.argtypes = [ctypes.c_int, P, P, P, P, I64, I64, ctypes.c_int, ctypes.c_int,
                                       I64, I64, P, P, ctypes.c_int]
    lib.oracle_e4m3_rn.restype = ctypes.c_uint8
    lib.oracle_e4m3_rn.argtypes = [ctypes.c_float]
    lib.oracle_e2m1_rn.restype = ctypes.c_uint8
    lib.oracle_e2m1_rn.argtypes = [ctypes.c_float]
    lib.oracle_quantize_nvfp4_v2.restype = ctypes.c_int
    lib.oracle_quantize_nvfp4_v2.argtypes = [P, I64, I64, P]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _fmt(name: str) -> int:
    if name not in FORMATS:
        raise ValueError(f"unknown format {name!r}")
    return FORMATS[name]


def max_threads() -> int:
    return _load().oracle_max_threads()


def fp16(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    out = np.empty(c.shape, np.float64)
    _load().oracle_fp16_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_array(_ptr(c), _ptr(out), c.size)
    return out


def e2m1(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e2m1_array(_ptr(c), _ptr(out), c.size)
    return out


def block_weights(fmt: str) -> int:
    return _load().oracle_block_weights(_fmt(fmt))


def block_bytes(fmt: str) -> int:
    return _load().oracle_block_bytes(_fmt(fmt))


def row_bytes(fmt: str, k: int) -> int:
    return _load().oracle_row_bytes(_fmt(fmt), k)


def _wbytes(w) -> np.ndarray:
    a = np.ascontiguousarray(w)
    return a.view(np.uint8).reshape(-1)


def decode(fmt: str, w, m: int, k: int) -> np.ndarray:
    """Exact decoded weights, f64 [m][k]."""
    wb = _wbytes(w)
    rb = row_bytes(fmt, k)
    if rb == 0 and k:
        raise ValueError("k is not a whole number of blocks")
    if wb.size < m * rb:
        raise ValueError("weight buffer too small")
    out = np.empty((m, k), np.float64)
    lib = _load()
    for r in range(m):
        rc = lib.oracle_decode_row(_fmt(fmt), _ptr(wb) + r * rb, k, _ptr(out) + r * k * 8)
        if rc:
            raise ValueError(f"decode failed ({rc})")
    return out


def nvfp4_repack_v2(v1, m: int, k: int) -> np.ndarray:
    """NVFP4 36-byte-group rows -> V2 rows (codes, then the scale stream)."""
    src = np.ascontiguousarray(np.asarray(v1, dtype=np.uint8).reshape(-1))
    if src.size != m * row_bytes("nvfp4", k):
        raise ValueError("v1 has the wrong size")
    out = np.empty(m * row_bytes("nvfp4_v2", k), np.uint8)
    rc = _load().oracle_nvfp4_repack_v2(_ptr(src), _ptr(out), m, k)
    if rc != 0:
        raise ValueError(f"oracle_nvfp4_repack_v2: status {rc}")
    return out


def dequant(fmt: str, w, m: int, k: int, tensor_scale: float = 1.0) -> np.ndarray:
    """f32 [m][k]: each decoded value (times tensor_scale for nvfp4), rounded once."""
    wb = _wbytes(w)
    out = np.empty((m, k), np.float32)
    rc = _load().oracle_dequant(_fmt(fmt), _ptr(wb), m, k, float(np.float32(tensor_scale)), _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequant failed ({rc})")
    return out


def matmul(fmt: str, w, x, m: int, k: int, n: int, threads: int = 0):
    """(dst, absmag), both f64 [n][m]: dst = sum_k W[m,k] X[n,k], absmag = sum_k |W X|."""
    wb = _wbytes(w)
    xa = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if xa.size < n * k:
        raise ValueError("x too small")
    dst = np.empty((n, m), np.float64)
    am = np.empty((n, m), np.float64)
    rc = _load().oracle_matmul(_fmt(fmt), _ptr(wb), _ptr(xa), m, k, n, _ptr(dst), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_matmul failed ({rc})")
    return dst, am


def matmul_entries(fmt: str, w, x, m: int, k: int, n: int, ni, mj, threads: int = 0):
    """dst and absmag at the entries (ni[e], mj[e]) only."""
    wb = _wbytes(w)
    xa = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    mj = np.ascontiguousarray(mj, dtype=np.int64)
    dst = np.empty(ni.size, np.float64)
    am = np.empty(ni.size, np.float64)
    rc = _load().oracle_matmul_entries(_fmt(fmt), _ptr(wb), _ptr(xa), m, k, n, ni.size, _ptr(ni), _ptr(mj),
                                       _ptr(dst), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_matmul_entries failed ({rc})")
    return dst, am


def moe_gate_up(fmt: str, mats, scales, x, in_f: int, n_ff: int, n_used: int, t: int,
                row0: int = 0, nrows: int | None = None, threads: int = 0):
    """(y, absmag), f64 [2][n_pairs][n_ff]; mats is a list of 2*n_pairs packed
    matrices indexed plane*n_pairs + pair.  Rows outside [row0, row0+nrows) are NaN."""
    n_pairs = t * n_used
    if len(mats) != 2 * n_pairs:
        raise ValueError("need 2*n_pairs matrices")
    nrows = n_ff if nrows is None else nrows
    keep = [_wbytes(a) for a in mats]
    table = np.array([_ptr(a) for a in keep], dtype=np.uint64)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    xa = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    y = np.full((2, n_pairs, n_ff), np.nan)
    am = np.full((2, n_pairs, n_ff), np.nan)
    rc = _load().oracle_moe_gate_up(_fmt(fmt), _ptr(table), _ptr(sc), _ptr(xa), in_f, n_ff, n_used, t,
                                    row0, nrows, _ptr(y), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_moe_gate_up failed ({rc})")
    return y, am


def quantize_q8_1(x, rows: int, k: int):
    """(q int8 [rows][k], d float32 [rows][k/32]): Q8_1 blocks of 32 values,
    d = amax/127, q = x*(1/d) rounded half away from zero, all in float32."""
    xa = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if xa.size != rows * k:
        raise ValueError("x has the wrong size")
    q = np.empty((rows, k), np.int8)
    d = np.empty((rows, k // 32 if k > 0 else 0), np.float32)
    rc = _load().oracle_quantize_q8_1(_ptr(xa), rows, k, _ptr(q), _ptr(d))
    if rc:
        raise ValueError(f"oracle_quantize_q8_1 failed ({rc})")
    return q, d


def e4m3_rn(v: float) -> int:
    """E4M3FN code nearest to v >= 0 (ties to even, saturating at 448)."""
    return int(_load().oracle_e4m3_rn(float(v)))


def e2m1_rn(v: float) -> int:
    """E2M1 code nearest to v (ties to even, saturating at +-6, sign kept)."""
    return int(_load().oracle_e2m1_rn(float(v)))


def quantize_nvfp4_v2(x, rows: int, k: int) -> np.ndarray:
    """x [rows][k] f32 -> NVFP4 V2 rows (uint8 [rows * k/32*18]): per 16 values
    scale = E4M3 nearest to amax/6, codes = E2M1 nearest to x/scale, decided
    in float32."""
    xa = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if xa.size != rows * k:
        raise ValueError("x has the wrong size")
    out = np.empty(rows * row_bytes("nvfp4_v2", k), np.uint8)
    rc = _load().oracle_quantize_nvfp4_v2(_ptr(xa), rows, k, _ptr(out))
    if rc:
        raise ValueError(f"oracle_quantize_nvfp4_v2 failed ({rc})")
    return out


def moe_gate_up_q8(fmt: str, mats, scales, q, d, in_f: int, n_ff: int, n_used: int, t: int,
                   row0: int = 0, nrows: int | None = None, threads: int = 0):
    """moe_gate_up with each token's activation given as Q8_1 blocks (q, d):
    x[tok][c] = q[tok][c] * d[tok][c // 32]."""
    n_pairs = t * n_used
    if len(mats) != 2 * n_pairs:
        raise ValueError("need 2*n_pairs matrices")
    nrows = n_ff if nrows is None else nrows
    keep = [_wbytes(a) for a in mats]
    table = np.array([_ptr(a) for a in keep], dtype=np.uint64)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    qa = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    da = np.ascontiguousarray(d, dtype=np.float32).reshape(-1)
    if qa.size != t * in_f or da.size != t * (in_f // 32):
        raise ValueError("q or d has the wrong size")
    y = np.full((2, n_pairs, n_ff), np.nan)
    am = np.full((2, n_pairs, n_ff), np.nan)
    rc = _load().oracle_moe_gate_up_q8(_fmt(fmt), _ptr(table), _ptr(sc), _ptr(qa), _ptr(da), in_f, n_ff, n_used,
                                       t, row0, nrows, _ptr(y), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_moe_gate_up_q8 failed ({rc})")
    return y, am


def moe_down(fmt: str, mats, scales, h, n_ff: int, gin: int, n_used: int, t: int,
             row0: int = 0, nrows: int | None = None, threads: int = 0):
    """(y, absmag), f64 [t][gin]: y[i][r] = sum over the token's pairs j =
    i*n_used + u of scales[j] * (W_j[r] . h[j]); mats is a list of t*n_used
    packed [gin][n_ff] matrices, h is [t*n_used][n_ff].  Rows outside
    [row0, row0+nrows) are NaN."""
    n_pairs = t * n_used
    if len(mats) != n_pairs:
        raise ValueError("need t*n_used matrices")
    nrows = gin if nrows is None else nrows
    keep = [_wbytes(a) for a in mats]
    table = np.array([_ptr(a) for a in keep], dtype=np.uint64)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    ha = np.ascontiguousarray(h, dtype=np.float32).reshape(-1)
    y = np.full((t, gin), np.nan)
    am = np.full((t, gin), np.nan)
    rc = _load().oracle_moe_down(_fmt(fmt), _ptr(table), _ptr(sc), _ptr(ha), n_ff, gin, n_used, t,
                                 row0, nrows, _ptr(y), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_moe_down failed ({rc})")
    return y, am


def moe_down_q8(fmt: str, mats, scales, q, d, n_ff: int, gin: int, n_used: int, t: int,
                row0: int = 0, nrows: int | None = None, threads: int = 0):
    """moe_down with each pair's activation given as Q8_1 blocks (q, d):
    h[j][c] = q[j][c] * d[j][c // 32]."""
    n_pairs = t * n_used
    if len(mats) != n_pairs:
        raise ValueError("need t*n_used matrices")
    nrows = gin if nrows is None else nrows
    keep = [_wbytes(a) for a in mats]
    table = np.array([_ptr(a) for a in keep], dtype=np.uint64)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    qa = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    da = np.ascontiguousarray(d, dtype=np.float32).reshape(-1)
    if qa.size != n_pairs * n_ff or da.size != n_pairs * (n_ff // 32):
        raise ValueError("q or d has the wrong size")
    y = np.full((t, gin), np.nan)
    am = np.full((t, gin), np.nan)
    rc = _load().oracle_moe_down_q8(_fmt(fmt), _ptr(table), _ptr(sc), _ptr(qa), _ptr(da), n_ff, gin, n_used, t,
                                    row0, nrows, _ptr(y), _ptr(am), threads)
    if rc:
        raise ValueError(f"oracle_moe_down_q8 failed ({rc})")
    return y, am
