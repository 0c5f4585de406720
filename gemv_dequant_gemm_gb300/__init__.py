"""Python binding of the qmm C ABI (include/qmm.h): argument marshalling only.

Every computation runs in the CUDA kernels of ``libqmm.so``; this module only
turns torch tensors (or raw integer device pointers) into the C arguments and
status codes into exceptions.  There is no fallback: if the library cannot be
loaded, importing the functions raises.

Names follow the C ABI: ``qmm_create``, ``qmm_destroy``, ``qmm_gemm``,
``qmm_gemv``, ``qmm_moe_gemv``, ``qmm_moe_down``, ``qmm_quantize_q8_1``, ``qmm_moe_gemv_q8``,
``qmm_moe_down_q8``, ``qmm_moe_gemv_q8_fused``, ``qmm_moe_down_q8_fused``, ``qmm_quantize_nvfp4``, ``qmm_gemm_fp4``, ``qmm_nvfp4_repack_v2``, ``qmm_dequant``, ``qmm_sync_status``,
``qmm_row_bytes``, ``qmm_gemm_workspace_bytes``, ``qmm_moe_down_workspace_bytes``,
``qmm_strerror``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmm.so")

# qmm_dtype values (include/qmm.h)
F32, Q4_0, Q8_0, Q4_K, Q6_K, NVFP4, NVFP4_V2 = 0, 1, 2, 3, 4, 5, 6
DTYPES = {"f32": F32, "q4_0": Q4_0, "q8_0": Q8_0, "q4_k": Q4_K, "q6_k": Q6_K, "nvfp4": NVFP4, "nvfp4_v2": NVFP4_V2}
GEMV_MAX_N = 8

STATUS = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED", 3: "QMM_ERR_SHAPE",
          4: "QMM_ERR_ALIGN", 5: "QMM_ERR_ARCH", 6: "QMM_ERR_CUDA", 7: "QMM_ERR_TIMEOUT",
          8: "QMM_ERR_WORKSPACE", 9: "QMM_ERR_OVERLAP"}

# Every symbol include/qmm.h and include/qmm_testing.h declare.
EXPORTS = ("qmm_create", "qmm_destroy", "qmm_strerror", "qmm_block_weights", "qmm_block_bytes",
           "qmm_row_bytes", "qmm_gemm_workspace_bytes", "qmm_gemm", "qmm_gemv", "qmm_moe_gemv",
           "qmm_moe_down_workspace_bytes", "qmm_moe_down", "qmm_nvfp4_repack_v2", "qmm_quantize_q8_1",
           "qmm_moe_gemv_q8", "qmm_moe_down_q8", "qmm_moe_gemv_q8_fused", "qmm_moe_down_q8_fused",
           "qmm_quantize_nvfp4", "qmm_gemm_fp4",
           "qmm_dequant", "qmm_sync_status", "qmm_gemm_noalloc", "qmm_gemm_noalloc_status",
           "qmm_testing_set_wait_limit_ns",
           "qmm_testing_skip_first_stage_load")


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_strerror(status)})")


_lib = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libqmm.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        from . import build as _build
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing; run gemv_dequant_gemm_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "qmm_create": (I, [I, ctypes.POINTER(P)]),
        "qmm_destroy": (I, [P]),
        "qmm_strerror": (ctypes.c_char_p, [I]),
        "qmm_block_weights": (I64, [I]),
        "qmm_block_bytes": (I64, [I]),
        "qmm_row_bytes": (I64, [I, I64]),
        "qmm_gemm_workspace_bytes": (SZ, [I, I64, I64, I64]),
        "qmm_gemm": (I, [P, I, P, P, P, I64, I64, I64, P, SZ, P]),
        "qmm_gemv": (I, [P, I, P, P, P, I64, I64, I64, P]),
        "qmm_moe_gemv": (I, [P, I, P, P, P, P, I64, I64, I, I, P]),
        "qmm_moe_down_workspace_bytes": (SZ, [I64, I, I]),
        "qmm_moe_down": (I, [P, I, P, P, P, P, I64, I64, I, I, P, SZ, P]),
        "qmm_dequant": (I, [P, I, P, P, I64, I64, ctypes.c_float, P]),
        "qmm_quantize_q8_1": (I, [P, P, P, P, I64, I64, P]),
        "qmm_quantize_nvfp4": (I, [P, P, P, I64, I64, P]),
        "qmm_gemm_fp4": (I, [P, P, P, P, I64, I64, I64, P]),
        "qmm_moe_gemv_q8": (I, [P, I, P, P, P, P, P, I64, I64, I, I, P]),
        "qmm_moe_down_q8": (I, [P, I, P, P, P, P, P, I64, I64, I, I, P, SZ, P]),
        "qmm_moe_gemv_q8_fused": (I, [P, I, P, P, P, P, I64, I64, I, I, P]),
        "qmm_moe_down_q8_fused": (I, [P, I, P, P, P, P, I64, I64, I, I, P, SZ, P]),
        "qmm_nvfp4_repack_v2": (I, [P, P, P, I64, I64, P]),
        "qmm_sync_status": (I, [P, P]),
        "qmm_gemm_noalloc": (I, [I, P, P, P, I64, I64, I64, P]),
        "qmm_gemm_noalloc_status": (I, [P]),
        "qmm_testing_set_wait_limit_ns": (I, [P, ctypes.c_uint64]),
        "qmm_testing_skip_first_stage_load": (I, [P, I]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _strerror(status: int) -> str:
    try:
        return load(False).qmm_strerror(status).decode()
    except Exception:  # the message is best effort; the status code is authoritative
        return "?"


def _dt(t) -> int:
    if isinstance(t, str):
        return DTYPES[t]
    return int(t)


def _ptr(a) -> int | None:
    """Device address of a torch tensor, or an int address as is."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise QmmError(status, where)


def qmm_strerror(status: int) -> str:
    return load().qmm_strerror(status).decode()


def qmm_block_weights(t) -> int:
    return load().qmm_block_weights(_dt(t))


def qmm_block_bytes(t) -> int:
    return load().qmm_block_bytes(_dt(t))


def qmm_row_bytes(t, k: int) -> int:
    return load().qmm_row_bytes(_dt(t), k)


def qmm_gemm_workspace_bytes(t, m: int, k: int, n: int) -> int:
    return load().qmm_gemm_workspace_bytes(_dt(t), m, k, n)


def qmm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().qmm_create(device, ctypes.byref(h)), "qmm_create")
    return h.value


def qmm_destroy(h: int) -> None:
    _check(load().qmm_destroy(h), "qmm_destroy")


def qmm_gemm(h, t, w, x, dst, m, k, n, workspace=None, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()
    _check(load().qmm_gemm(h, _dt(t), _ptr(w), _ptr(x), _ptr(dst), m, k, n, _ptr(workspace), workspace_bytes,
                           _stream(stream)), "qmm_gemm")


def qmm_gemv(h, t, w, x, dst, m, k, n, stream=None) -> None:
    _check(load().qmm_gemv(h, _dt(t), _ptr(w), _ptr(x), _ptr(dst), m, k, n, _stream(stream)), "qmm_gemv")


def qmm_moe_gemv(h, t, w_ptrs, scales, x, y, in_f, n_ff, n_used, t_tokens, stream=None) -> None:
    _check(load().qmm_moe_gemv(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(x), _ptr(y), in_f, n_ff, n_used,
                               t_tokens, _stream(stream)), "qmm_moe_gemv")


def qmm_moe_down_workspace_bytes(gin: int, n_used: int, t_tokens: int) -> int:
    return load().qmm_moe_down_workspace_bytes(gin, n_used, t_tokens)


def qmm_moe_down(h, t, w_ptrs, scales, hact, y, n_ff, gin, n_used, t_tokens, workspace=None, workspace_bytes=None,
                 stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()
    _check(load().qmm_moe_down(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(hact), _ptr(y), n_ff, gin, n_used,
                               t_tokens, _ptr(workspace), workspace_bytes, _stream(stream)), "qmm_moe_down")


Q8_MAX_K = 8192


def qmm_quantize_q8_1(h, x, q, d, rows, k, stream=None) -> None:
    _check(load().qmm_quantize_q8_1(h, _ptr(x), _ptr(q), _ptr(d), rows, k, _stream(stream)), "qmm_quantize_q8_1")


def qmm_moe_gemv_q8(h, t, w_ptrs, scales, q, d, y, in_f, n_ff, n_used, t_tokens, stream=None) -> None:
    _check(load().qmm_moe_gemv_q8(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(q), _ptr(d), _ptr(y), in_f, n_ff,
                                  n_used, t_tokens, _stream(stream)), "qmm_moe_gemv_q8")


def qmm_moe_down_q8(h, t, w_ptrs, scales, q, d, y, n_ff, gin, n_used, t_tokens, workspace=None, workspace_bytes=None,
                    stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()
    _check(load().qmm_moe_down_q8(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(q), _ptr(d), _ptr(y), n_ff, gin,
                                  n_used, t_tokens, _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_down_q8")


def qmm_moe_gemv_q8_fused(h, t, w_ptrs, scales, x, y, in_f, n_ff, n_used, t_tokens, stream=None) -> None:
    _check(load().qmm_moe_gemv_q8_fused(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(x), _ptr(y), in_f, n_ff,
                                        n_used, t_tokens, _stream(stream)), "qmm_moe_gemv_q8_fused")


def qmm_moe_down_q8_fused(h, t, w_ptrs, scales, x, y, n_ff, gin, n_used, t_tokens, workspace=None,
                          workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()
    _check(load().qmm_moe_down_q8_fused(h, _dt(t), _ptr(w_ptrs), _ptr(scales), _ptr(x), _ptr(y), n_ff, gin,
                                        n_used, t_tokens, _ptr(workspace), workspace_bytes, _stream(stream)),
           "qmm_moe_down_q8_fused")


def qmm_quantize_nvfp4(h, x, xq, rows, k, stream=None) -> None:
    _check(load().qmm_quantize_nvfp4(h, _ptr(x), _ptr(xq), rows, k, _stream(stream)), "qmm_quantize_nvfp4")


def qmm_gemm_fp4(h, w, xq, dst, m, k, n, stream=None) -> None:
    _check(load().qmm_gemm_fp4(h, _ptr(w), _ptr(xq), _ptr(dst), m, k, n, _stream(stream)), "qmm_gemm_fp4")


def qmm_nvfp4_repack_v2(h, v1, v2, m, k, stream=None) -> None:
    _check(load().qmm_nvfp4_repack_v2(h, _ptr(v1), _ptr(v2), m, k, _stream(stream)), "qmm_nvfp4_repack_v2")


def qmm_dequant(h, t, w, out, m, k, tensor_scale=1.0, stream=None) -> None:
    _check(load().qmm_dequant(h, _dt(t), _ptr(w), _ptr(out), m, k, float(tensor_scale), _stream(stream)),
           "qmm_dequant")


def qmm_sync_status(h, stream=None) -> int:
    """Synchronize and return the latched device status code (0 = ok); never raises."""
    return load().qmm_sync_status(h, _stream(stream))


NOALLOC_SCRATCH_BYTES = 8 << 20


def qmm_gemm_noalloc(t, w, x, dst, m, k, n, stream=None) -> None:
    """qmm_gemm without a handle or workspace, for callers that cannot allocate
    device memory; its scratch is a static device array of the library (calls
    share it, so they must not overlap on the GPU)."""
    _check(load().qmm_gemm_noalloc(_dt(t), _ptr(w), _ptr(x), _ptr(dst), m, k, n, _stream(stream)),
           "qmm_gemm_noalloc")


def qmm_gemm_noalloc_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status latched by
    qmm_gemm_noalloc calls on the current device (0 = ok); never raises."""
    return load().qmm_gemm_noalloc_status(_stream(stream))


def qmm_testing_set_wait_limit_ns(h, limit_ns: int) -> None:
    _check(load().qmm_testing_set_wait_limit_ns(h, limit_ns), "qmm_testing_set_wait_limit_ns")


def qmm_testing_skip_first_stage_load(h, enable: bool) -> None:
    _check(load().qmm_testing_skip_first_stage_load(h, int(bool(enable))), "qmm_testing_skip_first_stage_load")
