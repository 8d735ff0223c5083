"""ctypes declarations of libcq's C ABI (include/cq.h).

Loading fails loudly: there is no fallback implementation behind these
names. ``load()`` returns the CDLL with every exported function typed.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcq.so")

c_int, c_float, c_size_t, c_uint32, c_uint64 = (
    ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64)
c_void_p, c_char_p = ctypes.c_void_p, ctypes.c_char_p
P = ctypes.POINTER

CQ_OK = 0
CQ_ERR_ARG, CQ_ERR_SHAPE, CQ_ERR_FORMAT, CQ_ERR_IO = -1, -2, -3, -4
CQ_ERR_CUDA, CQ_ERR_TIMEOUT, CQ_ERR_NOMEM, CQ_ERR_INDEX = -5, -6, -7, -8
CQ_X_F32, CQ_X_I8, CQ_X_F32Q = 0, 1, 2
CQ_GEMV_MAX_BATCH = 16
CQ_MAX_GROUPED = 256
CQ_GEMM_NOALLOC_MAX_ELEMS = 2 * 1024 * 1024
CQ_DTYPE_FP16, CQ_DTYPE_FP32, CQ_DTYPE_CQ, CQ_DTYPE_RAW = 1, 2, 3, 4

ERROR_NAMES = {
    CQ_ERR_ARG: "CQ_ERR_ARG", CQ_ERR_SHAPE: "CQ_ERR_SHAPE", CQ_ERR_FORMAT: "CQ_ERR_FORMAT",
    CQ_ERR_IO: "CQ_ERR_IO", CQ_ERR_CUDA: "CQ_ERR_CUDA", CQ_ERR_TIMEOUT: "CQ_ERR_TIMEOUT",
    CQ_ERR_NOMEM: "CQ_ERR_NOMEM", CQ_ERR_INDEX: "CQ_ERR_INDEX",
}


class GemvDesc(ctypes.Structure):
    _fields_ = [
        ("blob", c_void_p), ("x", c_void_p), ("x_scale", c_void_p), ("y", c_void_p),
        ("codebook", P(c_float)),
        ("out", c_int), ("in_", c_int), ("group", c_int), ("bits", c_int),
        ("x_dtype", c_int), ("B", c_int),
    ]


class GemmDesc(ctypes.Structure):
    _fields_ = [
        ("blob", c_void_p), ("Xq", c_void_p), ("x_scale", c_void_p), ("Y", c_void_p),
        ("codebook", P(c_float)),
        ("out", c_int), ("in_", c_int), ("group", c_int), ("bits", c_int), ("M", c_int),
    ]


class KvGeom(ctypes.Structure):
    _fields_ = [
        ("n_q_heads", c_int), ("n_kv_heads", c_int), ("head_dim_k", c_int), ("head_dim_v", c_int),
        ("k_bits", c_int), ("v_bits", c_int), ("k_codebook", P(c_float)), ("v_codebook", P(c_float)),
        ("scale", c_float),
    ]


class KvSeq(ctypes.Structure):
    _fields_ = [
        ("k_cache", c_void_p), ("v_cache", c_void_p), ("q", c_void_p), ("o", c_void_p),
        ("cap", c_int), ("n_tokens", c_int),
    ]


class TensorDesc(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_uint8), ("ndim", ctypes.c_uint8), ("shape", c_uint32 * 4),
        ("nbytes", c_uint64), ("group", c_uint32), ("bits", c_uint32), ("data", c_void_p),
    ]


# name -> (restype, argtypes); every symbol include/cq.h declares
SIGNATURES = {
    "cq_last_error": (c_char_p, []),
    "cq_version": (c_int, []),
    "cq_levels": (c_int, [c_int]),
    "cq_code_width": (c_int, [c_int]),
    "cq_codebook_init": (c_int, [c_int, c_int, P(c_float), c_size_t, P(c_size_t)]),
    "cq_packed_bytes": (c_uint64, [c_int, c_int, c_int, c_int]),
    "cq_encode": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_void_p]),
    "cq_act_quant_int8": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "cq_gemv": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_int,
                        c_void_p, c_int, c_void_p, c_void_p]),
    "cq_gemv_grouped": (c_int, [P(GemvDesc), c_int, c_void_p]),
    "cq_gemv_shared": (c_int, [P(c_void_p), P(c_int), c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_int,
                               c_void_p, c_int, P(c_void_p), c_void_p]),
    "cq_gemm": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_void_p,
                        c_int, c_void_p, c_void_p]),
    "cq_gemm_grouped": (c_int, [P(GemmDesc), c_int, c_void_p]),
    "cq_gemm_noalloc": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_void_p,
                                c_int, c_void_p, c_void_p]),
    "cq_gather_rows": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P(c_float), c_void_p, c_int,
                               c_void_p, c_void_p]),
    "cq_kv_write": (c_int, [c_void_p, c_int, c_int, c_int, P(c_float), c_void_p, c_int, c_int, c_void_p]),
    "cq_kv_attend": (c_int, [P(KvGeom), P(KvSeq), c_int, c_void_p]),
    "cq_device_status": (c_int, [c_void_p]),
    "cq_selftest_wait_timeout": (c_int, [c_void_p]),
    "cq_selftest_dirty_counters": (c_int, [c_void_p]),
    "cq_cact_write": (c_int, [c_char_p, P(TensorDesc), c_int, P(c_float), c_uint32]),
    "cq_cact_open": (c_int, [c_char_p, P(c_void_p)]),
    "cq_cact_open_memory": (c_int, [c_void_p, c_uint64, P(c_void_p)]),
    "cq_cact_count": (c_int, [c_void_p]),
    "cq_cact_codebook": (c_int, [c_void_p, P(c_float)]),
    "cq_cact_default_group": (c_uint32, [c_void_p]),
    "cq_cact_tensor": (c_int, [c_void_p, c_int, P(TensorDesc)]),
    "cq_cact_close": (None, [c_void_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Loads libcq.so (built by ``hadamard_rotated_codebook_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(the CQ kernels have no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class CQError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def check(code: int) -> int:
    if code != CQ_OK:
        raise CQError(code, load().cq_last_error().decode(errors="replace"))
    return code
