"""Oracle for Cactus Quants (CQ) -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU restatement (C99, double precision, explicit Hadamard
matrix) of what the CQ hot path computes: the encoder (rotate, norm, nearest
level, pack), the dequantiser and the matrix product over packed weights.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product package never does.

Sources (page title, section):
  * "The .cact format" (cactuscompute.com blog): "Cactus Quants",
    "How the kernel reads it".
  * "The .cact archive and Cactus Quants" (needle.js tutorial):
    "Shared codebooks", "Anatomy of a CQ matrix", "2-bit"/"4-bit"/"3-bit",
    "Reconstructing one group".
  * OpenNeedle docs/reference.md: CQ quantisation recipe, file format,
    rotated-domain identity, fake_quant_act.

Every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py``; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libcq_oracle.so")
_SRC = os.path.join(_HERE, "cq_oracle.c")


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (gcc); returns the path."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "cq_oracle.h"))
    ):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        d, f, i, l = ctypes.c_double, ctypes.c_float, ctypes.c_int, ctypes.c_long
        u8, u16 = ctypes.c_uint8, ctypes.c_uint16
        sig = {
            "cqo_hadamard": (i, [i, P(d)]),
            "cqo_lloyd_max_normal": (i, [i, i, d, P(d)]),
            "cqo_lloyd_max_samples": (i, [P(d), l, i, i, P(d)]),
            "cqo_f32_to_f16": (u16, [f]),
            "cqo_f16_to_f32": (f, [u16]),
            "cqo_levels": (i, [i]),
            "cqo_width": (i, [i]),
            "cqo_packed_bytes": (ctypes.c_uint64, [i, i, i, i]),
            "cqo_encode": (l, [P(f), i, i, i, i, P(f), P(u8), P(u8), d]),
            "cqo_unpack": (i, [P(u8), i, i, i, i, P(i), P(u16)]),
            "cqo_dequant": (i, [P(u8), i, i, i, i, P(f), P(d)]),
            "cqo_matmul": (None, [P(d), i, i, P(d), i, P(d), P(d)]),
            "cqo_matmul_rotated": (i, [P(u8), i, i, i, i, P(f), P(d), i, P(d)]),
            "cqo_act_quant_int8": (None, [P(f), i, i, P(ctypes.c_int8), P(f)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ------------------------------------------------------------------ helpers

def levels(bits: int) -> int:
    return lib().cqo_levels(bits)


def width(bits: int) -> int:
    return lib().cqo_width(bits)


def in_padded(n_in: int, group: int = 128) -> int:
    return (n_in + group - 1) // group * group


def hadamard(n: int) -> np.ndarray:
    H = np.empty((n, n), dtype=np.float64)
    if lib().cqo_hadamard(n, _ptr(H, ctypes.c_double)) != 0:
        raise ValueError("n must be a power of two")
    return H


def lloyd_max_normal(L: int, max_iter: int = 1_000_000, tol: float = 1e-15):
    c = np.empty(L, dtype=np.float64)
    it = lib().cqo_lloyd_max_normal(L, max_iter, tol, _ptr(c, ctypes.c_double))
    if it < 0:
        raise ValueError("bad arguments")
    return c, it


def lloyd_max_samples(x: np.ndarray, L: int, iters: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    c = np.empty(L, dtype=np.float64)
    if lib().cqo_lloyd_max_samples(_ptr(x, ctypes.c_double), x.size, L, iters,
                                   _ptr(c, ctypes.c_double)) != 0:
        raise ValueError("bad arguments")
    return c


def analytic_codebook(bits: int, group: int = 128) -> np.ndarray:
    """Oracle-side codebook: Lloyd-Max on N(0,1) divided by sqrt(group), as
    fp32; ternary uses the constant 1.2240064 printed in the needle.js
    tutorial ("Shared codebooks"); binary (bits=1) is the two-level
    Lloyd-Max quantiser, whose centroids are closed-form ("The .cact format",
    "Cactus Quants": binary packs eight codes per byte)."""
    if bits == 5:
        c = 1.2240064 / np.sqrt(group)
        return np.array([-c, 0.0, c], dtype=np.float32)
    c, _ = lloyd_max_normal(1 << bits)
    return (c / np.sqrt(group)).astype(np.float32)


def f32_to_f16_bits(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib().cqo_f32_to_f16(float(v)) for v in x], dtype=np.uint16)


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib().cqo_f16_to_f32(int(v)) for v in h], dtype=np.float32)


def packed_bytes(out: int, n_in: int, group: int, bits: int) -> int:
    return int(lib().cqo_packed_bytes(out, n_in, group, bits))


def encode(W: np.ndarray, bits: int, codebook: np.ndarray, group: int = 128,
           eps: float = 1e-6):
    """Returns (blob uint8, flags uint8[out, in_pad], n_flagged)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    out, n_in = W.shape
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    blob = np.zeros(packed_bytes(out, n_in, group, bits), dtype=np.uint8)
    flags = np.zeros((out, in_padded(n_in, group)), dtype=np.uint8)
    n = lib().cqo_encode(_ptr(W, ctypes.c_float), out, n_in, group, bits,
                         _ptr(cb, ctypes.c_float), _ptr(blob, ctypes.c_uint8),
                         _ptr(flags, ctypes.c_uint8), eps)
    if n < 0:
        raise ValueError("cqo_encode rejected its arguments")
    return blob, flags, int(n)


def unpack(blob: np.ndarray, out: int, n_in: int, bits: int, group: int = 128):
    ip = in_padded(n_in, group)
    codes = np.zeros((out, ip), dtype=np.int32)
    norms = np.zeros((out, ip // group), dtype=np.uint16)
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    if lib().cqo_unpack(_ptr(blob, ctypes.c_uint8), out, n_in, group, bits,
                        _ptr(codes, ctypes.c_int), _ptr(norms, ctypes.c_uint16)) != 0:
        raise ValueError("bad arguments")
    return codes, norms


def dequant(blob: np.ndarray, out: int, n_in: int, bits: int, codebook,
            group: int = 128) -> np.ndarray:
    What = np.zeros((out, n_in), dtype=np.float64)
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    if lib().cqo_dequant(_ptr(blob, ctypes.c_uint8), out, n_in, group, bits,
                         _ptr(cb, ctypes.c_float), _ptr(What, ctypes.c_double)) != 0:
        raise ValueError("bad arguments")
    return What


def gather_rows(blob: np.ndarray, out: int, n_in: int, bits: int, codebook, idx,
                group: int = 128) -> np.ndarray:
    """Rows ``idx`` of the dequantised table, by definition: every row
    rebuilt group by group as n * H c[q] ("The .cact archive and Cactus
    Quants", "Reconstructing one group"), then the indexed rows selected.
    Indices must lie in [0, out)."""
    What = dequant(blob, out, n_in, bits, codebook, group)
    return What[np.asarray(idx, dtype=np.int64)]


def matmul(What: np.ndarray, X: np.ndarray):
    """Returns (Y[B, out], Bound[B, out]) in float64."""
    What = np.ascontiguousarray(What, dtype=np.float64)
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float64)
    out, n_in = What.shape
    B = X.shape[0]
    Y = np.zeros((B, out)); Bd = np.zeros((B, out))
    lib().cqo_matmul(_ptr(What, ctypes.c_double), out, n_in, _ptr(X, ctypes.c_double),
                     B, _ptr(Y, ctypes.c_double), _ptr(Bd, ctypes.c_double))
    return Y, Bd


def matmul_rotated(blob, out: int, n_in: int, bits: int, codebook, X,
                   group: int = 128) -> np.ndarray:
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float64)
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    Y = np.zeros((X.shape[0], out))
    if lib().cqo_matmul_rotated(_ptr(blob, ctypes.c_uint8), out, n_in, group, bits,
                                _ptr(cb, ctypes.c_float), _ptr(X, ctypes.c_double),
                                X.shape[0], _ptr(Y, ctypes.c_double)) != 0:
        raise ValueError("bad arguments")
    return Y


def act_quant_int8(X: np.ndarray):
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float32)
    B, n_in = X.shape
    Q = np.zeros((B, n_in), dtype=np.int8)
    S = np.zeros(B, dtype=np.float32)
    lib().cqo_act_quant_int8(_ptr(X, ctypes.c_float), B, n_in,
                             _ptr(Q, ctypes.c_int8), _ptr(S, ctypes.c_float))
    return Q, S


# ------------------------------------------------------------ KV cache --
# A CQ key or value cache is a CQ matrix whose rows are tokens: row t holds
# the n_kv_heads head vectors of token t side by side, encoded like weights
# ("The .cact format", "Five regions": the kv_bits field, and "How the
# kernel reads it": the same path serves the KV cache; OpenNeedle
# docs/reference.md: below 8 bits the KV cache goes through the CQ
# quantiser).

def _cache_geometry(n_in: int, bits: int, group: int = 128):
    ip = in_padded(n_in, group)
    return ip * width(bits) // 8, ip // group  # code bytes per row, groups per row


def kv_write(cache: np.ndarray, cap: int, n_in: int, bits: int, codebook, rows,
             t0: int, group: int = 128):
    """Encodes ``rows`` [n, n_in] as a CQ matrix and stores its code rows and
    norms at rows t0 .. t0+n-1 of ``cache`` (uint8, packed_bytes(cap, ...)
    bytes; modified in place). Returns (flags, n_flagged) of the encode."""
    rows = np.ascontiguousarray(np.atleast_2d(rows), dtype=np.float32)
    n = rows.shape[0]
    if t0 < 0 or t0 + n > cap:
        raise ValueError("rows outside the cache")
    if n == 0:
        return np.zeros((0, in_padded(n_in, group)), dtype=np.uint8), 0
    rb, ng = _cache_geometry(n_in, bits, group)
    blob, flags, nflag = encode(rows, bits, codebook, group)
    cache[t0 * rb:(t0 + n) * rb] = blob[:n * rb]
    nb = cap * rb + 2 * ng * t0
    cache[nb:nb + 2 * ng * n] = blob[n * rb:]
    return flags, nflag


def kv_rows_blob(cache: np.ndarray, cap: int, n_in: int, bits: int, n: int,
                 group: int = 128) -> np.ndarray:
    """The CQ blob of the first n rows of a cache of cap rows."""
    rb, ng = _cache_geometry(n_in, bits, group)
    return np.concatenate([cache[:n * rb], cache[cap * rb:cap * rb + 2 * ng * n]])


def attend(K: np.ndarray, V: np.ndarray, q: np.ndarray, n_kv_heads: int, scale: float):
    """Decode-step attention by its definition, in float64:
    o[b] = sum_t p[b, t] V[t, head h], p[b] = softmax_t(scale * <q[b], K[t, head h]>),
    h = b // (n_q_heads / n_kv_heads): consecutive query heads share one
    key/value head (grouped-query attention; OpenNeedle docs/reference.md:
    two query heads per KV head). K [T, n_kv_heads*dk], V [T, n_kv_heads*dv],
    q [n_q_heads, dk]. Returns (o [n_q_heads, dv], p [n_q_heads, T]); with
    T = 0 both are empty sums (o = 0)."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    Hq, dk = q.shape
    T = K.shape[0]
    dv = V.shape[1] // n_kv_heads
    per = Hq // n_kv_heads
    o = np.zeros((Hq, dv))
    P = np.zeros((Hq, T))
    for b in range(Hq):
        h = b // per
        if T == 0:
            continue
        s = scale * (K[:, h * dk:(h + 1) * dk] @ q[b])
        e = np.exp(s - s.max())
        p = e / e.sum()
        o[b] = p @ V[:, h * dv:(h + 1) * dv]
        P[b] = p
    return o, P


def kv_attend(k_cache, v_cache, cap: int, n_tokens: int, q, n_kv_heads: int,
              head_dim_k: int, head_dim_v: int, k_bits: int, v_bits: int,
              k_codebook, v_codebook, scale: float):
    """Attention over the first n_tokens rows of two CQ caches: the rows are
    dequantised (n * H c[q] per group) and ``attend`` applies. Returns
    (o, p, K_hat, V_hat)."""
    in_k, in_v = n_kv_heads * head_dim_k, n_kv_heads * head_dim_v
    Kh = dequant(kv_rows_blob(k_cache, cap, in_k, k_bits, n_tokens), n_tokens, in_k,
                 k_bits, k_codebook) if n_tokens else np.zeros((0, in_k))
    Vh = dequant(kv_rows_blob(v_cache, cap, in_v, v_bits, n_tokens), n_tokens, in_v,
                 v_bits, v_codebook) if n_tokens else np.zeros((0, in_v))
    o, P = attend(Kh, Vh, q, n_kv_heads, scale)
    return o, P, Kh, Vh
