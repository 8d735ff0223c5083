"""Cactus Quants (CQ) on GB300: Hadamard-rotated codebook encode, GEMV and
GEMM over CQ-packed weights, and a .cact-shaped container.

Thin binding over libcq's C ABI (include/cq.h): every function here only
checks and marshals arguments (torch tensors for device memory and the
current CUDA stream) and calls the entry point of the same name. All
arithmetic of the hot path runs in the CUDA kernels of libcq.so; if the
library is missing the import fails rather than falling back.

Page citations use the page title and section:
  "The .cact format" (cactuscompute.com blog), "The .cact archive and Cactus
  Quants" (needle.js tutorial), OpenNeedle docs/reference.md.
"""
from __future__ import annotations

import contextlib
import ctypes
from dataclasses import dataclass
from typing import Iterable, Optional, Sequence

import numpy as np
import torch

from . import _capi
from ._capi import (CQ_DTYPE_CQ, CQ_DTYPE_FP16, CQ_DTYPE_FP32, CQ_DTYPE_RAW, CQ_X_F32,
                    CQ_X_F32Q, CQ_X_I8, CQError, GemmDesc, GemvDesc, KvGeom, KvSeq, TensorDesc, check)

GROUP = 128

__all__ = [
    "cq_levels", "cq_code_width", "cq_codebook_init", "cq_packed_bytes", "cq_encode",
    "cq_act_quant_int8", "cq_gemv", "cq_gemv_grouped", "cq_gemv_shared", "cq_gemm", "cq_gemm_grouped", "cq_gemm_noalloc",
    "cq_gather_rows", "cq_kv_write", "cq_kv_attend", "cq_device_status", "cq_cact_write", "cq_cact_open", "cq_cact_open_memory", "CactReader",
    "CQError", "library_path", "GROUP",
]


def _lib():
    return _capi.load()


def library_path() -> str:
    return _capi.LIB_PATH


def _stream(device: Optional[torch.device] = None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dev_ptr(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _io_ptr(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    """Pointer to a GEMV activation, scale or output: a CUDA tensor, or a
    pinned (page-locked) host tensor, which the kernels read or write in
    place over the host link (unified addressing)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _on(device):
    """Makes `device` current for a library call: the library keeps its
    per-device state (SM count, status word, workspaces, the fixed scratch
    array) for the device that is current when it is called. When it is
    current already, nothing is switched (the common case costs one query)."""
    dev = torch.device(device) if not isinstance(device, torch.device) else device
    if dev.index is None or dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def _check_blob(blob: torch.Tensor, out: int, n_in: int, group: int, bits: int, name: str = "blob"):
    """A blob shorter than its geometry would be read past its end on the
    device, which the C ABI (a bare pointer) cannot see. Invalid geometries
    (size 0) are left to the library, which reports them."""
    need = cq_packed_bytes(out, n_in, group, bits)
    if isinstance(blob, torch.Tensor) and blob.numel() < need:
        raise ValueError(f"{name} holds {blob.numel()} bytes, the CQ matrix needs {need}")


def _codebook_arg(codebook, bits: int):
    cb = np.ascontiguousarray(np.asarray(
        codebook.detach().cpu() if isinstance(codebook, torch.Tensor) else codebook,
        dtype=np.float32))
    if cb.size != cq_levels(bits):
        raise ValueError(f"codebook for bits={bits} needs {cq_levels(bits)} levels, got {cb.size}")
    return cb, cb.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


# ------------------------------------------------------------------- host

def cq_levels(bits: int) -> int:
    return _lib().cq_levels(bits)


def cq_code_width(bits: int) -> int:
    return _lib().cq_code_width(bits)


def cq_codebook_init(bits: int, group: int = GROUP) -> np.ndarray:
    """Analytic Lloyd-Max codebook of N(0,1) divided by sqrt(group) (fp32);
    ternary (bits=5) levels +-1.2240064/sqrt(group) and 0."""
    n = ctypes.c_size_t(0)
    check(_lib().cq_codebook_init(bits, group, None, 0, ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.float32)
    check(_lib().cq_codebook_init(bits, group, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                  out.size, None))
    return out


def cq_packed_bytes(out: int, n_in: int, group: int, bits: int) -> int:
    return int(_lib().cq_packed_bytes(out, n_in, group, bits))


# ----------------------------------------------------------------- device

def cq_encode(W: torch.Tensor, bits: int, codebook, group: int = GROUP,
              blob: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Encodes fp32 W[out, in] (CUDA) into a CQ blob (uint8, CUDA)."""
    if W.dim() != 2:
        raise ValueError("W must be 2-D [out, in]")
    out, n_in = W.shape
    nbytes = cq_packed_bytes(out, n_in, group, bits)
    if blob is None:
        blob = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    elif blob.numel() != nbytes:
        raise ValueError(f"blob must hold {nbytes} bytes")
    _, cbp = _codebook_arg(codebook, bits)
    with _on(W.device):
        check(_lib().cq_encode(_dev_ptr(W, torch.float32, "W"), out, n_in, group, bits, cbp,
                               _dev_ptr(blob, torch.uint8, "blob"), _stream(W.device)))
    return blob


def cq_act_quant_int8(X: torch.Tensor, Xq: Optional[torch.Tensor] = None,
                      s: Optional[torch.Tensor] = None):
    """Per-token int8 quantisation of fp32 X[M, in]; returns (Xq int8, s fp32)."""
    X2 = X if X.dim() == 2 else X.reshape(1, -1)
    M, n_in = X2.shape
    if Xq is None:
        Xq = torch.empty((M, n_in), dtype=torch.int8, device=X.device)
    if s is None:
        s = torch.empty(M, dtype=torch.float32, device=X.device)
    if tuple(Xq.shape) != (M, n_in) or s.numel() != M:
        raise ValueError("Xq must be [M, in] and s [M]")
    with _on(X.device):
        check(_lib().cq_act_quant_int8(_dev_ptr(X2, torch.float32, "X"), M, n_in,
                                       _dev_ptr(Xq, torch.int8, "Xq"), _dev_ptr(s, torch.float32, "s"),
                                       _stream(X.device)))
    return Xq, s


def _gemv_desc(blob, out, n_in, bits, codebook, x, x_scale, y, group, keep, quantize=False):
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    B = x2.shape[0]
    if x2.shape[1] != n_in:
        raise ValueError(f"x has {x2.shape[1]} columns, matrix has in={n_in}")
    if quantize and x2.dtype != torch.float32:
        raise TypeError("quantize=True needs fp32 activations")
    if x2.dtype == torch.float32:
        xdt, xs = (CQ_X_F32Q if quantize else CQ_X_F32), None
    elif x2.dtype == torch.int8:
        xdt = CQ_X_I8
        if x_scale is None:
            raise ValueError("int8 activations need x_scale")
        if x_scale.numel() < B:
            raise ValueError(f"x_scale has {x_scale.numel()} entries, the batch has {B}")
        xs = _io_ptr(x_scale, torch.float32, "x_scale")
    else:
        raise TypeError("x must be float32 or int8")
    if y is None:
        y = torch.empty((B, out), dtype=torch.float32, device=blob.device)
    elif y.numel() < B * out:
        raise ValueError(f"y holds {y.numel()} values, the product has {B * out}")
    _check_blob(blob, out, n_in, group, bits)
    cb, cbp = _codebook_arg(codebook, bits)
    keep.append(cb)
    d = GemvDesc(blob=_dev_ptr(blob, torch.uint8, "blob"), x=_io_ptr(x2, x2.dtype, "x"),
                 x_scale=xs, y=_io_ptr(y, torch.float32, "y"), codebook=cbp, out=out, in_=n_in,
                 group=group, bits=bits, x_dtype=xdt, B=B)
    return d, y


def cq_gemv(blob: torch.Tensor, out: int, n_in: int, bits: int, codebook, x: torch.Tensor,
            x_scale: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
            group: int = GROUP, quantize: bool = False) -> torch.Tensor:
    """y[B, out] = W_hat x over one CQ blob; x fp32 [B, in] or int8 with
    per-token scales x_scale[B]. quantize=True: fp32 x is quantised per token
    to int8 inside the call (as cq_act_quant_int8 does) before the product."""
    keep = []
    d, y = _gemv_desc(blob, out, n_in, bits, codebook, x, x_scale, y, group, keep, quantize)
    with _on(blob.device):
        check(_lib().cq_gemv_grouped(ctypes.byref(d), 1, _stream(blob.device)))
    return y


def cq_gemv_grouped(items: Sequence[dict]) -> list:
    """Runs many GEMVs in one launch. Each item is a dict with keys blob,
    out, in, bits, codebook, x and optionally x_scale, y, group, quantize.
    Returns the ys."""
    if not items:
        return []
    keep, ds, ys = [], [], []
    for it in items:
        d, y = _gemv_desc(it["blob"], it["out"], it["in"], it["bits"], it["codebook"], it["x"],
                          it.get("x_scale"), it.get("y"), it.get("group", GROUP), keep, it.get("quantize", False))
        ds.append(d)
        ys.append(y)
    arr = (GemvDesc * len(ds))(*ds)
    with _on(items[0]["blob"].device):
        check(_lib().cq_gemv_grouped(arr, len(ds), _stream(items[0]["blob"].device)))
    return ys


def cq_gemv_shared(blobs: Sequence[torch.Tensor], outs: Sequence[int], n_in: int, bits: int, codebook,
                   x: torch.Tensor, x_scale: Optional[torch.Tensor] = None, group: int = GROUP) -> list:
    """y_j = W_j x for matrices that share the activation x (Q/K/V/gate of a
    layer), in one launch. Returns the list of y_j [B, outs[j]]."""
    if len(blobs) != len(outs) or not blobs:
        raise ValueError("blobs and outs must be non-empty and of equal length")
    B = x.shape[0] if x.dim() == 2 else 1
    ys = [torch.empty((B, o), dtype=torch.float32, device=blobs[0].device) for o in outs]
    keep = []
    d, _ = _gemv_desc(blobs[0], outs[0], n_in, bits, codebook, x, x_scale, ys[0], group, keep)
    n = len(blobs)
    bp = (ctypes.c_void_p * n)(*[_dev_ptr(b, torch.uint8, "blob") for b in blobs])
    op = (ctypes.c_int * n)(*outs)
    yp = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    for b, o in zip(blobs, outs):
        _check_blob(b, o, n_in, group, bits)
    cb, cbp = _codebook_arg(codebook, bits)
    with _on(blobs[0].device):
        check(_lib().cq_gemv_shared(bp, op, n, n_in, group, bits, cbp, d.x, d.x_dtype, d.x_scale, d.B, yp,
                                    _stream(blobs[0].device)))
    return ys


class GemvPlan:
    """Prebuilt descriptor array for repeated grouped GEMV calls on the same
    buffers (the decode step): only the ctypes call remains per step."""

    def __init__(self, items: Sequence[dict]):
        self._keep, ds, self.ys = [], [], []
        for it in items:
            d, y = _gemv_desc(it["blob"], it["out"], it["in"], it["bits"], it["codebook"], it["x"],
                              it.get("x_scale"), it.get("y"), it.get("group", GROUP), self._keep,
                              it.get("quantize", False))
            ds.append(d)
            self.ys.append(y)
        self._items = list(items)  # keep tensors alive
        self._arr = (GemvDesc * len(ds))(*ds)
        self._n = len(ds)
        self._device = items[0]["blob"].device

    def run(self, stream: Optional[torch.cuda.Stream] = None):
        st = ctypes.c_void_p((stream or torch.cuda.current_stream(self._device)).cuda_stream)
        with _on(self._device):
            check(_lib().cq_gemv_grouped(self._arr, self._n, st))
        return self.ys


def _gemm_checks(blob, out, n_in, bits, Xq, x_scale, Y, group):
    """Sizes the C ABI cannot see: a short blob or scale buffer would be
    read past its end on the device."""
    if Xq.dim() != 2 or Xq.shape[1] != n_in:
        raise ValueError("Xq must be [M, in]")
    M = Xq.shape[0]
    if x_scale.numel() != M:
        raise ValueError(f"x_scale has {x_scale.numel()} entries, Xq has {M} rows")
    if Y is not None and tuple(Y.shape) != (M, out):
        raise ValueError(f"Y must be [{M}, {out}]")
    _check_blob(blob, out, n_in, group, bits)
    return M


def _gemm_desc(blob, out, n_in, bits, codebook, Xq, x_scale, Y, group, keep):
    M = _gemm_checks(blob, out, n_in, bits, Xq, x_scale, Y, group)
    if Y is None:
        Y = torch.empty((M, out), dtype=torch.float32, device=Xq.device)
    cb, cbp = _codebook_arg(codebook, bits)
    keep.append(cb)
    d = GemmDesc(blob=_dev_ptr(blob, torch.uint8, "blob"), Xq=_dev_ptr(Xq, torch.int8, "Xq"),
                 x_scale=_dev_ptr(x_scale, torch.float32, "x_scale"), Y=_dev_ptr(Y, torch.float32, "Y"),
                 codebook=cbp, out=out, in_=n_in, group=group, bits=bits, M=M)
    return d, Y


def cq_gemm(blob: torch.Tensor, out: int, n_in: int, bits: int, codebook, Xq: torch.Tensor,
            x_scale: torch.Tensor, Y: Optional[torch.Tensor] = None, group: int = GROUP) -> torch.Tensor:
    """Y[M, out] = s[m] * W_hat Xq[m] on the tensor cores (int8 per-token activations)."""
    keep = []
    d, Y = _gemm_desc(blob, out, n_in, bits, codebook, Xq, x_scale, Y, group, keep)
    with _on(Xq.device):
        check(_lib().cq_gemm_grouped(ctypes.byref(d), 1, _stream(Xq.device)))
    return Y


def cq_gemm_noalloc(blob: torch.Tensor, out: int, n_in: int, bits: int, codebook, Xq: torch.Tensor,
                    x_scale: torch.Tensor, Y: torch.Tensor, group: int = GROUP) -> torch.Tensor:
    """cq_gemm for callers that cannot allocate device memory while they run:
    the rotated activations live in a fixed array inside the library (at most
    CQ_GEMM_NOALLOC_MAX_ELEMS = M * in_pad fp16 values). Y must be given.
    Calls share that array, so calls that overlap on the GPU race."""
    cb, cbp = _codebook_arg(codebook, bits)
    if Y is None:
        raise ValueError("cq_gemm_noalloc writes into a caller-owned Y [M, out]")
    M = _gemm_checks(blob, out, n_in, bits, Xq, x_scale, Y, group)
    # the library picks the scratch array of the current device
    with _on(Xq.device):
        check(_lib().cq_gemm_noalloc(_dev_ptr(blob, torch.uint8, "blob"), out, n_in, group, bits, cbp,
                                     _dev_ptr(Xq, torch.int8, "Xq"), _dev_ptr(x_scale, torch.float32, "x_scale"),
                                     M, _dev_ptr(Y, torch.float32, "Y"), _stream(Xq.device)))
    return Y


def cq_gemm_grouped(items: Sequence[dict]) -> list:
    """Items: dicts with blob, out, in, bits, codebook, Xq, x_scale and optionally Y."""
    if not items:
        return []
    keep, ds, Ys = [], [], []
    for it in items:
        d, Y = _gemm_desc(it["blob"], it["out"], it["in"], it["bits"], it["codebook"], it["Xq"],
                          it["x_scale"], it.get("Y"), it.get("group", GROUP), keep)
        ds.append(d)
        Ys.append(Y)
    arr = (GemmDesc * len(ds))(*ds)
    with _on(items[0]["Xq"].device):
        check(_lib().cq_gemm_grouped(arr, len(ds), _stream(items[0]["Xq"].device)))
    return Ys


def cq_gather_rows(blob: torch.Tensor, out: int, n_in: int, bits: int, codebook, idx: torch.Tensor,
                   dst: Optional[torch.Tensor] = None, group: int = GROUP) -> torch.Tensor:
    """dst[i] = W_hat[idx[i]] (fp32 [n, in]): only the indexed rows of the CQ
    table are decoded. An index outside [0, out) gives a zero row, reported by
    a later cq_device_status as CQError(CQ_ERR_INDEX)."""
    if idx.dim() != 1:
        raise ValueError("idx must be one-dimensional")
    n = idx.shape[0]
    if dst is None:
        dst = torch.empty((n, n_in), dtype=torch.float32, device=idx.device)
    if dst.shape != (n, n_in):
        raise ValueError("dst must be [n, in]")
    _check_blob(blob, out, n_in, group, bits)
    cb, cbp = _codebook_arg(codebook, bits)
    with _on(idx.device):
        check(_lib().cq_gather_rows(_dev_ptr(blob, torch.uint8, "blob"), out, n_in, group, bits, cbp,
                                    _dev_ptr(idx, torch.int32, "idx"), n, _dev_ptr(dst, torch.float32, "dst"),
                                    _stream(idx.device)))
    return dst


def cq_kv_write(cache: torch.Tensor, cap: int, n_in: int, bits: int, codebook, rows: torch.Tensor,
                t0: int) -> None:
    """Encodes rows [n, n_in] (fp32, device) into rows t0 .. t0+n-1 of a CQ
    cache of ``cap`` rows (uint8 device tensor of cq_packed_bytes(cap, n_in,
    128, bits) bytes)."""
    rows2 = rows if rows.dim() == 2 else rows.reshape(1, -1)
    if rows2.shape[1] != n_in:
        raise ValueError(f"rows have {rows2.shape[1]} columns, cache rows have {n_in}")
    _check_blob(cache, cap, n_in, GROUP, bits, "cache")
    cb, cbp = _codebook_arg(codebook, bits)
    with _on(cache.device):
        check(_lib().cq_kv_write(_dev_ptr(cache, torch.uint8, "cache"), cap, n_in, bits, cbp,
                                 _dev_ptr(rows2, torch.float32, "rows"), t0, rows2.shape[0],
                                 _stream(cache.device)))


def cq_kv_attend(seqs: Sequence[dict], n_q_heads: int, n_kv_heads: int, head_dim_k: int,
                 head_dim_v: int, k_bits: int, v_bits: int, k_codebook, v_codebook,
                 scale: float) -> list:
    """Decode-step attention over CQ caches for several sequences (one
    launch per 256). Each item has k_cache, v_cache (uint8 device tensors),
    cap, n_tokens, q [n_q_heads, head_dim_k] fp32 and optionally o. Returns
    the o tensors [n_q_heads, head_dim_v]."""
    if not seqs:
        return []
    kcb, kp = _codebook_arg(k_codebook, k_bits)
    vcb, vp = _codebook_arg(v_codebook, v_bits)
    geom = KvGeom(n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim_k=head_dim_k,
                  head_dim_v=head_dim_v, k_bits=k_bits, v_bits=v_bits, k_codebook=kp,
                  v_codebook=vp, scale=scale)
    outs, arr = [], (KvSeq * len(seqs))()
    for i, it in enumerate(seqs):
        q = it["q"]
        if tuple(q.shape) != (n_q_heads, head_dim_k):
            raise ValueError(f"q has shape {tuple(q.shape)}, expected {(n_q_heads, head_dim_k)}")
        o = it.get("o")
        if o is None:
            o = torch.empty((n_q_heads, head_dim_v), dtype=torch.float32, device=q.device)
        outs.append(o)
        arr[i] = KvSeq(k_cache=_dev_ptr(it["k_cache"], torch.uint8, "k_cache"),
                       v_cache=_dev_ptr(it["v_cache"], torch.uint8, "v_cache"),
                       q=_dev_ptr(q, torch.float32, "q"), o=_dev_ptr(o, torch.float32, "o"),
                       cap=it["cap"], n_tokens=it["n_tokens"])
    with _on(seqs[0]["q"].device):
        check(_lib().cq_kv_attend(ctypes.byref(geom), arr, len(seqs), _stream(seqs[0]["q"].device)))
    return outs


def cq_device_status(device: Optional[torch.device] = None) -> int:
    """Reads and clears the device status word of bounded waits (raises
    CQError(CQ_ERR_TIMEOUT) if one gave up)."""
    with _on(device if device is not None else torch.cuda.current_device()):
        return check(_lib().cq_device_status(_stream(device)))


# -------------------------------------------------------------- container

@dataclass
class CactTensor:
    dtype: int
    shape: tuple
    nbytes: int
    group: int
    bits: int
    data: bytes


def _tensor_desc(t) -> tuple:
    """Accepts a CactTensor or a dict(dtype, shape, data, group=0, bits=0)."""
    if isinstance(t, dict):
        t = CactTensor(dtype=t["dtype"], shape=tuple(t["shape"]), nbytes=len(t["data"]),
                       group=t.get("group", 0), bits=t.get("bits", 0), data=bytes(t["data"]))
    buf = ctypes.create_string_buffer(t.data, len(t.data))
    shp = (ctypes.c_uint32 * 4)(*(list(t.shape) + [0] * (4 - len(t.shape))))
    d = TensorDesc(dtype=t.dtype, ndim=len(t.shape), shape=shp, nbytes=len(t.data),
                   group=t.group, bits=t.bits, data=ctypes.cast(buf, ctypes.c_void_p))
    return d, buf


def cq_cact_write(path: str, tensors: Iterable, codebook28, default_group: int = GROUP) -> None:
    ds, bufs = [], []
    for t in tensors:
        d, b = _tensor_desc(t)
        ds.append(d)
        bufs.append(b)
    arr = (TensorDesc * max(1, len(ds)))(*ds)
    cb = np.ascontiguousarray(np.asarray(codebook28, dtype=np.float32))
    if cb.size != 28:
        raise ValueError("the container codebook has 28 floats (CQ2|CQ3|CQ4)")
    check(_lib().cq_cact_write(path.encode(), arr, len(ds),
                               cb.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), default_group))


class CactReader:
    """Validated view of a container; tensors are copied out as bytes."""

    def __init__(self, handle: ctypes.c_void_p):
        self._h = handle

    def __len__(self):
        return _lib().cq_cact_count(self._h)

    def codebook(self) -> np.ndarray:
        out = np.zeros(28, dtype=np.float32)
        check(_lib().cq_cact_codebook(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))))
        return out

    def default_group(self) -> int:
        return int(_lib().cq_cact_default_group(self._h))

    def tensor(self, i: int) -> CactTensor:
        d = TensorDesc()
        check(_lib().cq_cact_tensor(self._h, i, ctypes.byref(d)))
        data = ctypes.string_at(d.data, d.nbytes) if d.nbytes else b""
        return CactTensor(dtype=d.dtype, shape=tuple(d.shape[: d.ndim]), nbytes=d.nbytes,
                          group=d.group, bits=d.bits, data=data)

    def close(self):
        if self._h:
            _lib().cq_cact_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cq_cact_open(path: str) -> CactReader:
    h = ctypes.c_void_p()
    check(_lib().cq_cact_open(path.encode(), ctypes.byref(h)))
    return CactReader(h)


def cq_cact_open_memory(data: bytes) -> CactReader:
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    check(_lib().cq_cact_open_memory(ctypes.cast(buf, ctypes.c_void_p), len(data), ctypes.byref(h)))
    return CactReader(h)
