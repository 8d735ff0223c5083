"""cq_gemm_noalloc: the GEMM for callers that cannot allocate device memory
while they run (an engine that reserves all device memory up front, or a
thread that must stay out of the CUDA allocator). It keeps the rotated
activations in a fixed array inside the library instead of a workspace grown
with cudaMalloc. Its results must match cq_gemm's, call after call, since
every call reuses the same array.

This file is collected last on purpose (pytest orders files by name)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import MATMUL_TOL, sub_blob

pytestmark = pytest.mark.gpu


def _rand_blob(out, n_in, bits, seed):
    ip = O.in_padded(n_in)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, seed, ternary=bits == 5)


def _call_noalloc(lib, blob, out, n_in, bits, cb, Xq, xs, Y):
    cbp = np.ascontiguousarray(cb, dtype=np.float32)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.cq_gemm_noalloc(blob.data_ptr(), out, n_in, 128, bits,
                               cbp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                               Xq.data_ptr(), xs.data_ptr(), Xq.shape[0], Y.data_ptr(), stream)


def test_noalloc_matches_cq_gemm_on_consecutive_calls():
    import hadamard_rotated_codebook_gb300 as C
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    # two calls in a row with different shapes and widths share the array
    for out, n_in, M, bits, seed in ((300, 640, 130, 2, 1), (512, 512, 256, 4, 2)):
        blob_np = _rand_blob(out, n_in, bits, 40 + seed)
        cb = O.analytic_codebook(bits)
        q, s = O.act_quant_int8(S.normal((M, n_in), 50 + seed).numpy())
        blob = torch.from_numpy(blob_np).cuda()
        Xq, xs = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
        Y_ref = C.cq_gemm(blob, out, n_in, bits, cb, Xq, xs)
        Y = torch.full((M, out), float("nan"), device="cuda")
        assert _call_noalloc(lib, blob, out, n_in, bits, cb, Xq, xs, Y) == 0, lib.cq_last_error()
        torch.cuda.synchronize()
        # tolerance of the product tests: |dy| <= 2e-3 * sum |w| |x|
        What = O.dequant(sub_blob(blob_np, out, n_in, bits, np.arange(out)), out, n_in, bits, cb)
        xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
        _, bound = O.matmul(What, xt)
        diff = np.abs(Y.cpu().numpy().astype(np.float64) - Y_ref.cpu().numpy())
        assert np.all(diff <= MATMUL_TOL * bound), float(np.max(diff / bound))


def test_noalloc_rejects_sizes_beyond_its_array():
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    M = _capi.CQ_GEMM_NOALLOC_MAX_ELEMS // 512 + 1
    cb = O.analytic_codebook(2)
    blob = torch.zeros(O.packed_bytes(8, 512, 128, 2), dtype=torch.uint8, device="cuda")
    Xq = torch.zeros((M, 512), dtype=torch.int8, device="cuda")
    xs = torch.ones(M, device="cuda")
    Y = torch.zeros((M, 8), device="cuda")
    assert _call_noalloc(lib, blob, 8, 512, 2, cb, Xq, xs, Y) == _capi.CQ_ERR_SHAPE
    assert b"exceeds the fixed scratch" in lib.cq_last_error()
