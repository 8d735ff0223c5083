"""cq_gemm_noalloc: the GEMM for callers that cannot allocate device memory
while they run (an engine that reserves all device memory up front, or a
thread that must stay out of the CUDA allocator). It keeps its scratch --
rotated activations of inputs wider than 512, padded copies of activations a
tensor map cannot address -- in a fixed array inside the library instead of
a workspace grown with cudaMalloc. Its results must match the oracle's (and
cq_gemm's), call after call, since every call reuses the same array, and
repeated calls must not change the device's free memory.

This file is collected last on purpose (pytest orders files by name)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import MATMUL_TOL, check_matmul

pytestmark = pytest.mark.gpu


def _rand_blob(out, n_in, bits, seed):
    ip = O.in_padded(n_in)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, seed, ternary=bits == 5)


def _call_noalloc(lib, blob, out, n_in, bits, cb, Xq, xs, Y, stream=None):
    cbp = np.ascontiguousarray(cb, dtype=np.float32)
    st = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    return lib.cq_gemm_noalloc(blob.data_ptr(), out, n_in, 128, bits,
                               cbp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                               Xq.data_ptr(), xs.data_ptr(), Xq.shape[0], Y.data_ptr(), st)


def _case(out, n_in, M, bits, seed, misalign=0):
    """A random blob and int8 activations; with misalign > 0 the activation
    rows start `misalign` bytes past a 16-byte boundary. Returns device
    tensors and the oracle's product and bound."""
    blob_np = _rand_blob(out, n_in, bits, 40 + seed)
    cb = O.analytic_codebook(bits)
    q, s = O.act_quant_int8(S.normal((M, n_in), 50 + seed).numpy())
    blob = torch.from_numpy(blob_np).cuda()
    buf = torch.zeros(M * n_in + 16, dtype=torch.int8, device="cuda")
    Xq = buf[misalign:misalign + M * n_in].view(M, n_in)
    Xq.copy_(torch.from_numpy(q))
    xs = torch.from_numpy(s).cuda()
    What = O.dequant(blob_np, out, n_in, bits, cb)
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    y_ref, bound = O.matmul(What, xt)
    return blob, cb, Xq, xs, y_ref, bound


# (out, in, M, bits, seed, misalign): the rotated path (in > 512), the direct
# tensor-map path (in = 512), the padded-copy path (rows not a multiple of 16
# bytes, and rows that are but start off a 16-byte boundary)
CASES = [(300, 640, 130, 2, 1, 0), (512, 512, 256, 4, 2, 0), (96, 200, 70, 3, 3, 0), (128, 512, 33, 5, 4, 1)]


def test_noalloc_matches_the_oracle_on_consecutive_calls():
    import hadamard_rotated_codebook_gb300 as C
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    for out, n_in, M, bits, seed, mis in CASES:
        blob, cb, Xq, xs, y_ref, bound = _case(out, n_in, M, bits, seed, mis)
        Y = torch.full((M, out), float("nan"), device="cuda")
        assert _call_noalloc(lib, blob, out, n_in, bits, cb, Xq, xs, Y) == 0, lib.cq_last_error()
        torch.cuda.synchronize()
        check_matmul(Y.cpu().numpy(), y_ref, bound, f"noalloc {out}x{n_in} M={M} bits={bits} misalign={mis}")
        # and within the same tolerance of cq_gemm's output
        Y_ref = C.cq_gemm(blob, out, n_in, bits, cb, Xq, xs)
        diff = np.abs(Y.cpu().numpy().astype(np.float64) - Y_ref.cpu().numpy())
        assert np.all(diff <= MATMUL_TOL * bound), float(np.max(diff / bound))


def test_noalloc_python_wrapper_and_no_new_device_memory():
    """The Python wrapper reaches the same entry point. Once every path has
    been called (the first call on a device resolves the array's address and
    loads the kernels), further calls on a stream the library has never seen
    leave the device's free memory unchanged: cq_gemm on that stream would
    have to allocate its workspace (4 MiB for the 2048 x 1024 case)."""
    import hadamard_rotated_codebook_gb300 as C
    cases = [_case(*c) for c in CASES] + [_case(64, 1024, 2048, 2, 5, 0)]
    shapes = [(c[0], c[1], c[3]) for c in CASES] + [(64, 1024, 2)]
    Ys = [torch.empty((Xq.shape[0], out), device="cuda") for (blob, cb, Xq, xs, _, _), (out, _, _) in
          zip(cases, shapes)]
    for (blob, cb, Xq, xs, _, _), (out, n_in, bits), Y in zip(cases, shapes, Ys):
        C.cq_gemm_noalloc(blob, out, n_in, bits, cb, Xq, xs, Y)  # set-up and kernel loading
    torch.cuda.synchronize()
    fresh = torch.cuda.Stream()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(fresh):
        for _rep in range(2):
            for (blob, cb, Xq, xs, _, _), (out, n_in, bits), Y in zip(cases, shapes, Ys):
                Y.fill_(float("nan"))
                C.cq_gemm_noalloc(blob, out, n_in, bits, cb, Xq, xs, Y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    for (blob, cb, Xq, xs, y_ref, bound), (out, n_in, bits), Y in zip(cases, shapes, Ys):
        check_matmul(Y.cpu().numpy(), y_ref, bound, f"wrapper {out}x{n_in} bits={bits}")


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
