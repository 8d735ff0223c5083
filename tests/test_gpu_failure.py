"""Failure detection without a GPU fault: a bounded device wait that nothing
completes gives up, records its code in the device status word, and the
host reads CQ_ERR_TIMEOUT; the context stays usable afterwards."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_host_sees_timeout():
    import hadamard_rotated_codebook_gb300 as C
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.cq_device_status(st) == _capi.CQ_OK  # clean to begin with
    assert lib.cq_selftest_wait_timeout(st) == _capi.CQ_OK
    assert lib.cq_device_status(st) == _capi.CQ_ERR_TIMEOUT
    assert b"0x4748ffff" in lib.cq_last_error()
    assert lib.cq_device_status(st) == _capi.CQ_OK  # read-and-clear
    # the context still works: a GEMM after the give-up is correct
    out, n_in, M, bits = 128, 256, 64, 2
    ip = O.in_padded(n_in)
    blob = S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, 71)
    cb = O.analytic_codebook(bits)
    q, s = O.act_quant_int8(S.normal((M, n_in), 72).numpy())
    Y = C.cq_gemm(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    What = O.dequant(blob, out, n_in, bits, cb)
    ref, bound = O.matmul(What, q.astype(np.float64) * s.astype(np.float64)[:, None])
    assert np.all(np.abs(Y.cpu().numpy() - ref) <= 2e-3 * bound)


def test_status_read_after_give_up_zeroes_split_counters():
    """The split GEMV's per-tile counters are left zero by every launch and
    zeroed when allocated; a launch that gave up midway could leave some
    set. With them set (a diagnostic fills them), the k-sliced sums of a
    4096 x 4096 matrix are not written; the status read that reports a
    give-up zeroes them, and the next call has the bits of a clean one."""
    import hadamard_rotated_codebook_gb300 as C
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.cq_device_status(st) == _capi.CQ_OK
    out = n_in = 4096  # 256 row tiles, too few for the SMs' warps: k-sliced
    blob = torch.from_numpy(S.random_blob(out * n_in * 2 // 8, out * n_in // 128, 73)).cuda()
    cb = O.analytic_codebook(2)
    x = S.normal((1, n_in), 74).cuda()
    y0 = C.cq_gemv(blob, out, n_in, 2, cb, x).clone()
    assert lib.cq_selftest_dirty_counters(st) == _capi.CQ_OK
    y_bad = C.cq_gemv(blob, out, n_in, 2, cb, x, y=torch.zeros_like(y0))
    torch.cuda.synchronize()
    assert not torch.equal(y_bad, y0)  # no k-slice saw itself last
    assert lib.cq_selftest_wait_timeout(st) == _capi.CQ_OK
    assert lib.cq_device_status(st) == _capi.CQ_ERR_TIMEOUT  # ... and the counters are zero again
    y1 = C.cq_gemv(blob, out, n_in, 2, cb, x, y=torch.zeros_like(y0))
    torch.cuda.synchronize()
    assert torch.equal(y1, y0)
