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
