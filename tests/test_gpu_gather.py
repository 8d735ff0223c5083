"""GPU parity of cq_gather_rows (row-gather dequantisation of a CQ table)
against the oracle's dequantised rows."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import gather_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _rand_blob(out, n_in, bits, seed):
    ip = O.in_padded(n_in)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, seed, ternary=bits == 5)


def _bound(blob, out, n_in, bits, cb, rows):
    return gather_bound(blob, out, n_in, bits, cb, rows)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("n_in", [384, 300])
def test_gather_matches_oracle(C, bits, n_in):
    out = 200
    cb = O.analytic_codebook(bits)
    blob = _rand_blob(out, n_in, bits, 60 + bits)
    rng = np.random.RandomState(bits * 7 + n_in)
    idx = rng.randint(0, out, size=97).astype(np.int32)
    idx[5] = idx[6]  # a repeated row
    dst = C.cq_gather_rows(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    ref = O.gather_rows(blob, out, n_in, bits, cb, idx)
    bound = _bound(blob, out, n_in, bits, cb, idx)
    assert np.all(np.abs(got - ref) <= bound), float((np.abs(got - ref) / bound).max())


def test_gather_closed_form_single_code(C):
    """All codes equal to j and norm n: the row is n*c_j*sqrt(128) at the
    first position of each group and zero elsewhere."""
    cb = O.analytic_codebook(4)
    out, n_in = 2, 256
    blob = np.zeros(O.packed_bytes(out, n_in, 128, 4), dtype=np.uint8)
    blob[:128] = 0x77   # row 0: every code 7
    blob[128:256] = 0xCC  # row 1: every code 12
    blob[256:264] = np.array([0x3C00, 0x4000, 0x3800, 0x4400], dtype="<u2").view(np.uint8)  # 1, 2 | 0.5, 4
    dst = C.cq_gather_rows(torch.from_numpy(blob).cuda(), out, n_in, 4, cb,
                           torch.tensor([1, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    for i, (row, code, ns) in enumerate([(1, 12, (0.5, 4.0)), (0, 7, (1.0, 2.0))]):
        for g, n in enumerate(ns):
            want = n * float(np.float32(cb[code])) * math.sqrt(128)
            assert abs(got[i, 128 * g] - want) <= 1e-6 * abs(want)
            assert np.all(np.abs(got[i, 128 * g + 1:128 * (g + 1)]) <= 1e-6 * abs(want))


def test_gather_empty_and_out_of_range(C):
    cb = O.analytic_codebook(2)
    out, n_in = 64, 256
    blob = _rand_blob(out, n_in, 2, 71)
    bdev = torch.from_numpy(blob).cuda()
    empty = C.cq_gather_rows(bdev, out, n_in, 2, cb, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert empty.shape == (0, n_in)
    C.cq_device_status()  # clean slate
    idx = torch.tensor([3, out, -1, 10], dtype=torch.int32, device="cuda")
    dst = C.cq_gather_rows(bdev, out, n_in, 2, cb, idx)
    with pytest.raises(C.CQError) as e:
        C.cq_device_status()
    assert e.value.code == C._capi.CQ_ERR_INDEX
    got = dst.cpu().numpy().astype(np.float64)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    ref = O.gather_rows(blob, out, n_in, 2, cb, [3, 10])
    assert np.all(np.abs(got[[0, 3]] - ref) <= _bound(blob, out, n_in, 2, cb, [3, 10]))
    C.cq_device_status()  # the word was cleared by the read above


def test_gather_full_table_sampled(C):
    """The 8192 x 512 CQ4 head table of the Needle-shaped set, 65536 token
    ids; 64 sampled outputs checked against the oracle's rows."""
    out, n_in = 8192, 512
    cb = O.analytic_codebook(4)
    blob = _rand_blob(out, n_in, 4, 72)
    rng = np.random.RandomState(73)
    idx = rng.randint(0, out, size=65536).astype(np.int32)
    dst = C.cq_gather_rows(torch.from_numpy(blob).cuda(), out, n_in, 4, cb, torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    C.cq_device_status()
    pick = np.sort(rng.choice(idx.size, 64, replace=False))
    rows = idx[pick]
    from tests.gpu_helpers import sub_blob
    sb = sub_blob(blob, out, n_in, 4, rows)
    ref = O.dequant(sb, len(rows), n_in, 4, cb)
    got = dst.cpu().numpy()[pick].astype(np.float64)
    bound = _bound(sb, len(rows), n_in, 4, cb, np.arange(len(rows)))
    assert np.all(np.abs(got - ref) <= bound)
