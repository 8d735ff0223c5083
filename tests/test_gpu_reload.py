"""The outlier encode workload end to end: 16 fp32 matrices of 8192x8192
(N(0, 0.02^2), 1% of entries scaled by 20) encoded on the GPU to CQ2 at
group 128, written to the container, read back, and reloaded matrices
multiplied at batch 1 on the GPU, checked against the oracle.

Pages: "The .cact format" ("Five regions": the blobs are what the kernel
consumes, as stored; "Versions"), "The .cact archive and Cactus Quants"
("Anatomy of a CQ matrix", "Keep the quantized views")."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import check_matmul, compare_encodings, sub_blob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _codebook28():
    return np.concatenate([O.analytic_codebook(2), O.analytic_codebook(3), O.analytic_codebook(4)])


def test_outlier_set_encode_write_read_gemv(C, tmp_path):
    out, n_in = S.ENCODE_SHAPE
    n = S.ENCODE_COUNT
    cb = O.analytic_codebook(2)
    nb = O.packed_bytes(out, n_in, 128, 2)
    blobs = []
    n_boundary = 0
    for i in range(n):
        W = S.encode_matrix(i, device="cuda")
        blob = C.cq_encode(W, 2, cb).cpu().numpy()
        assert blob.size == nb
        if i % 5 == 0:  # the encoder on sampled rows of every fifth matrix
            rows = np.array([0, 1 + 97 * i, 4096 + i, out - 1])
            ref, flags, _ = O.encode(W[torch.from_numpy(rows).cuda()].cpu().numpy(), 2, cb)
            nbd, _ = compare_encodings(sub_blob(blob, out, n_in, 2, rows), ref, flags, len(rows), n_in, 2)
            n_boundary += nbd
        blobs.append(blob)
        del W
    print(f"encoder: {n_boundary} boundary coordinates in the sampled rows")

    path = str(tmp_path / "outliers.cact")
    C.cq_cact_write(path, [dict(dtype=3, shape=(out, n_in), data=b.tobytes(), group=128, bits=2) for b in blobs],
                    _codebook28(), 128)
    with C.cq_cact_open(path) as r:
        assert len(r) == n and r.default_group() == 128
        cb_file = r.codebook()[:4]
        np.testing.assert_array_equal(cb_file, cb)
        for i in range(n):
            t = r.tensor(i)
            assert (t.dtype, t.shape, t.group, t.bits) == (3, (out, n_in), 128, 2)
            assert t.data == blobs[i].tobytes(), f"tensor {i}: reloaded bytes differ from the written ones"
        reloaded = {i: r.tensor(i).data for i in (0, 9, n - 1)}

    # batch-1 products over reloaded blobs, with the codebook read from the file
    rows = np.array([0, 5, 1000, 4095, 4096, 6001, out - 2, out - 1])
    for i, data in reloaded.items():
        blob_dev = torch.frombuffer(bytearray(data), dtype=torch.uint8).cuda()
        x = S.normal((1, n_in), 8100 + i)
        y = C.cq_gemv(blob_dev, out, n_in, 2, cb_file, x.cuda()).cpu().numpy()
        # the bytes as they were on the device before the round trip (the
        # product of an input this wide sums its partial results in any
        # order, so the two agree within the tolerance, not bit for bit)
        y_dev = C.cq_gemv(torch.from_numpy(blobs[i]).cuda(), out, n_in, 2, cb, x.cuda()).cpu().numpy()
        blob_np = np.frombuffer(data, dtype=np.uint8)
        What = O.dequant(sub_blob(blob_np, out, n_in, 2, rows), len(rows), n_in, 2, cb_file)
        y_ref, bound = O.matmul(What, x.numpy())
        worst = check_matmul(y[:, rows], y_ref, bound, f"reloaded matrix {i}")
        check_matmul(y_dev[:, rows], y_ref, bound, f"device matrix {i}")
        print(f"matrix {i}: max |err|/bound {worst:.3e}")
