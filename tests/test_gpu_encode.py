"""GPU parity of the encoder and the int8 activation quantiser against the
oracle on identical seeded inputs.

Codes must be bit-exact except at coordinates the oracle flags as lying
within 1e-6 of a decision boundary (counted and reported); fp16 norms must
be bit-exact; int8 activations and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import compare_encodings

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _encode_both(C, W, bits, codebook=None):
    cb = O.analytic_codebook(bits) if codebook is None else codebook
    blob_ref, flags, nflag = O.encode(W.numpy(), bits, cb)
    blob = C.cq_encode(W.cuda(), bits, cb)
    torch.cuda.synchronize()
    return blob.cpu().numpy(), blob_ref, flags


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("shape", [(512, 512), (3, 129), (33, 200), (1, 1), (130, 1024)])
def test_encode_parity(C, bits, shape):
    W = S.normal(shape, 7 + bits, S.W_STD)
    g, r, flags = _encode_both(C, W, bits)
    nb, nbm = compare_encodings(g, r, flags, shape[0], shape[1], bits)
    print(f"bits={bits} shape={shape}: {nb} boundary coordinates, {nbm} differ")


@pytest.mark.parametrize("bits", [2, 4])
def test_encode_heavy_tails_and_outliers(C, bits):
    W = S.with_outliers(S.student_t4((64, 1024), 11, S.W_STD), 12)
    g, r, flags = _encode_both(C, W, bits)
    compare_encodings(g, r, flags, 64, 1024, bits)


def test_encode_empirical_codebook(C):
    """The kernels take any strictly increasing codebook, e.g. the
    asymmetric empirical one a file carries."""
    x = np.random.RandomState(0).randn(400000)
    cb = (O.lloyd_max_samples(x, 4, 200) / np.sqrt(128)).astype(np.float32)
    W = S.normal((96, 384), 21, S.W_STD)
    g, r, flags = _encode_both(C, W, 2, cb)
    compare_encodings(g, r, flags, 96, 384, 2)


def test_encode_special_groups(C):
    """Zero groups, all-ones groups (exact ties), a basis vector, huge and
    tiny scales (the fp64 norm path), padding."""
    W = torch.zeros((8, 300))
    W[1] = 1.0
    W[2, 5] = 1.0
    W[3] = S.normal((300,), 3, 1e-20)
    W[4] = S.normal((300,), 4, 1e15)
    W[5, :128] = 0.25
    W[6] = S.normal((300,), 6, 1.0)
    W[7, 299] = -3.0
    for bits in (2, 3, 4, 5):
        g, r, flags = _encode_both(C, W, bits)
        compare_encodings(g, r, flags, 8, 300, bits)


def test_encode_ties_match_oracle_tie_rule(C):
    """All-ones rows put 127 exact zeros per group on the middle boundary of
    the symmetric codebook; the tie rule (smaller index) must hold on the
    GPU too, so these flagged coordinates must still agree."""
    W = torch.ones((4, 256))
    g, r, flags = _encode_both(C, W, 2)
    cg, _ = O.unpack(g, 4, 256, 2)
    cr, _ = O.unpack(r, 4, 256, 2)
    assert np.array_equal(cg, cr)
    assert np.all(cg[:, 1:128] == 1)


def test_encode_full_size_sampled_rows(C):
    """8192x8192 with 1% outliers, encoded whole on the GPU in the launch
    configuration of the benchmark; the oracle re-encodes sampled rows."""
    W = S.encode_matrix(0, device="cuda")
    blob = C.cq_encode(W, 2, O.analytic_codebook(2))
    torch.cuda.synchronize()
    rows = np.array([0, 1, 777, 4095, 4096, 8190, 8191])
    Wr = W[torch.from_numpy(rows).cuda()].cpu().numpy()
    blob_ref, flags, _ = O.encode(Wr, 2, O.analytic_codebook(2))
    from tests.gpu_helpers import sub_blob
    g = sub_blob(blob.cpu().numpy(), 8192, 8192, 2, rows)
    compare_encodings(g, blob_ref, flags, len(rows), 8192, 2)


def test_encode_decode_step_set_sampled(C):
    mats = S.decode_step_mats()
    from tests.gpu_helpers import sub_blob
    for m in mats[::9] + [mats[-1]]:
        W = S.decode_weights(m)
        blob = C.cq_encode(W.cuda(), m.bits, O.analytic_codebook(m.bits)).cpu().numpy()
        rows = np.arange(0, m.out, max(1, m.out // 16))
        blob_ref, flags, _ = O.encode(W.numpy()[rows], m.bits, O.analytic_codebook(m.bits))
        compare_encodings(sub_blob(blob, m.out, m.n_in, m.bits, rows), blob_ref, flags,
                          len(rows), m.n_in, m.bits)


@pytest.mark.parametrize("shape", [(1, 512), (55, 512), (7, 129), (2048, 512), (3, 1)])
def test_act_quant_bit_exact(C, shape):
    X = S.normal(shape, 31, 1.0)
    X[0, 0] = 0.0
    if shape[0] > 2:
        X[2] = 0.0  # an all-zero token
    q_ref, s_ref = O.act_quant_int8(X.numpy())
    q, s = C.cq_act_quant_int8(X.cuda())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy(), s_ref)
