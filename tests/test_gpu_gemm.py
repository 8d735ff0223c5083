"""GPU parity of cq_gemm / cq_gemm_grouped (int8 per-token activations)
against the oracle's dense fp64 product. x_t = s_t * q_t exactly as handed
to the GPU."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import check_matmul, sub_blob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _rand_blob(out, n_in, bits, seed):
    ip = O.in_padded(n_in)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, seed, ternary=bits == 5)


def _tokens(M, n_in, seed):
    q, s = O.act_quant_int8(S.normal((M, n_in), seed).numpy())
    return q, s


def _check(C, blob, out, n_in, bits, cb, q, s, rows=None, toks=None, what=""):
    Y = C.cq_gemm(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    Y = Y.cpu().numpy()
    rows = np.arange(out) if rows is None else rows
    toks = np.arange(q.shape[0]) if toks is None else toks
    xt = q[toks].astype(np.float64) * s[toks].astype(np.float64)[:, None]
    What = O.dequant(sub_blob(blob, out, n_in, bits, rows), len(rows), n_in, bits, cb)
    y_ref, bound = O.matmul(What, xt)
    return check_matmul(Y[np.ix_(toks, rows)], y_ref, bound, what)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("M", [1, 64, 130])
def test_gemm_small(C, bits, M):
    out, n_in = 200, 384
    blob = _rand_blob(out, n_in, bits, 10 + bits)
    q, s = _tokens(M, n_in, 20 + M)
    _check(C, blob, out, n_in, bits, O.analytic_codebook(bits), q, s, what=f"cq{bits} M={M}")


@pytest.mark.parametrize("shape", [(1, 128), (3, 129), (129, 300), (512, 512)])
def test_gemm_ragged(C, shape):
    out, n_in = shape
    blob = _rand_blob(out, n_in, 2, 33)
    q, s = _tokens(67, n_in, 34)
    _check(C, blob, out, n_in, 2, O.analytic_codebook(2), q, s, what=f"ragged {shape}")


def test_gemm_oracle_encoded_weights(C):
    W = S.normal((256, 512), 3, S.W_STD)
    cb = O.analytic_codebook(2)
    blob, _, _ = O.encode(W.numpy(), 2, cb)
    q, s = _tokens(64, 512, 4)
    _check(C, blob, 256, 512, 2, cb, q, s, what="encoded")


@pytest.mark.parametrize("M", [64, 256, 2048])
def test_gemm_grouped_prefill_full_size_sampled(C, M):
    """The Needle-shaped matrix set at prefill M (one rotation per distinct
    activation, one grouped GEMM launch per code width); sampled tokens and
    rows of a third of the matrices are checked against the oracle."""
    mats = S.decode_step_mats()
    cbs = {b: O.analytic_codebook(b) for b in (2, 4)}
    blobs_np = [_rand_blob(m.out, m.n_in, m.bits, 9100 + i) for i, m in enumerate(mats)]
    acts = [_tokens(M, 512, 3000 + a) for a in range(S.n_activations(mats))]
    items = []
    for i, m in enumerate(mats):
        items.append(dict(blob=torch.from_numpy(blobs_np[i]).cuda(), out=m.out, **{"in": m.n_in}, bits=m.bits,
                          codebook=cbs[m.bits], Xq=torch.from_numpy(acts[m.act][0]).cuda(),
                          x_scale=torch.from_numpy(acts[m.act][1]).cuda()))
    Ys = C.cq_gemm_grouped(items)
    torch.cuda.synchronize()
    rng = np.random.RandomState(M)
    for i, m in enumerate(mats):
        if i % 3 and i != len(mats) - 1:
            continue
        rows = np.sort(rng.choice(m.out, 16, replace=False))
        toks = np.sort(rng.choice(M, min(M, 16), replace=False))
        q, s = acts[m.act]
        xt = q[toks].astype(np.float64) * s[toks].astype(np.float64)[:, None]
        What = O.dequant(sub_blob(blobs_np[i], m.out, m.n_in, m.bits, rows), len(rows), m.n_in, m.bits, cbs[m.bits])
        y_ref, bound = O.matmul(What, xt)
        check_matmul(Ys[i].cpu().numpy()[np.ix_(toks, rows)], y_ref, bound, f"{m.name} M={M}")


def test_gemm_empty(C):
    cb = O.analytic_codebook(2)
    Y = C.cq_gemm(torch.zeros(O.packed_bytes(4, 0, 128, 2), dtype=torch.uint8, device="cuda"), 4, 0, 2, cb,
                  torch.zeros((3, 0), dtype=torch.int8, device="cuda"), torch.ones(3, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


def test_gemm_grouped_mixed_inputs(C):
    """One grouped call over inputs above 512 (rotated activations), at most
    512 and aligned (activations read in place), and rows that are not a
    multiple of 16 bytes (padded copies), across all code widths."""
    M = 200
    shapes = [(300, 640, 2), (256, 512, 4), (129, 300, 3), (64, 128, 5), (200, 384, 2)]
    items, refs = [], []
    for i, (out, n_in, bits) in enumerate(shapes):
        cb = O.analytic_codebook(bits)
        blob = _rand_blob(out, n_in, bits, 700 + i)
        q, s = _tokens(M, n_in, 800 + i)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=bits, codebook=cb,
                          Xq=torch.from_numpy(q).cuda(), x_scale=torch.from_numpy(s).cuda()))
        refs.append((blob, out, n_in, bits, cb, q, s))
    Ys = C.cq_gemm_grouped(items)
    torch.cuda.synchronize()
    for Y, (blob, out, n_in, bits, cb, q, s) in zip(Ys, refs):
        xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
        What = O.dequant(blob, out, n_in, bits, cb)
        y_ref, bound = O.matmul(What, xt)
        check_matmul(Y.cpu().numpy(), y_ref, bound, f"mixed out={out} in={n_in} bits={bits}")


def test_gemm_misaligned_activation_rows(C):
    """Activations whose base address is not 16-byte aligned take the padded
    copy; the result is the same as for an aligned copy of the same values."""
    out, n_in, M = 256, 256, 70
    cb = O.analytic_codebook(2)
    blob = torch.from_numpy(_rand_blob(out, n_in, 2, 901)).cuda()
    q, s = _tokens(M, n_in, 902)
    buf = torch.zeros(M * n_in + 16, dtype=torch.int8, device="cuda")
    Xmis = buf[3:3 + M * n_in].view(M, n_in)
    Xmis.copy_(torch.from_numpy(q).cuda())
    assert Xmis.data_ptr() % 16 != 0
    xs = torch.from_numpy(s).cuda()
    Y1 = C.cq_gemm(blob, out, n_in, 2, cb, Xmis, xs)
    Y2 = C.cq_gemm(blob, out, n_in, 2, cb, torch.from_numpy(q).cuda(), xs)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    _check(C, blob.cpu().numpy(), out, n_in, 2, cb, q, s, what="misaligned")
