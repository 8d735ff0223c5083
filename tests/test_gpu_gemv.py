"""GPU parity of cq_gemv / cq_gemv_grouped against the oracle's dense
product (dequantise with the explicit Hadamard matrix, multiply in fp64).
Blobs come from the oracle encoder or are seeded random byte strings; no
oracle input comes from the CUDA path."""
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


def _oracle_y(blob, out, n_in, bits, cb, xt):
    What = O.dequant(blob, out, n_in, bits, cb)
    return O.matmul(What, xt)


def _rand_blob(out, n_in, bits, seed):
    ip = O.in_padded(n_in)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // 128, seed, ternary=bits == 5)


def _run(C, blob, out, n_in, bits, cb, x, xs=None):
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda(),
                  None if xs is None else xs.cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_gemv_single_matrix_config(C, bits):
    """512x512, W ~ N(0, 0.02^2) seed 0 encoded by the oracle, x ~ N(0,1)
    seed 1, batch 1 (CQ3/CQ4/ternary on the same shape)."""
    W = S.normal((512, 512), 0, S.W_STD)
    x = S.normal((1, 512), 1)
    cb = O.analytic_codebook(bits)
    blob, _, _ = O.encode(W.numpy(), bits, cb)
    y = _run(C, blob, 512, 512, bits, cb, x)
    y_ref, bound = _oracle_y(blob, 512, 512, bits, cb, x.numpy())
    worst = check_matmul(y, y_ref, bound, f"cq{bits}")
    print(f"cq{bits}: max |err|/bound {worst:.2e}")


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("B", [1, 2, 5, 16])
@pytest.mark.parametrize("shape", [(1, 128), (3, 129), (37, 200), (300, 1024)])
def test_gemv_shapes_batches_fp32(C, bits, B, shape):
    out, n_in = shape
    blob = _rand_blob(out, n_in, bits, 100 + out + n_in + bits)
    cb = O.analytic_codebook(bits)
    x = S.normal((B, n_in), 3 + B)
    y = _run(C, blob, out, n_in, bits, cb, x)
    y_ref, bound = _oracle_y(blob, out, n_in, bits, cb, x.numpy())
    check_matmul(y, y_ref, bound, f"bits={bits} B={B} {shape}")


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("B", [1, 16])
def test_gemv_int8_activations(C, bits, B):
    out, n_in = 260, 640
    blob = _rand_blob(out, n_in, bits, 55 + B)
    cb = O.analytic_codebook(bits)
    X = S.normal((B, n_in), 9)
    q, s = O.act_quant_int8(X.numpy())
    y = _run(C, blob, out, n_in, bits, cb, torch.from_numpy(q), torch.from_numpy(s))
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    y_ref, bound = _oracle_y(blob, out, n_in, bits, cb, xt)
    check_matmul(y, y_ref, bound, f"int8 bits={bits} B={B}")


def test_gemv_empirical_codebook(C):
    x0 = np.random.RandomState(0).randn(400000)
    cb = (O.lloyd_max_samples(x0, 4, 200) / np.sqrt(128)).astype(np.float32)
    blob = _rand_blob(128, 512, 2, 77)
    x = S.normal((1, 512), 78)
    y = _run(C, blob, 128, 512, 2, cb, x)
    y_ref, bound = _oracle_y(blob, 128, 512, 2, cb, x.numpy())
    check_matmul(y, y_ref, bound, "empirical")


def test_gemv_long_input_large_batch(C):
    """Input long enough that a batch of 16 splits the reduction over
    several work items."""
    out, n_in = 64, 14336
    blob = _rand_blob(out, n_in, 3, 5)
    cb = O.analytic_codebook(3)
    x = S.normal((16, n_in), 6)
    y = _run(C, blob, out, n_in, 3, cb, x)
    y_ref, bound = _oracle_y(blob, out, n_in, 3, cb, x.numpy())
    check_matmul(y, y_ref, bound, "long input")


def test_gemv_zero_weights_and_empty(C):
    cb = O.analytic_codebook(2)
    blob = np.zeros(O.packed_bytes(5, 256, 128, 2), dtype=np.uint8)
    y = _run(C, blob, 5, 256, 2, cb, S.normal((2, 256), 1))
    assert np.all(y == 0)
    # in = 0: the product is defined and zero
    y = C.cq_gemv(torch.zeros(0, dtype=torch.uint8, device="cuda"), 4, 0, 2, cb,
                  torch.zeros((1, 0), device="cuda"))
    assert torch.all(y == 0)
    # out = 0: nothing to do
    y = C.cq_gemv(torch.zeros(0, dtype=torch.uint8, device="cuda"), 0, 128, 2, cb,
                  torch.zeros((1, 128), device="cuda"))
    assert y.shape == (1, 0)


def _decode_items(C, mats, blobs, xq, xs, cbs):
    items = []
    for m, b in zip(mats, blobs):
        items.append(dict(blob=b, out=m.out, **{"in": m.n_in}, bits=m.bits, codebook=cbs[m.bits],
                          x=xq[m.act], x_scale=xs[m.act]))
    return items


def test_gemv_grouped_decode_step_full_size(C):
    """The full Needle-shaped decode step (136 matrices, one launch) on
    seeded random blobs and int8 per-token activations; the oracle checks 24
    sampled rows of every matrix."""
    mats = S.decode_step_mats()
    cbs = {b: O.analytic_codebook(b) for b in (2, 4)}
    blobs_np = [_rand_blob(m.out, m.n_in, m.bits, 9000 + i) for i, m in enumerate(mats)]
    blobs = [torch.from_numpy(b).cuda() for b in blobs_np]
    qs, ss = [], []
    for a in range(S.n_activations(mats)):
        q, s = O.act_quant_int8(S.decode_activation(a).numpy())
        qs.append(q)
        ss.append(s)
    xq = [torch.from_numpy(q).cuda() for q in qs]
    xs = [torch.from_numpy(s).cuda() for s in ss]
    ys = C.cq_gemv_grouped(_decode_items(C, mats, blobs, xq, xs, cbs))
    torch.cuda.synchronize()
    rng = np.random.RandomState(0)
    for i, m in enumerate(mats):
        rows = np.sort(rng.choice(m.out, 24, replace=False))
        sb = sub_blob(blobs_np[i], m.out, m.n_in, m.bits, rows)
        xt = qs[m.act].astype(np.float64) * ss[m.act].astype(np.float64)[:, None]
        y_ref, bound = _oracle_y(sb, len(rows), m.n_in, m.bits, cbs[m.bits], xt)
        check_matmul(ys[i].cpu().numpy()[:, rows], y_ref, bound, m.name)


def test_gemv_grouped_equals_single_calls(C):
    """Grouping changes only the launch: each output equals its single call
    up to fp32 summation order."""
    mats = S.decode_step_mats(layers=2)
    cbs = {b: O.analytic_codebook(b) for b in (2, 4)}
    blobs = [torch.from_numpy(_rand_blob(m.out, m.n_in, m.bits, 300 + i)).cuda() for i, m in enumerate(mats)]
    xs = [S.normal((1, 512), 400 + a).cuda() for a in range(S.n_activations(mats))]
    items = [dict(blob=b, out=m.out, **{"in": m.n_in}, bits=m.bits, codebook=cbs[m.bits], x=xs[m.act])
             for m, b in zip(mats, blobs)]
    ys = C.cq_gemv_grouped(items)
    for it, yg in zip(items, ys):
        y1 = C.cq_gemv(it["blob"], it["out"], it["in"], it["bits"], it["codebook"], it["x"])
        assert torch.allclose(y1, yg, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("B", [1, 4])
def test_gemv_shared_input_qkvg(C, B):
    """Shared-input entry point: Q, K, V and gate of one Needle layer read one
    int8 activation; results are bit-identical to the grouped call over the
    same matrices and match the oracle."""
    outs, n_in, bits = [512, 256, 256, 512], 512, 2
    cb = O.analytic_codebook(bits)
    blobs_np = [_rand_blob(o, n_in, bits, 510 + j) for j, o in enumerate(outs)]
    blobs = [torch.from_numpy(b).cuda() for b in blobs_np]
    q, s = O.act_quant_int8(S.normal((B, n_in), 520 + B).numpy())
    xq, xs = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    ys = C.cq_gemv_shared(blobs, outs, n_in, bits, cb, xq, xs)
    items = [dict(blob=b, out=o, **{"in": n_in}, bits=bits, codebook=cb, x=xq, x_scale=xs)
             for b, o in zip(blobs, outs)]
    yg = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    for j in range(len(outs)):
        assert ys[j].shape == (B, outs[j])
        assert torch.equal(ys[j], yg[j])
        y_ref, bound = _oracle_y(blobs_np[j], outs[j], n_in, bits, cb, xt)
        check_matmul(ys[j].cpu().numpy(), y_ref, bound, f"shared mat {j}")


def test_gemv_shared_rejects_bad_counts(C):
    cb = O.analytic_codebook(2)
    x = torch.zeros((1, 128), device="cuda")
    with pytest.raises(ValueError):
        C.cq_gemv_shared([], [], 128, 2, cb, x)
    blobs = [torch.zeros(O.packed_bytes(8, 128, 128, 2), dtype=torch.uint8, device="cuda")] * 300
    with pytest.raises(C.CQError):
        C.cq_gemv_shared(blobs, [8] * 300, 128, 2, cb, x)


@pytest.mark.parametrize("shape", S.SWEEP_SHAPES)
@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("B", [1, 16])
def test_gemv_sweep_full_size_sampled(C, shape, bits, B):
    """Width sweep at full size (4096x4096, 14336x4096) in the benchmark's
    launch configuration; the oracle checks 8 sampled rows."""
    out, n_in = shape
    blob = _rand_blob(out, n_in, bits, 700 + bits + out // 1024)
    cb = O.analytic_codebook(bits)
    x = S.normal((B, n_in), 800 + B)
    y = _run(C, blob, out, n_in, bits, cb, x)
    rows = np.array([0, 1, out // 3, out // 2, out - 129, out - 2, out - 1, 17])
    y_ref, bound = _oracle_y(sub_blob(blob, out, n_in, bits, rows), len(rows), n_in, bits, cb, x.numpy())
    check_matmul(y[:, rows], y_ref, bound, f"sweep {shape} cq{bits} B={B}")


@pytest.mark.parametrize("B", [1, 3])
def test_gemv_host_resident_activations_and_outputs(C, B):
    """x, x_scale and y in pinned host memory: the kernels read and write them
    in place, and the result is bit-identical to the device-resident call."""
    out, n_in, bits = 272, 640, 2
    blob = torch.from_numpy(_rand_blob(out, n_in, bits, 61)).cuda()
    cb = O.analytic_codebook(bits)
    q, s = O.act_quant_int8(S.normal((B, n_in), 62).numpy())
    xq_d, xs_d = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    y_d = C.cq_gemv(blob, out, n_in, bits, cb, xq_d, xs_d)
    xq_h, xs_h = torch.from_numpy(q).pin_memory(), torch.from_numpy(s).pin_memory()
    y_h = torch.full((B, out), float("nan")).pin_memory()
    C.cq_gemv(blob, out, n_in, bits, cb, xq_h, xs_h, y=y_h)
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_d.cpu())


def test_gemv_grouped_mixed_widths_activations_and_batches(C):
    """One grouped call over many small matrices of every tensor-core width
    (CQ2, ternary, CQ4, binary), inputs of 1 to 12 groups, batches 1 to 4,
    fp32 and int8 activations, some shared between consecutive matrices:
    the launch cuts these into runs that cross matrix, activation and width
    boundaries. Every output is checked against the oracle."""
    rng = np.random.RandomState(41)
    items, refs = [], []
    x_prev = None
    for i in range(60):
        bits = [2, 5, 4, 1][i % 4] if i < 40 else 2
        n_in = int(rng.choice([128, 200, 384, 512, 1000, 1536]))
        out = int(rng.choice([1, 16, 40, 129, 256, 300]))
        B = int(rng.choice([1, 2, 3, 4]))
        if x_prev is not None and x_prev[0].shape[1] == n_in and rng.rand() < 0.5:
            x, xs, xt = x_prev  # shares the previous matrix's activation
        elif rng.rand() < 0.5:
            xf = S.normal((B, n_in), 600 + i)
            x, xs, xt = xf.cuda(), None, xf.numpy().astype(np.float64)
        else:
            q, s = O.act_quant_int8(S.normal((B, n_in), 600 + i).numpy())
            x, xs = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
            xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
        x_prev = (x, xs, xt)
        cb = O.analytic_codebook(bits)
        blob = _rand_blob(out, n_in, bits, 650 + i)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=bits, codebook=cb, x=x,
                          x_scale=xs))
        refs.append(_oracle_y(blob, out, n_in, bits, cb, xt))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for i, (y, (y_ref, bound)) in enumerate(zip(ys, refs)):
        check_matmul(y.cpu().numpy(), y_ref, bound, f"item {i}")
