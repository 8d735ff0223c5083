"""GPU parity for groups of 64 and binary (1-bit) CQ codes ("The .cact
format", "Cactus Quants": binary packs eight codes per byte with closed-form
centroids; OpenNeedle docs/reference.md tests group 64 and 128): encoder,
fp32 GEMV and row gather against the oracle on identical seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import check_matmul, compare_encodings, sub_blob

pytestmark = pytest.mark.gpu

GEOMS = [(64, 1), (64, 2), (64, 3), (64, 4), (64, 5), (128, 1)]


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _rand_blob(out, n_in, bits, group, seed):
    ip = O.in_padded(n_in, group)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // group, seed, ternary=bits == 5)


@pytest.mark.parametrize("group,bits", GEOMS)
@pytest.mark.parametrize("shape", [(512, 512), (3, 65), (33, 200), (1, 1), (130, 1000), (3, 64), (7, 320)])
def test_encode_parity(C, group, bits, shape):
    W = S.normal(shape, 70 + bits + group, S.W_STD)
    cb = O.analytic_codebook(bits, group)
    ref, flags, _ = O.encode(W.numpy(), bits, cb, group)
    got = C.cq_encode(W.cuda(), bits, cb, group=group)
    torch.cuda.synchronize()
    nb, nbm = compare_encodings(got.cpu().numpy(), ref, flags, shape[0], shape[1], bits, group)
    print(f"group={group} bits={bits} {shape}: {nb} boundary coordinates, {nbm} differ")


@pytest.mark.parametrize("group,bits", [(64, 2), (128, 1)])
def test_encode_outliers_full_width(C, group, bits):
    """4096 x 4096 with 1% outliers x20 (the encode workload's recipe at a
    smaller size)."""
    W = S.with_outliers(S.normal((4096, 4096), 80, S.W_STD), 81)
    cb = O.analytic_codebook(bits, group)
    got = C.cq_encode(W.cuda(), bits, cb, group=group).cpu().numpy()
    rows = np.array([0, 1, 977, 2048, 4095])
    ref, flags, _ = O.encode(W.numpy()[rows], bits, cb, group)
    compare_encodings(sub_blob(got, 4096, 4096, bits, rows, group), ref, flags, len(rows), 4096, bits, group)


@pytest.mark.parametrize("group,bits", GEOMS)
@pytest.mark.parametrize("B", [1, 3, 16])
@pytest.mark.parametrize("shape", [(1, 64), (3, 65), (37, 200), (300, 1024)])
def test_gemv_parity(C, group, bits, B, shape):
    out, n_in = shape
    blob = _rand_blob(out, n_in, bits, group, 90 + out + n_in + bits + group)
    cb = O.analytic_codebook(bits, group)
    x = S.normal((B, n_in), 91 + B)
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda(), group=group)
    torch.cuda.synchronize()
    y_ref, bound = O.matmul(O.dequant(blob, out, n_in, bits, cb, group), x.numpy())
    check_matmul(y.cpu().numpy(), y_ref, bound, f"g{group} cq{bits} B={B} {shape}")


@pytest.mark.parametrize("group,bits", [(64, 2), (64, 4), (128, 1)])
def test_gemv_int8_and_grouped_with_group128(C, group, bits):
    """int8 activations; one grouped launch mixing these matrices with
    group-128 CQ2 ones (which take the tensor-core path)."""
    n_in = 640
    q, s = O.act_quant_int8(S.normal((2, n_in), 92).numpy())
    xq, xs = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    items, refs = [], []
    for j, (g, b) in enumerate([(group, bits), (128, 2), (group, bits)]):
        out = 96 + 16 * j
        blob = _rand_blob(out, n_in, b, g, 93 + j)
        cb = O.analytic_codebook(b, g)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=b, codebook=cb,
                          x=xq, x_scale=xs, group=g))
        refs.append(O.matmul(O.dequant(blob, out, n_in, b, cb, g), xt))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for y, (y_ref, bound) in zip(ys, refs):
        check_matmul(y.cpu().numpy(), y_ref, bound, f"grouped g{group} cq{bits}")


@pytest.mark.parametrize("group,bits", [(64, 2), (128, 1)])
def test_gemv_full_size_sampled(C, group, bits):
    out, n_in = 4096, 4096
    blob = _rand_blob(out, n_in, bits, group, 94)
    cb = O.analytic_codebook(bits, group)
    x = S.normal((1, n_in), 95)
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda(), group=group).cpu().numpy()
    rows = np.array([0, 1, 1234, 2047, 4095])
    sb = sub_blob(blob, out, n_in, bits, rows, group)
    y_ref, bound = O.matmul(O.dequant(sb, len(rows), n_in, bits, cb, group), x.numpy())
    check_matmul(y[:, rows], y_ref, bound, f"full g{group} cq{bits}")


def _gather_bound(blob, out, n_in, bits, group, cb, rows):
    """fp32 transform of one group (log2(group) rounded stages over partial
    sums bounded by sum|c|, then one rounded scaling): |err| <= 1e-6 *
    n/sqrt(group) * sum_k |c[q_k]| per element."""
    codes, norms = O.unpack(blob, out, n_in, bits, group)
    lv = np.zeros(16)
    if bits == 5:
        c = float(cb[2])
        lv[1], lv[2], lv[3] = c, -2.0 * c, -c
    else:
        lv[:len(cb)] = np.asarray(cb, dtype=np.float64)
    n = O.f16_bits_to_f32(norms).astype(np.float64).reshape(norms.shape)
    ng = codes.shape[1] // group
    s = np.abs(lv[codes]).reshape(out, ng, group).sum(axis=2) * n / math.sqrt(group)
    return np.repeat(s, group, axis=1)[:, :n_in][rows] * 1e-6


@pytest.mark.parametrize("group,bits", GEOMS)
@pytest.mark.parametrize("n_in", [64, 96, 192, 200, 512])
def test_gather_parity(C, group, bits, n_in):
    out = 50
    blob = _rand_blob(out, n_in, bits, group, 96 + n_in + bits + group)
    cb = O.analytic_codebook(bits, group)
    idx = np.array([3, 0, 49, 3, 17, 17, 48], dtype=np.int32)
    got = C.cq_gather_rows(torch.from_numpy(blob).cuda(), out, n_in, bits, cb,
                           torch.from_numpy(idx).cuda(), group=group).cpu().numpy()
    ref = O.gather_rows(blob, out, n_in, bits, cb, idx, group)
    bound = _gather_bound(blob, out, n_in, bits, group, cb, idx)
    assert np.all(np.abs(got - ref) <= bound), f"g{group} cq{bits} in={n_in}"


def test_gather_out_of_range_group64(C):
    out, n_in = 8, 192
    blob = _rand_blob(out, n_in, 2, 64, 97)
    cb = O.analytic_codebook(2, 64)
    got = C.cq_gather_rows(torch.from_numpy(blob).cuda(), out, n_in, 2, cb,
                           torch.tensor([1, 8, -1], dtype=torch.int32, device="cuda"), group=64)
    with pytest.raises(C.CQError):
        C.cq_device_status()
    g = got.cpu().numpy()
    assert np.all(g[1:] == 0)
    ref = O.gather_rows(blob, out, n_in, 2, cb, [1], 64)
    assert np.all(np.abs(g[0] - ref[0]) <= _gather_bound(blob, out, n_in, 2, 64, cb, [1])[0])


@pytest.mark.parametrize("group,bits", [(64, 1), (64, 2), (64, 4), (128, 1), (128, 4)])
@pytest.mark.parametrize("B", [1, 3])
@pytest.mark.parametrize("shape", [(200, 2048), (37, 4096)])
def test_gemv_wide_inputs(C, group, bits, B, shape):
    """Inputs of 16 to 32 spans of 128 take the split tensor-core products
    (a rotation launch, then per-warp units; groups of 64 as two chains per
    span with their own norms), ragged row counts included."""
    out, n_in = shape
    blob = _rand_blob(out, n_in, bits, group, 98 + out + bits + group + B)
    cb = O.analytic_codebook(bits, group)
    x = S.normal((B, n_in), 99 + B)
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda(), group=group)
    torch.cuda.synchronize()
    y_ref, bound = O.matmul(O.dequant(blob, out, n_in, bits, cb, group), x.numpy())
    check_matmul(y.cpu().numpy(), y_ref, bound, f"wide g{group} cq{bits} B={B} {shape}")


def test_gemv_more_wide_matrices_than_one_launch_holds(C):
    """210 wide matrices (16 rows each, in = 2048; CQ2 and binary at group
    128 interleaved) in one grouped call: more than one split launch holds
    (128 matrices), so each code width's set is cut in two launches."""
    items, refs = [], []
    x = S.normal((2, 2048), 120)
    xd = x.cuda()
    for j in range(210):
        group, bits = ((128, 2), (128, 1))[j % 2]
        blob = _rand_blob(16, 2048, bits, group, 2000 + j)
        cb = O.analytic_codebook(bits, group)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=16, **{"in": 2048}, bits=bits, codebook=cb,
                          x=xd, group=group))
        if j % 23 == 0:  # the oracle checks a sample
            refs.append((j, O.matmul(O.dequant(blob, 16, 2048, bits, cb, group), x.numpy())))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for j, (y_ref, bound) in refs:
        check_matmul(ys[j].cpu().numpy(), y_ref, bound, f"matrix {j}")


def _gemm_check(C, group, bits, out, n_in, M, seed, toks=None):
    blob = _rand_blob(out, n_in, bits, group, seed)
    cb = O.analytic_codebook(bits, group)
    q, s = O.act_quant_int8(S.normal((M, n_in), seed + 1).numpy())
    Y = C.cq_gemm(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda(), group=group)
    torch.cuda.synchronize()
    toks = np.arange(M) if toks is None else np.asarray(toks)
    xt = q[toks].astype(np.float64) * s[toks].astype(np.float64)[:, None]
    y_ref, bound = O.matmul(O.dequant(blob, out, n_in, bits, cb, group), xt)
    check_matmul(Y.cpu().numpy()[toks], y_ref, bound, f"gemm g{group} cq{bits} M={M} {out}x{n_in}")


@pytest.mark.parametrize("group,bits", [(64, 1), (64, 2), (64, 3), (64, 4), (64, 5), (128, 1)])
@pytest.mark.parametrize("shape", [(200, 384), (3, 128), (512, 512)])
@pytest.mark.parametrize("M", [64, 2048])
def test_gemm_parity(C, group, bits, shape, M):
    """Tensor-core product over int8 tokens: groups of 64 (each half of a
    128-wide span rotated by H_64 with its own norm) and binary codes."""
    out, n_in = shape
    toks = None if M <= 64 else [0, 1, 130, 1023, 1500, 2047]
    _gemm_check(C, group, bits, out, n_in, M, 300 + bits + group + out, toks)


@pytest.mark.parametrize("shape", [(130, 1000), (64, 4096)])
@pytest.mark.parametrize("M", [64, 2048])
def test_gemm_binary_rotated_activations(C, shape, M):
    """Binary codes on inputs wider than 512 (the product over rotated
    activations), ragged input width included."""
    out, n_in = shape
    toks = None if M <= 64 else [0, 5, 999, 2047]
    _gemm_check(C, 128, 1, out, n_in, M, 400 + out, toks)


def test_gemm_grouped_mixes_group64_binary_and_cq2(C):
    n_in = 256
    q, s = O.act_quant_int8(S.normal((70, n_in), 410).numpy())
    xq, xs = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    items, refs = [], []
    for j, (g, b) in enumerate([(64, 2), (128, 1), (128, 2), (64, 1), (64, 4)]):
        out = 90 + 40 * j
        blob = _rand_blob(out, n_in, b, g, 411 + j)
        cb = O.analytic_codebook(b, g)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=b, codebook=cb,
                          Xq=xq, x_scale=xs, group=g))
        refs.append(O.matmul(O.dequant(blob, out, n_in, b, cb, g), xt))
    Ys = C.cq_gemm_grouped(items)
    torch.cuda.synchronize()
    for j, (Y, (y_ref, bound)) in enumerate(zip(Ys, refs)):
        check_matmul(Y.cpu().numpy(), y_ref, bound, f"grouped item {j}")


@pytest.mark.parametrize("n_in", [200, 640])
def test_gemm_group64_rejects_unsupported_widths(C, n_in):
    """Groups of 64 in the product: whole 128-wide spans, at most 512 inputs."""
    blob = _rand_blob(8, n_in, 2, 64, 420)
    q = torch.zeros((4, n_in), dtype=torch.int8, device="cuda")
    s = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(C.CQError):
        C.cq_gemm(torch.from_numpy(blob).cuda(), 8, n_in, 2, O.analytic_codebook(2, 64), q, s, group=64)
