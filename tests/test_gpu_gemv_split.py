"""GPU parity of the split GEMV products (inputs of 16 groups and more at
group 128, batches of 1 to 4, 1-, 2-, 3- and 4-bit codes and ternary): units of
(matrix, k-slice, 16-row tile), k-slices of a tile summed in slice order by
the last one to finish. Checked against the oracle's dense product on the
same seeded inputs; repeated calls must give the same bits."""
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


def _rows(out):
    r = [0, 1, 15, 16, out // 3, out // 2, out - 17, out - 16, out - 1]
    return np.array(sorted({min(max(v, 0), out - 1) for v in r}))


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("B", [1, 2, 4])
@pytest.mark.parametrize("shape", [(4096, 4096), (4100, 3000), (129, 16384), (40, 2048), (33, 640)])
def test_split_single_matrices(C, bits, B, shape):
    """One matrix per call: 4096 rows (k-sliced in four), a ragged last tile
    and an input that is not a multiple of 128, a 16384-wide input over nine
    tiles (deep k-slices), and a matrix of three tiles."""
    out, n_in = shape
    blob = _rand_blob(out, n_in, bits, 3100 + bits + B + out % 97)
    cb = O.analytic_codebook(bits)
    x = S.normal((B, n_in), 3200 + B)
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda())
    torch.cuda.synchronize()
    rows = _rows(out)
    y_ref, bound = O.matmul(O.dequant(sub_blob(blob, out, n_in, bits, rows), len(rows), n_in, bits, cb), x.numpy())
    check_matmul(y.cpu().numpy()[:, rows], y_ref, bound, f"split {shape} bits={bits} B={B}")


@pytest.mark.parametrize("B", [1, 3])
def test_split_int8_activations(C, B):
    out, n_in, bits = 520, 4096, 2
    blob = _rand_blob(out, n_in, bits, 3300 + B)
    cb = O.analytic_codebook(bits)
    q, s = O.act_quant_int8(S.normal((B, n_in), 3310 + B).numpy())
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    y_ref, bound = O.matmul(O.dequant(blob, out, n_in, bits, cb), xt)
    check_matmul(y.cpu().numpy(), y_ref, bound, f"split int8 B={B}")


def test_split_repeat_calls_bit_identical(C):
    """The tile counters are cleared by every call's rotation launch and the
    k-slices are added in slice order: the same call gives the same bits,
    also with another k-sliced call in between and from a CUDA graph."""
    out, n_in, bits = 1000, 8192, 2
    blob = torch.from_numpy(_rand_blob(out, n_in, bits, 3400)).cuda()
    other = torch.from_numpy(_rand_blob(300, 4096, 1, 3401)).cuda()
    cb, cb1 = O.analytic_codebook(bits), O.analytic_codebook(1)
    x = S.normal((2, n_in), 3402).cuda()
    x2 = S.normal((1, 4096), 3403).cuda()
    y0 = C.cq_gemv(blob, out, n_in, bits, cb, x).clone()
    for _ in range(3):
        C.cq_gemv(other, 300, 4096, 1, cb1, x2)
        y1 = C.cq_gemv(blob, out, n_in, bits, cb, x)
        torch.cuda.synchronize()
        assert torch.equal(y0, y1)
    y = torch.empty_like(y0)
    plan = C.GemvPlan([dict(blob=blob, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=x, y=y)])
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        plan.run(st)  # grows the workspace before capture
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        plan.run(st)
    for _ in range(3):
        y.zero_()
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        assert torch.equal(y, y0)


def test_split_grouped_with_every_other_route(C):
    """One grouped call whose matrices go to the split products (CQ2, CQ3,
    CQ4, binary at batch <= 4, group 64), the sliced products (batch 8) and
    the decode kernel (short inputs): every output against the oracle."""
    specs = [(300, 4096, 2, 128, 1), (200, 2048, 4, 128, 2), (64, 3000, 1, 128, 1), (150, 2048, 3, 128, 1),
             (96, 2048, 2, 64, 1), (130, 2048, 2, 128, 8), (256, 512, 2, 128, 1), (333, 4096, 5, 128, 4)]
    items, refs = [], []
    for i, (out, n_in, bits, group, B) in enumerate(specs):
        ip = O.in_padded(n_in, group)
        blob = S.random_blob(out * ip * O.width(bits) // 8, out * ip // group, 3500 + i, ternary=bits == 5)
        cb = O.analytic_codebook(bits, group)
        x = S.normal((B, n_in), 3520 + i)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=bits, codebook=cb,
                          x=x.cuda(), group=group))
        refs.append(O.matmul(O.dequant(blob, out, n_in, bits, cb, group), x.numpy()))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for i, (y, (y_ref, bound)) in enumerate(zip(ys, refs)):
        check_matmul(y.cpu().numpy(), y_ref, bound, f"item {i} {specs[i]}")


# ---- groups of 64 (two 64-point transforms and two norms per 128-span) ----

def _rand_blob64(out, n_in, bits, seed):
    return S.random_blob(out * n_in * O.width(bits) // 8, out * n_in // 64, seed, ternary=bits == 5)


@pytest.mark.parametrize("bits", [1, 2, 4])
@pytest.mark.parametrize("B", [1, 2, 4])
@pytest.mark.parametrize("shape", [(4096, 4096), (4100, 3072), (129, 16384), (40, 256)])
def test_split_group64_single_matrices(C, bits, B, shape):
    """Groups of 64 on the split products: 4096 rows (k-sliced), a ragged
    last tile, a 16384-wide input (deep k-slices) and two spans only."""
    out, n_in = shape
    blob = _rand_blob64(out, n_in, bits, 3600 + bits + B + out % 89)
    cb = O.analytic_codebook(bits, 64)
    x = S.normal((B, n_in), 3700 + B)
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, x.cuda(), group=64)
    torch.cuda.synchronize()
    rows = _rows(out)
    sb = sub_blob(blob, out, n_in, bits, rows, 64)
    y_ref, bound = O.matmul(O.dequant(sb, len(rows), n_in, bits, cb, 64), x.numpy())
    check_matmul(y.cpu().numpy()[:, rows], y_ref, bound, f"split g64 {shape} bits={bits} B={B}")


@pytest.mark.parametrize("B", [1, 4])
def test_split_group64_int8_activations(C, B):
    out, n_in, bits = 300, 2048, 2
    blob = _rand_blob64(out, n_in, bits, 3800 + B)
    cb = O.analytic_codebook(bits, 64)
    q, s = O.act_quant_int8(S.normal((B, n_in), 3810 + B).numpy())
    y = C.cq_gemv(torch.from_numpy(blob).cuda(), out, n_in, bits, cb, torch.from_numpy(q).cuda(),
                  torch.from_numpy(s).cuda(), group=64)
    torch.cuda.synchronize()
    xt = q.astype(np.float64) * s.astype(np.float64)[:, None]
    y_ref, bound = O.matmul(O.dequant(blob, out, n_in, bits, cb, 64), xt)
    check_matmul(y.cpu().numpy(), y_ref, bound, f"split g64 int8 B={B}")


def test_split_group64_and_group128_read_one_activation(C):
    """One activation read by group-64 and group-128 matrices in one call:
    each group size gets its own rotation of it (the halves of a span are
    not mixed for groups of 64), and the two go to separate split launches."""
    n_in, B = 4096, 2
    x = S.normal((B, n_in), 3900)
    xd = x.cuda()
    specs = [(520, 64, 2), (300, 128, 2), (200, 64, 1), (260, 128, 4), (100, 64, 4)]
    items, refs = [], []
    for i, (out, group, bits) in enumerate(specs):
        blob = (_rand_blob64(out, n_in, bits, 3910 + i) if group == 64 else _rand_blob(out, n_in, bits, 3910 + i))
        cb = O.analytic_codebook(bits, group)
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=out, **{"in": n_in}, bits=bits, codebook=cb,
                          x=xd, group=group))
        refs.append(O.matmul(O.dequant(blob, out, n_in, bits, cb, group), x.numpy()))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for i, (y, (y_ref, bound)) in enumerate(zip(ys, refs)):
        check_matmul(y.cpu().numpy(), y_ref, bound, f"item {i} {specs[i]}")


def test_split_group64_falls_back_to_streamed(C):
    """128 group-64 matrices of 16 x 4096, each with its own batch-4
    activation: no split plan fits every block's fragments (each unit is its
    own (matrix, k-slice) pair), so the call hands them to the streamed
    kernel. Every output still matches the oracle, as do those of group-128
    CQ2 matrices in the same call (the sliced kernel)."""
    items, refs = [], []
    cb64, cb128 = O.analytic_codebook(2, 64), O.analytic_codebook(2)
    for j in range(130):
        group = 128 if j >= 128 else 64
        blob = _rand_blob64(16, 4096, 2, 4000 + j) if group == 64 else _rand_blob(16, 4096, 2, 4000 + j)
        x = S.normal((4, 4096), 4200 + j)
        cb = cb64 if group == 64 else cb128
        items.append(dict(blob=torch.from_numpy(blob).cuda(), out=16, **{"in": 4096}, bits=2, codebook=cb,
                          x=x.cuda(), group=group))
        if j % 17 == 0 or j >= 127:
            refs.append((j, O.matmul(O.dequant(blob, 16, 4096, 2, cb, group), x.numpy())))
    ys = C.cq_gemv_grouped(items)
    torch.cuda.synchronize()
    for j, (y_ref, bound) in refs:
        check_matmul(ys[j].cpu().numpy(), y_ref, bound, f"matrix {j}")


def test_split_group64_repeat_calls_bit_identical(C):
    out, n_in = 2000, 8192
    blob = torch.from_numpy(_rand_blob64(out, n_in, 2, 4300)).cuda()
    cb = O.analytic_codebook(2, 64)
    x = S.normal((3, n_in), 4301).cuda()
    y0 = C.cq_gemv(blob, out, n_in, 2, cb, x, group=64).clone()
    for _ in range(3):
        y1 = C.cq_gemv(blob, out, n_in, 2, cb, x, group=64)
        torch.cuda.synchronize()
        assert torch.equal(y0, y1)
