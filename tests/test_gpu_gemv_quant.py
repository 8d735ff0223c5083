"""GPU checks of CQ_X_F32Q activations (fp32, quantised per token inside the
GEMV call with the activation quantiser's rule, OpenNeedle reference
fake_quant_act): on every GEMV route the outputs are bit-identical to
cq_act_quant_int8 followed by the int8 call, and match the oracle's product
of the dequantised matrix with the oracle's quantised activations."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import check_matmul

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _blob(out, n_in, bits, group, seed):
    ip = O.in_padded(n_in, group)
    return S.random_blob(out * ip * O.width(bits) // 8, out * ip // group, seed, ternary=bits == 5)


def _pair(C, specs, seed, host_x=False):
    """One grouped call with quantize=True and the same call on explicitly
    quantised int8 activations; returns both outputs and the oracle refs."""
    items_q, items_i, refs = [], [], []
    acts = {}
    for i, (out, n_in, bits, group, B, a) in enumerate(specs):
        if a not in acts:
            x = S.normal((B, n_in), seed + 100 * a) * 3.0
            if a % 3 == 2:
                x[0] = 0.0  # an all-zero token: scale 1, product 0
            xd = x.pin_memory() if host_x else x.cuda()
            q, s = C.cq_act_quant_int8(x.cuda())
            acts[a] = (x, xd, q, s)
        x, xd, q, s = acts[a]
        blob = _blob(out, n_in, bits, group, seed + i)
        cb = O.analytic_codebook(bits, group)
        bd = torch.from_numpy(blob).cuda()
        items_q.append(dict(blob=bd, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=xd, group=group,
                            quantize=True))
        items_i.append(dict(blob=bd, out=out, **{"in": n_in}, bits=bits, codebook=cb, x=q, x_scale=s, group=group))
        qo, so = O.act_quant_int8(x.numpy())
        xt = qo.astype(np.float64) * so.astype(np.float64)[:, None]
        refs.append(O.matmul(O.dequant(blob, out, n_in, bits, cb, group), xt))
    yq = C.cq_gemv_grouped(items_q)
    yi = C.cq_gemv_grouped(items_i)
    torch.cuda.synchronize()
    return yq, yi, refs


def test_decode_step_shapes_quantise_in_the_call(C):
    """The decode kernel's shapes (inputs below 2048 at group 128, batch <=
    4): Q/K/V/gate-like matrices sharing one activation, an O-like matrix
    and a CQ4 head with their own, a ternary matrix; one all-zero token."""
    specs = [(512, 512, 2, 128, 1, 0), (256, 512, 2, 128, 1, 0), (256, 512, 2, 128, 1, 0),
             (512, 512, 2, 128, 1, 0), (512, 512, 2, 128, 1, 1), (1024, 512, 4, 128, 1, 2),
             (300, 640, 5, 128, 3, 3), (77, 1000, 2, 128, 4, 4)]
    yq, yi, refs = _pair(C, specs, 5000)
    for i, (a, b, (y_ref, bound)) in enumerate(zip(yq, yi, refs)):
        assert torch.equal(a, b), f"item {i} {specs[i]}: not the bits of the int8 call"
        check_matmul(a.cpu().numpy(), y_ref, bound, f"item {i} {specs[i]}")


def test_other_routes_quantise_first(C):
    """Shapes the decode kernel does not take quantise into a workspace first:
    wide inputs on the split products, groups of 64, 3-bit codes on the
    streamed kernel, batch 8 on the sliced products, group 64 on a ragged
    input (fp32 kernel); two of them share an activation."""
    specs = [(300, 4096, 2, 128, 2, 0), (200, 4096, 2, 64, 2, 0), (150, 2048, 3, 128, 1, 1),
             (130, 2048, 2, 128, 8, 2), (40, 200, 2, 64, 3, 3)]
    yq, yi, refs = _pair(C, specs, 5200)
    for i, (a, b, (y_ref, bound)) in enumerate(zip(yq, yi, refs)):
        assert torch.equal(a, b), f"item {i} {specs[i]}: not the bits of the int8 call"
        check_matmul(a.cpu().numpy(), y_ref, bound, f"item {i} {specs[i]}")


def test_pinned_host_activations(C):
    """fp32 activations in pinned host memory, read in place by the kernels
    (the decode kernel and the quantiser of the other routes)."""
    specs = [(512, 512, 2, 128, 1, 0), (8192 // 8, 512, 4, 128, 1, 1), (260, 4096, 2, 128, 1, 2)]
    yq, yi, refs = _pair(C, specs, 5400, host_x=True)
    for i, (a, b, (y_ref, bound)) in enumerate(zip(yq, yi, refs)):
        assert torch.equal(a, b), f"item {i} {specs[i]}"
        check_matmul(a.cpu().numpy(), y_ref, bound, f"item {i} {specs[i]}")


def test_single_call_wrapper_and_graph_replay(C):
    """cq_gemv(..., quantize=True), then the same call from a CUDA graph
    with new activation values copied in before each replay."""
    out, n_in = 520, 512
    blob = torch.from_numpy(_blob(out, n_in, 2, 128, 5600)).cuda()
    cb = O.analytic_codebook(2)
    x = S.normal((2, n_in), 5601).cuda()
    y = C.cq_gemv(blob, out, n_in, 2, cb, x, quantize=True)
    q, s = C.cq_act_quant_int8(x)
    assert torch.equal(y, C.cq_gemv(blob, out, n_in, 2, cb, q, s))
    plan = C.GemvPlan([dict(blob=blob, out=out, **{"in": n_in}, bits=2, codebook=cb, x=x, quantize=True)])
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        plan.run(st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        plan.run(st)
    for k in range(3):
        xn = S.normal((2, n_in), 5610 + k).cuda()
        x.copy_(xn)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        q, s = C.cq_act_quant_int8(xn)
        assert torch.equal(plan.ys[0], C.cq_gemv(blob, out, n_in, 2, cb, q, s))


def test_quantize_needs_fp32(C):
    blob = torch.from_numpy(_blob(16, 128, 2, 128, 5700)).cuda()
    q = torch.zeros((1, 128), dtype=torch.int8, device="cuda")
    with pytest.raises(TypeError):
        C.cq_gemv(blob, 16, 128, 2, O.analytic_codebook(2), q, torch.ones(1, device="cuda"), quantize=True)
