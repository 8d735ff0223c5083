"""Pins for the oracle: each test checks the oracle against something other
than itself -- values printed on the pages, closed forms, textbook special
cases, library routines, invariants -- so that a plausible mistake anywhere
in it (a dropped term, a wrong sign or index, a transposed operand) fails.

Page citations use the page title and section:
  [CF] "The .cact format" (cactuscompute.com blog)
  [NJ] "The .cact archive and Cactus Quants" (needle.js tutorial)
  [ON] OpenNeedle docs/reference.md
"""
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden_floats(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return np.array(vals)


def _read_golden_kv(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                kv[k] = float(v)
    return kv


# ------------------------------------------------------------------ Hadamard

@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_hadamard_integer_orthogonality(n):
    """[CF] "Cactus Quants": H is symmetric and orthogonal. In integers the
    unnormalised matrix satisfies H0 H0^T = n I exactly."""
    H = O.hadamard(n)
    H0 = np.rint(H * math.sqrt(n)).astype(np.int64)
    assert np.all(np.abs(H0) == 1)
    assert np.array_equal(H0 @ H0.T, n * np.eye(n, dtype=np.int64))
    assert np.array_equal(H0, H0.T)
    assert np.allclose(H @ H, np.eye(n), atol=1e-14)


def test_hadamard_is_sylvester_natural_order():
    """[ON] names the Sylvester/Walsh-Hadamard matrix; scipy builds the
    Sylvester construction in natural order."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    for n in (8, 128):
        H0 = np.rint(O.hadamard(n) * math.sqrt(n)).astype(np.int64)
        assert np.array_equal(H0, scipy_linalg.hadamard(n))


# ----------------------------------------------------------------- codebooks

def test_lloyd_max_two_levels_closed_form():
    """Two-level Lloyd-Max for N(0,1) is +-E|X| = +-sqrt(2/pi)."""
    c, _ = O.lloyd_max_normal(2)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-13
    assert abs(c[0] + math.sqrt(2 / math.pi)) < 1e-13


def test_lloyd_max_three_levels_is_the_ternary_constant():
    """[NJ] "Shared codebooks" prints the ternary levels {-1.2240064, 0,
    +1.2240064}/sqrt(group); [CF] says they are analytic. The 3-level
    Lloyd-Max fixed point reproduces the printed constant to its digits."""
    c, _ = O.lloyd_max_normal(3)
    assert abs(c[1]) < 1e-15
    assert abs(c[2] - 1.2240064) < 5e-8 and abs(c[0] + 1.2240064) < 5e-8


def test_lloyd_max_four_levels_matches_stated_values():
    """CQ2 analytic levels quoted to four places for the CQ2 codebook:
    +-0.4528 and +-1.5104 before the 1/sqrt(128) scale."""
    c, _ = O.lloyd_max_normal(4)
    assert np.allclose(c, [-1.5104, -0.4528, 0.4528, 1.5104], atol=5e-5)


@pytest.mark.parametrize("L", [4, 8])
def test_lloyd_max_minimises_distortion(L):
    """The fixed point must be the minimiser of the mean squared error
    integral, found here by a generic optimiser with numerical quadrature
    (no centroid formula involved)."""
    integrate = pytest.importorskip("scipy.integrate")
    optimize = pytest.importorskip("scipy.optimize")

    def mse(half):
        pos = np.sort(np.abs(half))
        c = np.concatenate([-pos[::-1], pos])
        t = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
        tot = 0.0
        for j in range(L):
            tot += integrate.quad(
                lambda x, cj=c[j]: (x - cj) ** 2 * math.exp(-x * x / 2) / math.sqrt(2 * math.pi),
                t[j], t[j + 1], epsabs=1e-13, epsrel=1e-13)[0]
        return tot

    x0 = np.linspace(0.2, 2.0, L // 2)
    res = optimize.minimize(mse, x0, method="Nelder-Mead",
                            options={"xatol": 1e-10, "fatol": 1e-15, "maxiter": 20000})
    opt = np.sort(np.abs(res.x))
    c, _ = O.lloyd_max_normal(L)
    assert np.allclose(c[L // 2:], opt, atol=2e-5)
    # and its distortion is no larger than the optimiser's
    assert mse(c[L // 2:]) <= res.fun + 1e-12


def test_empirical_codebook_reproduces_printed_header():
    """[ON] CQ section: RandomState(0).randn(400000), quantile start, 200
    Lloyd-Max iterations, divide by sqrt(128), fp32 -- reproduces the CQ2
    header codebook it prints, exactly in fp32."""
    printed = _read_golden_floats("cq2_header_codebook.txt").astype(np.float32)
    x = np.random.RandomState(0).randn(400000)
    c = O.lloyd_max_samples(x, 4, 200)
    got = (c / np.sqrt(128)).astype(np.float32)
    assert np.array_equal(got, printed)
    # the printed codebook is not symmetric (the page says so)
    assert printed[0] != -printed[3]


# ---------------------------------------------------------------------- fp16

def test_fp16_conversion_matches_numpy():
    rng = np.random.RandomState(7)
    vals = np.concatenate([
        rng.randn(20000).astype(np.float32),
        (rng.randn(5000) * 1e-5).astype(np.float32),     # fp16 subnormals
        (rng.randn(5000) * 3e4).astype(np.float32),      # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 1e-8, 2.0 ** -24,
                  2.0 ** -25, 3 * 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11,
                  2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, np.inf, -np.inf],
                 dtype=np.float32),
    ])
    got = O.f32_to_f16_bits(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    back = O.f16_bits_to_f32(ref)
    assert np.array_equal(back, ref.view(np.float16).astype(np.float32))


# ------------------------------------------------------------ byte accounting

def test_blob_size_formula_reproduces_needle2_size_table():
    """[NJ] "Anatomy of a CQ matrix" gives the blob length; [ON] prints the
    Needle-2 totals. The shapes follow from [ON]'s geometry table."""
    ref = _read_golden_kv("needle2_cq_sizes.txt")
    layer_cq2 = [(512, 512), (256, 512), (256, 512), (512, 512), (512, 512)]  # Q K V gate O
    engram_cq2 = [(4 * 8192, 128), (512, 512), (512, 512)]  # tables, key, value
    cq2 = layer_cq2 * 27 + engram_cq2 * 2
    cq4 = [(8192, 512), (27 * 4, 2048), (27 * 4, 2048), (27 * 16, 2048)]  # embedding, phi pre/post/res
    assert len(cq2) == ref["cq2_tensors"] and len(cq4) == ref["cq4_tensors"]
    el2 = sum(o * i for o, i in cq2)
    el4 = sum(o * i for o, i in cq4)
    assert el2 == ref["cq2_elements"] and el4 == ref["cq4_elements"]
    b2 = sum(O.packed_bytes(o, i, 128, 2) for o, i in cq2)
    b4 = sum(O.packed_bytes(o, i, 128, 4) for o, i in cq4)
    norms = sum(o * (i // 128) * 2 for o, i in cq2 + cq4)
    assert b2 == ref["cq2_bytes"] and b4 == ref["cq4_bytes"]
    assert norms == ref["fp16_norm_bytes"]
    assert round((2 * el2 + 4 * el4) / (el2 + el4), 6) == ref["cq_weighted_code_bits"]


def test_bits_per_weight():
    """[CF] "Cactus Quants": bits + 16/group -> 2.125 (CQ2), 4.125 (CQ4)."""
    for bits, bpw in ((2, 2.125), (4, 4.125), (3, 3.125), (5, 2.125)):
        assert O.packed_bytes(1024, 4096, 128, bits) * 8 / (1024 * 4096) == bpw


def test_padding_to_group():
    """[NJ]: the input axis is zero-padded to a multiple of the group."""
    assert O.packed_bytes(3, 129, 128, 2) == 3 * 256 * 2 // 8 + 3 * 2 * 2
    assert O.packed_bytes(0, 512, 128, 2) == 0
    assert O.packed_bytes(5, 512, 100, 2) == 0  # group must be a power of two


# ------------------------------------------------------------------- packing

def _blob_with_row(row_bytes: bytes, out=1, n_in=128, bits=2):
    blob = np.zeros(O.packed_bytes(out, n_in, 128, bits), dtype=np.uint8)
    blob[: len(row_bytes)] = np.frombuffer(row_bytes, dtype=np.uint8)
    return blob


def test_unpack_two_bit_lsb_first():
    """[NJ] "2-bit": four indices per byte, first column in the lowest bits."""
    blob = _blob_with_row(bytes([0b11100100, 0b00011011]))
    codes, _ = O.unpack(blob, 1, 128, 2)
    assert list(codes[0, :8]) == [0, 1, 2, 3, 3, 2, 1, 0]


def test_unpack_four_bit_low_nibble_first():
    """[NJ] "4-bit": two indices per byte, low nibble first."""
    blob = _blob_with_row(bytes([0x21, 0xF0]), bits=4)
    codes, _ = O.unpack(blob, 1, 128, 4)
    assert list(codes[0, :4]) == [1, 2, 0, 15]


def test_unpack_three_bit_crosses_bytes():
    """[NJ] "3-bit" (16-bit window) and [ON] (8 codes -> one word -> 3
    little-endian bytes): codes 0..7 pack to 0xFAC688."""
    blob = _blob_with_row(bytes([0x88, 0xC6, 0xFA]), bits=3)
    codes, _ = O.unpack(blob, 1, 128, 3)
    assert list(codes[0, :8]) == list(range(8))


def test_norms_follow_codes_region():
    """[NJ] "Anatomy of a CQ matrix": all rows' packed indices, then all
    fp16 norms [out][in_pad/group]."""
    out, n_in = 2, 256
    blob = np.zeros(O.packed_bytes(out, n_in, 128, 2), dtype=np.uint8)
    base = out * 256 * 2 // 8
    h = np.array([0x3C00, 0x4000, 0x4200, 0x4400], dtype="<u2")  # 1, 2, 3, 4
    blob[base:] = h.view(np.uint8)
    _, norms = O.unpack(blob, out, n_in, 2)
    assert norms.tolist() == [[0x3C00, 0x4000], [0x4200, 0x4400]]


# ------------------------------------------------------------------- encoder

def _cq2():
    return O.analytic_codebook(2)


def test_encode_unit_vector_all_outer_codes():
    """w = a*e_0: r = a*(row 0 of H) = a/sqrt(128) everywhere, so u_k =
    1/sqrt(128) = 0.0884, which is closer to the outer level 0.1335 than to
    0.0400: every code is 3, and the norm is exactly a."""
    W = np.zeros((1, 128), dtype=np.float32)
    W[0, 0] = 0.75
    blob, flags, nflag = O.encode(W, 2, _cq2())
    codes, norms = O.unpack(blob, 1, 128, 2)
    assert np.all(codes == 3) and nflag == 0
    assert norms[0, 0] == np.float16(0.75).view(np.uint16)


@pytest.mark.parametrize("i", [1, 5, 77, 127])
def test_encode_basis_vector_follows_hadamard_row(i):
    """w = e_i: r_k = H[i][k] = (-1)^popcount(i&k)/sqrt(128): code 3 where
    the sign is +, code 0 where it is -. Catches a transposed or re-ordered
    Hadamard matrix."""
    W = np.zeros((1, 128), dtype=np.float32)
    W[0, i] = 1.0
    blob, _, _ = O.encode(W, 2, _cq2())
    codes, _ = O.unpack(blob, 1, 128, 2)
    sign = np.array([(-1) ** bin(i & k).count("1") for k in range(128)])
    assert np.array_equal(codes[0], np.where(sign > 0, 3, 0))


@pytest.mark.parametrize("cb_kind", ["analytic", "empirical"])
def test_encode_ties_go_to_smaller_index(cb_kind):
    """[ON]: equal distances pick the smaller index. w = 1 (all ones) gives
    u = e_0: code 3 at k=0; u_k = 0 elsewhere, which with the symmetric
    codebook ties levels 1 and 2 (-> 1) and with the printed empirical one is
    nearer level 1. Exact zeros sit on the middle decision boundary of the
    symmetric codebook, so they are flagged."""
    cb = _cq2() if cb_kind == "analytic" else _read_golden_floats(
        "cq2_header_codebook.txt").astype(np.float32)
    W = np.ones((1, 128), dtype=np.float32)
    blob, flags, nflag = O.encode(W, 2, cb)
    codes, norms = O.unpack(blob, 1, 128, 2)
    assert codes[0, 0] == 3 and np.all(codes[0, 1:] == 1)
    assert norms[0, 0] == np.float16(math.sqrt(128)).view(np.uint16)
    if cb_kind == "analytic":
        assert nflag == 127 and flags[0, 0] == 0


def test_encode_zero_group():
    """A zero group: n = 0, u = 0, every coordinate ties to the lower middle
    level; the stored norm is zero so the group reconstructs to zero."""
    W = np.zeros((2, 256), dtype=np.float32)
    W[1, 200] = 2.0  # second group of row 1 is non-zero
    blob, _, _ = O.encode(W, 2, _cq2())
    codes, norms = O.unpack(blob, 2, 256, 2)
    assert np.all(codes[0] == 1) and np.all(norms[0] == 0)
    assert np.all(codes[1, :128] == 1) and norms[1, 0] == 0
    What = O.dequant(blob, 2, 256, 2, _cq2())
    assert np.all(What[0] == 0) and np.all(What[1, :128] == 0)


def test_encode_ternary_crumbs():
    """[NJ] "Shared codebooks": bits=5 is the ternary marker; [ON]: signed
    2-bit crumbs. e_0 -> u = +1/sqrt(128) = 0.0884 > c/2 = 0.0541 -> +c ->
    crumb 01; -e_0 -> -c -> crumb 11; 0.2*e_0 + rest gives zeros."""
    cb = O.analytic_codebook(5)
    W = np.zeros((2, 128), dtype=np.float32)
    W[0, 0] = 1.0
    W[1, 0] = -1.0
    blob, _, _ = O.encode(W, 5, cb)
    codes, _ = O.unpack(blob, 2, 128, 5)
    assert np.all(codes[0] == 1) and np.all(codes[1] == 3)
    What = O.dequant(blob, 2, 128, 5, cb)
    c = float(cb[2])
    # all-equal levels +c reconstruct to n*c*sqrt(128)*e_0
    assert abs(What[0, 0] - c * math.sqrt(128)) < 1e-12
    assert np.allclose(What[0, 1:], 0, atol=1e-15)
    assert abs(What[1, 0] + c * math.sqrt(128)) < 1e-12


def test_encode_scale_by_power_of_two():
    """Scaling W by 2^k scales r and n exactly and leaves u, hence the codes,
    unchanged; the fp16 norms scale exactly while they stay normal."""
    rng = np.random.RandomState(3)
    W = (rng.randn(4, 384) * 0.02).astype(np.float32)
    b1, _, _ = O.encode(W, 3, O.analytic_codebook(3))
    b2, _, _ = O.encode(W * 8, 3, O.analytic_codebook(3))
    c1, n1 = O.unpack(b1, 4, 384, 3)
    c2, n2 = O.unpack(b2, 4, 384, 3)
    assert np.array_equal(c1, c2)
    assert np.array_equal(O.f16_bits_to_f32(n1) * 8, O.f16_bits_to_f32(n2))


def test_encode_sign_flip_mirrors_codes():
    """With a symmetric codebook, -W maps code q to L-1-q (no exact ties in
    random data), and keeps the norm."""
    rng = np.random.RandomState(4)
    W = (rng.randn(3, 256) * 0.02).astype(np.float32)
    cb = O.analytic_codebook(4)
    assert np.array_equal(cb, -cb[::-1])
    b1, _, _ = O.encode(W, 4, cb)
    b2, _, _ = O.encode(-W, 4, cb)
    c1, n1 = O.unpack(b1, 3, 256, 4)
    c2, n2 = O.unpack(b2, 3, 256, 4)
    assert np.array_equal(c1, 15 - c2) and np.array_equal(n1, n2)


@pytest.mark.parametrize("bits,dist", [(2, 0.1175), (3, 0.03454), (4, 0.009497)])
def test_reconstruction_error_matches_lloyd_max_distortion(bits, dist):
    """For Gaussian groups the rotated direction is close to Gaussian, so the
    relative squared reconstruction error approaches the textbook Lloyd-Max
    distortion for unit variance (Max 1960): 0.1175, 0.03454, 0.009497.
    A transposed H, a wrong norm or a wrong level would miss by far."""
    rng = np.random.RandomState(5)
    W = (rng.randn(64, 512) * 0.02).astype(np.float32)
    blob, _, _ = O.encode(W, bits, O.analytic_codebook(bits))
    What = O.dequant(blob, 64, 512, bits, O.analytic_codebook(bits))
    rel = np.sum((What - W) ** 2) / np.sum(W.astype(np.float64) ** 2)
    assert abs(rel - dist) < 0.12 * dist


def test_dequant_closed_form_single_code_pattern():
    """[NJ] "Reconstructing one group": all codes j with norm n give
    w_hat = n*c_j*(1,...,1).H = n*c_j*sqrt(128)*e_0."""
    cb = _cq2()
    blob = np.zeros(O.packed_bytes(1, 128, 128, 2), dtype=np.uint8)
    blob[:32] = 0b10101010  # every code = 2
    blob[32:34] = np.array([0x4000], dtype="<u2").view(np.uint8)  # n = 2.0
    What = O.dequant(blob, 1, 128, 2, cb)
    assert abs(What[0, 0] - 2.0 * float(cb[2]) * math.sqrt(128)) < 1e-12
    assert np.allclose(What[0, 1:], 0.0, atol=1e-14)


def test_padding_columns_are_zero_and_cropped():
    rng = np.random.RandomState(6)
    W = (rng.randn(3, 200) * 0.02).astype(np.float32)
    Wpad = np.zeros((3, 256), dtype=np.float32)
    Wpad[:, :200] = W
    b1, _, _ = O.encode(W, 2, _cq2())
    b2, _, _ = O.encode(Wpad, 2, _cq2())
    assert np.array_equal(b1, b2)
    D1 = O.dequant(b1, 3, 200, 2, _cq2())
    D2 = O.dequant(b2, 3, 256, 2, _cq2())
    assert np.array_equal(D1, D2[:, :200])


def test_encode_rejects_unsorted_codebook():
    with pytest.raises(ValueError):
        O.encode(np.zeros((1, 128), np.float32), 2,
                 np.array([0.1, -0.1, 0.2, 0.3], dtype=np.float32))


# ------------------------------------------------------------------- product

@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_rotated_identity_matches_dense_product(bits):
    """[ON] and [NJ] "Reconstructing one group": <w_hat_g, x_g> =
    n * <c[q], H x_g>. The dense route (dequantise, then multiply) and the
    rotated route must agree to rounding."""
    rng = np.random.RandomState(10 + bits)
    W = (rng.randn(9, 300) * 0.02).astype(np.float32)
    X = rng.randn(3, 300)
    cb = O.analytic_codebook(bits)
    blob, _, _ = O.encode(W, bits, cb)
    What = O.dequant(blob, 9, 300, bits, cb)
    Y1, Bd = O.matmul(What, X)
    Y2 = O.matmul_rotated(blob, 9, 300, bits, cb, X)
    assert np.max(np.abs(Y1 - Y2) / Bd) < 1e-12


def test_matmul_matches_numpy():
    rng = np.random.RandomState(11)
    A = rng.randn(7, 33)
    X = rng.randn(4, 33)
    Y, Bd = O.matmul(A, X)
    assert np.allclose(Y, X @ A.T, rtol=1e-13, atol=1e-13)
    assert np.allclose(Bd, np.abs(X) @ np.abs(A).T, rtol=1e-13)


# ---------------------------------------------------------- activation quant

def test_act_quant_worked_examples():
    """[ON] fake_quant_act: s = absmax/127, round (half to even), clamp.
    x = [127, 0.5, 1.5, 2.5, -126.5] -> s = 1 -> q = [127, 0, 2, 2, -126]."""
    Q, S = O.act_quant_int8(np.array([[127.0, 0.5, 1.5, 2.5, -126.5]], np.float32))
    assert S[0] == 1.0 and Q[0].tolist() == [127, 0, 2, 2, -126]
    Q, S = O.act_quant_int8(np.zeros((1, 5), np.float32))
    assert S[0] == 1.0 and np.all(Q == 0)


def test_act_quant_error_bound():
    rng = np.random.RandomState(12)
    X = rng.randn(8, 512).astype(np.float32)
    Q, S = O.act_quant_int8(X)
    amax = np.abs(X).max(axis=1)
    assert np.allclose(S, amax / 127, rtol=1e-7)
    assert np.all(np.abs(Q).max(axis=1) == 127)
    err = np.abs(Q * S[:, None].astype(np.float64) - X)
    assert np.all(err <= 0.5 * S[:, None] * (1 + 1e-6))


def test_gather_rows_selects_in_order_with_repeats():
    """Row gather ("Reconstructing one group" applied to indexed rows only):
    row r of a 3-row table has every code equal to r and norm 2^r, so its
    dequantised group is 2^r * c_r * sqrt(128) * e_0; gathering [2, 0, 2, 1]
    must return those rows in that order."""
    cb = _cq2()
    out = 3
    blob = np.zeros(O.packed_bytes(out, 128, 128, 2), dtype=np.uint8)
    for r, byte in enumerate((0b00000000, 0b01010101, 0b10101010)):
        blob[32 * r: 32 * (r + 1)] = byte
    norms = np.array([0x3C00, 0x4000, 0x4400], dtype="<u2")  # 1, 2, 4
    blob[96:102] = norms.view(np.uint8)
    got = O.gather_rows(blob, out, 128, 2, cb, [2, 0, 2, 1])
    for i, r in enumerate([2, 0, 2, 1]):
        assert abs(got[i, 0] - (2.0 ** r) * float(cb[r]) * math.sqrt(128)) < 1e-12
        assert np.allclose(got[i, 1:], 0.0, atol=1e-14)


# ------------------------------------------------------------ KV cache --
# Attention pins: closed forms of the softmax-weighted sum that a dropped
# scale, a wrong head mapping, a transposed operand or an unstable softmax
# would break.

def test_attend_single_token_returns_its_value_slice():
    """One token: the softmax weight is 1 whatever the logit, so each head
    returns its key/value head's slice of the value row."""
    rng = np.random.RandomState(1)
    K, V, q = rng.randn(1, 2 * 3), rng.randn(1, 2 * 5), rng.randn(4, 3)
    o, P = O.attend(K, V, q, 2, 0.7)
    assert np.array_equal(P, np.ones((4, 1)))
    for b in range(4):
        h = b // 2
        assert np.array_equal(o[b], V[0, 5 * h:5 * h + 5])


def test_attend_zero_query_averages_values():
    """q = 0 (or scale 0): every logit is 0, the weights are uniform and the
    output is the mean of the value rows."""
    rng = np.random.RandomState(2)
    K, V = rng.randn(7, 8), rng.randn(7, 8)
    o, P = O.attend(K, V, np.zeros((2, 8)), 1, 0.35)
    assert np.allclose(P, 1.0 / 7.0, rtol=0, atol=1e-15)
    assert np.allclose(o, np.tile(V.mean(axis=0), (2, 1)), rtol=0, atol=1e-14)
    o2, _ = O.attend(K, V, rng.randn(2, 8), 1, 0.0)
    assert np.allclose(o2, o, rtol=0, atol=1e-14)


def test_attend_two_tokens_logistic_closed_form():
    """Two tokens with logits a and b: the weight of the second is the
    logistic function of scale * (b - a)."""
    K = np.array([[1.0, 0.0], [0.0, 1.0]])
    V = np.array([[2.0, -1.0], [5.0, 3.0]])
    q = np.array([[0.25, 1.75]])
    scale = 0.8
    w1 = 1.0 / (1.0 + math.exp(-scale * (1.75 - 0.25)))
    o, P = O.attend(K, V, q, 1, scale)
    assert abs(P[0, 1] - w1) < 1e-15 and abs(P[0, 0] - (1 - w1)) < 1e-15
    assert np.allclose(o[0], (1 - w1) * V[0] + w1 * V[1], rtol=0, atol=1e-14)


def test_attend_grouped_query_heads_use_their_kv_head():
    """Four query heads over two key/value heads: heads 0, 1 read key head 0
    (columns 0..1) and heads 2, 3 read key head 1 (columns 2..3). Token 0's
    key points along q in head 0 only, token 1's in head 1 only, so each
    query head picks one token's value slice of its own head."""
    K = np.array([[40.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 40.0, 0.0]])
    V = np.array([[1.0, 2.0, 3.0, 4.0],
                  [5.0, 6.0, 7.0, 8.0]])
    q = np.tile(np.array([[1.0, 0.0]]), (4, 1))
    o, _ = O.attend(K, V, q, 2, 1.0)
    e = math.exp(-40.0)
    for b in (0, 1):  # token 0 dominates, value head 0 = columns 0..1
        assert np.allclose(o[b], ([1.0, 2.0] + e * np.array([5.0, 6.0])) / (1 + e), rtol=0, atol=1e-15)
    for b in (2, 3):  # token 1 dominates, value head 1 = columns 2..3
        assert np.allclose(o[b], ([7.0, 8.0] + e * np.array([3.0, 4.0])) / (1 + e), rtol=0, atol=1e-15)


def test_attend_large_logits_do_not_overflow():
    """Logits of order 1e4 would overflow exp without the max shift; the
    result is the value row of the largest logit."""
    K = np.array([[1.0], [2.0], [1.5]]) * 1e4
    V = np.array([[1.0, 0.0], [0.0, 1.0], [9.0, 9.0]])
    o, P = O.attend(K, V, np.array([[1.0]]), 1, 1.0)
    assert np.all(np.isfinite(o)) and np.array_equal(o[0], [0.0, 1.0])


def test_attend_no_tokens_gives_zero():
    o, P = O.attend(np.zeros((0, 4)), np.zeros((0, 6)), np.ones((2, 4)), 1, 1.0)
    assert o.shape == (2, 6) and not o.any() and P.shape == (2, 0)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_kv_write_in_pieces_equals_one_encode(bits):
    """Writing the rows of a cache in three pieces, out of order, gives the
    blob that encoding the whole matrix at once gives ([CF] "How the kernel
    reads it": the KV cache uses the weight path); rows never written stay
    as they were."""
    rng = np.random.RandomState(3 + bits)
    n_in, T = 96, 11
    rows = (rng.randn(T, n_in) * 0.5).astype(np.float32)
    cb = O.analytic_codebook(bits)
    whole, _, _ = O.encode(rows, bits, cb)
    cache = np.zeros(O.packed_bytes(T, n_in, 128, bits), dtype=np.uint8)
    for a, b in ((4, 9), (0, 4), (9, 11)):
        O.kv_write(cache, T, n_in, bits, cb, rows[a:b], a)
    assert np.array_equal(cache, whole)
    big = np.full(O.packed_bytes(T + 5, n_in, 128, bits), 0xA5, dtype=np.uint8)
    O.kv_write(big, T + 5, n_in, bits, cb, rows, 0)
    assert np.array_equal(O.kv_rows_blob(big, T + 5, n_in, bits, T), whole)
    rb = O.in_padded(n_in) * O.width(bits) // 8
    assert np.all(big[T * rb:(T + 5) * rb] == 0xA5)  # rows past T untouched


def test_kv_attend_ignores_rows_past_n_tokens_and_single_row_is_exact():
    """Rows past n_tokens may hold anything (0xFF: NaN norms); with one row
    the output is that row's dequantised value slice, n * H c[q] per group
    ([NJ] "Reconstructing one group")."""
    rng = np.random.RandomState(4)
    Hkv, dk, dv, cap = 2, 48, 64, 9
    cb = O.analytic_codebook(2)
    kc = np.full(O.packed_bytes(cap, Hkv * dk, 128, 2), 0xFF, dtype=np.uint8)
    vc = np.full(O.packed_bytes(cap, Hkv * dv, 128, 2), 0xFF, dtype=np.uint8)
    O.kv_write(kc, cap, Hkv * dk, 2, cb, rng.randn(5, Hkv * dk), 0)
    O.kv_write(vc, cap, Hkv * dv, 2, cb, rng.randn(5, Hkv * dv), 0)
    q = rng.randn(4, dk)
    o, P, Kh, Vh = O.kv_attend(kc, vc, cap, 5, q, Hkv, dk, dv, 2, 2, cb, cb, 0.2)
    assert np.all(np.isfinite(o)) and Kh.shape == (5, Hkv * dk)
    o1, _, _, Vh1 = O.kv_attend(kc, vc, cap, 1, q, Hkv, dk, dv, 2, 2, cb, cb, 0.2)
    codes, norms = O.unpack(O.kv_rows_blob(vc, cap, Hkv * dv, 2, 1), 1, Hkv * dv, 2)
    n = O.f16_bits_to_f32(norms)[0]
    row = n * O.hadamard(128) @ cb[codes[0]].astype(np.float64)  # normalised H
    for b in range(4):
        h = b // 2
        assert np.allclose(o1[b], row[h * dv:(h + 1) * dv], rtol=0, atol=1e-12)


# ------------------------------------------------ binary codes and group 64
# [CF] "Cactus Quants": binary weights pack eight per byte and have
# closed-form centroids; OpenNeedle docs/reference.md tests group 64 and 128.

def test_binary_centroids_closed_form():
    """The two-level Lloyd-Max quantiser of N(0,1) has centroids
    +-E|X| = +-sqrt(2/pi) (the conditional mean of a half-normal)."""
    c, _ = O.lloyd_max_normal(2)
    assert np.allclose(c, [-math.sqrt(2 / math.pi), math.sqrt(2 / math.pi)], rtol=0, atol=1e-12)
    for g in (64, 128):
        cb = O.analytic_codebook(1, g)
        assert np.allclose(cb, np.float32(np.array([-1, 1]) * math.sqrt(2 / math.pi) / math.sqrt(g)), rtol=0, atol=0)


def _brute_encode(W, group, cb):
    """Brute force with scipy's Hadamard matrix: codes of the nearest level to
    u = H w / |w| per group (ties to the smaller index), and fp32 norms."""
    from scipy.linalg import hadamard as sh
    H = sh(group).astype(np.float64) / math.sqrt(group)
    out, n_in = W.shape
    ip = O.in_padded(n_in, group)
    Wp = np.zeros((out, ip)); Wp[:, :n_in] = W
    codes = np.zeros((out, ip), dtype=np.int64); norms = np.zeros((out, ip // group))
    for o in range(out):
        for g in range(ip // group):
            w = Wp[o, g * group:(g + 1) * group]
            n = np.float32(np.sqrt(np.sum(w * w)))
            u = (H @ w) / max(float(n), 1e-12)
            d = np.abs(u[:, None] - cb.astype(np.float64)[None, :])
            codes[o, g * group:(g + 1) * group] = np.argmin(d, axis=1)
            norms[o, g] = n
    return codes, norms


@pytest.mark.parametrize("bits,group", [(1, 128), (1, 64), (2, 64), (3, 64), (4, 64)])
def test_encode_matches_brute_force(bits, group):
    """Codes and norms for binary codes and 64-wide groups against a direct
    computation with an independently built Hadamard matrix."""
    rng = np.random.RandomState(40 + bits + group)
    W = (rng.randn(3, 200) * 0.02).astype(np.float32)
    cb = O.analytic_codebook(bits, group)
    blob, flags, _ = O.encode(W, bits, cb, group)
    codes, norms = O.unpack(blob, 3, 200, bits, group)
    bc, bn = _brute_encode(W, group, cb)
    assert np.array_equal(codes[flags == 0], bc[flags == 0])
    assert np.array_equal(O.f16_bits_to_f32(norms).reshape(bn.shape), bn.astype(np.float16).astype(np.float32))


def test_binary_packing_eight_codes_per_byte():
    """One continuous LSB-first stream per row ([CF] "Cactus Quants"):
    binary code k of a row is bit k % 8 of byte k // 8; a row of 256 codes
    takes 32 bytes, then the fp16 norms follow."""
    rng = np.random.RandomState(44)
    W = (rng.randn(2, 256) * 0.02).astype(np.float32)
    cb = O.analytic_codebook(1)
    blob, _, _ = O.encode(W, 1, cb)
    assert blob.size == O.packed_bytes(2, 256, 128, 1) == 2 * 32 + 2 * 2 * 2
    codes, _ = O.unpack(blob, 2, 256, 1)
    assert np.array_equal(blob[:64], np.packbits(codes.astype(np.uint8).reshape(-1), bitorder="little"))


@pytest.mark.parametrize("group", [64, 128])
def test_binary_dequant_closed_form(group):
    """All codes 1 with norm n give n * c * (1,...,1) H = n * c * sqrt(group) * e_0
    in every group ([NJ] "Reconstructing one group")."""
    cb = O.analytic_codebook(1, group)
    nb = O.packed_bytes(1, 2 * group, group, 1)
    blob = np.zeros(nb, dtype=np.uint8)
    blob[:2 * group // 8] = 0xFF
    blob[2 * group // 8:] = np.array([0x4000, 0x3C00], dtype="<u2").view(np.uint8)  # n = 2, 1
    What = O.dequant(blob, 1, 2 * group, 1, cb, group)
    for g, n in ((0, 2.0), (1, 1.0)):
        seg = What[0, g * group:(g + 1) * group]
        assert abs(seg[0] - n * float(cb[1]) * math.sqrt(group)) < 1e-12
        assert np.allclose(seg[1:], 0.0, atol=1e-14)


def test_binary_reconstruction_error_matches_distortion():
    """The 1-bit Lloyd-Max quantiser of N(0,1) has distortion 1 - 2/pi; the
    relative squared reconstruction error of Gaussian groups approaches it
    (at group 64 and 128)."""
    rng = np.random.RandomState(45)
    W = (rng.randn(64, 512) * 0.02).astype(np.float32)
    for group in (64, 128):
        cb = O.analytic_codebook(1, group)
        blob, _, _ = O.encode(W, 1, cb, group)
        What = O.dequant(blob, 64, 512, 1, cb, group)
        rel = np.sum((What - W) ** 2) / np.sum(W.astype(np.float64) ** 2)
        assert abs(rel - (1 - 2 / math.pi)) < 0.06 * (1 - 2 / math.pi)


@pytest.mark.parametrize("bits,group", [(1, 128), (1, 64), (2, 64), (4, 64), (5, 64)])
def test_rotated_identity_other_geometries(bits, group):
    """The rotated route n <c[q], H x_g> equals the dense product for binary
    codes and 64-wide groups."""
    rng = np.random.RandomState(46 + bits + group)
    W = (rng.randn(5, 200) * 0.02).astype(np.float32)
    X = rng.randn(2, 200)
    cb = O.analytic_codebook(bits, group)
    blob, _, _ = O.encode(W, bits, cb, group)
    Y1, Bd = O.matmul(O.dequant(blob, 5, 200, bits, cb, group), X)
    Y2 = O.matmul_rotated(blob, 5, 200, bits, cb, X, group)
    assert np.max(np.abs(Y1 - Y2) / Bd) < 1e-12
