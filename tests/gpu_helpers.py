"""Shared helpers of the GPU parity tests (comparison rules only). The
benchmark's oracle leg reuses the same rules for its parity statistics."""
import math

import numpy as np

import oracle as O

# Tolerances for products over CQ weights: |y - y_ref| <= 2e-3 * sum|w||x|
# per element and cosine >= 0.99999 per output vector.
MATMUL_TOL = 2e-3
COS_MIN = 0.99999


def check_matmul(y, y_ref, bound, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    ratio = err / np.maximum(bound, 1e-300)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert np.all(err <= MATMUL_TOL * bound + 1e-30), f"{what}: max |err|/bound = {worst:.3e}"
    for b in range(y.shape[0]):
        ny, nr = np.linalg.norm(y[b]), np.linalg.norm(y_ref[b])
        if nr == 0:
            assert ny == 0, f"{what}: row {b} should be exactly zero"
            continue
        cos = float(np.dot(y[b], y_ref[b]) / (ny * nr))
        assert cos >= COS_MIN, f"{what}: cosine {cos:.8f} in row {b}"
    return worst


def sub_blob(blob, out, n_in, bits, rows, group=128):
    """Blob of a subset of rows (codes of those rows, then their norms)."""
    ip = O.in_padded(n_in, group)
    rb = ip * O.width(bits) // 8
    ng = ip // group
    codes = blob[: out * rb].reshape(out, rb)[rows]
    norms = blob[out * rb:].reshape(out, ng * 2)[rows]
    return np.concatenate([codes.ravel(), norms.ravel()])


def compare_encodings(blob_gpu, blob_ref, flags, out, n_in, bits, group=128):
    """Codes must be equal except at flagged boundary coordinates; norms
    must be bit-exact. Returns (n_boundary, n_boundary_mismatch)."""
    cg, ng_ = O.unpack(blob_gpu, out, n_in, bits, group)
    cr, nr = O.unpack(blob_ref, out, n_in, bits, group)
    assert np.array_equal(ng_, nr), f"{int((ng_ != nr).sum())} fp16 norms differ"
    diff = cg != cr
    bad = diff & (flags == 0)
    assert not bad.any(), f"{int(bad.sum())} codes differ away from decision boundaries"
    return int(flags.sum()), int((diff & (flags != 0)).sum())


def attention_bound(Kh, Vh, q, P, o_ref, n_kv_heads, scale):
    """Per-element tolerance of decode attention over CQ caches, derived
    from the product rule. Each logit is a product over CQ weights (the key
    cache), so it may be off by d_t = scale * 2e-3 * sum_i |k_t,i||q_i|; with
    d = max_t d_t every softmax weight moves by a factor within e^(+-2d), so
    o moves by at most (e^(2d) - 1) * sum_t p_t |v_t - o|. The value sum is a
    product over CQ weights taken in the rotated domain, group by group,
    which bounds its error in a coordinate of group g by
    2e-3 * sum_t p_t ||v_t,g||_2 (the 2-norm of row t's group g)."""
    Hq, dk = q.shape
    per = Hq // n_kv_heads
    dv = Vh.shape[1] // n_kv_heads
    ng = (Vh.shape[1] + 127) // 128
    gnorm = [np.linalg.norm(Vh[:, 128 * g:128 * (g + 1)], axis=1) for g in range(ng)]  # [T] each
    bound = np.zeros_like(o_ref)
    for b in range(Hq):
        h = b // per
        if Kh.shape[0] == 0:
            continue
        kh, vh = Kh[:, h * dk:(h + 1) * dk], Vh[:, h * dv:(h + 1) * dv]
        d = scale * MATMUL_TOL * float((np.abs(kh) @ np.abs(q[b])).max())
        spread = P[b] @ np.abs(vh - o_ref[b])
        gsum = np.array([float(P[b] @ gnorm[g]) for g in range(ng)])
        cols = (h * dv + np.arange(dv)) // 128  # the group of each of the head's columns
        bound[b] = np.expm1(2 * d) * spread + MATMUL_TOL * gsum[cols]
    return bound


def check_attention(o, o_ref, bound, what=""):
    o = np.asarray(o, dtype=np.float64)
    err = np.abs(o - o_ref)
    worst = float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0
    assert np.all(err <= bound + 1e-30), f"{what}: max |err|/bound = {worst:.3e}"
    for b in range(o.shape[0]):
        no, nr = np.linalg.norm(o[b]), np.linalg.norm(o_ref[b])
        if nr == 0:
            assert no == 0, f"{what}: head {b} should be exactly zero"
            continue
        cos = float(np.dot(o[b], o_ref[b]) / (no * nr))
        assert cos >= COS_MIN, f"{what}: cosine {cos:.8f} in head {b}"
    return worst


def gather_bound(blob, out, n_in, bits, cb, rows):
    """Per-element bound of the row gather's fp32 arithmetic: the 128-point
    transform adds seven rounded stages over values bounded by sum|c[q]|,
    then one rounded scaling by n/sqrt(128): |err| <= 1e-6 * n/sqrt(128) *
    sum_k |c[q_k]| per group (a factor ~16 above 8 * 2^-24)."""
    codes, norms = O.unpack(blob, out, n_in, bits)
    lv = np.zeros(16)
    if bits == 5:
        c = float(cb[2])
        lv[1], lv[2], lv[3] = c, -2.0 * c, -c
    else:
        lv[:len(cb)] = np.asarray(cb, dtype=np.float64)
    n = O.f16_bits_to_f32(norms).astype(np.float64).reshape(norms.shape)
    ng = codes.shape[1] // 128
    s = np.abs(lv[codes]).reshape(out, ng, 128).sum(axis=2) * n / math.sqrt(128)  # [out][ng]
    b = np.repeat(s, 128, axis=1)[:, :n_in]
    return 1e-6 * b[rows] + 1e-30
