"""Shared helpers of the GPU parity tests (comparison rules only)."""
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


def sub_blob(blob, out, n_in, bits, rows):
    """Blob of a subset of rows (codes of those rows, then their norms)."""
    ip = O.in_padded(n_in)
    rb = ip * O.width(bits) // 8
    ng = ip // 128
    codes = blob[: out * rb].reshape(out, rb)[rows]
    norms = blob[out * rb:].reshape(out, ng * 2)[rows]
    return np.concatenate([codes.ravel(), norms.ravel()])


def compare_encodings(blob_gpu, blob_ref, flags, out, n_in, bits):
    """Codes must be equal except at flagged boundary coordinates; norms
    must be bit-exact. Returns (n_boundary, n_boundary_mismatch)."""
    cg, ng_ = O.unpack(blob_gpu, out, n_in, bits)
    cr, nr = O.unpack(blob_ref, out, n_in, bits)
    assert np.array_equal(ng_, nr), f"{int((ng_ != nr).sum())} fp16 norms differ"
    diff = cg != cr
    bad = diff & (flags == 0)
    assert not bad.any(), f"{int(bad.sum())} codes differ away from decision boundaries"
    return int(flags.sum()), int((diff & (flags != 0)).sum())
