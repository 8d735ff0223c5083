"""GPU parity of the CQ KV cache (cq_kv_write, cq_kv_attend) against the
oracle: cache rows encoded by the oracle's encoder, attention by definition
over the oracle's dequantised rows in fp64. Caches are seeded random blobs or
oracle encodings; no oracle input comes from the CUDA path."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests.gpu_helpers import attention_bound, check_attention, compare_encodings

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _width(Hkv, d):
    return Hkv * d


def _filled_cache(cap, width, bits, n, seed, fill=0xFF):
    """Random rows 0..n-1; rows n..cap-1 hold `fill` bytes (0xFF: NaN norms)."""
    blob = S.kv_cache_blob(cap, width, bits, seed)
    ip = O.in_padded(width)
    rb, ng = ip * O.width(bits) // 8, ip // 128
    blob[n * rb:cap * rb] = fill
    blob[cap * rb + 2 * ng * n:] = fill
    return blob


def _run_and_check(C, geom, kb, vb, seqs_np, scale, what):
    Hq, Hkv, dk, dv = geom
    cbk, cbv = O.analytic_codebook(kb), O.analytic_codebook(vb)
    items = []
    for (kc, vc, cap, n, q) in seqs_np:
        items.append(dict(k_cache=torch.from_numpy(kc).cuda(), v_cache=torch.from_numpy(vc).cuda(),
                          cap=cap, n_tokens=n, q=torch.from_numpy(q).float().cuda()))
    outs = C.cq_kv_attend(items, Hq, Hkv, dk, dv, kb, vb, cbk, cbv, scale)
    torch.cuda.synchronize()
    worst = 0.0
    for i, (kc, vc, cap, n, q) in enumerate(seqs_np):
        o_ref, P, Kh, Vh = O.kv_attend(kc, vc, cap, n, q.astype(np.float32).astype(np.float64),
                                       Hkv, dk, dv, kb, vb, cbk, cbv, np.float32(scale))
        o = outs[i].cpu().numpy()
        if n == 0:
            assert np.all(o == 0), f"{what}: empty sequence {i} must give zeros"
            continue
        bound = attention_bound(Kh, Vh, q.astype(np.float32).astype(np.float64), P, o_ref, Hkv, scale)
        worst = max(worst, check_attention(o, o_ref, bound, f"{what} seq {i} (n={n})"))
    return worst


GEOMS = [(12, 2, 48, 64), (8, 4, 64, 64), (16, 1, 128, 128), (1, 1, 32, 200), (6, 3, 40, 24), (4, 2, 256, 96)]


@pytest.mark.parametrize("geom", GEOMS)
@pytest.mark.parametrize("bits", [(2, 2), (4, 4), (3, 2), (5, 4), (2, 3)])
def test_kv_attend_matches_oracle(C, geom, bits):
    """Ragged batch in one call: sequences of 1, 7, 128, 129, 300 and 0
    tokens, each cache with 13 spare rows of 0xFF bytes past n_tokens."""
    Hq, Hkv, dk, dv = geom
    kb, vb = bits
    rng = np.random.RandomState(sum(geom) + 10 * kb + vb)
    seqs = []
    for j, n in enumerate([1, 7, 128, 129, 300, 0]):
        cap = n + 13
        kc = _filled_cache(cap, _width(Hkv, dk), kb, n, 100 + j)
        vc = _filled_cache(cap, _width(Hkv, dv), vb, n, 200 + j)
        seqs.append((kc, vc, cap, n, rng.randn(Hq, dk).astype(np.float32)))
    worst = _run_and_check(C, geom, kb, vb, seqs, 1.0 / math.sqrt(dk), f"{geom} bits={bits}")
    print(f"{geom} bits={bits}: max |err|/bound {worst:.2e}")


def test_kv_attend_long_sequences_merge_chunks(C):
    """Sequences of 8192 and 3001 tokens split over many blocks whose
    partial results are merged; a short one rides in the same launch."""
    geom = (12, 2, 48, 64)
    rng = np.random.RandomState(7)
    seqs = []
    for j, n in enumerate([8192, 3001, 5]):
        kc = _filled_cache(n + 3, 96, 2, n, 300 + j)
        vc = _filled_cache(n + 3, 128, 2, n, 400 + j)
        seqs.append((kc, vc, n + 3, n, rng.randn(12, 48).astype(np.float32)))
    _run_and_check(C, geom, 2, 2, seqs, 1.0 / math.sqrt(48), "long")


def test_kv_attend_more_than_256_sequences(C):
    """300 sequences: the call is split into launches of at most 256."""
    geom = (8, 4, 64, 64)
    rng = np.random.RandomState(8)
    seqs = []
    for j in range(300):
        n = int(rng.randint(1, 200))
        kc = _filled_cache(n, 256, 4, n, 1000 + j)
        vc = _filled_cache(n, 256, 2, n, 2000 + j)
        seqs.append((kc, vc, n, n, rng.randn(8, 64).astype(np.float32)))
    _run_and_check(C, geom, 4, 2, seqs, 0.125, "300 seqs")


def test_kv_attend_peaked_and_flat_logits(C):
    """Large key norms make the softmax nearly one-hot (logits of order
    100); scale 0 makes it exactly uniform (the mean of the value rows)."""
    geom = (4, 2, 64, 64)
    rng = np.random.RandomState(9)
    n = 257
    kc = S.kv_cache_blob(n, 128, 2, 11, norm_lo=200.0, norm_hi=400.0)
    vc = S.kv_cache_blob(n, 128, 4, 12)
    q = rng.randn(4, 64).astype(np.float32)
    _run_and_check(C, geom, 2, 4, [(kc, vc, n, n, q)], 0.125, "peaked")
    _run_and_check(C, geom, 2, 4, [(kc, vc, n, n, q)], 0.0, "flat")


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("width", [96, 128, 300])
def test_kv_write_matches_oracle(C, bits, width):
    """Rows written in two pieces into a cache of 40 rows: codes equal the
    oracle's (boundary coordinates excepted), norms bit-exact, rows outside
    the pieces untouched."""
    cap = 40
    cb = O.analytic_codebook(bits)
    rows = S.normal((cap, width), 50 + bits + width).numpy()
    ref = np.full(O.packed_bytes(cap, width, 128, bits), 0xA5, dtype=np.uint8)
    flags = np.zeros((cap, O.in_padded(width)), dtype=np.uint8)
    for a, b in ((5, 17), (17, 33)):
        f, _ = O.kv_write(ref, cap, width, bits, cb, rows[a:b], a)
        flags[a:b] = f
    dev = torch.full((ref.size,), 0xA5, dtype=torch.uint8, device="cuda")
    rows_d = torch.from_numpy(rows).cuda()
    for a, b in ((5, 17), (17, 33)):
        C.cq_kv_write(dev, cap, width, bits, cb, rows_d[a:b].contiguous(), a)
    torch.cuda.synchronize()
    got = dev.cpu().numpy()
    compare_encodings(got, ref, flags, cap, width, bits)
    ip = O.in_padded(width)
    rb = ip * O.width(bits) // 8
    assert np.all(got[:5 * rb] == 0xA5) and np.all(got[33 * rb:cap * rb] == 0xA5)


def test_kv_attend_full_size_sampled(C):
    """The benchmark's workload (256 sequences x 8192 tokens, Needle 3
    attention geometry, CQ2 keys and values) in one call; the oracle checks
    four sampled sequences."""
    g = S.KV_GEOM
    Hq, Hkv, dk, dv = g["n_q_heads"], g["n_kv_heads"], g["head_dim_k"], g["head_dim_v"]
    T, nseq, bits = S.KV_TOKENS, S.KV_SEQS, S.KV_BITS
    cb = O.analytic_codebook(bits)
    kb_np = [S.kv_cache_blob(T, Hkv * dk, bits, 5000 + i) for i in range(nseq)]
    vb_np = [S.kv_cache_blob(T, Hkv * dv, bits, 6000 + i) for i in range(nseq)]
    qs = [S.normal((Hq, dk), 7000 + i).numpy() for i in range(nseq)]
    items = [dict(k_cache=torch.from_numpy(k).cuda(), v_cache=torch.from_numpy(v).cuda(), cap=T,
                  n_tokens=T, q=torch.from_numpy(q).cuda()) for k, v, q in zip(kb_np, vb_np, qs)]
    outs = C.cq_kv_attend(items, Hq, Hkv, dk, dv, bits, bits, cb, cb, 1.0 / math.sqrt(dk))
    torch.cuda.synchronize()
    scale = np.float32(1.0 / math.sqrt(dk))
    for i in (0, 1, 137, 255):
        o_ref, P, Kh, Vh = O.kv_attend(kb_np[i], vb_np[i], T, T, qs[i].astype(np.float64), Hkv, dk, dv,
                                       bits, bits, cb, cb, scale)
        bound = attention_bound(Kh, Vh, qs[i].astype(np.float64), P, o_ref, Hkv, float(scale))
        check_attention(outs[i].cpu().numpy(), o_ref, bound, f"full-size seq {i}")
