"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
side of every comparison. Holds no CQ arithmetic: only random tensors and
the shapes of the workloads.

Workloads (the pages ship no data; the shapes follow the Needle-2 geometry
in OpenNeedle docs/reference.md -- width 512, 27 layers, 8 query heads and
4 key/value heads of 64, vocabulary 8192, tied CQ4 embedding head):

* ``single``:  one CQ2 matrix 512x512, W ~ N(0, 0.02^2) seed 0, x ~ N(0,1)
  seed 1, batch 1.
* ``decode``:  27 layers x {Q 512x512, K 256x512, V 256x512, gate 512x512,
  O 512x512} in CQ2 plus the head 8192x512 in CQ4 (136 matrices); weights
  N(0, 0.02^2) with seed 1000+index (layer-major, Q K V gate O, head last);
  activations N(0,1) with one vector per layer shared by Q/K/V/gate (the
  shared rotated input of OpenNeedle's fused QKVG path), one for O and one
  for the head, seeds 2000+activation index; int8 per token on the device.
* ``prefill``: the same matrix set with M tokens of activations per input.
* ``sweep``:   4096x4096 and 14336x4096, W = 0.02 * t4 (Student t, nu = 4,
  z / sqrt(chi2_4 / 4) from five seeded normals), x ~ N(0,1).
* ``encode``:  16 matrices 8192x8192 ~ N(0, 0.02^2), each entry scaled by 20
  with independent probability 0.01 (outliers).
* ``kv``:      decode-step attention over CQ key/value caches in the Needle 3
  attention geometry ("Porting Needle 3", "The geometry, for the header": 12
  query heads of 48 over 2 key/value heads, value heads of 64, context
  8192): 256 sequences of 8192 cached tokens, CQ2 keys and values. Caches
  are seeded random blobs (random codes, fp16 norms uniform in [1, 8)) so
  that the logits spread over several units; queries N(0, 1); logit scale
  1/sqrt(48).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

import torch

W_STD = 0.02


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def student_t4(shape, seed: int, scale: float = W_STD, device="cpu") -> torch.Tensor:
    """scale * z / sqrt(chi2_4/4), chi2_4 = sum of four squared normals."""
    g = _gen(seed, device)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(4):
        chi += torch.randn(shape, generator=g, device=device, dtype=torch.float32) ** 2
    return scale * z / torch.sqrt(chi / 4)


def with_outliers(W: torch.Tensor, seed: int, prob: float = 0.01, factor: float = 20.0) -> torch.Tensor:
    g = _gen(seed, W.device)
    mask = torch.rand(W.shape, generator=g, device=W.device) < prob
    return torch.where(mask, W * factor, W)


@dataclass(frozen=True)
class Mat:
    name: str
    out: int
    n_in: int
    bits: int
    w_seed: int
    act: int  # activation index


def decode_step_mats(layers: int = 27) -> List[Mat]:
    mats = []
    idx = 0
    for l in range(layers):
        for nm, out in (("q", 512), ("k", 256), ("v", 256), ("gate", 512), ("o", 512)):
            act = 2 * l + (1 if nm == "o" else 0)
            mats.append(Mat(f"l{l}.{nm}", out, 512, 2, 1000 + idx, act))
            idx += 1
    mats.append(Mat("head", 8192, 512, 4, 1000 + idx, 2 * layers))
    return mats


def n_activations(mats: List[Mat]) -> int:
    return max(m.act for m in mats) + 1


def act_seed(a: int) -> int:
    return 2000 + a


def decode_weights(m: Mat, device="cpu") -> torch.Tensor:
    return normal((m.out, m.n_in), m.w_seed, W_STD, device)


def decode_activation(a: int, tokens: int = 1, n_in: int = 512, device="cpu") -> torch.Tensor:
    return normal((tokens, n_in), act_seed(a), 1.0, device)


SWEEP_SHAPES = [(4096, 4096), (14336, 4096)]
SWEEP_BITS = [2, 3, 4, 5]
SWEEP_BATCHES = [1, 16]
ENCODE_SHAPE = (8192, 8192)
ENCODE_COUNT = 16


def single_weights(device="cpu") -> torch.Tensor:
    """The single 512x512 CQ2 matrix: N(0, 0.02^2), seed 0."""
    return normal((512, 512), 0, W_STD, device)


def single_activation(device="cpu") -> torch.Tensor:
    """Its batch-1 activation: N(0, 1), seed 1."""
    return normal((1, 512), 1, 1.0, device)


def sweep_weights(shape, bits: int, device="cpu") -> torch.Tensor:
    """Width-sweep weights: 0.02 * Student t (4 dof), one seed per shape and width."""
    seed = 3000 + 10 * SWEEP_SHAPES.index(tuple(shape)) + SWEEP_BITS.index(bits)
    return student_t4(tuple(shape), seed, W_STD, device)


def sweep_activation(B: int, n_in: int, device="cpu") -> torch.Tensor:
    """Width-sweep activations: fp32 N(0, 1), [B, n_in]."""
    return normal((B, n_in), 3500 + B, 1.0, device)


def encode_matrix(i: int, device="cpu", shape=ENCODE_SHAPE) -> torch.Tensor:
    W = normal(shape, 5000 + i, W_STD, device)
    return with_outliers(W, 6000 + i)


def random_blob(code_bytes: int, n_norms: int, seed: int, ternary: bool = False,
                norm_lo: float = 0.05, norm_hi: float = 0.5) -> "np.ndarray":
    """A seeded CQ blob of random content: `code_bytes` random code bytes
    (for ternary only the crumbs 00, 01, 11) followed by `n_norms` fp16
    norms uniform in [norm_lo, norm_hi). Any such byte string is a valid
    blob, so products over it can be checked without an encoder."""
    import numpy as np

    rng = np.random.RandomState(seed)
    if ternary:
        crumbs = rng.choice(np.array([0, 1, 3], dtype=np.uint8), size=(code_bytes, 4))
        codes = (crumbs[:, 0] | (crumbs[:, 1] << 2) | (crumbs[:, 2] << 4) | (crumbs[:, 3] << 6)).astype(np.uint8)
    else:
        codes = rng.randint(0, 256, size=code_bytes).astype(np.uint8)
    norms = rng.uniform(norm_lo, norm_hi, size=n_norms).astype(np.float16)
    return np.concatenate([codes, norms.view(np.uint8)])


# ------------------------------------------------------------------ kv --
KV_GEOM = dict(n_q_heads=12, n_kv_heads=2, head_dim_k=48, head_dim_v=64)
KV_SEQS, KV_TOKENS, KV_BITS = 256, 8192, 2


def kv_cache_blob(cap: int, width: int, bits: int, seed: int, norm_lo: float = 1.0,
                  norm_hi: float = 8.0) -> "np.ndarray":
    """A seeded random CQ cache of `cap` rows of `width` columns."""
    ip = (width + 127) // 128 * 128
    w = 2 if bits == 5 else bits
    return random_blob(cap * ip * w // 8, cap * ip // 128, seed, ternary=bits == 5,
                       norm_lo=norm_lo, norm_hi=norm_hi)
