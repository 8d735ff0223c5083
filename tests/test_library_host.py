"""Host-side checks of libcq (no GPU needed): the library loads, exports
every entry point include/cq.h declares, and its host logic (codebooks,
byte accounting, argument validation) agrees with the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def C():
    from hadamard_rotated_codebook_gb300 import build
    build.build()
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "cq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(cq_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(C):
    from hadamard_rotated_codebook_gb300 import _capi
    lib = ctypes.CDLL(C.library_path())
    declared = _declared_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), f"libcq.so does not export {name}"
    # and the binding types every one of them
    assert set(declared) == set(_capi.SIGNATURES)


def test_library_is_built_for_sm103a(C):
    # the build recipe is the one the package ships; check its arch flags
    from hadamard_rotated_codebook_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
def test_codebook_init_matches_oracle(C, bits):
    np.testing.assert_array_equal(C.cq_codebook_init(bits, 128), O.analytic_codebook(bits, 128))
    np.testing.assert_array_equal(C.cq_codebook_init(bits, 64), O.analytic_codebook(bits, 64))


def test_codebook_init_query_and_errors(C):
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    n = ctypes.c_size_t(0)
    assert lib.cq_codebook_init(4, 128, None, 0, ctypes.byref(n)) == 0 and n.value == 16
    assert lib.cq_codebook_init(6, 128, None, 0, None) == _capi.CQ_ERR_ARG
    assert lib.cq_codebook_init(2, 100, None, 0, None) == _capi.CQ_ERR_ARG
    buf = (ctypes.c_float * 2)()
    assert lib.cq_codebook_init(2, 128, buf, 2, None) == _capi.CQ_ERR_ARG
    assert b"need 4" in lib.cq_last_error()


def test_levels_and_widths(C):
    for bits in (1, 2, 3, 4, 5):
        assert C.cq_levels(bits) == O.levels(bits)
        assert C.cq_code_width(bits) == O.width(bits)
    assert C.cq_levels(0) == -1 and C.cq_code_width(7) == -1


def test_packed_bytes_matches_oracle(C):
    rng = np.random.RandomState(0)
    for _ in range(200):
        out, n_in = int(rng.randint(0, 5000)), int(rng.randint(0, 9000))
        group = int(2 ** rng.randint(3, 9))
        bits = int(rng.choice([2, 3, 4, 5]))
        assert C.cq_packed_bytes(out, n_in, group, bits) == O.packed_bytes(out, n_in, group, bits)
    assert C.cq_packed_bytes(4, 4, 96, 2) == 0
    assert C.cq_packed_bytes(-1, 4, 128, 2) == 0


def test_device_entry_points_reject_bad_arguments_before_launch(C):
    """Argument errors come back as status codes with a message, before any
    CUDA call (this host has no GPU)."""
    from hadamard_rotated_codebook_gb300 import _capi
    lib = _capi.load()
    cb = (ctypes.c_float * 4)(-0.1, -0.03, 0.03, 0.1)
    bad = (ctypes.c_float * 4)(-0.1, 0.03, -0.03, 0.1)
    assert lib.cq_encode(None, 4, 128, 32, 2, cb, None, None) == _capi.CQ_ERR_SHAPE
    assert b"group = 64 or 128" in lib.cq_last_error()
    assert lib.cq_encode(None, 4, 128, 64, 2, cb, None, None) == _capi.CQ_ERR_ARG  # group 64 taken; null W
    # the GEMM takes groups of 64 on whole 128-wide spans up to 512 inputs;
    # the sizes pass and the unaligned pointers are the error
    g64 = _capi.GemmDesc(blob=1, Xq=1, x_scale=1, Y=1, codebook=cb, out=4, in_=128, group=64, bits=2, M=8)
    assert lib.cq_gemm_grouped(ctypes.byref(g64), 1, None) == _capi.CQ_ERR_ARG
    for n_in in (192, 640):
        g64.in_ = n_in
        assert lib.cq_gemm_grouped(ctypes.byref(g64), 1, None) == _capi.CQ_ERR_SHAPE
        assert b"groups of 64" in lib.cq_last_error()
    b1 = (ctypes.c_float * 2)(-0.07, 0.07)
    g1 = _capi.GemmDesc(blob=1, Xq=1, x_scale=1, Y=1, codebook=b1, out=4, in_=1000, group=128, bits=1, M=8)
    assert lib.cq_gemm_grouped(ctypes.byref(g1), 1, None) == _capi.CQ_ERR_ARG  # binary codes taken
    assert lib.cq_encode(None, 4, 128, 128, 2, bad, None, None) == _capi.CQ_ERR_ARG
    assert b"increasing" in lib.cq_last_error()
    assert lib.cq_encode(None, 4, 128, 128, 7, cb, None, None) == _capi.CQ_ERR_ARG
    assert lib.cq_encode(None, 4, 128, 128, 2, cb, None, None) == _capi.CQ_ERR_ARG  # null W
    assert lib.cq_encode(None, 0, 128, 128, 2, cb, None, None) == _capi.CQ_OK  # empty: no work
    d = _capi.GemvDesc(blob=1, x=1, x_scale=None, y=1, codebook=cb, out=4, in_=128, group=128,
                       bits=2, x_dtype=_capi.CQ_X_F32, B=17)
    assert lib.cq_gemv_grouped(ctypes.byref(d), 1, None) == _capi.CQ_ERR_SHAPE
    assert b"descriptor 0" in lib.cq_last_error()
    d.B, d.x_dtype = 1, _capi.CQ_X_I8
    assert lib.cq_gemv_grouped(ctypes.byref(d), 1, None) == _capi.CQ_ERR_ARG  # no scales
    d.x_dtype = 3
    assert lib.cq_gemv_grouped(ctypes.byref(d), 1, None) == _capi.CQ_ERR_ARG  # unknown activation type
    assert b"x_dtype" in lib.cq_last_error()
    d.x_dtype, d.blob = _capi.CQ_X_F32Q, 8  # quantised in the call: no scales needed; a misaligned blob
    assert lib.cq_gemv_grouped(ctypes.byref(d), 1, None) == _capi.CQ_ERR_ARG  # is the next check to fail
    assert b"16-byte aligned" in lib.cq_last_error()
    d.blob = 1
    assert lib.cq_gemv_grouped(ctypes.byref(d), 0, None) == _capi.CQ_ERR_ARG
    g = _capi.GemmDesc(blob=1, Xq=1, x_scale=None, Y=1, codebook=cb, out=4, in_=128, group=128,
                       bits=2, M=8)
    assert lib.cq_gemm_grouped(ctypes.byref(g), 1, None) == _capi.CQ_ERR_ARG
    assert lib.cq_act_quant_int8(None, 2, 8, None, None, None) == _capi.CQ_ERR_ARG
    bl = (ctypes.c_void_p * 2)(1, 1)
    outs = (ctypes.c_int * 2)(4, 4)
    ys = (ctypes.c_void_p * 2)(1, 1)
    assert lib.cq_gemv_shared(bl, outs, 0, 128, 128, 2, cb, 1, _capi.CQ_X_F32, None, 1, ys, None) == _capi.CQ_ERR_ARG
    assert lib.cq_gemv_shared(None, outs, 2, 128, 128, 2, cb, 1, _capi.CQ_X_F32, None, 1, ys, None) == _capi.CQ_ERR_ARG
    assert lib.cq_gemv_shared(bl, outs, 2, 128, 128, 2, cb, 1, _capi.CQ_X_F32, None, 17, ys, None) == _capi.CQ_ERR_SHAPE
    geom = _capi.KvGeom(n_q_heads=12, n_kv_heads=5, head_dim_k=48, head_dim_v=64, k_bits=2, v_bits=2,
                        k_codebook=cb, v_codebook=cb, scale=0.1)
    seq = _capi.KvSeq(k_cache=16, v_cache=16, q=16, o=16, cap=4, n_tokens=5)
    assert lib.cq_kv_attend(ctypes.byref(geom), ctypes.byref(seq), 1, None) == _capi.CQ_ERR_SHAPE  # 12 % 5
    geom.n_kv_heads = 2
    assert lib.cq_kv_attend(ctypes.byref(geom), ctypes.byref(seq), 1, None) == _capi.CQ_ERR_SHAPE  # n > cap
    assert b"sequence 0" in lib.cq_last_error()
    seq.n_tokens, seq.k_cache = 4, 8
    assert lib.cq_kv_attend(ctypes.byref(geom), ctypes.byref(seq), 1, None) == _capi.CQ_ERR_ARG  # alignment
    geom.head_dim_k = 300
    assert lib.cq_kv_attend(ctypes.byref(geom), ctypes.byref(seq), 1, None) == _capi.CQ_ERR_SHAPE  # 600 > 512
    assert lib.cq_kv_attend(ctypes.byref(geom), ctypes.byref(seq), 0, None) == _capi.CQ_ERR_ARG
    assert lib.cq_kv_write(None, 4, 96, 2, cb, None, 2, 3, None) == _capi.CQ_ERR_SHAPE  # rows past cap
    assert lib.cq_kv_write(None, 4, 96, 2, cb, None, 0, 2, None) == _capi.CQ_ERR_ARG   # null cache
    assert lib.cq_kv_write(None, 4, 96, 2, cb, None, 1, 0, None) == _capi.CQ_OK        # nothing to write


def test_binding_requires_the_library(tmp_path, monkeypatch):
    """No silent fallback: a missing libcq.so is an ImportError."""
    from hadamard_rotated_codebook_gb300 import _capi
    monkeypatch.setattr(_capi, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_capi, "_lib", None)
    with pytest.raises(ImportError):
        _capi.load()
