"""Container writer/reader (host only): round trip, layout as the pages
define it, and the reader's refusal of malformed files before it exposes
any byte. Pages: "The .cact format" ("Five regions", "Reading one
yourself", "Versions"); "The .cact archive and Cactus Quants" ("Header",
"Tensor directory", "Anatomy of a CQ matrix")."""
import struct

import numpy as np
import pytest

import oracle as O


@pytest.fixture(scope="module")
def C():
    from hadamard_rotated_codebook_gb300 import build
    build.build()
    import hadamard_rotated_codebook_gb300 as pkg
    return pkg


def _codebook28():
    return np.concatenate([O.analytic_codebook(2), O.analytic_codebook(3), O.analytic_codebook(4)])


def _sample_tensors():
    rng = np.random.RandomState(1)
    W = (rng.randn(40, 300) * 0.02).astype(np.float32)
    blob, _, _ = O.encode(W, 2, O.analytic_codebook(2))
    W4 = (rng.randn(7, 128) * 0.02).astype(np.float32)
    blob4, _, _ = O.encode(W4, 4, O.analytic_codebook(4))
    f16 = rng.randn(33).astype(np.float16)
    f32 = rng.randn(2, 3, 5).astype(np.float32)
    raw = b"tokenizer bytes \x00\x01\x02"
    return [
        dict(dtype=3, shape=(40, 300), data=blob.tobytes(), group=128, bits=2),
        dict(dtype=1, shape=(33,), data=f16.tobytes()),
        dict(dtype=2, shape=(2, 3, 5), data=f32.tobytes()),
        dict(dtype=3, shape=(7, 128), data=blob4.tobytes(), group=128, bits=4),
        dict(dtype=4, shape=(len(raw),), data=raw),
        dict(dtype=2, shape=(0,), data=b""),
    ]


def test_round_trip(C, tmp_path):
    path = str(tmp_path / "m.cact")
    ts = _sample_tensors()
    cb = _codebook28()
    C.cq_cact_write(path, ts, cb, 128)
    with C.cq_cact_open(path) as r:
        assert len(r) == len(ts)
        np.testing.assert_array_equal(r.codebook(), cb)
        assert r.default_group() == 128
        for i, t in enumerate(ts):
            got = r.tensor(i)
            assert got.dtype == t["dtype"] and got.shape == tuple(t["shape"])
            assert got.data == t["data"]
            assert got.group == t.get("group", 0) and got.bits == t.get("bits", 0)


def test_layout_matches_the_pages_record_format(C, tmp_path):
    """Parse the file with struct exactly as the pages' Python reader does:
    44-byte '<BBHIIIIQQII' records (dtype, ndim, pad, shape[4], offset,
    nbytes, group, bits), blobs at absolute 64-byte-aligned offsets, dtype
    codes 1 FP16, 2 FP32, 3 CQ, 4 RAW."""
    path = str(tmp_path / "m.cact")
    ts = _sample_tensors()
    C.cq_cact_write(path, ts, _codebook28(), 128)
    b = open(path, "rb").read()
    tag, ver, hb, n, cbl, grp = struct.unpack_from("<6I", b, 0)
    assert tag == 0x42475143 and ver == 1 and hb == 64 and n == len(ts) and cbl == 28 and grp == 128
    cb = np.frombuffer(b, dtype="<f4", count=28, offset=64)
    np.testing.assert_array_equal(cb, _codebook28())
    off = 64 + 28 * 4
    for t in ts:
        dtype, ndim, pad, s0, s1, s2, s3, start, nbytes, group, bits = struct.unpack_from("<BBHIIIIQQII", b, off)
        assert struct.calcsize("<BBHIIIIQQII") == 44
        assert dtype == t["dtype"] and ndim == len(t["shape"]) and pad == 0
        assert (s0, s1, s2, s3)[:ndim] == tuple(t["shape"]) and all(v == 0 for v in (s0, s1, s2, s3)[ndim:])
        assert start % 64 == 0 and b[start:start + nbytes] == t["data"]
        assert group == t.get("group", 0) and bits == t.get("bits", 0)
        off += 44


def test_cq_blob_length_formula(C, tmp_path):
    """[NJ] "Anatomy of a CQ matrix": nbytes = out*in_pad*b/8 + out*(in_pad/g)*2."""
    ts = _sample_tensors()
    assert len(ts[0]["data"]) == 40 * 384 * 2 // 8 + 40 * 3 * 2


def _good_file(C, tmp_path):
    path = str(tmp_path / "good.cact")
    C.cq_cact_write(path, _sample_tensors(), _codebook28(), 128)
    return bytearray(open(path, "rb").read())


def _expect_format_error(C, data, needle):
    from hadamard_rotated_codebook_gb300 import CQError
    with pytest.raises(CQError) as ei:
        C.cq_cact_open_memory(bytes(data))
    assert "CQ_ERR_FORMAT" in str(ei.value) and needle in str(ei.value), str(ei.value)


REC0 = 64 + 28 * 4


def test_reader_refuses_needle_tags(C, tmp_path):
    """[CF] "Versions": an engine handed another generation's tag refuses
    with a message rather than guessing."""
    b = _good_file(C, tmp_path)
    for tag, gen in ((0x05E12A83, "Needle 2"), (0x05E12A84, "Needle 3")):
        struct.pack_into("<I", b, 0, tag)
        _expect_format_error(C, b, gen)
    struct.pack_into("<I", b, 0, 0xDEADBEEF)
    _expect_format_error(C, b, "unknown tag")


def test_reader_bounds_and_alignment(C, tmp_path):
    """[NJ] "Tensor directory": a malformed offset must fail before
    allocation or indexing."""
    good = _good_file(C, tmp_path)
    b = bytearray(good)
    struct.pack_into("<Q", b, REC0 + 20, 2 ** 64 - 64)  # offset wraps when nbytes is added
    _expect_format_error(C, b, "outside")
    b = bytearray(good)
    struct.pack_into("<Q", b, REC0 + 28, 2 ** 64 - 1)  # nbytes huge
    _expect_format_error(C, b, "outside")
    b = bytearray(good)
    off = struct.unpack_from("<Q", b, REC0 + 20)[0]
    struct.pack_into("<Q", b, REC0 + 20, off + 8)
    _expect_format_error(C, b, "aligned")
    b = bytearray(good)
    struct.pack_into("<Q", b, REC0 + 20, 64)
    _expect_format_error(C, b, "overlaps")
    _expect_format_error(C, good[: len(good) - 10], "outside")  # truncated last blob
    _expect_format_error(C, good[:40], "truncated")
    b = bytearray(good)
    struct.pack_into("<I", b, 12, 10 ** 6)  # directory larger than the file
    _expect_format_error(C, b, "does not fit")


def test_reader_record_semantics(C, tmp_path):
    good = _good_file(C, tmp_path)
    b = bytearray(good)
    b[REC0 + 1] = 5  # ndim
    _expect_format_error(C, b, "ndim")
    b = bytearray(good)
    b[REC0] = 9  # dtype
    _expect_format_error(C, b, "dtype")
    b = bytearray(good)
    struct.pack_into("<I", b, REC0 + 36, 96)  # group not a power of two
    _expect_format_error(C, b, "power of two")
    b = bytearray(good)
    struct.pack_into("<Q", b, REC0 + 28, struct.unpack_from("<Q", b, REC0 + 28)[0] - 2)
    _expect_format_error(C, b, "inconsistent")
    b = bytearray(good)
    struct.pack_into("<I", b, REC0 + 40, 6)  # bits
    _expect_format_error(C, b, "bits")
    rec1 = REC0 + 44  # FP16 record with a wrong byte count
    b = bytearray(good)
    struct.pack_into("<I", b, rec1 + 4, 34)
    _expect_format_error(C, b, "does not match")
    b = bytearray(good)
    struct.pack_into("<I", b, 40, 7)  # reserved header field
    _expect_format_error(C, b, "reserved")
    b = bytearray(good)
    struct.pack_into("<f", b, 64, float("nan"))
    _expect_format_error(C, b, "codebook")


def test_writer_rejects_inconsistent_cq_record(C, tmp_path):
    from hadamard_rotated_codebook_gb300 import CQError
    ts = _sample_tensors()
    ts[0] = dict(ts[0], data=ts[0]["data"][:-2])
    with pytest.raises(CQError):
        C.cq_cact_write(str(tmp_path / "bad.cact"), ts, _codebook28(), 128)
    assert not (tmp_path / "bad.cact").exists()


def test_missing_file_is_io_error(C, tmp_path):
    from hadamard_rotated_codebook_gb300 import CQError
    with pytest.raises(CQError) as ei:
        C.cq_cact_open(str(tmp_path / "nope.cact"))
    assert "CQ_ERR_IO" in str(ei.value)


def test_round_trip_binary_and_group64_records(C, tmp_path):
    """Binary codes (bits 1, eight per byte) and 64-wide groups are valid
    records ([CF] "Cactus Quants"): the reader checks their byte counts with
    the same formula and hands back the blobs unchanged; a record whose
    nbytes disagrees is refused."""
    rng = np.random.RandomState(2)
    W = (rng.randn(9, 256) * 0.02).astype(np.float32)
    b1, _, _ = O.encode(W, 1, O.analytic_codebook(1, 128), 128)
    b64, _, _ = O.encode(W, 2, O.analytic_codebook(2, 64), 64)
    assert b1.size == 9 * 256 // 8 + 9 * 2 * 2 and b64.size == 9 * 256 // 4 + 9 * 4 * 2
    ts = [dict(dtype=3, shape=(9, 256), data=b1.tobytes(), group=128, bits=1),
          dict(dtype=3, shape=(9, 256), data=b64.tobytes(), group=64, bits=2)]
    path = str(tmp_path / "g.cact")
    C.cq_cact_write(path, ts, _codebook28(), 128)
    with C.cq_cact_open(path) as r:
        for i, t in enumerate(ts):
            got = r.tensor(i)
            assert got.data == t["data"] and got.group == t["group"] and got.bits == t["bits"]
    bad = [dict(dtype=3, shape=(9, 256), data=b1.tobytes()[:-2], group=128, bits=1)]
    with pytest.raises(C.CQError):
        C.cq_cact_write(str(tmp_path / "bad.cact"), bad, _codebook28(), 128)
