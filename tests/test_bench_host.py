"""Host logic of bench.py on the CPU: the DRAM-traffic records are reported
only while the kernel sources still hash to the build they were taken on."""
import os

import numpy as np

import bench


def test_traffic_records_name_existing_sources():
    csrc = os.path.join(bench.ROOT, "hadamard_rotated_codebook_gb300", "csrc")
    assert set(bench.NCU_TRAFFIC) <= set(bench.KERNEL_SOURCES)
    for kernel, (key, nbytes) in bench.NCU_TRAFFIC.items():
        assert len(key) == 16 and int(key, 16) >= 0
        assert nbytes > 0
        for name in bench.KERNEL_SOURCES[kernel]:
            assert os.path.isfile(os.path.join(csrc, name)), name


def test_traffic_follows_the_source_hash(monkeypatch):
    kernel, (key, nbytes) = next(iter(bench.NCU_TRAFFIC.items()))
    monkeypatch.setattr(bench, "_src_hash", lambda *names: key)
    assert bench.ncu_traffic(kernel) == nbytes
    monkeypatch.setattr(bench, "_src_hash", lambda *names: "0" * 16)
    assert bench.ncu_traffic(kernel) is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_source_hash_changes_with_any_named_file(tmp_path, monkeypatch):
    pkg = tmp_path / "hadamard_rotated_codebook_gb300" / "csrc"
    pkg.mkdir(parents=True)
    (pkg / "a.cu").write_text("kernel a\n")
    (pkg / "b.h").write_text("header\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._src_hash("a.cu", "b.h")
    (pkg / "b.h").write_text("header changed\n")
    assert bench._src_hash("a.cu", "b.h") != h0


def _fake_run():
    """A tiny decode-shaped sample whose 'GPU' outputs are the oracle's own,
    plus one sampled GEMV line and one encode line."""
    import numpy as np

    import oracle as O
    import synthetic as S
    mats = [S.Mat("a", 64, 256, 2, 0, 0), S.Mat("b", 40, 256, 4, 1, 1)]
    cbs = {2: O.analytic_codebook(2), 4: O.analytic_codebook(4)}
    rng = np.random.RandomState(3)
    Ws = [(rng.randn(m.out, m.n_in) * 0.02).astype(np.float32) for m in mats]
    blobs = [O.encode(W, m.bits, cbs[m.bits])[0] for W, m in zip(Ws, mats)]
    Xq, xs = O.act_quant_int8(rng.randn(2, 256).astype(np.float32))
    ys = []
    for m, b in zip(mats, blobs):
        xt = Xq[m.act:m.act + 1].astype(np.float64) * np.float64(xs[m.act])
        ys.append(O.matmul(O.dequant(b, m.out, m.n_in, m.bits, cbs[m.bits]), xt)[0][0].astype(np.float32))
    rows = [bench.sample_rows(m.out, 4) for m in mats]
    samples = bench.Samples()
    samples.add(("parity",), "decode", wl=dict(mats=mats, blobs=blobs, cbs=cbs, Xq=Xq, xs=xs, y=ys,
                                                w_rows=[(r, W[r]) for r, W in zip(rows, Ws)]))
    x = rng.randn(3, 256)
    r = np.arange(10)
    sub = bench.host_sub_blob(blobs[0], 64, 256, 2, r)
    y = O.matmul(O.dequant(sub, 10, 256, 2, cbs[2]), x)[0]
    samples.add(("sweep", "line"), "gemv", blob=sub, rows=r, n_in=256, bits=2, group=128, cb=cbs[2], x=x,
                y=y.astype(np.float32))
    samples.add(("sweep", "line_encode"), "encode", W=Ws[1][:5], blob=bench.host_sub_blob(blobs[1], 40, 256, 4,
                                                                                        np.arange(5)),
                bits=4, group=128, cb=cbs[4])
    return samples


def test_oracle_leg_reports_parity_and_both_baselines():
    """The oracle leg fills the CPU baseline (one thread and all cores, with
    the core count and CPU model) and the parity objects; outputs equal to
    the oracle's pass, encodings from the oracle have no mismatches."""
    samples = _fake_run()
    result = {}
    bench.oracle_leg(result, samples, budget_s=5.0)
    cb = result["cpu_baseline"]
    assert cb["cores"] >= 1 and cb["kind"] == "oracle" and cb["value"] > 0 and cb["cpu_model"]
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    par = result["parity"]
    assert par["pass"] and par["max_err_over_bound"] < 1e-3 and par["outputs_checked"] == 104
    assert par["encode"]["pass"] and par["encode"]["code_mismatch"] == 0 and par["encode"]["norm_mismatch"] == 0
    assert result["sweep"]["line"]["parity"]["pass"]
    assert result["sweep"]["line_encode"]["parity"]["coords"] == 5 * 256


def test_oracle_leg_flags_a_wrong_output():
    samples = _fake_run()
    dec = samples.items[0]["wl"]
    dec["y"][1] = dec["y"][1].copy()
    dec["y"][1][7] += 0.05 * (abs(dec["y"][1][7]) + 1.0)  # one output off by far more than the bound
    line = samples.items[1]
    line["y"] = line["y"] * 1.01
    result = {}
    bench.oracle_leg(result, samples, budget_s=5.0)
    assert not result["parity"]["pass"] and result["parity"]["max_err_over_bound"] > 2e-3
    assert not result["sweep"]["line"]["parity"]["pass"]


def test_sample_rows_span_the_range():
    r = bench.sample_rows(8192, 16)
    assert r[0] == 0 and r[-1] == 8191 and len(r) == 16 and (np.diff(r) > 0).all()
    assert list(bench.sample_rows(5, 16)) == [0, 1, 2, 3, 4]
