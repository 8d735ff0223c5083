"""Host logic of bench.py on the CPU: the DRAM-traffic records are reported
only while the kernel sources still hash to the build they were taken on."""
import os

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
