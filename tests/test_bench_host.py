"""Host-side logic of bench.py: the code hash that keys recorded DRAM counters and
the lookup of those records (no GPU needed)."""
import json
import shutil

import pytest

import bench


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    """A copy of the kernel sources and the traffic records under a scratch root."""
    csrc = tmp_path / "quant_dequant_gemv_gb300" / "csrc"
    shutil.copytree(bench.ROOT / "quant_dequant_gemv_gb300" / "csrc", csrc)
    (tmp_path / "profiles").mkdir()
    shutil.copy(bench.ROOT / "profiles" / "dram_traffic.json", tmp_path / "profiles" / "dram_traffic.json")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    # key the copied records to the copied sources, so that the tests below check
    # the hashing alone, whether or not the committed records are current
    rec = tmp_path / "profiles" / "dram_traffic.json"
    d = json.loads(rec.read_text())
    for e in d.values():
        e["source_hash"] = bench.kernel_source_hash(tuple(e.get("excluded_sources", ())))
    rec.write_text(json.dumps(d))
    return tmp_path


def test_committed_records_resolve():
    # A record taken on other kernel code reads as None (the bench then reports no
    # traffic); that is expected between a kernel change and the next capture.
    d = json.loads((bench.ROOT / "profiles" / "dram_traffic.json").read_text())
    assert "step/b1" in d
    stale = []
    for key, e in d.items():
        workload, b = key.split("/b")
        got = bench.recorded_traffic(workload, int(b))
        assert got in (None, e["bytes_per_launch"]), key
        if got is None:
            stale.append(key)
    if stale:
        pytest.skip(f"records taken on earlier kernel code: {stale}")


def test_hash_ignores_comments_and_blank_lines(fake_root):
    f = fake_root / "quant_dequant_gemv_gb300" / "csrc" / "qdq_stream1.cu"
    h0 = bench.kernel_source_hash()
    f.write_text("// a new comment line\n\n" + f.read_text().replace("{\n", "{  // trailing comment\n", 1))
    assert bench.kernel_source_hash() == h0
    assert bench.recorded_traffic("step", 1) is not None


def test_code_change_voids_the_records(fake_root):
    f = fake_root / "quant_dequant_gemv_gb300" / "csrc" / "qdq_stream1.cu"
    f.write_text(f.read_text() + "\nstatic int changed_code_line = 1;\n")
    assert bench.recorded_traffic("step", 1) is None


def test_excluded_source_does_not_void_the_records(fake_root):
    d = json.loads((fake_root / "profiles" / "dram_traffic.json").read_text())
    assert "qdq_mma.cu" in d["step/b1"]["excluded_sources"]
    f = fake_root / "quant_dequant_gemv_gb300" / "csrc" / "qdq_mma.cu"
    f.write_text(f.read_text() + "\nstatic int changed_code_line = 1;\n")
    assert bench.recorded_traffic("step", 1) == d["step/b1"]["bytes_per_launch"]


def test_missing_record_is_none(fake_root):
    assert bench.recorded_traffic("step", 7) is None
    assert bench.recorded_traffic("no_such_workload", 1) is None
