"""Host logic of bench.py that needs no GPU: reading ncu's per-launch DRAM counters, the
DRAM traffic record keyed by the kernel sources, and the launches one bench step makes."""
import json

import pytest

import bench

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
          '"Metric Value"')


def _csv(path, launches):
    """An ncu --csv log: its banner lines, then one row per (launch, metric)."""
    lines = ["==PROF== Connected to process 1 (/usr/bin/python3)", HEADER]
    for i, (rd, wr, unit) in enumerate(launches):
        for name, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr),
                        ("gpu__time_duration.sum", "12.5")):
            u = "usecond" if name.startswith("gpu__") else unit
            lines.append(f'"{i}","1","python3","h","k","1","7","(64, 1, 1)","(9, 1, 1)","0",'
                         f'"10.3","Command line profiler metrics","{name}","{u}","{v}"')
    path.write_text("\n".join(lines) + "\n")
    return str(path)


def test_ncu_dram_bytes_sums_read_and_write_per_launch(tmp_path):
    p = _csv(tmp_path / "a.csv", [("5,153,792", "1000", "byte"), ("2.5", "0.5", "Mbyte"),
                                  ("3", "1", "Kbyte")])
    assert bench.ncu_dram_bytes(p) == pytest.approx([5_154_792, 3_000_000, 4_000])


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.traffic_per_launch("decompress_kernel", 1e6) is None  # no record
    good = {"source_sha256": bench.kernel_source_hash("decompress_kernel"),
            "dram_bytes_per_word": 2.5}
    rec.write_text(json.dumps({"kernels": {"decompress_kernel": good}}))
    assert bench.traffic_per_launch("decompress_kernel", 1e6) == pytest.approx(2.5e6)
    assert bench.traffic_per_launch("compress_kernel", 1e6) is None  # no entry
    stale = dict(good, source_sha256="0" * 64)
    rec.write_text(json.dumps({"kernels": {"decompress_kernel": stale}}))
    assert bench.traffic_per_launch("decompress_kernel", 1e6) is None


def test_write_traffic_checks_the_launch_count(tmp_path, monkeypatch):
    pytest.importorskip("torch")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    L = bench.launches_per_step(4096)
    assert L == 6  # AlexNet layer 0 takes two 32 Mi-word segments, the others one each
    ok = [("1", "1", "Mbyte")] * L
    c = _csv(tmp_path / "c.csv", ok)
    d = _csv(tmp_path / "d.csv", ok)
    assert bench.write_traffic([c, d], 4096) == 0
    rec = json.loads((tmp_path / "traffic.json").read_text())
    for k in ("compress_kernel", "decompress_kernel"):
        assert rec["kernels"][k]["launches"] == L
        assert rec["kernels"][k]["dram_bytes"] == pytest.approx(2e6 * L)
        assert rec["kernels"][k]["source_sha256"] == bench.kernel_source_hash(k)
    short = _csv(tmp_path / "s.csv", ok[:-1])
    with pytest.raises(SystemExit):
        bench.write_traffic([c, short], 4096)
