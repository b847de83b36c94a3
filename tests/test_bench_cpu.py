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


def test_write_traffic_records_bytes_per_word_of_one_launch_each(tmp_path, monkeypatch):
    pytest.importorskip("torch")
    import math

    import workloads
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    words = sum(math.prod(s.shape) for s in workloads.googlenet_specs(16))
    assert words == 3_020_193_792 // 16  # batch 16 is 1/16 of the batch-256 workload
    c = _csv(tmp_path / "c.csv", [("3", "1", "Gbyte")])
    d = _csv(tmp_path / "d.csv", [("1", "3", "Gbyte")])
    assert bench.write_traffic([c, d], 4096, 16) == 0
    rec = json.loads((tmp_path / "traffic.json").read_text())
    assert rec["words_per_launch"] == words
    for k in ("compress_kernel", "decompress_kernel"):
        assert rec["kernels"][k]["dram_bytes"] == pytest.approx(4e9)
        assert rec["kernels"][k]["dram_bytes_per_word"] == pytest.approx(4e9 / words)
        assert rec["kernels"][k]["gpu_time_us"] == pytest.approx(12.5)
        assert rec["kernels"][k]["source_sha256"] == bench.kernel_source_hash(k)
    # scaled to a full-size launch by its words
    assert bench.traffic_per_launch("compress_kernel", 16 * words) == pytest.approx(64e9)
    two = _csv(tmp_path / "two.csv", [("1", "1", "Mbyte")] * 2)
    with pytest.raises(SystemExit):
        bench.write_traffic([c, two], 4096, 16)


def test_host_cpu_reports_cores_and_a_model():
    cores, model = bench.host_cpu()
    assert cores >= 1 and isinstance(model, str) and model


def test_clock_sampler_falls_back_without_nvml():
    # no NVIDIA driver here: the NVML sampler is unavailable and nvidia-smi takes over
    s = bench.clock_sampler(None)
    assert isinstance(s, (bench.NvmlSampler, bench.ClockSampler))
    if isinstance(s, bench.NvmlSampler):
        assert s.available()
