"""Host logic of bench.py that needs no GPU: the attention traffic record
(parsed from an ncu --csv metrics log, tied to a digest of the attention
source, reported as stale once that source changes)."""
import json

import pytest

import bench

CSV = '''"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void sp::exchange_kernel<16, false>(sp::ExchangeParams, int, int)","1","7","(256, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","402653184"
"1","1","python","h","void sp::tc::attn_tc_kernel<128, false>(sp::tc::TcParams)","1","7","(320, 1, 1)","(6176, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","1.45"
"1","1","python","h","void sp::tc::attn_tc_kernel<128, false>(sp::tc::TcParams)","1","7","(320, 1, 1)","(6176, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","426.97"
"1","1","python","h","void sp::tc::attn_tc_kernel<128, false>(sp::tc::TcParams)","1","7","(320, 1, 1)","(6176, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","msecond","28.92"
'''


@pytest.fixture
def record_file(tmp_path, monkeypatch):
    path = tmp_path / "attention_dram.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    return path


def test_record_and_read_traffic(tmp_path, record_file):
    log = tmp_path / "ncu.csv"
    log.write_text("==PROF== Connected\n" + CSV)
    rec = bench.record_traffic(str(log), "c5", "ncu --metrics ... python bench.py")
    assert rec["launches"] == 1
    assert rec["dram_read_bytes"] == 1_450_000_000 and rec["dram_write_bytes"] == 426_970_000
    assert bench.attention_traffic("c5") == (1_876_970_000, f"ncu, attention source {rec['source_digest']}")
    assert bench.attention_traffic("c3")[0] is None


def test_stale_record_gives_no_traffic(record_file):
    record_file.write_text(json.dumps({"c5": {"dram_bytes_per_launch": 5, "source_digest": "0" * 16}}))
    value, why = bench.attention_traffic("c5")
    assert value is None and "stale" in why


def test_missing_record_gives_no_traffic(record_file):
    assert bench.attention_traffic("c5") == (None, "no ncu record")


def test_bench_reads_no_markdown():
    src = open(bench.__file__).read()
    assert ".md" not in src
