"""Host logic of the benchmark, on the CPU: a step whose decode kernel reported a non-zero device
status word refuses its line, the DRAM-traffic record is used only for the kernel sources it was
taken on, and the clock samples are summarised with every throttle reason that was active."""
import pytest
import torch

import bench


def _problem_with_status(word: int):
    pb = bench.Problem.__new__(bench.Problem)        # no device: only the workspace and the plan
    pb.ws = torch.zeros(64, dtype=torch.uint8)
    pb.ws[16:20] = torch.tensor([word], dtype=torch.int32).view(torch.uint8)
    pb.plan = type("Plan", (), {"status_offset": 16})()
    return pb


def test_nonzero_status_word_refuses_the_line(monkeypatch):
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    ok = _problem_with_status(0)
    assert ok.status() == 0
    ok.check("clean step")
    bad = _problem_with_status(0x12)
    assert bad.status() == 0x12
    with pytest.raises(RuntimeError, match="status 0x12"):
        bad.check("step whose pipeline wait expired")


def test_traffic_record_only_for_matching_sources(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# workload  digest  bytes\nwl_a 1111aaaa 123\nwl_a 2222bbbb 456\nwl_b 2222bbbb 789\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda tu="decode_tc.cu": "2222bbbb")
    assert bench.profiled_traffic("wl_a") == 456.0
    assert bench.profiled_traffic("wl_b") == 789.0
    assert bench.profiled_traffic("wl_c") is None
    monkeypatch.setattr(bench, "kernel_source_digest", lambda tu="decode_tc.cu": "3333cccc")
    assert bench.profiled_traffic("wl_a") is None


def test_source_digest_follows_the_kernel_and_headers_only(monkeypatch, tmp_path):
    csrc = tmp_path / "quantized_kv_paged_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in (("decode_tc.cu", "kernel"), ("common.cuh", "helpers"), ("api.h", "decls"),
                       ("other.cu", "another kernel")):
        (csrc / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_source_digest()
    (csrc / "other.cu").write_text("another kernel, changed")
    assert bench.kernel_source_digest() == d0
    (csrc / "common.cuh").write_text("helpers, changed")
    d1 = bench.kernel_source_digest()
    assert d1 != d0
    (csrc / "decode_tc.cu").write_text("kernel, changed")
    assert bench.kernel_source_digest() != d1
    assert bench.kernel_source_digest("other.cu") != bench.kernel_source_digest()
    assert len(d0) == 16 and all(ch in "0123456789abcdef" for ch in d0)


def test_clock_summary_reports_median_and_active_reasons():
    c = bench.ClockSampler(0)
    c.lines = [
        "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1400.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1001.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "[N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "truncated line",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = ["1500, 2070, 800.0, 0x8, Not Active, Active, Not Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_thermal_slowdown"]
    c.lines = []
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
