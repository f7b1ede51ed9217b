"""Host logic of bench.py that decides what the JSON line reports (no GPU).

- roofline.traffic comes from profiles/dram_traffic.txt only while the
  kernel source still has the digest the counters were taken on;
- the peaks come from MEASURED_PEAKS.json, with a labelled fallback;
- every line of the committed traffic file names a kernel, workload and
  source that bench.py actually looks up.
"""
import hashlib
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lookups():
    """(kernel, source, workload) triples bench.py passes to profiled_traffic."""
    text = open(os.path.join(ROOT, "bench.py")).read()
    calls = re.findall(r'profiled_traffic\(\s*"([^"]+)",\s*([^,]+),\s*"([^"]+)"\)', text)
    out = []
    for kernel, src, workload in calls:
        src = src.strip()
        if src.startswith('"'):
            src = src.strip('"')
        else:   # a variable: its string literal is assigned above the call
            m = re.search(rf'{re.escape(src)}\s*=\s*"([^"]+)"', text)
            assert m, f"cannot resolve the source of {kernel}"
            src = m.group(1)
        out.append((kernel, src, workload))
    return out


def test_traffic_needs_the_current_digest(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel source v1\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:12]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment\n"
        f"my_kernel wl {digest} 1234\n"
        f"my_kernel other_wl {digest} 99\n"
        "other_kernel wl 000000000000 5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_digest("k.cu") == digest
    assert bench.profiled_traffic("my_kernel", "k.cu", "wl") == 1234.0
    assert bench.profiled_traffic("my_kernel", "k.cu", "other_wl") == 99.0
    assert bench.profiled_traffic("my_kernel", "k.cu", "missing") is None
    src.write_text("kernel source v2\n")   # the kernel changed since the capture
    assert bench.profiled_traffic("my_kernel", "k.cu", "wl") is None


def test_traffic_without_a_file_is_null(tmp_path, monkeypatch):
    (tmp_path / "k.cu").write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("my_kernel", "k.cu", "wl") is None


def test_peaks_measured_or_labelled_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    hbm, bf16, src = bench.measured_peaks()
    assert src == "fallback" and hbm == 6800.0 and bf16 == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6787.6,
                                                               "bf16_tflops": 1907.2}))
    hbm, bf16, src = bench.measured_peaks()
    assert src == "measured" and hbm == 6787.6 and bf16 == 1907.2


def test_committed_traffic_lines_are_looked_up():
    lookups = _lookups()
    assert {k for k, _, _ in lookups} >= {"kda_prefill_tc_kernel", "kda_decode_kernel",
                                           "kda_qkv_prologue_kernel"}
    known = {(k, w): s for k, s, w in lookups}
    for line in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        kernel, workload, digest, nbytes = line.split()
        assert (kernel, workload) in known, f"bench.py never reads {kernel} {workload}"
        assert re.fullmatch(r"[0-9a-f]{12}", digest)
        assert float(nbytes) > 0
        assert os.path.exists(os.path.join(ROOT, known[(kernel, workload)]))


def test_clock_summary_inside_nearest_and_reasons():
    """Clock samples inside the timed region are summarised (median SM clock,
    max clock, active throttle reasons); a region shorter than the sampling
    period falls back to the nearest sample and says so."""
    s = bench.ClockSampler(0)

    def row(mhz, *active):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        return ["0", str(mhz), "2070", "900.0", "0x0"] + ["Active" if n in active else "Not Active" for n in names]
    s.samples = [(10.00, row(2070)), (10.02, row(1950, "sw_power_cap")), (10.04, row(2070)),
                 (10.50, row(1500, "hw_slowdown"))]
    out = s.summary(9.99, 10.05)
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and "note" not in out
    near = s.summary(10.45, 10.46)
    assert near["samples"] == 1 and near["sm_mhz"] == 1500.0 and near["reasons"] == ["hw_slowdown"]
    assert "nearest" in near["note"]
    assert bench.ClockSampler(0).summary(0, 1)["reasons"] == ["unavailable"]
