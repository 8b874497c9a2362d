"""Host-side pieces of bench.py that need no GPU: the DRAM-traffic record
looked up from the committed ncu summaries (null once the kernel source has
changed or for another workload), and the parsing of the clock samples taken
during a timed region (median SM clock, throttle reasons, samples outside
the region ignored)."""
import hashlib
import json
import os
import time

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_matches_the_committed_capture():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    assert records, "no traffic records committed"
    for kernel, rec in records.items():
        src = os.path.join(ROOT, rec["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        assert h == rec["source_sha256_16"], f"{kernel}: capture predates the current {rec['source']}"
        got = bench.traffic_record(kernel, rec["workload"])
        assert got == float(rec["bytes_per_launch"])
        assert bench.traffic_record(kernel, rec["workload"] + " (another workload)") is None
    assert bench.traffic_record("no_such_kernel", "any") is None


def test_traffic_record_is_null_for_a_changed_source(tmp_path, monkeypatch):
    # a copy of the repository's record pointing at a source whose bytes differ
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "k.cu"
    src.write_text("// one version\n")
    rec = {"fa_x_kernel": {"bytes_per_launch": 123.0, "source": "k.cu",
                           "source_sha256_16": hashlib.sha256(b"// one version\n").hexdigest()[:16],
                           "workload": "w"}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("fa_x_kernel", "w") == 123.0
    src.write_text("// another version\n")
    assert bench.traffic_record("fa_x_kernel", "w") is None


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


class _FakeThread:
    def join(self, timeout=None):
        pass


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    s.proc, s.t, s.lines = _FakeProc(), _FakeThread(), lines
    return s


def test_clock_samples_inside_the_region_only():
    t0 = time.time()
    row = "0, {mhz}, 2070, {w}, 0x0, Not Active, Not Active, Not Active, {cap}"
    lines = [
        (t0 - 1.0, row.format(mhz=1200, w=100, cap="Not Active")),   # before the region
        (t0 + 0.05, row.format(mhz=2070, w=900, cap="Not Active")),
        (t0 + 0.10, row.format(mhz=2040, w=1300, cap="Active")),
        (t0 + 0.15, row.format(mhz=2070, w=1000, cap="Not Active")),
        (t0 + 5.0, row.format(mhz=900, w=100, cap="Not Active")),     # well after it
        (t0 + 0.12, "garbled line"),
    ]
    got = _sampler_with(lines).stop(t0, t0 + 0.2)
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070.0
    assert got["sm_max_mhz"] == 2070.0
    assert got["power_w_max"] == 1300.0
    assert got["reasons"] == ["sw_power_cap"]


def test_clock_reasons_that_reject_a_run_are_reported():
    t0 = time.time()
    lines = [(t0 + 0.01, "0, 1500, 2070, 700, 0x8, Not Active, Active, Not Active, Not Active")]
    got = _sampler_with(lines).stop(t0, t0 + 0.1)
    assert got["reasons"] == ["hw_thermal_slowdown"]
    assert got["sm_mhz"] == 1500.0


def test_clock_sampler_without_nvidia_smi():
    got = bench.ClockSampler(0).stop(0.0, 1.0)   # never started
    assert got["samples"] == 0 and got["sm_mhz"] is None
