"""bench.py's clock sampler on CPU, against a stand-in nvidia-smi that prints
one CSV sample every 50 ms: the sampler is live before the timed region,
keeps only the samples taken inside it, falls back to the first sample after
a region shorter than the period (and says so), parses the throttle reasons,
and reports "unsampled" when no nvidia-smi exists."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

FAKE = """#!{py}
import sys, time
n = 0
while True:
    n += 1
    mhz = 1800 if n % 2 else 2000
    cap = "Active" if n % 3 == 0 else "Not Active"
    print(f"0, 00000000:1B:00.0, {{mhz}}, 2070, 700.5, 0x4, Not Active, Not Active, Not Active, {{cap}}",
          flush=True)
    time.sleep(0.05)
"""


def fake_smi(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE.format(py=sys.executable))
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")


def test_samples_inside_the_region(tmp_path, monkeypatch):
    fake_smi(tmp_path, monkeypatch)
    with bench.ClockSampler(bus_id="00000000:1B:00.0", period_ms=50) as clk:
        assert clk.lines, "the sampler is live before the region starts"
        time.sleep(0.2)                    # samples before the region are not counted
        clk.region_start()
        time.sleep(0.6)
        clk.region_end()
        time.sleep(0.2)                    # nor those after it
    s = clk.summary()
    assert s["sampled"] == "timed region"
    assert 6 <= s["samples"] <= 16
    assert s["sm_max_mhz"] == 2070.0 and s["sm_mhz"] in (1800.0, 1900.0, 2000.0)
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 700.5


def test_short_region_takes_the_next_sample(tmp_path, monkeypatch):
    fake_smi(tmp_path, monkeypatch)
    with bench.ClockSampler(period_ms=50) as clk:
        time.sleep(0.12)
        clk.region_start()
        clk.region_end()                   # far shorter than the period
    s = clk.summary()
    assert s["samples"] == 1
    assert s["sampled"].startswith("first sample after")


def test_other_gpus_are_filtered(tmp_path, monkeypatch):
    fake_smi(tmp_path, monkeypatch)
    with bench.ClockSampler(bus_id="00000000:99:00.0", period_ms=50) as clk:
        clk.region_start()
        time.sleep(0.2)
        clk.region_end()
    assert clk.summary()["reasons"] == ["unsampled"]


def test_no_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler() as clk:
        clk.region_start()
        clk.region_end()
    assert clk.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
