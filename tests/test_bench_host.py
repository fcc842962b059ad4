"""bench.py host logic without a GPU: the clock sampler's window selection and parsing, with
fake samples, fake nvidia-smi output and a fake NVML poller (nothing here queries a device)."""
import io
import os
import sys
import threading
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_summary_uses_the_samples_inside_the_window():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, 1500.0, 2032.0, []), (2.0, 2032.0, 2032.0, []),
                 (2.5, 2000.0, 2032.0, ["sw_power_cap"]), (3.0, 2032.0, 2032.0, []),
                 (9.0, 800.0, 2032.0, ["hw_slowdown"])]
    s = c.summary(1.9, 3.1)
    assert s["samples"] == 3 and s["sampled"] == "timed window"
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]  # the slowdown outside the window is not counted


def test_summary_falls_back_to_the_nearest_samples():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, 2032.0, 2032.0, []), (5.0, 1000.0, 2032.0, ["hw_thermal_slowdown"]),
                 (2.2, 2010.0, 2032.0, [])]
    s = c.summary(2.0, 2.1)  # no sample inside a 0.1 s window
    assert s["samples"] == 3 and s["sampled"].startswith("nearest")
    assert c.summary(0.0, 1.0)["samples"] == 1
    assert bench.ClockSampler(0).summary(0.0, 1.0)["reasons"] == ["unsampled"]


def test_nvidia_smi_lines_are_parsed():
    c = bench.ClockSampler(0)

    class P:
        stdout = io.StringIO(
            "2032, 2032, 700.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "1800, 2032, 1100.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "[N/A], 2032, 0, 0, Not Active, Not Active, Not Active, Not Active\n"
            "short line\n")
    c.proc = P()
    c._read()
    assert [(s[1], s[2], s[3]) for s in c.samples] == [(2032.0, 2032.0, []),
                                                      (1800.0, 2032.0, ["sw_power_cap"])]


def test_nvml_reason_bits():
    c = bench.ClockSampler(0)
    bits = iter([0x0, 0x4, 0x8 | 0x40, 0x20])
    state = {"n": 0}

    def sm():
        state["n"] += 1
        if state["n"] > 4:
            raise OSError("done")  # ends the poller
        return 2032.0

    c.nvml = (sm, 2032.0, lambda: next(bits))
    c.running = True
    t = threading.Thread(target=c._poll_nvml)
    t.start()
    t.join(timeout=5)
    assert [s[3] for s in c.samples] == [[], ["sw_power_cap"],
                                         ["hw_slowdown", "hw_thermal_slowdown"],
                                         ["sw_thermal_slowdown"]]
    assert c.summary(0.0, time.time() + 1)["source"] == "nvml"


def test_visible_device_index_maps_to_the_nvml_index():
    c = bench.ClockSampler(1)
    old = os.environ.get("CUDA_VISIBLE_DEVICES")
    try:
        os.environ["CUDA_VISIBLE_DEVICES"] = "3,5"
        assert c._nvml_index() == 5
        os.environ["CUDA_VISIBLE_DEVICES"] = ""
        assert c._nvml_index() == 1
    finally:
        if old is None:
            os.environ.pop("CUDA_VISIBLE_DEVICES", None)
        else:
            os.environ["CUDA_VISIBLE_DEVICES"] = old
