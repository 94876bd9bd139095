"""Host logic of bench.py that needs no GPU: the roofline denominator
follows the regime the timed region ran in, and the script refuses to run as
several ranks or on several GPUs (the library is for single-GPU processes)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"bf16_tflops": 1925.7, "bf16_tflops_sustained": 1709.8, "hbm_gbs": 6784.2}


def test_short_region_without_power_cap_is_burst():
    # 20 launches of 0.5718 ms: 11.4 ms, no throttle reason in the samples
    assert bench.timing_regime(11.4, {"reasons": []}) == "burst"
    r = bench.tensor_roofline(1922.9, "burst", PEAKS)
    assert r["peak"] == 1925.7 and r["frac"] == pytest.approx(0.9985, abs=1e-4)
    assert r["frac_sustained"] == pytest.approx(1922.9 / 1709.8)
    assert r["regime"] == "burst" and "burst" in r["peak_source"]


def test_power_cap_or_long_region_is_sustained():
    assert bench.timing_regime(300.0, {"reasons": ["sw_power_cap"]}) == "sustained"
    assert bench.timing_regime(1500.0, {"reasons": []}) == "sustained"
    assert bench.timing_regime(1500.0, None) == "sustained"
    r = bench.tensor_roofline(1710.0, "sustained", PEAKS)
    assert r["peak"] == 1709.8 and r["frac_burst"] == pytest.approx(1710.0 / 1925.7)


def test_fallback_peaks_without_measured_file():
    assert bench.tensor_roofline(1000.0, "burst", None)["peak"] == bench.FALLBACK_BURST_TFLOPS
    r = bench.tensor_roofline(1000.0, "sustained", None)
    assert r["peak"] == bench.FALLBACK_SUSTAINED_TFLOPS and r["peak_source"].startswith("of fallback")


def test_throughput():
    assert bench.throughput(4.0, 2e12, 3) == pytest.approx(2e12 * 3 / 4e-3 / 1e12)


@pytest.mark.parametrize("env,args", [({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}, []),
                                      ({}, ["--gpus", "2"])])
def test_refuses_several_ranks_or_gpus(env, args):
    e = dict(os.environ)
    e.update(env)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3"] + args,
                       env=e, capture_output=True, text=True, timeout=300)
    assert r.returncode == 2
    assert "single-GPU" in r.stderr
    assert r.stdout == ""
