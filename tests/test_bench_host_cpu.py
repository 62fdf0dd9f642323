"""bench.py's host-side arithmetic and evidence handling, on CPU: the
algorithmic bytes behind `value` and `roofline.achieved`, the number of
weight copies rotated so every launch reads HBM, the DRAM traffic taken
from a committed ncu summary only while the kernel source is unchanged, the
clock summary of the timed region, and the peak table."""

import importlib.util
import json
import math
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes(bench):
    # O projection at m = 16: n*k/2 code bytes, n*k/16 E4M3 scales, A and C in BF16
    n = k = 8192
    assert bench.algo_bytes(16, n, k) == 33554432 + 4194304 + 262144 + 262144
    # MXFP4: one E8M0 scale per 32
    assert bench.algo_bytes(16, n, k, 32) == 33554432 + 2097152 + 262144 + 262144
    # the m = 16 decode step (four Llama-3-70B linears): 485.7 MB, so a
    # 106.86 us step moves 4.545 TB/s
    shapes = [(10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)]
    step = sum(bench.algo_bytes(16, n, k) for n, k in shapes)
    assert step == 485_687_296
    assert step / 106.86e-6 / 1e9 == pytest.approx(4545.0, rel=1e-3)


def test_weight_rotation_outruns_l2(bench):
    l2 = 126 * 2**20
    # R = max(2, ceil(3 L2 / W)): the copies a launch cycles through hold
    # at least three L2s, so no launch finds its weights in L2
    for wbytes in (37_748_736, 47_185_920, 264_241_152, 132_120_576, 1 << 20):
        r = bench.rotation_copies(wbytes, l2)
        assert r == max(2, math.ceil(3 * l2 / wbytes))
        assert r * wbytes >= 3 * l2 or r == 2
    assert bench.rotation_copies(37_748_736, l2) == 11     # O: the bench's 11 copies
    assert bench.rotation_copies(264_241_152, l2) == 2     # gate_up


def test_ncu_traffic_only_for_the_profiled_source(bench, tmp_path, monkeypatch):
    # the committed decode summary gives its traffic while it pins the
    # current kernel source, else nothing
    import hashlib
    summary = open(os.path.join(ROOT, "profiles", "gemm_nvfp4_decode_m16.txt")).read()
    digest = hashlib.sha256(open(os.path.join(ROOT, "fp4_weight_only_gb300", "csrc", "gemm.cu"),
                                 "rb").read()).hexdigest()[:16]
    pinned = f"gemm.cu sha256 prefix: {digest}" in summary
    assert bench.ncu_traffic("gemm_nvfp4_decode_m16.txt") == (122099201.0 if pinned else None)
    assert bench.ncu_traffic("no_such_summary.txt") is None
    # a copy of the tree whose kernel source differs by one byte: no traffic
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "fp4_weight_only_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, "profiles", "gemm_nvfp4_decode_m16.txt"), tmp_path / "profiles")
    src = open(os.path.join(ROOT, "fp4_weight_only_gb300", "csrc", "gemm.cu"), "rb").read()
    (csrc / "gemm.cu").write_bytes(src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("gemm_nvfp4_decode_m16.txt") == (122099201.0 if pinned else None)
    (csrc / "gemm.cu").write_bytes(src + b"\n")
    assert bench.ncu_traffic("gemm_nvfp4_decode_m16.txt") is None


def _sampler(bench, rows):
    s = object.__new__(bench.ClockSampler)
    import threading
    s.lock = threading.Lock()
    s.rows = rows
    return s


def test_clock_summary_takes_the_timed_region(bench):
    idle = ["Not Active"] * 5
    cap = ["Active", "Not Active", "Not Active", "Not Active", "Active"]
    rows = [(0.0, 1000.0, 2070.0, idle),           # before the timed region
            (10.0, 2070.0, 2070.0, idle),
            (10.2, 2055.0, 2070.0, cap),
            (10.4, 2070.0, 2070.0, idle),
            (30.0, 900.0, 2070.0, idle)]           # after it
    s = _sampler(bench, rows)
    out = s.summary([(10.0, 10.5)])
    assert out["samples_in_timed_region"] == 3 and out["samples"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    # no sample inside a window: every sample is summarised, and said so
    out = s.summary([(50.0, 51.0)])
    assert out["samples_in_timed_region"] == 0 and out["samples"] == 5
    hot = ["Active", "Not Active", "Active", "Not Active", "Not Active"]
    out = _sampler(bench, [(1.0, 1500.0, 2070.0, hot)]).summary([(0.0, 2.0)])
    assert out["reasons"] == ["hw_thermal_slowdown"]
    empty = _sampler(bench, []).summary([(0.0, 1.0)])
    assert empty["sm_mhz"] is None and empty["samples"] == 0


def test_peaks_measured_or_fallback(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["source"] == "fallback" and fb["hbm_gbs"] == 6800.0 and fb["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6791.4, "bf16_tflops": 1869.0}))
    m = bench.load_peaks()
    assert m["source"] == "measured" and m["hbm_gbs"] == 6791.4
    assert m["bf16_tflops_sustained"] == 1869.0     # burst figure when no sustained one is given
