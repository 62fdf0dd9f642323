"""The plan queries on the GPU: the device's limits are the ones the GEMM
plans with, and the planned workspace is exactly what a GEMM needs.

The planner's decisions themselves are checked on CPU (test_planner_cpu.py);
here petit_device_limits() is tied to the device and the plan to real
launches: one byte less than the planned workspace is refused before
anything is enqueued, the planned size runs and matches the oracle.
"""

import ctypes

import pytest
import torch

from fp4_weight_only_gb300 import synth
from tests.gpu_util import assert_parity, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu

ERR_WORKSPACE = 4


def test_device_limits(cuda_lib):
    sms, pairs = cuda_lib.device_limits()
    assert sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert 1 <= pairs <= sms // 2


@pytest.mark.parametrize("m,n,k,fmt", [(16, 10240, 8192, "nvfp4"), (128, 8192, 8192, "nvfp4"),
                                       (256, 57344, 8192, "mxfp4"), (70, 1024, 1152, "nvfp4_f16"),
                                       (512, 8192, 28672, "mxfp4")])
def test_planned_workspace_is_the_gemm_workspace(cuda_lib, m, n, k, fmt):
    p = cuda_lib.plan(m, n, k, fmt)
    assert p["workspace_bytes"] == cuda_lib.workspace_bytes(m, n, k, fmt)
    sms, pairs = cuda_lib.device_limits()
    assert cuda_lib.plan(m, n, k, fmt, sms, pairs) == p


@pytest.mark.parametrize("m,pair_mode", [(100, 0), (200, 2)])
def test_gemm_runs_in_exactly_the_planned_workspace(cuda_lib, m, pair_mode):
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=91 + m)
    codes, scales = oracle_quantize(w, "mxfp4")
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "mxfp4")
    a = synth.activations(m, k, seed=92).cuda()
    L = cuda_lib.load()
    cuda_lib.set_pair_mode(pair_mode)
    try:
        p = cuda_lib.plan(m, n, k, "mxfp4")
        need = p["workspace_bytes"]
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

        def call(nbytes):
            return L.petit_gemm_bf16_mxfp4(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(rep.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), m, n, k,
                                           ctypes.c_void_p(ws.data_ptr()), nbytes, stream)
        assert call(need - 1) == ERR_WORKSPACE
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all(), "a refused call enqueued work"
        assert call(need) == 0
        torch.cuda.synchronize()
    finally:
        cuda_lib.set_pair_mode(0)
    assert_parity(out, oracle_reference(a.cpu(), codes, scales, "mxfp4"), f"m={m} pairs={pair_mode}")


def test_tuner_times_every_tile_shape(cuda_lib):
    from fp4_weight_only_gb300 import tune
    m, n, k = 40, 1024, 1024
    rows, planned, planned_us = tune.tune(m, n, k, "nvfp4", iters=8)
    want = {(bn, ku, mode) for bn, ku in tune.candidates(k)
            for mode in ((1, 2) if bn >= 128 else (1,))}
    assert {(r["bn"], r["ku"], r["pair_mode"]) for r in rows} == want
    assert all(r["us"] > 0 for r in rows) and planned_us > 0
    assert [r["us"] for r in rows] == sorted(r["us"] for r in rows)
    assert planned == cuda_lib.plan(m, n, k, "nvfp4")   # settings restored
