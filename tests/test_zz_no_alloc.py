"""The NVFP4 GEMM entry point that allocates nothing (built-in scratch array).

Some callers cannot allocate device memory when they call the GEMM: plug-ins
whose host framework owns all device memory and forbids allocation inside
their enqueue call, and latency-critical serving loops that cannot afford
cudaMalloc's implicit device synchronisation.  They use
petit_gemm_bf16_nvfp4_noalloc, whose split-K scratch is a fixed array in the
library's device image.

Its results are checked against the FP64 oracle and against the workspace
entry point, on two calls in a row (the second call must not be disturbed by
what the first left in the shared array).  This file is collected last, so a
failure here does not hide the results of the other tests; it also passes
when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from tests.gpu_util import assert_parity, compare, oracle_quantize, oracle_reference, to_device_packed, MAX_ABS_REL, REL_L2

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_oracle_and_workspace_entry_point(cuda_lib):
    L = cuda_lib.load()
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=31)
    codes, scales = oracle_quantize(w, "nvfp4", 1.0)
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    # two calls in a row with different m (different tile heights and
    # split-K layouts in the shared scratch)
    for m in (16, 5):
        a = synth.activations(m, k, seed=40 + m)
        a_dev = a.cuda()
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.petit_gemm_bf16_nvfp4_noalloc(_p(a_dev), _p(rep), ctypes.c_float(1.0), _p(out),
                                             m, n, k, _stream())
        assert st == 0, cuda_lib.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert_parity(out, oracle_reference(a, codes, scales, "nvfp4"), f"noalloc m={m}")
        # and against the entry point with a caller workspace
        ref_ws = cuda_lib.gemm(a_dev, rep, n, "nvfp4", 1.0)
        torch.cuda.synchronize()
        mx, l2 = compare(out, ref_ws.float().cpu().numpy().astype(np.float64))
        assert mx <= MAX_ABS_REL and l2 <= REL_L2, (m, mx, l2)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    L = cuda_lib.load()
    n, k, m = 1024, 1024, 256
    a = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    rep = torch.zeros(n * k // 2 + n * k // 16, dtype=torch.uint8, device="cuda")
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    st = L.petit_gemm_bf16_nvfp4_noalloc(_p(a), _p(rep), ctypes.c_float(1.0), _p(c), m, n, k,
                                         _stream())
    assert st == 4   # PETIT_ERR_WORKSPACE: needs more than the built-in scratch
