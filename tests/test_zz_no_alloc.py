"""The GEMM entry point that allocates nothing (built-in scratch array).

Callers that cannot allocate device memory when they call the GEMM -- code
running during CUDA graph capture, plug-ins whose framework owns device
memory, serving loops that cannot afford cudaMalloc's implicit
synchronisation -- use petit_gemm_bf16_nvfp4_noalloc.  This file is collected
last, so a failure here does not hide the results of the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from tests.gpu_util import MAX_ABS_REL, REL_L2, compare

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point(cuda_lib):
    L = cuda_lib.load()
    n, k = 1024, 2048
    fw = cuda_lib.FP4Weight(synth.weights(n, k, seed=31, device="cuda"), "nvfp4", 1.0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row: the second must not be disturbed by the first
    # call's leftovers in the shared scratch array
    for m in (16, 5):
        a = synth.activations(m, k, seed=40 + m, device="cuda")
        ref = cuda_lib.gemm(a, fw.rep, n, "nvfp4", 1.0)
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.petit_gemm_bf16_nvfp4_noalloc(_p(a), _p(fw.rep), ctypes.c_float(1.0), _p(out),
                                             m, n, k, stream)
        assert st == 0, cuda_lib.STATUS.get(st, st)
        torch.cuda.synchronize()
        mx, l2 = compare(out, ref.float().cpu().numpy().astype(np.float64))
        assert mx <= MAX_ABS_REL and l2 <= REL_L2, (m, mx, l2)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    L = cuda_lib.load()
    n, k, m = 1024, 1024, 256
    a = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    rep = torch.zeros(n * k // 2 + n * k // 16, dtype=torch.uint8, device="cuda")
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    st = L.petit_gemm_bf16_nvfp4_noalloc(_p(a), _p(rep), ctypes.c_float(1.0), _p(c), m, n, k,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4   # PETIT_ERR_WORKSPACE: needs more than the built-in scratch
