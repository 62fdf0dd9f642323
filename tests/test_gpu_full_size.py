"""Full-size parity, in the launch configuration bench.py times.

Each workload the method is measured on runs at its full size through the
same binding call as the bench; the oracle checks sampled output columns
(every weight row it needs is quantised by the oracle itself: quantisation
is row-local, so the sampled rows' codes do not depend on the other rows):

* NVFP4 decode, m = 16, the four Llama-3-70B linears (g = 1);
* MXFP4 decode, m in {1, 4, 8, 16}, and MXFP4 at m = 256, same shapes;
* NVFP4 prefill, m = 256, activations with 0.1 % N(0, 20) outliers and the
  per-tensor global scale g = amax / (6 * 448);
* NVFP4 m sweep 1 .. 1024 at n = k = 8192, and m = n = k = 4096.
"""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import quantize
from tests.gpu_util import assert_parity, oracle_quantize, oracle_reference

pytestmark = pytest.mark.gpu

SHAPES = list(synth.LLAMA3_70B_SHAPES.items())


def _sample_rows(n, count=48):
    """Rows spread over all 128-row tiles, including the first and last rows."""
    rows = np.unique(np.concatenate([np.linspace(0, n - 1, count).astype(np.int64), [0, 127, n - 128, n - 1]]))
    return rows


def _prepare(cuda_lib, n, k, fmt, seed, g=1.0):
    w = synth.weights(n, k, seed=seed, device="cuda")
    wp, sp = cuda_lib.quantize(w, fmt, g)
    rep = cuda_lib.repack(wp, sp, fmt)
    del wp, sp
    return w, rep


def _check(cuda_lib, w, rep, a, fmt, g, what):
    n = w.shape[0]
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a.cuda(), rep, n, fmt, g, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rows = _sample_rows(n)
    codes, scales = oracle_quantize(w[rows].cpu(), fmt, g)
    assert_parity(c[:, rows], oracle_reference(a, codes, scales, fmt, g), what)


@pytest.mark.parametrize("name,nk", SHAPES)
def test_nvfp4_decode_llama(cuda_lib, name, nk):
    n, k = nk
    w, rep = _prepare(cuda_lib, n, k, "nvfp4", seed=101)
    a = synth.activations(16, k, seed=201)
    _check(cuda_lib, w, rep, a, "nvfp4", 1.0, f"{name} m=16")


@pytest.mark.parametrize("name,nk", SHAPES)
def test_mxfp4_decode_llama(cuda_lib, name, nk):
    n, k = nk
    w, rep = _prepare(cuda_lib, n, k, "mxfp4", seed=102)
    for m in (1, 4, 8, 16):
        a = synth.activations(m, k, seed=202 + m)
        _check(cuda_lib, w, rep, a, "mxfp4", 1.0, f"{name} m={m}")


@pytest.mark.parametrize("name,nk", SHAPES)
def test_mxfp4_prefill_llama_m256(cuda_lib, name, nk):
    """MXFP4 at m = 256 (the prefill size bench.py also reports for MXFP4):
    gate_up and down run 256-row activation tiles, QKV and O two 128-row
    tiles."""
    n, k = nk
    w, rep = _prepare(cuda_lib, n, k, "mxfp4", seed=106)
    a = synth.activations(256, k, seed=206, outlier_frac=0.001, outlier_std=20.0)
    _check(cuda_lib, w, rep, a, "mxfp4", 1.0, f"{name} mxfp4 m=256")


@pytest.mark.parametrize("name,nk", SHAPES)
def test_nvfp4_prefill_llama_global_scale(cuda_lib, name, nk):
    n, k = nk
    w = synth.weights(n, k, seed=103, device="cuda")
    amax_cpu = np.float32(w.cpu().float().abs().max().item())
    g = float(quantize.nvfp4_global_scale(np.array([amax_cpu], dtype=np.float32)))
    # the GPU side derives g with its own max-abs and scale kernels
    g_gpu = cuda_lib.nvfp4_global_scale(cuda_lib.absmax(w).item())
    assert np.float32(g_gpu) == np.float32(g)
    wp, sp = cuda_lib.quantize(w, "nvfp4", g_gpu)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    del wp, sp
    a = synth.activations(256, k, seed=203, outlier_frac=0.001, outlier_std=20.0)
    _check(cuda_lib, w, rep, a, "nvfp4", g, f"{name} m=256")


def test_nvfp4_m_sweep(cuda_lib):
    n = k = 8192
    w, rep = _prepare(cuda_lib, n, k, "nvfp4", seed=104)
    for m in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024):
        a = synth.activations(m, k, seed=300 + m)
        _check(cuda_lib, w, rep, a, "nvfp4", 1.0, f"m={m}")
    w, rep = _prepare(cuda_lib, 4096, 4096, "nvfp4", seed=105)
    a = synth.activations(4096, 4096, seed=400)
    _check(cuda_lib, w, rep, a, "nvfp4", 1.0, "m=n=k=4096")
