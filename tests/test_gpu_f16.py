"""FP16-activation variant (FP16 A x NVFP4 W -> FP16 C) vs the oracle.

* repack for the FP16 layout + dequant hook reproduce the oracle's Wq as
  binary16, bit for bit, for every code and every positive E4M3 scale;
* one-hot activations make C bit-exact to columns of Wq;
* tolerance parity (max|C - ref| <= 1e-2 max|ref|, rel-L2 <= 4e-3) over
  ragged m and with a global scale, and at full size on the Llama-3-70B
  decode shapes (sampled columns).
"""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import gemm as ogemm
from oracle import quantize
from tests.gpu_util import assert_parity, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu


def _f16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _prep(cuda_lib, w, g=1.0):
    codes, scales = oracle_quantize(w, "nvfp4", g)
    wp, sp = to_device_packed(codes, scales)
    return codes, scales, cuda_lib.repack(wp, sp, "nvfp4_f16")


def test_repack_dequant_f16_bitexact(cuda_lib):
    n, k = 256, 128 * 16
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    codes[7, :16] = np.arange(16)
    scales = np.tile(np.arange(1, 127, dtype=np.uint8), (n * k // 16) // 126 + 1)[: n * k // 16]
    scales = scales.reshape(n, k // 16)
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "nvfp4_f16")
    got = _f16_bits(cuda_lib.dequant(rep, n, k, "nvfp4_f16"))
    np.testing.assert_array_equal(got, ogemm.dequantize_f16_bits(codes, scales))


@pytest.mark.parametrize("m,n,k", [(16, 256, 2048), (200, 384, 640)])
def test_f16_one_hot_is_bit_exact(cuda_lib, m, n, k):
    w = synth.weights(n, k, seed=22)
    codes, scales, rep = _prep(cuda_lib, w)
    rng = np.random.default_rng(m + k)
    cols = rng.permutation(k)[:m]
    a = synth.one_hot_activations(m, k, cols).to(torch.float16).cuda()
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a, rep, n, "nvfp4_f16", 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    expect = ogemm.dequantize_f16_bits(codes, scales)[:, cols].T
    got = _f16_bits(c)
    zero = (expect & 0x7FFF) == 0
    assert np.all((got == expect) | (zero & ((got & 0x7FFF) == 0)))


@pytest.mark.parametrize("m", [1, 16, 33, 100, 256, 300])
def test_f16_parity_ragged_m(cuda_lib, m):
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=23)
    g = float(quantize.nvfp4_global_scale(w.float().numpy()))
    codes, scales, rep = _prep(cuda_lib, w, g)
    a = synth.activations(m, k, seed=24 + m).to(torch.float16)
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a.cuda(), rep, n, "nvfp4_f16", g, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0 and c.dtype == torch.float16
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4", g), f"f16 m={m}")


@pytest.mark.parametrize("name", ["gate_up", "down"])
def test_f16_decode_llama_full_size(cuda_lib, name):
    n, k = synth.LLAMA3_70B_SHAPES[name]
    w = synth.weights(n, k, seed=25, device="cuda")
    wp, sp = cuda_lib.quantize(w, "nvfp4", 1.0)
    rep = cuda_lib.repack(wp, sp, "nvfp4_f16")
    del wp, sp
    a = synth.activations(16, k, seed=26).to(torch.float16)
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a.cuda(), rep, n, "nvfp4_f16", 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rows = np.unique(np.concatenate([np.linspace(0, n - 1, 48).astype(np.int64), [0, n - 1]]))
    codes, scales = oracle_quantize(w[rows].cpu(), "nvfp4", 1.0)
    assert_parity(c[:, rows], oracle_reference(a, codes, scales, "nvfp4"), f"f16 {name}")
