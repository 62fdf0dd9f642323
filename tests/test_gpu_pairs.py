"""CTA-pair GEMM kernel (cta_group::2, two CTAs per 256-row weight tile pair)
vs the FP64 oracle.

The pair kernel is chosen by the planner for 256-row activation tiles and
for 128-row tiles of large matrices; here mode 2 forces it wherever it
applies (n a multiple of 256, 128- or 256-row tiles), so small problems
exercise it.  One-hot activations make C bit-exact to the dequantised
weights: this pins the split of the activation rows between the two CTAs
(the MMA's N halves), the weight tile each CTA decodes and the output
columns each CTA writes.  Tolerance parity covers ragged m, split-K tails,
both formats and the FP16 layout; the pair kernel and the single-CTA kernel
agree within the tolerances, and repeated launches are bit-identical.
"""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import gemm as ogemm
from oracle import quantize
from tests.gpu_util import assert_parity, bf16_bits, compare, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu


@pytest.fixture()
def pairs(cuda_lib):
    """CTA pairs wherever they apply, restored to the default afterwards."""
    cuda_lib.set_pair_mode(2)
    yield cuda_lib
    cuda_lib.set_pair_mode(0)
    cuda_lib.set_tile_config(0, 0)


def _prep(lib, w, fmt, g=1.0):
    codes, scales = oracle_quantize(w, "nvfp4" if fmt == "nvfp4_f16" else fmt, g)
    wp, sp = to_device_packed(codes, scales)
    rep = lib.repack(wp, sp, fmt)
    torch.cuda.synchronize()
    return codes, scales, rep


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,n,k,bn", [(200, 512, 640, 256), (100, 768, 1024, 128), (256, 512, 2048, 128),
                                      (40, 512, 1024, 128)])
def test_pair_one_hot_is_bit_exact(pairs, fmt, m, n, k, bn):
    w = synth.weights(n, k, seed=7 + m)
    codes, scales, rep = _prep(pairs, w, fmt)
    rng = np.random.default_rng(m + n + k)
    cols = rng.permutation(k)[:m]
    a = synth.one_hot_activations(m, k, cols).cuda()
    pairs.set_tile_config(bn, 1)
    ws = pairs.Workspace()
    c = pairs.gemm(a, rep, n, fmt, 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    expect = ogemm.dequantize_bf16_bits(codes, scales, fmt)[:, cols].T
    got = bf16_bits(c)
    zero = (expect & 0x7FFF) == 0
    bad = ~((got == expect) | (zero & ((got & 0x7FFF) == 0)))
    assert not bad.any(), f"{int(bad.sum())} mismatches, first at {np.argwhere(bad)[:4].tolist()}"


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "nvfp4_f16"])
@pytest.mark.parametrize("m", [65, 128, 129, 255, 256, 300, 512])
def test_pair_parity_ragged_m(pairs, fmt, m):
    n, k = 1024, 4096          # 4 tile pairs x 32 k-units: split tiles over the pairs
    w = synth.weights(n, k, seed=11)
    qfmt = "nvfp4" if fmt == "nvfp4_f16" else fmt
    g = float(quantize.nvfp4_global_scale(w.float().numpy())) if qfmt == "nvfp4" else 1.0
    codes, scales, rep = _prep(pairs, w, fmt, g)
    a = synth.activations(m, k, seed=12 + m)
    if fmt == "nvfp4_f16":
        a = a.to(torch.float16)
    ws = pairs.Workspace()
    c = pairs.gemm(a.cuda(), rep, n, fmt, g, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert_parity(c, oracle_reference(a, codes, scales, qfmt, g), f"{fmt} m={m}")


def test_pair_and_single_cta_kernels_agree_and_repeat(cuda_lib):
    n, k, m = 2048, 4096, 200
    w = synth.weights(n, k, seed=13)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    a = synth.activations(m, k, seed=14).cuda()
    ref = oracle_reference(a.cpu(), codes, scales, "nvfp4")
    out = {}
    try:
        for mode in (2, 1):
            cuda_lib.set_pair_mode(mode)
            ws = cuda_lib.Workspace()
            first = cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws).clone()
            for _ in range(8):
                assert torch.equal(cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws), first)
            assert ws.status() == 0
            assert_parity(first, ref, f"pair mode {mode}")
            out[mode] = first
    finally:
        cuda_lib.set_pair_mode(0)
    mx, l2 = compare(out[2], out[1].float().cpu().numpy().astype(np.float64))
    assert mx <= 1e-2 and l2 <= 4e-3, (mx, l2)


def test_pair_full_size_gate_up_prefill(cuda_lib):
    """The planner's default for Llama-3-70B gate_up at m = 256 (CTA pairs,
    256-row tiles), sampled output columns against the oracle."""
    n, k, m = 57344, 8192, 256
    w = synth.weights(n, k, seed=15, device="cuda")
    g = cuda_lib.nvfp4_global_scale(cuda_lib.absmax(w).item())
    wp, sp = cuda_lib.quantize(w, "nvfp4", g)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    torch.cuda.synchronize()
    a = synth.activations(m, k, seed=16).cuda()
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a, rep, n, "nvfp4", g, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rows = np.concatenate([np.arange(0, 256), np.arange(n - 256, n), np.arange(300, n, 977)])
    codes, scales = oracle_quantize(w[rows].cpu(), "nvfp4", g)
    assert_parity(c[:, rows], oracle_reference(a.cpu(), codes, scales, "nvfp4", g), "gate_up m=256")


@pytest.mark.parametrize("n,m", [(16384, 100), (57344, 200)])
def test_full_tiles_write_no_row_past_m(cuda_lib, n, m):
    """Whole 128/256-row output tiles are written through the shared-memory
    stage in 256-byte row segments; with m not a multiple of the tile height
    (n = 16384: one 128-row tile per CTA on 128 CTAs; n = 57344: CTA pairs,
    256-row tiles) no row past m may be written, and sampled columns match
    the oracle."""
    k = 8192
    w = synth.weights(n, k, seed=17, device="cuda")
    g = cuda_lib.nvfp4_global_scale(cuda_lib.absmax(w).item())
    wp, sp = cuda_lib.quantize(w, "nvfp4", g)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    torch.cuda.synchronize()
    a = synth.activations(m, k, seed=18).cuda()
    guard = 16
    buf = torch.full((m + guard, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a, rep, n, "nvfp4", g, workspace=ws, out=buf[:m])
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.isnan(buf[m:].float()).all(), "a row past m was written"
    assert not torch.isnan(c.float()).any()
    rows = np.concatenate([np.arange(0, 128), np.arange(n - 128, n), np.arange(200, n, 1013)])
    codes, scales = oracle_quantize(w[rows].cpu(), "nvfp4", g)
    assert_parity(c[:, rows], oracle_reference(a.cpu(), codes, scales, "nvfp4", g), f"n={n} m={m}")
