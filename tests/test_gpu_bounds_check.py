"""The bounds-checking build of the library (_petit_check.so) on the GPU.

In this build the GEMM kernel checks every global-memory access, bulk and
tensor copy and shared- or tensor-memory buffer index against its buffer
before use; a failed check skips the access, stops the CTA and records
PETIT_ERR_BOUNDS.  Illegal addresses from a wrong index or copy coordinate
are the failure the CUTLASS FP4 article describes (sections 5.1 and 7); this
build turns them into a status.

* Every kernel shape (tile heights 16..256, one or two chunks per unit,
  split tiles, ragged m), the CTA-pair kernel, both formats, the FP16
  layout, the grouped MoE launch and the no-allocation entry point run with
  all checks passing:
  status OK and results within the oracle tolerances.
* A check is made to fail without any access leaving its real buffer: the
  extents the checks use are lowered (weights, then C) below the true ones.
  The kernel then reports PETIT_ERR_BOUNDS and returns; no store reaches C
  beyond the lowered extent; after the status read the same workspace gives
  correct results again.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import quantize
from tests.gpu_util import assert_parity, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu

OK, ERR_BOUNDS = 0, 8


@pytest.fixture(scope="module")
def chk(cuda_lib):
    """The binding, with every call routed through the bounds-checking build."""
    with cuda_lib.bounds_checked() as lib:
        assert lib.petit_bounds_checking() == 1
        yield cuda_lib
        assert lib.petit_check_set_limits(-1, -1) == 0


def _prep(lib, w, fmt, g=1.0):
    codes, scales = oracle_quantize(w, "nvfp4" if fmt == "nvfp4_f16" else fmt, g)
    wp, sp = to_device_packed(codes, scales)
    rep = lib.repack(wp, sp, fmt)
    torch.cuda.synchronize()
    return codes, scales, rep


@pytest.mark.parametrize("bn,ku", [(16, 1), (16, 2), (32, 2), (64, 1), (64, 2), (128, 1), (256, 1)])
def test_every_tile_shape_passes_its_checks(chk, bn, ku):
    n, k, m = 512, 2048, 70          # ragged m, several tiles, split tiles
    w = synth.weights(n, k, seed=bn + ku)
    codes, scales, rep = _prep(chk, w, "nvfp4")
    a = synth.activations(m, k, seed=bn)
    ws = chk.Workspace()
    chk.set_tile_config(bn, ku)
    try:
        c = chk.gemm(a.cuda(), rep, n, "nvfp4", 1.0, workspace=ws)
    finally:
        chk.set_tile_config(0, 0)
    assert ws.status() == OK
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), f"bn={bn} ku={ku}")


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("m", [40, 200])
def test_cta_pairs_pass_their_checks(chk, bn, m):
    """The CTA-pair kernel (forced), including a tile whose second half of
    activation rows lies entirely past m."""
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=bn + m)
    codes, scales, rep = _prep(chk, w, "mxfp4")
    a = synth.activations(m, k, seed=m)
    ws = chk.Workspace()
    chk.set_pair_mode(2)
    chk.set_tile_config(bn, 1)
    try:
        c = chk.gemm(a.cuda(), rep, n, "mxfp4", 1.0, workspace=ws)
    finally:
        chk.set_tile_config(0, 0)
        chk.set_pair_mode(0)
    assert ws.status() == OK
    assert_parity(c, oracle_reference(a, codes, scales, "mxfp4"), f"pairs bn={bn} m={m}")


@pytest.mark.parametrize("fmt,m,k", [("nvfp4", 16, 4096), ("nvfp4", 5, 3968), ("mxfp4", 16, 4096),
                                     ("mxfp4", 200, 1024), ("nvfp4_f16", 33, 2048)])
def test_planner_shapes_pass_their_checks(chk, fmt, m, k):
    n = 1024
    w = synth.weights(n, k, seed=m + k)
    qfmt = "nvfp4" if fmt == "nvfp4_f16" else fmt
    g = float(quantize.nvfp4_global_scale(w.float().numpy())) if qfmt == "nvfp4" else 1.0
    codes, scales, rep = _prep(chk, w, fmt, g)
    a = synth.activations(m, k, seed=m)
    if fmt == "nvfp4_f16":
        a = a.to(torch.float16)
    ws = chk.Workspace()
    c = chk.gemm(a.cuda(), rep, n, fmt, g, workspace=ws)
    assert ws.status() == OK
    assert_parity(c, oracle_reference(a, codes, scales, qfmt, g), fmt)


def test_moe_and_noalloc_pass_their_checks(chk):
    E, n, k = 6, 512, 1024
    off = [0, 5, 5, 40, 41, 41, 60]                  # empty experts, ragged groups
    reps, cs = [], []
    for e in range(E):
        codes, scales, rep = _prep(chk, synth.weights(n, k, seed=70 + e), "mxfp4")
        reps.append(rep)
        cs.append((codes, scales))
    rep_all = torch.cat(reps)
    torch.cuda.synchronize()
    a = synth.activations(off[-1], k, seed=71)
    ws = chk.Workspace()
    c = chk.moe_gemm(a.cuda(), rep_all, off, n, "mxfp4", workspace=ws)
    assert ws.status() == OK
    for e in range(E):
        if off[e + 1] > off[e]:
            codes, scales = cs[e]
            assert_parity(c[off[e]:off[e + 1]],
                          oracle_reference(a[off[e]:off[e + 1]], codes, scales, "mxfp4"), f"e{e}")
    # the entry point with the library's own scratch
    L = chk.load()
    codes, scales, rep = _prep(chk, synth.weights(n, k, seed=72), "nvfp4")
    a = synth.activations(16, k, seed=73)
    out = torch.empty((16, n), dtype=torch.bfloat16, device="cuda")
    st = L.petit_gemm_bf16_nvfp4_noalloc(ctypes.c_void_p(a.cuda().data_ptr()),
                                         ctypes.c_void_p(rep.data_ptr()), ctypes.c_float(1.0),
                                         ctypes.c_void_p(out.data_ptr()), 16, n, k,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == OK
    torch.cuda.synchronize()
    assert_parity(out, oracle_reference(a, codes, scales, "nvfp4"), "noalloc")


def _limited(chk, weight_bytes, c_elems, fn):
    L = chk.load()
    assert L.petit_check_set_limits(weight_bytes, c_elems) == 0
    try:
        return fn()
    finally:
        assert L.petit_check_set_limits(-1, -1) == 0


@pytest.mark.parametrize("m", [16, 200])
def test_failed_weight_check_reports_bounds_and_recovers(chk, m):
    """m = 16: single CTAs; m = 200: CTA pairs (256-row tiles), where the CTA
    that stops leaves its partner to run out its bounded waits and both
    meet at the final cluster barrier."""
    n, k = 1024, 8192                 # split tiles: arrival counters in use
    w = synth.weights(n, k, seed=81)
    codes, scales, rep = _prep(chk, w, "nvfp4")
    a = synth.activations(m, k, seed=82).cuda()
    ws = chk.Workspace()
    # only the first half of the weights count as readable
    _limited(chk, rep.numel() // 2, -1, lambda: chk.gemm(a, rep, n, "nvfp4", workspace=ws))
    assert ws.status() == ERR_BOUNDS
    assert ws.status() == OK          # the read cleared the word (and the counters)
    c = chk.gemm(a, rep, n, "nvfp4", workspace=ws)
    assert ws.status() == OK
    assert_parity(c, oracle_reference(a.cpu(), codes, scales, "nvfp4"), "after recovery")


@pytest.mark.parametrize("m", [16, 200])
def test_failed_output_check_stops_before_the_extent(chk, m):
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=83)
    codes, scales, rep = _prep(chk, w, "mxfp4")
    a = synth.activations(m, k, seed=84).cuda()
    ws = chk.Workspace()
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    limit = (m * n) // 2 + 77
    _limited(chk, -1, limit, lambda: chk.gemm(a, rep, n, "mxfp4", workspace=ws, out=out))
    assert ws.status() == ERR_BOUNDS
    tail = out.view(-1)[limit:].float().cpu().numpy()
    assert np.isnan(tail).all(), "a store passed the lowered extent of C"
    c = chk.gemm(a, rep, n, "mxfp4", workspace=ws)
    assert ws.status() == OK
    assert_parity(c, oracle_reference(a.cpu(), codes, scales, "mxfp4"), "after recovery")
