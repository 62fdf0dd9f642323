"""MoE grouped GEMM (C ABI) vs the oracle, one plain GEMM per expert.

Expert e's output rows [off[e], off[e+1]) must equal the oracle's
g_e * A[rows] . Wq_e^T within the usual tolerances; empty experts, a single
busy expert, repeated launches (bit-identical) and full-size Mixtral-like
shapes (sampled columns) are covered."""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import quantize
from tests.gpu_util import assert_parity, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu


def _experts(cuda_lib, E, n, k, fmt, seed, device_quant=False):
    reps, ws_cpu, gs = [], [], []
    for e in range(E):
        if device_quant:
            w = synth.weights(n, k, seed=seed + e, device="cuda")
            g = cuda_lib.nvfp4_global_scale(cuda_lib.absmax(w).item()) if fmt == "nvfp4" else 1.0
            wp, sp = cuda_lib.quantize(w, fmt, g)
        else:
            w = synth.weights(n, k, seed=seed + e)
            g = float(quantize.nvfp4_global_scale(w.float().numpy())) if fmt == "nvfp4" else 1.0
            codes, scales = oracle_quantize(w, fmt, g)
            wp, sp = to_device_packed(codes, scales)
        reps.append(cuda_lib.repack(wp, sp, fmt))
        ws_cpu.append(w)
        gs.append(g)
    rep = torch.cat(reps)
    # a GEMM reads its weights while the kernel before it on the stream is
    # still finishing, so the copy that wrote them must have completed
    torch.cuda.synchronize()
    return rep, ws_cpu, gs


def _check(cuda_lib, c, a, ws_cpu, gs, off, fmt, rows=None):
    for e in range(len(off) - 1):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        w = ws_cpu[e] if rows is None else ws_cpu[e][rows].cpu()
        codes, scales = oracle_quantize(w.cpu(), fmt, gs[e])
        got = c[lo:hi] if rows is None else c[lo:hi][:, rows]
        assert_parity(got, oracle_reference(a[lo:hi], codes, scales, fmt, gs[e]), f"expert {e}")


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
@pytest.mark.parametrize("tokens,top_k", [(16, 2), (200, 2)])
def test_moe_matches_per_expert_oracle(cuda_lib, fmt, tokens, top_k):
    E, n, k = 8, 512, 1024
    off = synth.moe_expert_offsets(tokens, E, top_k, seed=tokens)
    rep, ws_cpu, gs = _experts(cuda_lib, E, n, k, fmt, seed=90)
    a = synth.activations(off[-1], k, seed=91)
    ws = cuda_lib.Workspace()
    c = cuda_lib.moe_gemm(a.cuda(), rep, off, n, fmt, gs, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _check(cuda_lib, c, a, ws_cpu, gs, off, fmt)


def test_moe_edge_routings_and_repeats(cuda_lib):
    E, n, k = 6, 256, 1152
    rep, ws_cpu, gs = _experts(cuda_lib, E, n, k, "mxfp4", seed=95)
    ws = cuda_lib.Workspace()
    for off in ([0, 0, 0, 40, 40, 40, 40],            # one busy expert
                [0, 1, 1, 130, 131, 300, 301],        # empty, single-row and multi-tile experts
                [0, 0, 0, 0, 0, 0, 0]):               # nothing routed: a no-op
        a = synth.activations(max(off[-1], 1), k, seed=off[-1])[: off[-1]]
        if off[-1] == 0:
            c = torch.empty((0, n), dtype=torch.bfloat16, device="cuda")
            cuda_lib.moe_gemm(a.cuda(), rep, off, n, "mxfp4", workspace=ws, out=c)
            continue
        first = cuda_lib.moe_gemm(a.cuda(), rep, off, n, "mxfp4", workspace=ws).clone()
        for _ in range(5):
            assert torch.equal(cuda_lib.moe_gemm(a.cuda(), rep, off, n, "mxfp4", workspace=ws), first)
        _check(cuda_lib, first, a, ws_cpu, gs, off, "mxfp4")
    assert ws.status() == 0


@pytest.mark.parametrize("tokens", [16, 256])
def test_moe_mixtral_shape_full_size(cuda_lib, tokens):
    """E = 8, top-2, gate_up of a Mixtral-8x7B-like layer (n = 28672,
    k = 4096), MXFP4; oracle on sampled columns of every expert."""
    E, n, k = 8, 28672, 4096
    off = synth.moe_expert_offsets(tokens, E, 2, seed=7)
    rep, ws_gpu, gs = _experts(cuda_lib, E, n, k, "mxfp4", seed=97, device_quant=True)
    a = synth.activations(off[-1], k, seed=98)
    ws = cuda_lib.Workspace()
    c = cuda_lib.moe_gemm(a.cuda(), rep, off, n, "mxfp4", workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rows = np.unique(np.concatenate([np.linspace(0, n - 1, 24).astype(np.int64), [0, n - 1]]))
    _check(cuda_lib, c, a, ws_gpu, gs, off, "mxfp4", rows=rows)
