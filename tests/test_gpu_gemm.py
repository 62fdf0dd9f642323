"""GPU GEMM (C ABI, tcgen05 path) vs the FP64 oracle.

* one-hot activations with g = 1 make C bit-exact to the dequantised weights
  (pins the repack layout, the tensor-memory operand layout and the stream-K
  reduction through the whole path);
* seeded N(0,1) x N(0,0.02) problems within the tolerances
  max|C - ref| <= 1e-2 max|ref| and rel-L2 <= 4e-3, over ragged m, several
  tiles and split-K tails, NVFP4 (with and without global scale) and MXFP4;
* special cases: A = 0, all-zero weights, outlier activations;
* determinism and workspace reuse.
"""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import gemm as ogemm
from oracle import quantize
from tests.gpu_util import assert_parity, bf16_bits, oracle_quantize, oracle_reference, to_device_packed

pytestmark = pytest.mark.gpu


def _prep(cuda_lib, w, fmt, g=1.0):
    codes, scales = oracle_quantize(w, fmt, g)
    wp, sp = to_device_packed(codes, scales)
    return codes, scales, cuda_lib.repack(wp, sp, fmt)


def _gemm(cuda_lib, a, rep, n, fmt, g=1.0):
    """One GEMM with its own workspace; no bounded wait may have run out."""
    ws = cuda_lib.Workspace()
    c = cuda_lib.gemm(a, rep, n, fmt, g, workspace=ws)
    assert ws.status() == 0, "device status: a pipeline wait timed out"
    return c


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,n,k", [(1024, 1024, 1024), (16, 256, 2048), (200, 384, 640)])
def test_one_hot_is_bit_exact(cuda_lib, fmt, m, n, k):
    w = synth.weights(n, k, seed=5)
    codes, scales, rep = _prep(cuda_lib, w, fmt)
    rng = np.random.default_rng(m + n + k)
    cols = rng.permutation(k)[:m] if m <= k else rng.integers(0, k, m)
    a = synth.one_hot_activations(m, k, cols).cuda()
    c = _gemm(cuda_lib, a, rep, n, fmt, 1.0)
    torch.cuda.synchronize()
    wq_bits = ogemm.dequantize_bf16_bits(codes, scales, fmt)      # [n, k]
    expect = wq_bits[:, cols].T                                   # C[i, :] = Wq[:, cols[i]]
    got = bf16_bits(c)
    # -0.0 weights give +0.0 sums; compare values for zeros, bits otherwise
    zero = (expect & 0x7FFF) == 0
    assert np.all((got == expect) | (zero & ((got & 0x7FFF) == 0)))


@pytest.mark.parametrize("m", [16, 200])
def test_mxfp4_one_and_two_multiply_chunks_one_hot(cuda_lib, m):
    """MXFP4 weights whose second 128-row tile is scaled by 2^20: its chunks
    hold E8M0 codes above 128 and take the two-multiply decode, the others
    the one-multiply decode.  One-hot activations make C bit-exact to Wq."""
    n, k = 384, 1024
    w = synth.weights(n, k, seed=15)
    w[128:256] *= 2.0 ** 20                     # exact in BF16
    codes, scales, rep = _prep(cuda_lib, w, "mxfp4")
    assert (scales[128:256] > 128).any() and (scales[:128] <= 128).all()
    rng = np.random.default_rng(m)
    cols = rng.integers(0, k, m)
    a = synth.one_hot_activations(m, k, cols).cuda()
    c = _gemm(cuda_lib, a, rep, n, "mxfp4", 1.0)
    torch.cuda.synchronize()
    expect = ogemm.dequantize_bf16_bits(codes, scales, "mxfp4")[:, cols].T
    got = bf16_bits(c)
    zero = (expect & 0x7FFF) == 0
    assert np.all((got == expect) | (zero & ((got & 0x7FFF) == 0)))


@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 16, 17, 33, 64, 65, 100, 128, 255, 256, 300])
def test_nvfp4_parity_ragged_m(cuda_lib, m):
    n, k = 1024, 1024
    w = synth.weights(n, k, seed=1)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    a = synth.activations(m, k, seed=m)
    c = _gemm(cuda_lib, a.cuda(), rep, n, "nvfp4", 1.0)
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), f"m={m}")


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("m", [4, 40, 130])
def test_odd_chunk_count(cuda_lib, fmt, m):
    """k = 9 x 128: pipeline units of a single 128-k chunk at every m."""
    n, k = 256, 1152
    w = synth.weights(n, k, seed=12)
    codes, scales, rep = _prep(cuda_lib, w, fmt)
    a = synth.activations(m, k, seed=13)
    c = _gemm(cuda_lib, a.cuda(), rep, n, fmt, 1.0)
    assert_parity(c, oracle_reference(a, codes, scales, fmt), f"m={m}")


@pytest.mark.parametrize("m", [1, 4, 8, 16, 100])
def test_mxfp4_parity(cuda_lib, m):
    n, k = 768, 2048
    w = synth.weights(n, k, seed=2)
    codes, scales, rep = _prep(cuda_lib, w, "mxfp4")
    a = synth.activations(m, k, seed=10 + m)
    c = _gemm(cuda_lib, a.cuda(), rep, n, "mxfp4")
    assert_parity(c, oracle_reference(a, codes, scales, "mxfp4"), f"m={m}")


@pytest.mark.parametrize("m", [16, 256])
def test_nvfp4_global_scale_and_outliers(cuda_lib, m):
    """Prefill-style inputs: 0.1% N(0,20) activation outliers, g = amax/(6*448)."""
    n, k = 640, 1536
    w = synth.weights(n, k, seed=3)
    g = float(quantize.nvfp4_global_scale(w.float().numpy()))
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4", g)
    a = synth.activations(m, k, seed=4, outlier_frac=0.001, outlier_std=20.0)
    c = _gemm(cuda_lib, a.cuda(), rep, n, "nvfp4", g)
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4", g), f"m={m}")


def test_special_cases(cuda_lib):
    n, k = 256, 512
    w = synth.weights(n, k, seed=6)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    z = torch.zeros((7, k), dtype=torch.bfloat16, device="cuda")
    c = _gemm(cuda_lib, z, rep, n, "nvfp4")
    assert torch.all(c == 0)
    # all-zero weights (zero codes, smallest positive scale)
    zw = torch.zeros((n, k), dtype=torch.bfloat16)
    codes0, scales0, rep0 = _prep(cuda_lib, zw, "nvfp4")
    assert np.all(codes0 == 0)
    a = synth.activations(9, k, seed=7).cuda()
    assert torch.all(_gemm(cuda_lib, a, rep0, n, "nvfp4") == 0)
    # all-ones activations give (BF16-rounded) row sums
    ones = torch.ones((1, k), dtype=torch.bfloat16, device="cuda")
    assert_parity(_gemm(cuda_lib, ones, rep, n, "nvfp4"),
                  oracle_reference(ones.cpu(), codes, scales, "nvfp4"), "ones")


def test_deterministic_and_workspace_reuse(cuda_lib):
    n, k = 1024, 2048
    w = synth.weights(n, k, seed=8)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    ws = cuda_lib.Workspace()
    outs = []
    for m in (16, 100, 16, 3, 16):
        a = synth.activations(m, k, seed=21).cuda()
        outs.append((m, cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws).clone()))
    assert ws.status() == 0
    c16 = [c for m, c in outs if m == 16]
    assert all(torch.equal(c16[0], c) for c in c16[1:])
    for m, c in outs:
        a = synth.activations(m, k, seed=21)
        assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), f"m={m}")
    # status word and arrival counters (256 + 4096 bytes) are left at zero;
    # the partials may hold data
    buf = ws.buf.cpu()
    assert int(buf[:4352].count_nonzero()) == 0


def test_bounded_wait_reports_timeout(cuda_lib):
    """Failure detection: a wait that nobody satisfies runs out and reports,
    and the context stays usable afterwards."""
    ws = cuda_lib.Workspace()
    cuda_lib.selftest_timeout(ws, 2000)
    assert ws.status() == 7                      # PETIT_ERR_TIMEOUT
    assert ws.status() == 0                      # cleared by the read
    n, k = 256, 256
    w = synth.weights(n, k, seed=9)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    a = synth.activations(4, k, seed=9)
    c = cuda_lib.gemm(a.cuda(), rep, n, "nvfp4", workspace=ws)
    assert ws.status() == 0
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), "after timeout")


@pytest.mark.parametrize("bn,ku", [(16, 1), (16, 2), (32, 1), (32, 2), (64, 1), (64, 2), (128, 1), (256, 1)])
def test_forced_tile_config(cuda_lib, bn, ku):
    """Every (BN, KU) kernel forced on one problem: m = 70 spans several
    16/32/64-row tiles and a ragged tail; k = 2048 gives split tiles."""
    n, k, m = 512, 2048, 70
    w = synth.weights(n, k, seed=90)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    a = synth.activations(m, k, seed=91)
    cuda_lib.set_tile_config(bn, ku)
    try:
        c = _gemm(cuda_lib, a.cuda(), rep, n, "nvfp4", 1.0)
    finally:
        cuda_lib.set_tile_config(0, 0)
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), f"bn={bn} ku={ku}")


def test_timeout_recovery_clears_arrival_counters(cuda_lib):
    """A kernel that stops early on a timeout can leave split-tile arrival
    counters raised.  Reading the status clears them with the status word, so
    the next split-K GEMM on the same workspace is correct again.  The
    aborted state is made on the host: status word = timeout, every counter
    dirty."""
    n, k, m = 1024, 8192, 16          # 256 units over the SMs: many split tiles
    w = synth.weights(n, k, seed=19)
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
    a = synth.activations(m, k, seed=19)
    ws = cuda_lib.Workspace()
    buf = ws.ensure(cuda_lib.workspace_bytes(m, n, k))
    words = buf[:4352].view(torch.int32)
    words[0] = 1                        # the timeout bit
    words[64:].fill_(3)                 # counters region [256, 4352)
    torch.cuda.synchronize()
    assert ws.status() == 7
    assert int(buf[:4352].count_nonzero()) == 0
    c = cuda_lib.gemm(a.cuda(), rep, n, "nvfp4", workspace=ws)
    assert ws.status() == 0
    assert_parity(c, oracle_reference(a, codes, scales, "nvfp4"), "after recovery")


# m -> the kernel's activation tile N (16/32/64/128/256) and chunks per unit;
# k/128 odd forces one chunk per unit.  Repeated launches catch pipeline
# races (a lost or aliased barrier phase shows up as a timeout status or a
# changed result).
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,k", [(8, 4096), (24, 4096), (48, 4096), (48, 3968), (100, 4096),
                                 (200, 4096), (300, 2048), (16, 3968)])
def test_every_tile_config_repeated(cuda_lib, fmt, m, k):
    n = 2048
    w = synth.weights(n, k, seed=m + k)
    codes, scales, rep = _prep(cuda_lib, w, fmt)
    a = synth.activations(m, k, seed=m).cuda()
    ws = cuda_lib.Workspace()
    first = cuda_lib.gemm(a, rep, n, fmt, 1.0, workspace=ws).clone()
    for _ in range(12):
        again = cuda_lib.gemm(a, rep, n, fmt, 1.0, workspace=ws)
        assert torch.equal(again, first)
    assert ws.status() == 0
    rows = np.arange(0, n, 37)
    assert_parity(first[:, rows], oracle_reference(a.cpu(), codes[rows], scales[rows], fmt), f"m={m}")


def test_large_prefill_tile(cuda_lib):
    """m = 256 on a matrix large enough for 256-row activation tiles (one
    dequantisation per weight for all rows); oracle on sampled columns."""
    m, n, k = 256, 8192, 16384
    w = synth.weights(n, k, seed=31, device="cuda")
    wp, sp = cuda_lib.quantize(w, "nvfp4", 1.0)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    a = synth.activations(m, k, seed=32, outlier_frac=0.001, outlier_std=20.0).cuda()
    c = _gemm(cuda_lib, a, rep, n, "nvfp4", 1.0)
    rows = np.concatenate([np.arange(0, 256, 5), np.arange(n - 300, n, 7)])
    # quantisation is row-local: the oracle quantises just the sampled rows
    codes, scales = oracle_quantize(w[rows].cpu(), "nvfp4", 1.0)
    assert_parity(c[:, rows], oracle_reference(a.cpu(), codes, scales, "nvfp4"), "m=256 large")


def test_workspace_shared_across_shapes(cuda_lib):
    """One workspace serves problems with different tile counts back to back
    (the partials of one must never land on the counters of another)."""
    probs = []
    for i, (m, n, k) in enumerate([(16, 256, 4096), (16, 8192, 1024), (200, 512, 2048), (64, 4096, 1024)]):
        w = synth.weights(n, k, seed=40 + i)
        codes, scales, rep = _prep(cuda_lib, w, "nvfp4")
        a = synth.activations(m, k, seed=50 + i)
        rows = np.arange(0, n, 29)
        probs.append((a.cuda(), rep, n, rows, oracle_reference(a, codes[rows], scales[rows], "nvfp4")))
    ws = cuda_lib.Workspace()
    for rnd in range(3):
        for j, (a, rep, n, rows, ref) in enumerate(probs):
            c = cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws)
            assert_parity(c[:, rows], ref, f"round {rnd} problem {j}")
    assert ws.status() == 0


def test_back_to_back_prefill_tiles(cuda_lib):
    """Kernels with 128- and 256-row activation tiles launched back to back
    (no host synchronisation) on large matrices reproduce, bit for bit, the
    results of isolated launches; the isolated results match the oracle on
    sampled columns.  Guards the pipeline's barrier protocol, where a
    consumer that skipped a phase once read a stage before it had landed."""
    m = 256
    probs = []
    for i, (n, k) in enumerate([(8192, 8192), (8192, 28672)]):
        w = synth.weights(n, k, seed=60 + i, device="cuda")
        wp, sp = cuda_lib.quantize(w, "nvfp4", 1.0)
        rep = cuda_lib.repack(wp, sp, "nvfp4")
        a = synth.activations(m, k, seed=70 + i).cuda()
        ws = cuda_lib.Workspace()
        ref = cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws).clone()
        torch.cuda.synchronize()
        assert ws.status() == 0
        rows = np.arange(3, n, 517)
        codes, scales = oracle_quantize(w[rows].cpu(), "nvfp4", 1.0)
        assert_parity(ref[:, rows], oracle_reference(a.cpu(), codes, scales, "nvfp4"), f"n={n} k={k}")
        del w, wp, sp
        probs.append((a, rep, n, ws, ref))
    outs = []
    for _ in range(6):
        for a, rep, n, ws, _ in probs:
            outs.append(cuda_lib.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws))
    torch.cuda.synchronize()
    for j, c in enumerate(outs):
        assert torch.equal(c, probs[j % 2][4]), f"launch {j}"
    assert all(p[3].status() == 0 for p in probs)


def test_device_global_scale_in_graph(cuda_lib):
    """The device-pointer global scale: same bits as the host-scale call, and
    a captured CUDA graph picks up a new value on replay (g doubled -> every
    BF16 output exactly doubled)."""
    n, k, m = 1024, 2048, 16
    w = synth.weights(n, k, seed=80)
    g0 = float(quantize.nvfp4_global_scale(w.float().numpy()))
    codes, scales, rep = _prep(cuda_lib, w, "nvfp4", g0)
    a = synth.activations(m, k, seed=81).cuda()
    ref = _gemm(cuda_lib, a, rep, n, "nvfp4", g0)
    gdev = torch.tensor([g0], dtype=torch.float32, device="cuda")
    ws = cuda_lib.Workspace()
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    cuda_lib.gemm(a, rep, n, "nvfp4", gdev, workspace=ws, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            cuda_lib.gemm(a, rep, n, "nvfp4", gdev, workspace=ws, out=out)
        gdev.fill_(2.0 * g0)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.float(), 2.0 * ref.float())
    assert ws.status() == 0
    assert_parity(ref, oracle_reference(a.cpu(), codes, scales, "nvfp4", g0), "device g")
