"""The host-side planner through petit_plan_gemm / petit_plan_moe, on CPU.

The plan queries take the device's SM count and CTA-pair capacity as
arguments, so the planner's decisions and the stream-K ranges the kernel
will use are checked here without a GPU: every range non-empty and the
ranges covering the units exactly once, the tile-height and chunk rules of
petit.h, CTA pairs under each pair mode, tile-aligned ranges for 128-row
tiles, the shortened ranges of the CTAs that start last (decode tiles
only), the forced tile shapes, the workspace formula, and the MoE tile
choice.  GB300: 152 SMs, 76 resident CTA pairs.
"""

import itertools
import math

import pytest

from fp4_weight_only_gb300 import binding

SMS, PAIRS = 152, 76
LLAMA = [("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192), ("down", 8192, 28672)]
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(autouse=True)
def _planner_defaults():
    binding.set_tile_config(0, 0)
    binding.set_pair_mode(0)
    yield
    binding.set_tile_config(0, 0)
    binding.set_pair_mode(0)


def _check_plan(p, m, n, k, sms=SMS, pairs=PAIRS, groups_rows=None):
    """Invariants that hold for every plan."""
    pair = p["cta_pairs"]
    assert p["bn"] in (16, 32, 64, 128, 256)
    assert p["ku"] in (1, 2) and (p["ku"] == 1 or p["bn"] <= 64)
    assert p["units_per_tile"] == k // 128 // p["ku"]
    tile_rows = 256 if pair else 128
    rows = groups_rows if groups_rows is not None else [m]
    tiles = sum(math.ceil(r / p["bn"]) for r in rows) * (n // tile_rows)
    assert p["num_tiles"] == tiles
    assert p["units"] == tiles * p["units_per_tile"]
    assert 1 <= p["num_ranges"] <= (pairs if pair else sms)
    assert p["num_ranges"] <= p["units"]
    assert p["num_ctas"] == p["num_ranges"] * (2 if pair else 1)
    s = p["range_starts"]
    assert len(s) == p["num_ranges"] + 1 and s[0] == 0 and s[-1] == p["units"]
    assert all(b > a for a, b in zip(s, s[1:])), "every range holds at least one unit"
    # status word + counters (4352 bytes), then two BN x 128 FP32 partial
    # slots per CTA (the formula petit.h gives for the no-allocation scratch)
    assert p["workspace_bytes"] == 4352 + 1024 * p["num_ctas"] * p["bn"]


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "nvfp4_f16"])
@pytest.mark.parametrize("m", [1, 5, 16, 17, 32, 33, 64, 65, 96, 128, 129, 200, 256, 300, 512, 1024])
def test_llama_plans_hold_the_invariants(fmt, m):
    for _, n, k in LLAMA:
        _check_plan(binding.plan(m, n, k, fmt, SMS, PAIRS), m, n, k)


@pytest.mark.parametrize("n,k", [(128, 128), (256, 384), (1024, 1152), (384, 8192), (8192, 128)])
@pytest.mark.parametrize("sms", [1, 7, 16, 152, 1024])
def test_small_and_odd_problems_hold_the_invariants(n, k, sms):
    for m, mode in itertools.product([1, 40, 130, 256, 700], [0, 1, 2]):
        binding.set_pair_mode(mode)
        _check_plan(binding.plan(m, n, k, "nvfp4", sms, PAIRS), m, n, k, sms=sms)


def test_tile_height_and_chunks_follow_m():
    # single GEMMs on a large matrix (gate_up): bn is the smallest of
    # 16..256 that holds m, two 128-k chunks per unit for bn <= 64
    n, k = 57344, 8192
    for m, bn in [(1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64), (65, 128),
                  (128, 128), (129, 256), (256, 256), (4096, 256)]:
        p = binding.plan(m, n, k, "nvfp4", SMS, PAIRS)
        assert (p["bn"], p["ku"]) == (bn, 2 if bn <= 64 else 1), m
    # an odd number of 128-k chunks keeps one chunk per unit
    assert binding.plan(16, 1024, 3 * 128, "nvfp4", SMS, PAIRS)["ku"] == 1


def test_small_matrices_keep_128_row_tiles():
    # N = 256 halves the work units; below 48 units per SM the planner keeps
    # two 128-row tiles (O and QKV at m = 256), above it takes 256 (gate_up)
    assert binding.plan(256, 8192, 8192, "nvfp4", SMS, PAIRS)["bn"] == 128
    assert binding.plan(256, 10240, 8192, "nvfp4", SMS, PAIRS)["bn"] == 128
    assert binding.plan(256, 57344, 8192, "nvfp4", SMS, PAIRS)["bn"] == 256
    assert binding.plan(256, 8192, 28672, "nvfp4", SMS, PAIRS)["bn"] == 256


def test_cta_pairs_by_mode():
    shapes = [(m, n, k) for m in (100, 128, 200, 256, 512) for _, n, k in LLAMA]
    for m, n, k in shapes:
        auto = binding.plan(m, n, k, "mxfp4", SMS, PAIRS)
        binding.set_pair_mode(1)
        never = binding.plan(m, n, k, "mxfp4", SMS, PAIRS)
        binding.set_pair_mode(2)
        always = binding.plan(m, n, k, "mxfp4", SMS, PAIRS)
        binding.set_pair_mode(0)
        assert not never["cta_pairs"]
        # pairs apply to 128/256-row tiles with n a multiple of 256
        assert always["cta_pairs"] == (always["bn"] >= 128 and n % 256 == 0)
        if auto["cta_pairs"]:
            assert auto["bn"] >= 128
        if auto["bn"] == 256:
            assert auto["cta_pairs"], "256-row tiles always run on CTA pairs"
        # no pair capacity: single CTAs whatever the mode
        binding.set_pair_mode(2)
        assert not binding.plan(m, n, k, "mxfp4", SMS, 0)["cta_pairs"]
        binding.set_pair_mode(0)
    # n not a multiple of 256: never pairs
    binding.set_pair_mode(2)
    assert not binding.plan(256, 8192 + 128, 8192, "nvfp4", SMS, PAIRS)["cta_pairs"]


def test_pairs_where_they_pay():
    # 128-row tiles: pairs on the large matrix only (gate_up, 224 x 64
    # pair units >= 100 per resident pair), single CTAs on O and QKV
    assert binding.plan(128, 57344, 8192, "nvfp4", SMS, PAIRS)["cta_pairs"]
    assert not binding.plan(128, 8192, 8192, "nvfp4", SMS, PAIRS)["cta_pairs"]
    assert not binding.plan(128, 10240, 8192, "nvfp4", SMS, PAIRS)["cta_pairs"]
    p = binding.plan(256, 57344, 8192, "nvfp4", SMS, PAIRS)
    assert p["cta_pairs"] and p["num_ranges"] == PAIRS and p["num_ctas"] == 2 * PAIRS


def test_tile_aligned_ranges_for_128_row_tiles():
    # O at m = 128: 64 tiles of 64 units; two ranges per tile on 128 CTAs
    # beat 152 ranges that cross tile boundaries
    p = binding.plan(128, 8192, 8192, "nvfp4", SMS, PAIRS)
    assert (p["bn"], p["num_ranges"], p["cta_pairs"]) == (128, 128, False)
    assert p["range_starts"] == list(range(0, p["units"] + 1, 32))
    # O at m = 256: one whole tile per CTA
    p = binding.plan(256, 8192, 8192, "nvfp4", SMS, PAIRS)
    assert p["num_ranges"] == 128
    assert all(s % p["units_per_tile"] == 0 for s in p["range_starts"])
    # QKV: 80 tiles; whole tiles on 80 CTAs cost more than crossing
    # boundaries on all 152 SMs
    assert binding.plan(128, 10240, 8192, "nvfp4", SMS, PAIRS)["num_ranges"] == SMS


def test_ranges_of_late_ctas_are_shorter_at_decode_only():
    for m in (1, 16, 32, 64):
        for _, n, k in LLAMA:
            s = binding.plan(m, n, k, "nvfp4", SMS, PAIRS)["range_starts"]
            lens = [b - a for a, b in zip(s, s[1:])]
            assert lens[-1] < lens[0], (m, n, k)
            assert max(lens[:100]) - min(lens[:100]) <= 1   # the early CTAs share evenly
            assert sum(lens[-8:]) / 8 < sum(lens[:100]) / 100   # the last ones get less
    for m in (128, 256, 512):
        for _, n, k in LLAMA:
            s = binding.plan(m, n, k, "nvfp4", SMS, PAIRS)["range_starts"]
            lens = [b - a for a, b in zip(s, s[1:])]
            assert max(lens) - min(lens) <= 1, (m, n, k)   # even split


def test_forced_tile_shapes():
    for bn, ku in [(16, 1), (16, 2), (32, 2), (64, 1), (64, 2), (128, 1), (256, 1)]:
        binding.set_tile_config(bn, ku)
        p = binding.plan(70, 8192, 8192, "nvfp4", SMS, PAIRS)
        assert (p["bn"], p["ku"]) == (bn, ku)
        _check_plan(p, 70, 8192, 8192)
        # a k with an odd number of 128-k chunks runs one chunk per unit
        assert binding.plan(70, 1024, 384, "nvfp4", SMS, PAIRS)["ku"] == 1
    for bad in [(128, 2), (48, 1), (16, 3), (0, 1)]:
        with pytest.raises(binding.PetitError):
            binding.set_tile_config(*bad)


def test_moe_tile_height_minimises_dequantised_tiles():
    n, k = 28672, 4096
    # expected tile heights worked by hand from the rule below
    cases = {
        (0, 4, 12, 14, 19, 22, 24, 28, 32): 16,            # 16 tokens: 8 tiles at any bn
        (0, 159, 258, 286, 335, 378, 441, 487, 512): 128,  # 256 tokens: 35/19/11/9/16 tiles
        (0, 40, 40, 41): 64,                               # 4/3/2/2/4: the first least
        # one expert is a single GEMM: m = 200 asks for 256-row tiles, but
        # 224 x 32 units at N = 256 are under 48 per SM, so 128; the rule
        # stops at m = 256, so m = 300 keeps 256
        (0, 200): 128,
        (0, 300): 256,
    }
    for off, want_bn in cases.items():
        p = binding.moe_plan(list(off), n, k, "mxfp4", SMS, PAIRS)
        assert p["bn"] == want_bn, off
        rows = [b - a for a, b in zip(off, off[1:])]
        _check_plan(p, None, n, k, groups_rows=rows)
        assert not p["cta_pairs"] or len(rows) == 1
        if len(rows) > 1:
            # the least work: activation tiles summed over experts, a
            # 256-row tile counted as two
            def cost(bn):
                return sum(math.ceil(r / bn) for r in rows) * (bn // 128 if bn > 128 else 1)
            best = min(cost(bn) for bn in (16, 32, 64, 128, 256))
            assert cost(p["bn"]) == best
    # no routed tokens: nothing planned
    p = binding.moe_plan([0, 0, 0], n, k, "mxfp4", SMS, PAIRS)
    assert p["units"] == 0 and p["num_ranges"] == 0 and p["range_starts"] == []


def test_plan_errors():
    L = binding.load()
    info = binding.PlanInfo()

    def st(m=16, n=1024, k=1024, fmt=0, sms=SMS, pairs=PAIRS, out=True, starts=None, max_r=0):
        return L.petit_plan_gemm(m, n, k, fmt, sms, pairs, binding.ctypes.byref(info) if out else None,
                                 starts, max_r)
    assert st() == OK
    assert st(out=False) == INVALID
    assert st(m=0) == INVALID
    assert st(fmt=7) == INVALID
    assert st(sms=0) == INVALID and st(sms=1025) == INVALID
    assert st(pairs=-1) == INVALID and st(pairs=161) == INVALID
    assert st(n=1000) == UNSUPPORTED and st(k=100) == UNSUPPORTED
    assert st(m=(1 << 24) + 1) == UNSUPPORTED
    short = (binding.ctypes.c_int64 * 10)()
    # 8 tiles x 4 units = 32 ranges: 33 entries needed
    assert st(starts=short, max_r=10) == INVALID
    assert info.num_ranges == 32                       # the plan itself is still written
    off = (binding.ctypes.c_int64 * 3)(0, 5, 3)        # decreasing offsets
    assert L.petit_plan_moe(off, 2, 1024, 1024, 1, SMS, PAIRS, binding.ctypes.byref(info), None, 0) == INVALID
    off = (binding.ctypes.c_int64 * 3)(0, 5, 9)
    assert L.petit_plan_moe(off, 2, 1024, 1024, 2, SMS, PAIRS, binding.ctypes.byref(info), None, 0) == INVALID


def test_tune_plan_only_cli(capsys):
    from fp4_weight_only_gb300 import tune
    assert tune.main(["--m", "128", "--n", "8192", "--k", "8192", "--plan-only",
                      "--sms", str(SMS), "--pairs", str(PAIRS), "--json"]) == 0
    import json
    assert json.loads(capsys.readouterr().out) == binding.plan(128, 8192, 8192, "nvfp4", SMS, PAIRS)
    assert tune.main(["--m", "16", "--n", "1024", "--k", "1024", "--fmt", "mxfp4", "--plan-only",
                      "--sms", str(SMS), "--pairs", str(PAIRS)]) == 0
    assert capsys.readouterr().out.startswith("bn=16 ku=2 single ranges=32")
    # two 128-k chunks per unit only where k holds an even number of them
    assert (16, 2) in tune.candidates(1024) and (16, 2) not in tune.candidates(384)
    assert all(ku == 1 for _, ku in tune.candidates(1152))
