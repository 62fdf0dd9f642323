"""C-ABI library: builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments before touching the device (no compute calls)."""

import ctypes
import os
import re

import pytest

from fp4_weight_only_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "petit.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(petit_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("petit_repack_nvfp4", "petit_repack_mxfp4", "petit_gemm_bf16_nvfp4",
                     "petit_gemm_bf16_mxfp4", "petit_dequant_bf16", "petit_gemm_workspace_bytes",
                     "petit_get_device_status", "petit_layout_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(binding.SIGNATURES), "binding signatures out of date with the header"


def test_host_only_entry_points(lib):
    assert lib.petit_layout_version() >= 1
    for s in range(9):
        assert lib.petit_status_string(s)
    assert lib.petit_status_string(8) == b"device-side index check failed"
    assert lib.petit_status_string(99) == b"unknown status"
    assert lib.petit_repacked_bytes(8192, 8192, 0) == 8192 * 4096 + 8192 * 512
    # MXFP4: codes, scales and a 16-byte flag field per 128 x 128 chunk
    assert lib.petit_repacked_bytes(8192, 8192, 1) == 8192 * 4096 + 8192 * 256 + 64 * 64 * 16
    assert lib.petit_repacked_bytes(8192, 8192, 7) == 0
    assert lib.petit_nvfp4_global_scale(ctypes.c_float(2688.0)) == 1.0


P = ctypes.c_void_p


def test_argument_validation_without_gpu(lib):
    a = P(0x10000)        # aligned fake addresses: validation must reject before any use
    bad = P(0x10008)
    NULL = P(0)
    s = P(0)
    # null pointer / m < 1
    assert lib.petit_gemm_bf16_nvfp4(NULL, a, 1.0, a, 16, 1024, 1024, a, 1 << 20, s) == 1
    assert lib.petit_gemm_bf16_nvfp4(a, a, 1.0, a, 0, 1024, 1024, a, 1 << 20, s) == 1
    assert lib.petit_gemm_bf16_nvfp4(a, a, -1.0, a, 16, 1024, 1024, a, 1 << 20, s) == 1
    # shapes: n, k multiples of 128
    assert lib.petit_gemm_bf16_nvfp4(a, a, 1.0, a, 16, 1000, 1024, a, 1 << 20, s) == 2
    assert lib.petit_gemm_bf16_mxfp4(a, a, a, 16, 1024, 1056, a, 1 << 20, s) == 2
    # alignment
    assert lib.petit_gemm_bf16_nvfp4(bad, a, 1.0, a, 16, 1024, 1024, a, 1 << 20, s) == 3
    # workspace missing
    assert lib.petit_gemm_bf16_mxfp4(a, a, a, 16, 1024, 1024, NULL, 0, s) == 4
    assert lib.petit_repack_nvfp4(a, a, a, 100, 1024, s) == 2
    assert lib.petit_repack_mxfp4(a, NULL, a, 128, 128, s) == 1
    assert lib.petit_dequant_bf16(a, 5, a, 128, 128, s) == 1
    assert lib.petit_quantize_nvfp4(a, ctypes.c_float(0.0), a, a, 4, 32, s) == 1
    assert lib.petit_quantize_mxfp4(a, a, a, 4, 48, s) == 2
    assert lib.petit_absmax_bf16(a, 0, a, s) == 1
    assert lib.petit_selftest_timeout(a, 16, 100, s) == 4
    assert lib.petit_selftest_timeout(a, 256, 0, s) == 1
    assert lib.petit_get_device_status(NULL, 4608, s) == 1
    assert lib.petit_get_device_status(a, 16, s) == 1
    # sizes are 0 for invalid shapes
    assert lib.petit_gemm_workspace_bytes(16, 1000, 1024, 0) == 0
    assert lib.petit_gemm_workspace_bytes(0, 1024, 1024, 0) == 0


def test_no_device_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = P(0x10000)
    # valid arguments, but no usable device: a CUDA error status, never a crash
    assert lib.petit_gemm_bf16_nvfp4(a, a, 1.0, a, 16, 1024, 1024, a, 1 << 30, P(0)) == 6
    assert lib.petit_gemm_workspace_bytes(16, 1024, 1024, 0) == 0


def test_pair_mode_validation(lib):
    for mode in (0, 1, 2):
        assert lib.petit_set_pair_mode(mode) == 0
    assert lib.petit_set_pair_mode(3) == 1
    assert lib.petit_set_pair_mode(-1) == 1
    assert lib.petit_set_pair_mode(0) == 0


def test_tile_config_override_validation(lib):
    assert lib.petit_set_tile_config(48, 1) == 1
    assert lib.petit_set_tile_config(128, 2) == 1
    assert lib.petit_set_tile_config(16, 3) == 1
    assert lib.petit_set_tile_config(256, 1) == 0
    assert lib.petit_set_tile_config(0, 0) == 0


def test_bounds_checking_build_loads_and_differs_only_in_checks(lib):
    """The bounds-checking build (_petit_check.so) has the same ABI; only it
    accepts test limits for its index checks."""
    chk = binding.load_check()
    names = declared_functions()
    assert not [n for n in names if not hasattr(chk, n)]
    assert lib.petit_bounds_checking() == 0
    assert chk.petit_bounds_checking() == 1
    assert lib.petit_check_set_limits(1024, -1) == 1    # normal build: no checks to limit
    assert chk.petit_check_set_limits(1024, -1) == 0
    assert chk.petit_check_set_limits(-1, -1) == 0
    assert chk.petit_layout_version() == lib.petit_layout_version()
    assert chk.petit_repacked_bytes(4096, 4096, 1) == lib.petit_repacked_bytes(4096, 4096, 1)


def test_binding_has_no_cpu_fallback(lib):
    """The Python entry points refuse host tensors instead of computing on
    the CPU, and with no GPU the device queries fail with a status."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = torch.zeros(16, 1024, dtype=torch.bfloat16)
    rep = torch.zeros(binding.load().petit_repacked_bytes(1024, 1024, 0), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        binding.gemm(a, rep, 1024, "nvfp4")
    with pytest.raises(ValueError, match="CUDA"):
        binding.quantize(torch.zeros(128, 128, dtype=torch.bfloat16), "nvfp4")
    with pytest.raises(ValueError, match="CUDA"):
        binding.FP4Weight(torch.zeros(128, 128, dtype=torch.bfloat16), "mxfp4")
    with pytest.raises(binding.PetitError) as e:
        binding.device_limits()
    assert e.value.status == 6
    # the plan itself needs no device
    assert binding.plan(16, 1024, 1024, "nvfp4", num_sms=152, pair_capacity=76)["bn"] == 16
