"""Thin ctypes binding of the C ABI in include/petit.h.

Argument marshalling only: every computation runs in the CUDA library.  The
functions take torch tensors for device memory and use torch's current CUDA
stream.  If the library cannot be built or loaded, :func:`load` raises --
there is no CPU fallback.
"""

import contextlib
import ctypes
import functools
import os
import threading

import torch

from . import build as _build

PETIT_FMT_NVFP4 = 0
PETIT_FMT_MXFP4 = 1
PETIT_FMT_NVFP4_F16 = 2
FORMATS = {"nvfp4": PETIT_FMT_NVFP4, "mxfp4": PETIT_FMT_MXFP4, "nvfp4_f16": PETIT_FMT_NVFP4_F16}

STATUS = {
    0: "PETIT_OK",
    1: "PETIT_ERR_INVALID_ARG",
    2: "PETIT_ERR_UNSUPPORTED_SHAPE",
    3: "PETIT_ERR_MISALIGNED",
    4: "PETIT_ERR_WORKSPACE",
    5: "PETIT_ERR_ARCH",
    6: "PETIT_ERR_CUDA",
    7: "PETIT_ERR_TIMEOUT",
    8: "PETIT_ERR_BOUNDS",
}

_lib = None
_lock = threading.Lock()

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_c_sz = ctypes.c_size_t


class PlanInfo(ctypes.Structure):
    """petit_plan_info_t"""
    _fields_ = [("bn", ctypes.c_int32), ("ku", ctypes.c_int32), ("cta_pairs", ctypes.c_int32),
                ("num_ranges", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("units_per_tile", ctypes.c_int32), ("num_tiles", ctypes.c_int64),
                ("units", ctypes.c_int64), ("workspace_bytes", ctypes.c_uint64)]


# name -> (restype, argtypes)
SIGNATURES = {
    "petit_layout_version": (ctypes.c_int, []),
    "petit_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "petit_repacked_bytes": (_c_sz, [_c_i64, _c_i64, ctypes.c_int]),
    "petit_gemm_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "petit_absmax_bf16": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_p]),
    "petit_nvfp4_global_scale": (ctypes.c_float, [ctypes.c_float]),
    "petit_quantize_nvfp4": (ctypes.c_int, [_c_p, ctypes.c_float, _c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_quantize_mxfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_repack_nvfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_repack_mxfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_repack_nvfp4_f16": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_dequant_f16": (ctypes.c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_gemm_f16_nvfp4": (ctypes.c_int, [_c_p, _c_p, ctypes.c_float, _c_p, _c_i64, _c_i64, _c_i64,
                                            _c_p, _c_sz, _c_p]),
    "petit_dequant_bf16": (ctypes.c_int, [_c_p, ctypes.c_int, _c_p, _c_i64, _c_i64, _c_p]),
    "petit_gemm_bf16_nvfp4": (ctypes.c_int, [_c_p, _c_p, ctypes.c_float, _c_p, _c_i64, _c_i64, _c_i64,
                                             _c_p, _c_sz, _c_p]),
    "petit_gemm_bf16_mxfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_sz,
                                             _c_p]),
    "petit_gemm_bf16_nvfp4_dscale": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                                    _c_p, _c_sz, _c_p]),
    "petit_gemm_bf16_nvfp4_noalloc": (ctypes.c_int, [_c_p, _c_p, ctypes.c_float, _c_p, _c_i64, _c_i64, _c_i64,
                                                     _c_p]),
    "petit_moe_workspace_bytes": (_c_sz, [_c_p, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "petit_moe_gemm_bf16_mxfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i64, _c_i64, _c_p,
                                                 _c_sz, _c_p]),
    "petit_moe_gemm_bf16_nvfp4": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i64, _c_i64,
                                                 _c_p, _c_sz, _c_p]),
    "petit_get_device_status": (ctypes.c_int, [_c_p, _c_sz, _c_p]),
    "petit_set_tile_config": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "petit_set_pair_mode": (ctypes.c_int, [ctypes.c_int]),
    "petit_bounds_checking": (ctypes.c_int, []),
    "petit_check_set_limits": (ctypes.c_int, [_c_i64, _c_i64]),
    "petit_selftest_timeout": (ctypes.c_int, [_c_p, _c_sz, ctypes.c_uint32, _c_p]),
    "petit_plan_gemm": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(PlanInfo), _c_p, _c_i64]),
    "petit_plan_moe": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_i64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.POINTER(PlanInfo), _c_p, _c_i64]),
    "petit_device_limits": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
}


class PetitError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def _open(path):
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(build=True):
    """Build (if stale) and load the CUDA library; raises on failure."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _open(_build.build() if build else _build.LIB)
    return _lib


_check_lib = None


def load_check(build=True):
    """Build (if stale) and load the bounds-checking build of the library
    (``_petit_check.so``: same API; the GEMM kernel checks every buffer
    index and copy and reports a failed check as PETIT_ERR_BOUNDS)."""
    global _check_lib
    with _lock:
        if _check_lib is None:
            _check_lib = _open(_build.build_check() if build else _build.CHECK_LIB)
    return _check_lib


@contextlib.contextmanager
def bounds_checked():
    """Inside the block every call of this module goes through the
    bounds-checking build (process-wide; not for concurrent use)."""
    global _lib
    chk = load_check()
    prev = load()
    _lib = chk
    try:
        yield chk
    finally:
        _lib = prev


def lib_path():
    return _build.LIB


def _check(status, where):
    if status != 0:
        raise PetitError(status, where)


# The raw handle of torch's current stream without building a Stream object
# (a per-call cost on the GEMM path); the public call where it is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return t.data_ptr()


def _need(t, dtype, name):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous CUDA {dtype} tensor")


# ---------------------------------------------------------------------- API
def layout_version():
    return load().petit_layout_version()


def absmax(x):
    """max |x| of a BF16 CUDA tensor, as a 1-element FP32 CUDA tensor."""
    _need(x, torch.bfloat16, "x")
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(load().petit_absmax_bf16(_ptr(x), x.numel(), _ptr(out), _stream()), "absmax")
    return out


def nvfp4_global_scale(amax):
    return float(load().petit_nvfp4_global_scale(ctypes.c_float(float(amax))))


def quantize(W, fmt="nvfp4", global_scale=1.0):
    """BF16 [n, k] -> (packed codes uint8 [n, k/2], scales uint8 [n, k/G])."""
    _need(W, torch.bfloat16, "W")
    n, k = W.shape
    group = 16 if fmt == "nvfp4" else 32
    wp = torch.empty((n, k // 2), dtype=torch.uint8, device=W.device)
    sp = torch.empty((n, max(k // group, 1)), dtype=torch.uint8, device=W.device)
    L = load()
    if fmt == "nvfp4":
        st = L.petit_quantize_nvfp4(_ptr(W), ctypes.c_float(global_scale), _ptr(wp), _ptr(sp), n, k, _stream())
    else:
        st = L.petit_quantize_mxfp4(_ptr(W), _ptr(wp), _ptr(sp), n, k, _stream())
    _check(st, "quantize_" + fmt)
    return wp, sp


def repack(w_packed, scales, fmt="nvfp4"):
    """Packed codes [n, k/2] + scales -> one repacked uint8 buffer."""
    _need(w_packed, torch.uint8, "w_packed")
    _need(scales, torch.uint8, "scales")
    n, half_k = w_packed.shape
    k = half_k * 2
    L = load()
    out = torch.empty(max(L.petit_repacked_bytes(n, k, FORMATS[fmt]), 1), dtype=torch.uint8,
                      device=w_packed.device)
    fn = {"nvfp4": L.petit_repack_nvfp4, "mxfp4": L.petit_repack_mxfp4,
          "nvfp4_f16": L.petit_repack_nvfp4_f16}[fmt]
    _check(fn(_ptr(w_packed), _ptr(scales), _ptr(out), n, k, _stream()), "repack_" + fmt)
    return out


def dequant(rep, n, k, fmt="nvfp4"):
    """Repacked weights -> Wq [n, k] (test hook; bit-exact): BF16, or FP16 for
    the "nvfp4_f16" layout."""
    if fmt == "nvfp4_f16":
        out = torch.empty((n, k), dtype=torch.float16, device=rep.device)
        _check(load().petit_dequant_f16(_ptr(rep), _ptr(out), n, k, _stream()), "dequant_f16")
        return out
    out = torch.empty((n, k), dtype=torch.bfloat16, device=rep.device)
    _check(load().petit_dequant_bf16(_ptr(rep), FORMATS[fmt], _ptr(out), n, k, _stream()), "dequant")
    return out


@functools.lru_cache(maxsize=1024)
def workspace_bytes(m, n, k, fmt="nvfp4"):
    return int(load().petit_gemm_workspace_bytes(m, n, k, FORMATS[fmt]))


class Workspace:
    """A zero-filled device workspace that grows on demand."""

    def __init__(self, device=None, nbytes=0):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes):
        if nbytes > self.buf.numel():
            self.buf = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
        return self.buf

    def status(self):
        """PETIT_OK (0) or the error the kernels recorded (clears it)."""
        return load().petit_get_device_status(_ptr(self.buf), self.buf.numel(), _stream())


def gemm(A, rep, n, fmt="nvfp4", global_scale=1.0, workspace=None, out=None):
    """C[m, n] = g * A @ dequant(W)^T in BF16 (FP32 accumulation).  For NVFP4,
    `global_scale` is a float or a one-element FP32 CUDA tensor (read by the
    kernel, so a CUDA graph picks up a changed value on replay).  With the
    "nvfp4_f16" layout, A and C are FP16."""
    act = torch.float16 if fmt == "nvfp4_f16" else torch.bfloat16
    _need(A, act, "A")
    m, k = A.shape
    ws = workspace or Workspace(A.device)
    need = workspace_bytes(m, n, k, fmt)
    if need == 0:
        raise PetitError(2, "gemm workspace size")
    buf = ws.ensure(need)
    C = out if out is not None else torch.empty((m, n), dtype=act, device=A.device)
    L = load()
    if fmt == "nvfp4_f16":
        st = L.petit_gemm_f16_nvfp4(_ptr(A), _ptr(rep), ctypes.c_float(global_scale), _ptr(C),
                                    m, n, k, _ptr(buf), buf.numel(), _stream())
    elif fmt == "nvfp4" and isinstance(global_scale, torch.Tensor):
        _need(global_scale, torch.float32, "global_scale")
        st = L.petit_gemm_bf16_nvfp4_dscale(_ptr(A), _ptr(rep), _ptr(global_scale), _ptr(C),
                                            m, n, k, _ptr(buf), buf.numel(), _stream())
    elif fmt == "nvfp4":
        st = L.petit_gemm_bf16_nvfp4(_ptr(A), _ptr(rep), ctypes.c_float(global_scale), _ptr(C),
                                     m, n, k, _ptr(buf), buf.numel(), _stream())
    else:
        st = L.petit_gemm_bf16_mxfp4(_ptr(A), _ptr(rep), _ptr(C), m, n, k, _ptr(buf), buf.numel(),
                                     _stream())
    _check(st, "gemm_" + fmt)
    return C


def moe_gemm(A, rep, expert_offsets, n, fmt="mxfp4", global_scales=None, workspace=None, out=None):
    """Grouped GEMM of an MoE layer: rows [off[e], off[e+1]) of A (BF16,
    grouped by expert) times expert e's weights; `rep` holds the experts'
    repacked weights back to back; `expert_offsets` is a host sequence of
    E + 1 ints; `global_scales` (NVFP4) a host sequence of E floats."""
    _need(A, torch.bfloat16, "A")
    T, k = A.shape
    off = (ctypes.c_int64 * len(expert_offsets))(*[int(x) for x in expert_offsets])
    E = len(expert_offsets) - 1
    if int(off[E]) != T:
        raise ValueError("expert_offsets[-1] must equal A.shape[0]")
    L = load()
    ws = workspace or Workspace(A.device)
    need = int(L.petit_moe_workspace_bytes(off, E, n, k, FORMATS[fmt]))
    if need == 0 and T > 0:
        raise PetitError(2, "moe workspace size")
    buf = ws.ensure(max(need, 256))
    C = out if out is not None else torch.empty((T, n), dtype=torch.bfloat16, device=A.device)
    if fmt == "mxfp4":
        st = L.petit_moe_gemm_bf16_mxfp4(_ptr(A), _ptr(rep), off, E, _ptr(C), n, k, _ptr(buf),
                                         buf.numel(), _stream())
    else:
        gs = (ctypes.c_float * E)(*[float(x) for x in (global_scales or [1.0] * E)])
        st = L.petit_moe_gemm_bf16_nvfp4(_ptr(A), _ptr(rep), gs, off, E, _ptr(C), n, k, _ptr(buf),
                                         buf.numel(), _stream())
    _check(st, "moe_gemm_" + fmt)
    return C


def set_tile_config(bn=0, ku=0):
    """Force the GEMM tile shape (bn activation rows, ku 128-k chunks per
    unit) for later calls in this process; (0, 0) restores the planner."""
    _check(load().petit_set_tile_config(int(bn), int(ku)), "set_tile_config")
    workspace_bytes.cache_clear()


def set_pair_mode(mode=0):
    """CTA pairs (cta_group::2) for 128/256-row tiles in later calls of this
    process: 0 where the planner expects a gain, 1 never, 2 wherever they
    apply."""
    _check(load().petit_set_pair_mode(int(mode)), "set_pair_mode")
    workspace_bytes.cache_clear()


_MAX_RANGES = 1025   # kernel grids have at most 1024 work ranges


def _limits(num_sms, pair_capacity):
    """The given SM count and pair capacity, the current device's for any left out."""
    if num_sms is None or pair_capacity is None:
        dev_sms, dev_pc = device_limits()
        num_sms = dev_sms if num_sms is None else num_sms
        pair_capacity = dev_pc if pair_capacity is None else pair_capacity
    return int(num_sms), int(pair_capacity)


def _plan_result(info, starts):
    d = {f: getattr(info, f) for f, _ in PlanInfo._fields_}
    d["cta_pairs"] = bool(d["cta_pairs"])
    d["range_starts"] = list(starts[:info.num_ranges + 1]) if info.num_ranges else []
    return d


def plan(m, n, k, fmt="nvfp4", num_sms=None, pair_capacity=None):
    """The plan of a GEMM (tile shape, CTA pairs, work units and ranges,
    workspace bytes) on a device with num_sms SMs and pair_capacity resident
    CTA pairs; by default the current device's (petit_device_limits).  With
    both given, no GPU is needed."""
    L = load()
    num_sms, pair_capacity = _limits(num_sms, pair_capacity)
    info = PlanInfo()
    starts = (ctypes.c_int64 * _MAX_RANGES)()
    _check(L.petit_plan_gemm(int(m), int(n), int(k), FORMATS[fmt], num_sms, pair_capacity,
                             ctypes.byref(info), starts, _MAX_RANGES), "plan_gemm")
    return _plan_result(info, starts)


def moe_plan(expert_offsets, n, k, fmt="mxfp4", num_sms=None, pair_capacity=None):
    """:func:`plan` for the grouped MoE GEMM (expert_offsets: E + 1 row offsets)."""
    L = load()
    num_sms, pair_capacity = _limits(num_sms, pair_capacity)
    E = len(expert_offsets) - 1
    off = (ctypes.c_int64 * (E + 1))(*[int(x) for x in expert_offsets])
    info = PlanInfo()
    starts = (ctypes.c_int64 * _MAX_RANGES)()
    _check(L.petit_plan_moe(off, E, int(n), int(k), FORMATS[fmt], num_sms, pair_capacity,
                            ctypes.byref(info), starts, _MAX_RANGES), "plan_moe")
    return _plan_result(info, starts)


def device_limits():
    """(SM count, resident CTA pairs) of the current device, as the GEMMs plan with."""
    sms, pc = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().petit_device_limits(ctypes.byref(sms), ctypes.byref(pc)), "device_limits")
    return sms.value, pc.value


def selftest_timeout(workspace, timeout_us=1000):
    _check(load().petit_selftest_timeout(_ptr(workspace.buf), workspace.buf.numel(), timeout_us, _stream()),
           "selftest_timeout")


class FP4Weight:
    """Offline-prepared FP4 weight: quantised, repacked, ready for gemm()."""

    def __init__(self, W, fmt="nvfp4", global_scale=None):
        n, k = W.shape
        self.n, self.k, self.fmt = n, k, fmt
        if fmt in ("nvfp4", "nvfp4_f16"):
            if global_scale is None:
                global_scale = 1.0
            elif global_scale == "amax":
                global_scale = nvfp4_global_scale(absmax(W).item())
            self.global_scale = float(global_scale)
        else:
            self.global_scale = 1.0
        w_packed, scales = quantize(W, "mxfp4" if fmt == "mxfp4" else "nvfp4", self.global_scale)
        self.rep = repack(w_packed, scales, fmt)

    def __call__(self, A, workspace=None, out=None):
        return gemm(A, self.rep, self.n, self.fmt, self.global_scale, workspace, out)
