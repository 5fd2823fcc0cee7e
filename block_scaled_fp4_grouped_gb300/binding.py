"""ctypes binding of libnvfp4_ggemm.so (include/nvfp4_ggemm.h).

Argument marshalling only: every function here forwards to the C entry point
of the same name; all compute runs in the library's CUDA kernels. The
library must be built (`python -m block_scaled_fp4_grouped_gb300.build`);
loading fails loudly otherwise. There is no CPU fallback.

`GroupedGemm` is a convenience wrapper that takes lists of torch tensors and
the current torch stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
# NVFP4_GGEMM_LIB names another build of the library to load instead (for
# example the device-check build, libnvfp4_ggemm_debug.so)
LIB_PATH = os.environ.get("NVFP4_GGEMM_LIB") or os.path.join(_PKG, "libnvfp4_ggemm.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libnvfp4_ggemm_debug.so")

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_ALIGNMENT = 2
NVFP4_ERR_UNSUPPORTED_SHAPE = 3
NVFP4_ERR_UNSUPPORTED_DEVICE = 4
NVFP4_ERR_CUDA = 5
NVFP4_ERR_TIMEOUT = 6
NVFP4_ERR_DEVICE_FAULT = 7
NVFP4_ERR_NOT_PREPARED = 8

NVFP4_SF_RAW = 0
NVFP4_SF_ATOM = 1
NVFP4_SF_FUSED = 0
NVFP4_SF_RELAYOUT = 1

# Every function the header declares (checked by the CPU tests).
EXPORTED = (
    "nvfp4_ggemm_default_options",
    "nvfp4_ggemm_plan",
    "nvfp4_ggemm_run",
    "nvfp4_ggemm_run_host",
    "nvfp4_ggemm_prepare_b_scales",
    "nvfp4_ggemm_sync_status",
    "nvfp4_ggemm_destroy",
    "nvfp4_sf_relayout",
    "nvfp4_sf_atom_bytes",
    "nvfp4_ggemm_plan_info",
    "nvfp4_status_string",
    "nvfp4_ggemm_version",
    "nvfp4_ggemm_run_noalloc",
    "nvfp4_ggemm_schedule",
    "nvfp4_ggemm_schedule_units",
    "nvfp4_ggemm_plan_shapes",
    "nvfp4_ggemm_run_strided",
    "nvfp4_ggemm_plan_batched",
    "nvfp4_ggemm_run_batched",
)


class nvfp4_ggemm_options_t(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("sf_layout", ctypes.c_int32),
        ("sf_path", ctypes.c_int32),
        ("cache_b_scales", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_uint64),
        ("tile_n", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32),
        ("debug_skip_load", ctypes.c_int32),
        ("b_stages", ctypes.c_int32),
        ("a_stages", ctypes.c_int32),
        ("serial_launch", ctypes.c_int32),
        ("b_static", ctypes.c_int32),
        ("debug_check_fail", ctypes.c_int32),
        ("row_units", ctypes.c_int32),
    ]


class nvfp4_ggemm_plan_info_t(ctypes.Structure):
    _fields_ = [
        ("tile_n", ctypes.c_int32),
        ("b_stages", ctypes.c_int32),
        ("a_stages", ctypes.c_int32),
        ("chunks", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("sm_count", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("kernels_per_run", ctypes.c_int32),
        ("sf_path", ctypes.c_int32),
        ("row_units", ctypes.c_int32),
        ("split_acc", ctypes.c_int32),
    ]


class NativeLibraryMissing(RuntimeError):
    pass


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {nvfp4_status_string(status)} (status {status})")


_lib = None
_VP = ctypes.c_void_p
_VPP = ctypes.POINTER(ctypes.c_void_p)


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once). Raises NativeLibraryMissing when it
    has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise NativeLibraryMissing(
            f"{LIB_PATH} is missing: build it with `python -m block_scaled_fp4_grouped_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    L.nvfp4_ggemm_default_options.restype = None
    L.nvfp4_ggemm_default_options.argtypes = [ctypes.POINTER(nvfp4_ggemm_options_t)]
    L.nvfp4_ggemm_plan.restype = ctypes.c_int
    L.nvfp4_ggemm_plan.argtypes = [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                                   ctypes.POINTER(nvfp4_ggemm_options_t)]
    for fn in ("nvfp4_ggemm_run", "nvfp4_ggemm_run_host"):
        f = getattr(L, fn)
        f.restype = ctypes.c_int
        f.argtypes = [_VP, _VPP, _VPP, _VPP, _VPP, _VPP, _VP]
    L.nvfp4_ggemm_prepare_b_scales.restype = ctypes.c_int
    L.nvfp4_ggemm_prepare_b_scales.argtypes = [_VP, _VPP, _VP]
    L.nvfp4_ggemm_sync_status.restype = ctypes.c_int
    L.nvfp4_ggemm_sync_status.argtypes = [_VP, _VP, ctypes.POINTER(ctypes.c_uint32)]
    L.nvfp4_ggemm_destroy.restype = ctypes.c_int
    L.nvfp4_ggemm_destroy.argtypes = [_VP]
    L.nvfp4_sf_relayout.restype = ctypes.c_int
    L.nvfp4_sf_relayout.argtypes = [_VP, _VP, ctypes.c_int32, ctypes.c_int32, _VP]
    L.nvfp4_sf_atom_bytes.restype = ctypes.c_uint64
    L.nvfp4_sf_atom_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.nvfp4_ggemm_plan_info.restype = ctypes.c_int
    L.nvfp4_ggemm_plan_info.argtypes = [_VP, ctypes.POINTER(nvfp4_ggemm_plan_info_t)]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    L.nvfp4_status_string.argtypes = [ctypes.c_int]
    L.nvfp4_ggemm_version.restype = ctypes.c_int
    L.nvfp4_ggemm_version.argtypes = []
    L.nvfp4_ggemm_run_noalloc.restype = ctypes.c_int
    L.nvfp4_ggemm_run_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                          ctypes.c_int32, _VPP, _VPP, _VPP, _VPP, _VPP, _VP,
                                          ctypes.POINTER(ctypes.c_uint32)]
    L.nvfp4_ggemm_schedule.restype = ctypes.c_int
    L.nvfp4_ggemm_schedule.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.nvfp4_ggemm_schedule_units.restype = ctypes.c_int
    L.nvfp4_ggemm_schedule_units.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.nvfp4_ggemm_run_strided.restype = ctypes.c_int
    L.nvfp4_ggemm_run_strided.argtypes = [_VP, _VPP, _VPP, _VPP, _VPP, _VPP, ctypes.POINTER(ctypes.c_int32), _VP]
    L.nvfp4_ggemm_plan_shapes.restype = ctypes.c_int
    L.nvfp4_ggemm_plan_shapes.argtypes = [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]
    L.nvfp4_ggemm_plan_batched.restype = ctypes.c_int
    L.nvfp4_ggemm_plan_batched.argtypes = [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int, ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]
    L.nvfp4_ggemm_run_batched.restype = ctypes.c_int
    L.nvfp4_ggemm_run_batched.argtypes = [_VP, _VPP, _VPP, _VPP, _VPP, _VPP, ctypes.POINTER(ctypes.c_int64), _VP]
    _lib = L
    return L


# ----------------------------------------------------------------- marshalling

def _ptr(x) -> int:
    """Address of a torch tensor, numpy array, ctypes object or integer."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    if isinstance(x, ctypes.c_void_p):
        return int(x.value or 0)
    raise TypeError(f"cannot take the address of {type(x)!r}")


def _ptr_array(xs: Optional[Sequence]):
    if xs is None:
        return None
    arr = (ctypes.c_void_p * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x) or None
    return arr


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:
            pass
        return 0
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    return int(stream)


# ------------------------------------------------------------- C entry points

def nvfp4_ggemm_default_options() -> nvfp4_ggemm_options_t:
    opt = nvfp4_ggemm_options_t()
    lib().nvfp4_ggemm_default_options(ctypes.byref(opt))
    return opt


def _i32_array(vals: Sequence[int]):
    return (ctypes.c_int32 * max(1, len(vals)))(*[int(v) for v in vals])


def nvfp4_ggemm_plan(device: int, M: Sequence[int], N, K,
                     opt: Optional[nvfp4_ggemm_options_t] = None) -> Tuple[int, Optional[int]]:
    """N and K: one value for every group (nvfp4_ggemm_plan) or one per group
    (nvfp4_ggemm_plan_shapes)."""
    handle = _VP()
    m = _i32_array(M)
    o = ctypes.byref(opt) if opt is not None else None
    if isinstance(N, (list, tuple)) or isinstance(K, (list, tuple)):
        Ns = list(N) if isinstance(N, (list, tuple)) else [int(N)] * len(M)
        Ks = list(K) if isinstance(K, (list, tuple)) else [int(K)] * len(M)
        st = lib().nvfp4_ggemm_plan_shapes(ctypes.byref(handle), int(device), len(M), m, _i32_array(Ns),
                                           _i32_array(Ks), o)
    else:
        st = lib().nvfp4_ggemm_plan(ctypes.byref(handle), int(device), len(M), m, int(N), int(K), o)
    return st, (handle.value if st == NVFP4_OK else None)


def nvfp4_ggemm_run(plan: int, A, B, SFA, SFB, C, stream=None) -> int:
    return lib().nvfp4_ggemm_run(plan, _ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB),
                                 _ptr_array(C), _stream(stream))


def nvfp4_ggemm_plan_batched(device: int, M: Sequence[int], N, K, batch: int,
                             opt: Optional[nvfp4_ggemm_options_t] = None) -> Tuple[int, Optional[int]]:
    """A plan of len(M) groups of `batch` problems each; N and K one value or one per group."""
    handle = _VP()
    Ns = list(N) if isinstance(N, (list, tuple)) else [int(N)] * len(M)
    Ks = list(K) if isinstance(K, (list, tuple)) else [int(K)] * len(M)
    o = ctypes.byref(opt) if opt is not None else None
    st = lib().nvfp4_ggemm_plan_batched(ctypes.byref(handle), int(device), len(M), int(batch), _i32_array(M),
                                        _i32_array(Ns), _i32_array(Ks), o)
    return st, (handle.value if st == NVFP4_OK else None)


def nvfp4_ggemm_run_batched(plan: int, A, B, SFA, SFB, C, batch_stride: Sequence[int], stream=None) -> int:
    """One pointer per group (its batch 0) and 5 byte strides per group:
    A, B, SFA, SFB, C."""
    strides = (ctypes.c_int64 * max(1, len(batch_stride)))(*[int(v) for v in batch_stride])
    return lib().nvfp4_ggemm_run_batched(plan, _ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB),
                                         _ptr_array(C), strides, _stream(stream))


def nvfp4_ggemm_run_strided(plan: int, A, B, SFA, SFB, C, ldc: Sequence[int], stream=None) -> int:
    """nvfp4_ggemm_run with a row stride (fp16 elements) for every C[g]."""
    return lib().nvfp4_ggemm_run_strided(plan, _ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB),
                                         _ptr_array(C), _i32_array(ldc), _stream(stream))


def nvfp4_ggemm_run_host(plan: int, A, B, SFA, SFB, C, stream=None) -> int:
    return lib().nvfp4_ggemm_run_host(plan, _ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB),
                                      _ptr_array(C), _stream(stream))


def nvfp4_ggemm_prepare_b_scales(plan: int, SFB, stream=None) -> int:
    return lib().nvfp4_ggemm_prepare_b_scales(plan, _ptr_array(SFB), _stream(stream))


def nvfp4_ggemm_sync_status(plan: int, stream=None) -> Tuple[int, int]:
    detail = ctypes.c_uint32(0)
    st = lib().nvfp4_ggemm_sync_status(plan, _stream(stream), ctypes.byref(detail))
    return st, int(detail.value)


def nvfp4_ggemm_destroy(plan: Optional[int]) -> int:
    return lib().nvfp4_ggemm_destroy(plan)


def nvfp4_sf_relayout(src, dst, rows: int, K: int, stream=None) -> int:
    return lib().nvfp4_sf_relayout(_ptr(src), _ptr(dst), int(rows), int(K), _stream(stream))


def nvfp4_sf_atom_bytes(rows: int, K: int) -> int:
    return int(lib().nvfp4_sf_atom_bytes(int(rows), int(K)))


def nvfp4_ggemm_plan_info(plan: int) -> nvfp4_ggemm_plan_info_t:
    info = nvfp4_ggemm_plan_info_t()
    st = lib().nvfp4_ggemm_plan_info(plan, ctypes.byref(info))
    if st != NVFP4_OK:
        raise Nvfp4Error(st, "nvfp4_ggemm_plan_info")
    return info


def nvfp4_status_string(status: int) -> str:
    try:
        return lib().nvfp4_status_string(int(status)).decode()
    except NativeLibraryMissing:
        return f"status {status}"


def nvfp4_ggemm_version() -> int:
    return int(lib().nvfp4_ggemm_version())


def nvfp4_ggemm_run_noalloc(M: Sequence[int], N: int, K: int, A, B, SFA, SFB, C, stream=None,
                            wait: bool = False) -> Tuple[int, int]:
    """The allocation-free grouped GEMM on the current device (raw scales).
    With wait=True the call waits for the stream and also returns the device
    error word. Returns (status, error word)."""
    m = (ctypes.c_int32 * max(1, len(M)))(*[int(v) for v in M])
    word = ctypes.c_uint32(0)
    st = lib().nvfp4_ggemm_run_noalloc(len(M), m, int(N), int(K), _ptr_array(A), _ptr_array(B),
                                       _ptr_array(SFA), _ptr_array(SFB), _ptr_array(C), _stream(stream),
                                       ctypes.byref(word) if wait else None)
    return st, int(word.value)


def nvfp4_ggemm_schedule(M: Sequence[int], N, tile_n: int = 0, max_ctas: int = 148, K=256) -> Tuple[int, List[int]]:
    """Per-CTA chunk ranges a plan would use (host only). N and K: one value
    for every group or one per group. Returns (status, cta_begin[0..grid])."""
    Ns = list(N) if isinstance(N, (list, tuple)) else [int(N)] * len(M)
    Ks = list(K) if isinstance(K, (list, tuple)) else [int(K)] * len(M)
    out = (ctypes.c_int32 * (max(1, int(max_ctas)) + 1))()
    grid = ctypes.c_int32(0)
    st = lib().nvfp4_ggemm_schedule(len(M), _i32_array(M), _i32_array(Ns), _i32_array(Ks), int(tile_n),
                                    int(max_ctas), out, ctypes.byref(grid))
    if st != NVFP4_OK:
        return st, []
    return st, [int(out[i]) for i in range(grid.value + 1)] if grid.value > 0 else [0]


def nvfp4_ggemm_schedule_units(M: Sequence[int], N, tile_n: int = 0, max_ctas: int = 148, K=256,
                               row_units: int = 0) -> Tuple[int, List[int], int, int]:
    """Per-CTA chunk ranges for units of row_units 128-row tiles (0: the
    plan's own choice). Returns (status, cta_begin[0..grid], units, split_acc)."""
    Ns = list(N) if isinstance(N, (list, tuple)) else [int(N)] * len(M)
    Ks = list(K) if isinstance(K, (list, tuple)) else [int(K)] * len(M)
    out = (ctypes.c_int32 * (max(1, int(max_ctas)) + 1))()
    grid, units, split = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().nvfp4_ggemm_schedule_units(len(M), _i32_array(M), _i32_array(Ns), _i32_array(Ks), int(tile_n),
                                          int(max_ctas), int(row_units), out, ctypes.byref(grid),
                                          ctypes.byref(units), ctypes.byref(split))
    if st != NVFP4_OK:
        return st, [], 0, 0
    cb = [int(out[i]) for i in range(grid.value + 1)] if grid.value > 0 else [0]
    return st, cb, int(units.value), int(split.value)


# -------------------------------------------------------------- convenience

def make_options(sf_layout: str = "raw", sf_path: str = "fused", cache_b_scales: bool = False,
                 wait_timeout_ns: int = 0, tile_n: int = 0, max_ctas: int = 0,
                 debug_skip_load: int = 0, b_stages: int = 0, a_stages: int = 0,
                 serial_launch: bool = False, b_static: int = 0,
                 debug_check_fail: int = 0, row_units: int = 0) -> nvfp4_ggemm_options_t:
    opt = nvfp4_ggemm_default_options()
    opt.sf_layout = {"raw": NVFP4_SF_RAW, "atom": NVFP4_SF_ATOM}[sf_layout]
    opt.sf_path = {"fused": NVFP4_SF_FUSED, "relayout": NVFP4_SF_RELAYOUT}[sf_path]
    opt.cache_b_scales = 1 if cache_b_scales else 0
    if wait_timeout_ns:
        opt.wait_timeout_ns = int(wait_timeout_ns)
    opt.tile_n = int(tile_n)
    opt.max_ctas = int(max_ctas)
    opt.debug_skip_load = int(debug_skip_load)
    opt.b_stages = int(b_stages)
    opt.a_stages = int(a_stages)
    opt.serial_launch = 1 if serial_launch else 0
    opt.b_static = int(b_static)  # False/True = 0/1; 2 = every input static
    opt.debug_check_fail = int(debug_check_fail)
    opt.row_units = int(row_units)
    return opt


class GroupedGemm:
    """A plan plus calls on torch tensors (lists of per-group tensors).

    A[g] uint8 [M_g, K/2], B[g] uint8 [N, K/2], SFA[g] / SFB[g] uint8 scale
    codes (raw [rows, K/16] or atom layout), C[g] float16 [M_g, N]."""

    def __init__(self, M: Sequence[int], N: int, K: int, device: int = 0, batch: int = 1, **options):
        self.M = [int(m) for m in M]
        # N and K: one value for every group, or one per group
        self.N = [int(n) for n in N] if isinstance(N, (list, tuple)) else int(N)
        self.K = [int(k) for k in K] if isinstance(K, (list, tuple)) else int(K)
        self.batch = int(batch)
        self.opt = make_options(**options)
        if self.batch != 1:
            st, handle = nvfp4_ggemm_plan_batched(device, self.M, self.N, self.K, self.batch, self.opt)
        else:
            st, handle = nvfp4_ggemm_plan(device, self.M, self.N, self.K, self.opt)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_plan")
        self.handle = handle

    def info(self) -> nvfp4_ggemm_plan_info_t:
        return nvfp4_ggemm_plan_info(self.handle)

    def run(self, A, B, SFA, SFB, C, stream=None) -> None:
        st = nvfp4_ggemm_run(self.handle, A, B, SFA, SFB, C, stream)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_run")

    def run_strided(self, A, B, SFA, SFB, C, ldc, stream=None) -> None:
        st = nvfp4_ggemm_run_strided(self.handle, A, B, SFA, SFB, C, ldc, stream)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_run_strided")

    def run_batched(self, A, B, SFA, SFB, C, batch_stride: Sequence[int], stream=None) -> None:
        st = nvfp4_ggemm_run_batched(self.handle, A, B, SFA, SFB, C, batch_stride, stream)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_run_batched")

    def bind(self, A, B, SFA, SFB, C, ldc: Optional[Sequence[int]] = None) -> "BoundCall":
        """Marshal one set of per-group buffers once, for repeated calls on
        them (the per-call cost is then one C call)."""
        return BoundCall(self, A, B, SFA, SFB, C, ldc)

    def bind_host(self, A, B, SFA, SFB, C) -> "BoundCall":
        """bind for nvfp4_ggemm_run_host: host buffers marshalled once."""
        return BoundCall(self, A, B, SFA, SFB, C, host=True)

    def run_host(self, A, B, SFA, SFB, C, stream=None) -> None:
        st = nvfp4_ggemm_run_host(self.handle, A, B, SFA, SFB, C, stream)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_run_host")

    def prepare_b_scales(self, SFB, stream=None) -> None:
        st = nvfp4_ggemm_prepare_b_scales(self.handle, SFB, stream)
        if st != NVFP4_OK:
            raise Nvfp4Error(st, "nvfp4_ggemm_prepare_b_scales")

    def sync_status(self, stream=None) -> Tuple[int, int]:
        return nvfp4_ggemm_sync_status(self.handle, stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            nvfp4_ggemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class BoundCall:
    """nvfp4_ggemm_run (or _run_strided, or _run_host) on one fixed set of
    buffers: the pointer arrays are built once and the tensors are kept
    alive for as long as this object is."""

    def __init__(self, gemm: GroupedGemm, A, B, SFA, SFB, C, ldc=None, host: bool = False):
        self.gemm = gemm
        self.host = host
        self._keep = (A, B, SFA, SFB, C)
        self._args = (_ptr_array(A), _ptr_array(B), _ptr_array(SFA), _ptr_array(SFB), _ptr_array(C))
        self._ldc = _i32_array(ldc) if ldc is not None else None

    def __call__(self, stream=None) -> None:
        L = lib()
        if self.host:
            st = L.nvfp4_ggemm_run_host(self.gemm.handle, *self._args, _stream(stream))
            name = "nvfp4_ggemm_run_host"
        elif self._ldc is None:
            st = L.nvfp4_ggemm_run(self.gemm.handle, *self._args, _stream(stream))
            name = "nvfp4_ggemm_run"
        else:
            st = L.nvfp4_ggemm_run_strided(self.gemm.handle, *self._args, self._ldc, _stream(stream))
            name = "nvfp4_ggemm_run_strided"
        if st != NVFP4_OK:
            raise Nvfp4Error(st, name)
