"""CPU oracle for the NVFP4 block-scaled grouped GEMM (plain C, fp64).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package; the library under
`block_scaled_fp4_grouped_gb300/` never does, and it shares no code with it.

The C source (`nvfp4_oracle.c`) is the definition written out:
C_g = RN_fp16(sum_k e2m1(A)*e4m3(SFA)*e2m1(B)*e4m3(SFB)) with fp64 sums in
ascending k and one direct fp64 -> fp16 rounding (the custom_kernel
docstring of submission 503584 fixes shapes and dtypes).

Every function here is pinned by `tests/test_oracle.py` against things
other than itself: torch's float8_e4m3fn decoding, numpy's float16 rounding,
exact rational arithmetic on tiny inputs, numpy fp64 matmul where the sum is
provably exact, closed-form E2M1 values, invariants, and the CuTe atom
layout printed by submission 402102.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")


def build(mutant: int = 0, out: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc and return its path.

    `mutant` > 0 plants one deliberate mistake (see the C source); only the
    test that checks the pins catch mistakes builds those."""
    os.makedirs(_BUILD, exist_ok=True)
    if out is None:
        out = os.path.join(_BUILD, "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so")
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)


def _ptr(a: Optional[np.ndarray], t):
    if a is None:
        return ctypes.cast(None, t)
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes front end of one oracle build."""

    def __init__(self, path: Optional[str] = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        lib.oracle_init.restype = None
        lib.oracle_e2m1.restype = ctypes.c_double
        lib.oracle_e2m1.argtypes = [ctypes.c_int]
        lib.oracle_e4m3.restype = ctypes.c_double
        lib.oracle_e4m3.argtypes = [ctypes.c_int]
        lib.oracle_fp16_rne.restype = ctypes.c_uint16
        lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
        lib.oracle_fp16_rne_array.restype = None
        lib.oracle_fp16_rne_array.argtypes = [ctypes.c_long, _f64p, _u16p]
        lib.oracle_group_gemm.restype = ctypes.c_int
        lib.oracle_group_gemm.argtypes = [ctypes.c_int] * 3 + [_u8p] * 4 + [_u16p, _f64p, ctypes.c_int]
        lib.oracle_group_entries.restype = ctypes.c_int
        lib.oracle_group_entries.argtypes = ([ctypes.c_int] * 3 + [_u8p] * 4 +
                                             [ctypes.c_int, _i32p, _i32p, _u16p, _f64p])
        lib.oracle_sf_relayout.restype = ctypes.c_int
        lib.oracle_sf_relayout.argtypes = [ctypes.c_int, ctypes.c_int, _u8p, _u8p]
        lib.oracle_mutant_id.restype = ctypes.c_int
        lib.oracle_init()
        self.lib = lib

    # -- scalar pieces ------------------------------------------------------
    def e2m1(self, code: int) -> float:
        return self.lib.oracle_e2m1(int(code))

    def e4m3(self, code: int) -> float:
        return self.lib.oracle_e4m3(int(code))

    def fp16_rne(self, x) -> np.ndarray:
        """fp64 -> fp16 bit patterns (uint16), rounding to nearest even."""
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_fp16_rne_array(a.size, _ptr(a, _f64p), _ptr(out, _u16p))
        return out.reshape(np.shape(x))

    # -- one group ------------------------------------------------------------
    def group_gemm(self, A: np.ndarray, B: np.ndarray, SFA: np.ndarray, SFB: np.ndarray,
                   K: int, want_exact: bool = False, nthreads: int = 0
                   ) -> Tuple[np.ndarray, Optional[np.ndarray], int]:
        """Returns (C fp16 [M,N] as float16, fp64 sums or None, exact flag)."""
        M, N = int(A.shape[0]), int(B.shape[0])
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
        SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
        assert A.shape == (M, K // 2) and B.shape == (N, K // 2)
        assert SFA.shape == (M, K // 16) and SFB.shape == (N, K // 16)
        C = np.empty((M, N), dtype=np.uint16)
        X = np.empty((M, N), dtype=np.float64) if want_exact else None
        rc = self.lib.oracle_group_gemm(M, N, K, _ptr(A, _u8p), _ptr(B, _u8p), _ptr(SFA, _u8p),
                                        _ptr(SFB, _u8p), _ptr(C, _u16p), _ptr(X, _f64p), int(nthreads))
        if rc < 0:
            raise ValueError(f"oracle_group_gemm failed ({rc})")
        return C.view(np.float16), X, rc

    def group_entries(self, A, B, SFA, SFB, K: int, rows: Sequence[int], cols: Sequence[int]
                      ) -> Tuple[np.ndarray, np.ndarray]:
        M, N = int(A.shape[0]), int(B.shape[0])
        r = np.ascontiguousarray(rows, dtype=np.int32)
        c = np.ascontiguousarray(cols, dtype=np.int32)
        o16 = np.empty(r.shape, dtype=np.uint16)
        ox = np.empty(r.shape, dtype=np.float64)
        rc = self.lib.oracle_group_entries(M, N, K, _ptr(np.ascontiguousarray(A), _u8p),
                                           _ptr(np.ascontiguousarray(B), _u8p),
                                           _ptr(np.ascontiguousarray(SFA), _u8p),
                                           _ptr(np.ascontiguousarray(SFB), _u8p),
                                           int(r.size), _ptr(r, _i32p), _ptr(c, _i32p),
                                           _ptr(o16, _u16p), _ptr(ox, _f64p))
        if rc < 0:
            raise ValueError("oracle_group_entries: bad argument")
        return o16.view(np.float16), ox

    # -- whole grouped problem ------------------------------------------------
    def grouped(self, prob, want_exact: bool = False, nthreads: int = 0):
        """C for every group of a `synth.Problem`; returns (list of C, list of sums or None)."""
        Cs, Xs = [], []
        for g in range(prob.G):
            C, X, _ = self.group_gemm(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K,
                                      want_exact=want_exact, nthreads=nthreads)
            Cs.append(C)
            Xs.append(X)
        return Cs, (Xs if want_exact else None)

    # -- scale re-layout --------------------------------------------------------
    def sf_relayout(self, sf: np.ndarray, K: int) -> np.ndarray:
        R = int(sf.shape[0])
        sf = np.ascontiguousarray(sf, dtype=np.uint8)
        assert sf.shape == (R, K // 16)
        out = np.full((((R + 127) // 128) * (K // 64) * 512,), 0xAA, dtype=np.uint8)
        rc = self.lib.oracle_sf_relayout(R, K, _ptr(sf, _u8p), _ptr(out, _u8p))
        if rc < 0:
            raise ValueError("oracle_sf_relayout: K must be a multiple of 64")
        return out


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from the committed source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
