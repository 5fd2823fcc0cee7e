"""Pins for the CPU oracle: each check compares it with something other than
itself (torch's float8_e4m3fn decoding, numpy's float16 rounding, exact
rational arithmetic, numpy fp64 matmul where the sum is provably exact,
closed-form E2M1 values, invariants, the CuTe atom printed on the pages).

Each `pin_*` function takes an `oracle.Oracle` and raises AssertionError on a
mismatch, so `test_oracle_mutants.py` can run the same pins against oracle
builds with a planted mistake and show that some pin catches each one.
"""
from __future__ import annotations

import ast
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# E2M1 magnitudes for codes 0..7 (OCP Microscaling formats v1.0, FP4 E2M1):
# 0, 0.5 (the one subnormal), 1, 1.5, 2, 3, 4, 6. Codes 8..15 are the same
# magnitudes with the sign bit (bit 3) set.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_lib(codes) -> np.ndarray:
    """E4M3 decode through torch's float8_e4m3fn dtype (a library route)."""
    t = torch.tensor(np.asarray(codes, dtype=np.uint8).ravel(), dtype=torch.uint8)
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(np.shape(codes))


def e2m1_indep(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    mag = np.asarray(E2M1_MAGNITUDES)[c & 7]
    return np.where(c & 8, -mag, mag)


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """[R, K/2] bytes -> [R, K] codes, even k in the low nibble."""
    R, H = q.shape
    out = np.empty((R, 2 * H), dtype=np.int64)
    out[:, 0::2] = q & 15
    out[:, 1::2] = q >> 4
    return out


def decode_indep(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    codes = unpack_nibbles(q)
    K = codes.shape[1]
    scales = np.repeat(e4m3_lib(sf), 16, axis=1)[:, :K]
    return e2m1_indep(codes) * scales


def same_fp16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Element-wise equality of fp16 results, +0 == -0, inf == inf (same sign)."""
    a = np.asarray(a, dtype=np.float16)
    b = np.asarray(b, dtype=np.float16)
    return (a == b) | (np.isnan(a) & np.isnan(b))


# ---------------------------------------------------------------- rationals

_FP16_POS = None


def _fp16_positive_finite():
    global _FP16_POS
    if _FP16_POS is None:
        bits = np.arange(0, 0x7C00, dtype=np.uint16)
        vals = bits.view(np.float16).astype(np.float64)
        _FP16_POS = (bits, [Fraction(float(v)) for v in vals])
    return _FP16_POS


def fp16_round_exact(x: Fraction) -> int:
    """Nearest fp16 of an exact rational by search over every finite value;
    ties to the even bit pattern; |x| >= 65520 overflows to infinity."""
    bits, vals = _fp16_positive_finite()
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a >= 65520:
        return sign | 0x7C00
    lo, hi = 0, len(vals) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if vals[mid] <= a:
            lo = mid
        else:
            hi = mid
    if vals[hi] <= a:
        lo = hi
    if vals[lo] == a or lo == len(vals) - 1:
        return sign | int(bits[lo])
    dl, dh = a - vals[lo], vals[lo + 1] - a
    if dl < dh:
        return sign | int(bits[lo])
    if dh < dl:
        return sign | int(bits[lo + 1])
    pick = lo if int(bits[lo]) % 2 == 0 else lo + 1
    return sign | int(bits[pick])


def exact_sum_rational(A, B, SFA, SFB, K, m, n) -> Fraction:
    a = unpack_nibbles(A[m:m + 1])[0]
    b = unpack_nibbles(B[n:n + 1])[0]
    s = Fraction(0)
    for k in range(K):
        va = Fraction(float(e2m1_indep(a[k]))) * Fraction(float(e4m3_lib(SFA[m, k // 16])))
        vb = Fraction(float(e2m1_indep(b[k]))) * Fraction(float(e4m3_lib(SFB[n, k // 16])))
        s += va * vb
    return s


# --------------------------------------------------------------------- pins

def pin_e4m3_table(o):
    codes = np.arange(256)
    lib = e4m3_lib(codes)
    ours = np.array([o.e4m3(c) for c in codes])
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan), "NaN codes differ"
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], lib[~nan]), "E4M3 decode differs from torch float8_e4m3fn"


def pin_e2m1_table(o):
    ours = np.array([o.e2m1(c) for c in range(16)])
    assert np.array_equal(np.abs(ours[:8]), np.asarray(E2M1_MAGNITUDES)), ours
    assert np.array_equal(ours[8:], -ours[:8]) and np.signbit(ours[8:]).all()
    # Library route: an E2M1 value (sign s, exponent e with bias 1, mantissa
    # m) equals the E4M3 value with the same sign, exponent e+6 (bias 7) and
    # mantissa m<<2; the one E2M1 subnormal 0.5 is the E4M3 normal 2^-1.
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0 and m == 0:
            byte = s << 7
        elif e == 0:
            byte = (s << 7) | (6 << 3)
        else:
            byte = (s << 7) | ((e + 6) << 3) | (m << 2)
        assert ours[c] == e4m3_lib([byte])[0], (c, ours[c])


def pin_fp16_rounding(o):
    rng = np.random.default_rng(123)
    xs = [rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),
          np.array([0.0, -0.0, 65504.0, 65519.999, 65520.0, 65536.0, 1e30, -65520.0, -65519.0,
                    2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -25 * 1.0000001, 2.0 ** -14,
                    2.0 ** -14 - 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2048 + 1, 2048 + 3])]
    # every exact halfway point between consecutive fp16 values in a few binades
    f = np.arange(0, 0x7BFF, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    g = np.arange(1, 0x7C00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    xs.append((f + g) / 2)
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    mids = (lo.view(np.float16).astype(np.float64) + (lo + 1).view(np.float16).astype(np.float64)) / 2
    xs.append(mids[::11])
    xs.append(-mids[::13])
    x = np.concatenate(xs)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16)
    ours = o.fp16_rne(x).view(np.float16)
    bad = ~same_fp16(ours, ref)
    assert not bad.any(), list(zip(x[bad][:5], ours[bad][:5], ref[bad][:5]))


def _random_codes(rng, shape, allow_negative_scales=True):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN scales
    if not allow_negative_scales:
        c &= 0x7F
    return c


def pin_bruteforce_tiny(o):
    rng = np.random.default_rng(7)
    for trial in range(12):
        M, N = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        K = [32, 48][trial % 2]
        A = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
        B = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        SFA = _random_codes(rng, (M, K // 16))
        SFB = _random_codes(rng, (N, K // 16))
        C, X, _ = o.group_gemm(A, B, SFA, SFB, K, want_exact=True)
        for m in range(M):
            for n in range(N):
                ex = exact_sum_rational(A, B, SFA, SFB, K, m, n)
                assert Fraction(float(X[m, n])) == ex, (trial, m, n)
                want = np.array([fp16_round_exact(ex)], dtype=np.uint16).view(np.float16)
                assert same_fp16(C[m, n], want[0]), (trial, m, n, C[m, n], want[0])


def pin_no_double_rounding(o):
    # one row/column pair whose exact sum is 16 + 2^-7 + 2^-20: the 2^-20 term
    # breaks the fp16 tie at 16 + 2^-7 (correct result 16 + 2^-6), but is only
    # half an fp32 ulp at 16, so rounding through fp32 would give 16.
    K = 48
    A = np.zeros((1, K // 2), np.uint8)
    B = np.zeros((1, K // 2), np.uint8)
    A[0, 0] = 6; A[0, 8] = 1; A[0, 16] = 1    # e2m1 4.0 at k=0, 0.5 at k=16 and k=32
    B[0, 0] = 6; B[0, 8] = 1; B[0, 16] = 1
    SFA = np.array([[0x38, 0x20, 0x01]], np.uint8)  # 1, 2^-3, 2^-9
    SFB = np.array([[0x38, 0x28, 0x01]], np.uint8)  # 1, 2^-2, 2^-9
    C, X, _ = o.group_gemm(A, B, SFA, SFB, K, want_exact=True)
    ex = exact_sum_rational(A, B, SFA, SFB, K, 0, 0)
    assert ex == 16 + Fraction(1, 2 ** 7) + Fraction(1, 2 ** 20)
    want = np.array([fp16_round_exact(ex)], np.uint16).view(np.float16)[0]
    assert float(want) == 16 + 2.0 ** -6
    assert same_fp16(C[0, 0], want), (C[0, 0], want)


def pin_products_16x16(o):
    K = 256
    A = np.zeros((16, K // 2), np.uint8)
    B = np.zeros((16, K // 2), np.uint8)
    A[:, 0] = np.arange(16)  # code i at k = 0 (low nibble), zero elsewhere
    B[:, 0] = np.arange(16)
    one = np.full((16, K // 16), 0x38, np.uint8)
    C, X, exact = o.group_gemm(A, B, one, one, K, want_exact=True)
    v = e2m1_indep(np.arange(16))
    prod = np.outer(v, v)
    assert exact == 1
    assert np.array_equal(X, prod)
    assert same_fp16(C, prod.astype(np.float16)).all()


def pin_matmul_single_group(o):
    rng = np.random.default_rng(11)
    from block_scaled_fp4_grouped_gb300 import synth
    for (M, N, K) in [(40, 72, 256), (3, 129, 512), (130, 5, 1024)]:
        A = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
        B = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        SFA = synth.scale_codes(rng, (M, K // 16))
        SFB = synth.scale_codes(rng, (N, K // 16))
        C, X, exact = o.group_gemm(A, B, SFA, SFB, K, want_exact=True, nthreads=3)
        assert exact == 1
        ref = decode_indep(A, SFA) @ decode_indep(B, SFB).T  # exact in fp64 here
        assert np.array_equal(X, ref)
        assert same_fp16(C, ref.astype(np.float16)).all()


def pin_exact_power_of_two_scales(o):
    rng = np.random.default_rng(5)
    M, N, K = 17, 33, 2048
    A = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    SFA = np.full((M, K // 16), 0x28, np.uint8)  # 2^-2
    SFB = np.full((N, K // 16), 0x40, np.uint8)  # 2^1
    C, X, exact = o.group_gemm(A, B, SFA, SFB, K, want_exact=True)
    codes_a, codes_b = unpack_nibbles(A), unpack_nibbles(B)
    # closed form: scales factor out of the sum
    ref = (e2m1_indep(codes_a) @ e2m1_indep(codes_b).T) * 0.25 * 2.0
    assert exact == 1 and np.array_equal(X, ref)
    assert same_fp16(C, ref.astype(np.float16)).all()


def _two_term_rows(K: int, big: int):
    """One row of A (and the same row of B) whose products are `big` terms of
    (4 * 2^8)^2 = 2^20 (E2M1 code 6 under scale code 0x78) followed by one
    term of (0.5 * 2^-9)^2 = 2^-20 (E2M1 code 1 under the smallest E4M3
    code 0x01), zeros after it. `big` is a multiple of 16."""
    codes = np.zeros((1, K), np.int64)
    codes[0, :big] = 6
    codes[0, big] = 1
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((1, K // 16), 0x38, np.uint8)
    sf[0, : big // 16] = 0x78
    sf[0, big // 16] = 0x01
    return q, sf


def pin_exactness_flag(o):
    """The `exact` flag promises that the fp64 sum in ascending k is the exact
    real sum. Checked against exact rationals on two rows: 2048 * 2^20 + 2^-20
    = 2^31 + 2^-20 needs 52 significant bits (fp64 holds 53: the sum is
    exact, and the flag must say so); 8192 * 2^20 + 2^-20 = 2^33 + 2^-20 needs
    54 (fp64 rounds the last term away: the flag must be 0)."""
    for big, want_exact in ((2048, 1), (8192, 0)):
        K = big + 16
        q, sf = _two_term_rows(K, big)
        C, X, exact = o.group_gemm(q, q, sf, sf, K, want_exact=True)
        true_sum = Fraction(big) * 2 ** 20 + Fraction(1, 2 ** 20)
        assert (Fraction(float(X[0, 0])) == true_sum) == bool(want_exact), (big, X[0, 0])
        if exact == 1:  # soundness: a sum declared exact is exact
            assert Fraction(float(X[0, 0])) == true_sum, (big, exact)
        assert exact == want_exact, (big, exact)


def pin_invariants(o):
    rng = np.random.default_rng(3)
    from block_scaled_fp4_grouped_gb300 import synth
    M, N, K = 6, 10, 128
    A = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    SFA = synth.scale_codes(rng, (M, K // 16))
    SFB = synth.scale_codes(rng, (N, K // 16))
    _, X, _ = o.group_gemm(A, B, SFA, SFB, K, want_exact=True)
    # zero A gives zero C
    C0, X0, _ = o.group_gemm(np.zeros_like(A), B, SFA, SFB, K, want_exact=True)
    assert not X0.any() and not C0.astype(np.float64).any()
    for (m, j) in [(0, 0), (5, 7), (2, 3)]:
        # the contribution of slice j of row m: keep only k in [16j, 16j+16)
        Aj = np.zeros_like(A)
        Aj[:, 8 * j:8 * j + 8] = A[:, 8 * j:8 * j + 8]
        _, Xj, _ = o.group_gemm(Aj, B, SFA, SFB, K, want_exact=True)
        S2 = SFA.copy()
        S2[m, j] += 8  # exponent + 1: the scale doubles exactly
        _, X2, _ = o.group_gemm(A, B, S2, SFB, K, want_exact=True)
        d = X2 - X
        assert np.array_equal(d[m], Xj[m]), (m, j)
        others = np.ones(M, bool)
        others[m] = False
        assert not d[others].any()
    for (n, j) in [(0, 0), (9, 7), (4, 2)]:
        Bj = np.zeros_like(B)
        Bj[:, 8 * j:8 * j + 8] = B[:, 8 * j:8 * j + 8]
        _, Xj, _ = o.group_gemm(A, Bj, SFA, SFB, K, want_exact=True)
        S2 = SFB.copy()
        S2[n, j] += 8
        _, X2, _ = o.group_gemm(A, B, SFA, S2, K, want_exact=True)
        d = X2 - X
        assert np.array_equal(d[:, n], Xj[:, n]), (n, j)
        others = np.ones(N, bool)
        others[n] = False
        assert not d[:, others].any()


def _golden_atom():
    spec = {}
    with open(os.path.join(GOLDEN, "sf_atom_layout.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split(None, 1)
                spec[key] = val
    return spec


def _cute_offset(coord: int, shape, stride) -> int:
    """Evaluate one mode of a CuTe layout: split `coord` colexicographically
    over the (nested) shape and sum coordinate * stride."""
    if isinstance(shape, int):
        return coord * stride
    off = 0
    for s, d in zip(shape, stride):
        size = int(np.prod(_flatten(s)))
        off += _cute_offset(coord % size, s, d)
        coord //= size
    return off


def _flatten(x):
    if isinstance(x, int):
        return [x]
    out = []
    for e in x:
        out += _flatten(e)
    return out


def pin_relayout(o):
    spec = _golden_atom()
    shape = ast.literal_eval(spec["atom_shape"])
    stride = ast.literal_eval(spec["atom_stride"])
    atom_bytes = int(spec["atom_bytes"])
    rows_per_atom = int(np.prod(_flatten(shape[0])))
    k_per_atom = int(np.prod(_flatten(shape[1])))
    assert (rows_per_atom, k_per_atom, atom_bytes) == (128, 64, 512)
    rng = np.random.default_rng(9)
    for (R, K) in [(300, 512), (128, 64), (1, 256), (129, 192)]:
        sf = rng.integers(0, 256, (R, K // 16)).astype(np.uint8)
        out = o.sf_relayout(sf, K)
        rblocks = (R + 127) // 128
        assert out.size == rblocks * (K // 64) * atom_bytes
        want = np.zeros_like(out)
        for r in range(rblocks * 128):
            for k in range(0, K, 16):
                atom = eval(spec["atom_index"], {}, {"row": r, "K": K, "k": k})
                off = (_cute_offset(r % rows_per_atom, shape[0], stride[0]) +
                       _cute_offset(k % k_per_atom, shape[1], stride[1]))
                want[atom * atom_bytes + off] = sf[r, k // 16] if r < R else 0
        assert np.array_equal(out, want), (R, K)


ALL_PINS = [
    pin_e4m3_table,
    pin_e2m1_table,
    pin_fp16_rounding,
    pin_bruteforce_tiny,
    pin_no_double_rounding,
    pin_products_16x16,
    pin_matmul_single_group,
    pin_exact_power_of_two_scales,
    pin_exactness_flag,
    pin_invariants,
    pin_relayout,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_oracle_thread_count_independent(oracle_lib):
    from block_scaled_fp4_grouped_gb300 import synth
    prob = synth.make_problem("custom", seed=1, M=[37], N=200, K=768)
    c1, x1, _ = oracle_lib.group_gemm(prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], prob.K,
                                      want_exact=True, nthreads=1)
    c7, x7, _ = oracle_lib.group_gemm(prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], prob.K,
                                      want_exact=True, nthreads=7)
    assert np.array_equal(x1, x7) and np.array_equal(c1.view(np.uint16), c7.view(np.uint16))


def test_oracle_entries_match_full(oracle_lib):
    from block_scaled_fp4_grouped_gb300 import synth
    prob = synth.make_problem("custom", seed=2, M=[50], N=90, K=512)
    C, X, _ = oracle_lib.group_gemm(prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], prob.K,
                                    want_exact=True)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 50, 40)
    cols = rng.integers(0, 90, 40)
    e16, ex = oracle_lib.group_entries(prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], prob.K, rows, cols)
    assert np.array_equal(ex, X[rows, cols])
    assert same_fp16(e16, C[rows, cols]).all()


def test_group_independence(oracle_lib):
    """Permuting the group order permutes the results and changes nothing else."""
    from block_scaled_fp4_grouped_gb300 import synth
    prob = synth.make_problem("custom", seed=4, M=[8, 24, 16], N=40, K=256)
    Cs, _ = oracle_lib.grouped(prob)
    for g in [2, 0, 1]:
        C, _, _ = oracle_lib.group_gemm(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K)
        assert np.array_equal(C.view(np.uint16), Cs[g].view(np.uint16))


def test_generated_sums_are_exact(oracle_lib):
    """The generated distributions keep every fp64 partial sum exact, so the
    oracle is the correctly rounded value (checked on the largest K)."""
    from block_scaled_fp4_grouped_gb300 import synth
    prob = synth.make_problem("custom", seed=0, M=[4], N=8, K=7168)
    _, _, exact = oracle_lib.group_gemm(prob.A[0], prob.B[0], prob.SFA[0], prob.SFB[0], prob.K)
    assert exact == 1
