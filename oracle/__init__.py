"""CPU oracle for the FP8 block-scaled GEMM and the MXFP8 GEMM.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product path never does. It shares no
code with the CUDA library.

``fp8bs_oracle.c`` holds the fp64 definition (dequantise -> naive triple loop ->
one bf16 rounding; skill card "FlyDSL fp8 blockscale GEMM", section
"Procedure" step 1, and PR "1x32 ue8m0 (MXFP8) 8-wave FlyDSL GEMM for gfx950",
section "Correctness"). This module loads it with ctypes and adds a
pure-Python exact evaluation with ``fractions.Fraction`` for tiny inputs,
which the tests use as brute force.

Every function here is pinned by tests/test_oracle_pins.py; nothing is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0_decode.restype = ctypes.c_double
        lib.oracle_ue8m0_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_max_threads.restype = ctypes.c_int
        p = ctypes.c_void_p
        i = ctypes.c_int
        for name in ("oracle_blockscale", "oracle_blockscale_blockpartial", "oracle_mxfp8"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [p, p, p, p, i, i, i, i, i, p, p]
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def ue8m0_decode(code: int) -> float:
    return _load().oracle_ue8m0_decode(int(code))


def bf16_rne(x: float) -> int:
    return int(_load().oracle_bf16_rne(float(x)))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _run(name, A, s_a, B, s_b, M, N, K, rows, want_exact):
    lib = _load()
    r0, r1 = (0, M) if rows is None else rows
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    C = np.empty((r1 - r0, N), dtype=np.uint16)
    Ce = np.empty((r1 - r0, N), dtype=np.float64) if want_exact else None
    rc = getattr(lib, name)(_ptr(A), _ptr(s_a), _ptr(B), _ptr(s_b), M, N, K, r0, r1, _ptr(C), _ptr(Ce))
    if rc != 0:
        raise RuntimeError(f"{name} failed ({rc})")
    return (C, Ce) if want_exact else C


def blockscale(A, a_scale, B, b_scale, rows=None, exact=False):
    """bf16 bits (uint16 [rows, N]) of the blockscale GEMM; a_scale is logical [M, K/128]."""
    M, K = A.shape
    N = B.shape[0]
    sa = np.ascontiguousarray(a_scale, dtype=np.float32)
    sb = np.ascontiguousarray(b_scale, dtype=np.float32)
    assert sa.shape == (M, K // 128) and sb.shape == ((N + 127) // 128, K // 128)
    return _run("oracle_blockscale", A, sa, B, sb, M, N, K, rows, exact)


def tensorscale(A, B, alpha, rows=None):
    """C = bf16(alpha * A.B^T), the promote-free ceiling twin (skill card "FlyDSL fp8
    blockscale GEMM", section "Bottleneck diagnosis"). It is exactly the blockscale
    definition with every a_scale equal to alpha and every b_scale equal to 1, so it
    is computed by that function (same fp64 sums, one bf16 rounding)."""
    M, K = A.shape
    N = B.shape[0]
    sa = np.full((M, K // 128), np.float32(alpha), dtype=np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), dtype=np.float32)
    return blockscale(A, sa, B, sb, rows=rows)


def e4m3_encode(y) -> np.ndarray:
    """fp32 values -> OCP E4M3FN codes (uint8), rounded to the nearest
    representable value with ties to the even mantissa, saturating at +-448;
    the sign of a value that rounds to zero is kept (0x80 for -0).

    From the format definition: a normal E4M3 value in the binade
    [2^E, 2^(E+1)), E = -6..8, is a multiple of 2^(E-3) (three fraction
    bits); below 2^-6 the values are the subnormal multiples of 2^-9. So the
    nearest value is rint(|y| / quantum) * quantum (numpy's rint rounds half
    to even, and the quotient of an fp32 by a power of two is exact in fp64);
    a quotient of 16 lands on 2^(E+1), the first value of the next binade.
    This is the store-side conversion of the fp8 partial in skill card "FlyDSL
    prefill MoE stage-2 fp8 partial", procedure step 2, with the saturation
    of the conversion the kernel uses (values past 448 are clamped, no NaN is
    produced from a finite value)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    if np.isnan(y).any():
        raise ValueError("NaN input")
    a = np.abs(y)
    _, e = np.frexp(a)                       # a in [2^(e-1), 2^e)
    E = np.maximum(e - 1, -6)                # binade; the subnormals share the quantum of E = -6
    quantum = np.ldexp(1.0, E - 3)
    v = np.minimum(np.rint(a / quantum) * quantum, 448.0)
    # value -> code
    code = np.zeros(a.shape, dtype=np.int64)
    sub = v < 2.0 ** -6
    code[sub] = np.rint(v[sub] / 2.0 ** -9).astype(np.int64)           # exponent field 0
    nv = v[~sub]
    _, e2 = np.frexp(nv)
    E2 = e2 - 1                                                        # nv in [2^E2, 2^(E2+1))
    mant = np.rint(nv / np.ldexp(1.0, E2 - 3)).astype(np.int64) - 8     # 0..7
    code[~sub] = ((E2 + 7) << 3) | mant
    code |= np.where(np.signbit(y), 0x80, 0)
    return code.astype(np.uint8)


def blockscale_e4m3out(A, a_scale, B, b_scale, c_scale, rows=None):
    """The blockscale GEMM with an E4M3 C: codes = e4m3(c_scale * C), C the
    exact sum rounded to fp32 and multiplied by the fp32 c_scale in fp32, the
    precision in which the kernel takes the same decision (its sum is fp32).
    Returns (codes uint8 [rows, N], y float32 [rows, N]: the value that was
    rounded, for judging ties near a rounding boundary)."""
    _, exact = blockscale(A, a_scale, B, b_scale, rows=rows, exact=True)
    y = (exact.astype(np.float32) * np.float32(c_scale)).astype(np.float32)
    return e4m3_encode(y), y


def mxfp8_e4m3out(A, a_e8m0, B, b_e8m0, c_scale, rows=None):
    """The MXFP8 GEMM with an E4M3 C, as blockscale_e4m3out: (codes, y)."""
    _, exact = mxfp8(A, a_e8m0, B, b_e8m0, rows=rows, exact=True)
    y = (exact.astype(np.float32) * np.float32(c_scale)).astype(np.float32)
    return e4m3_encode(y), y


def moe_leaders(block_expert, num_experts, pair=True) -> np.ndarray:
    """Leader descriptor of a sorted block -> expert table (skill card "FlyDSL
    decode MoE stage-1 blkmap", procedure step 2): for every run of k adjacent
    blocks of one expert, ceil(k/2) leaders, each the first block of a pair
    (value b | 1 << 30) or a trailing solo block (value b); without pairing,
    every block leads itself. Blocks whose expert is outside [0, num_experts)
    lead nothing. Walks the table run by run."""
    be = [int(v) for v in block_expert]
    out = []
    b = 0
    while b < len(be):
        r = b
        while r < len(be) and be[r] == be[b]:
            r += 1
        if 0 <= be[b] < num_experts:
            k = r - b
            if pair:
                out.extend((b + i) | ((1 << 30) if i + 1 < k else 0) for i in range(0, k, 2))
            else:
                out.extend(range(b, r))
        b = r
    return np.array(out, dtype=np.int32)


def moe_gemm(A, a_scale, B, b_scale, block_expert, num_experts, block_rows=64):
    """Grouped blockscale GEMM by its definition: every row of a sort block of
    expert e is the blockscale GEMM of that row with B[e], b_scale[e] (a_scale
    logical [M, K/128], B [E, N, K], b_scale [E, ceil(N/128), K/128]). Returns
    (C bf16 bits [M, N], mask of the rows that are defined: blocks with an
    expert in range)."""
    M, K = A.shape
    N = B.shape[1]
    be = np.asarray(block_expert)
    C = np.zeros((M, N), dtype=np.uint16)
    defined = np.zeros(M, dtype=bool)
    for e in range(num_experts):
        blocks = np.nonzero(be == e)[0]
        if len(blocks) == 0:
            continue
        rows = (blocks[:, None] * block_rows + np.arange(block_rows)[None, :]).ravel()
        C[rows] = blockscale(np.ascontiguousarray(A[rows]), np.ascontiguousarray(a_scale[rows]),
                             np.ascontiguousarray(B[e]), np.ascontiguousarray(b_scale[e]))
        defined[rows] = True
    return C, defined


def blockscale_blockpartial(A, a_scale, B, b_scale, rows=None, exact=False):
    M, K = A.shape
    N = B.shape[0]
    sa = np.ascontiguousarray(a_scale, dtype=np.float32)
    sb = np.ascontiguousarray(b_scale, dtype=np.float32)
    return _run("oracle_blockscale_blockpartial", A, sa, B, sb, M, N, K, rows, exact)


def mxfp8(A, a_e8m0, B, b_e8m0, rows=None, exact=False):
    """bf16 bits (uint16 [rows, N]) of the MXFP8 GEMM; scales are ue8m0 bytes [rows, K/32]."""
    M, K = A.shape
    N = B.shape[0]
    ea = np.ascontiguousarray(a_e8m0, dtype=np.uint8)
    eb = np.ascontiguousarray(b_e8m0, dtype=np.uint8)
    assert ea.shape == (M, K // 32) and eb.shape == (N, K // 32)
    return _run("oracle_mxfp8", A, ea, B, eb, M, N, K, rows, exact)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Exact rational evaluation (brute force for tiny inputs).

def e4m3_fraction(code: int) -> Fraction:
    """E4M3FN code -> exact value as a Fraction (NaN code raises)."""
    s, e, m = code >> 7, (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        raise ValueError("NaN code")
    v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))
    return -v if s else v


def fraction_to_bf16_bits(q: Fraction) -> int:
    """Correctly rounded (nearest, ties to even) bf16 of an exact rational."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qexp = max(e, -126) - 7
    scaled = a / (Fraction(2) ** qexp)
    fl = scaled.numerator // scaled.denominator
    rem = scaled - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    value = Fraction(fl) * (Fraction(2) ** qexp)
    if value > Fraction(255) * Fraction(2) ** 120:
        return sign | 0x7F80
    bits = int(np.array([float(value)], dtype=np.float32).view(np.uint32)[0])
    return sign | ((bits >> 16) & 0x7FFF)


def exact_blockscale(A, a_scale, B, b_scale):
    """Exact rational C (list of lists of Fraction) of the blockscale definition."""
    M, K = A.shape
    N = B.shape[0]
    fa = [[e4m3_fraction(int(c)) for c in row] for row in A]
    fb = [[e4m3_fraction(int(c)) for c in row] for row in B]
    out = []
    for m in range(M):
        row = []
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sa = Fraction(float(a_scale[m, k // 128]))
                sb = Fraction(float(b_scale[n // 128, k // 128]))
                acc += (fa[m][k] * sa) * (fb[n][k] * sb)
            row.append(acc)
        out.append(row)
    return out


def exact_mxfp8(A, a_e8m0, B, b_e8m0):
    M, K = A.shape
    N = B.shape[0]
    fa = [[e4m3_fraction(int(c)) for c in row] for row in A]
    fb = [[e4m3_fraction(int(c)) for c in row] for row in B]
    out = []
    for m in range(M):
        row = []
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sa = Fraction(2) ** (int(a_e8m0[m, k // 32]) - 127)
                sb = Fraction(2) ** (int(b_e8m0[n, k // 32]) - 127)
                acc += (fa[m][k] * sa) * (fb[n][k] * sb)
            row.append(acc)
        out.append(row)
    return out
