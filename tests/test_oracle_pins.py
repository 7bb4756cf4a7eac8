"""Pins of the CPU oracle against things other than itself (CPU only).

Each test fixes one part of the oracle with something independent of its code:
a library decoder, exact rational arithmetic, a closed form, an invariant of the
definition, or a hand-derived worked example under tests/golden/.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---- P1: decoders ----------------------------------------------------------

def test_e4m3_decoder_matches_torch_for_all_codes():
    torch = pytest.importorskip("torch")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


def test_e4m3_decoder_golden_anchors():
    for code, val in _golden_rows("e4m3_anchors.txt"):
        got = oracle.e4m3_decode(int(code, 16))
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_decoder_matches_exact_fraction():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert Fraction(oracle.e4m3_decode(c)) == oracle.e4m3_fraction(c)


def test_ue8m0_decoder():
    for c in range(255):
        assert oracle.ue8m0_decode(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(oracle.ue8m0_decode(255))


# ---- P2: bf16 rounding -----------------------------------------------------

def test_bf16_rne_matches_exact_rational_rounding():
    rng = np.random.Generator(np.random.PCG64(1234))
    # random magnitudes over the whole bf16 range, incl. subnormals and overflow
    xs = list(rng.standard_normal(40000) * np.exp2(rng.uniform(-140, 130, 40000)))
    # values with random 53-bit mantissas near 1
    xs += list(rng.uniform(-4, 4, 20000))
    # exact ties and ties +- 1 ulp of double, at several magnitudes
    for e in (-133, -130, -126, -100, -1, 0, 7, 100, 127):
        for mant in range(128, 256, 7):
            base = math.ldexp(mant, e - 7)
            tie = base + math.ldexp(1, e - 8) if e >= -126 else None
            if tie is not None:
                xs += [tie, -tie, math.nextafter(tie, 0), math.nextafter(tie, math.inf)]
    # subnormal-range ties (quantum 2^-133)
    for m in range(0, 128, 3):
        t = math.ldexp(2 * m + 1, -134)
        xs += [t, -t, math.nextafter(t, 0), math.nextafter(t, 1)]
    # overflow boundary: max bf16, midpoint to 2^128, and just below
    mx = math.ldexp(255, 120)
    mid = math.ldexp(511, 119)
    xs += [mx, -mx, mid, math.nextafter(mid, 0), math.ldexp(1, 128), 1e300, -1e300, 0.0, -0.0, 5e-324]
    for x in xs:
        x = float(x)
        assert oracle.bf16_rne(x) == oracle.fraction_to_bf16_bits(Fraction(x)) or \
            (x == 0 and oracle.bf16_rne(x) in (0, 0x8000)), x


def test_bf16_rne_special_values():
    assert oracle.bf16_rne(math.inf) == 0x7F80
    assert oracle.bf16_rne(-math.inf) == 0xFF80
    assert oracle.bf16_rne(-0.0) == 0x8000
    assert (oracle.bf16_rne(math.nan) & 0x7F80) == 0x7F80 and (oracle.bf16_rne(math.nan) & 0x7F)


# ---- golden worked examples -----------------------------------------------

def _tiny_blockscale_inputs():
    M, N, K = 3, 2, 256
    A = np.zeros((M, K), np.uint8)
    A[0, :] = 0x38
    A[1, :] = 0x40
    A[2, :136] = 0x38
    B = np.zeros((N, K), np.uint8)
    B[0, :] = 0x38
    B[1, :] = 0xB0
    sa = np.array([[0.5, 0.25], [1.0, 3.0], [1.0, 1.0]], np.float32)
    sb = np.array([[2.0, 0.125]], np.float32)
    return A, sa, B, sb


def test_golden_tiny_blockscale():
    A, sa, B, sb = _tiny_blockscale_inputs()
    C, Ce = oracle.blockscale(A, sa, B, sb, exact=True)
    Cf = oracle.bf16_bits_to_float(C)
    for m, n, exact, bf in _golden_rows("tiny_blockscale.txt"):
        m, n = int(m), int(n)
        assert Ce[m, n] == float(exact)
        assert Cf[m, n] == float(bf)


def test_golden_tiny_mxfp8():
    A = np.full((1, 64), 0x38, np.uint8)
    B = np.full((1, 64), 0x3C, np.uint8)
    ea = np.array([[127, 130]], np.uint8)
    eb = np.array([[126, 127]], np.uint8)
    C, Ce = oracle.mxfp8(A, ea, B, eb, exact=True)
    for m, n, exact, bf in _golden_rows("tiny_mxfp8.txt"):
        assert Ce[int(m), int(n)] == float(exact)
        assert oracle.bf16_bits_to_float(C)[int(m), int(n)] == float(bf)


# ---- P3: exact brute force on tiny random inputs --------------------------

def _random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3A     # no NaN codes (outside the contract)
    return c


@pytest.mark.parametrize("seed,M,N,K", [(0, 2, 3, 128), (1, 3, 2, 256), (2, 4, 4, 128), (3, 1, 130, 128)])
def test_blockscale_brute_force_exact(seed, M, N, K):
    rng = np.random.Generator(np.random.PCG64(seed))
    A = _random_codes(rng, (M, K))
    B = _random_codes(rng, (N, K))
    sa = rng.uniform(1e-4, 2.0, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(1e-5, 0.5, ((N + 127) // 128, K // 128)).astype(np.float32)
    C = oracle.blockscale(A, sa, B, sb)
    ex = oracle.exact_blockscale(A, sa, B, sb)
    for m in range(M):
        for n in range(N):
            assert C[m, n] == oracle.fraction_to_bf16_bits(ex[m][n]), (m, n)


@pytest.mark.parametrize("seed,M,N,K", [(0, 2, 3, 64), (1, 3, 2, 128), (2, 2, 2, 256)])
def test_mxfp8_brute_force_exact(seed, M, N, K):
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    A = _random_codes(rng, (M, K))
    B = _random_codes(rng, (N, K))
    ea = rng.integers(110, 140, size=(M, K // 32), dtype=np.uint8)
    eb = rng.integers(110, 140, size=(N, K // 32), dtype=np.uint8)
    C = oracle.mxfp8(A, ea, B, eb)
    ex = oracle.exact_mxfp8(A, ea, B, eb)
    for m in range(M):
        for n in range(N):
            assert C[m, n] == oracle.fraction_to_bf16_bits(ex[m][n]), (m, n)


# ---- P4: unit scales reduce to a plain fp8 GEMM ----------------------------

def _decode_array(codes):
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_unit_scales_equal_plain_fp8_gemm():
    rng = np.random.Generator(np.random.PCG64(7))
    M, N, K = 24, 136, 1024
    A = _random_codes(rng, (M, K))
    B = _random_codes(rng, (N, K))
    ref = _decode_array(A) @ _decode_array(B).T     # every partial sum is exact in fp64 here
    _, Ce = oracle.blockscale(A, np.ones((M, K // 128), np.float32), B,
                              np.ones(((N + 127) // 128, K // 128), np.float32), exact=True)
    assert np.array_equal(Ce, ref)
    _, Ce2 = oracle.mxfp8(A, np.full((M, K // 32), 127, np.uint8), B,
                          np.full((N, K // 32), 127, np.uint8), exact=True)
    assert np.array_equal(Ce2, ref)


# ---- P5: linearity in one per-block scale ----------------------------------

def test_linearity_in_one_block_scale():
    x = workloads.make_blockscale_inputs(64, 256, 512, seed=3)
    _, C0 = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, exact=True)
    m, kb, alpha = 17, 2, 3.5
    sa2 = x.a_scale.copy()
    sa2[m, kb] *= np.float32(alpha)
    _, C1 = oracle.blockscale(x.A, sa2, x.B, x.b_scale, exact=True)
    dA = _decode_array(x.A[m, kb * 128:(kb + 1) * 128])
    dB = _decode_array(x.B[:, kb * 128:(kb + 1) * 128])
    S = dB @ dA                                        # unscaled block partial per column
    sb = x.b_scale[np.arange(256) // 128, kb].astype(np.float64)
    pred = (float(sa2[m, kb]) - float(x.a_scale[m, kb])) * sb * S
    diff = C1[m] - C0[m]
    assert np.allclose(diff, pred, rtol=1e-12, atol=1e-14 * np.abs(C0[m]).max())
    other = np.arange(64) != m
    assert np.array_equal(C1[other], C0[other])


# ---- P6: power-of-two scaling is exact ------------------------------------

def test_power_of_two_scale_doubles_row_exactly():
    x = workloads.make_mxfp8_inputs(16, 64, 256, seed=5)
    C0, E0 = oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0, exact=True)
    ea = x.a_e8m0.copy()
    ea[5] += 1
    C1, E1 = oracle.mxfp8(x.A, ea, x.B, x.b_e8m0, exact=True)
    assert np.array_equal(E1[5], 2 * E0[5])
    assert np.array_equal(oracle.bf16_bits_to_float(C1[5]), 2 * oracle.bf16_bits_to_float(C0[5]))
    assert np.array_equal(C1[np.arange(16) != 5], C0[np.arange(16) != 5])
    # blockscale with every a_scale of one row multiplied by 2^-3
    y = workloads.make_blockscale_inputs(16, 128, 256, seed=6)
    D0, F0 = oracle.blockscale(y.A, y.a_scale, y.B, y.b_scale, exact=True)
    sa = y.a_scale.copy()
    sa[9] *= np.float32(0.125)
    D1, F1 = oracle.blockscale(y.A, sa, y.B, y.b_scale, exact=True)
    assert np.array_equal(F1[9], F0[9] * 0.125)
    assert np.array_equal(oracle.bf16_bits_to_float(D1[9]), oracle.bf16_bits_to_float(D0[9]) * np.float32(0.125))


# ---- P7: integer inputs with a known exact product ------------------------

def test_integer_inputs_exact():
    rng = np.random.Generator(np.random.PCG64(11))
    M, N, K = 40, 72, 256
    vals = rng.integers(-1, 2, size=(M, K))
    wals = rng.integers(-1, 2, size=(N, K))
    code = {-1: 0xB8, 0: 0x00, 1: 0x38}
    A = np.vectorize(code.get)(vals).astype(np.uint8)
    B = np.vectorize(code.get)(wals).astype(np.uint8)
    ref = vals.astype(np.int64) @ wals.astype(np.int64).T
    C = oracle.blockscale(A, np.ones((M, 2), np.float32), B, np.ones((1, 2), np.float32))
    assert np.array_equal(oracle.bf16_bits_to_float(C), ref.astype(np.float32))
    C2 = oracle.mxfp8(A, np.full((M, 8), 127, np.uint8), B, np.full((N, 8), 127, np.uint8))
    assert np.array_equal(oracle.bf16_bits_to_float(C2), ref.astype(np.float32))


# ---- P8: definition form vs block-partial form -----------------------------

def test_definition_form_matches_block_partial_form():
    x = workloads.make_blockscale_inputs(96, 200, 768, seed=2)
    C0, E0 = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, exact=True)
    C1, E1 = oracle.blockscale_blockpartial(x.A, x.a_scale, x.B, x.b_scale, exact=True)
    # the two summation orders differ by fp64 rounding only: bounded by
    # K * 2^-53 * sum_k |a_k b_k| (standard recursive-summation bound)
    KB = 768 // 128
    da = np.abs(_decode_array(x.A)) * np.repeat(x.a_scale.astype(np.float64), 128, axis=1)
    db = np.abs(_decode_array(x.B)) * np.repeat(np.repeat(x.b_scale.astype(np.float64), 128, axis=0)[:200], 128, axis=1)
    bound = (da @ db.T) * (768 + KB) * 2.0 ** -53
    assert np.all(np.abs(E0 - E1) <= bound)
    mism = np.nonzero(C0 != C1)
    # only near-ties may differ, and then by one bf16 ulp
    assert len(mism[0]) <= 2
    for m, n in zip(*mism):
        assert abs(int(C0[m, n]) - int(C1[m, n])) == 1


# ---- P9: blockscale <-> MXFP8 cross case -----------------------------------

def test_blockscale_equals_mxfp8_with_power_of_two_scales():
    rng = np.random.Generator(np.random.PCG64(9))
    M, N, K = 33, 257, 384
    A = _random_codes(rng, (M, K))
    B = _random_codes(rng, (N, K))
    ja = rng.integers(-6, 6, size=(M, K // 128))
    jb = rng.integers(-6, 6, size=((N + 127) // 128, K // 128))
    sa = np.ldexp(np.float32(1), ja).astype(np.float32)
    sb = np.ldexp(np.float32(1), jb).astype(np.float32)
    ea = np.repeat(ja + 127, 4, axis=1).astype(np.uint8)                       # [M, K/32]
    eb = np.repeat(np.repeat(jb + 127, 128, axis=0)[:N], 4, axis=1).astype(np.uint8)  # [N, K/32]
    C1, E1 = oracle.blockscale(A, sa, B, sb, exact=True)
    C2, E2 = oracle.mxfp8(A, ea, B, eb, exact=True)
    assert np.array_equal(E1, E2)
    assert np.array_equal(C1, C2)


# ---- P10: zeros --------------------------------------------------------------

def test_zero_operand_gives_positive_zero():
    x = workloads.make_blockscale_inputs(8, 16, 128, seed=0)
    C = oracle.blockscale(np.zeros_like(x.A), x.a_scale, x.B, x.b_scale)
    assert np.all(C == 0)
    y = workloads.make_mxfp8_inputs(8, 16, 128, seed=0)
    C = oracle.mxfp8(y.A, y.a_e8m0, np.zeros_like(y.B), y.b_e8m0)
    assert np.all(C == 0)


def test_row_range_matches_full():
    x = workloads.make_blockscale_inputs(64, 96, 256, seed=4)
    full = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale)
    part = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, rows=(10, 37))
    assert np.array_equal(part, full[10:37])


def test_tensorscale_oracle_is_the_exact_gemm_times_alpha():
    """The twin's oracle against exact rational arithmetic: with alpha = 1 every
    output is the correctly rounded bf16 of the exact sum of code products, and a
    power-of-two alpha scales every output exactly."""
    rng = np.random.Generator(np.random.PCG64(12))
    M, N, K = 5, 7, 256
    A = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0     # no NaN codes
    B[(B & 0x7F) == 0x7F] = 0
    fa = [[oracle.e4m3_fraction(int(c)) for c in row] for row in A]
    fb = [[oracle.e4m3_fraction(int(c)) for c in row] for row in B]
    want = np.array([[oracle.fraction_to_bf16_bits(sum(x * y for x, y in zip(fa[m], fb[n])))
                      for n in range(N)] for m in range(M)], dtype=np.uint16)
    one = oracle.tensorscale(A, B, 1.0)
    assert np.array_equal(one, want)
    four = oracle.tensorscale(A, B, 4.0)
    assert np.array_equal(oracle.bf16_bits_to_float(four), 4.0 * oracle.bf16_bits_to_float(one))


# ---- E4M3 output (the fp8 store of skill card "FlyDSL prefill MoE stage-2 fp8 partial")

def _e4m3_values():
    """The 126 positive finite E4M3FN values by code (1..126), from torch's decoder."""
    torch = pytest.importorskip("torch")
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_encoder_round_trips_every_finite_code():
    vals = _e4m3_values()
    codes = np.array([c for c in range(256) if not np.isnan(vals[c])], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(vals[codes].astype(np.float32)), codes)


def test_e4m3_encoder_ties_go_to_even_and_neighbours_to_nearest():
    vals = _e4m3_values()
    for c in range(0, 126):
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)            # exact: E4M3 midpoints have 5 significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == even, c
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1e9))
        assert oracle.e4m3_encode(np.array([below]))[0] == c
        assert oracle.e4m3_encode(np.array([above]))[0] == c + 1
        assert oracle.e4m3_encode(np.array([-mid]))[0] == 0x80 | even


def test_e4m3_encoder_saturates_and_keeps_the_sign_of_zero():
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    tiny = np.array([0.0, 2.0 ** -11, -0.0, -(2.0 ** -11)], dtype=np.float32)   # below half the smallest subnormal
    assert list(oracle.e4m3_encode(tiny)) == [0x00, 0x00, 0x80, 0x80]


def test_e4m3_encoder_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(31))
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-14, 6, 100000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_blockscale_e4m3out_on_integer_inputs():
    """Integer codes, unit block scales: the sums are exact integers, known from an
    integer matmul; c_scale = 1/8 and the result is torch's E4M3 cast of sum/8."""
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(32))
    M, N, K = 6, 20, 256
    va = rng.integers(-2, 3, size=(M, K))
    vb = rng.integers(-2, 3, size=(N, K))
    enc = {v: oracle.e4m3_encode(np.array([v], dtype=np.float32))[0] for v in (-2, -1, 0, 1, 2)}
    A = np.vectorize(enc.get)(va).astype(np.uint8)
    B = np.vectorize(enc.get)(vb).astype(np.uint8)
    sa = np.ones((M, K // 128), np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), np.float32)
    codes, y = oracle.blockscale_e4m3out(A, sa, B, sb, 0.125)
    exact = (va @ vb.T).astype(np.float64) / 8
    assert np.array_equal(y, exact.astype(np.float32))
    ref = torch.from_numpy(np.clip(exact, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(codes, ref.numpy())


# ---- grouped MoE stage-1 (skill card "FlyDSL decode MoE stage-1 blkmap")

P30 = 1 << 30


def test_moe_leaders_worked_example():
    """Runs of 3, 1, 2, (unused), 4 blocks: ceil(k/2) leaders per run, pairs
    first, a trailing odd block solo (procedure step 2); the count is the valid
    blocks minus the pairs (procedure step 3)."""
    table = [0, 0, 0, 1, 2, 2, -1, 3, 3, 3, 3]
    assert oracle.moe_leaders(table, 4, pair=True).tolist() == [0 | P30, 2, 3, 4 | P30, 7 | P30, 9 | P30]
    assert oracle.moe_leaders(table, 4, pair=False).tolist() == [0, 1, 2, 3, 4, 5, 7, 8, 9, 10]
    # an expert id past the expert count leads nothing
    assert oracle.moe_leaders([0, 5, 5, 1], 4, pair=True).tolist() == [0, 3]
    assert oracle.moe_leaders([], 4).tolist() == []


def test_moe_leaders_cover_every_valid_block_once():
    rng = np.random.Generator(np.random.PCG64(41))
    for _ in range(50):
        E = int(rng.integers(1, 9))
        runs = rng.integers(1, 6, size=int(rng.integers(1, 12)))
        experts = np.sort(rng.choice(np.arange(-1, E + 1), size=len(runs)))
        table = np.repeat(experts, runs)
        lead = oracle.moe_leaders(table, E, pair=True)
        covered = []
        for v in lead.tolist():
            b, two = v & (P30 - 1), bool(v & P30)
            covered.append(b)
            if two:
                assert table[b + 1] == table[b]
                covered.append(b + 1)
        valid = [b for b in range(len(table)) if 0 <= table[b] < E]
        assert sorted(covered) == valid
        pairs = sum(1 for v in lead.tolist() if v & P30)
        assert len(lead) == len(valid) - pairs


def test_moe_gemm_oracle_reduces_to_the_dense_gemm():
    """One expert owning every block is the dense blockscale GEMM; E identical
    experts under any block map give the same rows; unused blocks are undefined."""
    x = workloads.make_moe_inputs(192, 2, 4, 256, 256, seed=3)
    M = x.A.shape[0]
    dense = oracle.blockscale(x.A, x.a_scale, x.B[0], x.b_scale[0])
    one = np.zeros(x.n_blocks, np.int32)
    C, d = oracle.moe_gemm(x.A, x.a_scale, x.B, x.b_scale, one, 4)
    assert d.all() and np.array_equal(C, dense)
    Bsame = np.repeat(x.B[:1], 4, axis=0)
    sbsame = np.repeat(x.b_scale[:1], 4, axis=0)
    C2, d2 = oracle.moe_gemm(x.A, x.a_scale, Bsame, sbsame, x.block_expert, 4)
    assert d2.all() and np.array_equal(C2, dense)
    partial = x.block_expert.copy()
    partial[-1] = -1
    C3, d3 = oracle.moe_gemm(x.A, x.a_scale, x.B, x.b_scale, partial, 4)
    assert not d3[M - 64:].any() and d3[:M - 64].all()


def test_moe_routing_layout():
    x = workloads.make_moe_inputs(300, 3, 8, 128, 256, seed=4, skew=1.0)
    assert x.A.shape[0] == 64 * x.n_blocks and np.all(np.diff(x.block_expert) >= 0)
    real = x.row_token >= 0
    assert real.sum() == 300 * 3                      # every (token, slot) routed once
    for b in range(x.n_blocks):                        # padding only at the end of an expert's rows
        rows = x.row_token[64 * b:64 * b + 64]
        if (rows < 0).any():
            assert np.all(rows[np.argmax(rows < 0):] < 0)
    assert np.all(x.A[~real] == 0)


def test_mxfp8_e4m3out_on_integer_inputs():
    """Integer codes with unit ue8m0 scales (byte 127): exact integer sums; c_scale
    = 1/4 and the codes are torch's E4M3 cast of sum/4."""
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(33))
    M, N, K = 5, 24, 128
    va = rng.integers(-2, 3, size=(M, K))
    vb = rng.integers(-2, 3, size=(N, K))
    enc = {v: oracle.e4m3_encode(np.array([v], dtype=np.float32))[0] for v in (-2, -1, 0, 1, 2)}
    A = np.vectorize(enc.get)(va).astype(np.uint8)
    B = np.vectorize(enc.get)(vb).astype(np.uint8)
    ea = np.full((M, K // 32), 127, np.uint8)
    eb = np.full((N, K // 32), 127, np.uint8)
    codes, y = oracle.mxfp8_e4m3out(A, ea, B, eb, 0.25)
    exact = (va @ vb.T).astype(np.float64) / 4
    assert np.array_equal(y, exact.astype(np.float32))
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
