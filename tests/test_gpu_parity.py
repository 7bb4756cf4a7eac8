"""GPU path vs the CPU oracle (needs a GB300).

Every case goes through the C ABI (via the ctypes binding) on seeded inputs and
compares element by element with the oracle: bit-exact where the result is an
exact integer, within the stated tolerance otherwise.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import compare, compare_e4m3, compare_rows, run_blockscale, run_mxfp8, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_block_scaled_e4m3_gb300  # noqa: F401  (fails loudly if the library is missing)


def _int_codes(vals):
    lut = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    return np.vectorize(lut.get)(vals).astype(np.uint8)


# ---------------------------------------------------------------- exact cases

@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (200, 136, 384)])
def test_blockscale_integer_inputs_bit_exact(M, N, K):
    rng = np.random.Generator(np.random.PCG64(M + N + K))
    va = rng.integers(-1, 2, size=(M, K))
    vb = rng.integers(-1, 2, size=(N, K))
    A, B = _int_codes(va), _int_codes(vb)
    sa = np.ones((M, K // 128), np.float32)
    sb = np.ones(((N + 127) // 128, K // 128), np.float32)
    got = run_blockscale(A, sa, B, sb)
    ref = oracle.blockscale(A, sa, B, sb)
    assert np.array_equal(got, ref)
    exact = va @ vb.T
    if np.abs(exact).max() <= 256:          # every such integer is a bf16 value
        assert np.array_equal(oracle.bf16_bits_to_float(got), exact.astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 136, 384)])
def test_mxfp8_integer_inputs_bit_exact(M, N, K):
    rng = np.random.Generator(np.random.PCG64(7 + M))
    va = rng.integers(-1, 2, size=(M, K))
    vb = rng.integers(-1, 2, size=(N, K))
    A, B = _int_codes(va), _int_codes(vb)
    ea = np.full((M, K // 32), 127, np.uint8)
    eb = np.full((N, K // 32), 127, np.uint8)
    got = run_mxfp8(A, ea, B, eb)
    assert np.array_equal(got, oracle.mxfp8(A, ea, B, eb))


def test_blockscale_per_block_scales_bit_exact():
    """Integer operands, power-of-two scales that differ per row, per K block and per N block."""
    M, N, K = 256, 384, 512
    rng = np.random.Generator(np.random.PCG64(21))
    A = _int_codes(rng.integers(-2, 3, size=(M, K)))
    B = _int_codes(rng.integers(-2, 3, size=(N, K)))
    sa = np.ldexp(np.float32(1), rng.integers(-3, 4, size=(M, K // 128))).astype(np.float32)
    sb = np.ldexp(np.float32(1), rng.integers(-3, 4, size=(N // 128, K // 128))).astype(np.float32)
    assert np.array_equal(run_blockscale(A, sa, B, sb), oracle.blockscale(A, sa, B, sb))


def test_mxfp8_per_group_scales_bit_exact():
    """Integer operands with ue8m0 scales that differ per row and per 32-wide group:
    pins which tensor-memory scale byte each row and K slice uses."""
    M, N, K = 256, 512, 512
    rng = np.random.Generator(np.random.PCG64(22))
    A = _int_codes(rng.integers(-2, 3, size=(M, K)))
    B = _int_codes(rng.integers(-2, 3, size=(N, K)))
    ea = rng.integers(124, 131, size=(M, K // 32)).astype(np.uint8)
    eb = rng.integers(124, 131, size=(N, K // 32)).astype(np.uint8)
    got = run_mxfp8(A, ea, B, eb)
    ref = oracle.mxfp8(A, ea, B, eb)
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        raise AssertionError(f"{len(bad)} mismatches, rows%128 {np.unique(bad[:, 0] % 128)[:20]}, "
                             f"cols%256 {np.unique(bad[:, 1] % 256)[:20]}")


def test_zero_operand_gives_zero():
    x = workloads.make_blockscale_inputs(256, 256, 256, seed=1)
    got = run_blockscale(np.zeros_like(x.A), x.a_scale, x.B, x.b_scale)
    assert np.all(got == 0)


# -------------------------------------------------------- tolerance cases

def test_blockscale_small_config_seed0():
    """256 x 512 x 512, the smallest workload, full output."""
    x = workloads.make_blockscale_inputs(256, 512, 512, seed=0)
    compare(run_blockscale(x.A, x.a_scale, x.B, x.b_scale), oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale),
            "bs 256x512x512")


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (64, 128, 256), (127, 136, 128), (129, 264, 768),
                                   (300, 520, 1280), (513, 1032, 384), (1000, 2056, 1024)])
def test_blockscale_tails(M, N, K):
    x = workloads.make_blockscale_inputs(M, N, K, seed=M)
    compare(run_blockscale(x.A, x.a_scale, x.B, x.b_scale), oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale),
            f"bs {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (64, 256, 256), (127, 136, 1280), (300, 520, 2048),
                                   (1024, 640, 1280)])
def test_mxfp8_tails(M, N, K):
    x = workloads.make_mxfp8_inputs(M, N, K, seed=M)
    compare(run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0),
            f"mx {M}x{N}x{K}")


def test_scales_are_applied():
    """A changed scale must change exactly the rows / blocks it governs."""
    x = workloads.make_blockscale_inputs(256, 512, 512, seed=5)
    base = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    sa = x.a_scale.copy()
    sa[37, 2] *= np.float32(4.0)
    changed = run_blockscale(x.A, sa, x.B, x.b_scale)
    diff_rows = np.unique(np.argwhere(changed != base)[:, 0])
    assert diff_rows.tolist() == [37]
    sb = x.b_scale.copy()
    sb[3, 1] *= np.float32(0.25)
    changed = run_blockscale(x.A, x.a_scale, x.B, sb)
    cols = np.unique(np.argwhere(changed != base)[:, 1])
    assert cols.min() >= 384 and cols.max() < 512
    y = workloads.make_mxfp8_inputs(256, 512, 512, seed=5)
    mbase = run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
    eb = y.b_e8m0.copy()
    eb[300, :] += 1
    ch = run_mxfp8(y.A, y.a_e8m0, y.B, eb)
    assert np.unique(np.argwhere(ch != mbase)[:, 1]).tolist() == [300]
    assert np.array_equal(oracle.bf16_bits_to_float(ch[:, 300]), 2 * oracle.bf16_bits_to_float(mbase[:, 300]))


def test_blockscale_and_mxfp8_agree_on_power_of_two_scales():
    rng = np.random.Generator(np.random.PCG64(9))
    M, N, K = 256, 384, 768
    x = workloads.make_blockscale_inputs(M, N, K, seed=9)
    ja = rng.integers(-8, -2, size=(M, K // 128))
    jb = rng.integers(-10, -4, size=((N + 127) // 128, K // 128))
    sa = np.ldexp(np.float32(1), ja).astype(np.float32)
    sb = np.ldexp(np.float32(1), jb).astype(np.float32)
    ea = np.repeat(ja + 127, 4, axis=1).astype(np.uint8)
    eb = np.repeat(np.repeat(jb + 127, 128, axis=0)[:N], 4, axis=1).astype(np.uint8)
    g1 = run_blockscale(x.A, sa, x.B, sb)
    g2 = run_mxfp8(x.A, ea, x.B, eb)
    ref = oracle.blockscale(x.A, sa, x.B, sb)
    compare(g1, ref, "bs pow2")
    compare(g2, ref, "mx pow2")


def test_repeat_calls_bitwise_identical_and_config_recorded():
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_blockscale_inputs(512, 1024, 1024, seed=3)
    a = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    cid = f.last_config_id()
    b = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    assert np.array_equal(a, b)
    assert f.decode_config(cid)["kind"].startswith("blockscale")


def test_pack_a_scale_bit_exact():
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    rng = np.random.Generator(np.random.PCG64(4))
    for M, K in [(1, 128), (5, 256), (130, 768), (4097, 7168)]:
        sa = rng.standard_normal((M, K // 128)).astype(np.float32)
        out = f.pack_a_scale(to_dev(sa), K)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), workloads.a_scale_to_kmajor(sa))


# every built kernel configuration, forced through the override
# one-CTA 128x256, 128x128 (one CTA per tile), 128x256 stream-K, three-stage
# 128x256 (both schedules), CTA-pair 256x256 (both schedules)
BS_CONFIGS = [1256411, 1128611, 1256412, 1256311, 1256312, 3256411, 3256412]
MX_CONFIGS = [2256411, 2128611, 2256412, 2128612, 5256611]


@pytest.fixture
def override():
    import fp8_block_scaled_e4m3_gb300 as f
    yield f.set_config_override
    f.set_config_override(0)


@pytest.mark.parametrize("cfg", BS_CONFIGS)
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (300, 520, 1280), (513, 1032, 384), (1, 8, 128)])
def test_blockscale_every_config(override, cfg, M, N, K):
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    override(cfg - (cfg // 10 % 10) * 10 + raster * 10)
    x = workloads.make_blockscale_inputs(M, N, K, seed=cfg % 97 + M)
    got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    assert f.last_config_id() == cfg - (cfg // 10 % 10) * 10 + raster * 10
    compare(got, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), f"bs cfg {cfg} {M}x{N}x{K}")


@pytest.mark.parametrize("cfg", BS_CONFIGS)
def test_blockscale_every_config_integer_exact(override, cfg):
    override(cfg)
    rng = np.random.Generator(np.random.PCG64(5))
    M, N, K = 384, 640, 512
    A = _int_codes(rng.integers(-2, 3, size=(M, K)))
    B = _int_codes(rng.integers(-2, 3, size=(N, K)))
    sa = np.ldexp(np.float32(1), rng.integers(-3, 4, size=(M, K // 128))).astype(np.float32)
    sb = np.ldexp(np.float32(1), rng.integers(-3, 4, size=((N + 127) // 128, K // 128))).astype(np.float32)
    assert np.array_equal(run_blockscale(A, sa, B, sb), oracle.blockscale(A, sa, B, sb))


@pytest.mark.parametrize("cfg", MX_CONFIGS)
@pytest.mark.parametrize("M,N,K", [(300, 520, 1280), (129, 136, 256)])
def test_mxfp8_every_config(override, cfg, M, N, K):
    override(cfg)
    x = workloads.make_mxfp8_inputs(M, N, K, seed=cfg % 89 + M)
    compare(run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0),
            f"mx cfg {cfg} {M}x{N}x{K}")


def test_config_override_rejects_unbuilt_ids():
    import fp8_block_scaled_e4m3_gb300 as f
    with pytest.raises(f.Fp8bsError):
        f.set_config_override(1999911)
    f.set_config_override(0)


def _packed_reference(e8m0, K):
    """The packed scale layout written out from its definition in include/fp8bs.h."""
    rows = e8m0.shape[0]
    RB, KS = (rows + 127) // 128, K // 128
    out = np.zeros(RB * KS * 512, np.uint8)
    for rb in range(RB):
        for ks in range(KS):
            base = (rb * KS + ks) * 512
            for r in range(128):
                if rb * 128 + r < rows:
                    for j in range(4):
                        out[base + (r % 32) * 16 + (r // 32) * 4 + j] = e8m0[rb * 128 + r, 4 * ks + j]
    return out


@pytest.mark.parametrize("rows,K", [(1, 128), (130, 256), (257, 1280)])
def test_pack_mx_scales_bit_exact(rows, K):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    rng = np.random.Generator(np.random.PCG64(rows))
    e = rng.integers(0, 255, size=(rows, K // 32), dtype=np.uint8)
    out = torch.full((f.packed_scale_bytes(rows, K),), 0xAB, dtype=torch.uint8, device="cuda")
    f.pack_mx_scales(to_dev(e), K, out=out)
    assert np.array_equal(out.cpu().numpy(), _packed_reference(e, K))


@pytest.mark.parametrize("M,N,K", [(200, 136, 384), (1024, 640, 1280)])
def test_mxfp8_packed_entry_matches_oracle(M, N, K):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_mxfp8_inputs(M, N, K, seed=M + 1)
    a_sf = f.pack_mx_scales(to_dev(x.a_e8m0), K)
    b_sf = f.pack_mx_scales(to_dev(x.b_e8m0), K)
    C = f.gemm_mxfp8_packed(to_dev(x.A), a_sf, to_dev(x.B), b_sf)
    assert f.get_status() == 0
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    compare(got, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), f"mx packed {M}x{N}x{K}")


def test_m_zero_is_noop():
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    A = torch.empty((0, 128), dtype=torch.uint8, device="cuda")
    B = torch.zeros((8, 128), dtype=torch.uint8, device="cuda")
    sa = torch.zeros((1, 0), dtype=torch.float32, device="cuda")
    sb = torch.ones((1, 1), dtype=torch.float32, device="cuda")
    C = f.gemm_blockscale(A, sa, B, sb)
    assert C.shape == (0, 8)


# ------------------------------------------------ full-size workloads (whole output)

def _check_full_size(kind, M, N, K, seed):
    """The workload at its full size in the configuration the library chooses
    (the one the benchmark times), compared element by element with the oracle
    over the whole of C."""
    x = workloads.make_inputs(kind, M, N, K, seed)
    if kind == "bs":
        got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
        ref = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale)
    else:
        got = run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)
        ref = oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)
    return compare_rows(got, ref, f"{kind} {M}x{N}x{K} seed {seed}")


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("name", ["bs_narrowN_4096x2048x7168", "bs_narrowN_16384x1536x7168",
                                  "bs_Klight_16384x7168x768", "bs_wideN_4096x65536x1536"])
def test_full_blockscale(name, seed):
    w = workloads.WORKLOADS[name]
    assert seed in w["seeds"]
    _check_full_size("bs", w["M"], w["N"], w["K"], seed)


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("M", [1024, 2048, 4096, 16384])
@pytest.mark.parametrize("N,K", [(5120, 2048), (8192, 1280)])
def test_full_mxfp8(M, N, K, seed):
    _check_full_size("mx", M, N, K, seed)


@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("M,N,K", [(4096, 2048, 7168), (1000, 2824, 1408), (384, 256, 128), (4096, 5120, 384),
                                   (512, 512, 8192), (600, 520, 4096)])
def test_blockscale_pair_kernel_full_output(override, M, N, K, sched):
    """The CTA-pair kernel (256 x 256 tiles, whole-tile C buffer) on the whole
    of C, one pair per tile and stream-K: the full-size narrow-N workload;
    ragged shapes whose last pair tile is cut in M (the odd CTA's rows past M)
    and in N (a 128-column half past N); a shape with several tiles per CTA
    pair and few K blocks (the tile buffer's reuse across tiles; under
    stream-K, whole waves first and then tiles of three K blocks cut between
    pairs); and, under stream-K, tiles whose K blocks are cut between four
    pairs, so that a finisher adds three partials, with every row of the odd
    CTA of the last M tile past M (no hand-off for those warps)."""
    import fp8_block_scaled_e4m3_gb300 as f
    cid = 3256400 + 10 * (1 if M >= N else 0) + sched
    override(cid)
    x = workloads.make_blockscale_inputs(M, N, K, seed=M + N)
    got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    assert f.last_config_id() == cid
    compare_rows(got, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), f"bs pair {M}x{N}x{K}")


def test_raster_group_sizes_give_the_same_bits(override):
    """The tile order (raster direction and group size) changes which CTA computes
    which tile, never a tile's arithmetic: every order gives the same bits, for
    both GEMMs and with a group that does not divide the panel count."""
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_blockscale_inputs(600, 1800, 512, seed=91)
    y = workloads.make_mxfp8_inputs(600, 1800, 512, seed=92)
    ref_bs = ref_mx = None
    try:
        for raster in (0, 1):
            override(1256401 + 10 * raster)
            for group in (1, 2, 3, 8):
                f.set_raster_group(group)
                got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
                ref_bs = got if ref_bs is None else ref_bs
                assert np.array_equal(got, ref_bs), (raster, group)
        override(0)
        for group in (1, 4, 7):
            f.set_raster_group(group)
            got = run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
            ref_mx = got if ref_mx is None else ref_mx
            assert np.array_equal(got, ref_mx), group
    finally:
        f.set_raster_group(0)
    compare(ref_bs, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), "raster groups, blockscale")
    compare(ref_mx, oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), "raster groups, mxfp8")


# ---------------------------------------------------------------- stream-K
@pytest.mark.parametrize("cfg", [1256402, 1256302])
def test_stream_k_repeated_calls_same_bits(override, cfg):
    """Twenty back-to-back calls of a stream-K configuration on a shape with
    whole waves before the stream-K range (raster 0): the first matches the
    oracle, every later one gives the same bits (the hand-off order is fixed).
    With three stages a stage's uses alternate between step parities; this is
    the case that exposed a parity wait two phases behind its barrier."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 2048, 8192, 1536
    override(cfg)
    x = workloads.make_blockscale_inputs(M, N, K, seed=81)
    dA, dB = to_dev(x.A), to_dev(x.B)
    dsa, dsb = to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.b_scale)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(64 << 20, dtype=torch.int32, device="cuda")
    f.gemm_blockscale(dA, dsa, dB, dsb, C=C)
    assert f.get_status() == 0 and f.last_config_id() == cfg
    first = C.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    compare_rows(first, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), f"stream-K {cfg} first call")
    for i in range(19):
        flush.fill_(i)
        C.fill_(float("nan"))
        f.gemm_blockscale(dA, dsa, dB, dsb, C=C)
        assert f.get_status() == 0
        assert np.array_equal(C.view(torch.int16).cpu().numpy().view(np.uint16), first), f"call {i + 2} differs"


@pytest.mark.parametrize("cfg", [1256412])
@pytest.mark.parametrize("M,N,K", [(256, 512, 7168), (130, 264, 3840), (1100, 776, 2048)])
def test_stream_k_tiles_cut_between_many_ctas(override, cfg, M, N, K):
    """Few tiles and long K: each tile is cut between several CTAs (every one but
    the first publishing a partial), and ragged M/N tails sit in cut tiles."""
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    cid = cfg - (cfg // 10 % 10) * 10 + raster * 10
    override(cid)
    x = workloads.make_blockscale_inputs(M, N, K, seed=M + N)
    got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    assert f.last_config_id() == cid
    compare(got, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), f"stream-K {cid} {M}x{N}x{K}")


def test_stream_k_back_to_back_calls_use_fresh_partials(override):
    """Consecutive calls reuse the pooled workspace: each must see only its own
    partials (per-call tokens, flags reset by the finishers)."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(1256412)
    M, N, K = 512, 768, 4096
    xs = [workloads.make_blockscale_inputs(M, N, K, seed=s) for s in (21, 22)]
    dev = [(to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.B),
            to_dev(np.ascontiguousarray(x.b_scale))) for x in xs]
    outs = [f.gemm_blockscale(*d) for d in (dev[0], dev[1], dev[0])]   # no sync in between
    assert f.get_status() == 0
    bits = [o.view(torch.int16).cpu().numpy().view(np.uint16) for o in outs]
    for b, x in zip(bits, (xs[0], xs[1], xs[0])):
        compare(b, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), "stream-K back to back")
    assert np.array_equal(bits[0], bits[2])


def test_blockscale_cuda_graph_replay(override):
    """Both schedules captured in a CUDA graph (the stream-K workspace becomes a
    graph allocation) and replayed on new input contents."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 384, 640, 2048
    for cid in (1256411, 1256412):
        override(cid)
        x0, x1 = (workloads.make_blockscale_inputs(M, N, K, seed=s) for s in (31, 32))
        d = [to_dev(x0.A), to_dev(workloads.a_scale_to_kmajor(x0.a_scale)), to_dev(x0.B),
             to_dev(np.ascontiguousarray(x0.b_scale))]
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        f.gemm_blockscale(*d, C=C)          # first call outside the capture (device set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            f.gemm_blockscale(*d, C=C)
        for x in (x1, x0, x1):
            d[0].copy_(to_dev(x.A))
            d[1].copy_(to_dev(workloads.a_scale_to_kmajor(x.a_scale)))
            d[2].copy_(to_dev(x.B))
            d[3].copy_(to_dev(np.ascontiguousarray(x.b_scale)))
            C.zero_()
            g.replay()
            assert f.get_status() == 0
            got = C.view(torch.int16).cpu().numpy().view(np.uint16)
            compare(got, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), f"graph replay {cid}")
        del g


def test_stream_k_after_whole_waves(override):
    """320 tiles on 152 SMs under stream-K: one wave one CTA per tile, then
    stream-K over the remaining 168 tiles, whose ranges start mid-tile. Checked
    on whole row blocks from both parts."""
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 5120, 2048, 2048
    if f.device_info()["num_sms"] != 152:
        pytest.skip("the wave split below is worked out for 152 SMs")
    override(1256412)
    x = workloads.make_blockscale_inputs(M, N, K, seed=77)
    got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    assert f.last_config_id() == 1256412
    # raster N-inner (M >= N): tile t = 8 * mb + nb; tiles 0..151 come first
    rows = np.concatenate([np.arange(mb * 128, mb * 128 + 128) for mb in (0, 18, 19, 25, 39)])
    ref = oracle.blockscale(x.A[rows], x.a_scale[rows], x.B, x.b_scale)
    compare(got[rows], ref, "stream-K after whole waves")


@pytest.mark.parametrize("cid", [2256401, 2256402])
def test_mxfp8_cuda_graph_replay(override, cid):
    """fp8mx_gemm (scale pack + GEMM, pooled workspace; stream-K workspace too)
    captured in a CUDA graph and replayed on new input contents."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(cid)
    M, N, K = 300, 520, 1280
    x0, x1 = (workloads.make_mxfp8_inputs(M, N, K, seed=s) for s in (41, 42))
    d = [to_dev(x0.A), to_dev(x0.a_e8m0), to_dev(x0.B), to_dev(x0.b_e8m0)]
    for entry in (f.gemm_mxfp8,):
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        entry(*d, C=C)                      # first call outside the capture (device set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            entry(*d, C=C)
        for x in (x1, x0):
            for dst, src in zip(d, (x.A, x.a_e8m0, x.B, x.b_e8m0)):
                dst.copy_(to_dev(src))
            C.zero_()
            g.replay()
            assert f.get_status() == 0
            got = C.view(torch.int16).cpu().numpy().view(np.uint16)
            compare(got, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), f"graph replay {entry.__name__}")
        del g


@pytest.mark.parametrize("width", [256, 128])
@pytest.mark.parametrize("M,N,K", [(256, 512, 7168), (130, 264, 3840), (1100, 776, 2048), (32, 5120, 2048),
                                   (1, 520, 1280), (70, 1024, 4096)])
def test_mxfp8_stream_k_tiles_cut_between_many_ctas(override, width, M, N, K):
    """MXFP8 under stream-K, both tile widths: few tiles (decode-like M
    included, where only the live row groups hand off), each accumulated in
    pieces by several CTAs; ragged tails inside cut tiles."""
    import fp8_block_scaled_e4m3_gb300 as f
    cid = (2256402 if width == 256 else 2128602) + (10 if M >= N else 0)
    override(cid)
    x = workloads.make_mxfp8_inputs(M, N, K, seed=M + N + 5)
    got = run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)
    assert f.last_config_id() == cid
    compare(got, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), f"mx stream-K {M}x{N}x{K}")


def test_mxfp8_stream_k_back_to_back_calls(override):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(2256402)
    M, N, K = 256, 1024, 4096
    xs = [workloads.make_mxfp8_inputs(M, N, K, seed=s) for s in (51, 52)]
    dev = [(to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0)) for x in xs]
    outs = [f.gemm_mxfp8(*d) for d in (dev[0], dev[1], dev[0])]   # no sync in between
    assert f.get_status() == 0
    bits = [o.view(torch.int16).cpu().numpy().view(np.uint16) for o in outs]
    for b, x in zip(bits, (xs[0], xs[1], xs[0])):
        compare(b, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), "mx stream-K back to back")
    assert np.array_equal(bits[0], bits[2])


def test_mxfp8_stream_k_after_whole_waves(override):
    """320 tiles of 16 K steps on 152 SMs under stream-K: one wave one CTA per
    tile, then stream-K over the rest (ranges start mid-tile); whole row blocks
    from both."""
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 5120, 2048, 2048
    if f.device_info()["num_sms"] != 152:
        pytest.skip("the wave split below is worked out for 152 SMs")
    override(2256412)
    x = workloads.make_mxfp8_inputs(M, N, K, seed=78)
    got = run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)
    assert f.last_config_id() == 2256412
    rows = np.concatenate([np.arange(mb * 128, mb * 128 + 128) for mb in (0, 18, 19, 25, 39)])
    compare(got[rows], oracle.mxfp8(x.A[rows], x.a_e8m0[rows], x.B, x.b_e8m0), "mx stream-K after whole waves")


# ------------------------------------------------ promote-free ceiling twin
@pytest.mark.parametrize("cfg", [4256411, 4128611, 4256412])
@pytest.mark.parametrize("M,N,K", [(300, 520, 1280), (129, 136, 256), (1, 8, 128), (640, 768, 7168)])
def test_tensorscale_every_config(override, cfg, M, N, K):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    cid = cfg - (cfg // 10 % 10) * 10 + raster * 10
    override(cid)
    x = workloads.make_tensorscale_inputs(M, N, K, seed=M + K)
    alpha = float(x.alpha)
    out = f.gemm_tensorscale(to_dev(x.A), to_dev(x.B), alpha)
    assert f.get_status() == 0
    assert f.last_config_id() == cid
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    compare(got, oracle.tensorscale(x.A, x.B, alpha), f"tensorscale {cid} {M}x{N}x{K}")


def test_tensorscale_integer_exact():
    """Small integer codes and a power-of-two alpha: every fp32 sum is exact, so the
    twin must equal the oracle bit for bit."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    rng = np.random.Generator(np.random.PCG64(9))
    M, N, K = 384, 640, 1024
    A = _int_codes(rng.integers(-2, 3, size=(M, K)))
    B = _int_codes(rng.integers(-2, 3, size=(N, K)))
    out = f.gemm_tensorscale(to_dev(A), to_dev(B), 0.25)
    assert f.get_status() == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.tensorscale(A, B, 0.25))


# ------------------------------------------------ E4M3 output (epilogue fusion)
def _c_scale(x, rows=None):
    """16 / rms(C) rounded to a power of two, from the oracle's bf16 result: the
    pre-store values sit mid-range in E4M3."""
    ref = oracle.bf16_bits_to_float(oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, rows=rows)).astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    return float(2.0 ** np.round(np.log2(16.0 / rms)))


def _run_e4m3out(x, c_scale):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    out = f.gemm_blockscale_e4m3out(to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.B),
                                    to_dev(np.ascontiguousarray(x.b_scale)), c_scale)
    assert f.get_status() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("cfg", [1256411, 1128611, 1256412])
@pytest.mark.parametrize("M,N,K", [(300, 528, 1280), (129, 144, 256), (1, 16, 128), (640, 768, 7168)])
def test_blockscale_e4m3out_every_config(override, cfg, M, N, K):
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    cid = cfg - (cfg // 10 % 10) * 10 + raster * 10
    override(cid)
    x = workloads.make_blockscale_inputs(M, N, K, seed=M + 3 * N)
    s = _c_scale(x)
    got = _run_e4m3out(x, s)
    assert f.last_config_id() == cid
    codes, y = oracle.blockscale_e4m3out(x.A, x.a_scale, x.B, x.b_scale, s)
    compare_e4m3(got, codes, y, s, f"e4m3out {cid} {M}x{N}x{K}")


def test_blockscale_e4m3out_saturates():
    """A c_scale far too large: every output of magnitude > 448 / c_scale is +-448."""
    x = workloads.make_blockscale_inputs(256, 512, 512, seed=9)
    s = _c_scale(x) * 64
    got = _run_e4m3out(x, s)
    codes, y = oracle.blockscale_e4m3out(x.A, x.a_scale, x.B, x.b_scale, s)
    assert (np.abs(y) > 448).mean() > 0.1
    assert np.all((got[np.abs(y) > 464] & 0x7F) == 0x7E)
    compare_e4m3(got, codes, y, s, "e4m3out saturating")


def test_blockscale_e4m3out_full_size_sampled_rows():
    """16384x7168x768 (the K-light layer whose C write the fp8 store halves):
    sampled whole rows against the oracle. C has rms ~0.02 * sqrt(768) = 0.55,
    so c_scale = 32 puts it mid-range."""
    M, N, K = 16384, 7168, 768
    x = workloads.make_blockscale_inputs(M, N, K, seed=0)
    rng = np.random.Generator(np.random.PCG64(123))
    rows = np.sort(rng.choice(M, 48, replace=False))
    s = 32.0
    got = _run_e4m3out(x, s)
    codes, y = oracle.blockscale_e4m3out(x.A[rows], x.a_scale[rows], x.B, x.b_scale, s)
    compare_e4m3(got[rows], codes, y, s, "e4m3out 16384x7168x768")


def test_e4m3out_feeds_the_next_gemm_with_one_scale():
    """The consumer side: C8 is the A operand of a second blockscale GEMM whose
    a_scale is 1/c_scale everywhere (the same scale, one source of truth)."""
    M, N1, K1, N2 = 256, 1024, 2048, 384
    x = workloads.make_blockscale_inputs(M, N1, K1, seed=44)
    z = workloads.make_blockscale_inputs(1, N2, N1, seed=46)      # its B: [N2, N1] with 128x128 block scales
    s = _c_scale(x)
    c8 = _run_e4m3out(x, s)
    codes, y = oracle.blockscale_e4m3out(x.A, x.a_scale, x.B, x.b_scale, s)
    compare_e4m3(c8, codes, y, s, "first GEMM")
    sa2 = np.full((M, N1 // 128), np.float32(1.0 / s), dtype=np.float32)
    got = run_blockscale(c8, sa2, z.B, z.b_scale)
    compare(got, oracle.blockscale(codes, sa2, z.B, z.b_scale), "E4M3 C as the next A")


# ------------------------------------------------ grouped MoE stage-1 GEMM
def _moe_dev(x):
    return (to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.B), to_dev(x.b_scale),
            to_dev(x.block_expert))


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("case", ["empty", "one", "mixed", "chunks", "long_run"])
def test_moe_leaders_kernel_matches_oracle(pair, case):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    rng = np.random.Generator(np.random.PCG64(7))
    E = 16
    if case == "empty":
        table = np.zeros(0, np.int32)
    elif case == "one":
        table = np.array([3], np.int32)
    elif case == "mixed":
        table = np.repeat(np.sort(rng.choice(np.arange(-1, E + 2), 40)), rng.integers(1, 6, 40)).astype(np.int32)
    elif case == "chunks":   # runs that straddle the 1024-block chunks of the scan
        table = np.repeat(np.arange(E), rng.integers(150, 260, E)).astype(np.int32)
    else:                    # one run of 2501 blocks, then others
        table = np.concatenate([np.full(2501, 2), np.full(3, 5), np.full(1030, 7), [-1, -1]]).astype(np.int32)
    be = torch.from_numpy(table).cuda() if len(table) else torch.zeros(0, dtype=torch.int32, device="cuda")
    lead, n = f.moe_leaders(be, E, pair=pair)
    torch.cuda.synchronize()
    want = oracle.moe_leaders(table, E, pair=pair)
    assert int(n.item()) == len(want)
    assert np.array_equal(lead.cpu().numpy()[:len(want)], want)


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("cid", [0, 1256401, 1128601])
def test_moe_gemm_matches_oracle(override, pair, cid):
    """Skewed routing (runs of 1..many blocks: pairs and solo tails), an unused
    block, both tile widths; rows of the unused block keep their sentinel."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    if cid:
        override(cid)
    x = workloads.make_moe_inputs(512, 2, 8, 384, 512, seed=11, skew=1.2)
    x.block_expert[-1] = -1                       # the last block is unused
    A, sa, B, sb, be = _moe_dev(x)
    lead, n = f.moe_leaders(be, 8, pair=pair)
    C = torch.full((x.A.shape[0], 384), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.gemm_moe(A, sa, B, sb, be, lead, n, C=C)
    assert f.get_status() == 0
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    want, defined = oracle.moe_gemm(x.A, x.a_scale, x.B, x.b_scale, x.block_expert, 8)
    assert not defined.all() and np.all(got[~defined] == got[~defined][0])   # untouched sentinel rows
    assert np.isnan(oracle.bf16_bits_to_float(got[~defined])).all()
    compare(got[defined], want[defined], f"moe pair={pair} cid={cid}")


def test_moe_gemm_graph_replay_with_new_routing():
    """Descriptor + GEMM captured once in a CUDA graph; replays after the
    block -> expert table changes in place give the new routing's result."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_moe_inputs(512, 2, 8, 256, 512, seed=12, skew=0.8)
    A, sa, B, sb, be = _moe_dev(x)
    lead = torch.empty(x.n_blocks, dtype=torch.int32, device="cuda")
    n = torch.empty(1, dtype=torch.int32, device="cuda")
    C = torch.empty((x.A.shape[0], 256), dtype=torch.bfloat16, device="cuda")
    f.moe_leaders(be, 8, leaders=lead, n_leaders=n)
    f.gemm_moe(A, sa, B, sb, be, lead, n, C=C)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f.moe_leaders(be, 8, leaders=lead, n_leaders=n)
        f.gemm_moe(A, sa, B, sb, be, lead, n, C=C)
    for table in (7 - x.block_expert, x.block_expert):
        be.copy_(torch.from_numpy(np.ascontiguousarray(table, dtype=np.int32)).cuda())
        g.replay()
        assert f.get_status() == 0
        got = C.view(torch.int16).cpu().numpy().view(np.uint16)
        want, _ = oracle.moe_gemm(x.A, x.a_scale, x.B, x.b_scale, table, 8)
        compare(got, want, "moe graph replay")
    del g


def test_moe_gemm_layer_sized_sampled_blocks():
    """1024 tokens, top-8 of 32 experts, N = 1536, K = 2048: every row of a
    sample of sort blocks against the oracle."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_moe_inputs(1024, 8, 32, 1536, 2048, seed=13, skew=0.5)
    A, sa, B, sb, be = _moe_dev(x)
    lead, n = f.moe_leaders(be, 32)
    C = f.gemm_moe(A, sa, B, sb, be, lead, n)
    assert f.get_status() == 0
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    rng = np.random.Generator(np.random.PCG64(14))
    for b in rng.choice(x.n_blocks, 6, replace=False):
        e = int(x.block_expert[b])
        rows = slice(64 * b, 64 * b + 64)
        want = oracle.blockscale(x.A[rows], x.a_scale[rows], x.B[e], x.b_scale[e])
        compare(got[rows], want, f"moe block {b}")


@pytest.mark.parametrize("cfg", [2256411, 2128611, 2256412, 2128612])
@pytest.mark.parametrize("M,N,K", [(300, 528, 1280), (129, 144, 256), (1, 16, 128)])
def test_mxfp8_e4m3out_every_config(override, cfg, M, N, K):
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    cid = cfg - (cfg // 10 % 10) * 10 + raster * 10
    override(cid)
    x = workloads.make_mxfp8_inputs(M, N, K, seed=M + 5 * N)
    ref = oracle.bf16_bits_to_float(oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)).astype(np.float64)
    s = float(2.0 ** np.round(np.log2(16.0 / (np.sqrt(np.mean(ref ** 2)) or 1.0))))
    got = f.gemm_mxfp8_e4m3out(to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0), s).cpu().numpy()
    assert f.get_status() == 0
    assert f.last_config_id() == cid - cid % 10 + 1     # the E4M3-output MXFP8 kernel runs one CTA per tile
    codes, y = oracle.mxfp8_e4m3out(x.A, x.a_e8m0, x.B, x.b_e8m0, s)
    compare_e4m3(got, codes, y, s, f"mx e4m3out {cid} {M}x{N}x{K}")


def test_shutdown_then_calls_set_up_again():
    """fp8bs_shutdown releases the pools; the next calls (pooled stream-K and
    scale workspaces included) set the device up again and are correct."""
    import fp8_block_scaled_e4m3_gb300 as f
    x = workloads.make_blockscale_inputs(256, 512, 7168, seed=61)   # stream-K shape (pooled workspace)
    y = workloads.make_mxfp8_inputs(200, 264, 1280, seed=62)        # scale pack (pooled workspace)
    want_x = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale)
    want_y = oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
    for _ in range(2):
        compare(run_blockscale(x.A, x.a_scale, x.B, x.b_scale), want_x, "bs around shutdown")
        compare(run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), want_y, "mx around shutdown")
        f.shutdown()


# ------------------------------------------------ seeded random shapes, every entry point
def _random_shapes(seed, n):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        M = int(rng.choice([1, 7, 64, 127, 128, 129, 200, 255, 256, 383, 520, 777]))
        N = int(rng.choice([16, 48, 128, 144, 256, 272, 400, 512, 528, 784]))
        K = 128 * int(rng.integers(1, 25))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("M,N,K", _random_shapes(2026, 12))
def test_random_shapes_every_entry_point(override, M, N, K):
    """Seeded random shapes (tails in M and N, K from 128 to 3072) through every
    entry point and every configuration that accepts the shape."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    raster = 1 if M >= N else 0
    x = workloads.make_blockscale_inputs(M, N, K, seed=M * 31 + N * 7 + K)
    want = oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale)
    for cfg in (0, 1256401, 1128601, 1256402, 3256401, 3256402):
        if cfg:
            override(cfg + raster * 10)
        compare(run_blockscale(x.A, x.a_scale, x.B, x.b_scale), want, f"bs cfg {cfg} {M}x{N}x{K}")
    override(0)
    y = workloads.make_mxfp8_inputs(M, N, K, seed=M * 13 + N + K)
    want_mx = oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
    for cfg in (0, 2256401, 2128601, 2256402, 2128602, 5256601):
        if cfg:
            override(cfg + raster * 10)
        compare(run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), want_mx, f"mx cfg {cfg} {M}x{N}x{K}")
    override(0)
    t = workloads.make_tensorscale_inputs(M, N, K, seed=M + N * 3 + K)
    for cfg in (0, 4256401, 4128601, 4256402):
        if cfg:
            override(cfg + raster * 10)
        got = f.gemm_tensorscale(to_dev(t.A), to_dev(t.B), float(t.alpha))
        assert f.get_status() == 0
        compare(got.view(torch.int16).cpu().numpy().view(np.uint16), oracle.tensorscale(t.A, t.B, float(t.alpha)),
                f"twin cfg {cfg} {M}x{N}x{K}")
    override(0)
    if N % 16 == 0:
        s = _c_scale(x)
        codes, yv = oracle.blockscale_e4m3out(x.A, x.a_scale, x.B, x.b_scale, s)
        compare_e4m3(_run_e4m3out(x, s), codes, yv, s, f"bs e4m3 {M}x{N}x{K}")


def _finite_codes(rng, shape):
    """Uniformly random E4M3 codes over all 254 finite encodings: both zeros,
    every subnormal, every normal up to +-448 (0x7F and 0xFF, the NaNs, skipped)."""
    r = rng.integers(0, 254, size=shape)
    return (r + (r >= 0x7F)).astype(np.uint8)


@pytest.mark.parametrize("M,N,K", [(200, 136, 384), (300, 520, 1280)])
def test_uniform_random_codes_every_entry_point(override, M, N, K):
    """The whole E4M3 code range on the GPU: uniformly random finite codes on
    both operands (subnormals and +-448 included), with scales near 2^-9 per
    side so that C is O(1) and the absolute term of the tolerance matters;
    tail shapes, through every blockscale and MXFP8 kernel."""
    rng = np.random.Generator(np.random.PCG64(M * 7 + N + K))
    A = _finite_codes(rng, (M, K))
    B = _finite_codes(rng, (N, K))
    sa = (rng.uniform(0.5, 1.0, size=(M, K // 128)) * 2.0 ** -9).astype(np.float32)
    sb = (rng.uniform(0.5, 1.0, size=((N + 127) // 128, K // 128)) * 2.0 ** -9).astype(np.float32)
    want = oracle.blockscale(A, sa, B, sb)
    assert np.abs(oracle.bf16_bits_to_float(want)).max() > 1.0   # O(1) outputs, not all below the tolerance
    raster = 1 if M >= N else 0
    for cfg in (0, 1256401, 1128601, 1256402, 1256301, 3256401, 3256402):
        if cfg:
            override(cfg + raster * 10)
        compare(run_blockscale(A, sa, B, sb), want, f"bs codes cfg {cfg} {M}x{N}x{K}")
    override(0)
    ea = rng.integers(117, 120, size=(M, K // 32)).astype(np.uint8)   # 2^-10 .. 2^-8
    eb = rng.integers(117, 120, size=(N, K // 32)).astype(np.uint8)
    want_mx = oracle.mxfp8(A, ea, B, eb)
    for cfg in (0, 2256401, 2128601, 2256402, 5256601):
        if cfg:
            override(cfg + raster * 10)
        compare(run_mxfp8(A, ea, B, eb), want_mx, f"mx codes cfg {cfg} {M}x{N}x{K}")
    override(0)


# ------------------------------------------------ size limits
def test_maximum_k_every_entry_point():
    """K at its limit (2^20, 8192 K blocks of one tile): blockscale (stream-K cuts
    the single tile between many CTAs), MXFP8, the twin and the E4M3 output."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 2, 16, 1 << 20
    x = workloads.make_blockscale_inputs(M, N, K, seed=71)
    compare(run_blockscale(x.A, x.a_scale, x.B, x.b_scale), oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale),
            "bs K=2^20")
    codes, yv = oracle.blockscale_e4m3out(x.A, x.a_scale, x.B, x.b_scale, 4.0)
    compare_e4m3(_run_e4m3out(x, 4.0), codes, yv, 4.0, "bs e4m3 K=2^20")
    y = workloads.make_mxfp8_inputs(M, N, K, seed=72)
    compare(run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), "mx K=2^20")
    t = workloads.make_tensorscale_inputs(M, N, K, seed=73)
    got = f.gemm_tensorscale(to_dev(t.A), to_dev(t.B), float(t.alpha))
    assert f.get_status() == 0
    compare(got.view(torch.int16).cpu().numpy().view(np.uint16), oracle.tensorscale(t.A, t.B, float(t.alpha)),
            "twin K=2^20")


def test_tall_m_sampled_rows():
    """M = 2^17 rows (a_scale row stride, tile and row indices far from small
    values): sampled rows of blockscale and MXFP8 against the oracle."""
    M, N, K = 1 << 17, 16, 128
    rng = np.random.Generator(np.random.PCG64(74))
    rows = np.sort(rng.choice(M, 64, replace=False))
    rows[-1] = M - 1
    x = workloads.make_blockscale_inputs(M, N, K, seed=75)
    got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
    compare(got[rows], oracle.blockscale(x.A[rows], x.a_scale[rows], x.B, x.b_scale), "bs M=2^17")
    y = workloads.make_mxfp8_inputs(M, N, K, seed=76)
    got = run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
    compare(got[rows], oracle.mxfp8(y.A[rows], y.a_e8m0[rows], y.B, y.b_e8m0), "mx M=2^17")


@pytest.mark.parametrize("M,N,K", [(4096, 1280, 1280), (4100, 776, 384), (257, 264, 3840), (1, 16, 128)])
def test_mxfp8_pair_kernel(override, M, N, K):
    """The CTA-pair MXFP8 kernel (256 x 256 tiles over two SMs): M and N tails,
    an odd number of 128-row B blocks, a single row; and the E4M3 output, which
    runs through the one-CTA kernel when the pair is forced."""
    import fp8_block_scaled_e4m3_gb300 as f
    cid = 5256601 + (10 if M >= N else 0)
    override(cid)
    y = workloads.make_mxfp8_inputs(M, N, K, seed=M + 3 * N + K)
    got = run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0)
    assert f.last_config_id() == cid
    compare(got, oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), f"mx pair {M}x{N}x{K}")
    if N % 16 == 0:
        s = 16.0
        c8 = f.gemm_mxfp8_e4m3out(to_dev(y.A), to_dev(y.a_e8m0), to_dev(y.B), to_dev(y.b_e8m0), s).cpu().numpy()
        assert f.get_status() == 0
        assert f.decode_config(f.last_config_id())["kind"] == "mxfp8"
        codes, yv = oracle.mxfp8_e4m3out(y.A, y.a_e8m0, y.B, y.b_e8m0, s)
        compare_e4m3(c8, codes, yv, s, f"mx pair e4m3 fallback {M}x{N}x{K}")


def test_mxfp8_pair_graph_replay_and_repeat(override):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(5256611)
    M, N, K = 1024, 512, 1280
    x0, x1 = (workloads.make_mxfp8_inputs(M, N, K, seed=s) for s in (81, 82))
    d = [to_dev(x0.A), to_dev(x0.a_e8m0), to_dev(x0.B), to_dev(x0.b_e8m0)]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    f.gemm_mxfp8(*d, C=C)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f.gemm_mxfp8(*d, C=C)
    for x in (x1, x0, x1):
        for dst, src in zip(d, (x.A, x.a_e8m0, x.B, x.b_e8m0)):
            dst.copy_(to_dev(src))
        g.replay()
        assert f.get_status() == 0
        compare(C.view(torch.int16).cpu().numpy().view(np.uint16), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0),
                "mx pair graph replay")
    del g


# ------------------------------------------------ MXFP8 decode kernel (selectable)
# (M, N, K, slices on 152 SMs): one slice (K = 128; or 512 tiles, several
# waves); 2..8 slices in a cluster; ragged N; M of one to four 32-row groups.
DECODE_CASES = [(1, 5120, 2048, 3), (32, 5120, 2048, 3), (33, 8192, 1280, 2), (128, 1536, 2048, 8),
                (5, 1000, 896, 7), (3, 136, 128, 1), (9, 1024, 6144, 8), (100, 2048, 768, 6),
                (20, 3840, 2048, 5), (64, 65536, 256, 1)]


@pytest.mark.parametrize("M,N,K,slices", DECODE_CASES)
def test_mxfp8_decode_kernel(override, M, N, K, slices):
    """The decode kernel (K slices of one 128-column tile in a thread-block
    cluster, partials added in distributed shared memory): oracle parity and
    the same bits on a repeat call, at every slice count it takes."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(6128601)
    y = workloads.make_mxfp8_inputs(M, N, K, seed=M + N + K)
    d = (to_dev(y.A), to_dev(y.a_e8m0), to_dev(y.B), to_dev(y.b_e8m0))
    c1 = f.gemm_mxfp8(*d)
    assert f.get_status() == 0
    assert f.last_config_id() == 6128601
    c2 = f.gemm_mxfp8(*d)
    assert f.get_status() == 0
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    compare(c1.view(torch.int16).cpu().numpy().view(np.uint16), oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0),
            f"mx decode {M}x{N}x{K} ({slices} slices)")


def test_mxfp8_decode_kernel_falls_back(override):
    """Shapes and outputs the decode kernel does not take run the one-CTA
    128-wide kernel: more than one row of tiles, a K needing more than 8
    slices, an E4M3 C."""
    import fp8_block_scaled_e4m3_gb300 as f
    override(6128601)
    for M, N, K in [(129, 256, 512), (17, 512, 7168)]:
        y = workloads.make_mxfp8_inputs(M, N, K, seed=7)
        compare(run_mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0), oracle.mxfp8(y.A, y.a_e8m0, y.B, y.b_e8m0),
                f"mx decode fallback {M}x{N}x{K}")
        assert f.last_config_id() == 2128601
    y = workloads.make_mxfp8_inputs(16, 1024, 2048, seed=8)
    c8 = f.gemm_mxfp8_e4m3out(to_dev(y.A), to_dev(y.a_e8m0), to_dev(y.B), to_dev(y.b_e8m0), 16.0).cpu().numpy()
    assert f.get_status() == 0
    assert f.last_config_id() == 2128601
    codes, yv = oracle.mxfp8_e4m3out(y.A, y.a_e8m0, y.B, y.b_e8m0, 16.0)
    compare_e4m3(c8, codes, yv, 16.0, "mx decode e4m3 fallback")


def test_mxfp8_decode_kernel_graph_replay(override):
    """Captured once, replayed on new contents: the cluster hand-off holds no
    state between launches."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    override(6128601)
    M, N, K = 16, 2048, 2048
    x0, x1 = (workloads.make_mxfp8_inputs(M, N, K, seed=s) for s in (91, 92))
    d = [to_dev(x0.A), to_dev(x0.a_e8m0), to_dev(x0.B), to_dev(x0.b_e8m0)]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    f.gemm_mxfp8(*d, C=C)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f.gemm_mxfp8(*d, C=C)
    for x in (x1, x0, x1):
        for dst, src in zip(d, (x.A, x.a_e8m0, x.B, x.b_e8m0)):
            dst.copy_(to_dev(src))
        g.replay()
        assert f.get_status() == 0
        compare(C.view(torch.int16).cpu().numpy().view(np.uint16), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0),
                "mx decode graph replay")
    del g
