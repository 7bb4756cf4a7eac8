"""The seeded input generators follow their stated recipe (CPU only)."""
import numpy as np

import workloads as w


def _all_values():
    return w._E4M3_POS


def test_e4m3_rne_is_nearest_ties_to_even():
    rng = np.random.Generator(np.random.PCG64(0))
    vals = _all_values()
    mids = (vals[:-1] + vals[1:]) / 2                        # exact ties (all representable in fp32)
    y = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 0.01,
                        mids, -mids, vals, -vals, [0.0, -0.0, 448.0, -448.0]]).astype(np.float32)
    codes = w.e4m3_rne(y)
    got = np.where(codes & 0x80, -1.0, 1.0) * vals[codes & 0x7F]
    yd = y.astype(np.float64)
    dist = np.abs(np.abs(yd)[:, None] - vals[None, :])
    best = dist.min(axis=1)
    assert np.all(np.abs(np.abs(got) - np.abs(yd)) == best)
    tie = (dist == best[:, None]).sum(axis=1) == 2
    assert np.all((codes[tie] & 1) == 0)
    assert np.all((codes[yd < 0] & 0x80) == 0x80)


def test_ue8m0_exponent_is_exact_ceil_log2():
    rng = np.random.Generator(np.random.PCG64(1))
    amax = np.concatenate([np.abs(rng.standard_normal(10000)) * 4,
                           448.0 * np.exp2(np.arange(-20, 20)).astype(np.float32)]).astype(np.float32)
    e = w.ue8m0_from_amax(amax).astype(np.int64) - 127
    q = (amax / np.float32(448)).astype(np.float64)
    assert np.all(np.exp2(e.astype(np.float64)) >= q)
    assert np.all(np.exp2(e.astype(np.float64) - 1) < q)
    assert w.ue8m0_from_amax(np.zeros(1, np.float32))[0] == 127


def test_blockscale_quantiser_recipe():
    x = w.make_blockscale_inputs(130, 200, 384, seed=1)
    assert x.a_scale.shape == (130, 3) and x.b_scale.shape == (2, 3)
    # every block reaches the saturation code 448 (scale = amax/448 within fp32 rounding)
    blk = (x.A.reshape(130, 3, 128) & 0x7F).max(axis=2)
    assert np.all(blk >= 0x7D)
    assert np.all(x.A & 0x7F != 0x7F)


def test_mx_quantiser_recipe():
    x = w.make_mxfp8_inputs(64, 96, 256, seed=2)
    assert x.a_e8m0.shape == (64, 8) and x.b_e8m0.shape == (96, 8)
    assert np.all(x.A & 0x7F != 0x7F)
    assert np.all((x.a_e8m0 > 100) & (x.a_e8m0 < 140))


def test_tensorscale_quantiser_recipe():
    x = w.make_tensorscale_inputs(70, 40, 256, seed=5)
    # one scale per tensor: the largest |value| of each tensor maps to the code 448
    assert (x.A & 0x7F).max() >= 0x7D and (x.B & 0x7F).max() >= 0x7D
    assert np.all(x.A & 0x7F != 0x7F) and np.all(x.B & 0x7F != 0x7F)
    rng = np.random.Generator(np.random.PCG64(5))
    a = rng.standard_normal((70, 256), dtype=np.float32)
    b = rng.standard_normal((40, 256), dtype=np.float32) * np.float32(0.02)
    sa, sb = np.abs(a).max() / np.float32(448), np.abs(b).max() / np.float32(448)
    assert x.alpha == np.float32(np.float32(sa) * np.float32(sb))


def test_generators_are_deterministic():
    a = w.make_blockscale_inputs(64, 128, 256, seed=3)
    b = w.make_blockscale_inputs(64, 128, 256, seed=3)
    assert a.digest() == b.digest()
    c = w.make_blockscale_inputs(64, 128, 256, seed=4)
    assert a.digest() != c.digest()


def test_a_scale_kmajor_layout():
    sa = np.arange(7 * 3, dtype=np.float32).reshape(7, 3)
    km = w.a_scale_to_kmajor(sa)
    assert km.shape == (3, 8)
    for m in range(7):
        for kb in range(3):
            assert km[kb, m] == sa[m, kb]
    assert np.all(km[:, 7] == 0)
