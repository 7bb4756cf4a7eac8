"""C-ABI library: loads, exports every declared symbol, host-side checks and
layout helpers (CPU only; no call here reaches a CUDA launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import fp8_block_scaled_e4m3_gb300 as f
    return f


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8(?:bs|mx)_\w+)\s*\(", txt)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "fp8bs_gemm" in names and "fp8mx_gemm" in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIBRARY_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_shape_rules_rejected_before_launch(lib):
    L = lib.lib()
    P = ctypes.c_void_p(16)   # never dereferenced: shape checks come first
    for f in (L.fp8bs_gemm, L.fp8mx_gemm):
        assert f(P, P, P, P, P, 4, 8, 100, None) == -3        # K % 128
        assert f(P, P, P, P, P, 4, 8, 0, None) == -3          # K < 128
        assert f(P, P, P, P, P, 4, 12, 128, None) == -3       # N % 8
        assert f(P, P, P, P, P, 4, 0, 128, None) == -3        # N < 8
        assert f(P, P, P, P, P, -1, 8, 128, None) == -3       # M < 0
        assert f(P, P, P, P, P, 4, 8, (1 << 20) + 128, None) == -3
        assert f(None, None, None, None, None, 0, 8, 128, None) == 0   # M == 0 is a no-op
        assert f(None, P, P, P, P, 4, 8, 128, None) == -1
        assert f(P, P, P, P, None, 4, 8, 128, None) == -1


def test_tensorscale_entry_checks_before_launch(lib):
    L = lib.lib()
    f = L.fp8bs_gemm_tensorscale
    P = ctypes.c_void_p(1 << 20)
    one = ctypes.c_float(1.0)
    assert f(P, P, P, 4, 8, 100, one, None) == -3         # K % 128
    assert f(P, P, P, 4, 12, 128, one, None) == -3        # N % 8
    assert f(P, P, P, -1, 8, 128, one, None) == -3        # M < 0
    assert f(None, None, None, 0, 8, 128, one, None) == 0  # M == 0 is a no-op
    assert f(None, P, P, 4, 8, 128, one, None) == -1
    assert f(ctypes.c_void_p((1 << 20) + 8), P, P, 4, 8, 128, one, None) == -2
    assert f(P, P, ctypes.c_void_p((1 << 20) + 8), 4, 8, 128, one, None) == -2
    for cid in (4256411, 4128611, 4256401, 4128601, 4256412):
        assert L.fp8bs_set_config_override(cid) == 0
        assert lib.decode_config(cid)["kind"] == "tensorscale"
    assert L.fp8bs_set_config_override(4128612) == -3     # stream-K with the 256-wide tile only
    assert L.fp8bs_set_config_override(0) == 0


def test_e4m3out_entry_checks_before_launch(lib):
    L = lib.lib()
    f = L.fp8bs_gemm_e4m3out
    P = ctypes.c_void_p(1 << 20)
    one = ctypes.c_float(1.0)
    assert f(P, P, P, P, P, one, 4, 24, 128, None) == -3        # N % 16 (E4M3 rows of whole 16-byte units)
    assert f(P, P, P, P, P, one, 4, 32, 100, None) == -3        # K % 128
    assert f(None, None, None, None, None, one, 0, 32, 128, None) == 0
    assert f(None, P, P, P, P, one, 4, 32, 128, None) == -1
    assert f(P, P, P, P, ctypes.c_void_p((1 << 20) + 8), one, 4, 32, 128, None) == -2
    g = L.fp8mx_gemm_e4m3out
    assert g(P, P, P, P, P, one, 4, 24, 128, None) == -3        # N % 16
    assert g(None, None, None, None, None, one, 0, 32, 128, None) == 0
    assert g(None, P, P, P, P, one, 4, 32, 128, None) == -1


def test_alignment_rejected_before_launch(lib):
    L = lib.lib()
    a16 = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    odd4 = ctypes.c_void_p((1 << 20) + 2)
    assert L.fp8bs_gemm(odd, a16, a16, a16, a16, 4, 8, 128, None) == -2
    assert L.fp8bs_gemm(a16, odd, a16, a16, a16, 4, 8, 128, None) == -2
    assert L.fp8bs_gemm(a16, a16, a16, odd4, a16, 4, 8, 128, None) == -2
    assert L.fp8bs_gemm(a16, a16, a16, a16, odd, 4, 8, 128, None) == -2
    assert L.fp8mx_gemm(a16, odd4, a16, a16, a16, 4, 8, 128, None) == -2
    assert L.fp8mx_gemm(a16, a16, odd, a16, a16, 4, 8, 128, None) == -2


def test_layout_helpers_bit_exact(lib):
    L = lib.lib()
    for M in list(range(1, 131)):
        ld = (M + 3) // 4 * 4
        assert L.fp8bs_a_scale_ld(M) == ld
        for K in (128, 256, 768):
            KB = K // 128
            for kb in range(KB):
                for m in (0, M // 2, M - 1):
                    assert L.fp8bs_a_scale_index(m, kb, M) == kb * ld + m
    for K in (128, 256, 768, 7168):
        KB = K // 128
        for n in range(0, 300, 7):
            for kb in range(KB):
                assert L.fp8bs_b_scale_index(n, kb, K) == (n // 128) * KB + kb
                for g in range(4 * kb, 4 * kb + 4):
                    assert L.fp8mx_scale_index(n, g, K) == n * (K // 32) + g


def test_sf_atom_layout_is_a_bijection(lib):
    L = lib.lib()
    seen = set()
    for r in range(128):
        for j in range(4):
            off = L.fp8mx_sf_atom_offset(r, j)
            assert off == (r % 32) * 16 + (r // 32) * 4 + j
            seen.add(off)
    assert seen == set(range(512))


def test_config_selection(lib):
    # wide tiles for the large shapes, the narrow tile when a wide grid would starve the SMs
    # blockscale: wide one-CTA tiles for the large shape classes, the narrow tile
    # when a wide grid would starve the SMs
    # one CTA per tile from M = 2048: the CTA-pair kernel (256 x 256 tiles, four
    # stages, whole-tile C buffer), K-light shapes included
    for M, N, K in [(4096, 2048, 7168), (2048, 2048, 7168), (4096, 65536, 1536), (8192, 8192, 3072),
                    (16384, 7168, 2048), (16384, 7168, 768), (16384, 7168, 1152), (4096, 4096, 512)]:
        c = lib.decode_config(lib.select_config("bs", M, N, K, 152))
        assert c["kind"] == "blockscale_pair" and c["block_n"] == 256 and c["stages"] == 4, (M, N, K, c)
    # stream-K shapes keep the one-CTA kernel
    for M, N, K in [(16384, 1536, 7168), (1024, 2048, 7168)]:
        c = lib.decode_config(lib.select_config("bs", M, N, K, 152))
        assert c["kind"] == "blockscale" and c["stages"] == 4 and c["schedule"] == "stream_k", (M, N, K, c)
    # below M = 2048 with few K blocks per tile (K <= 1024): the one-CTA three-stage instance
    for M, N, K in [(1024, 7168, 768), (1024, 4096, 512)]:
        c = lib.decode_config(lib.select_config("bs", M, N, K, 152))
        assert c["kind"] == "blockscale" and c["block_n"] == 256 and c["stages"] == 3, (M, N, K, c)
    assert lib.decode_config(lib.select_config("mx", 16384, 7168, 768, 152))["stages"] != 3
    assert lib.decode_config(lib.select_config("bs", 256, 512, 512, 152))["block_n"] == 128
    # mxfp8: wide tiles, the narrow tile when the wide grid would starve the SMs
    assert lib.decode_config(lib.select_config("mx", 16384, 5120, 2048, 152))["block_n"] == 256
    assert lib.decode_config(lib.select_config("mx", 256, 512, 512, 152))["block_n"] == 128
    assert lib.decode_config(lib.select_config("mx", 16384, 5120, 2048, 152))["kind"] == "mxfp8_pair"
    assert lib.decode_config(lib.select_config("mx", 2048, 8192, 1280, 152))["kind"] == "mxfp8"
    assert lib.select_config("mx", 16384, 8192, 1280, 152) == 5256611
    assert lib.lib().fp8bs_set_config_override(5256612) == -3   # no stream-K for the MXFP8 pair
    assert lib.lib().fp8bs_set_config_override(5128611) == -3
    # raster streams the larger operand
    assert lib.decode_config(lib.select_config("bs", 4096, 65536, 1536, 152))["raster"] == 0
    assert lib.decode_config(lib.select_config("bs", 16384, 1536, 7168, 152))["raster"] == 1
    assert lib.select_config("bs", 4, 12, 128, 152) == -3
    L = lib.lib()
    assert L.fp8bs_set_config_override(1999911) == -3      # no such kernel
    assert L.fp8bs_set_config_override(1160511) == -3      # the 160-wide tile was removed
    assert L.fp8bs_set_config_override(2128612) == 0       # the MXFP8 kernel's 128-wide tile has stream-K too
    assert L.fp8bs_set_config_override(4128612) == -3
    assert L.fp8bs_set_config_override(3256411) == 0       # the blockscale CTA-pair kernel: 256 x 256, four stages
    assert lib.decode_config(3256411)["kind"] == "blockscale_pair"
    assert L.fp8bs_set_config_override(3256412) == 0       # ... with the stream-K schedule
    assert lib.decode_config(3256412)["schedule"] == "stream_k"
    for bad in (3128811, 3256611, 3256311, 3256413):       # no other tile, stage count or schedule
        assert L.fp8bs_set_config_override(bad) == -3
    assert L.fp8bs_set_config_override(1256413) == -3      # no such schedule
    assert L.fp8bs_set_config_override(1128612) == -3      # stream-K runs with the 256-wide tile only
    # the MXFP8 decode kernel (K slices in clusters): selectable, one id only, never chosen by the rule
    assert L.fp8bs_set_config_override(6128601) == 0
    assert lib.decode_config(6128601)["kind"] == "mxfp8_decode"
    for bad in (6256601, 6128401, 6128602, 6128611):
        assert L.fp8bs_set_config_override(bad) == -3
    assert L.fp8bs_set_config_override(0) == 0
    assert L.fp8bs_set_raster_group(-1) == -3 and L.fp8bs_set_raster_group(4097) == -3
    assert L.fp8bs_set_raster_group(8) == 0 and L.fp8bs_set_raster_group(0) == 0
    for M, N, K in [(1, 5120, 2048), (32, 8192, 1280), (128, 5120, 2048)]:
        assert lib.decode_config(lib.select_config("mx", M, N, K, 152))["kind"] == "mxfp8"


def test_schedule_selection(lib):
    # Stream-K exactly when it shortens the longest CTA's K loop by >= 20 K
    # blocks (blockscale) or >= 13 K steps (MXFP8).
    sched = lambda M, N, K, sms=152: lib.decode_config(lib.select_config("bs", M, N, K, sms))["schedule"]
    assert sched(16384, 1536, 7168) == "stream_k"     # 768 tiles x 56: 336 -> 283 K blocks
    assert sched(8192, 2048, 7168) == "stream_k"      # 512 tiles x 56: 224 -> 189
    assert sched(256, 512, 7168) == "stream_k"        # 8 tiles x 56: 56 -> 3
    assert sched(4096, 2048, 7168) == "tile"          # 256 tiles x 56: 112 -> 95
    assert sched(2048, 2048, 7168) == "tile"          # 128 tiles x 56: 56 -> 48
    assert sched(16384, 7168, 768) == "tile"          # 3584 tiles x 6: 144 -> 142
    assert sched(4096, 65536, 1536) == "tile"         # 8192 tiles x 12: 648 -> 647
    assert sched(16384, 1536, 7168, sms=128) == "tile"  # 768 tiles = 6 full waves
    assert sched(4096, 2048, 128) == "tile"           # one K block: nothing to share
    assert sched(256, 512, 512) == "tile"             # 8 tiles x 4: 4 -> 1, not worth a hand-off
    assert sched(16, 2048, 7168) == "stream_k"        # decode: 8 tiles x 56, pieces of >= 7
    assert sched(128, 2048, 7168) == "tile"           # one row of tiles, four live row groups
    assert lib.decode_config(lib.select_config("bs", 128, 2048, 7168, 152))["block_n"] == 128
    mx = lambda M, N, K, sms=152: lib.decode_config(lib.select_config("mx", M, N, K, sms))["schedule"]
    assert mx(1024, 5120, 2048) == "stream_k"         # 160 tiles x 16: 32 -> 17
    assert mx(2048, 5120, 2048) == "stream_k"         # 320 tiles x 16: 48 -> 34
    assert mx(4096, 5120, 2048) == "tile"             # 640 tiles x 16: 80 -> 68
    assert mx(2048, 8192, 1280) == "tile"             # 512 tiles x 10: 40 -> 34
    assert mx(32, 5120, 2048) == "tile"               # 20 tiles x 16: 16 -> 8
    assert mx(16384, 5120, 2048) == "tile"            # 2560 tiles x 16: 272 -> 270
    assert mx(256, 512, 512) == "tile"


def test_shutdown_without_setup_is_a_noop(lib):
    assert lib.lib().fp8bs_shutdown() == 0
    lib.shutdown()


def test_status_strings(lib):
    L = lib.lib()
    for code in range(-7, 1):
        assert L.fp8bs_status_string(code)
    assert L.fp8bs_launches_per_call() == 1
