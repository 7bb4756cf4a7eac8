"""fp8mx_gemm_noalloc: the MXFP8 GEMM for callers that must not allocate.

Some callers cannot let a library allocate device memory while they call it:
engines that reserve all device memory up front and manage it themselves,
plugins that run inside a host framework which gives them no allocator, and
latency-critical paths that forbid allocator calls. fp8mx_gemm takes its
packed-scale workspace from a memory pool; fp8mx_gemm_noalloc uses a fixed
8 MiB device array built into the library instead. These tests call it through
the C ABI (ctypes, raw pointers) and compare it with the oracle, and bit for
bit with fp8mx_gemm wherever both calls ran the same kernel configuration.

This file is named so that pytest collects it last.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import workloads
from gpu_util import compare, to_dev

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    import fp8_block_scaled_e4m3_gb300 as f
    return f, f.lib()


def _call(L, fn, A, ea, B, eb, C, M, N, K):
    import torch
    return fn(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(ea.data_ptr()), ctypes.c_void_p(B.data_ptr()),
              ctypes.c_void_p(eb.data_ptr()), ctypes.c_void_p(C.data_ptr()), M, N, K,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _bits(C):
    import torch
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Sizes whose packed scales exceed the fixed array are refused on the host."""
    f, L = _lib()
    limit = L.fp8mx_noalloc_scratch_bytes()
    assert limit == 8 << 20
    K = 4096
    rows = (limit // ((K // 128) * 512)) * 128      # A alone fills the array; any N overflows it
    P = ctypes.c_void_p(1 << 20)
    assert L.fp8mx_gemm_noalloc(P, P, P, P, P, rows, 128, K, None) == -8
    assert L.fp8bs_status_string(-8)


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    f, L = _lib()
    # a larger call, then a smaller one that reuses (and must not depend on) the
    # array's leftover contents
    for (M, N, K, seed) in [(1000, 640, 1280, 11), (129, 264, 2048, 12)]:
        x = workloads.make_mxfp8_inputs(M, N, K, seed=seed)
        A, ea, B, eb = to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0)
        C_pool = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        C_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(L, L.fp8mx_gemm, A, ea, B, eb, C_pool, M, N, K) == 0
        cfg_pool = f.last_config_id()
        assert _call(L, L.fp8mx_gemm_noalloc, A, ea, B, eb, C_new, M, N, K) == 0
        cfg_new = f.last_config_id()
        assert f.get_status() == 0
        got = _bits(C_new)
        compare(got, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), f"noalloc vs oracle {M}x{N}x{K}")
        if cfg_new == cfg_pool:
            # same kernel and schedule on the same packed scales: the same bits
            assert np.array_equal(got, _bits(C_pool)), f"noalloc and fp8mx_gemm differ at {M}x{N}x{K}"


@pytest.mark.gpu
def test_noalloc_runs_the_pair_kernel_when_forced():
    """The CTA-pair kernel (chosen by the shape rule from M = 4096) needs no
    workspace, so a forced pair configuration runs under the allocation-free entry."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    f, L = _lib()
    M, N, K = 600, 776, 1280
    x = workloads.make_mxfp8_inputs(M, N, K, seed=14)
    A, ea, B, eb = to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.set_config_override(5256611)
    try:
        assert _call(L, L.fp8mx_gemm_noalloc, A, ea, B, eb, C, M, N, K) == 0
        assert f.get_status() == 0
        assert f.last_config_id() == 5256611
    finally:
        f.set_config_override(0)
    compare(_bits(C), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), "noalloc forced pair kernel")


_FRESH = textwrap.dedent("""
    import ctypes, sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    import workloads
    import fp8_block_scaled_e4m3_gb300 as f
    L = f.lib()
    M, N, K = 4096, 5120, 2048
    x = workloads.make_mxfp8_inputs(M, N, K, seed=21)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    A, ea, B, eb = dev(x.A), dev(x.a_e8m0), dev(x.B), dev(x.b_e8m0)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    outs, cfgs = [], []
    for rnd in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        # the first library call of the process (and, the second time, the first after shutdown)
        assert L.fp8mx_gemm_noalloc(P(A), P(ea), P(B), P(eb), P(C), M, N, K, s) == 0
        assert f.get_status() == 0
        cfgs.append(f.last_config_id())
        outs.append(C.view(torch.int16).cpu().numpy().view(np.uint16))
        assert L.fp8bs_shutdown() == 0
    np.save({out!r}, np.stack(outs))
    print(cfgs[0], cfgs[1])
""")


@pytest.mark.gpu
def test_noalloc_as_first_call_of_a_process_on_a_pair_kernel_shape(tmp_path):
    """In a fresh process whose first library call is fp8mx_gemm_noalloc (and again
    after fp8bs_shutdown), a shape for which the rule picks the CTA-pair kernel
    runs it with the allocation-free set-up alone."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    out = str(tmp_path / "noalloc_fresh.npy")
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT, out=out)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    cfg0, cfg1 = (int(v) for v in r.stdout.split())
    assert cfg0 // 1000000 == 5 and cfg1 == cfg0, (cfg0, cfg1)
    got = np.load(out)
    assert np.array_equal(got[0], got[1])
    M, N, K = 4096, 5120, 2048
    x = workloads.make_mxfp8_inputs(M, N, K, seed=21)
    compare(got[0], oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), "noalloc first call, pair kernel")


@pytest.mark.gpu
def test_noalloc_runs_the_decode_kernel_when_forced():
    """The MXFP8 decode kernel reduces its K slices in distributed shared
    memory, so it needs no workspace and runs under the allocation-free entry."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    f, L = _lib()
    M, N, K = 8, 1024, 2048
    x = workloads.make_mxfp8_inputs(M, N, K, seed=13)
    A, ea, B, eb = to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.set_config_override(6128601)
    try:
        assert _call(L, L.fp8mx_gemm_noalloc, A, ea, B, eb, C, M, N, K) == 0
        assert f.get_status() == 0
        assert f.last_config_id() == 6128601
    finally:
        f.set_config_override(0)
    compare(_bits(C), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), "noalloc decode kernel")
