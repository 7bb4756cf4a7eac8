"""fp8mx_gemm_noalloc: the MXFP8 GEMM for callers that must not allocate.

Some callers cannot let a library allocate device memory while they call it:
engines that reserve all device memory up front and manage it themselves,
plugins that run inside a host framework which gives them no allocator, and
latency-critical paths that forbid allocator calls. fp8mx_gemm takes its
packed-scale workspace from a memory pool; fp8mx_gemm_noalloc uses a fixed
8 MiB device array built into the library instead. These tests call it through
the C ABI (ctypes, raw pointers) and compare it with fp8mx_gemm.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_util import compare, to_dev


def _lib():
    import fp8_block_scaled_e4m3_gb300 as f
    return f, f.lib()


def _call(L, fn, A, ea, B, eb, C, M, N, K):
    import torch
    return fn(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(ea.data_ptr()), ctypes.c_void_p(B.data_ptr()),
              ctypes.c_void_p(eb.data_ptr()), ctypes.c_void_p(C.data_ptr()), M, N, K,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


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
def test_noalloc_matches_fp8mx_gemm_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f, L = _lib()
    # a larger call, then a smaller one that reuses (and must not depend on) the
    # array's leftover contents
    for (M, N, K, seed) in [(1000, 640, 1280, 11), (129, 264, 2048, 12)]:
        x = workloads.make_mxfp8_inputs(M, N, K, seed=seed)
        A, ea, B, eb = to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0)
        C_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        C_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(L, L.fp8mx_gemm, A, ea, B, eb, C_ref, M, N, K) == 0
        assert _call(L, L.fp8mx_gemm_noalloc, A, ea, B, eb, C_new, M, N, K) == 0
        assert f.get_status() == 0
        ref = C_ref.view(torch.int16).cpu().numpy().view(np.uint16)
        got = C_new.view(torch.int16).cpu().numpy().view(np.uint16)
        compare(got, ref, f"noalloc vs fp8mx_gemm {M}x{N}x{K}")


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
    compare(C.view(torch.int16).cpu().numpy().view(np.uint16), oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0),
            "noalloc decode kernel")
