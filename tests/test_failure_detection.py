"""Device-side wait limits: a wait that runs out is reported, not trapped (GPU).

The limit is set so short that the first pipeline wait which has to wait at
all runs out; the kernel must record FP8BS_ERR_DEVICE_TIMEOUT in the status
word, finish the work it already issued, free its tensor memory and return,
and the CUDA context must stay usable: the next call with the normal limit is
correct.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import compare, run_blockscale, run_mxfp8, to_dev

pytestmark = pytest.mark.gpu

TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _call(kind, x):
    """A callable that launches the path under test once on the inputs x and
    returns its output tensor."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    if kind in ("bs", "bs_sk", "bs_pair", "bs_pair_sk", "e4m3"):
        d = (to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.B), to_dev(x.b_scale))
        if kind == "e4m3":
            return lambda: f.gemm_blockscale_e4m3out(*d, 8.0)
        return lambda: f.gemm_blockscale(*d)
    if kind in ("mx", "mx_sk", "mx_pair", "mx_decode"):
        return lambda: f.gemm_mxfp8(to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0))
    if kind == "twin":
        return lambda: f.gemm_tensorscale(to_dev(x.A), to_dev(x.B), 1e-3)
    A, sa = to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale))
    B, sb, be = to_dev(x.B), to_dev(x.b_scale), to_dev(x.block_expert)

    def moe():
        lead, n = f.moe_leaders(be, x.num_experts)
        return f.gemm_moe(A, sa, B, sb, be, lead, n)
    return moe


OVERRIDE = {"bs_sk": 1256402, "bs_pair": 3256401, "bs_pair_sk": 3256402, "mx_sk": 2256402, "mx_pair": 5256601, "mx_decode": 6128601}


@pytest.mark.parametrize("kind", ["bs", "bs_sk", "bs_pair", "bs_pair_sk", "e4m3", "mx", "mx_sk", "mx_pair", "mx_decode", "twin", "moe"])
def test_every_path_reports_a_timeout_and_recovers(kind):
    """Stream-K included: a CTA that gives up never publishes its partial, and
    the finishers waiting for it run out of time as well instead of hanging.
    In the CTA-pair kernels a CTA whose partner gave up runs out of time on the
    partner's barriers, and the blockscale pair's store warp on the tile buffer.
    In the decode kernel's clusters every CTA still reaches both cluster
    barriers, and a partial marked invalid is never stored."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    if kind == "moe":
        x = workloads.make_moe_inputs(512, 2, 8, 256, 1024, seed=5, skew=1.0)
    elif kind == "mx_decode":   # one row of tiles, 8 K slices per cluster
        x = workloads.make_inputs("mx", 32, 1024, 2048, seed=4)
    else:
        x = workloads.make_inputs("mx" if kind.startswith("mx") else "bs", 256, 1024, 4096, seed=4)
    f.set_config_override(OVERRIDE.get(kind, 0))
    try:
        run = _call(kind, x)
        f.set_wait_limit_ns(200)
        try:
            run()
            assert f.get_status() == TIMEOUT
        finally:
            f.set_wait_limit_ns(0)
        assert f.get_status() == 0
        first = run()
        assert f.get_status() == 0
        second = run()            # a clean call after the recovered one: same bits (fresh stream-K tokens)
        assert f.get_status() == 0
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.uint8), second.view(torch.uint8))
    finally:
        f.set_config_override(0)


@pytest.mark.parametrize("kind", ["bs", "mx"])
def test_wait_timeout_reported_and_context_survives(kind):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    M, N, K = 512, 1024, 2048
    x = workloads.make_inputs(kind, M, N, K, seed=3)
    f.set_wait_limit_ns(200)          # 200 ns: any wait that is not already satisfied runs out
    try:
        if kind == "bs":
            f.gemm_blockscale(to_dev(x.A), to_dev(workloads.a_scale_to_kmajor(x.a_scale)), to_dev(x.B),
                              to_dev(x.b_scale))
        else:
            f.gemm_mxfp8(to_dev(x.A), to_dev(x.a_e8m0), to_dev(x.B), to_dev(x.b_e8m0))
        assert f.get_status() == TIMEOUT
    finally:
        f.set_wait_limit_ns(0)
    assert f.get_status() == 0        # read-and-clear
    # the context is intact: the same call with the normal limit is correct
    if kind == "bs":
        got = run_blockscale(x.A, x.a_scale, x.B, x.b_scale)
        compare(got, oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale), "bs after timeout")
    else:
        got = run_mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0)
        compare(got, oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0), "mx after timeout")
    torch.cuda.synchronize()
