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
