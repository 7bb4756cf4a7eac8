"""Helpers for the GPU tests: run the library on numpy inputs, compare to the oracle."""
import numpy as np

import oracle
import workloads

# Tolerance of the comparison: elementwise |gpu - oracle| <= ATOL + RTOL*|oracle|
# and ||gpu - oracle||_2 / ||oracle||_2 <= REL_L2 (the oracle's bf16 is the reference).
ATOL = 1e-2
RTOL = 1e-2
REL_L2 = 2e-3


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_blockscale(A, a_scale, B, b_scale, C=None):
    """GPU blockscale GEMM on numpy inputs (a_scale logical [M, K/128]); returns bf16 bits (uint16 numpy)."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    M, K = A.shape
    N = B.shape[0]
    dA = to_dev(A)
    dB = to_dev(B)
    dsa = to_dev(workloads.a_scale_to_kmajor(a_scale))
    dsb = to_dev(np.ascontiguousarray(b_scale, dtype=np.float32))
    out = f.gemm_blockscale(dA, dsa, dB, dsb, C=C)
    assert f.get_status() == 0
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def run_mxfp8(A, a_e8m0, B, b_e8m0, C=None):
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    out = f.gemm_mxfp8(to_dev(A), to_dev(a_e8m0), to_dev(B), to_dev(b_e8m0), C=C)
    assert f.get_status() == 0
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def compare(gpu_bits, ref_bits, what=""):
    """Apply the tolerance; return a dict of metrics (raises AssertionError on failure)."""
    g = oracle.bf16_bits_to_float(gpu_bits).astype(np.float64)
    o = oracle.bf16_bits_to_float(ref_bits).astype(np.float64)
    assert g.shape == o.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - o)
    bad = err > ATOL + RTOL * np.abs(o)
    nrm = np.linalg.norm(o)
    rel = float(np.linalg.norm(g - o) / nrm) if nrm > 0 else float(np.linalg.norm(g - o))
    cos = float(np.dot(g.ravel(), o.ravel()) / (np.linalg.norm(g) * nrm)) if nrm > 0 else 1.0
    m = {"maxabs": float(err.max()) if err.size else 0.0, "rel_l2": rel, "cos": cos,
         "n_out_of_tol": int(bad.sum()), "n": int(g.size)}
    if bad.any():
        idx = np.argwhere(bad)
        rows = np.unique(idx[:, 0] % 128)
        cols = np.unique(idx[:, 1] % 256)
        raise AssertionError(f"{what}: {m}; first bad {idx[:5].tolist()}, rows%128 {rows[:16].tolist()}, "
                             f"cols%256 {cols[:16].tolist()}")
    assert rel <= REL_L2, f"{what}: {m}"
    return m


def compare_rows(gpu_bits, ref_bits, what="", rows_per_chunk=512):
    """compare() over a large output in row chunks (the metrics are accumulated
    over the whole matrix; nothing of size M x N is held in float64)."""
    assert gpu_bits.shape == ref_bits.shape
    M = gpu_bits.shape[0]
    sq_err = sq_ref = sq_gpu = dot = 0.0
    maxabs = 0.0
    n_bad = 0
    first_bad = []
    for r0 in range(0, M, rows_per_chunk):
        g = oracle.bf16_bits_to_float(gpu_bits[r0:r0 + rows_per_chunk]).astype(np.float64)
        o = oracle.bf16_bits_to_float(ref_bits[r0:r0 + rows_per_chunk]).astype(np.float64)
        assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output in rows {r0}.."
        err = np.abs(g - o)
        bad = err > ATOL + RTOL * np.abs(o)
        if bad.any():
            n_bad += int(bad.sum())
            if len(first_bad) < 5:
                first_bad += (np.argwhere(bad)[:5] + [r0, 0]).tolist()
        maxabs = max(maxabs, float(err.max()) if err.size else 0.0)
        sq_err += float(np.sum(err * err))
        sq_ref += float(np.sum(o * o))
        sq_gpu += float(np.sum(g * g))
        dot += float(np.sum(g * o))
    rel = (sq_err / sq_ref) ** 0.5 if sq_ref > 0 else sq_err ** 0.5
    cos = dot / (sq_gpu * sq_ref) ** 0.5 if sq_ref > 0 and sq_gpu > 0 else 1.0
    m = {"maxabs": maxabs, "rel_l2": rel, "cos": cos, "n_out_of_tol": n_bad, "n": int(gpu_bits.size)}
    assert n_bad == 0, f"{what}: {m}; first bad {first_bad[:5]}"
    assert rel <= REL_L2, f"{what}: {m}"
    return m


def _e4m3_table():
    """Values of the 256 E4M3FN codes (NaN for 0x7F/0xFF), from the oracle's decoder."""
    return np.array([oracle.e4m3_decode(c) for c in range(256)], dtype=np.float64)


def compare_e4m3(gpu_codes, ref_codes, y, c_scale, what="", max_frac=1e-3):
    """E4M3 outputs: codes must be equal, except where the oracle's pre-rounding
    value y lies so close to the midpoint of two neighbouring E4M3 values that
    the kernel's own fp32 sum (another summation order) may fall on the other
    side; there either neighbour is correct. Returns the number of such cases."""
    t = _e4m3_table()
    g = gpu_codes.astype(np.int64)
    o = ref_codes.astype(np.int64)
    diff = g != o
    if not diff.any():
        return 0
    gv, ov, yy = t[g[diff]], t[o[diff]], y[diff].astype(np.float64)
    same_sign = np.sign(gv) * np.sign(ov) >= 0
    # neighbours: no E4M3 value strictly between the two
    lo, hi = np.minimum(np.abs(gv), np.abs(ov)), np.maximum(np.abs(gv), np.abs(ov))
    pos = np.sort(t[1:127])
    between = np.searchsorted(pos, hi, side="left") - np.searchsorted(pos, lo, side="right")
    adjacent = same_sign & (between == 0) & np.isfinite(gv) & np.isfinite(ov)
    mid = (gv + ov) / 2
    near = np.abs(yy - mid) <= 1e-4 * np.abs(mid) + 1e-3 * float(c_scale)
    ok = adjacent & near
    n = int(diff.sum())
    assert ok.all(), (f"{what}: {int((~ok).sum())} of {n} differing codes are not a tie within accumulation "
                      f"noise; first {np.argwhere(diff)[~ok][:5].tolist()}")
    assert n <= max_frac * g.size + 1, f"{what}: {n} near-tie differences of {g.size}"
    return n
