"""Seeded synthetic inputs for the FP8 block-scaled GEMM and its MXFP8 variant.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle. It draws Gaussian data and quantises it to OCP E4M3 codes with the
scale recipes below; it contains none of the GEMM arithmetic itself.

Recipes (the workloads the skill card "FlyDSL fp8 blockscale GEMM" measures,
section "When to use", shape table; and the PR "1x32 ue8m0 (MXFP8) 8-wave
FlyDSL GEMM for gfx950", section "Measured"):

* blockscale: A[M,K] ~ N(0,1), one fp32 scale per (row, 128-wide K block);
  B[N,K] ~ N(0,0.02), one fp32 scale per 128x128 block. scale = fp32(amax/448)
  (amax == 0 -> 1.0), code = e4m3_rne(clamp(fp32(x/scale), +-448)).
* mxfp8: A and B ~ N(0,1), one ue8m0 byte per (row, 32-wide K group):
  e = ceil(log2(fp32(amax/448))) computed exactly from the fp32 bits,
  byte = clamp(e+127, 0, 254) (amax == 0 -> 127), code = e4m3_rne(clamp(x/2^e, +-448)).

The random stream is numpy's PCG64 seeded with the integer seed; A is drawn
first ([M,K] row-major), then B ([N,K]).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

E4M3_MAX = 448.0
BLOCK_K = 128          # blockscale K block (and B's N block)
MX_GROUP = 32          # MXFP8 scale group along K

# Non-negative finite OCP E4M3FN values indexed by code 0x00..0x7E
# (bias 7; exponent field 0 is subnormal m*2^-9; 0x7F is NaN and never produced).
_codes = np.arange(0x7F, dtype=np.int64)
_exp = (_codes >> 3) & 0xF
_man = _codes & 0x7
_E4M3_POS = np.where(_exp == 0, _man * 2.0 ** -9,
                     (1.0 + _man / 8.0) * np.exp2(_exp.astype(np.float64) - 7.0))
assert np.all(np.diff(_E4M3_POS) > 0) and _E4M3_POS[-1] == E4M3_MAX


def e4m3_rne(y: np.ndarray) -> np.ndarray:
    """Round fp32 values with |y| <= 448 to the nearest E4M3 code, ties to even code.

    Returns uint8 codes. Values are compared in fp64, where every fp32 input and
    every E4M3 value (and midpoint) is exact, so the nearest/tie decision is exact.
    """
    y = np.asarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    flat_y = y.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_y.size, step):
        v = flat_y[i:i + step].astype(np.float64)
        a = np.abs(v)
        if np.any(a > E4M3_MAX) or np.any(np.isnan(a)):
            raise ValueError("e4m3_rne: input outside [-448, 448]")
        hi = np.searchsorted(_E4M3_POS, a, side="left")     # _E4M3_POS[hi-1] < a <= _E4M3_POS[hi]
        hi_c = np.minimum(hi, 0x7E)
        lo_c = np.maximum(hi - 1, 0)
        d_hi = _E4M3_POS[hi_c] - a
        d_lo = a - _E4M3_POS[lo_c]
        pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi_c & 1) == 0))
        code = np.where(hi == 0, 0, np.where(pick_hi, hi_c, lo_c)).astype(np.uint8)
        code |= np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
        flat_o[i:i + step] = code
    return out


def _quantise_with_scale(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x / scale in fp32 (scale broadcast), saturate to +-448, round to E4M3."""
    y = (x / scale).astype(np.float32)
    np.clip(y, -E4M3_MAX, E4M3_MAX, out=y)
    return e4m3_rne(y)


def fp32_block_scale(amax: np.ndarray) -> np.ndarray:
    """fp32(amax/448), with 1.0 where the block is all zero."""
    amax = amax.astype(np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def ue8m0_from_amax(amax: np.ndarray) -> np.ndarray:
    """Byte e+127 with e = ceil(log2(fp32(amax/448))), exact (no log2 rounding)."""
    amax = amax.astype(np.float32)
    q = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    frac, ex = np.frexp(q)              # q = frac * 2^ex, frac in [0.5, 1)
    e = np.where(frac == 0.5, ex - 1, ex).astype(np.int64)
    byte = np.clip(e + 127, 0, 254)
    byte = np.where(amax == 0, 127, byte)
    return byte.astype(np.uint8)


def quantise_blockscale_a(x: np.ndarray):
    """A[M,K] fp32 -> (codes uint8 [M,K], scales fp32 [M, K/128])."""
    M, K = x.shape
    assert K % BLOCK_K == 0
    xb = x.reshape(M, K // BLOCK_K, BLOCK_K)
    scale = fp32_block_scale(np.abs(xb).max(axis=2))
    codes = _quantise_with_scale(xb, scale[:, :, None]).reshape(M, K)
    return codes, scale


def quantise_blockscale_b(x: np.ndarray):
    """B[N,K] fp32 -> (codes uint8 [N,K], scales fp32 [ceil(N/128), K/128]).

    A partial last N block uses the amax of the rows it has.
    """
    N, K = x.shape
    assert K % BLOCK_K == 0
    NB, KB = -(-N // BLOCK_K), K // BLOCK_K
    pad = NB * BLOCK_K - N
    xp = np.pad(x, ((0, pad), (0, 0))) if pad else x
    xb = xp.reshape(NB, BLOCK_K, KB, BLOCK_K)
    scale = fp32_block_scale(np.abs(xb).max(axis=(1, 3)))
    codes = _quantise_with_scale(xb, scale[:, None, :, None]).reshape(NB * BLOCK_K, K)[:N]
    return np.ascontiguousarray(codes), scale


def quantise_mxfp8(x: np.ndarray):
    """X[R,K] fp32 -> (codes uint8 [R,K], ue8m0 bytes uint8 [R, K/32])."""
    R, K = x.shape
    assert K % MX_GROUP == 0
    xg = x.reshape(R, K // MX_GROUP, MX_GROUP)
    e = ue8m0_from_amax(np.abs(xg).max(axis=2))
    scale = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)
    codes = _quantise_with_scale(xg, scale[:, :, None]).reshape(R, K)
    return codes, e


def quantise_tensorscale(x: np.ndarray):
    """X fp32 -> (codes uint8, one fp32 scale amax/448 for the whole tensor)."""
    scale = fp32_block_scale(np.array(np.abs(x).max(), dtype=np.float32))
    return _quantise_with_scale(x, scale), np.float32(scale)


@dataclass
class BlockscaleInputs:
    M: int
    N: int
    K: int
    seed: int
    A: np.ndarray        # uint8 [M,K] E4M3 codes
    a_scale: np.ndarray  # fp32 [M, K/128], logical a_scale[m, kb]
    B: np.ndarray        # uint8 [N,K] E4M3 codes
    b_scale: np.ndarray  # fp32 [ceil(N/128), K/128]

    def digest(self) -> str:
        h = hashlib.sha256()
        for t in (self.A, self.a_scale, self.B, self.b_scale):
            h.update(np.ascontiguousarray(t).tobytes())
        return h.hexdigest()


@dataclass
class MxInputs:
    M: int
    N: int
    K: int
    seed: int
    A: np.ndarray        # uint8 [M,K]
    a_e8m0: np.ndarray   # uint8 [M, K/32]
    B: np.ndarray        # uint8 [N,K]
    b_e8m0: np.ndarray   # uint8 [N, K/32]

    def digest(self) -> str:
        h = hashlib.sha256()
        for t in (self.A, self.a_e8m0, self.B, self.b_e8m0):
            h.update(np.ascontiguousarray(t).tobytes())
        return h.hexdigest()


def make_blockscale_inputs(M: int, N: int, K: int, seed: int = 0, b_std: float = 0.02) -> BlockscaleInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, K), dtype=np.float32)
    b = rng.standard_normal((N, K), dtype=np.float32) * np.float32(b_std)
    A, sa = quantise_blockscale_a(a)
    del a
    B, sb = quantise_blockscale_b(b)
    return BlockscaleInputs(M, N, K, seed, A, sa, B, sb)


@dataclass
class TensorscaleInputs:
    M: int
    N: int
    K: int
    seed: int
    A: np.ndarray        # uint8 [M,K]
    B: np.ndarray        # uint8 [N,K]
    alpha: np.float32    # fp32(scale_A * scale_B)


def make_tensorscale_inputs(M: int, N: int, K: int, seed: int = 0, b_std: float = 0.02) -> TensorscaleInputs:
    """The blockscale recipe's distributions, quantised with one scale per tensor."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, K), dtype=np.float32)
    b = rng.standard_normal((N, K), dtype=np.float32) * np.float32(b_std)
    A, sa = quantise_tensorscale(a)
    del a
    B, sb = quantise_tensorscale(b)
    return TensorscaleInputs(M, N, K, seed, A, B, np.float32(sa * sb))


@dataclass
class MoeInputs:
    tokens: int
    top_k: int
    num_experts: int
    N: int
    K: int
    seed: int
    A: np.ndarray             # uint8 [64 * n_blocks, K]: routed rows sorted by expert, padded per expert
    a_scale: np.ndarray       # fp32 [64 * n_blocks, K/128] (padding rows: zeros with scale 1)
    B: np.ndarray             # uint8 [E, N, K]
    b_scale: np.ndarray       # fp32 [E, N/128, K/128]
    block_expert: np.ndarray  # int32 [n_blocks]
    row_token: np.ndarray     # int32 [64 * n_blocks]: source token of each row, -1 for padding

    @property
    def n_blocks(self) -> int:
        return int(self.block_expert.shape[0])


MOE_BLOCK_ROWS = 64


def make_moe_inputs(tokens: int, top_k: int, num_experts: int, N: int, K: int, seed: int = 0,
                    skew: float = 0.0, b_std: float = 0.02) -> MoeInputs:
    """Synthetic MoE stage-1 routing and operands. Each token picks top_k
    distinct experts with probability proportional to (e + 1)^-skew (0 =
    uniform); rows are grouped by expert in token order and each expert's count
    is padded up to whole sort blocks of 64 rows, the layout the MoE align/sort
    step produces. Token activations N(0,1) are quantised per (token, 128-wide K
    block) and gathered; the expert weights N(0, b_std) are quantised per 128x128
    block (N a multiple of 128, so no block spans two experts)."""
    assert N % BLOCK_K == 0 and K % BLOCK_K == 0 and top_k <= num_experts
    rng = np.random.Generator(np.random.PCG64(seed))
    p = (np.arange(num_experts) + 1.0) ** (-skew)
    p /= p.sum()
    choice = np.stack([rng.choice(num_experts, size=top_k, replace=False, p=p) for _ in range(tokens)])
    x = rng.standard_normal((tokens, K), dtype=np.float32)
    codes, scales = quantise_blockscale_a(x)
    del x
    w = rng.standard_normal((num_experts * N, K), dtype=np.float32) * np.float32(b_std)
    B, sb = quantise_blockscale_b(w)
    del w
    row_token, block_expert = [], []
    for e in range(num_experts):
        toks = np.nonzero((choice == e).any(axis=1))[0]
        nb = -(-len(toks) // MOE_BLOCK_ROWS)
        pad = nb * MOE_BLOCK_ROWS - len(toks)
        row_token.extend(toks.tolist() + [-1] * pad)
        block_expert.extend([e] * nb)
    row_token = np.array(row_token, dtype=np.int32)
    real = row_token >= 0
    A = np.zeros((len(row_token), K), dtype=np.uint8)
    a_scale = np.ones((len(row_token), K // BLOCK_K), dtype=np.float32)
    A[real] = codes[row_token[real]]
    a_scale[real] = scales[row_token[real]]
    return MoeInputs(tokens, top_k, num_experts, N, K, seed, A, a_scale,
                     np.ascontiguousarray(B.reshape(num_experts, N, K)),
                     np.ascontiguousarray(sb.reshape(num_experts, N // BLOCK_K, K // BLOCK_K)),
                     np.array(block_expert, dtype=np.int32), row_token)


def make_mxfp8_inputs(M: int, N: int, K: int, seed: int = 0) -> MxInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, K), dtype=np.float32)
    b = rng.standard_normal((N, K), dtype=np.float32)
    A, ea = quantise_mxfp8(a)
    del a
    B, eb = quantise_mxfp8(b)
    return MxInputs(M, N, K, seed, A, ea, B, eb)


def a_scale_to_kmajor(a_scale: np.ndarray) -> np.ndarray:
    """Logical a_scale[M, KB] -> the library's K-block-major layout [KB, round_up(M,4)] (zero pad)."""
    M, KB = a_scale.shape
    ld = (M + 3) // 4 * 4
    out = np.zeros((KB, ld), dtype=np.float32)
    out[:, :M] = a_scale.T
    return out


# The workloads: shapes and seeds of the pages' measured layers.
WORKLOADS = {
    "bs_tiny_256x512x512": dict(kind="bs", M=256, N=512, K=512, seeds=(0,)),
    "bs_narrowN_4096x2048x7168": dict(kind="bs", M=4096, N=2048, K=7168, seeds=(0, 1, 2, 3)),
    "bs_narrowN_16384x1536x7168": dict(kind="bs", M=16384, N=1536, K=7168, seeds=(0, 1, 2, 3)),
    "bs_Klight_16384x7168x768": dict(kind="bs", M=16384, N=7168, K=768, seeds=(0, 1, 2, 3)),
    "bs_wideN_4096x65536x1536": dict(kind="bs", M=4096, N=65536, K=1536, seeds=(0, 1, 2, 3)),
}
for _m in (1024, 2048, 4096, 16384):
    WORKLOADS[f"mx_{_m}x5120x2048"] = dict(kind="mx", M=_m, N=5120, K=2048, seeds=(0,))
    WORKLOADS[f"mx_{_m}x8192x1280"] = dict(kind="mx", M=_m, N=8192, K=1280, seeds=(0,))
# Grouped MoE stage-1 (gate+up) at decode-like token counts: synthetic routing
# (skill card "FlyDSL decode MoE stage-1 blkmap": sort blocks of 64 rows; the
# card's measured model is not reproduced, these are generic sizes).
WORKLOADS["moe_s1_T256_top8_E32_N1536_K2048"] = dict(kind="moe", tokens=256, top_k=8, experts=32, N=1536,
                                                      K=2048, skew=0.0, seeds=(0,))
WORKLOADS["moe_s1_T1024_top8_E32_N1536_K2048_skew1"] = dict(kind="moe", tokens=1024, top_k=8, experts=32,
                                                             N=1536, K=2048, skew=1.0, seeds=(0,))


def make_inputs(kind: str, M: int, N: int, K: int, seed: int = 0):
    if kind == "bs":
        return make_blockscale_inputs(M, N, K, seed)
    if kind == "mx":
        return make_mxfp8_inputs(M, N, K, seed)
    raise ValueError(kind)
