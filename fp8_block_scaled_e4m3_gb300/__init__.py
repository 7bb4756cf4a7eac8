"""FP8 block-scaled GEMM and MXFP8 GEMM on GB300 (sm_103a).

Entry points: gemm_blockscale, gemm_blockscale_e4m3out (E4M3 C), gemm_mxfp8,
gemm_mxfp8_packed, gemm_mxfp8_e4m3out, gemm_tensorscale (the promote-free
twin), moe_leaders + gemm_moe (grouped MoE stage-1 over 64-row sort blocks),
plus the layout helpers, status and configuration introspection.

Thin ctypes binding over libfp8bs.so (include/fp8bs.h). Every step of the
computation runs in the library's CUDA kernels; this module only checks
tensors, marshals pointers and the current CUDA stream, and raises on a
non-zero status. PyTorch provides device memory and streams.

There is no CPU fallback: if the library is missing, importing the package
raises ImportError with the build command.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libfp8bs.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(
        f"{LIBRARY_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python fp8_block_scaled_e4m3_gb300/_build.py` (needs nvcc for sm_103a)")

_lib = ctypes.CDLL(LIBRARY_PATH)
_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64

_SIGS = {
    "fp8bs_gemm": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "fp8bs_gemm_tensorscale": (_i, [_p, _p, _p, _i, _i, _i, ctypes.c_float, _p]),
    "fp8bs_gemm_e4m3out": (_i, [_p, _p, _p, _p, _p, ctypes.c_float, _i, _i, _i, _p]),
    "fp8bs_moe_leaders": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "fp8bs_shutdown": (_i, []),
    "fp8mx_gemm_e4m3out": (_i, [_p, _p, _p, _p, _p, ctypes.c_float, _i, _i, _i, _p]),
    "fp8bs_moe_gemm": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _p]),
    "fp8mx_gemm": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "fp8mx_gemm_packed": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "fp8mx_packed_scale_bytes": (_i64, [_i, _i]),
    "fp8mx_pack_scales": (_i, [_p, _p, _i, _i, _p]),
    "fp8mx_launches_per_call": (_i, []),
    "fp8mx_gemm_noalloc": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "fp8mx_noalloc_scratch_bytes": (_i64, []),
    "fp8bs_a_scale_ld": (_i64, [_i]),
    "fp8bs_a_scale_index": (_i64, [_i, _i, _i]),
    "fp8bs_b_scale_index": (_i64, [_i, _i, _i]),
    "fp8mx_scale_index": (_i64, [_i, _i, _i]),
    "fp8mx_sf_atom_offset": (_i, [_i, _i]),
    "fp8bs_pack_a_scale": (_i, [_p, _p, _i, _i, _p]),
    "fp8bs_get_status": (_i, [_p]),
    "fp8bs_status_string": (ctypes.c_char_p, [_i]),
    "fp8bs_last_config_id": (_i, []),
    "fp8bs_select_config": (_i, [_i, _i, _i, _i]),
    "fp8mx_select_config": (_i, [_i, _i, _i, _i]),
    "fp8bs_launches_per_call": (_i, []),
    "fp8bs_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "fp8bs_set_config_override": (_i, [_i]),
    "fp8bs_set_raster_group": (_i, [_i]),
    "fp8bs_device_info": (_i, [_p, _p]),
    "fp8bs_version": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

STATUS = {0: "FP8BS_OK", -1: "FP8BS_ERR_NULL", -2: "FP8BS_ERR_ALIGN", -3: "FP8BS_ERR_SHAPE",
          -4: "FP8BS_ERR_UNSUPPORTED_DEVICE", -5: "FP8BS_ERR_LAUNCH", -6: "FP8BS_ERR_DEVICE_TIMEOUT",
          -7: "FP8BS_ERR_CUDA", -8: "FP8BS_ERR_SCRATCH_TOO_SMALL"}


class Fp8bsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.fp8bs_status_string(code).decode()
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise Fp8bsError(rc, where)


def lib() -> ctypes.CDLL:
    """The loaded libfp8bs.so (for the C-ABI tests and the benchmark)."""
    return _lib


def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _fp8_ptr(t, name, shape):
    torch = _torch()
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError(f"{name} must be float8_e4m3fn or uint8 E4M3 codes, got {t.dtype}")
    return _dev_ptr(t, name, shape)


def _dev_ptr(t, name, shape):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def a_scale_ld(M: int) -> int:
    return int(_lib.fp8bs_a_scale_ld(M))


def gemm_blockscale(A, a_scale, B, b_scale, C=None, stream=None):
    """C[M,N] bf16 = sum_kb (A.B^T)_kb * a_scale[m,kb] * b_scale[n//128,kb].

    A: [M,K] E4M3; a_scale: fp32 [K/128, a_scale_ld(M)] K-block-major;
    B: [N,K] E4M3; b_scale: fp32 [ceil(N/128), K/128]; C: optional bf16 [M,N] output.
    """
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if a_scale.dtype != torch.float32 or b_scale.dtype != torch.float32 or C.dtype != torch.bfloat16:
        raise TypeError("scales must be float32 and C bfloat16")
    rc = _lib.fp8bs_gemm(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_scale, "a_scale", (K // 128, a_scale_ld(M))),
                         _fp8_ptr(B, "B", (N, K)), _dev_ptr(b_scale, "b_scale", ((N + 127) // 128, K // 128)),
                         _dev_ptr(C, "C", (M, N)), M, N, K, _stream_ptr(stream))
    _check(rc, "fp8bs_gemm")
    return C


def gemm_blockscale_e4m3out(A, a_scale, B, b_scale, c_scale, C8=None, stream=None):
    """C8[M,N] E4M3 codes (uint8) = e4m3(c_scale * the blockscale GEMM's fp32 sum),
    rounded to nearest even and saturated at +-448; decode(C8) / c_scale recovers C.
    Arguments as gemm_blockscale; N must be a multiple of 16."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C8 is None:
        C8 = torch.empty((M, N), dtype=torch.uint8, device=A.device)
    if a_scale.dtype != torch.float32 or b_scale.dtype != torch.float32:
        raise TypeError("scales must be float32")
    if C8.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("C8 must be uint8 or float8_e4m3fn")
    rc = _lib.fp8bs_gemm_e4m3out(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_scale, "a_scale", (K // 128, a_scale_ld(M))),
                                 _fp8_ptr(B, "B", (N, K)),
                                 _dev_ptr(b_scale, "b_scale", ((N + 127) // 128, K // 128)),
                                 _dev_ptr(C8, "C8", (M, N)), float(c_scale), M, N, K, _stream_ptr(stream))
    _check(rc, "fp8bs_gemm_e4m3out")
    return C8


def gemm_mxfp8_e4m3out(A, a_e8m0, B, b_e8m0, c_scale, C8=None, stream=None):
    """C8[M,N] E4M3 codes (uint8) = e4m3(c_scale * the MXFP8 GEMM's fp32 sum); N % 16 == 0."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C8 is None:
        C8 = torch.empty((M, N), dtype=torch.uint8, device=A.device)
    if C8.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("C8 must be uint8 or float8_e4m3fn")
    rc = _lib.fp8mx_gemm_e4m3out(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_e8m0, "a_e8m0", (M, K // 32)),
                                 _fp8_ptr(B, "B", (N, K)), _dev_ptr(b_e8m0, "b_e8m0", (N, K // 32)),
                                 _dev_ptr(C8, "C8", (M, N)), float(c_scale), M, N, K, _stream_ptr(stream))
    _check(rc, "fp8mx_gemm_e4m3out")
    return C8


MOE_BLOCK_ROWS = 64


def moe_leaders(block_expert, num_experts, pair=True, leaders=None, n_leaders=None, stream=None):
    """Leader descriptor of a sorted block->expert table (int32 [n_blocks], device):
    returns (leaders int32 [n_blocks], n_leaders int32 [1]), both on the device;
    leader value = first block | (covers two blocks) << 30. One kernel, no sync."""
    torch = _torch()
    n_blocks = int(block_expert.shape[0])
    if block_expert.dtype != torch.int32:
        raise TypeError("block_expert must be int32")
    if leaders is None:
        leaders = torch.empty((max(n_blocks, 1),), dtype=torch.int32, device=block_expert.device)
    if n_leaders is None:
        n_leaders = torch.empty((1,), dtype=torch.int32, device=block_expert.device)
    rc = _lib.fp8bs_moe_leaders(_dev_ptr(block_expert, "block_expert", (n_blocks,)), n_blocks, int(num_experts),
                                1 if pair else 0, _dev_ptr(leaders, "leaders", tuple(leaders.shape)),
                                _dev_ptr(n_leaders, "n_leaders", (1,)), _stream_ptr(stream))
    _check(rc, "fp8bs_moe_leaders")
    return leaders, n_leaders


def gemm_moe(A, a_scale, B, b_scale, block_expert, leaders, n_leaders, C=None, stream=None):
    """Grouped MoE blockscale GEMM over sort blocks of 64 rows.
    A: [64*n_blocks, K] E4M3 (sorted rows); a_scale: fp32 [K/128, a_scale_ld(64*n_blocks)];
    B: [E, N, K] E4M3; b_scale: fp32 [E, ceil(N/128), K/128]; C: bf16 [64*n_blocks, N]
    (rows of blocks whose expert is out of range are left as they are)."""
    torch = _torch()
    M, K = A.shape
    E, N, _ = B.shape
    n_blocks = int(block_expert.shape[0])
    if M != n_blocks * MOE_BLOCK_ROWS:
        raise ValueError(f"A has {M} rows, expected {n_blocks} blocks x {MOE_BLOCK_ROWS}")
    if C is None:
        C = torch.zeros((M, N), dtype=torch.bfloat16, device=A.device)
    rc = _lib.fp8bs_moe_gemm(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_scale, "a_scale", (K // 128, a_scale_ld(M))),
                             _fp8_ptr(B, "B", (E, N, K)),
                             _dev_ptr(b_scale, "b_scale", (E, (N + 127) // 128, K // 128)),
                             _dev_ptr(C, "C", (M, N)), _dev_ptr(block_expert, "block_expert", (n_blocks,)),
                             _dev_ptr(leaders, "leaders", tuple(leaders.shape)),
                             _dev_ptr(n_leaders, "n_leaders", (1,)), n_blocks, N, K, E, _stream_ptr(stream))
    _check(rc, "fp8bs_moe_gemm")
    return C


def gemm_tensorscale(A, B, alpha, C=None, stream=None):
    """C[M,N] bf16 = alpha * A.B^T: the promote-free ceiling twin of gemm_blockscale
    (same tiles and MMA work, one per-tensor scale). A: [M,K] E4M3; B: [N,K] E4M3."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16:
        raise TypeError("C must be bfloat16")
    rc = _lib.fp8bs_gemm_tensorscale(_fp8_ptr(A, "A", (M, K)), _fp8_ptr(B, "B", (N, K)), _dev_ptr(C, "C", (M, N)),
                                     M, N, K, float(alpha), _stream_ptr(stream))
    _check(rc, "fp8bs_gemm_tensorscale")
    return C


def gemm_mxfp8(A, a_e8m0, B, b_e8m0, C=None, stream=None):
    """C[M,N] bf16 = sum_k A[m,k] 2^(a_e8m0[m,k/32]-127) B[n,k] 2^(b_e8m0[n,k/32]-127).

    A: [M,K] E4M3; a_e8m0: uint8 [M, K/32]; B: [N,K] E4M3; b_e8m0: uint8 [N, K/32].
    """
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if a_e8m0.dtype != torch.uint8 or b_e8m0.dtype != torch.uint8 or C.dtype != torch.bfloat16:
        raise TypeError("ue8m0 scales must be uint8 and C bfloat16")
    rc = _lib.fp8mx_gemm(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_e8m0, "a_e8m0", (M, K // 32)),
                         _fp8_ptr(B, "B", (N, K)), _dev_ptr(b_e8m0, "b_e8m0", (N, K // 32)),
                         _dev_ptr(C, "C", (M, N)), M, N, K, _stream_ptr(stream))
    _check(rc, "fp8mx_gemm")
    return C


def packed_scale_bytes(rows: int, K: int) -> int:
    return int(_lib.fp8mx_packed_scale_bytes(rows, K))


def pack_mx_scales(e8m0, K: int, out=None, stream=None):
    """ue8m0 bytes [rows, K/32] -> the packed scale-factor layout gemm_mxfp8_packed takes."""
    torch = _torch()
    rows = e8m0.shape[0]
    if out is None:
        out = torch.empty((packed_scale_bytes(rows, K),), dtype=torch.uint8, device=e8m0.device)
    if e8m0.dtype != torch.uint8:
        raise TypeError("ue8m0 scales must be uint8")
    rc = _lib.fp8mx_pack_scales(_dev_ptr(e8m0, "e8m0", (rows, K // 32)),
                                _dev_ptr(out, "out", (packed_scale_bytes(rows, K),)), rows, K, _stream_ptr(stream))
    _check(rc, "fp8mx_pack_scales")
    return out


def gemm_mxfp8_packed(A, a_sf, B, b_sf, C=None, stream=None):
    """MXFP8 GEMM on packed scale factors (from pack_mx_scales); one kernel, no allocation."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if a_sf.dtype != torch.uint8 or b_sf.dtype != torch.uint8 or C.dtype != torch.bfloat16:
        raise TypeError("packed scales must be uint8 and C bfloat16")
    rc = _lib.fp8mx_gemm_packed(_fp8_ptr(A, "A", (M, K)), _dev_ptr(a_sf, "a_sf", (packed_scale_bytes(M, K),)),
                                _fp8_ptr(B, "B", (N, K)), _dev_ptr(b_sf, "b_sf", (packed_scale_bytes(N, K),)),
                                _dev_ptr(C, "C", (M, N)), M, N, K, _stream_ptr(stream))
    _check(rc, "fp8mx_gemm_packed")
    return C


def pack_a_scale(a_scale_rowmajor, K: int, out=None, stream=None):
    """Row-major logical a_scale [M, K/128] -> the K-block-major layout gemm_blockscale takes."""
    torch = _torch()
    M = a_scale_rowmajor.shape[0]
    if out is None:
        out = torch.empty((K // 128, a_scale_ld(M)), dtype=torch.float32, device=a_scale_rowmajor.device)
    rc = _lib.fp8bs_pack_a_scale(_dev_ptr(a_scale_rowmajor, "a_scale", (M, K // 128)),
                                 _dev_ptr(out, "out", (K // 128, a_scale_ld(M))), M, K, _stream_ptr(stream))
    _check(rc, "fp8bs_pack_a_scale")
    return out


def get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(_lib.fp8bs_get_status(_stream_ptr(stream)))


def last_config_id() -> int:
    return int(_lib.fp8bs_last_config_id())


def select_config(kind: str, M: int, N: int, K: int, num_sms: int) -> int:
    f = _lib.fp8bs_select_config if kind == "bs" else _lib.fp8mx_select_config
    return int(f(M, N, K, num_sms))


def decode_config(cid: int) -> dict:
    return {"kind": {1: "blockscale", 2: "mxfp8", 3: "blockscale_pair", 4: "tensorscale", 5: "mxfp8_pair",
                      6: "mxfp8_decode"}.get(cid // 1000000, "?"),
            "block_n": (cid // 1000) % 1000,
            "stages": (cid // 100) % 10, "raster": (cid // 10) % 10,
            "schedule": {1: "tile", 2: "stream_k"}.get(cid % 10, "?")}


def device_info() -> dict:
    """SM count and resident CTA pairs of the current device (as the library sees them)."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.fp8bs_device_info(ctypes.byref(a), ctypes.byref(b)), "fp8bs_device_info")
    return {"num_sms": a.value, "pair_clusters": b.value}


def set_config_override(config_id: int) -> None:
    """Force a kernel configuration (0 = choose by shape); see include/fp8bs.h."""
    _check(_lib.fp8bs_set_config_override(int(config_id)), "fp8bs_set_config_override")


def set_raster_group(group: int) -> None:
    """Tile-order group size of later launches (0 = default 1); see include/fp8bs.h."""
    _check(_lib.fp8bs_set_raster_group(int(group)), "fp8bs_set_raster_group")


def set_wait_limit_ns(ns: int) -> None:
    _lib.fp8bs_set_wait_limit_ns(int(ns))


def shutdown() -> None:
    """Release the library's per-device workspace pools (see fp8bs_shutdown)."""
    _check(_lib.fp8bs_shutdown(), "fp8bs_shutdown")


def version() -> str:
    return _lib.fp8bs_version().decode()
