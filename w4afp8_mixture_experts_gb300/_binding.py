"""ctypes binding of libw4a8moe.so: argument marshalling only.

Every step runs in the library's CUDA kernels; this module allocates outputs
with torch (device memory), passes raw pointers, sizes and the current CUDA
stream, and raises on a non-OK status.  There is no fallback: without the
built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_vp = ctypes.c_void_p
_c_sz = ctypes.c_size_t

_SIGS = {
    "w4a8_status_string": (ctypes.c_char_p, [_c_int]),
    "w4a8_last_error": (ctypes.c_char_p, []),
    "w4a8_abi_version": (_c_int, []),
    "w4a8_device_error": (_c_int, []),
    "moe_route_topk": (_c_int, [_c_vp, _c_i64, _c_i64, _c_int, _c_int, _c_vp, _c_vp, _c_vp]),
    "moe_permute": (_c_int, [_c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "moe_permute_ep": (_c_int, [_c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz,
                                _c_vp]),
    "fp8_quant_per_token_group": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp,
                                           _c_i64, _c_vp]),
    "fp8_quant_scatter_per_token_group": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                                                   _c_vp, _c_i64, _c_vp]),
    "w4a8_grouped_gemm": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                   _c_i64, _c_vp, _c_vp, _c_sz, _c_vp]),
    "w4a8_prepack_weights": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp]),
    "w4a8_grouped_gemm_silu": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                        _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_sz, _c_vp]),
    "w4a8_grouped_gemm_silu_unfused": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64,
                                                _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_sz, _c_vp]),
    "silu_mul_requant": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp]),
    "silu_mul_requant_rows": (_c_int, [_c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp]),
    "moe_unpermute_combine": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_vp]),
    "w4a8_linear": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp,
                             _c_sz, _c_vp]),
    "w4a8_workspace_bytes": (_c_sz, [_c_int, _c_i64, _c_i64, _c_i64, _c_i64]),
    "w4a8_linear_split_k": (_c_int, [_c_i64, _c_i64, _c_i64]),
    "w4a8_test_wait_timeout": (_c_int, [ctypes.c_uint64, _c_vp, _c_vp]),
    "w4a8_test_tile_list_limit": (_c_int, [_c_int]),
    "w4a8_grouped_gemm_plan": (_c_int, [_c_i64, _c_i64, _c_i64, ctypes.POINTER(_c_int)]),
    "w4a8_tile_cost": (ctypes.c_double, [_c_int, _c_i64]),
    "w4a8_expected_tile_cost": (ctypes.c_double, [_c_int, ctypes.c_double]),
    "w4a8_moe_forward": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_vp,
                                  _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "w4a8_moe_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, _c_i64, _c_int]),
    "w4a8_moe_forward_ep": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_vp, _c_i64,
                                     _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "w4a8_moe_forward_noalloc": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_vp,
                                          _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "w4a8_moe_noalloc_scratch_bytes": (_c_sz, []),
}


class MoeLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("topk_ids", "topk_w", "seg_indptr", "src2dst", "dst2src",
                                               "xq", "xs", "xc", "y13", "hq", "hs", "hc", "y2",
                                               "permute_ws")] + \
               [("scale_ld", ctypes.c_int64), ("total", ctypes.c_size_t)]


_lib = None


def load(path: str | None = None):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with w4afp8_mixture_experts_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    lib.w4a8_moe_workspace_layout.restype = _c_int
    lib.w4a8_moe_workspace_layout.argtypes = [_c_i64, _c_i64, _c_i64, _c_i64, _c_int, ctypes.POINTER(MoeLayout)]
    _lib = lib
    return lib


class W4A8Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} ({status})")
        self.status = status


def _check(status: int):
    if status != 0:
        lib = load()
        raise W4A8Error(status, lib.w4a8_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def scale_ld(m: int) -> int:
    """Leading dimension of an activation-scale tensor [K/128][ld] for m rows."""
    return max(4, (m + 3) // 4 * 4)


def _req(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


# ---------------------------------------------------------------------------

def moe_route_topk(logits, k: int, renormalize: bool = True):
    _req(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(load().moe_route_topk(_p(logits), T, E, k, int(bool(renormalize)), _p(ids), _p(w), _stream()))
    return ids, w


def moe_permute(topk_ids, E: int):
    _req(topk_ids, torch.int32, "topk_ids", 2)
    T, k = topk_ids.shape
    dev = topk_ids.device
    seg = torch.empty(E + 1, dtype=torch.int64, device=dev)
    s2d = torch.empty(T * k, dtype=torch.int32, device=dev)
    d2s = torch.empty(T * k, dtype=torch.int32, device=dev)
    need = int(load().w4a8_workspace_bytes(1, T * k, 0, 0, E))
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    _check(load().moe_permute(_p(topk_ids), T, k, E, _p(seg), _p(s2d), _p(d2s), _p(ws), need, _stream()))
    return seg, s2d, d2s


def moe_permute_ep(topk_ids, E: int, expert_map, E_local: int):
    """One expert-parallel shard's permutation: expert_map int32 [E] (local id or -1).
    Returns (seg_indptr int64 [E_local+1], src2dst int32 [T*k], dst2src int32 [T*k])."""
    _req(topk_ids, torch.int32, "topk_ids", 2)
    _req(expert_map, torch.int32, "expert_map", 1)
    T, k = topk_ids.shape
    dev = topk_ids.device
    seg = torch.empty(E_local + 1, dtype=torch.int64, device=dev)
    s2d = torch.empty(T * k, dtype=torch.int32, device=dev)
    d2s = torch.empty(T * k, dtype=torch.int32, device=dev)
    need = int(load().w4a8_workspace_bytes(1, T * k, 0, 0, E_local))
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    _check(load().moe_permute_ep(_p(topk_ids), T, k, E, _p(expert_map), E_local, _p(seg), _p(s2d), _p(d2s), _p(ws),
                                 need, _stream()))
    return seg, s2d, d2s


def fp8_quant_scatter_per_token_group(x, src2dst, k: int, m_out: int):
    """bf16 [T, K] -> codes uint8 [m_out, K], scales and gcorr fp32 [K/128, ld]: row t quantised once and
    written to rows src2dst[t*k + j] (-1 skipped; rows nothing maps to are left zero here)."""
    _req(x, torch.bfloat16, "x", 2)
    _req(src2dst, torch.int32, "src2dst", 1)
    T, K = x.shape
    ld = scale_ld(m_out)
    q = torch.zeros((m_out, K), dtype=torch.uint8, device=x.device)
    s = torch.zeros((max(1, K // 128), ld), dtype=torch.float32, device=x.device)
    c = torch.zeros((max(1, K // 128), ld), dtype=torch.float32, device=x.device)
    _check(load().fp8_quant_scatter_per_token_group(_p(x), T, K, _p(src2dst), k, m_out, _p(q), _p(s), _p(c), ld,
                                                    _stream()))
    return q, s, c


def fp8_quant_per_token_group(x, row_index=None, row_div: int = 1, m_out: int | None = None):
    """bf16 [M, K] -> (E4M3 codes uint8 [M_out, K], scales fp32 [K/128, ld], gcorr fp32 [K/128, ld])."""
    _req(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if row_index is not None:
        _req(row_index, torch.int32, "row_index", 1)
        m_out = row_index.numel() if m_out is None else m_out
    else:
        m_out = M
    ld = scale_ld(m_out)
    G = K // 128 if K % 128 == 0 else 1
    q = torch.empty((m_out, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((G, ld), dtype=torch.float32, device=x.device)
    c = torch.empty((G, ld), dtype=torch.float32, device=x.device)
    _check(load().fp8_quant_per_token_group(_p(x), M, K, _p(row_index), row_div, m_out, _p(q), _p(s), _p(c), ld,
                                            _stream()))
    return q, s, c


def w4a8_prepack_weights(w):
    """Canonical packed int4 uint8 [..., K/2] -> the GEMMs' prepacked layout (same shape)."""
    _req(w, torch.uint8, "w")
    out = torch.empty_like(w)
    K = w.shape[-1] * 2
    _check(load().w4a8_prepack_weights(_p(w), w.numel() // (K // 2), K, _p(out), _stream()))
    return out


def w4a8_grouped_gemm(A, a_scales, a_gcorr, B_prepacked, b_scales, seg_indptr):
    """A uint8 [M, K], a_scales [K/128, ld], a_gcorr [K/128, ld] or None (the library then computes the
    corrections from A in a workspace), B prepacked uint8 [E, N, K/2], b_scales [E, K/128, N] -> bf16 [M, N]."""
    _req(A, torch.uint8, "A", 2)
    _req(a_scales, torch.float32, "a_scales", 2)
    if a_gcorr is not None:
        _req(a_gcorr, torch.float32, "a_gcorr", 2)
    _req(B_prepacked, torch.uint8, "B_prepacked", 3)
    _req(b_scales, torch.float32, "b_scales", 3)
    _req(seg_indptr, torch.int64, "seg_indptr", 1)
    M, K = A.shape
    E, N, Kh = B_prepacked.shape
    if Kh * 2 != K or seg_indptr.numel() != E + 1 or (a_gcorr is not None and a_gcorr.shape != a_scales.shape):
        raise ValueError("shape mismatch")
    ws = None
    if a_gcorr is None:  # room for the corrections at this call's scale leading dimension
        ws = torch.empty((K // 128) * a_scales.shape[1] * 4, dtype=torch.uint8, device=A.device)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(load().w4a8_grouped_gemm(_p(A), _p(a_scales), _p(a_gcorr), a_scales.shape[1], _p(B_prepacked),
                                    _p(b_scales), _p(seg_indptr), E, N, K, M, _p(C), _p(ws),
                                    0 if ws is None else ws.numel(), _stream()))
    return C


def w4a8_grouped_gemm_silu(A, a_scales, a_gcorr, B_prepacked, b_scales, seg_indptr, fused: bool = True):
    """The w13 grouped GEMM (B_prepacked [E, 2I, K/2]: gate rows then up rows) followed by SiLU-and-Mul
    requantisation -> (codes uint8 [M, I], scales fp32 [I/128, ld], gcorr fp32 [I/128, ld]).  With
    fused=True the requantisation runs in the GEMM's epilogue when the tile plan allows (same bits)."""
    _req(A, torch.uint8, "A", 2)
    _req(a_scales, torch.float32, "a_scales", 2)
    if a_gcorr is not None:
        _req(a_gcorr, torch.float32, "a_gcorr", 2)
    _req(B_prepacked, torch.uint8, "B_prepacked", 3)
    _req(b_scales, torch.float32, "b_scales", 3)
    _req(seg_indptr, torch.int64, "seg_indptr", 1)
    M, K = A.shape
    E, N, Kh = B_prepacked.shape
    if Kh * 2 != K or seg_indptr.numel() != E + 1 or N % 256:
        raise ValueError("shape mismatch")
    I = N // 2
    ld = scale_ld(M)
    need = int(load().w4a8_workspace_bytes(4, M, N, K, E))
    if a_gcorr is None:
        need += (K // 128) * (a_scales.shape[1] - scale_ld(M)) * 4
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=A.device)
    q = torch.empty((M, I), dtype=torch.uint8, device=A.device)
    s = torch.empty((I // 128, ld), dtype=torch.float32, device=A.device)
    c = torch.empty((I // 128, ld), dtype=torch.float32, device=A.device)
    fn = load().w4a8_grouped_gemm_silu if fused else load().w4a8_grouped_gemm_silu_unfused
    _check(fn(_p(A), _p(a_scales), _p(a_gcorr), a_scales.shape[1], _p(B_prepacked), _p(b_scales), _p(seg_indptr), E,
              I, K, M, _p(q), _p(s), _p(c), ld, _p(ws), ws.numel(), _stream()))
    return q, s, c


def silu_mul_requant(gate_up):
    _req(gate_up, torch.bfloat16, "gate_up", 2)
    M, I2 = gate_up.shape
    I = I2 // 2
    ld = scale_ld(M)
    q = torch.empty((M, I), dtype=torch.uint8, device=gate_up.device)
    s = torch.empty((max(1, I // 128), ld), dtype=torch.float32, device=gate_up.device)
    c = torch.empty((max(1, I // 128), ld), dtype=torch.float32, device=gate_up.device)
    _check(load().silu_mul_requant(_p(gate_up), M, I, _p(q), _p(s), _p(c), ld, _stream()))
    return q, s, c


def moe_unpermute_combine(Y, src2dst, topk_w):
    _req(Y, torch.bfloat16, "Y", 2)
    _req(src2dst, torch.int32, "src2dst", 1)
    _req(topk_w, torch.float32, "topk_w", 2)
    T, k = topk_w.shape
    H = Y.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=Y.device)
    _check(load().moe_unpermute_combine(_p(Y), _p(src2dst), _p(topk_w), T, k, H, _p(out), _stream()))
    return out


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace of w4a8_linear (split-K partial sums, and room for the corrections when a_gcorr is None)."""
    return int(load().w4a8_workspace_bytes(3, M, N, K, 1))


def linear_split_k(M: int, N: int, K: int) -> int:
    """K splits w4a8_linear uses for this shape on the current device (1: none)."""
    return int(load().w4a8_linear_split_k(M, N, K))


def w4a8_linear(A, a_scales, a_gcorr, B_prepacked, b_scales, ws=None):
    """A uint8 [M, K], a_scales [K/128, ld], a_gcorr [K/128, ld] or None (computed by the library),
    B prepacked uint8 [N, K/2], b_scales [K/128, N] -> bf16 [M, N]."""
    _req(A, torch.uint8, "A", 2)
    _req(a_scales, torch.float32, "a_scales", 2)
    if a_gcorr is not None:
        _req(a_gcorr, torch.float32, "a_gcorr", 2)
    _req(B_prepacked, torch.uint8, "B_prepacked", 2)
    _req(b_scales, torch.float32, "b_scales", 2)
    M, K = A.shape
    N = B_prepacked.shape[0]
    if ws is None:
        need = linear_workspace_bytes(M, N, K)
        if a_gcorr is None:  # the corrections at this call's scale leading dimension
            need += (K // 128) * (a_scales.shape[1] - scale_ld(M)) * 4
        ws = torch.empty(need, dtype=torch.uint8, device=A.device) if need else None
    C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(load().w4a8_linear(_p(A), _p(a_scales), _p(a_gcorr), a_scales.shape[1], _p(B_prepacked), _p(b_scales),
                              M, N, K, _p(C), _p(ws), 0 if ws is None else ws.numel(), _stream()))
    return C


def moe_workspace_layout(T: int, H: int, I: int, E: int, k: int) -> MoeLayout:
    L = MoeLayout()
    _check(load().w4a8_moe_workspace_layout(T, H, I, E, k, ctypes.byref(L)))
    return L


def w4a8_moe_forward(x, logits, k: int, w13, w13_s, w2, w2_s, renormalize: bool = True, ws=None, out=None):
    """The whole layer.  x bf16 [T, H], logits fp32 [T, E], w13 prepacked uint8 [E, 2I, H/2],
    w13_s fp32 [E, H/128, 2I], w2 prepacked uint8 [E, H, I/2], w2_s fp32 [E, I/128, H] -> bf16 [T, H]."""
    _req(x, torch.bfloat16, "x", 2)
    _req(logits, torch.float32, "logits", 2)
    _req(w13, torch.uint8, "w13", 3)
    _req(w2, torch.uint8, "w2", 3)
    _req(w13_s, torch.float32, "w13_s", 3)
    _req(w2_s, torch.float32, "w2_s", 3)
    T, H = x.shape
    E = logits.shape[1]
    I = w13.shape[1] // 2
    need = int(load().w4a8_moe_workspace_bytes(T, H, I, E, k))
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().w4a8_moe_forward(_p(x), _p(logits), T, H, I, E, k, int(bool(renormalize)), _p(w13), _p(w13_s),
                                   _p(w2), _p(w2_s), _p(out), _p(ws), ws.numel(), _stream()))
    return out


def w4a8_moe_forward_ep(x, logits, k: int, expert_map, w13, w13_s, w2, w2_s, renormalize: bool = True, ws=None,
                        out=None):
    """One expert-parallel shard of the layer: routing over the E = logits.shape[1] experts, the rest over
    the E_local = w13.shape[0] local experts named by expert_map (int32 [E], local id or -1).  Returns
    this shard's share of the layer output, bf16 [T, H]."""
    _req(x, torch.bfloat16, "x", 2)
    _req(logits, torch.float32, "logits", 2)
    _req(expert_map, torch.int32, "expert_map", 1)
    _req(w13, torch.uint8, "w13", 3)
    _req(w2, torch.uint8, "w2", 3)
    _req(w13_s, torch.float32, "w13_s", 3)
    _req(w2_s, torch.float32, "w2_s", 3)
    T, H = x.shape
    E = logits.shape[1]
    E_local = w13.shape[0]
    I = w13.shape[1] // 2
    need = int(load().w4a8_moe_workspace_bytes(T, H, I, E, k))
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().w4a8_moe_forward_ep(_p(x), _p(logits), T, H, I, E, k, int(bool(renormalize)), _p(expert_map),
                                      E_local, _p(w13), _p(w13_s), _p(w2), _p(w2_s), _p(out), _p(ws), ws.numel(),
                                      _stream()))
    return out


def w4a8_moe_forward_noalloc(x, logits, k: int, w13, w13_s, w2, w2_s, out, renormalize: bool = True):
    """The whole layer into a caller-given `out`, with the intermediates kept in the
    library's fixed device array instead of a workspace (for callers that cannot
    allocate device memory).  Calls that overlap on the GPU race on that array."""
    _req(x, torch.bfloat16, "x", 2)
    _req(logits, torch.float32, "logits", 2)
    _req(out, torch.bfloat16, "out", 2)
    T, H = x.shape
    E = logits.shape[1]
    I = w13.shape[1] // 2
    _check(load().w4a8_moe_forward_noalloc(_p(x), _p(logits), T, H, I, E, k, int(bool(renormalize)), _p(w13),
                                           _p(w13_s), _p(w2), _p(w2_s), _p(out), _stream()))
    return out


def device_error() -> int:
    return int(load().w4a8_device_error())
