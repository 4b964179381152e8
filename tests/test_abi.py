"""The C ABI without a GPU: the library loads, exports every entry point the header declares,
and rejects bad arguments on the host before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a8moe.h")


@pytest.fixture(scope="module")
def clib():
    from w4afp8_mixture_experts_gb300 import build
    build.build()
    import w4afp8_mixture_experts_gb300._binding as b
    return b.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|const char\s*\*)\s*\**\s*(\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(clib):
    names = declared_functions()
    assert len(names) >= 16
    for n in ["moe_route_topk", "moe_permute", "fp8_quant_per_token_group", "w4a8_grouped_gemm",
              "silu_mul_requant", "moe_unpermute_combine", "w4a8_linear", "w4a8_prepack_weights",
              "w4a8_moe_forward", "w4a8_moe_forward_noalloc", "moe_permute_ep", "w4a8_moe_forward_ep",
              "fp8_quant_scatter_per_token_group", "silu_mul_requant_rows"]:
        assert n in names
    for n in names:
        assert hasattr(clib, n), n


def test_status_strings_and_version(clib):
    assert clib.w4a8_abi_version() == 4
    assert clib.w4a8_status_string(0) == b"ok"
    assert clib.w4a8_status_string(1) == b"invalid argument"
    assert clib.w4a8_status_string(4) == b"device-side wait timed out"


NULL = None
P16 = ctypes.c_void_p(16)  # a 16-byte aligned non-null dummy (never dereferenced: rejected first)


@pytest.mark.parametrize("call,msg", [
    (lambda L: L.moe_route_topk(P16, 4, 8, 9, 1, P16, P16, NULL), b"k=9"),
    (lambda L: L.moe_route_topk(P16, 4, 2000, 2, 1, P16, P16, NULL), b"E=2000"),
    (lambda L: L.moe_permute(P16, 4, 2, 0, P16, P16, P16, NULL, 0, NULL), b"E=0"),
    (lambda L: L.moe_permute(P16, 1024, 8, 256, P16, P16, P16, NULL, 0, NULL), b"workspace"),
    (lambda L: L.moe_permute_ep(P16, 4, 2, 8, NULL, 4, P16, P16, P16, NULL, 0, NULL), b"expert_map"),
    (lambda L: L.moe_permute_ep(P16, 4, 2, 8, P16, 0, P16, P16, P16, NULL, 0, NULL), b"E_local=0"),
    (lambda L: L.moe_permute_ep(P16, 1024, 8, 256, P16, 32, P16, P16, P16, NULL, 0, NULL), b"workspace"),
    (lambda L: L.fp8_quant_per_token_group(P16, 4, 100, NULL, 1, 4, P16, P16, NULL, 4, NULL), b"K=100"),
    (lambda L: L.fp8_quant_per_token_group(P16, 4, 128, NULL, 1, 4, P16, P16, NULL, 2, NULL), b"scale_ld"),
    (lambda L: L.fp8_quant_scatter_per_token_group(P16, 4, 100, P16, 2, 8, P16, P16, NULL, 8, NULL), b"K=100"),
    (lambda L: L.fp8_quant_scatter_per_token_group(P16, 4, 128, P16, 33, 8, P16, P16, NULL, 8, NULL), b"k=33"),
    (lambda L: L.w4a8_grouped_gemm(P16, P16, P16, 4, P16, P16, P16, 2, 256, 200, 4, P16, NULL, 0, NULL), b"K=200"),
    (lambda L: L.w4a8_grouped_gemm(P16, P16, P16, 4, P16, P16, P16, 2, 100, 256, 4, P16, NULL, 0, NULL), b"N=100"),
    (lambda L: L.w4a8_grouped_gemm(P16, P16, P16, 4, P16, P16, NULL, 2, 128, 256, 4, P16, NULL, 0, NULL),
     b"seg_indptr"),
    (lambda L: L.w4a8_linear(P16, P16, P16, 4, NULL, P16, 4, 128, 256, P16, NULL, 0, NULL), b"null"),
    # no caller corrections: the call computes them and needs (K/128) x ld fp32 of workspace
    (lambda L: L.w4a8_linear(P16, P16, NULL, 4, P16, P16, 4, 128, 256, P16, NULL, 0, NULL), b"workspace"),
    (lambda L: L.w4a8_grouped_gemm(P16, P16, NULL, 4, P16, P16, P16, 2, 128, 256, 4, P16, P16, 16, NULL),
     b"workspace"),
    (lambda L: L.w4a8_linear(P16, P16, ctypes.c_void_p(20), 4, P16, P16, 4, 128, 256, P16, NULL, 0, NULL),
     b"aligned"),
    (lambda L: L.silu_mul_requant(P16, 4, 100, P16, P16, NULL, 4, NULL), b"I=100"),
    (lambda L: L.silu_mul_requant_rows(P16, 4, P16, 100, P16, P16, NULL, 4, NULL), b"I=100"),
    (lambda L: L.moe_unpermute_combine(P16, P16, P16, 4, 2, 12, P16, NULL), b"H=12"),
    (lambda L: L.w4a8_prepack_weights(P16, 4, 12, P16, NULL), b"K=12"),
    (lambda L: L.w4a8_moe_forward(P16, P16, 4, 256, 256, 8, 2, 1, P16, P16, P16, P16, P16, P16, 10, NULL),
     b"workspace too small"),
    (lambda L: L.w4a8_moe_forward_noalloc(P16, P16, 4096, 7168, 2048, 8, 8, 1, P16, P16, P16, P16, P16, NULL),
     b"at most"),
    (lambda L: L.w4a8_moe_forward_ep(P16, P16, 4, 256, 256, 8, 2, 1, P16, 9, P16, P16, P16, P16, P16, P16,
                                     1 << 30, NULL), b"E_local=9"),
    (lambda L: L.w4a8_moe_forward_ep(P16, P16, 4, 256, 256, 8, 2, 1, NULL, 4, P16, P16, P16, P16, P16, P16,
                                     1 << 30, NULL), b"expert_map"),
])
def test_host_validation_rejects_before_launch(clib, call, msg):
    assert call(clib) == 1  # W4A8_ERR_INVALID_ARG
    assert msg in clib.w4a8_last_error()


def test_moe_workspace_layout(clib):
    import w4afp8_mixture_experts_gb300._binding as b
    L = b.moe_workspace_layout(64, 7168, 2048, 256, 8)
    offs = [getattr(L, n) for n in ("topk_ids", "topk_w", "seg_indptr", "src2dst", "dst2src", "xq", "xs", "xc",
                                    "y13", "hq", "hs", "hc", "y2")]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    P = 64 * 8
    assert L.scale_ld == P and L.total >= P * 7168 + P * 4096 * 2 + P * 2048 + P * 7168 * 2
    assert clib.w4a8_moe_workspace_bytes(64, 7168, 2048, 256, 8) == L.total
    assert clib.w4a8_moe_noalloc_scratch_bytes() == 64 << 20


def test_gemm_workspace_sizes(clib):
    # the corrections of M rows (ld = M rounded up to 4) over K/128 groups, after the split-K partials
    assert clib.w4a8_workspace_bytes(2, 300, 256, 1024, 8) == 8 * 300 * 4
    assert clib.w4a8_workspace_bytes(2, 5, 256, 1024, 8) == 8 * 8 * 4
    assert clib.w4a8_workspace_bytes(3, 1000, 128, 256, 1) == 2 * 1000 * 4  # no split at this shape
    assert clib.w4a8_workspace_bytes(2, 0, 256, 1024, 8) == 0
