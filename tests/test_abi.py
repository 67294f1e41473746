"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every entry point
include/nvfp4.h declares, answers the size queries, and rejects bad arguments before it touches
a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as nv
    return nv


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:nvfp4|mxfp4|sf)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("nvfp4_quantize", "nvfp4_gemm", "mxfp4_quantize", "mxfp4_grouped_gemm", "sf_swizzle",
                 "nvfp4_last_error", "nvfp4_sf_bytes", "nvfp4_check_status", "nvfp4_gemm_plan",
                 "nvfp4_gemm_workspace_size"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name


def test_size_queries(lib):
    assert lib.sf_bytes(1, 16, 16) == 128 * 4
    assert lib.sf_bytes(32, 1024, 16) == 128 * 64
    assert lib.sf_bytes(129, 7168, 16) == 256 * 448
    assert lib.sf_bytes(5, 96, 16) == 128 * 8
    assert lib.sf_bytes(300, 2048, 32) == 384 * 64
    assert lib.sf_bytes(-1, 16, 16) == 0
    assert lib.sf_bytes(4, 24, 16) == 0
    assert lib.sf_bytes(4, 32, 8) == 0
    assert lib.grouped_sf_bytes(32768, 128, 2048) == (32768 + 128 * 128) * 64
    assert lib.grouped_sf_bytes(10, 0, 64) == 0


def test_plan_selector_buckets(lib):
    """Without a device the selector plans for 152 SMs."""
    for m in (1, 4, 8, 16):
        p = lib.nvfp4_gemm_plan(m, 4096, 7168)
        # 32 weight tiles, K split 7 ways inside clusters (two CTAs per SM): 224 CTAs
        assert p["swap_ab"] == 1 and p["tile_n"] == 32 and p["splits"] == 7
        assert p["dp_tiles"] == 32 and p["sk_tiles"] == 0 and p["ctas"] == 224
    assert lib.nvfp4_gemm_plan(32, 4096, 7168)["tile_n"] == 32
    assert lib.nvfp4_gemm_plan(256, 4096, 7168)["tile_n"] == 256
    big = lib.nvfp4_gemm_plan(4096, 4096, 7168)
    # 256 tiles of 256x256, walked whole and persistently by 76 CTA pairs; K % 256 == 0, so a
    # ring stage holds two 256-wide K steps (3 stages)
    assert big["swap_ab"] == 0 and big["tile_m"] == 256 and big["tile_n"] == 256 and big["ctas"] == 152
    assert big["dp_tiles"] == 256 and big["sk_tiles"] == 0 and big["stages"] == 3
    ragged = lib.nvfp4_gemm_plan(300, 13056, 512)           # 3 x 51 single tiles -> 2 x 51 pair tiles
    assert ragged["tile_m"] == 256 and ragged["dp_tiles"] == 102 and ragged["ctas"] == 152
    # 64 pair tiles fill more than a quarter of the 76 pairs: pairs from 129 tokens on
    mid = lib.nvfp4_gemm_plan(1024, 4096, 7168)
    assert mid["tile_m"] == 256 and mid["dp_tiles"] == 64 and mid["ctas"] == 128
    # 16 pair tiles would fill too few: swap-AB, four-way cluster split-K
    assert lib.nvfp4_gemm_plan(256, 4096, 7168)["swap_ab"] == 1
    assert lib.nvfp4_gemm_plan(256, 14336, 4096)["tile_m"] == 256   # 56 pair tiles
    # short K (8 steps) at N >= 4096: 128 x 128 tiles over the whole K instead of split-K
    short = lib.nvfp4_gemm_plan(128, 7168, 2048)
    assert short["swap_ab"] == 0 and short["tile_n"] == 128 and short["splits"] == 1
    assert short["dp_tiles"] == 56 and short["sk_tiles"] == 0 and short["ctas"] == 56
    assert lib.nvfp4_gemm_plan(256, 4096, 2048)["dp_tiles"] == 64
    assert lib.nvfp4_gemm_plan(16, 7168, 2048)["swap_ab"] == 1     # up to 16 tokens: split-K
    assert lib.nvfp4_gemm_plan(128, 7168, 4096)["swap_ab"] == 1    # longer K, one token tile: split-K
    two = lib.nvfp4_gemm_plan(256, 7168, 4096)                      # two token tiles, K <= 4096
    assert two["swap_ab"] == 0 and two["dp_tiles"] == 112 and two["sk_tiles"] == 0 and two["ctas"] == 112
    assert lib.nvfp4_gemm_plan(256, 4096, 7168)["swap_ab"] == 1    # K = 7168: split-K
    small = lib.nvfp4_gemm_plan(32, 1024, 1024)            # 8 tiles x 4 stages: one stage per CTA
    assert small["splits"] == 4 and small["ctas"] == 32
    few = lib.nvfp4_gemm_plan(640, 1024, 2048)             # 40 tiles but only 2 stages per SM
    assert few["sk_tiles"] == 0 and few["ctas"] == 40
    deep = lib.nvfp4_gemm_plan(300, 1024, 16384)           # 24 tiles x 64 stages: stream-K
    assert deep["sk_tiles"] == 24 and deep["dp_tiles"] == 0 and deep["ctas"] == 152
    for m in (1, 32, 256, 1024, 4096):
        p = lib.nvfp4_gemm_plan(m, 4096, 7168)
        assert p["ctas"] >= 1 and p["stages"] >= 2
        if p["swap_ab"]:   # weight rows in 128-row tiles x token columns in tile_n tiles
            tiles = 32 * -(-m // p["tile_n"])
        else:
            tiles = -(-m // p["tile_m"]) * (4096 // p["tile_n"])
        assert p["dp_tiles"] + p["sk_tiles"] == tiles


def test_swap_plans_hold_every_token_in_one_tile(lib):
    """The swap-AB kernels read operand B's scales at scale-factor ID 0 (rows 0..tile_n-1 of a
    128-row scale block), so a swap plan must cover all M tokens with one tile."""
    for m in list(range(1, 40)) + [48, 63, 64, 65, 96, 127, 128, 129, 192, 255, 256]:
        for (n, k) in ((4096, 7168), (7168, 2048), (14336, 4096), (1024, 1024)):
            p = lib.nvfp4_gemm_plan(m, n, k)
            if p["swap_ab"]:
                assert p["tile_n"] >= m, (m, n, k, p)


def test_plan_invariants_over_a_shape_sweep(lib):
    """Every plan the selector makes (152 SMs without a device) is launchable and covers the
    output exactly once: swap-AB plans hold all tokens in one tile and split K at most 8 ways
    over one CTA per split; other plans never split inside a cluster; whole plus stream-K tiles
    are the output tiles; a workspace is needed exactly when tiles are split stream-K; short-K
    whole-tile plans never fall back to stream-K."""
    ms = [1, 2, 16, 17, 31, 32, 33, 64, 65, 100, 128, 129, 200, 256, 257, 300, 512, 1024, 2048, 4096, 6000]
    ns = [256, 512, 1024, 2048, 4096, 7168, 8192, 13056, 14336, 16384, 19456, 28672]
    ks = [256, 512, 768, 1536, 2048, 2304, 4096, 7168, 16384]
    for m in ms:
        for n in ns:
            for k in ks:
                p = lib.nvfp4_gemm_plan(m, n, k)
                ws = lib.gemm_workspace_size(m, n, k)
                where = (m, n, k, p)
                assert p["ctas"] >= 1 and p["stages"] >= 2 and p["tile_n"] in (32, 64, 128, 256), where
                k_steps = -(-k // 256)
                if p["swap_ab"]:
                    assert m <= 256 and p["tile_n"] >= m and p["tile_m"] == 128, where
                    assert 1 <= p["splits"] <= min(8, k_steps), where
                    assert p["dp_tiles"] == -(-n // 128) and p["sk_tiles"] == 0, where
                    assert p["ctas"] == p["dp_tiles"] * p["splits"] and ws == 0, where
                else:
                    assert p["splits"] == 1, where
                    tiles = -(-m // p["tile_m"]) * -(-n // p["tile_n"])
                    assert p["dp_tiles"] + p["sk_tiles"] == tiles, where
                    assert (ws > 0) == (p["sk_tiles"] > 0), where
                    if p["tile_m"] == 256:
                        assert p["tile_n"] == 256 and p["ctas"] % 2 == 0 and p["sk_tiles"] == 0, where
                    if m <= 256 and p["tile_m"] == 128:   # a short-K whole-tile plan
                        assert p["sk_tiles"] == 0 and p["ctas"] == min(tiles, 152), where


def test_workspace_size(lib):
    """Counters (one per split tile, padded to 256 B) + 2 fp32 slots of 128 x tile_n per CTA."""
    assert lib.gemm_workspace_size(1, 4096, 7168) == 0        # cluster split-K needs none
    assert lib.gemm_workspace_size(4096, 4096, 7168) == 0     # whole tiles
    assert lib.gemm_workspace_size(300, 1024, 16384) == 256 + 152 * 2 * 128 * 128 * 4
    assert lib.gemm_workspace_size(2048, 512, 65536) == 256 + 152 * 2 * 128 * 128 * 4
    assert lib.gemm_workspace_size(0, 4096, 7168) == 0


def _c(v):
    return ctypes.c_void_p(v)


def test_gemm_rejects_bad_arguments_without_a_device(lib):
    L = lib.lib
    A, S, D = 0x10000, 0x20000, 0x30000  # never dereferenced: validation fails first
    assert L.nvfp4_gemm(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 32, 1024, 1000, None, 0, 0, None) == 3  # k % 32
    assert L.nvfp4_gemm(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 32, 1000, 1024, None, 0, 0, None) == 3  # n % 32
    assert L.nvfp4_gemm(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), -1, 1024, 1024, None, 0, 0, None) == 1
    assert L.nvfp4_gemm(None, _c(S), _c(A), _c(S), _c(S), _c(D), 32, 1024, 1024, None, 0, 0, None) == 1
    assert L.nvfp4_gemm(_c(A + 16), _c(S), _c(A), _c(S), _c(S), _c(D), 32, 1024, 1024, None, 0, 0, None) == 2
    assert L.nvfp4_gemm(_c(A), _c(S + 8), _c(A), _c(S), _c(S), _c(D), 32, 1024, 1024, None, 0, 0, None) == 2
    assert L.nvfp4_gemm(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 32, 1024, 1024, None, 0, 1 << 20, None) == 1
    assert "k" in lib.last_error() or "flags" in lib.last_error()
    # zero rows: a legal no-op that needs no device
    assert L.nvfp4_gemm(None, None, None, None, None, None, 0, 1024, 1024, None, 0, 0, None) == 0


def test_fused_quantize_gemm_rejects_bad_arguments_without_a_device(lib):
    L = lib.lib
    X, G, B, S, D = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000  # never dereferenced
    q = L.nvfp4_quantize_gemm
    assert q(None, 1024, _c(G), _c(B), _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 1   # x
    assert q(_c(X), 1024, None, _c(B), _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 1   # gs
    assert q(_c(X), 512, _c(G), _c(B), _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 1   # ldx < k
    assert q(_c(X + 8), 1024, _c(G), _c(B), _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 2
    assert q(_c(X), 1028, _c(G), _c(B), _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 2  # ldx % 8
    assert q(_c(X), 1024, _c(G), _c(B), _c(S), _c(G), _c(D), 8, 1024, 1000, None, 0, 0, None) == 3  # k % 32
    assert q(_c(X), 1024, _c(G), None, _c(S), _c(G), _c(D), 8, 1024, 1024, None, 0, 0, None) == 1   # b
    assert q(None, 0, None, None, None, None, None, 0, 1024, 1024, None, 0, 0, None) == 0          # m = 0


def test_quantizers_reject_bad_arguments_without_a_device(lib):
    L = lib.lib
    X, G, Q, S = 0x10000, 0x20000, 0x30000, 0x40000
    assert L.nvfp4_quantize(_c(X), 4, 24, 24, _c(G), _c(Q), _c(S), 0, None) == 3     # k % 16
    assert L.nvfp4_quantize(_c(X), 4, 32, 20, _c(G), _c(Q), _c(S), 0, None) == 2     # ldx < k
    assert L.nvfp4_quantize(_c(X + 2), 4, 32, 32, _c(G), _c(Q), _c(S), 0, None) == 2
    assert L.nvfp4_quantize(None, 4, 32, 32, _c(G), _c(Q), _c(S), 0, None) == 1
    assert L.nvfp4_quantize(None, 0, 32, 32, None, None, None, 0, None) == 0
    assert L.mxfp4_quantize(_c(X), 4, 48, 48, None, 0, _c(Q), _c(S), 1 << 20, 0, None) == 3
    assert L.mxfp4_quantize(_c(X), 4, 64, 64, None, 0, _c(Q), _c(S), 16, 0, None) == 1   # sf too small
    assert L.mxfp4_quantize(_c(X), 4, 64, 64, _c(X), 2000, _c(Q), _c(S), 1 << 30, 0, None) == 1
    assert L.mxfp4_grouped_gemm(_c(X), _c(S), _c(X), 0, _c(X), _c(S), None, _c(Q), 4, 64, 64, 0, None) == 1
    assert L.nvfp4_grouped_gemm(_c(X), _c(S), _c(X), 513, _c(X), _c(S), None, _c(Q), 4, 64, 64, 0, None) == 1
    assert L.sf_swizzle(_c(X), _c(Q), -1, 4, 1, None) == 1
    assert L.sf_swizzle(_c(X), _c(Q), 4, 4, 7, None) == 1


def test_layout_conversion_rejects_bad_arguments_without_a_device(lib):
    L = lib.lib
    S, D = 0x10000, 0x90000
    assert L.nvfp4_sf_convert_layout(_c(S), _c(D), -1, 4, 1, None) == 1
    assert L.nvfp4_sf_convert_layout(_c(S), _c(D), 4, 4, 2, None) == 1          # direction
    assert L.nvfp4_sf_convert_layout(None, _c(D), 4, 4, 1, None) == 1
    assert L.nvfp4_sf_convert_layout(_c(S + 4), _c(D), 4, 4, 1, None) == 2      # alignment
    assert L.nvfp4_sf_convert_layout(_c(S), _c(S + 256), 4, 4, 1, None) == 1    # overlap (512 B)
    assert L.nvfp4_sf_convert_layout(None, None, 0, 4, 1, None) == 0            # empty: no-op
    # the SM103 layout is an NVFP4 layout: the MXFP4 entry points refuse the flag
    X, Q = 0x10000, 0x30000
    assert L.mxfp4_quantize(_c(X), 4, 64, 64, None, 0, _c(Q), _c(S), 1 << 20, lib.FLAG_SF_SM103, None) == 1


def test_moe_sort_workspace_size(lib):
    assert lib.moe_sort_workspace_size(4096, 128) == 128 * 128 * 4      # 32 tokens per CTA
    assert lib.moe_sort_workspace_size(1, 8) == 8 * 4
    assert lib.moe_sort_workspace_size(10 ** 6, 16) == 1024 * 16 * 4    # at most 1024 CTAs
    assert lib.moe_sort_workspace_size(-1, 8) == 0


def test_moe_steps_reject_bad_arguments_without_a_device(lib):
    L = lib.lib
    I, R, P, W, X, O, G, Q, S = (0x10000 * i for i in range(1, 10))   # never dereferenced
    ws = lib.moe_sort_workspace_size(16, 4)
    sort = L.moe_sort_by_expert
    assert sort(_c(I), 16, 33, 4, _c(R), _c(P), _c(P), _c(W), ws, 0, None) == 1      # topk > 32
    assert sort(_c(I), 16, 2, 1025, _c(R), _c(P), _c(P), _c(W), 1 << 30, 0, None) == 1  # experts > 1024
    assert sort(_c(I), (1 << 31) - 511, 1, 4, _c(R), _c(P), _c(P), _c(W), 1 << 30, 0, None) == 1  # slots > 2^31-512
    assert sort(_c(I), 16, 2, 4, _c(R), _c(P), _c(P), _c(W), ws - 1, 0, None) == 1   # workspace too small
    assert "workspace" in lib.last_error()
    assert sort(_c(I), 16, 2, 4, _c(R), _c(P), _c(P), _c(W), ws, 1 << 2, None) == 1  # flags
    assert sort(_c(I), 16, 2, 4, None, _c(P), _c(P), _c(W), ws, 0, None) == 1
    assert sort(_c(I), 16, 2, 4, _c(R + 4), _c(P), _c(P), _c(W), ws, 0, None) == 2   # row_offsets 8-B
    gather = L.moe_gather_rows
    assert gather(_c(X), 16, 60, 64, _c(P), 32, _c(O), 0, None) == 1                  # h % 8
    assert gather(_c(X), 16, 64, 56, _c(P), 32, _c(O), 0, None) == 1                  # ldx < h
    assert gather(_c(X + 8), 16, 64, 64, _c(P), 32, _c(O), 0, None) == 2
    assert gather(None, 16, 64, 64, _c(P), 32, _c(O), 0, None) == 1
    assert gather(None, 0, 64, 64, None, 0, None, 0, None) == 0                        # nothing to gather
    comb = L.moe_combine
    assert comb(_c(X), 32, _c(P), _c(G), 16, 0, 64, _c(O), 0, None) == 1              # topk < 1
    assert comb(_c(X), 32, _c(P), _c(G), 16, 2, 60, _c(O), 0, None) == 1              # h % 8
    assert comb(_c(X), 32, _c(P), _c(G + 2), 16, 2, 64, _c(O), 0, None) == 2
    assert comb(_c(X), 32, None, _c(G), 16, 2, 64, _c(O), 0, None) == 1
    assert comb(None, 0, None, None, 0, 2, 64, None, 0, None) == 0
    sfb = (128 + 128 * 4) * 16                                                         # t=40, E=4, k=256
    for f, k, ldx in ((L.nvfp4_quantize_experts, 256, 256), (L.nvfp4_silu_mul_quantize_experts, 256, 512)):
        assert f(_c(X), 40, 250, ldx, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 3   # k % 16
        assert f(_c(X), 40, k, ldx - 8, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 2  # ldx too short
        assert f(_c(X), 40, k, ldx, _c(R), 0, _c(G), _c(Q), _c(S), sfb, 0, None) == 1     # no experts
        assert f(_c(X), 40, k, ldx, _c(R), 4, _c(G), _c(Q), _c(S), sfb - 1, 0, None) == 1  # sf too small
        assert f(_c(X), 40, k, ldx, _c(R), 4, _c(G), _c(Q + 4), _c(S), sfb, 0, None) == 2  # q 8-B
        assert f(_c(X), 40, k, ldx, None, 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 1
        assert f(None, 0, k, ldx, None, 4, None, None, None, sfb, 0, None) == 0           # no rows
    gq = L.nvfp4_gather_quantize_experts                                               # x: 16 tokens
    assert gq(_c(X), -1, 256, 256, _c(P), 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 1   # tokens < 0
    assert gq(_c(X), 16, 256, 256, None, 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 1    # no src_rows
    assert gq(_c(X), 16, 256, 256, _c(P + 2), 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 2  # src 4-B
    assert gq(_c(X), 16, 250, 256, _c(P), 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 3   # k % 16
    assert gq(_c(X), 16, 256, 248, _c(P), 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb, 0, None) == 2   # ldx < k
    assert gq(_c(X), 16, 256, 256, _c(P), 40, _c(R), 4, _c(G), _c(Q), _c(S), sfb - 1, 0, None) == 1  # sf small
    assert gq(None, 0, 256, 256, None, 0, None, 4, None, None, None, sfb, 0, None) == 0          # no rows


def test_noalloc_gemm_refuses_what_nvfp4_gemm_refuses_without_a_device(lib):
    L = lib.lib
    A, S, D = 0x10000, 0x20000, 0x30000
    g = L.nvfp4_gemm_noalloc
    assert g(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 300, 1024, 16016, 0, None) == 3       # k % 32
    assert g(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 300, 1000, 16384, 0, None) == 3       # n % 32
    assert g(_c(A + 16), _c(S), _c(A), _c(S), _c(S), _c(D), 300, 1024, 16384, 0, None) == 2  # split plan, misaligned a
    assert g(None, _c(S), _c(A), _c(S), _c(S), _c(D), 300, 1024, 16384, 0, None) == 1
    assert g(_c(A), _c(S), _c(A), _c(S), _c(S), _c(D), 300, 1024, 16384, 1 << 20, None) == 1  # flags
    assert g(None, None, None, None, None, None, 0, 1024, 1024, 0, None) == 0
