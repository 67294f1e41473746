"""GPU parity of the NVFP4 GEMM against the fp64 oracle, within
|D - R| <= ulp_bf16(|R|) + 1e-5 * sum_k |alpha a b| per element."""
import numpy as np
import pytest
import torch

import synth
from cases import assert_within, dev, global_scale, nvfp4_operands, reference, scalar
from oracle import gemm as ogemm
from oracle import layout
from oracle import quant as oquant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m
    return m


def _run(nv, ops, flags=0):
    d = nv.nvfp4_gemm(dev(ops["qa"]), dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]),
                      flags=flags)
    torch.cuda.synchronize()
    nv.check_status()
    return d


def test_pr1_config(nv):
    """M=32, N=1024, K=1024, seed 0: A ~ N(0,1), B ~ N(0,0.02), oracle-quantised."""
    ops = nvfp4_operands(32, 1024, 1024, 0, outliers=False)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, "PR1")


@pytest.mark.parametrize("m,n,k", [
    (1, 32, 32), (3, 64, 96), (7, 96, 160), (16, 256, 256), (17, 128, 320), (33, 160, 544),
    (64, 512, 1024), (65, 384, 768), (100, 256, 2048), (128, 128, 256), (129, 256, 512),
    (200, 320, 1056), (256, 512, 512), (257, 256, 512), (300, 1024, 1024), (512, 768, 1536),
    (1000, 2048, 512), (640, 4096, 256)])
def test_shapes_and_ragged_tails(nv, m, n, k):
    ops = nvfp4_operands(m, n, k, seed=m + n + k)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"{m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [
    (300, 1024, 16384),   # 24 tiles x 64 K stages over 152 CTAs: up to 8 contributors per tile
    (1100, 256, 16384),   # BN=128, 18 tiles x 64 stages: tails of 76 rows in the last row block
    (512, 512, 16384),    # 16 tiles x 64 stages
    (2048, 512, 8224)])   # 64 tiles of 128x128, K tail of 32 (a short last stage)
def test_stream_k_splits(nv, m, n, k):
    """Shapes whose plan splits tiles stream-K (few tiles, long K), including ragged rows and a
    K tail; every output element checked."""
    p = nv.nvfp4_gemm_plan(m, n, k)
    assert p["sk_tiles"] > 0
    ops = nvfp4_operands(m, n, k, seed=11)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"stream-K {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [
    (300, 13056, 512),    # 2 row tiles: the second CTA of each last-row pair is past M (stores nothing)
    (520, 9984, 544),     # 8 valid rows in the last pair tile, K tail of 32 (a short last stage)
    (2304, 4096, 1024),   # 144 tiles over 76 pairs: accumulators handed back across CTAs
    (264, 14336, 1280),   # 2 K steps per stage, the last stage holding one (its second is zero-filled)
    (160, 12288, 768),    # fewer than 256 rows on pairs (M > 128 with many tiles), a half last stage
    (1024, 4096, 2560)])  # 64 tiles: one per pair, 5 two-step stages
def test_cta_pair_tiles(nv, m, n, k):
    """256 x 256 tiles computed by CTA pairs (cta_group::2): every output element checked."""
    p = nv.nvfp4_gemm_plan(m, n, k)
    assert p["tile_m"] == 256 and p["tile_n"] == 256 and p["ctas"] % 2 == 0
    ops = nvfp4_operands(m, n, k, seed=m + k)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"pair {m}x{n}x{k}")


def test_workspace_contract(nv):
    """An explicit workspace works, comes back all zero, gives bit-identical output on reuse;
    a short or missing workspace is refused before anything is launched."""
    m, n, k = 512, 512, 16384
    ops = nvfp4_operands(m, n, k, 0)
    args = (dev(ops["qa"]), dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]))
    need = nv.gemm_workspace_size(m, n, k)
    assert need > 0
    ws = nv.gemm_workspace(need)
    d0 = nv.nvfp4_gemm(*args, workspace=ws)
    d1 = nv.nvfp4_gemm(*args, workspace=ws)
    torch.cuda.synchronize()
    nv.check_status()
    assert int(torch.count_nonzero(ws[:256])) == 0          # arrival counters reset
    assert torch.equal(d0, d1)
    R, tol = reference(ops)
    assert_within(d0, R, tol, "explicit workspace")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_gemm(*args, workspace=ws[: need - 1])
    assert e.value.code == 1 and "workspace" in str(e.value)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_gemm(*args, workspace=ws[1:])
    assert e.value.code in (1, 2)
    L = nv.lib
    import ctypes
    c = lambda t: ctypes.c_void_p(t.data_ptr())
    d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    assert L.nvfp4_gemm(c(args[0]), c(args[1]), c(args[2]), c(args[3]), c(args[4]), c(d), m, n, k, None, 0, 0,
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 1


@pytest.mark.parametrize("m", [1, 4, 8, 16, 32, 64, 128, 256])
def test_decode_sweep_full_size(nv, m):
    """N=4096, K=7168 with 0.1% outlier channels, every output element checked."""
    ops = nvfp4_operands(m, 4096, 7168, 0)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"decode M={m}")


def test_prefill_4096_every_element(nv):
    """4096 x 4096 x 7168 (CTA pairs, 256 tiles over 76 pairs, 14 two-step stages per tile), every
    output element against the fp64 oracle."""
    m, n, k = 4096, 4096, 7168
    assert nv.nvfp4_gemm_plan(m, n, k)["tile_m"] == 256
    ops = nvfp4_operands(m, n, k, 0)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"prefill {m}x{n}x{k}, all elements")


@pytest.mark.parametrize("m,n,k", [(1024, 4096, 7168), (2048, 4096, 7168), (4096, 4096, 7168), (4096, 4096, 4096),
                                   (128, 7168, 2048)])
def test_prefill_sampled_rows(nv, m, n, k):
    """The five prefill shapes at full size (M >= 1024 run on CTA pairs), checked on whole
    128-row blocks at both ends plus seeded rows."""
    ops = nvfp4_operands(m, n, k, 0)
    d = _run(nv, ops)
    rng = np.random.default_rng(m + n + k)
    rows = np.unique(np.concatenate([np.arange(0, min(128, m)), np.arange(max(0, m - 128), m),
                                     rng.integers(0, m, 64)]))
    R, tol = reference(ops, rows)
    assert_within(d[torch.from_numpy(rows).cuda()], R, tol, f"prefill {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(17, 4096, 2048), (256, 4096, 1536), (200, 7168, 4096)])
def test_short_k_tiles_every_element(nv, m, n, k):
    """Short K at N >= 4096 takes 128 x 128 tiles over the whole K rather than split-K (from 17
    tokens on at K <= 2048, from 129 at K <= 4096); every element against the fp64 oracle (ragged
    token tiles, a K of 6 steps)."""
    p = nv.nvfp4_gemm_plan(m, n, k)
    assert p["swap_ab"] == 0 and p["splits"] == 1
    ops = nvfp4_operands(m, n, k, 5)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, f"short K {m}x{n}x{k}")


def test_one_hot_probes(nv):
    """A single nonzero FP4 element of A (value 3, block scale 2) against an all-ones B with
    unit scales: exactly one output row is 6, the rest 0.  Sweeps nibble parity, block index
    and row position inside the 128-row scale tile."""
    m, n, k = 160, 64, 512
    qb = np.full((n, k // 2), 0x22, dtype=np.uint8)
    sfb = layout.swizzle(np.full((n, k // 16), 0x38, dtype=np.uint8))
    for (r, kk) in [(0, 0), (1, 1), (31, 17), (32, 64), (63, 255), (95, 256), (127, 300), (128, 511), (159, 130)]:
        qa = np.zeros((m, k // 2), dtype=np.uint8)
        qa[r, kk // 2] = 0x5 if kk % 2 == 0 else 0x50
        sca = np.full((m, k // 16), 0x38, dtype=np.uint8)
        sca[r, kk // 16] = 0x40
        d = nv.nvfp4_gemm(dev(qa), dev(layout.swizzle(sca)), dev(qb), dev(sfb), scalar(1.0))
        torch.cuda.synchronize()
        got = d.float().cpu().numpy()
        want = np.zeros((m, n), dtype=np.float32)
        want[r, :] = 6.0
        assert np.array_equal(got, want), (r, kk, np.argwhere(got != want)[:4].tolist())


def test_random_codes_and_scales(nv):
    """Uniformly random data nibbles and random finite e4m3 scales (no quantiser involved)."""
    m, n, k = 96, 256, 1024
    rng = np.random.default_rng(7)
    qa = rng.integers(0, 256, (m, k // 2)).astype(np.uint8)
    qb = rng.integers(0, 256, (n, k // 2)).astype(np.uint8)
    sca = rng.integers(0x20, 0x48, (m, k // 16)).astype(np.uint8)
    scb = rng.integers(0x20, 0x48, (n, k // 16)).astype(np.uint8)
    ops = dict(qa=qa, sfa=layout.swizzle(sca), qb=qb, sfb=layout.swizzle(scb), alpha=np.float32(0.125), m=m, n=n, k=k)
    d = _run(nv, ops)
    R, tol = reference(ops)
    assert_within(d, R, tol, "random codes")


def test_pdl_and_determinism(nv):
    for (m, n, k) in [(8, 4096, 7168), (512, 1024, 2048)]:
        ops = nvfp4_operands(m, n, k, 3)
        d0 = _run(nv, ops)
        d1 = _run(nv, ops, flags=nv.FLAG_PDL)
        d2 = _run(nv, ops)
        assert torch.equal(d0, d1) and torch.equal(d0, d2)


@pytest.mark.parametrize("m", [256, 512])
def test_quant_then_gemm_chain_with_pdl(nv, m):
    """Device quantisation of the activation feeds the GEMM on the same stream with PDL, at the
    end-to-end shapes (M=512 runs on CTA pairs)."""
    n, k = 14336, 4096
    ops = nvfp4_operands(m, n, k, 0)
    xa = ops["xa"].cuda()
    qa, sfa = nv.nvfp4_quantize(xa, scalar(ops["gsa"]), flags=nv.FLAG_PDL)
    d = nv.nvfp4_gemm(qa, sfa, dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]), flags=nv.FLAG_PDL)
    torch.cuda.synchronize()
    nv.check_status()
    assert np.array_equal(qa.cpu().numpy(), ops["qa"]) and np.array_equal(sfa.cpu().numpy(), ops["sfa"])
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(m - 136, m),
                                     np.random.default_rng(m).integers(0, m, 32)]))
    R, tol = reference(ops, rows)
    assert_within(d[torch.from_numpy(rows).cuda()], R, tol, f"e2e M={m}")


def test_zero_rows_and_output_stride_contract(nv):
    ops = nvfp4_operands(4, 64, 64, 1)
    a = torch.zeros((0, 32), dtype=torch.uint8, device="cuda")
    d = nv.nvfp4_gemm(a, dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(1.0))
    assert d.shape == (0, 64)
