"""nvfp4_gemm_noalloc: the GEMM with the library's static split-K scratch instead of a caller
workspace.  Two calls in a row must reproduce, bit for bit, nvfp4_gemm with its own workspace
(the split order is fixed), on split and unsplit plans; a call after one that timed out must
start clean.  This file sorts last so that it also runs after every other GPU test."""
import pytest
import torch

from cases import assert_within, dev, nvfp4_operands, reference, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m
    return m


def _args(ops):
    return (dev(ops["qa"]), dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]))


@pytest.mark.parametrize("m,n,k,split", [
    (300, 1024, 16384, True),    # stream-K: partials in the static scratch
    (512, 512, 16384, True),
    (1, 4096, 7168, False),      # cluster split-K: no scratch
    (2048, 4096, 1024, False)])  # whole tiles
def test_two_calls_match_the_workspace_entry_point(nv, m, n, k, split):
    assert (nv.nvfp4_gemm_plan(m, n, k)["sk_tiles"] > 0) == split
    ops = nvfp4_operands(m, n, k, seed=21)
    args = _args(ops)
    ws = nv.gemm_workspace(nv.gemm_workspace_size(m, n, k))
    ref = nv.nvfp4_gemm(*args, workspace=ws)
    d1 = nv.nvfp4_gemm_noalloc(*args)
    d2 = nv.nvfp4_gemm_noalloc(*args)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.equal(d1, ref) and torch.equal(d2, ref)
    if m * n <= 300 * 1024:
        R, tol = reference(ops)
        assert_within(d1, R, tol, f"no-alloc {m}x{n}x{k}")


def test_dirty_counters_leave_split_tiles_unwritten(nv):
    """What the counter clearing guards against, shown on nvfp4_gemm with a caller workspace:
    arrival counters that do not start at zero (as a split call that timed out part way can
    leave them) make no CTA the last of its tile, so the split tiles are never written and the
    counters stay set.  nvfp4_gemm_noalloc clears its counters before every split launch."""
    m, n, k = 512, 512, 16384
    plan = nv.nvfp4_gemm_plan(m, n, k)
    assert plan["sk_tiles"] > 0 and plan["dp_tiles"] == 0
    ops = nvfp4_operands(m, n, k, seed=24)
    args = _args(ops)
    ws = nv.gemm_workspace(nv.gemm_workspace_size(m, n, k))
    counters = ws[:4 * plan["sk_tiles"]].view(torch.int32)
    counters.fill_(1000)                       # no arrival can see n - 1
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(*args, d=d, workspace=ws)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.isnan(d.float()).all()        # no split tile was finished
    assert (counters > 1000).all()             # and the counters are still set
    good = nv.nvfp4_gemm_noalloc(*args)
    torch.cuda.synchronize()
    nv.check_status()
    R, tol = reference(ops)
    assert_within(good, R, tol, "no-alloc beside a dirty workspace")


def test_call_after_a_timeout_starts_clean(nv):
    """A split call that times out (every CTA here gives up at its first stage); the next call
    on the static scratch must give the oracle's result."""
    m, n, k = 512, 512, 16384
    ops = nvfp4_operands(m, n, k, seed=22)
    args = _args(ops)
    nv.check_status()
    nv.nvfp4_gemm_noalloc(*args, flags=nv.FLAG_DEBUG_TIMEOUT | nv.FLAG_DEBUG_SKIP_FIRST_LOAD)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.check_status()
    assert e.value.code == 6
    d = nv.nvfp4_gemm_noalloc(*args)
    torch.cuda.synchronize()
    nv.check_status()
    R, tol = reference(ops)
    assert_within(d, R, tol, "no-alloc after time-out")


def test_refuses_what_nvfp4_gemm_refuses(nv):
    ops = nvfp4_operands(300, 1024, 16384, seed=23)
    a, sfa, b, sfb, al = _args(ops)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_gemm_noalloc(a, sfa, b, sfb, al, flags=1 << 20)
    assert e.value.code == 1
