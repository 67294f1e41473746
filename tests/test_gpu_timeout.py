"""The bounded pipeline waits on the GPU: a GEMM whose first K stage is never loaded (test
hook flag) gives up its wait after the short debug limit, reports NVFP4_ERR_TIMEOUT through
nvfp4_check_status, frees its resources, and leaves the context usable for the next call."""
import numpy as np
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


@pytest.mark.parametrize("m,n,k", [(8, 1024, 2048), (512, 512, 1024), (512, 512, 16384)])
def test_wait_times_out_and_context_survives(nv, m, n, k):
    ops = nvfp4_operands(m, n, k, 4)
    args = (dev(ops["qa"]), dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]))
    nv.check_status()                                    # start from a clean status word
    # a timed-out call may leave split-tile counters set: it gets a workspace of its own
    ws = nv.gemm_workspace(nv.gemm_workspace_size(m, n, k))
    nv.nvfp4_gemm(*args, flags=nv.FLAG_DEBUG_TIMEOUT | nv.FLAG_DEBUG_SKIP_FIRST_LOAD, workspace=ws)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.check_status()
    assert e.value.code == 6                             # NVFP4_ERR_TIMEOUT
    nv.check_status()                                    # the word was cleared
    d = nv.nvfp4_gemm(*args)                             # the next call works normally
    torch.cuda.synchronize()
    nv.check_status()
    R, tol = reference(ops)
    assert_within(d, R, tol, "after time-out")


def test_skip_hook_needs_the_debug_timeout(nv):
    """Without the short limit the hook is ignored (a 10 s stall is never what a caller wants)."""
    ops = nvfp4_operands(8, 256, 512, 5)
    d = nv.nvfp4_gemm(dev(ops["qa"]), dev(ops["sfa"]), dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"]),
                      flags=nv.FLAG_DEBUG_SKIP_FIRST_LOAD)
    torch.cuda.synchronize()
    nv.check_status()
    R, tol = reference(ops)
    assert_within(d, R, tol, "hook ignored")
