"""GPU parity of the SM103 scale layout: the layout-conversion kernel against the oracle, the
quantiser writing the SM103 layout (codes unchanged, scales = the converted SM100 scales: the
invariants of test_nvfp4_quant.py "test_scaled_fp4_quant_sm103_matches_sm100" on the vLLM fork
compare view "add pdl"), and the GEMM reading SM103-layout scales (bit-identical output)."""
import numpy as np
import pytest
import torch

import synth
from cases import assert_within, dev, global_scale, nvfp4_operands, reference, scalar
from oracle import layout
from oracle import quant as oquant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m
    return m


@pytest.mark.parametrize("rows,cols", [(1, 1), (5, 3), (128, 4), (130, 9), (256, 448), (1000, 112), (4096, 448)])
def test_conversion_kernel_matches_oracle(nv, rows, cols):
    rp, cp = layout.padded_shape(rows, cols)
    rng = np.random.default_rng(rows + 7 * cols)
    buf = rng.integers(0, 256, size=rp * cp).astype(np.uint8)   # padding bytes non-zero too
    src = dev(buf)
    fwd = nv.sf_convert_layout(src, rows, cols, to_sm103=True)
    torch.cuda.synchronize()
    want = layout.convert_layout(buf, rows, cols, to_sm103=True)
    assert np.array_equal(fwd.cpu().numpy(), want)
    back = nv.sf_convert_layout(fwd, rows, cols, to_sm103=False)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), buf)


@pytest.mark.parametrize("m,k", [(1, 64), (37, 160), (128, 7168), (300, 2048), (1025, 4096)])
def test_quantiser_sm103_layout(nv, m, k):
    x = synth.activation(m + k, m, k)
    gs = global_scale(x)
    xd, gsd = dev(x), scalar(gs)
    q0, sf0 = nv.nvfp4_quantize(xd, gsd)
    q1, sf1 = nv.nvfp4_quantize(xd, gsd, flags=nv.FLAG_SF_SM103)
    torch.cuda.synchronize()
    # codes do not depend on where the scales go
    assert torch.equal(q0, q1)
    # both equal the oracle quantiser (bit-exact) in their own layout
    oq, osf = oquant.nvfp4_quantize(x, gs)
    assert np.array_equal(q0.cpu().numpy(), oq)
    assert np.array_equal(sf0.cpu().numpy(), osf)
    assert np.array_equal(sf1.cpu().numpy(), layout.convert_layout(osf, m, k // 16, to_sm103=True))
    # and the conversion kernel maps the one onto the other
    conv = nv.sf_convert_layout(sf0, m, k // 16, to_sm103=True)
    torch.cuda.synchronize()
    assert torch.equal(conv, sf1)


@pytest.mark.parametrize("m,n,k", [(1, 4096, 7168), (32, 1024, 1024), (100, 256, 2048), (256, 512, 512),
                                   (1000, 2048, 512), (300, 1024, 16384)])
def test_gemm_reads_sm103_scales(nv, m, n, k):
    """Same operands, scales in either layout: identical bf16 output (same arithmetic), within
    the oracle tolerance."""
    ops = nvfp4_operands(m, n, k, seed=3 * m + n)
    sfa103 = layout.convert_layout(ops["sfa"], m, k // 16, to_sm103=True)
    sfb103 = layout.convert_layout(ops["sfb"], n, k // 16, to_sm103=True)
    a, b, al = dev(ops["qa"]), dev(ops["qb"]), scalar(ops["alpha"])
    d0 = nv.nvfp4_gemm(a, dev(ops["sfa"]), b, dev(ops["sfb"]), al)
    d1 = nv.nvfp4_gemm(a, dev(sfa103), b, dev(sfb103), al, flags=nv.FLAG_SF_SM103)
    d2 = nv.nvfp4_gemm(a, dev(sfa103), b, dev(sfb103), al, flags=nv.FLAG_SF_SM103 | nv.FLAG_PDL)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.equal(d0, d1) and torch.equal(d0, d2)
    if m * n * k <= 1 << 31:
        R, tol = reference(ops)
        assert_within(d1, R, tol, f"sm103 {m}x{n}x{k}")
