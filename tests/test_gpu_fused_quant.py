"""GPU parity of nvfp4_quantize_gemm (the activation quantised inside the GEMM): bit-identical to
nvfp4_quantize followed by nvfp4_gemm on the same inputs, and within the GEMM tolerance of the
oracle's quantise-then-GEMM on whole outputs; strided rows, the SM103 scale layout, PDL, the
refused shapes."""
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


def _two_kernels(nv, x, gs, qb, sfb, alpha, flags=0):
    q, sf = nv.nvfp4_quantize(x, gs, flags=flags)
    d = nv.nvfp4_gemm(q, sf, qb, sfb, alpha, flags=flags)
    return q, sf, d


# resident slices (m <= 64 at K = 7168), the ring (m = 128, 256), ragged token tiles, a K tail
@pytest.mark.parametrize("m,n,k", [(1, 4096, 7168), (5, 256, 544), (32, 1024, 1024), (33, 512, 768),
                                   (64, 4096, 7168), (100, 384, 2048), (128, 4096, 7168), (200, 1024, 512),
                                   (256, 4096, 7168)])
def test_bit_identical_to_quantize_then_gemm(nv, m, n, k):
    ops = nvfp4_operands(m, n, k, seed=m + n)
    x = ops["xa"].cuda()
    gs = scalar(ops["gsa"])
    qb, sfb, alpha = dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"])
    d = nv.nvfp4_quantize_gemm(x, gs, qb, sfb, alpha)
    _, _, ref = _two_kernels(nv, x, gs, qb, sfb, alpha)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.equal(d, ref)


@pytest.mark.parametrize("m,n,k", [(1, 512, 1024), (17, 768, 544), (64, 256, 2048), (129, 512, 512)])
def test_within_oracle_tolerance(nv, m, n, k):
    """Against the oracle's quantisation and fp64 GEMM, every element."""
    ops = nvfp4_operands(m, n, k, seed=3 * m + k)
    d = nv.nvfp4_quantize_gemm(ops["xa"].cuda(), scalar(ops["gsa"]), dev(ops["qb"]), dev(ops["sfb"]),
                               scalar(ops["alpha"]))
    torch.cuda.synchronize()
    nv.check_status()
    R, tol = reference(ops)
    assert_within(d, R, tol, f"fused {m}x{n}x{k}")


def test_strided_rows_pdl_and_sm103_scales(nv):
    m, n, k = 24, 1024, 2048
    ops = nvfp4_operands(m, n, k, seed=9)
    big = torch.zeros((m, k + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :k] = ops["xa"].cuda()
    x = big[:, :k]                       # row stride k + 64 elements
    gs = scalar(ops["gsa"])
    qb, sfb, alpha = dev(ops["qb"]), dev(ops["sfb"]), scalar(ops["alpha"])
    ref = _two_kernels(nv, x.contiguous(), gs, qb, sfb, alpha)[2]
    d = nv.nvfp4_quantize_gemm(x, gs, qb, sfb, alpha, flags=nv.FLAG_PDL)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.equal(d, ref)
    # weight scales in the SM103 layout: the kernel writes the activation's scales in it too
    sfb103 = torch.empty_like(sfb)
    nv.sf_convert_layout(sfb, n, k // 16, to_sm103=True, dst=sfb103)
    ref103 = _two_kernels(nv, x.contiguous(), gs, qb, sfb103, alpha, flags=nv.FLAG_SF_SM103)[2]
    d103 = nv.nvfp4_quantize_gemm(x, gs, qb, sfb103, alpha, flags=nv.FLAG_SF_SM103)
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.equal(d103, ref103) and torch.equal(d103, ref)


def test_refused_shapes_and_empty(nv):
    ops = nvfp4_operands(257, 256, 256, seed=1)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize_gemm(ops["xa"].cuda(), scalar(ops["gsa"]), dev(ops["qb"]), dev(ops["sfb"]),
                               scalar(ops["alpha"]))
    assert e.value.code == 3 and "m <= 256" in str(e.value)
    x0 = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    d0 = nv.nvfp4_quantize_gemm(x0, scalar(1.0), dev(ops["qb"]), dev(ops["sfb"]), scalar(1.0))
    assert d0.shape == (0, 256)
