"""GPU parity of the quantisers and the scale swizzle: bit-exact against the CPU oracle."""
import numpy as np
import pytest
import torch

import synth
from cases import dev, global_scale, scalar
from oracle import formats, layout
from oracle import quant as oquant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m
    return m


def _check_nvfp4(nv, x: torch.Tensor, gs, flags=0, ldx_pad=0):
    m, k = x.shape
    xd = x.cuda()
    if ldx_pad:
        big = torch.zeros((m, k + ldx_pad), dtype=torch.bfloat16, device="cuda")
        big[:, :k] = xd
        xd = big[:, :k]
    q, sf = nv.nvfp4_quantize(xd, scalar(gs), flags=flags)
    torch.cuda.synchronize()
    q_ref, sf_ref = oquant.nvfp4_quantize(x, gs)
    qg, sg = q.cpu().numpy(), sf.cpu().numpy()
    assert sg.size == sf_ref.size
    bad_q = np.argwhere(qg != q_ref)
    assert bad_q.size == 0, f"{len(bad_q)} data bytes differ, first at {bad_q[:3].tolist()}"
    bad_s = np.nonzero(sg != sf_ref)[0]
    assert bad_s.size == 0, f"{bad_s.size} scale bytes differ, first at {bad_s[:3].tolist()}"
    return q, sf


@pytest.mark.parametrize("m,k,pad", [(32, 1024, 0), (1, 7168, 0), (3, 96, 0), (130, 4096, 64),
                                     (256, 7168, 0), (512, 4096, 0), (1, 16, 0), (200, 48, 8)])
def test_nvfp4_quantize_matches_oracle(nv, m, k, pad):
    x = synth.activation(m + k, m, k)
    _check_nvfp4(nv, x, global_scale(x), ldx_pad=pad)


def test_nvfp4_quantize_other_global_scales(nv):
    x = synth.activation(11, 64, 512)
    for gs in (np.float32(1.0), np.float32(0.37), np.float32(3.0e4), global_scale(x) * np.float32(7.0)):
        _check_nvfp4(nv, x, gs)


def test_nvfp4_e2m1_rounding_exhaustive_bf16(nv):
    """gs = 1 and a block amax of 6 give scale 1.0 and inv = 1, so each data code is the e2m1
    rounding of the bf16 input itself: every bf16 value of magnitude < 8, both signs."""
    bits = np.arange(0, 0x8000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.abs(vals) < 8.0]
    vals = np.concatenate([vals, -vals])
    nblk = -(-len(vals) // 15)
    nblk += (-nblk) % 4                       # whole 64-element rows
    flat = np.zeros(nblk * 15, dtype=np.float32)
    flat[:len(vals)] = vals
    x = np.zeros((nblk, 16), dtype=np.float32)
    x[:, 0] = 6.0
    x[:, 1:] = flat.reshape(nblk, 15)
    x = x.reshape(nblk // 4, 64)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xt.float().numpy(), x)
    _check_nvfp4(nv, xt, np.float32(1.0))


def test_nvfp4_e4m3_scale_rounding_exhaustive_bf16(nv):
    """gs = 6: the scale of a block with amax a is e4m3(a) (6a/6 is exact), for every
    non-negative finite bf16 a."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    a = (bits << 16).view(np.float32)
    n = len(a)
    rows = -(-n // 4)
    x = np.zeros((rows * 4, 16), dtype=np.float32)
    x[:n, 0] = a
    x[:n, 5] = -a * 0.5
    xt = torch.from_numpy(x.reshape(rows, 64)).to(torch.bfloat16)
    _check_nvfp4(nv, xt, np.float32(6.0))


def test_nvfp4_sign_of_zero_and_zero_blocks(nv):
    x = np.zeros((4, 32), dtype=np.float32)
    x[0, :16] = -0.0
    x[1, 0] = 6.0
    x[1, 1:8] = [-0.1, -0.25, 0.25, -0.0, 0.0, 1e-30, -1e-30]
    x[2, 16:] = 1.0
    xt = torch.from_numpy(x).to(torch.bfloat16)
    q, _ = _check_nvfp4(nv, xt, np.float32(1.0))


def test_nvfp4_pdl_flag_is_bitwise_identical(nv):
    x = synth.activation(5, 256, 4096)
    gs = global_scale(x)
    q0, s0 = _check_nvfp4(nv, x, gs, flags=0)
    q1, s1 = _check_nvfp4(nv, x, gs, flags=nv.FLAG_PDL)
    assert torch.equal(q0, q1) and torch.equal(s0, s1)


def test_nvfp4_zero_rows_is_a_no_op(nv):
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q, sf = nv.nvfp4_quantize(x, scalar(1.0))
    assert q.numel() == 0 and sf.numel() == 0


@pytest.mark.parametrize("t,k", [(1, 32), (33, 2048), (300, 768), (128, 96)])
def test_mxfp4_quantize_dense_matches_oracle(nv, t, k):
    x = synth.activation(t * 3 + k, t, k)
    q, sf = nv.mxfp4_quantize(x.cuda())
    torch.cuda.synchronize()
    q_ref, sf_ref = oquant.mxfp4_quantize(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy()[:sf_ref.size], sf_ref)


def test_mxfp4_quantize_grouped_matches_oracle(nv):
    counts = torch.tensor([0, 1, 127, 128, 129, 0, 300, 5], dtype=torch.int64)
    ro = synth.moe_offsets(counts)
    t, k = int(ro[-1]), 256
    x = synth.activation(21, t, k)
    q, sf = nv.mxfp4_quantize(x.cuda(), row_offsets=ro.cuda())
    torch.cuda.synchronize()
    q_ref, sf_ref = oquant.mxfp4_quantize(x, ro.numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy()[:sf_ref.size], sf_ref)


def test_mxfp4_scale_rounding_exhaustive_bf16(nv):
    """Every non-negative finite bf16 amax: the ue8m0 code is the round-up of amax/6."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    a = (bits << 16).view(np.float32)
    rows = -(-len(a) // 2)
    x = np.zeros((rows * 2, 32), dtype=np.float32)
    x[:len(a), 3] = a
    xt = torch.from_numpy(x.reshape(rows, 64)).to(torch.bfloat16)
    q, sf = nv.mxfp4_quantize(xt.cuda())
    torch.cuda.synchronize()
    q_ref, sf_ref = oquant.mxfp4_quantize(xt)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (128, 4), (300, 37), (4096, 448)])
def test_sf_swizzle_matches_oracle(nv, rows, cols):
    mat = synth.random_bytes(rows * 7 + cols, rows * cols).view(rows, cols)
    sw = nv.sf_swizzle(mat.cuda(), rows, cols, True)
    torch.cuda.synchronize()
    want = layout.swizzle(mat.numpy())
    assert np.array_equal(sw.cpu().numpy(), want)
    back = nv.sf_swizzle(sw, rows, cols, False)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy().reshape(rows, cols), mat.numpy())
