"""The Python binding's argument checks, on the CPU: every wrapper runs against a stand-in for the
library's compute entry points (the size queries are the real ones), with CPU tensors standing
in for device tensors.  Valid calls -- the argument patterns of the GPU tests and the benchmark
-- reach the library; undersized, mistyped or strided outputs are refused before it."""
import numpy as np
import pytest
import torch


@pytest.fixture()
def nv(monkeypatch):
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m

    real = m._lib
    calls = []

    class FakeLib:
        nvfp4_sf_bytes = real.nvfp4_sf_bytes
        mxfp4_grouped_sf_bytes = real.mxfp4_grouped_sf_bytes
        moe_sort_workspace_size = real.moe_sort_workspace_size

        @staticmethod
        def nvfp4_last_error():
            return b""

        def __getattr__(self, name):
            def entry(*args):
                calls.append(name)
                return 0          # also leaves a queried workspace size at 0
            return entry

    monkeypatch.setattr(m, "_lib", FakeLib())
    monkeypatch.setattr(m, "_check_device", lambda t, name: None)
    monkeypatch.setattr(m, "_stream", lambda s: None)
    m.calls = calls
    return m


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.ones(shape, dtype=torch.float32)


def test_quantize_and_gemm_accept_the_usual_calls(nv):
    m, n, k = 33, 256, 512
    x = bf(m, k)
    q, sf = nv.nvfp4_quantize(x, f32(1))
    assert q.shape == (m, k // 2) and sf.numel() == nv.sf_bytes(m, k)
    nv.nvfp4_quantize(x, f32(1), u8(m, k // 2), u8(nv.sf_bytes(m, k)))             # the benchmark's form
    wb, sfb = u8(n, k // 2), u8(nv.sf_bytes(n, k))
    d = nv.nvfp4_gemm(q, sf, wb, sfb, f32(1))
    nv.nvfp4_gemm(q, sf, wb, sfb, f32(1), bf(m, n), workspace=u8(4096))
    nv.nvfp4_quantize_gemm(x, f32(1), wb, sfb, f32(1), d=d)
    nv.nvfp4_gemm_noalloc(q, sf, wb, sfb, f32(1), d)
    nv.nvfp4_gemm(u8(0, k // 2), sf, wb, sfb, f32(1))                               # no rows
    E = 3
    qe, sfe = u8(E, n, k // 2), u8(E, nv.sf_bytes(n, k, 32))
    for e in range(E):
        nv.mxfp4_quantize(bf(n, k), q=qe[e], sf=sfe[e])
    ro = torch.tensor([0, 10, 10, m], dtype=torch.int64)
    qa, sfa = nv.mxfp4_quantize(x, ro)
    nv.mxfp4_grouped_gemm(qa, sfa, ro, qe, sfe, None, bf(m, n))
    assert nv.calls.count("nvfp4_gemm") == 3 and "mxfp4_grouped_gemm" in nv.calls


def test_undersized_or_wrong_outputs_are_refused(nv):
    m, n, k = 8, 256, 512
    x = bf(m, k)
    q, sf = nv.nvfp4_quantize(x, f32(1))
    wb, sfb = u8(n, k // 2), u8(nv.sf_bytes(n, k))
    with pytest.raises(ValueError, match="q has"):
        nv.nvfp4_quantize(x, f32(1), q=u8(m, k // 2 - 1))
    with pytest.raises(ValueError, match="sf has"):
        nv.nvfp4_quantize(x, f32(1), sf=u8(nv.sf_bytes(m, k) - 1))
    with pytest.raises(ValueError, match="d has"):
        nv.nvfp4_gemm(q, sf, wb, sfb, f32(1), d=bf(m, n - 1))
    with pytest.raises(ValueError, match="contiguous"):
        nv.nvfp4_gemm(q, sf, wb, sfb, f32(1), d=bf(n, m).t())
    with pytest.raises(TypeError):
        nv.nvfp4_gemm(q, sf, wb, sfb, f32(1), d=torch.zeros((m, n), dtype=torch.float16))
    with pytest.raises(ValueError, match="d has"):
        nv.nvfp4_quantize_gemm(x, f32(1), wb, sfb, f32(1), d=bf(m - 1, n))
    E = 2
    ro = torch.tensor([0, 3, m], dtype=torch.int64)
    qa, sfa = nv.mxfp4_quantize(x, ro)
    with pytest.raises(ValueError, match="sfb has"):
        nv.mxfp4_grouped_gemm(qa, sfa, ro, u8(E, n, k // 2), u8(E, nv.sf_bytes(n, k, 32) - 1))
    with pytest.raises(ValueError, match="sfb has"):
        nv.nvfp4_grouped_gemm(qa, sfa, ro, u8(E, n, k // 2), u8(E * nv.sf_bytes(n, k, 16) - 1), f32(E))
    assert "nvfp4_gemm" not in nv.calls and "mxfp4_grouped_gemm" not in nv.calls


def test_layout_calls(nv):
    rows, cols = 300, 37
    pad = 384 * 40
    sw = nv.sf_swizzle(u8(rows, cols), rows, cols, True)
    assert sw.numel() == pad
    back = nv.sf_swizzle(sw, rows, cols, False)
    assert back.numel() == rows * cols
    with pytest.raises(ValueError, match="src has"):
        nv.sf_swizzle(u8(pad - 1), rows, cols, False)
    with pytest.raises(ValueError, match="dst has"):
        nv.sf_swizzle(u8(rows, cols), rows, cols, True, dst=u8(pad - 1))
    conv = nv.sf_convert_layout(sw, rows, cols, to_sm103=True)
    nv.sf_convert_layout(sw, rows, cols, to_sm103=False, dst=torch.empty_like(conv))
    with pytest.raises(ValueError, match="dst has"):
        nv.sf_convert_layout(sw, rows, cols, dst=u8(pad - 512))


def test_moe_steps(nv):
    T, E, topk, H, I = 16, 4, 2, 64, 32
    R = T * topk
    ids = torch.zeros((T, topk), dtype=torch.int32)
    ro, src, pos = nv.moe_sort_by_expert(ids, E)
    nv.moe_sort_by_expert(ids.t().contiguous().t(), E, out=(ro, src, pos))              # strided ids: copied
    xg = nv.moe_gather_rows(bf(T, H), src)
    nv.moe_gather_rows(bf(T, H), src, out=bf(R, H))
    gs = f32(E)
    q1, s1 = nv.nvfp4_quantize_experts(xg, ro, gs)
    nv.nvfp4_quantize_experts(xg, ro, gs, q=u8(R, H // 2), sf=u8(nv.expert_sf_bytes(R, E, H)))
    qg, sg = nv.nvfp4_gather_quantize_experts(bf(T, H), src, ro, gs)
    assert qg.shape == (R, H // 2) and sg.numel() == nv.expert_sf_bytes(R, E, H)
    nv.nvfp4_gather_quantize_experts(bf(T, H), src, ro, gs, q=u8(R, H // 2), sf=u8(nv.expert_sf_bytes(R, E, H)))
    qw, sfw = u8(E, 2 * I, H // 2), u8(E, nv.sf_bytes(2 * I, H, 16))
    h1 = nv.nvfp4_grouped_gemm(q1, s1, ro, qw, sfw, f32(E))
    q2, s2 = nv.nvfp4_silu_mul_quantize_experts(h1, ro, gs)
    assert q2.shape == (R, I // 2)
    y = nv.nvfp4_grouped_gemm(q2, s2, ro, u8(E, H, I // 2), u8(E, nv.sf_bytes(H, I, 16)), f32(E), d=bf(R, H))
    out = nv.moe_combine(y, pos, f32(T, topk))
    assert out.shape == (T, H)
    with pytest.raises(ValueError, match="out has"):
        nv.moe_gather_rows(bf(T, H), src, out=bf(R - 1, H))
    with pytest.raises(ValueError, match="weights must have shape"):
        nv.moe_combine(y, pos, f32(T, topk + 1))
    with pytest.raises(ValueError, match="gs has"):
        nv.nvfp4_quantize_experts(xg, ro, f32(E - 1))
    with pytest.raises(ValueError, match="q has"):
        nv.nvfp4_gather_quantize_experts(bf(T, H), src, ro, gs, q=u8(R - 1, H // 2))
    with pytest.raises(TypeError, match="src_rows"):
        nv.nvfp4_gather_quantize_experts(bf(T, H), src.long(), ro, gs)
    with pytest.raises(ValueError, match="pos has"):
        nv.moe_sort_by_expert(ids, E, out=(ro, src, torch.zeros(R - 1, dtype=torch.int32)))
    assert nv.calls.count("moe_combine") == 1


def test_device_check_names_the_tensor(monkeypatch):
    import nvfp4_block_scaled_bf16_gb300 as m
    with pytest.raises(TypeError, match="x must be a CUDA tensor"):
        m._check_device(np.zeros(3), "x")
    with pytest.raises(TypeError, match="q must be a CUDA tensor"):
        m._check_device(torch.zeros(3), "q")
