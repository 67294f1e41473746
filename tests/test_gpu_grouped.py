"""GPU parity of the MXFP4 grouped (MoE) GEMM against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from cases import assert_within, dev, scalar
from oracle import gemm as ogemm
from oracle import quant as oquant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as m
    return m


def _weights(seed, E, n, k):
    xb = synth.weight(seed, n, k, experts=E)
    qb = np.empty((E, n, k // 2), dtype=np.uint8)
    sfb = []
    for e in range(E):
        q, s = oquant.mxfp4_quantize(xb[e])
        qb[e] = q
        sfb.append(s)
    return qb, np.stack(sfb)


def _check(nv, counts, n, k, seed=0, alpha=None, experts_to_check=None):
    counts = torch.as_tensor(counts, dtype=torch.int64)
    E = counts.numel()
    ro = synth.moe_offsets(counts)
    t = int(ro[-1])
    xa = synth.activation(seed, t, k)
    qa, sfa = oquant.mxfp4_quantize(xa, ro.numpy())
    qb, sfb = _weights(seed, E, n, k)
    sfa_d = torch.zeros(nv.grouped_sf_bytes(t, E, k), dtype=torch.uint8, device="cuda")
    sfa_d[:sfa.size] = dev(sfa)
    d = nv.mxfp4_grouped_gemm(dev(qa), sfa_d, ro.cuda(), dev(qb), dev(sfb),
                              None if alpha is None else scalar(alpha))
    torch.cuda.synchronize()
    nv.check_status()
    out = ogemm.mxfp4_grouped_gemm(qa, sfa, ro.numpy(), qb, sfb, alpha, n, k, experts_to_check)
    for e, (Ae, Be, Re) in out.items():
        r0, r1 = int(ro[e]), int(ro[e + 1])
        if r1 == r0:
            continue
        tol = ogemm.tolerance(Re, ogemm.abs_product_sum(Ae, Be, 1.0 if alpha is None else alpha))
        assert_within(d[r0:r1], Re, tol, f"expert {e}")
    return d


def test_small_groups_with_empty_experts(nv):
    _check(nv, [3, 0, 130, 1, 0, 256, 129], 256, 512)


def test_alpha_and_k_tail(nv):
    _check(nv, [5, 200, 64], 128, 96 * 2, alpha=0.25)


def test_ragged_n_tiles(nv):
    """N = 288: each expert's 256-wide column tile and a 32-wide one (B rows past the expert's
    last belong to the next expert, their columns are not stored)."""
    _check(nv, [40, 0, 170, 7], 288, 256)


def test_largest_expert_count(nv):
    """1024 experts (the MXFP4 grouped GEMM's limit), most with 0..3 rows."""
    counts = np.random.default_rng(4).integers(0, 4, 1024).tolist()
    _check(nv, counts, 64, 64, seed=3)


def test_moe_gate_up_sampled_experts(nv):
    """E=128 experts, 4096 tokens top-8 (32768 rows), gate+up N=1536, K=2048; the oracle checks
    the smallest and largest experts and six seeded others."""
    counts = synth.moe_routing(0, 4096, 128, 8)
    order = torch.argsort(counts)
    rng = np.random.default_rng(0)
    pick = sorted(set([int(order[0]), int(order[-1])] + [int(v) for v in rng.integers(0, 128, 6)]))
    _check(nv, counts, 1536, 2048, experts_to_check=pick)


def test_moe_down_sampled_experts(nv):
    """The down projection of the same layer: 128 experts, 32768 rows, N=2048, K=768 (three K
    stages); the smallest and largest experts and six seeded others."""
    counts = synth.moe_routing(0, 4096, 128, 8)
    order = torch.argsort(counts)
    rng = np.random.default_rng(1)
    pick = sorted(set([int(order[0]), int(order[-1])] + [int(v) for v in rng.integers(0, 128, 6)]))
    _check(nv, counts, 2048, 768, seed=2, experts_to_check=pick)


def test_malformed_row_offsets_are_rejected_on_device(nv):
    """Offsets that do not end at the row count (or decrease) make the kernel do no work and
    nvfp4_check_status report NVFP4_ERR_INVALID_ARG; the output is left untouched."""
    E, n, k, t = 3, 128, 256, 64
    qa = torch.zeros((t, k // 2), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(nv.grouped_sf_bytes(t, E, k), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((E, n, k // 2), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros((E, nv.sf_bytes(n, k, 32)), dtype=torch.uint8, device="cuda")
    for bad in ([0, 10, 5, 64], [0, 10, 20, 60], [3, 10, 20, 64]):
        d = torch.full((t, n), 7.0, dtype=torch.bfloat16, device="cuda")
        nv.check_status()
        nv.mxfp4_grouped_gemm(qa, sfa, torch.tensor(bad, device="cuda"), qb, sfb, None, d)
        with pytest.raises(nv.NVFP4Error) as e:
            nv.check_status()
        assert e.value.code == 1
        assert bool((d == 7.0).all())
