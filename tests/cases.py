"""Shared test inputs: seeded synthetic operands quantised by the oracle, and the comparison
helpers the GPU parity tests use.  Nothing here calls the CUDA library."""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth
from oracle import gemm as ogemm
from oracle import quant as oquant

F32 = np.float32


def global_scale(x: torch.Tensor) -> np.float32:
    """gs = 448 * 6 / amax(x) in fp32 (FLOAT8_E4M3_MAX * FLOAT4_E2M1_MAX / amax)."""
    amax = F32(x.float().abs().max().item())
    return F32(2688.0) / amax


@functools.lru_cache(maxsize=4)
def _nvfp4_weight(n: int, k: int, seed: int):
    """B: weight [n,k] N(0,0.02) quantised by the oracle (shared by every M of a shape sweep;
    callers treat the arrays as read-only)."""
    xb = synth.weight(seed, n, k)
    gsb = global_scale(xb)
    qb, sfb = oquant.nvfp4_quantize(xb, gsb)
    return xb, gsb, qb, sfb


@functools.lru_cache(maxsize=16)
def nvfp4_operands(m: int, n: int, k: int, seed: int = 0, outliers: bool = True):
    """A: activation [m,k] N(0,1) (+x20 outlier channels), B: weight [n,k] N(0,0.02); both
    quantised to NVFP4 by the oracle with gs = 2688/amax; alpha = 1/(gsA*gsB) in fp32."""
    xa = synth.activation(seed, m, k, outliers=outliers)
    xb, gsb, qb, sfb = _nvfp4_weight(n, k, seed)
    gsa = global_scale(xa)
    qa, sfa = oquant.nvfp4_quantize(xa, gsa)
    alpha = F32(1.0) / (gsa * gsb)
    return dict(xa=xa, xb=xb, gsa=gsa, gsb=gsb, qa=qa, sfa=sfa, qb=qb, sfb=sfb, alpha=alpha, m=m, n=n, k=k)


def dev(a, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)) if isinstance(a, np.ndarray) else a
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def scalar(v) -> torch.Tensor:
    return torch.tensor([float(v)], dtype=torch.float32, device="cuda")


def reference(ops: dict, rows=None):
    """Oracle result R (fp64) and its tolerance for all rows or the given row subset."""
    m, n, k = ops["m"], ops["n"], ops["k"]
    A = ogemm.dequantize(ops["qa"], ops["sfa"], m, k, 16, "e4m3")
    B = ogemm.dequantize(ops["qb"], ops["sfb"], n, k, 16, "e4m3")
    if rows is not None:
        A = A[np.asarray(rows)]
    al = np.float64(ops["alpha"])
    R = al * (A @ B.T)
    tol = ogemm.tolerance(R, ogemm.abs_product_sum(A, B, ops["alpha"]))
    return R, tol


def assert_within(D: torch.Tensor, R: np.ndarray, tol: np.ndarray, what: str = "") -> float:
    """|D - R| <= tol elementwise; returns the worst |D - R| / tol."""
    d = D.float().cpu().numpy().astype(np.float64)
    assert d.shape == R.shape, (d.shape, R.shape)
    err = np.abs(d - R)
    bad = err > tol
    ratio = float(np.max(np.where(tol > 0, err / np.maximum(tol, 1e-300), np.where(err > 0, np.inf, 0.0))))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"[{i},{j}] got {d[i, j]!r} want {R[i, j]!r} tol {tol[i, j]:.3g}" for i, j in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; {detail}")
    return ratio
