"""Seeded synthetic inputs shared by the CPU oracle, the tests and the benchmark.

This module draws numbers and shapes workloads; it holds none of the NVFP4 /
MXFP4 arithmetic (no quantisation, no scale layout, no GEMM).  Every tensor it
returns lives in host memory.

Recipe (stated once, used everywhere):

* Random bits: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014), counter form: output ``i`` of stream ``s``
  is ``mix64(s + (i + 1) * 0x9E3779B97F4A7C15)`` with the published finaliser
  constants.  A stream is addressed by ``seed * 8 + t`` with ``t`` = 0 for
  activations, 1 for weights, 2 for the outlier-channel choice, 3 for router
  logits.
* Normals: Box-Muller in fp64 on consecutive output pairs,
  ``u1 = ((r0 >> 11) + 1) * 2**-53``, ``u2 = (r1 >> 11) * 2**-53``,
  ``z0 = sqrt(-2 ln u1) cos(2 pi u2)``, ``z1 = sqrt(-2 ln u1) sin(2 pi u2)``.
* Values are scaled in fp64, rounded to fp32 and then to bf16 (both RNE).
* Activation outliers: ``round(0.001 * K)`` distinct K-channels (at least one)
  picked by a partial Fisher-Yates shuffle driven by stream ``seed*8+2`` and
  multiplied by 20 before the rounding to bf16 (the "0.1% of channels scaled
  x20" of the decode and prefill workloads).
* Every generator takes an optional ``device``: the same steps then run there.  On a GPU the
  fp64 log / cos / sin may differ from the host's in the last bit, so a value can, rarely, round
  to a neighbouring bf16; the parity tests therefore draw on the host, and the benchmark draws
  its large timing inputs on the GPU.
* MoE routing: fp32 logits N(0,1) of shape [tokens, experts] from stream
  ``seed*8+3``, softmax over experts in fp32, top-k by a stable descending sort
  (ties go to the lower expert id); the per-expert row counts are what the
  grouped GEMM sees.
"""
from __future__ import annotations

import math

import torch

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

STREAM_ACT, STREAM_WEIGHT, STREAM_OUTLIER, STREAM_ROUTER = 0, 1, 2, 3

_CHUNK = 1 << 24


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit integer as a signed int64 value."""
    v &= _MASK64
    return v - (1 << 64) if v >> 63 else v


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def splitmix64(stream: int, start: int, count: int, device=None) -> torch.Tensor:
    """Outputs ``start .. start+count-1`` of SplitMix64 stream ``stream`` as int64 bit patterns."""
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    state = idx * _s64(GOLDEN) + _s64(stream)
    return _mix64(state)


def splitmix64_py(stream: int, count: int) -> list[int]:
    """Plain-Python SplitMix64 (unsigned ints); used to pin the vectorised form."""
    out, state = [], stream & _MASK64
    for _ in range(count):
        state = (state + GOLDEN) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * _M1) & _MASK64
        z = ((z ^ (z >> 27)) * _M2) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def normal(stream: int, count: int, device=None) -> torch.Tensor:
    """``count`` standard normals (fp64) from SplitMix64 stream ``stream`` by Box-Muller."""
    out = torch.empty(count, dtype=torch.float64, device=device)
    pairs = (count + 1) // 2
    done = 0
    while done < pairs:
        n = min(_CHUNK, pairs - done)
        r = splitmix64(stream, 2 * done, 2 * n, device).view(n, 2)
        u1 = (_lsr(r[:, 0], 11) + 1).to(torch.float64) * 2.0 ** -53
        u2 = _lsr(r[:, 1], 11).to(torch.float64) * 2.0 ** -53
        rad = torch.sqrt(-2.0 * torch.log(u1))
        th = (2.0 * math.pi) * u2
        z = torch.stack((rad * torch.cos(th), rad * torch.sin(th)), dim=1).reshape(-1)
        lo = 2 * done
        hi = min(count, lo + 2 * n)
        out[lo:hi] = z[: hi - lo]
        done += n
    return out


def to_bf16(v: torch.Tensor) -> torch.Tensor:
    """fp64 -> fp32 -> bf16, each step round-to-nearest-even."""
    return v.to(torch.float32).to(torch.bfloat16)


def outlier_channels(seed: int, k: int) -> torch.Tensor:
    """Distinct activation channels scaled x20: round(0.001*K) of them, at least one."""
    count = max(1, int(round(0.001 * k)))
    r = splitmix64(seed * 8 + STREAM_OUTLIER, 0, count)
    perm = list(range(k))
    for i in range(count):
        u = int(r[i].item()) & _MASK64
        j = i + u % (k - i)
        perm[i], perm[j] = perm[j], perm[i]
    return torch.tensor(sorted(perm[:count]), dtype=torch.int64)


def activation(seed: int, m: int, k: int, outliers: bool = True, std: float = 1.0, device=None) -> torch.Tensor:
    """bf16 activation [m, k]: N(0, std^2) with optional x20 outlier channels."""
    v = normal(seed * 8 + STREAM_ACT, m * k, device).view(m, k) * std
    if outliers and m > 0:
        v[:, outlier_channels(seed, k).to(v.device)] *= 20.0
    return to_bf16(v)


def weight(seed: int, n: int, k: int, std: float = 0.02, experts: int | None = None, device=None) -> torch.Tensor:
    """bf16 weight [n, k] (or [experts, n, k]) drawn N(0, std^2)."""
    shape = (n, k) if experts is None else (experts, n, k)
    count = math.prod(shape)
    return to_bf16(normal(seed * 8 + STREAM_WEIGHT, count, device).view(shape) * std)


def moe_topk(seed: int, tokens: int, experts: int, topk: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Softmax top-k routing of N(0,1) logits [tokens, experts]: (expert ids int32 [tokens, topk],
    routing weights fp32 [tokens, topk] = the chosen probabilities renormalised to sum 1).  Ties go
    to the lower expert id (stable sort)."""
    logits = normal(seed * 8 + STREAM_ROUTER, tokens * experts).to(torch.float32).view(tokens, experts)
    probs = torch.softmax(logits, dim=1)
    srt = torch.sort(probs, dim=1, descending=True, stable=True)
    ids, p = srt.indices[:, :topk], srt.values[:, :topk]
    return ids.to(torch.int32), (p / p.sum(dim=1, keepdim=True)).to(torch.float32)


def moe_routing(seed: int, tokens: int, experts: int, topk: int) -> torch.Tensor:
    """Per-expert row counts (int64 [experts]) from softmax top-k routing of N(0,1) logits."""
    ids, _ = moe_topk(seed, tokens, experts, topk)
    return torch.bincount(ids.to(torch.int64).reshape(-1), minlength=experts)


def moe_offsets(counts: torch.Tensor) -> torch.Tensor:
    """Row offsets [E+1] of expert-sorted rows (prefix sums of the counts)."""
    counts = counts.to(torch.int64)
    row = torch.zeros(counts.numel() + 1, dtype=torch.int64)
    row[1:] = torch.cumsum(counts, 0)
    return row


def random_bytes(stream: int, count: int) -> torch.Tensor:
    """``count`` uniformly random bytes (uint8) from a SplitMix64 stream."""
    words = (count + 7) // 8
    r = splitmix64(stream, 0, words)
    return r.view(torch.uint8)[:count].clone()
