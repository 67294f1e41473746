#!/usr/bin/env python
"""Benchmark of the NVFP4 quantise -> GEMM hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|e2e|moe|moe_nvfp4|pipeline]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

Workloads (synthetic, seeded; shapes and value distributions of the pages' benchmarks):
  decode   (default)  N=4096, K=7168, M in {1,4,8,16,32,64,128,256}.  One step quantises the
                      bf16 activation of every M on the device and multiplies it with its own
                      copy of the NVFP4 weight (8 distinct copies, 132 MB, so no GEMM finds its
                      weight in L2), quant and GEMM chained with programmatic dependent launch.
  prefill             (M,N,K) in {(1024,4096,7168), (2048,4096,7168), (4096,4096,7168),
                      (4096,4096,4096), (128,7168,2048)}, quant -> GEMM per shape.
  e2e                 bf16 activation [M,4096], M in {256,512}, weights [14336,4096]: quant ->
                      GEMM with PDL; the line also carries the time without PDL.
  moe                 MXFP4: 4096 tokens top-8 over 128 experts (32768 rows); quantise, then the
                      gate+up grouped GEMM (N=1536, K=2048) and the down grouped GEMM (N=2048,
                      K=768) on a second quantised activation.
  moe_nvfp4           a whole NVFP4 MoE layer (same shape as moe): expert sort, gather,
                      quantise, gate+up grouped GEMM, fused SiLU*mul + quantise, down grouped
                      GEMM, weighted combine, chained with PDL.
  pipeline            4 back-to-back quant->GEMM layers (N=K=7168, own weight per layer) at
                      M in {1,16,64,256,1024,2048,4096}; the line adds each M's 4-layer time
                      with and without PDL.
Each step is captured once in a CUDA graph and replayed; the L2 is flushed before every timed
step, outside the timed interval: a 512 MB write, then a 512 MB read of a second buffer, so the
step starts with none of its inputs in L2 and with L2 holding clean lines (as after the previous
layer's kernels), not 126 MB of dirty lines whose write-back would compete with the step's
reads.  `value` is GEMM TFLOPS over the whole step (quantisation time included); `roofline`
covers the GEMM kernel, timed on its own in a second graph of the step's GEMM launches.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "NVFP4 GEMM TFLOPS and % of binding roofline (FP4 peak or 8 TB/s HBM) vs M"
DECODE_MS = (1, 4, 8, 16, 32, 64, 128, 256)
PREFILL = ((1024, 4096, 7168), (2048, 4096, 7168), (4096, 4096, 7168), (4096, 4096, 4096), (128, 7168, 2048))
# FlashInfer PR 4865 B300 table (best of its SM100/SM103 kernels, ms), N=4096 K=7168: context only
PAGES_B300_DECODE_MS = {1: 0.0100, 4: 0.0099, 8: 0.0096, 16: 0.0097, 32: 0.0097, 64: 0.0094, 128: 0.0096, 256: 0.0091}
# same table, other shapes (us, faster of the two kernels): context only
PAGES_B300_PREFILL_US = {(1024, 4096, 7168): 13.4, (2048, 4096, 7168): 21.5, (4096, 4096, 7168): 36.7,
                         (4096, 4096, 4096): 25.1, (128, 7168, 2048): 6.1, (256, 14336, 4096): 12.6,
                         (512, 14336, 4096): 17.4}


def gemm_bytes(m, n, k):
    """Algorithmic bytes of one NVFP4 GEMM: packed A and B, their scales (unpadded), bf16 D."""
    return m * k // 2 + m * k // 16 + n * k // 2 + n * k // 16 + 2 * m * n


def grouped_bytes(experts, t, n, k):
    return experts * n * k * (1 / 2 + 1 / 32) + t * k * (1 / 2 + 1 / 32) + 2 * t * n


def quant_bytes(m, k, vec=16):
    return 2 * m * k + m * k // 2 + m * k // vec


def recorded_traffic(workload: str):
    """DRAM bytes per GEMM launch from the last ncu capture (profiles/gemm_traffic.json), or
    None when the GEMM sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for src in rec["kernel_sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec["kernel_sha256"] or workload not in rec:
        return None
    return rec[workload]["dram_bytes_per_launch_avg"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """SM clock and clock-event reasons sampled every ~1 ms through NVML (read-only queries)
    while the timed region runs.  If NVML cannot be loaded there are no samples: the line's
    `clocks` then carries null clocks and the reason NVML was unavailable."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: int):
        import threading
        self.samples, self.mask, self.max_mhz, self.err = [], 0, None, None
        self.stop_ev = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            nv.nvmlInit_v2()
            h = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                cnt = ctypes.c_uint()
                nv.nvmlDeviceGetCount_v2(ctypes.byref(cnt))
                if cnt.value != 1 or nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                    raise RuntimeError("NVML device not found")
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.nv, self.h = nv, h
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
        except Exception as e:  # noqa: BLE001
            self.err = f"NVML unavailable ({e})"
            self.t = None

    def _poll(self):
        mhz, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        get_r = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_ev.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if get_r(self.h, ctypes.byref(reasons)) == 0:
                self.mask |= reasons.value
            time.sleep(0.001)

    def stop(self) -> dict:
        if self.t is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.err]}
        self.stop_ev.set()
        self.t.join()
        reasons = sorted(v for k, v in self.REASONS.items() if self.mask & k)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "source": "NVML, 1 ms polling during the timed steps"}


# ---------------------------------------------------------------------------- workloads
class Workload:
    """Holds device buffers and knows how to run one step (quant -> GEMM chain)."""

    def __init__(self, nv, name: str):
        self.nv, self.name = nv, name
        self.launches = []         # callables, in order, each one kernel
        self.gemm_launches = []    # the GEMM kernels alone (roofline pass)
        self.flops = 0.0
        self.gemm_bytes = 0.0
        self.quant_bytes = 0.0
        self.h2d = []              # (device tensor, pinned host tensor) per step input
        self.d2h = []              # (host tensor, device tensor) per step output
        self.h2d_at = []           # per input: index of the first launch that reads it (default 0)
        self.d2h_after = []        # per output: index of the launch that writes it (default: last)
        self.config = {}
        self.extra = {}

    def step(self):
        for f in self.launches:
            f()

    def pack_transfers(self, align: int = 256, device: str = "cuda"):
        """Moves the step's inputs into one device buffer (each tensor becomes a view at an
        `align`-byte offset) with one pinned host image, and its outputs likewise, so that a step
        crosses the host link with one copy each way instead of one per tensor.  Must run before
        the launches are captured: the launch closures hold these tensor objects, which `set_`
        re-points in place.  Returns (h2d_bytes, d2h_bytes) per step."""
        moved, ranges = [], []
        for pairs, dev_at in ((self.h2d, 0), (self.d2h, 1)):
            if not pairs:
                moved.append(None)
                ranges.append([])
                continue
            offs, total = [], 0
            for p in pairs:
                t = p[dev_at]
                assert t.is_contiguous()
                offs.append(total)
                total += -(-t.numel() * t.element_size() // align) * align
            dbuf = torch.empty(total, dtype=torch.uint8, device=device)
            hbuf = torch.empty(total, dtype=torch.uint8)
            hbuf = hbuf.pin_memory() if device == "cuda" else hbuf
            for p, o in zip(pairs, offs):
                for t, buf in ((p[dev_at], dbuf), (p[1 - dev_at], hbuf)):
                    nb = t.numel() * t.element_size()
                    slot = buf[o:o + nb].view(t.dtype).view(t.shape)
                    slot.copy_(t)
                    t.set_(slot)
            moved.append((dbuf, hbuf))
            ranges.append([(o, e) for o, e in zip(offs, offs[1:] + [total])])
        self.h2d_buf, self.d2h_buf = moved
        self.h2d_ranges, self.d2h_ranges = ranges
        return tuple(0 if b is None else b[0].numel() for b in moved)

    def transfer_groups(self):
        """After `pack_transfers`: the input copies as [(launch index, start, end)] in packed
        order, neighbours read first by the same launch merged into one copy, and the output copies
        as [(launch index, start, end)], the launch being the one that writes those bytes."""
        last = len(self.launches) - 1
        groups = []
        for ranges, at, dflt in ((self.h2d_ranges, self.h2d_at, 0), (self.d2h_ranges, self.d2h_after, last)):
            out = []
            for j, (a, b) in enumerate(ranges):
                i = at[j] if j < len(at) else dflt
                assert 0 <= i <= last
                if out and out[-1][0] == i and out[-1][2] == a:
                    out[-1] = (i, out[-1][1], b)
                else:
                    out.append((i, a, b))
            groups.append(out)
        return groups


def _gs(x: torch.Tensor) -> float:
    return float(np.float32(2688.0) / np.float32(x.float().abs().max().item()))


def build_nvfp4_chain(nv, wl: Workload, shapes, weight_seed=0, weights_by_shape=None, pdl=True):
    flags = nv.FLAG_PDL if pdl else 0
    cache = {} if weights_by_shape is None else weights_by_shape
    # one zeroed split-K workspace serves every GEMM of the chain (they run in stream order)
    ws = nv.gemm_workspace(max(nv.gemm_workspace_size(m, n, k) for (m, n, k) in shapes))
    for i, (m, n, k) in enumerate(shapes):
        key = (n, k)
        if key not in cache:
            w = synth.weight(weight_seed, n, k)
            gsw = _gs(w)
            qb, sfb = nv.nvfp4_quantize(w.cuda(), torch.tensor([gsw], device="cuda"))
            cache[key] = (qb, sfb, gsw)
        qb, sfb, gsw = cache[key]
        qb, sfb = qb.clone(), sfb.clone()          # every GEMM streams its own weight copy
        x = synth.activation(i, m, k)
        gsa = _gs(x)
        xd = x.cuda()
        gs_d = torch.tensor([gsa], dtype=torch.float32, device="cuda")
        al_d = torch.tensor([float(np.float32(1.0) / (np.float32(gsa) * np.float32(gsw)))], device="cuda")
        q = torch.empty((m, k // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty(nv.sf_bytes(m, k), dtype=torch.uint8, device="cuda")
        d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        wl.launches.append(lambda xd=xd, gs_d=gs_d, q=q, sf=sf: nv.nvfp4_quantize(xd, gs_d, q, sf, flags=flags))
        g = (lambda q=q, sf=sf, qb=qb, sfb=sfb, al_d=al_d, d=d, f=flags:
             nv.nvfp4_gemm(q, sf, qb, sfb, al_d, d, flags=f, workspace=ws))
        wl.launches.append(g)
        wl.gemm_launches.append(g)
        wl.flops += 2.0 * m * n * k
        wl.gemm_bytes += gemm_bytes(m, n, k)
        wl.quant_bytes += quant_bytes(m, k)
        wl.h2d.append((xd, x.pin_memory()))
        wl.h2d_at.append(len(wl.launches) - 2)           # the quantiser reads it
        wl.d2h.append((torch.empty((m, n), dtype=torch.bfloat16).pin_memory(), d))
        wl.d2h_after.append(len(wl.launches) - 1)        # the GEMM writes it


def make_decode(nv):
    wl = Workload(nv, "decode")
    build_nvfp4_chain(nv, wl, [(m, 4096, 7168) for m in DECODE_MS])
    wl.config = {"workload": "decode sweep: NVFP4 quant->GEMM, N=4096 K=7168, M in 1,4,8,16,32,64,128,256",
                 "global_batch": sum(DECODE_MS), "n": 4096, "k": 7168, "ms": list(DECODE_MS),
                 "inputs": "activation N(0,1) with 0.1% outlier channels x20, weight N(0,0.02), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read); 8 distinct weight copies",
                 "parallelism": "replicas"}
    return wl


def make_prefill(nv):
    wl = Workload(nv, "prefill")
    build_nvfp4_chain(nv, wl, list(PREFILL))
    wl.config = {"workload": "prefill sweep: NVFP4 quant->GEMM, (M,N,K) in " + str(list(PREFILL)),
                 "global_batch": sum(s[0] for s in PREFILL),
                 "inputs": "activation N(0,1) with 0.1% outlier channels x20, weight N(0,0.02), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


def make_e2e(nv, pdl=True):
    wl = Workload(nv, "e2e")
    build_nvfp4_chain(nv, wl, [(256, 14336, 4096), (512, 14336, 4096)], pdl=pdl)
    wl.config = {"workload": "quant->GEMM with PDL: act bf16 [M,4096], M in 256,512, weight [14336,4096]",
                 "global_batch": 768, "pdl": pdl,
                 "inputs": "activation N(0,1) with outlier channels x20, weight N(0,0.02), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


def make_moe(nv):
    wl = Workload(nv, "moe")
    E, T, topk, H, I = 128, 4096, 8, 2048, 768
    counts = synth.moe_routing(0, T, E, topk)
    ro = synth.moe_offsets(counts)
    rows = int(ro[-1])
    ro_d = ro.cuda()
    specs = [("gate_up", 2 * I, H, 1), ("down", H, I, 2)]
    for name, n, k, seed in specs:
        wb = synth.weight(seed, n, k, experts=E)
        qb = torch.empty((E, n, k // 2), dtype=torch.uint8, device="cuda")
        sfb = torch.empty((E, nv.sf_bytes(n, k, 32)), dtype=torch.uint8, device="cuda")
        for e in range(E):
            nv.mxfp4_quantize(wb[e].cuda(), q=qb[e], sf=sfb[e])
        del wb
        x = synth.activation(seed + 10, rows, k, outliers=False)
        xd = x.cuda()
        q = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
        sf = torch.zeros(nv.grouped_sf_bytes(rows, E, k), dtype=torch.uint8, device="cuda")
        d = torch.empty((rows, n), dtype=torch.bfloat16, device="cuda")
        fl = nv.FLAG_PDL
        wl.launches.append(lambda xd=xd, q=q, sf=sf: nv.mxfp4_quantize(xd, ro_d, q, sf, flags=fl))
        g = (lambda q=q, sf=sf, qb=qb, sfb=sfb, d=d: nv.mxfp4_grouped_gemm(q, sf, ro_d, qb, sfb, None, d, flags=fl))
        wl.launches.append(g)
        wl.gemm_launches.append(g)
        wl.flops += 2.0 * rows * n * k
        wl.gemm_bytes += grouped_bytes(E, rows, n, k)
        wl.quant_bytes += quant_bytes(rows, k, 32)
        wl.h2d.append((xd, x.pin_memory()))
        wl.h2d_at.append(len(wl.launches) - 2)
        wl.d2h.append((torch.empty((rows, n), dtype=torch.bfloat16).pin_memory(), d))
        wl.d2h_after.append(len(wl.launches) - 1)
    wl.config = {"workload": "MXFP4 MoE: 128 experts, 4096 tokens top-8 (32768 rows); gate+up N=1536 K=2048, "
                             "down N=2048 K=768; quant + grouped GEMM each",
                 "global_batch": rows, "expert_rows_min": int(counts.min()), "expert_rows_max": int(counts.max()),
                 "inputs": "activation N(0,1), weight N(0,0.02), router logits N(0,1), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


def nvfp4_grouped_bytes(experts, t, n, k):
    return experts * n * k * (1 / 2 + 1 / 16) + t * k * (1 / 2 + 1 / 16) + 2 * t * n


def make_moe_nvfp4(nv):
    """A whole NVFP4 MoE layer (the f3 steps): sort -> gather + quantise (one kernel) -> gate+up
    grouped GEMM -> SiLU*mul + quantise -> down grouped GEMM -> combine, chained with PDL.  128 experts, 4096
    tokens top-8, hidden 2048, expert intermediate 768 (the MXFP4 MoE shape, NVFP4 formats)."""
    wl = Workload(nv, "moe_nvfp4")
    E, T, topk, H, I = 128, 4096, 8, 2048, 768
    ids, wts = synth.moe_topk(0, T, E, topk)
    x = synth.activation(20, T, H, outliers=False)
    ids_d, wts_d, xd = ids.cuda(), wts.cuda(), x.cuda()
    gs1 = torch.full((E,), _gs(x), dtype=torch.float32, device="cuda")
    specs = {}
    for name, n, k, seed in (("gate_up", 2 * I, H, 1), ("down", H, I, 2)):
        qb = torch.empty((E, n, k // 2), dtype=torch.uint8, device="cuda")
        sfb = torch.empty((E, nv.sf_bytes(n, k, 16)), dtype=torch.uint8, device="cuda")
        gsb = torch.empty(E, dtype=torch.float32)
        for e in range(E):
            w = synth.weight(seed * 1000 + e, n, k)
            gsb[e] = _gs(w)
            nv.nvfp4_quantize(w.cuda(), gsb[e:e + 1].cuda(), q=qb[e], sf=sfb[e])
        specs[name] = (qb, sfb, gsb)
    R = T * topk
    P = nv.FLAG_PDL
    ro = torch.empty(E + 1, dtype=torch.int64, device="cuda")
    src = torch.empty(R, dtype=torch.int32, device="cuda")
    pos = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    q1 = torch.empty((R, H // 2), dtype=torch.uint8, device="cuda")
    s1 = torch.empty(nv.expert_sf_bytes(R, E, H), dtype=torch.uint8, device="cuda")
    h1 = torch.empty((R, 2 * I), dtype=torch.bfloat16, device="cuda")
    q2 = torch.empty((R, I // 2), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(nv.expert_sf_bytes(R, E, I), dtype=torch.uint8, device="cuda")
    y = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    a1 = (1.0 / (gs1.cpu() * specs["gate_up"][2])).to(torch.float32).cuda()
    # the SiLU*mul output's global scale: calibrated once from a run of the first half
    nv.moe_sort_by_expert(ids_d, E)
    ro0, src0, _ = nv.moe_sort_by_expert(ids_d, E)
    xq, xs = nv.nvfp4_quantize_experts(nv.moe_gather_rows(xd, src0), ro0, gs1)
    hh = nv.nvfp4_grouped_gemm(xq, xs, ro0, specs["gate_up"][0], specs["gate_up"][1], a1)
    hf = hh.float()
    hamax = float((torch.nn.functional.silu(hf[:, :I]) * hf[:, I:]).abs().max().item())
    gs2 = torch.full((E,), float(np.float32(2688.0) / np.float32(hamax)), dtype=torch.float32, device="cuda")
    a2 = (1.0 / (gs2.cpu() * specs["down"][2])).to(torch.float32).cuda()
    del xq, xs, hh, hf
    L = wl.launches
    sort_ws = torch.empty(max(1, nv.moe_sort_workspace_size(T, E) // 4), dtype=torch.int32, device="cuda")
    L.append(lambda: nv.moe_sort_by_expert(ids_d, E, out=(ro, src, pos), workspace=sort_ws, flags=P))
    L.append(lambda: nv.nvfp4_gather_quantize_experts(xd, src, ro, gs1, q=q1, sf=s1, flags=P))
    g1 = (lambda: nv.nvfp4_grouped_gemm(q1, s1, ro, specs["gate_up"][0], specs["gate_up"][1], a1, d=h1, flags=P))
    L.append(g1)
    L.append(lambda: nv.nvfp4_silu_mul_quantize_experts(h1, ro, gs2, q=q2, sf=s2, flags=P))
    g2 = (lambda: nv.nvfp4_grouped_gemm(q2, s2, ro, specs["down"][0], specs["down"][1], a2, d=y, flags=P))
    L.append(g2)
    L.append(lambda: nv.moe_combine(y, pos, wts_d, out=out, flags=P))
    wl.gemm_launches += [g1, g2]
    wl.flops = 2.0 * R * (2 * I * H + H * I)
    wl.gemm_bytes = nvfp4_grouped_bytes(E, R, 2 * I, H) + nvfp4_grouped_bytes(E, R, H, I)
    wl.quant_bytes = quant_bytes(R, H) + quant_bytes(R, 2 * I)
    wl.h2d += [(xd, x.pin_memory()), (ids_d, ids.pin_memory()), (wts_d, wts.pin_memory())]
    wl.h2d_at += [1, 0, 5]                               # gather+quantise, sort, combine
    wl.d2h.append((torch.empty((T, H), dtype=torch.bfloat16).pin_memory(), out))
    wl.config = {"workload": "NVFP4 MoE layer: 128 experts, 4096 tokens top-8 (32768 rows), hidden 2048, intermediate "
                             "768; sort, gather+quantise, gate+up grouped GEMM (N=1536, K=2048), SiLU*mul+quantise, "
                             "down grouped GEMM (N=2048, K=768), combine",
                 "global_batch": R, "inputs": "activation N(0,1), expert weights N(0,0.02), router logits N(0,1), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


PIPE_MS = (1, 16, 64, 256, 1024, 2048, 4096)
PIPE_LAYERS = 4


def pipeline_shapes(m):
    return [(m, 7168, 7168)] * PIPE_LAYERS


def make_pipeline(nv):
    """Back-to-back quant->GEMM layers (vLLM fork compare view "add pdl",
    benchmark_nvfp4_sm103.py, benchmark_pdl_pipeline: 4 layers, N = K = 7168).  One step runs
    the 4-layer pipeline at every M of PIPE_MS; each layer streams its own weight copy (the page
    reuses one weight for all layers, which L2 would then hold after the first)."""
    wl = Workload(nv, "pipeline")
    cache = {}
    build_nvfp4_chain(nv, wl, [s for m in PIPE_MS for s in pipeline_shapes(m)], weights_by_shape=cache)
    wl.extra["weights"] = cache
    wl.config = {"workload": f"{PIPE_LAYERS}-layer quant->GEMM pipeline with PDL, N=K=7168, M in {','.join(map(str, PIPE_MS))}",
                 "global_batch": PIPE_LAYERS * sum(PIPE_MS), "layers": PIPE_LAYERS, "n": 7168, "k": 7168,
                 "inputs": "activation N(0,1) with 0.1% outlier channels x20, weight N(0,0.02), seed 0",
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


def make_custom(nv, shapes):
    wl = Workload(nv, "custom")
    build_nvfp4_chain(nv, wl, shapes)
    wl.config = {"workload": "NVFP4 quant->GEMM chain " + str(shapes), "global_batch": sum(s[0] for s in shapes),
                 "l2": "flushed before every timed step (512 MB write, then 512 MB read)", "parallelism": "replicas"}
    return wl


MAKERS = {"decode": make_decode, "prefill": make_prefill, "e2e": make_e2e, "moe": make_moe, "pipeline": make_pipeline,
          "moe_nvfp4": make_moe_nvfp4}


# ---------------------------------------------------------------------------- timing
def capture(fns) -> torch.cuda.CUDAGraph:
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in fns:   # warm-up outside capture: kernel attributes, module load
            f()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    torch.cuda.synchronize()
    return g


def capture_e2e(wl: Workload) -> torch.cuda.CUDAGraph:
    """The step with its host transfers in one graph: the input copies run in packed order on one
    side stream and each launch waits for the copies it reads first; each output is copied back
    on a second side stream once the launch that writes it has finished.  So the copies overlap
    the kernels instead of bracketing them."""
    (dbuf, hbuf), (odbuf, ohbuf) = wl.h2d_buf, wl.d2h_buf
    ins, outs = wl.transfer_groups()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        cin.wait_event(fork)
        cout.wait_event(fork)
        ready = {}
        with torch.cuda.stream(cin):
            for i, a, b in ins:
                dbuf[a:b].copy_(hbuf[a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cin)
                ready.setdefault(i, []).append(e)
        written = {}
        for i, a, b in outs:
            written.setdefault(i, []).append((a, b))
        for i, f in enumerate(wl.launches):
            for e in ready.get(i, []):
                main.wait_event(e)
            f()
            for a, b in written.get(i, []):
                e = torch.cuda.Event()
                e.record(main)
                cout.wait_event(e)
                with torch.cuda.stream(cout):
                    ohbuf[a:b].copy_(odbuf[a:b], non_blocking=True)
        for side in (cin, cout):
            e = torch.cuda.Event()
            e.record(side)
            main.wait_event(e)
    return g


class L2Flush:
    """Evicts the step's data from L2: writes a 512 MB buffer, then reads a second one, so what
    L2 holds afterwards is clean (no write-backs land inside the timed interval)."""

    def __init__(self):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(128 << 20, dtype=torch.int32, device="cuda")

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)
        self.r.sum()


def timed_replays(g, n: int, flush: L2Flush, before=None, after=None) -> list[float]:
    """Per-replay device times (ms), each after an L2 flush outside the timed interval."""
    out = []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush(i)
        a, b = evs[i]
        a.record()
        if before:
            before()
        g.replay()
        if after:
            after()
        b.record()
    torch.cuda.synchronize()
    for a, b in evs:
        out.append(a.elapsed_time(b))
    return out


# ---------------------------------------------------------------------------- per-config lines
# Every graded configuration on its own (the metric is "... vs M"): per GEMM, CUDA-event time
# with cold L2, throughput, and the fraction of the binding roofline
#   t_roof = max(flops / FP4 peak, algorithmic bytes / HBM peak),  frac = t_roof / t.
# "us_per_gemm": a PDL chain of R GEMMs of the shape with R distinct weight copies (the
# steady state of back-to-back layers), time / R; "single_us": one GEMM per graph replay
# (includes the graph's launch gap on the device, ~1-2 us, so it understates short kernels).
PER_CONFIG_REPS = 20


def _graph_ms(fns, flush, reps=PER_CONFIG_REPS, warm=3) -> float:
    g = capture(fns)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    t = statistics.mean(timed_replays(g, reps, flush))
    del g
    return t


def _qweight(nv, seed, n, k, dev="cuda"):
    w = synth.weight(seed, n, k, device=dev)
    gsw = _gs(w)
    qb, sfb = nv.nvfp4_quantize(w, torch.tensor([gsw], device=dev))
    del w
    return qb, sfb, gsw


def _qact(nv, seed, m, k, gsw, dev="cuda"):
    x = synth.activation(seed, m, k, device=dev)
    gsa = _gs(x)
    qa, sfa = nv.nvfp4_quantize(x, torch.tensor([gsa], device=dev))
    al = torch.tensor([float(np.float32(1.0) / (np.float32(gsa) * np.float32(gsw)))], device=dev)
    return x, gsa, qa, sfa, al


def _entry(kind, m, n, k, us, flops, nbytes, hbm, fp4, **extra):
    t = us * 1e-6
    t_hbm, t_fp4 = nbytes / (hbm * 1e9), flops / (fp4 * 1e12)
    e = {"config": kind, "m": m, "n": n, "k": k, "us_per_gemm": round(us, 3),
         "tflops": round(flops / t / 1e12, 1), "gbs": round(nbytes / t / 1e9, 1),
         "bound": "hbm" if t_hbm >= t_fp4 else "tensor", "roof_us": round(max(t_hbm, t_fp4) * 1e6, 3),
         "frac": round(max(t_hbm, t_fp4) / t, 4)}
    e.update(extra)
    return e


def per_config(nv, flush, hbm, fp4):
    P = nv.FLAG_PDL
    out = []

    def gemm_chain(shape, copies, seed):
        m, n, k = shape
        ws = nv.gemm_workspace(nv.gemm_workspace_size(m, n, k))
        qb, sfb, gsw = _qweight(nv, seed, n, k)
        ws_ = [(qb, sfb)] + [(qb.clone(), sfb.clone()) for _ in range(copies - 1)]
        _, _, qa, sfa, al = _qact(nv, seed + 100, m, k, gsw)
        d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        fns = [(lambda b=b, sb=sb: nv.nvfp4_gemm(qa, sfa, b, sb, al, d, flags=P, workspace=ws)) for b, sb in ws_]
        chain = _graph_ms(fns, flush) * 1e3 / copies
        single = _graph_ms(fns[:1], flush) * 1e3
        return chain, single

    for m in DECODE_MS:
        n, k = 4096, 7168
        chain, single = gemm_chain((m, n, k), 8, 0)
        out.append(_entry("decode", m, n, k, chain, 2.0 * m * n * k, gemm_bytes(m, n, k), hbm, fp4,
                          single_us=round(single, 3), chain=8,
                          pages_b300_us=round(PAGES_B300_DECODE_MS[m] * 1e3, 2)))
    for (m, n, k) in PREFILL:
        chain, single = gemm_chain((m, n, k), 2, 1)
        out.append(_entry("prefill", m, n, k, chain, 2.0 * m * n * k, gemm_bytes(m, n, k), hbm, fp4,
                          single_us=round(single, 3), chain=2,
                          pages_b300_us=PAGES_B300_PREFILL_US.get((m, n, k))))
    # quantiser -> GEMM, with and without programmatic dependent launch (4 pairs, own weights)
    for m in (256, 512):
        n, k = 14336, 4096
        qb, sfb, gsw = _qweight(nv, 2, n, k)
        wts = [(qb, sfb)] + [(qb.clone(), sfb.clone()) for _ in range(3)]
        res = {}
        for tag, fl in (("pdl", P), ("no_pdl", 0)):
            fns, gfns = [], []
            for i, (b, sb) in enumerate(wts):
                x, gsa, qa, sfa, al = _qact(nv, 200 + i, m, k, gsw)
                gs_d = torch.tensor([gsa], dtype=torch.float32, device="cuda")
                d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
                fns.append(lambda x=x, g=gs_d, q=qa, s_=sfa, fl=fl: nv.nvfp4_quantize(x, g, q, s_, flags=fl))
                g = (lambda q=qa, s_=sfa, b=b, sb=sb, al=al, d=d, fl=fl: nv.nvfp4_gemm(q, s_, b, sb, al, d, flags=fl))
                fns.append(g)
                gfns.append(g)
            res[tag] = _graph_ms(fns, flush) * 1e3 / len(wts)
            if tag == "pdl":
                res["gemm"] = _graph_ms(gfns, flush) * 1e3 / len(wts)
        out.append(_entry("e2e_gemm", m, n, k, res["gemm"], 2.0 * m * n * k, gemm_bytes(m, n, k), hbm, fp4,
                          quant_gemm_pdl_us=round(res["pdl"], 3), quant_gemm_no_pdl_us=round(res["no_pdl"], 3),
                          pdl_speedup=round(res["no_pdl"] / res["pdl"], 3), chain=len(wts),
                          pages_b300_us=PAGES_B300_PREFILL_US.get((m, n, k))))
        del wts, qb, sfb
    # MoE grouped GEMMs: 128 experts, 4096 tokens top-8; MXFP4 and NVFP4 formats
    E, T, topk, H, I = 128, 4096, 8, 2048, 768
    counts = synth.moe_routing(0, T, E, topk)
    ro = synth.moe_offsets(counts).cuda()
    rows = int(counts.sum())
    for fmt in ("mxfp4", "nvfp4"):
        for name, n, k, seed in (("gate_up", 2 * I, H, 1), ("down", H, I, 2)):
            wb = synth.weight(seed, n, k, experts=E, device="cuda")
            x = synth.activation(seed + 10, rows, k, outliers=False, device="cuda")
            d = torch.empty((rows, n), dtype=torch.bfloat16, device="cuda")
            if fmt == "mxfp4":
                qb = torch.empty((E, n, k // 2), dtype=torch.uint8, device="cuda")
                sfb = torch.empty((E, nv.sf_bytes(n, k, 32)), dtype=torch.uint8, device="cuda")
                for e in range(E):
                    nv.mxfp4_quantize(wb[e], q=qb[e], sf=sfb[e])
                qa, sfa = nv.mxfp4_quantize(x, ro)
                fn = (lambda: nv.mxfp4_grouped_gemm(qa, sfa, ro, qb, sfb, None, d, flags=P))
                nbytes = grouped_bytes(E, rows, n, k)
            else:
                qb = torch.empty((E, n, k // 2), dtype=torch.uint8, device="cuda")
                sfb = torch.empty((E, nv.sf_bytes(n, k, 16)), dtype=torch.uint8, device="cuda")
                gsb = torch.empty(E, dtype=torch.float32)
                for e in range(E):
                    gsb[e] = _gs(wb[e])
                    nv.nvfp4_quantize(wb[e], gsb[e:e + 1].cuda(), q=qb[e], sf=sfb[e])
                gsa = _gs(x)
                qa, sfa = nv.nvfp4_quantize_experts(x, ro, torch.full((E,), gsa, device="cuda"))
                al = (1.0 / (gsa * gsb)).to(torch.float32).cuda()
                fn = (lambda: nv.nvfp4_grouped_gemm(qa, sfa, ro, qb, sfb, al, d, flags=P))
                nbytes = nvfp4_grouped_bytes(E, rows, n, k)
            del wb, x
            us = _graph_ms([fn], flush) * 1e3
            out.append(_entry(f"moe_{fmt}_{name}", rows, n, k, us, 2.0 * rows * n * k, nbytes, hbm, fp4,
                              experts=E, expert_rows_min=int(counts.min()), expert_rows_max=int(counts.max())))
            del qb, sfb, qa, sfa, d
    torch.cuda.empty_cache()
    return out


def targets(per):
    """The two throughput targets, read off the per-config entries."""
    dec = [e for e in per if e["config"] == "decode" and e["m"] <= 32]
    pre = [e for e in per if e["config"] == "prefill" and e["m"] >= 2048]
    return {"decode_m_le_32_hbm_frac_min": min(e["frac"] for e in dec) if dec else None,
            "prefill_m_ge_2048_fp4_frac_min": min(e["frac"] for e in pre) if pre else None,
            "target": 0.70}


def barrier(dist_on: bool, device: str = "cuda"):
    if dist_on:
        torch.distributed.barrier()
    if device == "cuda":
        torch.cuda.synchronize()


def max_over_ranks(v: float, dist_on: bool, device: str = "cuda") -> float:
    """The slowest rank's time: every rank gets the maximum of `v` over the ranks."""
    if not dist_on:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Replicas each do `flops_per_rank` in at most `ms_max`: the job's aggregate rate."""
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


def run_ours(args, dist_on, rank, world):
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_bf16_gb300 as nv

    if args.shapes:
        shapes = [tuple(int(v) for v in s.split(",")) for s in args.shapes.split(";")]
        wl = make_custom(nv, shapes)
    else:
        wl = MAKERS[args.workload](nv)
    flush = L2Flush()
    h2d_bytes, d2h_bytes = wl.pack_transfers()
    step_graph = capture(wl.launches)
    gemm_graph = capture(wl.gemm_launches)
    for _ in range(args.warmup):
        step_graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K steps, barrier + synchronize on both sides
    clocks = Clocks(torch.cuda.current_device())
    barrier(dist_on)
    t_wall = time.perf_counter()
    step_ms = timed_replays(step_graph, args.steps, flush)
    barrier(dist_on)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dist_on)

    # ---- GEMM kernels alone (roofline of the dominant kernel)
    # Means, not medians: CUDA events resolve these short graphs only to ~2 us, so a median
    # snaps to that grid; the mean over many replays does not.
    gemm_ms = timed_replays(gemm_graph, max(3, min(args.steps, 100)), flush)
    gemm_mean = statistics.mean(gemm_ms)
    per_launch_ms = gemm_mean / len(wl.gemm_launches)
    quant_ms = max(0.0, ms - gemm_mean)

    # ---- end to end through the public API with host buffers
    # (inputs packed into one pinned image and one device buffer, outputs likewise: one copy each
    # way per step, the bytes counted from those buffers)
    def h2d():
        dbuf, hbuf = wl.h2d_buf
        dbuf.copy_(hbuf, non_blocking=True)

    def d2h():
        dbuf, hbuf = wl.d2h_buf
        hbuf.copy_(dbuf, non_blocking=True)

    n_e2e = max(3, min(args.steps, 50))
    seq_ms = statistics.mean(timed_replays(step_graph, n_e2e, flush, before=h2d, after=d2h))
    torch.cuda.synchronize()
    want = wl.d2h_buf[1].clone()
    # The same step with the copies overlapping the kernels, kept only if its outputs equal the
    # sequential step's bit for bit after the device inputs were cleared (a launch that read its
    # input before the copy landed would differ).
    try:
        e2e_graph = capture_e2e(wl)
        wl.h2d_buf[0].zero_()
        wl.d2h_buf[1].zero_()
        e2e_graph.replay()
        torch.cuda.synchronize()
        overlap = "yes" if torch.equal(wl.d2h_buf[1], want) else "no: outputs differ from the sequential step"
    except Exception as exc:  # capture refused: keep the sequential copies
        overlap = f"no: {type(exc).__name__}: {str(exc).splitlines()[0][:160] if str(exc) else ''}"
    if overlap == "yes":
        e2e_ms = statistics.mean(timed_replays(e2e_graph, n_e2e, flush))
    else:
        e2e_ms = seq_ms
    e2e_ms = max_over_ranks(e2e_ms, dist_on)
    seq_ms = max_over_ranks(seq_ms, dist_on)

    hbm, bf16, peak_kind = peaks()
    tflops = whole_job_tflops(wl.flops, world, ms)
    gemm_gbs = wl.gemm_bytes / (gemm_mean * 1e-3) / 1e9
    fp4_peak_tflops = bf16 * 6.0  # nominal dense FP4 : bf16 ratio 13.5 : 2.25
    gemm_tflops = wl.flops / (gemm_mean * 1e-3) / 1e12
    # binding roof of the step's GEMMs: max(flops / FP4 peak, bytes / HBM)
    t_roof = max(wl.flops / (fp4_peak_tflops * 1e12), wl.gemm_bytes / (hbm * 1e9))
    bound = "hbm" if wl.gemm_bytes / (hbm * 1e9) >= wl.flops / (fp4_peak_tflops * 1e12) else "tensor"
    if bound == "hbm":
        tr = recorded_traffic(wl.name)
        roof = {"bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gemm_gbs / hbm, 4), "traffic": None if tr is None else round(tr),
                "algorithmic_bytes_per_launch": round(wl.gemm_bytes / len(wl.gemm_launches))}
    else:
        roof = {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak_tflops, 1),
                "unit": "TFLOP/s", "frac": round(gemm_tflops / fp4_peak_tflops, 4), "traffic": None}
    roof.update({"kernel": "bs_gemm_kernel" if wl.name not in ("moe", "moe_nvfp4") else "bs_gemm_kernel (grouped)",
                 "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json hbm_gbs' if bound == 'hbm' else 'bf16_tflops x 6, the nominal fp4/bf16 ratio'})",
                 "per_launch_ms": round(per_launch_ms, 5), "binding_roof_frac": round(t_roof / (gemm_mean * 1e-3), 4),
                 "bytes_per_step": wl.gemm_bytes})

    line = {"metric": METRIC, "value": round(tflops, 2), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp4 (e2m1) x fp4, fp32 accumulate, bf16 out",
            "data": "synthetic", "config": wl.config,
            "roofline": roof,
            "e2e": {"value": round(whole_job_tflops(wl.flops, world, e2e_ms), 2), "unit": "TFLOPS",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                    "copies_overlap_kernels": overlap, "sequential_ms_per_step": round(seq_ms, 5)},
            "gpu_launches": len(wl.launches) * args.steps,
            "clocks": clk,
            "breakdown": {"gemm_ms": round(gemm_mean, 5), "quant_ms_est": round(quant_ms, 5),
                          "quant_bytes_per_step": wl.quant_bytes, "wall_s": round(wall, 3)}}
    if wl.name == "decode":
        line["pages_b300_context"] = {
            "gemm_only_ms_sum": round(sum(PAGES_B300_DECODE_MS.values()), 4),
            "note": "FlashInfer PR 4865 B300 best-kernel times for the same 8 GEMMs (GEMM only, other machine)"}
    if wl.name == "e2e":
        nopdl = make_e2e(nv, pdl=False)
        g2 = capture(nopdl.launches)
        for _ in range(args.warmup):
            g2.replay()
        t2 = timed_replays(g2, args.steps, flush)
        line["without_pdl_ms_per_step"] = round(max_over_ranks(statistics.mean(t2), dist_on), 5)
    if wl.name == "pipeline":
        # per M: the 4-layer pipeline alone, with and without PDL (the page's table)
        per_m = {}
        for m in PIPE_MS:
            row = {}
            for tag, pdl in (("pdl_us", True), ("no_pdl_us", False)):
                w_m = Workload(nv, "pipeline_m")
                build_nvfp4_chain(nv, w_m, pipeline_shapes(m), weights_by_shape=wl.extra["weights"], pdl=pdl)
                g_m = capture(w_m.launches)
                for _ in range(args.warmup):
                    g_m.replay()
                t_m = statistics.mean(timed_replays(g_m, max(3, min(args.steps, 50)), flush)) * 1e3
                row[tag] = round(max_over_ranks(t_m, dist_on), 2)
                del g_m, w_m
            row["pdl_tflops"] = round(2.0 * m * 7168 * 7168 * PIPE_LAYERS / (row["pdl_us"] * 1e-6) / 1e12, 2)
            row["pdl_speedup"] = round(row["no_pdl_us"] / row["pdl_us"], 3)
            per_m[str(m)] = row
        line["pipeline"] = per_m
    if args.per_config and wl.name == "decode":
        per = per_config(nv, flush, hbm, fp4_peak_tflops)
        line["per_config"] = per
        line["targets"] = targets(per)
        line["per_config_method"] = (
            "CUDA events, L2 flushed before every replay; us_per_gemm = PDL chain of `chain` GEMMs with "
            "distinct weight copies / chain; single_us = one GEMM per replay; frac = max(flops/FP4 peak, "
            "bytes/HBM peak) / time with the measured peaks (FP4 = bf16 burst x 6)")
    if rank == 0:
        line["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baseline(args.workload)
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- CPU oracle
def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_step(workload: str, n_rows_sample: int):
    """One bounded sample of the workload through the CPU oracle (quantise both operands,
    dequantise, fp64 GEMM); returns (flops done, seconds, description)."""
    from oracle import gemm as ogemm
    from oracle import quant as oquant
    if workload in ("moe", "moe_nvfp4"):
        shapes = [(256, 1536, 2048), (256, 2048, 768)]     # one average expert, both GEMMs
        fmt = "MXFP4" if workload == "moe" else "NVFP4"
        desc = f"one 256-row expert of each MoE GEMM (gate+up 1536x2048, down 2048x768), {fmt}"
    elif workload == "prefill":
        shapes = [(64, n_rows_sample, k) for (_, n, k) in PREFILL]
        desc = f"64 activation rows x {n_rows_sample} weight rows of each prefill shape"
    elif workload == "e2e":
        shapes = [(m, n_rows_sample, 4096) for m in (256, 512)]
        desc = f"both e2e M, {n_rows_sample} of 14336 weight rows"
    elif workload == "pipeline":
        shapes = [(min(m, 64), n_rows_sample, 7168) for m in PIPE_MS]
        desc = f"one layer per pipeline M (at most 64 activation rows), {n_rows_sample} of 7168 weight rows, K=7168"
    else:
        shapes = [(m, n_rows_sample, 7168) for m in DECODE_MS]
        desc = f"all 8 decode M, {n_rows_sample} of 4096 weight rows, K=7168"
    flops = 0.0
    t0 = time.perf_counter()
    for i, (m, n, k) in enumerate(shapes):
        xa = synth.activation(i, m, k)
        xb = synth.weight(0, n, k)
        if workload == "moe":   # (moe_nvfp4 samples the NVFP4 path below)
            qa, sfa = oquant.mxfp4_quantize(xa)
            qb, sfb = oquant.mxfp4_quantize(xb)
            A = ogemm.dequantize(qa, sfa, m, k, 32, "ue8m0")
            B = ogemm.dequantize(qb, sfb, n, k, 32, "ue8m0")
            _ = A @ B.T
        else:
            gsa = np.float32(2688.0) / np.float32(xa.float().abs().max().item())
            gsb = np.float32(2688.0) / np.float32(xb.float().abs().max().item())
            qa, sfa = oquant.nvfp4_quantize(xa, gsa)
            qb, sfb = oquant.nvfp4_quantize(xb, gsb)
            _ = ogemm.nvfp4_gemm(qa, sfa, qb, sfb, np.float32(1.0) / (gsa * gsb), m, n, k)
        flops += 2.0 * m * n * k
    return flops, time.perf_counter() - t0, desc


def cpu_baseline(workload: str) -> dict:
    flops, secs, desc = oracle_step(workload, 1024)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOPS", "cores": _cores(), "kind": "oracle",
            "sample": desc + f" ({secs:.1f} s, numpy fp64)"}


def run_reference(args, rank):
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_step(args.workload, 128)
    total_f, total_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s, desc = oracle_step(args.workload, 128)
        total_f += f
        total_s += s
    v = total_f / total_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload} (bounded sample through the CPU oracle)", "sample": desc},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOPS", "cores": _cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(MAKERS), default="decode")
    ap.add_argument("--shapes", default="", help="custom quant->GEMM chain, e.g. '32,4096,7168;1024,4096,7168'")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg (profiling runs)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the per-configuration lines (decode, prefill, e2e, MoE GEMMs one by one)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3   # at least three untimed warm-up steps
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    dist_on = world > 1
    if dist_on:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    run_ours(args, dist_on, rank, world)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
