"""GB300 (sm_103a) NVFP4 / MXFP4 block-scaled GEMM library -- Python binding of libnvfp4.so.

Thin ctypes marshalling over the C ABI in include/nvfp4.h: each function here has the name of
the C entry point it calls, takes torch CUDA tensors, allocates missing outputs with
torch.empty, checks what the library cannot see behind a bare pointer (device, dtype,
contiguity, size of every buffer), and passes raw pointers and the current CUDA stream.  All
arithmetic runs in the library's CUDA kernels; there is no CPU fallback.  Importing fails if
libnvfp4.so is missing (build it with ``python nvfp4_block_scaled_bf16_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnvfp4.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built: run `python nvfp4_block_scaled_bf16_gb300/build.py`")
_lib = ctypes.CDLL(_LIB_PATH)

_i64, _u32, _int, _vp, _sz = ctypes.c_int64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t

FLAG_PDL = 1 << 0
FLAG_SF_SM103 = 1 << 2
FLAG_DEBUG_TIMEOUT = 1 << 8
FLAG_DEBUG_SKIP_FIRST_LOAD = 1 << 9

STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_MISALIGNED",
          3: "NVFP4_ERR_UNSUPPORTED_SHAPE", 4: "NVFP4_ERR_UNSUPPORTED_DEVICE", 5: "NVFP4_ERR_CUDA",
          6: "NVFP4_ERR_TIMEOUT"}


class PlanT(ctypes.Structure):
    _fields_ = [("swap_ab", _int), ("tile_m", _int), ("tile_n", _int), ("splits", _int),
                ("stages", _int), ("ctas", _int), ("dp_tiles", _int), ("sk_tiles", _int)]


_SIGS = {
    "nvfp4_last_error": (ctypes.c_char_p, []),
    "nvfp4_sf_bytes": (_sz, [_i64, _i64, _int]),
    "mxfp4_grouped_sf_bytes": (_sz, [_i64, _int, _i64]),
    "nvfp4_quantize": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _u32, _vp]),
    "mxfp4_quantize": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _vp, _vp, _sz, _u32, _vp]),
    "nvfp4_gemm_plan": (_int, [_i64, _i64, _i64, ctypes.POINTER(PlanT)]),
    "nvfp4_gemm_workspace_size": (_int, [_i64, _i64, _i64, ctypes.POINTER(_sz)]),
    "nvfp4_gemm": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _u32, _vp]),
    "nvfp4_gemm_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _u32, _vp]),
    "nvfp4_quantize_gemm": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _u32, _vp]),
    "mxfp4_grouped_gemm": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _u32, _vp]),
    "sf_swizzle": (_int, [_vp, _vp, _i64, _i64, _int, _vp]),
    "nvfp4_sf_convert_layout": (_int, [_vp, _vp, _i64, _i64, _int, _vp]),
    "moe_sort_workspace_size": (_sz, [_i64, _int]),
    "moe_sort_by_expert": (_int, [_vp, _i64, _int, _int, _vp, _vp, _vp, _vp, _sz, _u32, _vp]),
    "moe_gather_rows": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _u32, _vp]),
    "nvfp4_quantize_experts": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _vp, _vp, _vp, _sz, _u32, _vp]),
    "nvfp4_gather_quantize_experts": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _int, _vp, _vp, _vp, _sz, _u32,
                                             _vp]),
    "nvfp4_silu_mul_quantize_experts": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _vp, _vp, _vp, _sz, _u32, _vp]),
    "nvfp4_grouped_gemm": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _u32, _vp]),
    "moe_combine": (_int, [_vp, _i64, _vp, _vp, _i64, _int, _i64, _vp, _u32, _vp]),
    "nvfp4_check_status": (_int, [_vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

lib = _lib  # raw ctypes handle (tests call entry points through it directly)
LIB_PATH = _LIB_PATH


class NVFP4Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


def last_error() -> str:
    return _lib.nvfp4_last_error().decode()


def _check(code: int) -> None:
    if code != 0:
        raise NVFP4Error(code, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_device(t, name):
    """The library launches on the current CUDA device; every tensor must live there."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    cur = torch.cuda.current_device()
    if t.get_device() != cur:
        raise ValueError(f"{name} is on cuda:{t.get_device()}, the current device is cuda:{cur}")


def _need(t, dtype, name, dim=None):
    _check_device(t, name)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions")


def _room(t, dtype, name, numel):
    """A buffer the kernels read or write `numel` elements of, densely from its first element (the
    library sees only the pointer, so its size is checked here)."""
    _need(t, dtype, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")


def _contig(t, stream):
    """`t` with dense rows.  A copy is made on the launch stream, so that the caching allocator
    cannot hand its memory out again before that stream's kernel has read it."""
    if t.is_contiguous():
        return t
    if stream is None:
        return t.contiguous()
    s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(stream)
    with torch.cuda.stream(s):
        return t.contiguous()


def sf_bytes(rows: int, k: int, sf_vec: int = 16) -> int:
    """Bytes of a 128x4-swizzled scale buffer: round_up(rows,128) * round_up(k/sf_vec, 4)."""
    return int(_lib.nvfp4_sf_bytes(rows, k, sf_vec))


def grouped_sf_bytes(total_rows: int, experts: int, k: int) -> int:
    return int(_lib.mxfp4_grouped_sf_bytes(total_rows, experts, k))


def nvfp4_gemm_plan(m: int, n: int, k: int) -> dict:
    p = PlanT()
    _check(_lib.nvfp4_gemm_plan(m, n, k, ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in PlanT._fields_}


def gemm_workspace_size(m: int, n: int, k: int) -> int:
    """Bytes of workspace nvfp4_gemm needs for (m, n, k) on the current device."""
    v = _sz(0)
    _check(_lib.nvfp4_gemm_workspace_size(m, n, k, ctypes.byref(v)))
    return int(v.value)


def gemm_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 workspace of at least nbytes (the library needs it zero before first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


_ws_cache: dict = {}


def _default_workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """One zeroed workspace per device, grown on demand and shared by every nvfp4_gemm call that
    passes none.  Calls on streams that may overlap must pass their own workspace."""
    ws = _ws_cache.get(device)
    if ws is None or ws.numel() < nbytes:
        ws = gemm_workspace(nbytes, device)
        _ws_cache[device] = ws
    return ws


def nvfp4_quantize(x, gs, q=None, sf=None, flags: int = 0, stream=None):
    """bf16 [m, k] -> (packed e2m1 uint8 [m, k/2], swizzled e4m3 scales uint8 [sf_bytes])."""
    _need(x, torch.bfloat16, "x", 2)
    _need(gs, torch.float32, "gs")
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    m, k = x.shape
    if q is None:
        q = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(sf_bytes(m, k, 16), dtype=torch.uint8, device=x.device)
    _room(q, torch.uint8, "q", m * (k // 2))
    _room(sf, torch.uint8, "sf", sf_bytes(m, k, 16))
    _check(_lib.nvfp4_quantize(_ptr(x), m, k, x.stride(0), _ptr(gs), _ptr(q), _ptr(sf), flags, _stream(stream)))
    return q, sf


def mxfp4_quantize(x, row_offsets=None, q=None, sf=None, flags: int = 0, stream=None):
    """bf16 [t, k] -> (packed e2m1 [t, k/2], ue8m0 scales); grouped per expert with row_offsets [E+1]."""
    _need(x, torch.bfloat16, "x", 2)
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    t, k = x.shape
    experts = 0
    if row_offsets is not None:
        _need(row_offsets, torch.int64, "row_offsets", 1)
        experts = row_offsets.numel() - 1
    need = grouped_sf_bytes(t, experts, k) if row_offsets is not None else sf_bytes(t, k, 32)
    if q is None:
        q = torch.empty((t, k // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.zeros(need, dtype=torch.uint8, device=x.device)
    _room(q, torch.uint8, "q", t * (k // 2))
    _room(sf, torch.uint8, "sf", 0)            # its capacity goes to the library, which checks it
    _check(_lib.mxfp4_quantize(_ptr(x), t, k, x.stride(0), _ptr(row_offsets), experts, _ptr(q), _ptr(sf),
                               sf.numel(), flags, _stream(stream)))
    return q, sf


def nvfp4_gemm(a, sfa, b, sfb, alpha, d=None, flags: int = 0, stream=None, workspace=None):
    """D[m, n] = bf16(alpha * deq(a) @ deq(b)^T); a [m, k/2], b [n, k/2] packed uint8.

    workspace: zero-filled uint8 CUDA tensor of at least gemm_workspace_size(m, n, k) bytes
    (the library leaves it zero after each call); None uses a per-device shared one."""
    _need(a, torch.uint8, "a", 2)
    _need(b, torch.uint8, "b", 2)
    _need(sfa, torch.uint8, "sfa")
    _need(sfb, torch.uint8, "sfb")
    _need(alpha, torch.float32, "alpha")
    m, kh = a.shape
    n = b.shape[0]
    if b.shape[1] != kh:
        raise ValueError("a and b disagree on K")
    for t_, name in ((a, "a"), (b, "b")):
        if not t_.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if sfa.numel() < sf_bytes(m, 2 * kh) or sfb.numel() < sf_bytes(n, 2 * kh):
        raise ValueError("scale buffers are too small")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _room(d, torch.bfloat16, "d", m * n)
    if workspace is None and m > 0:
        need = gemm_workspace_size(m, n, 2 * kh)
        if need:
            workspace = _default_workspace(need, a.device)
    if workspace is not None:
        _room(workspace, torch.uint8, "workspace", 0)   # the library checks its size
    _check(_lib.nvfp4_gemm(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(alpha), _ptr(d), m, n, 2 * kh,
                           _ptr(workspace), 0 if workspace is None else workspace.numel(), flags,
                           _stream(stream)))
    return d


def nvfp4_quantize_gemm(x, gs, b, sfb, alpha, d=None, flags: int = 0, stream=None):
    """nvfp4_gemm(*nvfp4_quantize(x, gs), b, sfb, alpha) in one kernel (1 <= m <= 256): x bf16
    [m, k] with contiguous rows, b [n, k/2] packed uint8; bit-identical to the two calls."""
    _need(x, torch.bfloat16, "x", 2)
    _need(gs, torch.float32, "gs")
    _need(b, torch.uint8, "b", 2)
    _need(sfb, torch.uint8, "sfb")
    _need(alpha, torch.float32, "alpha")
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    if not b.is_contiguous():
        raise ValueError("b must be contiguous")
    m, k = x.shape
    n = b.shape[0]
    if b.shape[1] * 2 != k:
        raise ValueError("x and b disagree on K")
    if sfb.numel() < sf_bytes(n, k):
        raise ValueError("sfb is too small")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _room(d, torch.bfloat16, "d", m * n)
    _check(_lib.nvfp4_quantize_gemm(_ptr(x), x.stride(0), _ptr(gs), _ptr(b), _ptr(sfb), _ptr(alpha), _ptr(d), m, n, k,
                                    None, 0, flags, _stream(stream)))
    return d


def nvfp4_gemm_noalloc(a, sfa, b, sfb, alpha, d=None, flags: int = 0, stream=None):
    """nvfp4_gemm with the library's static split-K scratch instead of a workspace (never
    allocates on the device beyond the output when d is None).  Not for concurrent use."""
    _need(a, torch.uint8, "a", 2)
    _need(b, torch.uint8, "b", 2)
    _need(sfa, torch.uint8, "sfa")
    _need(sfb, torch.uint8, "sfb")
    _need(alpha, torch.float32, "alpha")
    m, kh = a.shape
    n = b.shape[0]
    if b.shape[1] != kh:
        raise ValueError("a and b disagree on K")
    for t_, name in ((a, "a"), (b, "b")):
        if not t_.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if sfa.numel() < sf_bytes(m, 2 * kh) or sfb.numel() < sf_bytes(n, 2 * kh):
        raise ValueError("scale buffers are too small")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _room(d, torch.bfloat16, "d", m * n)
    _check(_lib.nvfp4_gemm_noalloc(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(alpha), _ptr(d), m, n, 2 * kh,
                                   flags, _stream(stream)))
    return d


def mxfp4_grouped_gemm(a, sfa, row_offsets, b, sfb, alpha=None, d=None, flags: int = 0, stream=None):
    """Per expert e: D[rows of e] = bf16(alpha * deq(A_e) @ deq(B_e)^T); b [E, n, k/2]."""
    _need(a, torch.uint8, "a", 2)
    _need(b, torch.uint8, "b", 3)
    _need(row_offsets, torch.int64, "row_offsets", 1)
    t, kh = a.shape
    experts, n, kb = b.shape
    if kb != kh or row_offsets.numel() != experts + 1:
        raise ValueError("shape mismatch")
    if not b.is_contiguous():
        raise ValueError("b must be contiguous")
    _need(sfa, torch.uint8, "sfa")
    _room(sfb, torch.uint8, "sfb", experts * sf_bytes(n, 2 * kh, 32))
    if alpha is not None:
        _room(alpha, torch.float32, "alpha", 1)
    if d is None:
        d = torch.empty((t, n), dtype=torch.bfloat16, device=a.device)
    _room(d, torch.bfloat16, "d", t * n)
    _check(_lib.mxfp4_grouped_gemm(_ptr(a), _ptr(sfa), _ptr(row_offsets), experts, _ptr(b), _ptr(sfb),
                                   _ptr(alpha), _ptr(d), t, n, 2 * kh, flags, _stream(stream)))
    return d


def sf_swizzle(src, rows: int, cols: int, to_swizzled: bool = True, dst=None, stream=None):
    """Row-major scale bytes [rows, cols] <-> 128x4 swizzled buffer."""
    padded = (-(-rows // 128) * 128) * (-(-cols // 4) * 4)
    _room(src, torch.uint8, "src", rows * cols if to_swizzled else padded)
    if dst is None:
        dst = torch.empty(padded if to_swizzled else rows * cols, dtype=torch.uint8, device=src.device)
    _room(dst, torch.uint8, "dst", padded if to_swizzled else rows * cols)
    _check(_lib.sf_swizzle(_ptr(src), _ptr(dst), rows, cols, 1 if to_swizzled else 0, _stream(stream)))
    return dst


def sf_convert_layout(src, rows: int, cols: int, to_sm103: bool = True, dst=None, stream=None):
    """Swizzled NVFP4 scale buffer: 128x4 ("SM100") layout <-> SM103 layout."""
    padded = (-(-rows // 128) * 128) * (-(-cols // 4) * 4)
    _room(src, torch.uint8, "src", padded)
    if dst is None:
        dst = torch.empty_like(src)
    _room(dst, torch.uint8, "dst", padded)
    _check(_lib.nvfp4_sf_convert_layout(_ptr(src), _ptr(dst), rows, cols, 1 if to_sm103 else 0, _stream(stream)))
    return dst


# ---------------------------------------------------------------- MoE steps (NVFP4)
def expert_sf_bytes(total_rows: int, experts: int, k: int) -> int:
    """Grouped NVFP4 scale buffer bound: (round_up(t,128) + 128 E) * round_up(k/16, 4)."""
    return (-(-total_rows // 128) * 128 + 128 * experts) * (-(-(k // 16) // 4) * 4)


def moe_sort_workspace_size(num_tokens: int, num_experts: int) -> int:
    return int(_lib.moe_sort_workspace_size(num_tokens, num_experts))


def moe_sort_by_expert(topk_ids, num_experts: int, out=None, workspace=None, flags: int = 0, stream=None):
    """int32 [T, topk] expert ids -> (row_offsets int64 [E+1], src_rows int32 [T*topk],
    pos int32 [T, topk]); stable: (token, slot) order inside an expert.  `out` may pass the
    three output tensors to fill."""
    _need(topk_ids, torch.int32, "topk_ids", 2)
    topk_ids = _contig(topk_ids, stream)
    T, topk = topk_ids.shape
    dv = topk_ids.device
    if out is None:
        out = (torch.empty(num_experts + 1, dtype=torch.int64, device=dv),
               torch.empty(T * topk, dtype=torch.int32, device=dv),
               torch.empty((T, topk), dtype=torch.int32, device=dv))
    ro, src, pos = out
    _room(ro, torch.int64, "row_offsets", num_experts + 1)
    _room(src, torch.int32, "src_rows", T * topk)
    _room(pos, torch.int32, "pos", T * topk)
    if workspace is None:
        workspace = torch.empty(max(1, moe_sort_workspace_size(T, num_experts) // 4), dtype=torch.int32, device=dv)
    _room(workspace, torch.int32, "workspace", 0)        # its size in bytes goes to the library
    _check(_lib.moe_sort_by_expert(_ptr(topk_ids), T, topk, num_experts, _ptr(ro), _ptr(src), _ptr(pos),
                                   _ptr(workspace), workspace.numel() * 4, flags, _stream(stream)))
    return ro, src, pos


def moe_gather_rows(x, src_rows, out=None, flags: int = 0, stream=None):
    """out[r] = x[src_rows[r]] (bf16 rows)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(src_rows, torch.int32, "src_rows", 1)
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    T, h = x.shape
    rows = src_rows.numel()
    if out is None:
        out = torch.empty((rows, h), dtype=torch.bfloat16, device=x.device)
    if not src_rows.is_contiguous():
        raise ValueError("src_rows must be contiguous")
    _room(out, torch.bfloat16, "out", rows * h)
    _check(_lib.moe_gather_rows(_ptr(x), T, h, x.stride(0), _ptr(src_rows), rows, _ptr(out), flags, _stream(stream)))
    return out


def nvfp4_quantize_experts(x, row_offsets, gs, q=None, sf=None, flags: int = 0, stream=None):
    """bf16 [t, k] (rows by expert) -> (packed e2m1 [t, k/2], grouped e4m3 scales); gs fp32 [E]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(row_offsets, torch.int64, "row_offsets", 1)
    _need(gs, torch.float32, "gs", 1)
    t, k = x.shape
    experts = row_offsets.numel() - 1
    if q is None:
        q = torch.empty((t, k // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(expert_sf_bytes(t, experts, k), dtype=torch.uint8, device=x.device)
    _room(row_offsets, torch.int64, "row_offsets", experts + 1)
    _room(gs, torch.float32, "gs", experts)
    _room(q, torch.uint8, "q", t * (k // 2))
    _room(sf, torch.uint8, "sf", 0)            # its capacity goes to the library, which checks it
    _check(_lib.nvfp4_quantize_experts(_ptr(x), t, k, x.stride(0), _ptr(row_offsets), experts, _ptr(gs), _ptr(q),
                                       _ptr(sf), sf.numel(), flags, _stream(stream)))
    return q, sf


def nvfp4_gather_quantize_experts(x, src_rows, row_offsets, gs, q=None, sf=None, flags: int = 0, stream=None):
    """Row r of the result quantises x[src_rows[r]]: moe_gather_rows + nvfp4_quantize_experts in one launch."""
    _need(x, torch.bfloat16, "x", 2)
    _need(src_rows, torch.int32, "src_rows", 1)
    _need(row_offsets, torch.int64, "row_offsets", 1)
    _need(gs, torch.float32, "gs", 1)
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    if not src_rows.is_contiguous():
        raise ValueError("src_rows must be contiguous")
    tokens, k = x.shape
    rows = src_rows.numel()
    experts = row_offsets.numel() - 1
    if q is None:
        q = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(expert_sf_bytes(rows, experts, k), dtype=torch.uint8, device=x.device)
    _room(row_offsets, torch.int64, "row_offsets", experts + 1)
    _room(gs, torch.float32, "gs", experts)
    _room(q, torch.uint8, "q", rows * (k // 2))
    _room(sf, torch.uint8, "sf", 0)            # its capacity goes to the library, which checks it
    _check(_lib.nvfp4_gather_quantize_experts(_ptr(x), tokens, k, x.stride(0), _ptr(src_rows), rows,
                                              _ptr(row_offsets), experts, _ptr(gs), _ptr(q), _ptr(sf), sf.numel(),
                                              flags, _stream(stream)))
    return q, sf


def nvfp4_silu_mul_quantize_experts(x, row_offsets, gs, q=None, sf=None, flags: int = 0, stream=None):
    """bf16 [t, 2I] = [gate | up] -> NVFP4 of h = bf16(silu(gate) * up): (q [t, I/2], grouped scales)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(row_offsets, torch.int64, "row_offsets", 1)
    _need(gs, torch.float32, "gs", 1)
    t, w = x.shape
    inter = w // 2
    experts = row_offsets.numel() - 1
    if q is None:
        q = torch.empty((t, inter // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(expert_sf_bytes(t, experts, inter), dtype=torch.uint8, device=x.device)
    _room(row_offsets, torch.int64, "row_offsets", experts + 1)
    _room(gs, torch.float32, "gs", experts)
    _room(q, torch.uint8, "q", t * (inter // 2))
    _room(sf, torch.uint8, "sf", 0)
    _check(_lib.nvfp4_silu_mul_quantize_experts(_ptr(x), t, inter, x.stride(0), _ptr(row_offsets), experts, _ptr(gs),
                                                _ptr(q), _ptr(sf), sf.numel(), flags, _stream(stream)))
    return q, sf


def nvfp4_grouped_gemm(a, sfa, row_offsets, b, sfb, alpha=None, d=None, flags: int = 0, stream=None):
    """Per expert e: D[rows of e] = bf16(alpha[e] * deq(A_e) @ deq(B_e)^T); b [E, n, k/2], alpha fp32 [E]."""
    _need(a, torch.uint8, "a", 2)
    _need(b, torch.uint8, "b", 3)
    _need(row_offsets, torch.int64, "row_offsets", 1)
    t, kh = a.shape
    experts, n, kb = b.shape
    if kb != kh or row_offsets.numel() != experts + 1 or (alpha is not None and alpha.numel() != experts):
        raise ValueError("shape mismatch")
    if not b.is_contiguous():
        raise ValueError("b must be contiguous")
    _need(sfa, torch.uint8, "sfa")
    _room(sfb, torch.uint8, "sfb", experts * sf_bytes(n, 2 * kh, 16))
    if alpha is not None:
        _room(alpha, torch.float32, "alpha", experts)
    if d is None:
        d = torch.empty((t, n), dtype=torch.bfloat16, device=a.device)
    _room(d, torch.bfloat16, "d", t * n)
    _check(_lib.nvfp4_grouped_gemm(_ptr(a), _ptr(sfa), _ptr(row_offsets), experts, _ptr(b), _ptr(sfb), _ptr(alpha),
                                   _ptr(d), t, n, 2 * kh, flags, _stream(stream)))
    return d


def moe_combine(y, pos, weights, out=None, flags: int = 0, stream=None):
    """out[t] = bf16(sum_j weights[t, j] * y[pos[t, j]]) (fp32, slot order)."""
    _need(y, torch.bfloat16, "y", 2)
    _need(pos, torch.int32, "pos", 2)
    _need(weights, torch.float32, "weights", 2)
    if not y.is_contiguous():
        raise ValueError("y must be contiguous")
    rows, h = y.shape
    T, topk = pos.shape
    if tuple(weights.shape) != (T, topk):
        raise ValueError(f"weights must have shape {(T, topk)}, got {tuple(weights.shape)}")
    pos, weights = _contig(pos, stream), _contig(weights, stream)
    if out is None:
        out = torch.empty((T, h), dtype=torch.bfloat16, device=y.device)
    _room(out, torch.bfloat16, "out", T * h)
    _check(_lib.moe_combine(_ptr(y), rows, _ptr(pos), _ptr(weights), T, topk, h, _ptr(out),
                            flags, _stream(stream)))
    return out


def check_status(stream=None) -> None:
    """Raise NVFP4Error(TIMEOUT) if a kernel gave up a bounded wait since the last check."""
    _check(_lib.nvfp4_check_status(_stream(stream)))
