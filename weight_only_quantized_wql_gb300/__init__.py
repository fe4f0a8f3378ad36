"""Weight-only quantised lm_head logits on GB300 -- Python binding of libwql.

Thin ctypes wrappers with the C ABI's names (``include/wql.h``).  They only
marshal arguments: torch tensors supply device memory and the current CUDA
stream, and every step of the computation runs in libwql's CUDA kernels.
There is no CPU or PyTorch fallback: if the library cannot be loaded, or a
tensor is not on a CUDA device, the call raises.

Functions
  wql_quantize(w, bits, group, scale_dtype, clip, fmt=FMT_SYM) -> QuantizedWeight
  wql_pack(nibbles) / wql_unpack(packed, k)
  wql_workspace_size(m, n, topk)                    -> bytes
  wql_logits(x, qw, bias=None, topk=0, workspace=None, out=None,
             candidates_only=False)             -> (logits, topk_idx, topk_val)
  wql_topk_rescore(x, w_ref, topk_idx, topk_val, logits, bias=None)
  wql_embed_gather(ids, qw, out_dtype=torch.float16, out=None) -> [*ids.shape, k]
  wql_status_string, wql_last_error, wql_launch_count
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import _build

__all__ = [
    "WQLError", "QuantizedWeight", "Workspace", "load", "wql_quantize", "wql_pack",
    "wql_unpack", "wql_workspace_size", "wql_logits", "wql_logits_noalloc", "wql_topk_rescore",
    "wql_embed_gather", "wql_debug_set_waits",
    "wql_status_string", "wql_last_error", "wql_launch_count", "F32", "F16", "BF16",
    "CLIP_RTN", "CLIP_MSE", "MAX_TOPK", "NOALLOC_SCRATCH_BYTES", "FMT_SYM", "FMT_E4M3",
    "FMT_ASYM",
]

F32, F16, BF16 = 0, 1, 2
CLIP_RTN, CLIP_MSE = 0, 1
FMT_SYM, FMT_E4M3, FMT_ASYM = 0, 1, 2    # wql_format
WEIGHT_STATIC = 0x100                    # flag ORed into the format field
MAX_TOPK = 16
MAX_CTAS = 1024
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
_CODE_DTYPE = {v: k for k, v in _DTYPE_CODE.items()}
_STATUS = {0: "WQL_OK", 1: "WQL_EINVAL", 2: "WQL_EUNSUPPORTED", 3: "WQL_ECUDA",
           4: "WQL_EWORKSPACE"}

_lock = threading.Lock()
_lib = None


class WQLError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn} failed: {_STATUS.get(status, status)}"
        if status == 3 and _lib is not None:
            msg += f" ({_lib.wql_last_error().decode()})"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class _WqlWeight(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("scale_dtype", ctypes.c_int32), ("format", ctypes.c_int32),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libwql.so (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libwql.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        lib.wql_quantize.restype = i32
        lib.wql_quantize.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, vp, vp, vp]
        lib.wql_quantize_ex.restype = i32
        lib.wql_quantize_ex.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp,
                                        vp]
        lib.wql_pack.restype = i32
        lib.wql_pack.argtypes = [vp, i64, i64, vp, vp]
        lib.wql_unpack.restype = i32
        lib.wql_unpack.argtypes = [vp, i64, i64, vp, vp]
        lib.wql_workspace_size.restype = sz
        lib.wql_workspace_size.argtypes = [i64, i64, i32]
        lib.wql_logits.restype = i32
        lib.wql_logits.argtypes = [vp, i32, i64, ctypes.POINTER(_WqlWeight), vp, vp, i32, vp,
                                   vp, vp, sz, vp]
        lib.wql_logits_noalloc.restype = i32
        lib.wql_logits_noalloc.argtypes = [vp, i32, i64, ctypes.POINTER(_WqlWeight), vp, vp,
                                           i32, vp, vp, vp]
        lib.wql_topk_rescore.restype = i32
        lib.wql_topk_rescore.argtypes = [vp, i32, i64, vp, i32, i64, i64, vp, i32, vp, vp, vp,
                                         vp]
        lib.wql_embed_gather.restype = i32
        lib.wql_embed_gather.argtypes = [vp, i64, ctypes.POINTER(_WqlWeight), i32, vp, vp]
        lib.wql_status_string.restype = ctypes.c_char_p
        lib.wql_status_string.argtypes = [i32]
        lib.wql_last_error.restype = ctypes.c_char_p
        lib.wql_last_error.argtypes = []
        lib.wql_launch_count.restype = ctypes.c_uint64
        lib.wql_launch_count.argtypes = []
        lib.wql_debug_set_waits.restype = i32
        lib.wql_debug_set_waits.argtypes = [i64, i32]
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        raise WQLError(fn, status)


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device) -> ctypes.c_void_p:
    """torch's current CUDA stream on `device` (the raw handle, read the
    cheap way when this torch build offers it)."""
    if _raw_stream is not None:
        idx = device.index if device.index is not None else torch.cuda.current_device()
        return ctypes.c_void_p(_raw_stream(idx))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


@dataclass
class QuantizedWeight:
    """Packed weight + scale table, in the layout wql.h documents."""
    qweight: torch.Tensor      # int32 [n, k/8] (bits 4), int8 / uint8 e4m3 [n, k] (bits 8)
    scales: torch.Tensor       # fp16/bf16 [n, k/group] (or [n, 1])
    bits: int
    group: int                 # 0 = one scale per row
    n: int
    k: int
    fmt: int = FMT_SYM         # wql_format
    zeros: torch.Tensor | None = None   # uint8 [n, k/group] zero points (FMT_ASYM)
    static: bool = False       # WQL_WEIGHT_STATIC: never written after quantisation, so
                               # calls may read it before the preceding kernel ends

    @property
    def scale_dtype(self) -> int:
        return _DTYPE_CODE[self.scales.dtype]

    def _struct(self) -> _WqlWeight:
        # built once per (qweight, scales) storage; calls reuse it
        zp = self.zeros.data_ptr() if self.zeros is not None else None
        key = (self.qweight.data_ptr(), self.scales.data_ptr(), self.bits, self.group,
               self.n, self.k, self.scales.dtype, self.fmt, zp, self.static)
        cached = self.__dict__.get("_st")
        if cached is None or cached[0] != key:
            fmt = self.fmt | (WEIGHT_STATIC if self.static else 0)
            cached = (key, _WqlWeight(self.bits, self.group, self.scale_dtype, fmt,
                                      self.n, self.k, key[0], key[1], zp))
            self.__dict__["_st"] = cached
        return cached[1]

    def nbytes(self) -> int:
        z = self.zeros.numel() if self.zeros is not None else 0
        return self.qweight.numel() * self.qweight.element_size() + \
            self.scales.numel() * self.scales.element_size() + z


class Workspace:
    """Zero-initialised device scratch for wql_logits, grown on demand."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf

    def error_word(self) -> int:
        """The kernels' sticky error word (0 = no bounded wait ever timed out).
        Reads device memory, so it synchronises with the current stream."""
        if self.buf is None:
            return 0
        return int(self.buf[4:8].view(torch.int32).item())

    def clear_error(self) -> None:
        """Zero the sticky error word (ordered on the current stream)."""
        if self.buf is not None:
            self.buf[4:8].zero_()


_default_ws: dict = {}


def wql_status_string(status: int) -> str:
    return load().wql_status_string(status).decode()


def wql_last_error() -> str:
    return load().wql_last_error().decode()


def wql_launch_count() -> int:
    return int(load().wql_launch_count())


def wql_debug_set_waits(budget_cycles: int = 0, stall_mma: bool = False) -> None:
    """Diagnostics for the timeout path (see wql.h); (0, False) restores the
    defaults."""
    _check("wql_debug_set_waits", load().wql_debug_set_waits(budget_cycles, int(stall_mma)))


_ws_sizes: dict = {}


def wql_workspace_size(m: int, n: int, topk: int) -> int:
    key = (m, n, topk)
    v = _ws_sizes.get(key)
    if v is None:
        v = _ws_sizes[key] = int(load().wql_workspace_size(m, n, topk))
    return v


def wql_quantize(w: torch.Tensor, bits: int, group: int, scale_dtype=torch.float16,
                 clip: int = CLIP_RTN, fmt: int = FMT_SYM) -> QuantizedWeight:
    """Quantise + pack a [n, k] fp32/fp16/bf16 CUDA weight (see wql.h;
    fmt FMT_E4M3 / FMT_ASYM go through wql_quantize_ex)."""
    lib = load()
    _cuda(w, "w")
    n, k = w.shape
    g = k if group == 0 else group
    if bits == 4:
        qw = torch.empty((n, k // 8), dtype=torch.int32, device=w.device)
    elif fmt == FMT_E4M3:
        qw = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    else:
        qw = torch.empty((n, k), dtype=torch.int8, device=w.device)
    sc = torch.empty((n, k // g if g else 0), dtype=scale_dtype, device=w.device)
    zeros = None
    if fmt == FMT_ASYM:
        zeros = torch.empty((n, k // g if g else 0), dtype=torch.uint8, device=w.device)
    _check("wql_quantize_ex", lib.wql_quantize_ex(
        _ptr(w), _DTYPE_CODE[w.dtype], n, k, fmt, bits, group, _DTYPE_CODE[scale_dtype], clip,
        _ptr(qw), _ptr(sc), _ptr(zeros), _stream(w.device)))
    return QuantizedWeight(qw, sc, bits, group, n, k, fmt, zeros)


def wql_pack(nibbles: torch.Tensor) -> torch.Tensor:
    lib = load()
    _cuda(nibbles, "nibbles")
    n, k = nibbles.shape
    out = torch.empty((n, k // 8), dtype=torch.int32, device=nibbles.device)
    _check("wql_pack", lib.wql_pack(_ptr(nibbles), n, k, _ptr(out), _stream(nibbles.device)))
    return out


def wql_unpack(packed: torch.Tensor, k: int) -> torch.Tensor:
    lib = load()
    _cuda(packed, "packed")
    n = packed.shape[0]
    out = torch.empty((n, k), dtype=torch.uint8, device=packed.device)
    _check("wql_unpack", lib.wql_unpack(_ptr(packed), n, k, _ptr(out), _stream(packed.device)))
    return out


def default_workspace(device=None) -> Workspace:
    dev = torch.device(device or "cuda")
    return _default_ws.setdefault((dev, torch.cuda.current_stream(dev)), Workspace(dev))


def wql_logits(x: torch.Tensor, qw: QuantizedWeight, bias: torch.Tensor | None = None,
               topk: int = 0, workspace: Workspace | None = None,
               out: torch.Tensor | None = None, topk_idx: torch.Tensor | None = None,
               topk_val: torch.Tensor | None = None, candidates_only: bool = False):
    """logits [m, n] (x.dtype), and top-K (idx int32, val fp32) when topk > 0.

    x of any leading shape is flattened to [m, k] (radiance_lmhead_int4.py,
    apply()); the logits are returned with x's leading shape.  With
    candidates_only (topk > 0) no logits are written (logits_out NULL) and
    None is returned in their place."""
    lib = load()
    lead = x.shape[:-1]
    x2 = x.reshape(-1, x.shape[-1])
    _cuda(x2, "x")
    m = x2.shape[0]
    if candidates_only and topk <= 0:
        raise ValueError("candidates_only needs topk > 0")
    if out is None and not candidates_only:
        out = torch.empty((m, qw.n), dtype=x.dtype, device=x.device)
    if topk > 0:
        if topk_idx is None:
            topk_idx = torch.empty((m, topk), dtype=torch.int32, device=x.device)
        if topk_val is None:
            topk_val = torch.empty((m, topk), dtype=torch.float32, device=x.device)
    need = wql_workspace_size(m, qw.n, topk)
    if workspace is None:
        workspace = default_workspace(x.device)
    ws = workspace.get(need)
    st = qw._struct()
    _check("wql_logits", lib.wql_logits(
        _ptr(x2), _DTYPE_CODE[x.dtype], m, ctypes.byref(st), _ptr(bias), _ptr(out), topk,
        _ptr(topk_idx) if topk > 0 else None, _ptr(topk_val) if topk > 0 else None,
        _ptr(ws), ws.numel(), _stream(x.device)))
    logits = out.reshape(*lead, qw.n) if out is not None else None
    if topk > 0:
        return logits, topk_idx.reshape(*lead, topk), topk_val.reshape(*lead, topk)
    return logits, None, None


NOALLOC_SCRATCH_BYTES = 4 << 20    # WQL_NOALLOC_SCRATCH_BYTES


def wql_logits_noalloc(x: torch.Tensor, qw: QuantizedWeight, bias: torch.Tensor | None = None,
                       topk: int = 0, out: torch.Tensor | None = None,
                       topk_idx: torch.Tensor | None = None,
                       topk_val: torch.Tensor | None = None):
    """wql_logits through the entry point that takes no workspace: the library
    uses its own fixed device scratch area (WQL_NOALLOC_SCRATCH_BYTES per
    device), for callers that cannot provide device memory.  Pass `out`,
    `topk_idx` and `topk_val` to keep this call free of allocations too (any
    that is None is allocated here, by torch, before the library call).
    Calls on one device share the area and must not overlap."""
    lib = load()
    lead = x.shape[:-1]
    x2 = x.reshape(-1, x.shape[-1])
    _cuda(x2, "x")
    m = x2.shape[0]
    if out is None:
        out = torch.empty((m, qw.n), dtype=x.dtype, device=x.device)
    if topk > 0:
        if topk_idx is None:
            topk_idx = torch.empty((m, topk), dtype=torch.int32, device=x.device)
        if topk_val is None:
            topk_val = torch.empty((m, topk), dtype=torch.float32, device=x.device)
    st = qw._struct()
    status = lib.wql_logits_noalloc(
        _ptr(x2), _DTYPE_CODE[x.dtype], m, ctypes.byref(st), _ptr(bias), _ptr(out), topk,
        _ptr(topk_idx) if topk > 0 else None, _ptr(topk_val) if topk > 0 else None,
        _stream(x.device))
    if status == 4:
        need = wql_workspace_size(min(m, 16), qw.n, topk)
        raise WQLError("wql_logits_noalloc", status,
                       f"needs {need} bytes of scratch for 16-row slices with top-{topk}; "
                       f"the fixed area holds {NOALLOC_SCRATCH_BYTES}")
    _check("wql_logits_noalloc", status)
    logits = out.reshape(*lead, qw.n)
    if topk > 0:
        return logits, topk_idx.reshape(*lead, topk), topk_val.reshape(*lead, topk)
    return logits, None, None


def wql_topk_rescore(x: torch.Tensor, w_ref: torch.Tensor, topk_idx: torch.Tensor,
                     topk_val: torch.Tensor, logits: torch.Tensor,
                     bias: torch.Tensor | None = None) -> None:
    """In place: exact rescoring of the top-K candidates (see wql.h)."""
    lib = load()
    x2 = x.reshape(-1, x.shape[-1])
    for t, name in ((x2, "x"), (w_ref, "w_ref"), (topk_idx, "topk_idx"),
                    (topk_val, "topk_val"), (logits, "logits")):
        _cuda(t, name)
    m, k = x2.shape
    n = w_ref.shape[0]
    topk = topk_idx.shape[-1]
    _check("wql_topk_rescore", lib.wql_topk_rescore(
        _ptr(x2), _DTYPE_CODE[x.dtype], m, _ptr(w_ref), _DTYPE_CODE[w_ref.dtype], n, k,
        _ptr(bias), topk, _ptr(topk_idx), _ptr(topk_val), _ptr(logits), _stream(x.device)))


def wql_embed_gather(ids: torch.Tensor, qw: QuantizedWeight, out_dtype=torch.float16,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Dequantised rows of the tied head for token ids (see wql.h): returns
    [*ids.shape, k] of out_dtype; ids outside [0, n) give rows of zeros."""
    lib = load()
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    flat = ids.reshape(-1)
    _cuda(flat, "ids")
    t = flat.numel()
    if out is None:
        out = torch.empty((t, qw.k), dtype=out_dtype, device=ids.device)
    _cuda(out, "out")
    st = qw._struct()
    _check("wql_embed_gather", lib.wql_embed_gather(
        _ptr(flat), t, ctypes.byref(st), _DTYPE_CODE[out.dtype], _ptr(out), _stream(ids.device)))
    return out.reshape(*ids.shape, qw.k)
