"""CPU oracle for the weight-only quantised lm_head path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library
(``weight_only_quantized_wql_gb300``) never imports it, and this package
imports nothing from the product.

The arithmetic lives in ``wql_oracle.c`` (plain C, binary64 accumulation,
built with ``-ffp-contract=off``); this module builds it with gcc and wraps
it with numpy arrays.  Each wrapper names the page section it follows:

* ``quantize``   -- radiance_lmhead_int4.py, ``quantize_int4_rows`` and its
  module constants (QMAX 7, nibble bias 8, clip ratios 1.0..0.8, bf16 scale
  rounded before q is chosen); int8 per "Fused WNA16 GEMM for tied quantized
  lm_head logits", Perf-evals rows W8-g128 and reviewer comment item 1.
* ``pack_int4`` / ``unpack_int4`` -- same page, Purpose ("packed along the
  input/hidden dim"), [N, K/8] int32 words; the in-word order is this
  library's: element 8i+j in nibble 4*(j%2) + j//2 of word i (even elements
  in bits 0..15, odd elements in bits 16..31).
* ``logits``     -- same page, Purpose: logits = X . dequant(Wq)^T, the dense
  weight never needed; binary64, k ascending.
* ``topk`` / ``rescore`` -- same page, reviewer comment item 2.
* ``embed_gather`` -- same page, Purpose (tied head: a token's input
  embedding is that row of the dequantised weight), rounded once to
  fp16 / bf16.
* ``e4m3_*``, ``quantize_fp8``, ``logits_fp8`` -- the per-channel fp8 head
  that radiance_lmhead_int4.py's module docstring compares against: e4m3
  from the format's definition, a per-row scale rounded before the codes
  are chosen, binary64 logits.
* ``quantize_asym_int4`` / ``logits_asym_int4`` -- zero-point int4 ("[CORE]
  Quantized lm-head Framework": the test model's lm_head uses sym=False):
  plain asymmetric round-to-nearest per group, w ~ (q - z) * s.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wql_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
CLIP_RATIOS = (1.0, 0.95, 0.9, 0.85, 0.8)


def build(force: bool = False) -> str:
    """Compile ``wql_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_quantize.restype = i32
        lib.oracle_quantize.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, vp, vp, vp, i32]
        lib.oracle_pack_int4.restype = i32
        lib.oracle_pack_int4.argtypes = [vp, i64, i64, vp]
        lib.oracle_pack_codes_int4.restype = i32
        lib.oracle_pack_codes_int4.argtypes = [vp, i64, i64, vp]
        lib.oracle_unpack_int4.restype = i32
        lib.oracle_unpack_int4.argtypes = [vp, i64, i64, vp]
        lib.oracle_logits.restype = i32
        lib.oracle_logits.argtypes = [vp, i32, i64, i64, vp, i32, vp, i32, i32, i64,
                                      vp, i32, vp, i64, vp, vp, i32]
        lib.oracle_topk.restype = i32
        lib.oracle_topk.argtypes = [vp, i64, i64, i32, vp, vp]
        lib.oracle_embed_gather.restype = i32
        lib.oracle_embed_gather.argtypes = [vp, i64, vp, i32, vp, i32, i64, i64, i64, i32, vp]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_f64_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_quantize_fp8.restype = i32
        lib.oracle_quantize_fp8.argtypes = [vp, i32, i64, i64, i32, vp, vp]
        lib.oracle_logits_fp8.restype = i32
        lib.oracle_logits_fp8.argtypes = [vp, i32, i64, i64, vp, vp, i32, i64, vp, vp]
        lib.oracle_quantize_asym_int4.restype = i32
        lib.oracle_quantize_asym_int4.argtypes = [vp, i32, i64, i64, i32, i32, vp, vp, vp]
        lib.oracle_logits_asym_int4.restype = i32
        lib.oracle_logits_asym_int4.argtypes = [vp, i32, i64, i64, vp, vp, vp, i32, i32, i64,
                                                vp, vp]
        lib.oracle_rescore.restype = i32
        lib.oracle_rescore.argtypes = [vp, i32, i64, i64, vp, i32, i64, vp, i32, vp, i32, vp, vp]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _as_bits(a: np.ndarray, dtype_code: int) -> np.ndarray:
    """fp32 arrays pass as float32; fp16/bf16 arrays pass as their uint16 bits."""
    if dtype_code == F32:
        assert a.dtype == np.float32
        return np.ascontiguousarray(a)
    assert a.dtype in (np.uint16, np.int16, np.float16), a.dtype
    return np.ascontiguousarray(a).view(np.uint16)


# --- scalar conversions (IEEE round-to-nearest-even, from the definitions) ---

def f32_to_f16_bits(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_f16(float(x)) for x in v], dtype=np.uint16)


def f32_to_bf16_bits(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(x)) for x in v], dtype=np.uint16)


def f16_bits_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f64(int(x)) for x in b], dtype=np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_f64(int(x)) for x in b], dtype=np.float64)


def scales_to_f64(bits: np.ndarray, scale_dtype: int) -> np.ndarray:
    conv = f16_bits_to_f64 if scale_dtype == F16 else bf16_bits_to_f64
    return conv(bits).reshape(np.shape(bits))


# --- quantiser, packing ----------------------------------------------------

def quantize(w: np.ndarray, w_dtype: int, bits: int, group: int, scale_dtype: int,
             clip: int, nthreads: int = 1):
    """Returns (q int8 [n,k] signed codes, scale bits uint16 [n, k/G], ratio idx int8)."""
    lib = _load()
    n, k = w.shape
    g = k if group == 0 else group
    wb = _as_bits(w, w_dtype)
    q = np.empty((n, k), dtype=np.int8)
    s = np.empty((n, k // g), dtype=np.uint16)
    r = np.empty((n, k // g), dtype=np.int8)
    rc = lib.oracle_quantize(_ptr(wb), w_dtype, n, k, bits, group, scale_dtype, clip,
                             _ptr(q), _ptr(s), _ptr(r), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_quantize rejected its arguments")
    return q, s, r


def quantize_packed(w: np.ndarray, w_dtype: int, bits: int, group: int, scale_dtype: int,
                    clip: int, nthreads: int = 1):
    """(qweight in the library layout, scale bits): int4 packed words or int8 codes."""
    q, s, _ = quantize(w, w_dtype, bits, group, scale_dtype, clip, nthreads)
    if bits == 4:
        n, k = q.shape
        out = np.empty((n, k // 8), dtype=np.uint32)
        if _load().oracle_pack_codes_int4(_ptr(q), n, k, _ptr(out)) != 0:
            raise ValueError("k must be a multiple of 8")
        return out.view(np.int32), s
    return q, s


def pack_int4(nibbles: np.ndarray) -> np.ndarray:
    """uint8 nibbles [n,k] in 0..15 -> int32 words [n, k/8]."""
    lib = _load()
    nib = np.ascontiguousarray(nibbles, dtype=np.uint8)
    n, k = nib.shape
    out = np.empty((n, k // 8), dtype=np.uint32)
    if lib.oracle_pack_int4(_ptr(nib), n, k, _ptr(out)) != 0:
        raise ValueError("k must be a multiple of 8")
    return out.view(np.int32)


def unpack_int4(packed: np.ndarray, k: int) -> np.ndarray:
    lib = _load()
    p = np.ascontiguousarray(packed).view(np.uint32)
    n = p.shape[0]
    out = np.empty((n, k), dtype=np.uint8)
    if lib.oracle_unpack_int4(_ptr(p), n, k, _ptr(out)) != 0:
        raise ValueError("k must be a multiple of 8")
    return out


# --- logits, top-K, rescoring ----------------------------------------------

def logits(x: np.ndarray, x_dtype: int, qweight: np.ndarray, bits: int,
           scales: np.ndarray, scale_dtype: int, group: int, n: int, k: int,
           bias: np.ndarray | None = None, rows: np.ndarray | None = None,
           nthreads: int = 1):
    """binary64 logits [m, len(rows) or n] and the matching sum |x*w| (A)."""
    lib = _load()
    xb = _as_bits(x, x_dtype)
    m = xb.shape[0]
    qw = np.ascontiguousarray(qweight)
    sc = np.ascontiguousarray(scales).view(np.uint16)
    bb = None if bias is None else _as_bits(bias, x_dtype)
    rr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = n if rr is None else rr.shape[0]
    out = np.empty((m, nrows), dtype=np.float64)
    absout = np.empty((m, nrows), dtype=np.float64)
    rc = lib.oracle_logits(_ptr(xb), x_dtype, m, k, _ptr(qw), bits, _ptr(sc), scale_dtype,
                           group, n, _ptr(bb), x_dtype, _ptr(rr), nrows, _ptr(out),
                           _ptr(absout), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_logits rejected its arguments")
    return out, absout


def topk(vals: np.ndarray, K: int):
    """Top-K per row of a float64 [m, n] array: value desc, index asc."""
    lib = _load()
    v = np.ascontiguousarray(vals, dtype=np.float64)
    m, n = v.shape
    idx = np.empty((m, K), dtype=np.int32)
    val = np.empty((m, K), dtype=np.float64)
    if lib.oracle_topk(_ptr(v), m, n, K, _ptr(idx), _ptr(val)) != 0:
        raise ValueError("bad K")
    return idx, val


def rescore(x: np.ndarray, x_dtype: int, wref: np.ndarray, wref_dtype: int,
            idx: np.ndarray, bias: np.ndarray | None = None):
    """binary64 dot of x rows with the reference-weight rows named in idx."""
    lib = _load()
    xb = _as_bits(x, x_dtype)
    wb = _as_bits(wref, wref_dtype)
    m, k = xb.shape
    n = wb.shape[0]
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    K = ii.shape[1]
    bb = None if bias is None else _as_bits(bias, x_dtype)
    out = np.empty((m, K), dtype=np.float64)
    absout = np.empty((m, K), dtype=np.float64)
    rc = lib.oracle_rescore(_ptr(xb), x_dtype, m, k, _ptr(wb), wref_dtype, n, _ptr(ii), K,
                            _ptr(bb), x_dtype, _ptr(out), _ptr(absout))
    if rc != 0:
        raise ValueError("oracle_rescore: index out of range")
    return out, absout


def embed_gather(ids: np.ndarray, qweight: np.ndarray, bits: int, scales: np.ndarray,
                 scale_dtype: int, group: int, n: int, k: int, out_dtype: int) -> np.ndarray:
    """uint16 bits [t, k] of RN_out(q * s) for rows ids (ids outside [0, n): +0)."""
    lib = _load()
    ii = np.ascontiguousarray(ids, dtype=np.int32).ravel()
    qw = np.ascontiguousarray(qweight)
    sc = np.ascontiguousarray(scales).view(np.uint16)
    g = k if group == 0 else group
    out = np.empty((ii.shape[0], k), dtype=np.uint16)
    rc = lib.oracle_embed_gather(_ptr(ii), ii.shape[0], _ptr(qw), bits, _ptr(sc), scale_dtype,
                                 g, n, k, out_dtype, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_embed_gather rejected its arguments")
    return out


def e4m3_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_f64(int(v)) for v in b], dtype=np.float64)


def f64_to_e4m3(values) -> np.ndarray:
    """Round to e4m3 (ties to even), saturating at +-448; NaN -> 0x7F."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib.oracle_f64_to_e4m3(float(x)) for x in v], dtype=np.uint8)


def quantize_fp8(w: np.ndarray, w_dtype: int, scale_dtype: int):
    """(e4m3 codes uint8 [n, k], per-row scale bits uint16 [n])."""
    lib = _load()
    n, k = w.shape
    wb = _as_bits(w, w_dtype)
    q = np.empty((n, k), dtype=np.uint8)
    s = np.empty(n, dtype=np.uint16)
    if lib.oracle_quantize_fp8(_ptr(wb), w_dtype, n, k, scale_dtype, _ptr(q), _ptr(s)) != 0:
        raise ValueError("oracle_quantize_fp8 rejected its arguments")
    return q, s


def logits_fp8(x: np.ndarray, x_dtype: int, q: np.ndarray, scales: np.ndarray,
               scale_dtype: int):
    """binary64 logits [m, n] of the fp8 head and the matching sum |x*w|."""
    lib = _load()
    xb = _as_bits(x, x_dtype)
    m, k = xb.shape
    qq = np.ascontiguousarray(q, dtype=np.uint8)
    n = qq.shape[0]
    sc = np.ascontiguousarray(scales).view(np.uint16)
    out = np.empty((m, n), dtype=np.float64)
    absout = np.empty((m, n), dtype=np.float64)
    lib.oracle_logits_fp8(_ptr(xb), x_dtype, m, k, _ptr(qq), _ptr(sc), scale_dtype, n,
                          _ptr(out), _ptr(absout))
    return out, absout


def quantize_asym_int4(w: np.ndarray, w_dtype: int, group: int, scale_dtype: int):
    """(codes uint8 [n, k] in 0..15, scale bits uint16 [n, k/G], zero points uint8 [n, k/G])."""
    lib = _load()
    n, k = w.shape
    wb = _as_bits(w, w_dtype)
    q = np.empty((n, k), dtype=np.uint8)
    s = np.empty((n, k // group), dtype=np.uint16)
    z = np.empty((n, k // group), dtype=np.uint8)
    if lib.oracle_quantize_asym_int4(_ptr(wb), w_dtype, n, k, group, scale_dtype, _ptr(q),
                                     _ptr(s), _ptr(z)) != 0:
        raise ValueError("oracle_quantize_asym_int4 rejected its arguments")
    return q, s, z


def logits_asym_int4(x: np.ndarray, x_dtype: int, q: np.ndarray, scales: np.ndarray,
                     zeros: np.ndarray, scale_dtype: int, group: int):
    """binary64 logits [m, n] of the zero-point int4 head and the matching sum |x*w|."""
    lib = _load()
    xb = _as_bits(x, x_dtype)
    m, k = xb.shape
    qq = np.ascontiguousarray(q, dtype=np.uint8)
    n = qq.shape[0]
    sc = np.ascontiguousarray(scales).view(np.uint16)
    zz = np.ascontiguousarray(zeros, dtype=np.uint8)
    out = np.empty((m, n), dtype=np.float64)
    absout = np.empty((m, n), dtype=np.float64)
    if lib.oracle_logits_asym_int4(_ptr(xb), x_dtype, m, k, _ptr(qq), _ptr(sc), _ptr(zz),
                                   scale_dtype, group, n, _ptr(out), _ptr(absout)) != 0:
        raise ValueError("oracle_logits_asym_int4 rejected its arguments")
    return out, absout


def tolerance(absacc: np.ndarray) -> np.ndarray:
    """Per-logit bound |gpu - oracle| <= 1e-3 + 2e-3 * sum_k |x_k * w_k|."""
    return 1e-3 + 2e-3 * absacc
