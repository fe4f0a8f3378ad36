"""Shared helpers for the GPU-vs-oracle parity tests.

The oracle always quantises the weight itself (from the same seeded input
tensor the GPU gets); no oracle input is ever taken from the CUDA path.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

NTHREADS = max(1, min(64, os.cpu_count() or 1))
TORCH_OF = {oracle.F32: torch.float32, oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


def np_bits(t: torch.Tensor) -> np.ndarray:
    """fp16/bf16 tensor -> its uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_input(t: torch.Tensor, code: int) -> np.ndarray:
    """A host array the oracle accepts for dtype `code` (float32 or uint16 bits)."""
    if code == oracle.F32:
        return t.detach().cpu().contiguous().numpy()
    return np_bits(t)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def oracle_quantized(w: torch.Tensor, w_code: int, bits: int, group: int, sdt: int, clip: int):
    return oracle.quantize_packed(np_input(w, w_code), w_code, bits, group, sdt, clip,
                                  nthreads=NTHREADS)


def assert_quantized_equal(qw, o_qw: np.ndarray, o_s: np.ndarray, rows=None):
    """Bit-exact comparison of the GPU's packed weight/scales with the oracle's."""
    g_q = qw.qweight.detach().cpu().numpy()
    g_s = np_bits(qw.scales)
    if rows is not None:
        g_q, g_s = g_q[rows], g_s[rows]
    if g_q.dtype == np.int32:
        o_q = o_qw.view(np.int32)
    else:
        o_q = o_qw
    bad_q = np.argwhere(g_q != o_q)
    bad_s = np.argwhere(g_s != o_s)
    assert bad_q.size == 0, f"{len(bad_q)} packed words differ, first at {bad_q[:3].tolist()}"
    assert bad_s.size == 0, f"{len(bad_s)} scales differ, first at {bad_s[:3].tolist()}"


def assert_logits_close(gpu: np.ndarray, ref: np.ndarray, absacc: np.ndarray, what=""):
    """|gpu - oracle| <= 1e-3 + 2e-3 * sum_k |x_k w_k|, element by element."""
    err = np.abs(gpu.astype(np.float64) - ref)
    tol = oracle.tolerance(absacc)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} logits out of tolerance; worst "
                           f"err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max()), float((err / tol).max())


def check_topk(g_idx: np.ndarray, g_val: np.ndarray, ref_row: np.ndarray, ref_abs: np.ndarray,
               K: int, g_logits: np.ndarray | None = None) -> int:
    """Top-K candidate check for one token row against the full oracle row.

    The GPU ranks its own fp32 logits, the oracle binary64 ones: the sets must
    agree except for near-ties -- an element may be swapped only if its
    oracle value lies within 2*delta of the oracle's K-th value, delta being
    the largest |gpu - oracle| seen on the row's candidates (their reported
    values and, when `g_logits` -- the row the kernel returned -- is given,
    the returned logits at the GPU's and the oracle's candidates: candidates
    chosen from the returned logits are exact up to their precision).
    Returns 1 if such a tie swap happened, else 0.  Values must match the
    oracle within the logit tolerance and be ordered value-descending,
    index-ascending."""
    o_idx, o_val = oracle.topk(ref_row[None, :], K)
    o_idx, o_val = o_idx[0], o_val[0]
    assert np.all(g_idx >= 0) and np.all(g_idx < ref_row.shape[0])
    assert len(set(g_idx.tolist())) == K, "duplicate candidates"
    ov = ref_row[g_idx]
    delta = float(np.max(np.abs(g_val.astype(np.float64) - ov)))
    if g_logits is not None:
        both = np.concatenate([g_idx, o_idx])
        delta = max(delta, float(np.max(np.abs(g_logits[both].astype(np.float64) -
                                               ref_row[both]))))
    tol = oracle.tolerance(ref_abs[g_idx])
    assert np.all(np.abs(g_val.astype(np.float64) - ov) <= tol), "candidate values off"
    order_ok = all((g_val[i] > g_val[i + 1]) or (g_val[i] == g_val[i + 1] and g_idx[i] < g_idx[i + 1])
                   for i in range(K - 1))
    assert order_ok, f"candidates not ordered: {g_val} {g_idx}"
    gs, os_ = set(g_idx.tolist()), set(o_idx.tolist())
    if gs == os_:
        return 0
    kth = o_val[-1]
    slack = 2 * delta + 1e-300
    for i in gs - os_:
        assert ref_row[i] >= kth - slack, f"GPU candidate {i} ({ref_row[i]}) far below K-th {kth}"
    for j in os_ - gs:
        assert ref_row[j] <= kth + slack, f"oracle candidate {j} ({ref_row[j]}) missed"
    return 1
