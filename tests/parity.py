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


# near-tie swaps seen by check_topk, per test (printed in the session summary)
TIE_LOG: dict = {}


def report_ties(name: str, swaps: int, rows: int) -> None:
    prev = TIE_LOG.get(name, (0, 0))
    TIE_LOG[name] = (prev[0] + swaps, prev[1] + rows)


def tc_rank_bound(ref_row: np.ndarray, ref_abs: np.ndarray, k: int) -> np.ndarray:
    """How far the tensor-core path's rounded logit of each row may lie from
    the exact one: the scale folded into fp16 weights (2^-11 relative per
    weight), the fp32 sums over k columns (k * 2^-22 relative, generous for
    the tensor cores' accumulation), the fp16 rounding of the output
    (2^-11 relative) and 2^-20 absolute for fp16 subnormals."""
    return (2.0 ** -11 + k * 2.0 ** -22) * ref_abs + 2.0 ** -11 * np.abs(ref_row) + 2.0 ** -20


def check_topk(g_idx: np.ndarray, g_val: np.ndarray, ref_row: np.ndarray, ref_abs: np.ndarray,
               K: int, tc_k: int | None = None) -> int:
    """Top-K candidate check for one token row against the full oracle row.

    The sets must agree except for near-ties.  Values must match the oracle
    within the logit tolerance and be ordered value-descending,
    index-ascending.  A GPU candidate i may stand in for an oracle candidate
    j only if the oracle's values are that close:
      * decode path (tc_k None): the GPU ranks the fp32 values it returns;
        L_j - L_i <= 2 * delta, delta the largest |value - oracle| over the
        GPU's candidates (fp32 values only);
      * tensor-core path (tc_k = k): the GPU ranks fp16-rounded logits;
        L_j - L_i <= b(i) + b(j) with b = tc_rank_bound.
    Returns the number of candidates swapped this way (0 when the sets are
    equal)."""
    o_idx, o_val = oracle.topk(ref_row[None, :], K)
    o_idx, o_val = o_idx[0], o_val[0]
    assert np.all(g_idx >= 0) and np.all(g_idx < ref_row.shape[0])
    assert len(set(g_idx.tolist())) == K, "duplicate candidates"
    ov = ref_row[g_idx]
    tol = oracle.tolerance(ref_abs[g_idx])
    assert np.all(np.abs(g_val.astype(np.float64) - ov) <= tol), "candidate values off"
    order_ok = all((g_val[i] > g_val[i + 1]) or (g_val[i] == g_val[i + 1] and g_idx[i] < g_idx[i + 1])
                   for i in range(K - 1))
    assert order_ok, f"candidates not ordered: {g_val} {g_idx}"
    gs, os_ = set(g_idx.tolist()), set(o_idx.tolist())
    if gs == os_:
        return 0
    extra, missed = sorted(gs - os_), sorted(os_ - gs)
    if tc_k is None:
        delta = float(np.max(np.abs(g_val.astype(np.float64) - ov)))
        for i in extra:
            for j in missed:
                assert ref_row[j] - ref_row[i] <= 2 * delta + 1e-300, \
                    f"swap {i} for {j}: oracle gap {ref_row[j] - ref_row[i]:.3e} > 2*delta {2 * delta:.3e}"
    else:
        b = tc_rank_bound(ref_row, ref_abs, tc_k)
        for i in extra:
            for j in missed:
                assert ref_row[j] - ref_row[i] <= b[i] + b[j], \
                    f"swap {i} for {j}: oracle gap {ref_row[j] - ref_row[i]:.3e} > bound {b[i] + b[j]:.3e}"
    return len(extra)
