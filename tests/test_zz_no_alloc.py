"""wql_logits_noalloc: the logits entry point that takes no workspace and
uses the library's fixed device scratch area instead.

Collected last on purpose (file name), so that it runs both after every other
GPU test in one process and, run on its own, as the first library call of a
fresh process (the call that does the one-time per-device setup).  The GPU
cases go through the C ABI and compare the new entry point with wql_logits
(caller workspace) within the logit tolerance, on two calls in a row; the
oracle supplies the tolerance's sum |x w| and an independent check.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wql_gb300 as wql
from weight_only_quantized_wql_gb300 import synth
from parity import assert_logits_close, check_topk, np_input, oracle_quantized, to_f64

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EWORKSPACE = 4
A = 0x7F0000100000  # aligned fake device address; the rejected call never uses it

# (bits, group, scale dtype, weight dtype, activation dtype, clip)
SCHEMES = [
    (4, 64, oracle.F16, oracle.F32, oracle.F16, 0),
    (8, 128, oracle.F16, oracle.F32, oracle.F16, 0),
    (4, 128, oracle.BF16, oracle.BF16, oracle.BF16, 1),
]
TORCH_OF = {oracle.F32: torch.float32, oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


def test_area_size_matches_header():
    text = open(os.path.join(ROOT, "include", "wql.h")).read()
    mt = re.search(r"#define WQL_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert mt and int(mt.group(1)) << int(mt.group(2)) == wql.NOALLOC_SCRATCH_BYTES


def test_every_valid_slice_fits_the_area():
    """The scratch a 16-row slice needs is bounded (top-K candidate slots and
    the counter block; it does not grow with the vocab), so the fixed area
    holds the largest one any valid call can ask for."""
    for topk in range(0, wql.MAX_TOPK + 1):
        for n in (1, 151936, 10 ** 6, 2 ** 31 - 1):
            assert wql.wql_workspace_size(16, n, topk) <= wql.NOALLOC_SCRATCH_BYTES


def test_invalid_call_is_rejected_before_any_cuda_call():
    """Argument errors are caught on the host (no GPU needed, nothing launched)."""
    lib = wql.load()
    st = wql._WqlWeight(4, 64, 1, 0, 1000, 512, A, A)
    before = lib.wql_launch_count()
    assert lib.wql_logits_noalloc(A, 1, 2, ctypes.byref(st), None, A, wql.MAX_TOPK + 1, A, A,
                                  None) == 1                       # WQL_EINVAL
    bad = wql._WqlWeight(4, 64, 1, 0, 1000, 100, A, A)             # k % 64 != 0
    assert lib.wql_logits_noalloc(A, 1, 2, ctypes.byref(bad), None, A, 0, None, None,
                                  None) == 2                       # WQL_EUNSUPPORTED
    assert lib.wql_launch_count() == before


@pytest.mark.gpu
@pytest.mark.parametrize("scheme", SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}s{s[2]}")
def test_noalloc_matches_workspace_entry_point(scheme):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    bits, group, sdt, wdt, xdt, clip = scheme
    n, k, K = 4099, 512, 8            # several CTAs, ragged 16-row tail
    w = synth.weight(n, k, wdt, seed=11)
    qw = wql.wql_quantize(w.to(dev), bits, group, TORCH_OF[sdt], clip)
    o_qw, o_s = oracle_quantized(w, wdt, bits, group, sdt, clip)
    ws = wql.Workspace(dev)
    for m in (1, 3, 16, 40):          # 40 = slices of 16 + 16 + 8
        x = synth.activations(m, k, xdt, seed=500 + m).to(dev)
        ref_logits, ref_idx, ref_val = wql.wql_logits(x, qw, topk=K, workspace=ws)
        outs = []
        for _ in range(2):            # two calls in a row, each into fresh outputs
            out = torch.full((m, n), float("nan"), dtype=x.dtype, device=dev)
            idx = torch.full((m, K), -7, dtype=torch.int32, device=dev)
            val = torch.full((m, K), float("nan"), dtype=torch.float32, device=dev)
            wql.wql_logits_noalloc(x, qw, topk=K, out=out, topk_idx=idx, topk_val=val)
            outs.append((out, idx, val))
        torch.cuda.synchronize()
        assert ws.error_word() == 0
        o_ref, absacc = oracle.logits(np_input(x.cpu(), xdt), xdt, o_qw, bits, o_s, sdt, group,
                                      n, k, nthreads=4)
        tol = oracle.tolerance(absacc)
        base = to_f64(ref_logits)
        for out, idx, val in outs:
            got = to_f64(out)
            assert np.all(np.isfinite(got))
            # against the existing entry point: each is within tol of the
            # oracle, so the two are within 2 * tol of each other
            diff = np.abs(got - base)
            assert np.all(diff <= 2 * tol), f"m={m}: max diff {diff.max():.3e}"
            assert_logits_close(got, o_ref, absacc, f"noalloc m={m}")
            g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
            r_idx = ref_idx.cpu().numpy()
            for r in range(m):
                check_topk(g_idx[r], g_val[r], o_ref[r], absacc[r], K)
                if set(g_idx[r].tolist()) != set(r_idx[r].tolist()):
                    # only an exact near-tie may differ; both must pass the oracle check
                    check_topk(r_idx[r], ref_val.cpu().numpy()[r], o_ref[r], absacc[r], K)
        # the two calls of the same kernel on the same inputs agree exactly
        assert torch.equal(outs[0][0], outs[1][0])
        assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])


@pytest.mark.gpu
def test_noalloc_large_vocab_with_topk():
    """A 400k-row vocab with top-16 in 16-row slices runs inside the fixed
    area and gives what the workspace entry point gives (same kernel, same
    inputs: identical outputs)."""
    dev = torch.device("cuda:0")
    n, k, K, m = 400_000, 128, 16, 16
    w = synth.weight(n, k, oracle.F32, seed=5)
    qw = wql.wql_quantize(w.to(dev), 4, 64, torch.float16, wql.CLIP_RTN)
    x = synth.activations(m, k, oracle.F16, seed=6).to(dev)
    ref = wql.wql_logits(x, qw, topk=K, workspace=wql.Workspace(dev))
    for _ in range(2):
        got = wql.wql_logits_noalloc(x, qw, topk=K)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
