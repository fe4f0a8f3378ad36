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


def test_oversize_call_is_rejected_before_any_cuda_call():
    """A vocab whose 16-row slice needs more than the fixed area is refused
    on the host (runs without a GPU: no CUDA call happens)."""
    lib = wql.load()
    n, k, topk = 400_000, 512, 8
    assert wql.wql_workspace_size(16, n, topk) > wql.NOALLOC_SCRATCH_BYTES
    st = wql._WqlWeight(4, 64, 1, 0, n, k, A, A)
    before = lib.wql_launch_count()
    status = lib.wql_logits_noalloc(A, 1, 16, ctypes.byref(st), None, A, topk, A, A, None)
    assert status == EWORKSPACE
    assert lib.wql_launch_count() == before
    # the same vocab without top-K needs only the counter block: accepted by the checks
    assert wql.wql_workspace_size(16, n, 0) <= wql.NOALLOC_SCRATCH_BYTES


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
def test_noalloc_oversize_raises_and_writes_nothing():
    dev = torch.device("cuda:0")
    n, k = 400_000, 128
    qw = wql.wql_quantize(torch.zeros(n, k, device=dev), 4, 64, torch.float16, wql.CLIP_RTN)
    m = 16                            # a full slice: 16 * n * 4 B of fp32 scratch > area
    assert wql.wql_workspace_size(m, n, 8) > wql.NOALLOC_SCRATCH_BYTES
    x = torch.ones(m, k, dtype=torch.float16, device=dev)
    out = torch.full((m, n), 3.0, dtype=torch.float16, device=dev)
    with pytest.raises(wql.WQLError, match="WQL_EWORKSPACE.*fixed area holds"):
        wql.wql_logits_noalloc(x, qw, topk=8, out=out)
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    # without top-K the same head fits: only the counter block is used
    logits, _, _ = wql.wql_logits_noalloc(x, qw, topk=0, out=out)
    torch.cuda.synchronize()
    assert bool((logits == 0).all())
