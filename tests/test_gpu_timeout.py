"""The bounded-wait timeout path of the tensor-core kernel, made to run out
on purpose without faulting or hanging anything.

wql_debug_set_waits(budget, stall_mma=True) makes the kernel's MMA warp
first wait on a barrier that nothing arrives on, with a budget of about a
millisecond: that wait runs out, the warp gives up, stops releasing the
rings it consumes, and every other role's waits run out after it (each a
budget long).  The producer still waits, with the full budget, for the
copies it issued, so nothing is in flight when the CTA ends.  The call must
return, the error word must be set, the top-K outputs must read -1 / NaN
(sticky on that workspace until cleared), and the next normal call must be
correct.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wql_gb300 as wql
from weight_only_quantized_wql_gb300 import synth
from parity import (assert_logits_close, check_topk, np_input, oracle_quantized, report_ties,
                    to_f64)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BUDGET = 2_000_000          # SM cycles, about 1 ms


@pytest.fixture(autouse=True)
def _restore_waits():
    torch.cuda.set_device(DEV)
    wql.load()
    yield
    wql.wql_debug_set_waits(0, False)


def _head():
    n, k = 4099, 512
    w = synth.weight(n, k, oracle.F32, seed=3)
    qw = wql.wql_quantize(w.to(DEV), 4, 64, torch.float16, wql.CLIP_RTN)
    o_qw, o_s = oracle_quantized(w, oracle.F32, 4, 64, oracle.F16, 0)
    return n, k, qw, o_qw, o_s


def _check_normal(x, qw, o_qw, o_s, n, k, ws, K=8):
    logits, idx, val = wql.wql_logits(x, qw, topk=K, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error_word() == 0
    m = x.shape[0]
    ref, absacc = oracle.logits(np_input(x.cpu(), oracle.F16), oracle.F16, o_qw, 4, o_s,
                                oracle.F16, 64, n, k, nthreads=8)
    assert_logits_close(to_f64(logits), ref, absacc, f"after timeout m={m}")
    tk = k if m > 16 else None
    ties = sum(check_topk(idx.cpu().numpy()[r], val.cpu().numpy()[r], ref[r], absacc[r], K, tk)
               for r in range(m))
    report_ties(f"timeout-recovery m={m}", ties, m)


def test_tensor_core_wait_timeout_is_reported_and_recovers():
    n, k, qw, o_qw, o_s = _head()
    m, K = 32, 8                              # the tensor-core kernel
    x = synth.activations(m, k, oracle.F16, seed=9).to(DEV)
    ws = wql.Workspace(DEV)
    wql.wql_debug_set_waits(BUDGET, True)
    logits, idx, val = wql.wql_logits(x, qw, topk=K, workspace=ws)
    torch.cuda.synchronize()                  # the call returned and the stream drained
    assert ws.error_word() & 2, f"error word {ws.error_word():#x}"
    assert (idx == -1).all()
    assert torch.isnan(val).all()
    # the GPU context is still usable: back to the defaults, the same
    # workspace keeps reporting the timeout until its error word is cleared
    wql.wql_debug_set_waits(0, False)
    _, idx2, val2 = wql.wql_logits(x, qw, topk=K, workspace=ws)
    torch.cuda.synchronize()
    assert (idx2 == -1).all() and torch.isnan(val2).all()
    ws.clear_error()
    _check_normal(x, qw, o_qw, o_s, n, k, ws)
    # and a fresh workspace is correct at once
    _check_normal(x, qw, o_qw, o_s, n, k, wql.Workspace(DEV))


def test_decode_kernel_has_no_waits_to_time_out():
    """m <= 16 runs the decode kernel, which has no waits: the diagnostic
    stall does not touch it and the call is correct."""
    n, k, qw, o_qw, o_s = _head()
    x = synth.activations(1, k, oracle.F16, seed=10).to(DEV)
    wql.wql_debug_set_waits(BUDGET, True)
    _check_normal(x, qw, o_qw, o_s, n, k, wql.Workspace(DEV))
