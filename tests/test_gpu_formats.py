"""GPU parity of the fp8 e4m3 per-row and the zero-point int4 formats, and
of the candidates-only mode (no logits written), against the CPU oracle.

fp8 e4m3 per row: the per-channel fp8 head that radiance_lmhead_int4.py's
module docstring compares against.  Zero-point int4: the sym=False lm_head
of "[CORE] Quantized lm-head Framework" (lm-eval table).  Candidates only:
"Fused WNA16 GEMM for tied quantized lm_head logits", reviewer comment
item 2 (a top-K consumer needs only the K candidates and their values).

Gates as for the symmetric formats: codes, scales and zero points
bit-exact; every logit within 1e-3 + 2e-3 * sum|x w|; top-K sets equal up
to exact near-ties.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wql_gb300 as wql
from weight_only_quantized_wql_gb300 import synth
from parity import (NTHREADS, assert_logits_close, check_topk, np_bits, np_input,
                    oracle_quantized, report_ties, to_f64)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TORCH_OF = {oracle.F32: torch.float32, oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch.cuda.set_device(DEV)
    wql.load()
    yield
    assert wql.default_workspace(DEV).error_word() == 0


def _edge_rows(k: int) -> torch.Tensor:
    """Rows that exercise clamps, ties, subnormal codes and zero scales."""
    rows = torch.zeros(8, k, dtype=torch.float32)
    rows[1, 5] = 1e-9                          # scale underflows in fp16 -> codes 0
    rows[2, :] = torch.linspace(-3, 3, k)
    rows[3, :8] = torch.tensor([448.0, -448.0, 3.5, -3.5, 0.5, 1.5, 2.5, -0.5])
    rows[4, :] = 1e-30
    rows[5, 0] = 3e38
    rows[5, 1:] = 1e-3                         # tiny values next to a huge one
    rows[6, :] = -0.02
    rows[7, ::2] = 0.013
    rows[7, 1::2] = -0.0009                    # codes in e4m3's subnormal range
    return rows


def _fp8_weight(n, k, wdt, sdt, seed=0, edges=True):
    w = synth.weight(n, k, wdt, seed=seed)
    if edges:
        w[:8] = _edge_rows(k).to(w.dtype)
    qw = wql.wql_quantize(w.to(DEV), 8, 0, TORCH_OF[sdt], wql.CLIP_RTN, fmt=wql.FMT_E4M3)
    o_q, o_s = oracle.quantize_fp8(np_input(w, wdt), wdt, sdt)
    return w, qw, o_q, o_s


def _asym_weight(n, k, group, wdt, sdt, seed=0, edges=True):
    w = synth.weight(n, k, wdt, seed=seed)
    if edges:
        w[:8] = _edge_rows(k).to(w.dtype)
        w[8, :] = torch.linspace(0.01, 0.5, k).to(w.dtype)     # all positive: z = 0
        w[9, :] = torch.linspace(-0.5, -0.01, k).to(w.dtype)   # all negative: z = 15
    qw = wql.wql_quantize(w.to(DEV), 4, group, TORCH_OF[sdt], wql.CLIP_RTN, fmt=wql.FMT_ASYM)
    o_q, o_s, o_z = oracle.quantize_asym_int4(np_input(w, wdt), wdt, group, sdt)
    return w, qw, o_q, o_s, o_z


# ---------------------------------------------------------------------------
# fp8 e4m3 per row
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wdt,sdt", [(oracle.F32, oracle.F16), (oracle.BF16, oracle.BF16),
                                     (oracle.F16, oracle.F16), (oracle.F32, oracle.BF16)])
@pytest.mark.parametrize("n,k", [(1000, 512), (77, 320), (16, 64)])
def test_fp8_quantize_bit_exact(wdt, sdt, n, k):
    w, qw, o_q, o_s = _fp8_weight(n, k, wdt, sdt, edges=n >= 8)
    torch.cuda.synchronize()
    g_q = qw.qweight.cpu().numpy()
    g_s = np_bits(qw.scales).reshape(-1)
    bad = np.argwhere(g_q != o_q)
    assert bad.size == 0, f"{len(bad)} e4m3 codes differ, first at {bad[:3].tolist()}"
    assert np.array_equal(g_s, o_s), "per-row scales differ"


@pytest.mark.parametrize("xdt,sdt", [(oracle.F16, oracle.F16), (oracle.BF16, oracle.BF16),
                                     (oracle.F16, oracle.BF16)])
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 9, 16, 17, 33])
def test_fp8_logits(xdt, sdt, m):
    n, k, K = 1000, 512, 8
    wdt = oracle.BF16 if xdt == oracle.BF16 else oracle.F32
    w, qw, o_q, o_s = _fp8_weight(n, k, wdt, sdt, seed=m, edges=False)
    x = synth.activations(m, k, xdt, seed=200 + m)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits_fp8(np_input(x, xdt), xdt, o_q, o_s, sdt)
    assert_logits_close(to_f64(logits), ref, absacc, f"fp8 m={m}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K) for r in range(m))
    report_ties(f"fp8 m={m}", ties, m)


def test_fp8_fullsize_head_m1():
    """The 248320 x 5120 head of the fp8 comparison (1.27 GB of codes) at
    M = 1 with top-8: the quantised rows of a 4096-row sample bit-exact, the
    logits there and at the candidates within tolerance, and no sampled row
    above the K-th candidate beyond the tolerance."""
    n, k, K = 248320, 5120, 8
    wl = synth.WORKLOADS["head_248320x5120_w4g128_mse"]
    w = synth.weight(n, k, wl.w_dtype, seed=wl.w_seed, device=DEV)
    qw = wql.wql_quantize(w, 8, 0, torch.bfloat16, wql.CLIP_RTN, fmt=wql.FMT_E4M3)
    x = synth.activations(1, k, wl.x_dtype, seed=wl.x_seed).to(DEV)
    logits, idx, val = wql.wql_logits(x, qw, topk=K)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(n, 4096, replace=False), idx[0].cpu().numpy()]))
    wr = w[torch.from_numpy(rows).to(DEV)].cpu()
    o_q, o_s = oracle.quantize_fp8(np_input(wr, wl.w_dtype), wl.w_dtype, oracle.BF16)
    assert np.array_equal(qw.qweight[torch.from_numpy(rows).to(DEV)].cpu().numpy(), o_q)
    assert np.array_equal(np_bits(qw.scales).reshape(-1)[rows], o_s)
    ref, absacc = oracle.logits_fp8(np_input(x.cpu(), wl.x_dtype), wl.x_dtype, o_q, o_s,
                                    oracle.BF16)
    got = to_f64(logits)[0, rows]
    assert_logits_close(got[None, :], ref, absacc, "fp8 full-size sample")
    pos = {int(r): i for i, r in enumerate(rows)}
    g_idx, g_val = idx[0].cpu().numpy(), val[0].cpu().numpy()
    cref = np.array([ref[0, pos[int(i)]] for i in g_idx])
    ctol = oracle.tolerance(np.array([absacc[0, pos[int(i)]] for i in g_idx]))
    assert np.all(np.abs(g_val - cref) <= ctol)
    kth = cref.min()
    others = np.array([j for j in range(len(rows)) if int(rows[j]) not in set(g_idx.tolist())])
    assert np.all(ref[0, others] <= kth + 2 * ctol.max()), "a sampled row beats the K-th candidate"


# ---------------------------------------------------------------------------
# zero-point int4
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wdt,sdt", [(oracle.F32, oracle.F16), (oracle.BF16, oracle.BF16),
                                     (oracle.F16, oracle.F16)])
@pytest.mark.parametrize("n,k,group", [(1000, 512, 128), (77, 1024, 256), (16, 384, 128)])
def test_asym_quantize_bit_exact(wdt, sdt, n, k, group):
    w, qw, o_q, o_s, o_z = _asym_weight(n, k, group, wdt, sdt)
    torch.cuda.synchronize()
    nib = wql.wql_unpack(qw.qweight, k).cpu().numpy()
    bad = np.argwhere(nib != o_q)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"
    assert np.array_equal(np_bits(qw.scales), o_s), "scales differ"
    assert np.array_equal(qw.zeros.cpu().numpy(), o_z), "zero points differ"


@pytest.mark.parametrize("xdt,sdt", [(oracle.F16, oracle.F16), (oracle.BF16, oracle.BF16),
                                     (oracle.F16, oracle.BF16)])
@pytest.mark.parametrize("m", [1, 3, 5, 9, 16, 33])
@pytest.mark.parametrize("k,group", [(512, 128), (768, 256)])
def test_asym_logits(xdt, sdt, m, k, group):
    n, K = 1000, 8
    wdt = oracle.BF16 if xdt == oracle.BF16 else oracle.F32
    w, qw, o_q, o_s, o_z = _asym_weight(n, k, group, wdt, sdt, seed=m, edges=False)
    x = synth.activations(m, k, xdt, seed=300 + m)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits_asym_int4(np_input(x, xdt), xdt, o_q, o_s, o_z, sdt, group)
    assert_logits_close(to_f64(logits), ref, absacc, f"asym m={m}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K) for r in range(m))
    report_ties(f"asym m={m} g{group}", ties, m)


# ---------------------------------------------------------------------------
# candidates only
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,group", [(4, 64), (8, 128), (4, 128)])
@pytest.mark.parametrize("m", [1, 5, 16, 40])
def test_candidates_only(bits, group, m):
    """logits_out NULL with top-K: no logits are written, and the candidates
    are those of a call that writes them (the same kernel for m <= 16), and
    within the oracle's near-tie rule at any m."""
    n, k, K = 4099, 512, 8
    w = synth.weight(n, k, oracle.F32, seed=7)
    qw = wql.wql_quantize(w.to(DEV), bits, group, torch.float16, wql.CLIP_RTN)
    o_qw, o_s = oracle_quantized(w, oracle.F32, bits, group, oracle.F16, 0)
    x = synth.activations(m, k, oracle.F16, seed=400 + m).to(DEV)
    ws = wql.Workspace(DEV)
    none, idx, val = wql.wql_logits(x, qw, topk=K, workspace=ws, candidates_only=True)
    assert none is None
    ref_l, ref_i, ref_v = wql.wql_logits(x, qw, topk=K, workspace=ws)
    torch.cuda.synchronize()
    if m <= 16:
        assert torch.equal(idx, ref_i) and torch.equal(val, ref_v)
    ref, absacc = oracle.logits(np_input(x.cpu(), oracle.F16), oracle.F16, o_qw, bits, o_s,
                                oracle.F16, group, n, k, nthreads=NTHREADS)
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K) for r in range(m))
    report_ties(f"candidates_only w{bits}g{group} m={m}", ties, m)
