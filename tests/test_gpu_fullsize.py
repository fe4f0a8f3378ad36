"""GPU parity at the full workload sizes, in the launch configuration the bench times.

Each workload is one of the pages' heads at its real shape ("Fused WNA16 GEMM
for tied quantized lm_head logits": Perf evals table and reviewer comment;
radiance_lmhead_int4.py: module docstring).  The weight is drawn on the
device (as the bench does), quantised by libwql, and the same tensor is
copied to the host for the oracle, which quantises it itself:

* quantisation and packing: the whole packed weight and scale table,
  bit-exact;
* logits: every token row at a seeded sample of vocab rows plus every row
  the GPU put in its top-K, within 1e-3 + 2e-3 * sum|x w|;
* top-K: for a few token rows per call the whole oracle row is computed and
  the candidate set must match up to near-ties; on the other rows the
  candidates' values must match and no sampled row may beat the K-th
  candidate by more than the tolerance;
* rescoring (151936 x 2048 int8 head): rescored values against a binary64
  dot with the fp16 reference rows, scattered into the logits, and the
  re-ranked best candidate.

Calls go through ``wql_logits(x, qw, topk=8)`` with the library's default
workspace, exactly as the bench issues them.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wql_gb300 as wql
from weight_only_quantized_wql_gb300 import synth
from parity import (NTHREADS, TORCH_OF, assert_logits_close, assert_quantized_equal,
                    check_topk, np_bits, np_input, oracle_quantized, report_ties, tc_rank_bound,
                    to_f64)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOPK = 8
N_SAMPLED_ROWS = 4096
FULL_ROWS_PER_CALL = 3        # token rows whose whole oracle row is computed (others)
WHOLE_ROWS_MAX_M = 16         # the 248320 x 5120 head: every token's whole row up to this m


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch.cuda.set_device(DEV)
    wql.load()
    yield
    assert wql.default_workspace(DEV).error_word() == 0


_CACHE = {}


def _quantised(name):
    """(workload, host W, GPU QuantizedWeight, oracle packed, oracle scales),
    built once per workload; the packed weight is checked bit-exact here."""
    if name in _CACHE:
        return _CACHE[name]
    _CACHE.clear()                    # one full-size head in memory at a time
    torch.cuda.empty_cache()
    wl = synth.WORKLOADS[name]
    w_dev = synth.weight(wl.n, wl.k, wl.w_dtype, seed=wl.w_seed, device=DEV)
    qw = wql.wql_quantize(w_dev, wl.bits, wl.group, TORCH_OF[wl.scale_dtype], wl.clip)
    w_host = w_dev.cpu()
    del w_dev
    o_qw, o_s = oracle_quantized(w_host, wl.w_dtype, wl.bits, wl.group, wl.scale_dtype,
                                 wl.clip)
    torch.cuda.synchronize()
    assert_quantized_equal(qw, o_qw, o_s)
    _CACHE[name] = (wl, w_host, qw, o_qw, o_s)
    return _CACHE[name]


def _sample_rows(n, seed, extra):
    rng = np.random.default_rng(seed)
    rows = rng.choice(n, size=min(n, N_SAMPLED_ROWS), replace=False)
    rows = np.concatenate([rows, np.arange(max(0, n - 16), n), np.asarray(extra).ravel()])
    return np.unique(rows.astype(np.int64))


def _check_call(wl, qw, o_qw, o_s, x, logits, idx, val, seed):
    """Sampled logits, whole-row top-K on some tokens (all of them for the
    248320 x 5120 head at m <= 16), and top-K validity against the sampled
    rows on the rest."""
    m = x.shape[0]
    x_host = np_input(x, wl.x_dtype)
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    gl = to_f64(logits)
    # the tensor-core path (m > 16, fp16 activations and scales) ranks rounded
    # logits; the decode kernel its fp32 values
    tc = m > 16 and wl.x_dtype == oracle.F16 and wl.scale_dtype == oracle.F16
    rows = _sample_rows(wl.n, seed, g_idx)
    ref, absacc = oracle.logits(x_host, wl.x_dtype, o_qw, wl.bits, o_s, wl.scale_dtype,
                                wl.group, wl.n, wl.k, rows=rows, nthreads=NTHREADS)
    assert_logits_close(gl[:, rows], ref, absacc, f"{wl.name} m={m} sampled rows")
    pos = {int(r): i for i, r in enumerate(rows)}
    if wl.n == 248320 and m <= WHOLE_ROWS_MAX_M:
        full = list(range(m))
    else:
        full = sorted({0, m // 2, m - 1})[:FULL_ROWS_PER_CALL]
    for t in range(m):
        cand = np.array([pos[int(i)] for i in g_idx[t]])
        o_cand = ref[t, cand]
        tol = oracle.tolerance(absacc[t, cand])
        assert np.all(np.abs(g_val[t].astype(np.float64) - o_cand) <= tol), \
            f"token {t}: candidate values off"
        if t in full:
            continue
        # no sampled row may beat the K-th candidate by more than the ranking
        # error: 2 * delta from the fp32 candidate values (decode kernel), or
        # the rounded-logit bound of both rows (tensor-core path)
        kc = int(np.argmin(o_cand))
        others = np.setdiff1d(np.arange(rows.size), cand)
        gap = ref[t, others] - o_cand[kc]
        if tc:
            b = tc_rank_bound(ref[t], absacc[t], wl.k)
            limit = b[cand[kc]] + b[others]
        else:
            limit = 2 * float(np.max(np.abs(g_val[t].astype(np.float64) - o_cand))) + 1e-300
        assert np.all(gap <= limit), f"token {t}: a sampled row beats the K-th candidate"
    ties = 0
    for t in full:
        ref_row, abs_row = oracle.logits(x_host[t:t + 1], wl.x_dtype, o_qw, wl.bits, o_s,
                                         wl.scale_dtype, wl.group, wl.n, wl.k,
                                         nthreads=NTHREADS)
        assert_logits_close(gl[t:t + 1], ref_row, abs_row, f"{wl.name} token {t} full row")
        ties += check_topk(g_idx[t], g_val[t], ref_row[0], abs_row[0], TOPK,
                           wl.k if tc else None)
    report_ties(f"fullsize {wl.name} m={m}", ties, len(full))


FULL = [("pr_fixture_50304x512_w4g64", 1),
        ("qwen_151936x1024_w4g64", 1), ("qwen_151936x1024_w4g64", 32),
        ("qwen_151936x1024_w4g64", 256),
        ("qwen_151936x1024_w8g128", 1), ("qwen_151936x1024_w8g128", 32),
        ("qwen_151936x1024_w8g128", 256),
        ("head_248320x5120_w4g128_mse", 1), ("head_248320x5120_w4g128_mse", 2),
        ("head_248320x5120_w4g128_mse", 3), ("head_248320x5120_w4g128_mse", 4),
        ("head_248320x5120_w4g128_mse", 5), ("head_248320x5120_w4g128_mse", 16)]


@pytest.mark.parametrize("name,m", FULL, ids=[f"{n}-M{m}" for n, m in FULL])
def test_fullsize_logits_topk(name, m):
    wl, w_host, qw, o_qw, o_s = _quantised(name)
    if wl.x_continues_w:
        # the 50304 x 512 fixture draws X from the same generator after W
        g = synth.generator(wl.w_seed, DEV)
        synth.weight(wl.n, wl.k, wl.w_dtype, device=DEV, gen=g)
        x = synth.activations(m, wl.k, wl.x_dtype, device=DEV, gen=g)
    else:
        x = synth.activations(m, wl.k, wl.x_dtype, seed=wl.x_seed + 1000 * m, device=DEV)
    logits, idx, val = wql.wql_logits(x, qw, topk=TOPK)
    torch.cuda.synchronize()
    _check_call(wl, qw, o_qw, o_s, x, logits, idx, val, seed=m)


def test_fullsize_int8_row_rescore():
    """151936 x 2048 int8 per-row head, M = 1 calls with top-8 followed by exact
    rescoring from the fp16 reference rows (reviewer comment items 1-2)."""
    wl, w_host, qw, o_qw, o_s = _quantised("qwen_151936x2048_w8row_rescore")
    w_ref = w_host.to(DEV)                       # the fp16 reference weight itself
    xs = synth.activations(wl.rows, wl.k, wl.x_dtype, seed=wl.x_seed, device=DEV)
    w_ref_host = np_input(w_host, wl.w_dtype)
    for r in (0, 1, 2047, wl.rows - 1):
        x = xs[r:r + 1].contiguous()
        logits, idx, val = wql.wql_logits(x, qw, topk=wl.rescore_k)
        torch.cuda.synchronize()
        _check_call(wl, qw, o_qw, o_s, x, logits, idx, val, seed=r)
        before = logits.clone()
        wql.wql_topk_rescore(x, w_ref, idx, val, logits)
        torch.cuda.synchronize()
        g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
        o_val, o_abs = oracle.rescore(np_input(x, wl.x_dtype), wl.x_dtype, w_ref_host,
                                      wl.w_dtype, g_idx)
        assert np.all(np.abs(g_val - o_val) <= oracle.tolerance(o_abs)), f"row {r}"
        assert np.all(np.diff(g_val[0]) <= 0)
        row = logits[0].cpu()
        sel = torch.tensor(g_idx[0], dtype=torch.long)
        assert torch.equal(row[sel], torch.tensor(g_val[0]).to(row.dtype))
        mask = torch.ones(wl.n, dtype=torch.bool)
        mask[sel] = False
        assert torch.equal(row[mask], before[0].cpu()[mask])
        # the rescored best candidate is the argmax of the exact fp16 rows among
        # the candidates, up to values the reference dot cannot separate
        best = int(np.argmax(o_val[0]))
        assert o_val[0, 0] >= o_val[0, best] - oracle.tolerance(o_abs[0, best])


@pytest.mark.parametrize("name", ["qwen_151936x1024_w4g64", "qwen_151936x1024_w8g128",
                                  "head_248320x5120_w4g128_mse"])
def test_fullsize_embed_gather(name):
    """Tied-embedding gather from the full head: 4096 seeded ids (and the
    first and last rows), bit-exact against the oracle's gather."""
    wl, w_host, qw, o_qw, o_s = _quantised(name)
    gen = torch.Generator().manual_seed(77)
    ids = torch.cat([torch.tensor([0, wl.n - 1], dtype=torch.int32),
                     torch.randint(0, wl.n, (4096,), generator=gen, dtype=torch.int32)])
    odt = wl.x_dtype
    out = wql.wql_embed_gather(ids.to(DEV), qw, out_dtype=TORCH_OF[odt])
    torch.cuda.synchronize()
    want = oracle.embed_gather(ids.numpy(), o_qw, wl.bits, o_s, wl.scale_dtype, wl.group,
                               wl.n, wl.k, odt)
    got = np_bits(out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} outputs differ, first at {bad[:3].tolist()}"
