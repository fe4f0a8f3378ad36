"""GPU parity: libwql (through its C ABI) against the CPU oracle, small shapes.

Shapes span several 16-row tiles, several CTAs and a ragged vocab tail; the
oracle quantises the same seeded weight itself and computes binary64 logits.
Gates: packing and quantisation bit-exact; every logit within
1e-3 + 2e-3 * sum|x w|; top-K sets equal up to exact near-ties.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wql_gb300 as wql
from weight_only_quantized_wql_gb300 import synth
from parity import (assert_logits_close, assert_quantized_equal, check_topk, np_bits,
                    np_input, oracle_quantized, report_ties, to_f64)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# (bits, group, scale dtype, weight dtype, activation dtype, clip)
SCHEMES = [
    (4, 64, oracle.F16, oracle.F32, oracle.F16, 0),
    (4, 128, oracle.BF16, oracle.BF16, oracle.BF16, 1),
    (4, 128, oracle.F16, oracle.F32, oracle.F16, 0),
    (4, 0, oracle.F16, oracle.F16, oracle.F16, 0),
    (8, 128, oracle.F16, oracle.F32, oracle.F16, 0),
    (8, 0, oracle.F16, oracle.F16, oracle.F16, 0),
    (8, 64, oracle.BF16, oracle.BF16, oracle.BF16, 1),
]
TORCH_OF = {oracle.F32: torch.float32, oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


def tc_k(m, xdt, sdt, k):
    """k when the call takes the tensor-core path (more than 16 tokens with
    fp16 activations and scales), else None: check_topk's rank bound."""
    return k if m > 16 and xdt == oracle.F16 and sdt == oracle.F16 else None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch.cuda.set_device(DEV)
    wql.load()
    yield
    # no bounded wait inside any kernel may have timed out
    assert wql.default_workspace(DEV).error_word() == 0


def _make(n, k, scheme, seed=0):
    bits, group, sdt, wdt, xdt, clip = scheme
    w = synth.weight(n, k, wdt, seed=seed)
    qw = wql.wql_quantize(w.to(DEV), bits, group, TORCH_OF[sdt], clip)
    o_qw, o_s = oracle_quantized(w, wdt, bits, group, sdt, clip)
    return w, qw, o_qw, o_s


@pytest.mark.parametrize("scheme", SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}s{s[2]}w{s[3]}c{s[5]}")
@pytest.mark.parametrize("n,k", [(1000, 512), (77, 256), (16, 320)])
def test_quantize_bit_exact(scheme, n, k):
    if scheme[1] and k % scheme[1]:
        pytest.skip("group does not divide k")
    w, qw, o_qw, o_s = _make(n, k, scheme)
    torch.cuda.synchronize()
    assert_quantized_equal(qw, o_qw, o_s)


def test_quantize_edge_values():
    # zero rows, a single outlier, exact ties for round-half-even, fp16 underflow
    n, k = 8, 128
    w = torch.zeros(n, k, dtype=torch.float32)
    w[1, 5] = 1e-9                    # scale underflows in fp16 -> codes 0
    w[2, :] = torch.linspace(-7, 7, k)
    w[3, :8] = torch.tensor([7.0, -7.0, 3.5, -3.5, 0.5, 1.5, 2.5, -0.5])
    w[4, :] = 1e-30
    w[5, 0] = 3e38
    w[6, :] = -0.02
    w[7, ::2] = 0.013
    for bits, group, sdt, clip in [(4, 64, oracle.F16, 0), (4, 64, oracle.BF16, 1),
                                   (8, 128, oracle.F16, 0), (8, 0, oracle.BF16, 1)]:
        qw = wql.wql_quantize(w.to(DEV), bits, group, TORCH_OF[sdt], clip)
        o_qw, o_s = oracle_quantized(w, oracle.F32, bits, group, sdt, clip)
        torch.cuda.synchronize()
        assert_quantized_equal(qw, o_qw, o_s)


def test_pack_unpack_against_oracle():
    nib = synth.random_nibbles(123, 96)
    packed = wql.wql_pack(nib.to(DEV))
    o = oracle.pack_int4(nib.numpy())
    assert np.array_equal(packed.cpu().numpy(), o)
    back = wql.wql_unpack(packed, 96)
    assert torch.equal(back.cpu(), nib)


@pytest.mark.parametrize("scheme", SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}s{s[2]}x{s[4]}")
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 9, 16, 17, 33])
def test_logits_small(scheme, m):
    n, k, K = 1000, 512, 8
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=m)
    x = synth.activations(m, k, xdt, seed=100 + m)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits(np_input(x, xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                nthreads=4)
    assert_logits_close(to_f64(logits), ref, absacc, f"m={m}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    tk = tc_k(m, xdt, sdt, k)
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K, tk) for r in range(m))
    report_ties(f"logits_small w{bits}g{group} m={m}", ties, m)


@pytest.mark.parametrize("n", [9, 16, 17, 31, 4099])
def test_logits_ragged_vocab_and_bias(n):
    k, m = 256, 4
    scheme = SCHEMES[0]
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=n)
    x = synth.activations(m, k, xdt, seed=7)
    b = synth.bias(n, xdt)
    K = min(8, n)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, bias=b.to(DEV), topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits(np_input(x, xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                bias=np_bits(b))
    assert_logits_close(to_f64(logits), ref, absacc, f"n={n}")
    ties = sum(check_topk(idx.cpu().numpy()[r], val.cpu().numpy()[r], ref[r], absacc[r], K)
               for r in range(m))
    report_ties(f"ragged n={n}", ties, m)


def test_logits_without_topk_and_leading_shape():
    n, k = 600, 256
    w, qw, o_qw, o_s = _make(n, k, SCHEMES[4])
    x = synth.activations(6, k, oracle.F16, seed=3).reshape(2, 3, k)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=0)
    torch.cuda.synchronize()
    assert logits.shape == (2, 3, n) and idx is None
    ref, absacc = oracle.logits(np_input(x.reshape(6, k), oracle.F16), oracle.F16, o_qw, 8, o_s,
                                oracle.F16, 128, n, k)
    assert_logits_close(to_f64(logits.reshape(6, n)), ref, absacc)


@pytest.mark.parametrize("xdt", [oracle.F16, oracle.BF16])
def test_topk_rescore(xdt):
    n, k, m, K = 3000, 512, 5, 8
    scheme = (8, 0, oracle.F16 if xdt == oracle.F16 else oracle.BF16, xdt, xdt, 0)
    bits, group, sdt, wdt, _, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme)
    x = synth.activations(m, k, xdt, seed=11)
    b = synth.bias(n, xdt)
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    logits, idx, val = wql.wql_logits(xd, qw, bias=bd, topk=K)
    before = logits.clone()
    wql.wql_topk_rescore(xd, wd, idx, val, logits, bias=bd)
    torch.cuda.synchronize()
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    o_val, o_abs = oracle.rescore(np_input(x, xdt), xdt, np_input(w, wdt), wdt, g_idx,
                                  bias=np_bits(b))
    assert np.all(np.abs(g_val - o_val) <= oracle.tolerance(o_abs))
    for r in range(m):
        assert np.all(np.diff(g_val[r]) <= 0)
        # rescored entries are scattered into the logits; the rest are untouched
        row = logits[r].cpu()
        ref_row = torch.tensor(g_val[r]).to(logits.dtype)
        assert torch.equal(row[torch.tensor(g_idx[r], dtype=torch.long)], ref_row)
        mask = torch.ones(n, dtype=torch.bool)
        mask[torch.tensor(g_idx[r], dtype=torch.long)] = False
        assert torch.equal(row[mask], before[r].cpu()[mask])


def test_empty_and_errors():
    n, k = 100, 256
    w, qw, o_qw, o_s = _make(n, k, SCHEMES[0])
    x = torch.empty(0, k, dtype=torch.float16, device=DEV)
    logits, _, _ = wql.wql_logits(x, qw, topk=0)
    assert logits.shape == (0, n)
    xx = synth.activations(2, k, oracle.F16).to(DEV)
    with pytest.raises(wql.WQLError):
        wql.wql_logits(xx, qw, topk=n + 1)
    with pytest.raises(wql.WQLError):
        wql.wql_logits(xx, qw, topk=wql.MAX_TOPK + 1)
    bad = wql.QuantizedWeight(qw.qweight, qw.scales, 4, 64, n, 200)
    with pytest.raises(wql.WQLError):
        wql.wql_logits(synth.activations(2, 200, oracle.F16).to(DEV), bad)


def test_workspace_reuse_across_calls():
    # the per-call ticket counter must be left at zero for the next call
    n, k = 5000, 256
    w, qw, o_qw, o_s = _make(n, k, SCHEMES[0])
    ws = wql.Workspace(DEV)
    x = synth.activations(3, k, oracle.F16, seed=5)
    ref, absacc = oracle.logits(np_input(x, oracle.F16), oracle.F16, o_qw, 4, o_s, oracle.F16,
                                64, n, k)
    for _ in range(5):
        logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=8, workspace=ws)
        torch.cuda.synchronize()
        ties = sum(check_topk(idx.cpu().numpy()[r], val.cpu().numpy()[r], ref[r], absacc[r], 8)
                   for r in range(3))
        report_ties("workspace reuse", ties, 3)


TC_SCHEMES = [s for s in SCHEMES if s[4] == oracle.F16 and s[2] == oracle.F16]


@pytest.mark.parametrize("scheme", TC_SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}")
@pytest.mark.parametrize("m,n", [(32, 1000), (48, 4099), (100, 1000), (256, 777), (300, 600)])
def test_logits_tensor_core_path(scheme, m, n):
    """m > 16 with fp16 activations runs the tcgen05 kernel (up to 256 tokens
    per launch, several launches beyond)."""
    k, K = 512, 8
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=m + n)
    x = synth.activations(m, k, xdt, seed=200 + m)
    b = synth.bias(n, xdt)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, bias=b.to(DEV), topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits(np_input(x, xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                bias=np_bits(b), nthreads=8)
    assert_logits_close(to_f64(logits), ref, absacc, f"m={m} n={n}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K, k) for r in range(m))
    report_ties(f"tensor_core w{bits}g{group} m={m} n={n}", ties, m)


@pytest.mark.parametrize("scheme", TC_SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}")
@pytest.mark.parametrize("m", [32, 256])
def test_tensor_core_topk_many_tiles_per_cta(scheme, m):
    """A vocab of ~2 tiles per CTA: after each CTA's first tile the top-K runs
    in its filtered mode (per-token thresholds, shared across CTAs)."""
    n, k, K = 40000, 128, 8
    bits, group, sdt, wdt, xdt, clip = scheme
    if group and k % group:
        pytest.skip("group does not divide k")
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=7 + m)
    x = synth.activations(m, k, xdt, seed=300 + m)
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits(np_input(x, xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                nthreads=16)
    assert_logits_close(to_f64(logits), ref, absacc, f"m={m}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K, k) for r in range(m))
    report_ties(f"tensor_core_many_tiles w{bits}g{group} m={m}", ties, m)


def _rowwise_weight(n, k, row_value):
    """W[r, :] = row_value(r): after quantisation every row is 7 * s_r (int4)."""
    vals = torch.tensor([row_value(r) for r in range(n)], dtype=torch.float32)
    return vals[:, None].expand(n, k).contiguous()


@pytest.mark.parametrize("m", [1, 4, 32, 256])
@pytest.mark.parametrize("order", ["increasing", "decreasing", "equal", "negative"])
def test_tensor_core_topk_adversarial_orders(m, order):
    """Logits that grow with the row index put the best rows last; decreasing
    ones put them first; negative ones (growing) give a negative selection
    threshold; equal logits must give the lowest indices, and every
    row ties with the threshold, so the thresholded candidate lists overflow
    and the exhaustive selection runs (decode kernel for m <= 16, selection
    kernel after the tensor-core kernel above)."""
    n, k, K = 40000, 128, 8
    f = {"increasing": lambda r: 0.01 + 1e-5 * r, "decreasing": lambda r: 0.5 - 1e-5 * r,
         "equal": lambda r: 0.02, "negative": lambda r: -0.5 + 1e-5 * r}[order]
    w = _rowwise_weight(n, k, f)
    qw = wql.wql_quantize(w.to(DEV), 4, 64, torch.float16, 0)
    o_qw, o_s = oracle_quantized(w, oracle.F32, 4, 64, oracle.F16, 0)
    gen = torch.Generator().manual_seed(11)
    x = (torch.rand(m, k, generator=gen) + 0.5).half()      # positive rows
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    ref, absacc = oracle.logits(np_input(x, oracle.F16), oracle.F16, o_qw, 4, o_s, oracle.F16,
                                64, n, k, nthreads=16)
    assert_logits_close(to_f64(logits), ref, absacc, order)
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    tk = k if m > 16 else None
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K, tk) for r in range(m))
    report_ties(f"adversarial {order} m={m}", ties, m)
    if order == "equal":
        # every row's logit is the same number: value ties go to the lowest indices
        assert (g_idx == np.arange(K)[None, :]).all(), g_idx[:2]


@pytest.mark.parametrize("scheme", SCHEMES, ids=lambda s: f"w{s[0]}g{s[1]}s{s[2]}")
@pytest.mark.parametrize("odt", [oracle.F16, oracle.BF16], ids=["f16", "bf16"])
def test_embed_gather_bit_exact(scheme, odt):
    """Tied-embedding gather: rows of the dequantised head for token ids,
    bit-exact against the oracle; duplicates, the first and last rows, and
    ids outside [0, n) (rows of zeros)."""
    n, k = 1000, 320 if scheme[1] in (0, 64) else 512
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=41)
    gen = torch.Generator().manual_seed(9)
    ids = torch.cat([torch.tensor([0, n - 1, 5, 5, -1, n, n + 7, -2147483648, 2147483647],
                                  dtype=torch.int32),
                     torch.randint(0, n, (300,), generator=gen, dtype=torch.int32)])
    out = wql.wql_embed_gather(ids.to(DEV), qw, out_dtype=TORCH_OF[odt])
    torch.cuda.synchronize()
    want = oracle.embed_gather(ids.numpy(), o_qw, bits, o_s, sdt, group, n, k, odt)
    assert out.shape == (ids.numel(), k) and out.dtype == TORCH_OF[odt]
    got = np_bits(out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} outputs differ, first at {bad[:3].tolist()}"


def test_embed_gather_shapes():
    n, k = 300, 256
    w, qw, o_qw, o_s = _make(n, k, SCHEMES[0])
    ids = torch.randint(0, n, (2, 3), generator=torch.Generator().manual_seed(2),
                        dtype=torch.int32)
    out = wql.wql_embed_gather(ids.to(DEV), qw)
    empty = wql.wql_embed_gather(torch.empty(0, dtype=torch.int32, device=DEV), qw)
    torch.cuda.synchronize()
    assert out.shape == (2, 3, k) and empty.shape == (0, k)
    want = oracle.embed_gather(ids.reshape(-1).numpy(), o_qw, 4, o_s, oracle.F16, 64, n, k,
                               oracle.F16)
    assert np.array_equal(np_bits(out.reshape(6, k)), want)


@pytest.mark.parametrize("scheme", [SCHEMES[0], SCHEMES[4], SCHEMES[1]],
                         ids=lambda s: f"w{s[0]}g{s[1]}s{s[2]}")
def test_static_weights_back_to_back(scheme):
    """WQL_WEIGHT_STATIC: the decode kernel copies the weight before the
    preceding kernel on the stream has finished.  Calls issued back to back
    (each one's X written by a copy kernel right before it) give exactly the
    results of calls without the flag, and match the oracle."""
    n, k, K = 4099, 512, 8
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=21)
    qs = wql.QuantizedWeight(qw.qweight, qw.scales, qw.bits, qw.group, qw.n, qw.k, static=True)
    ws1, ws2 = wql.Workspace(DEV), wql.Workspace(DEV)
    for m in (1, 4, 16):
        xs = [synth.activations(m, k, xdt, seed=600 + 10 * m + i) for i in range(4)]
        xd = torch.empty(m, k, dtype=TORCH_OF[xdt], device=DEV)
        outs = []
        for x in xs:              # copy X in, then the static call, back to back
            xd.copy_(x.to(DEV), non_blocking=True)
            outs.append(tuple(t.clone() for t in wql.wql_logits(xd, qs, topk=K, workspace=ws1)))
        torch.cuda.synchronize()
        for x, (lg, idx, val) in zip(xs, outs):
            rl, ri, rv = wql.wql_logits(x.to(DEV), qw, topk=K, workspace=ws2)
            torch.cuda.synchronize()
            assert torch.equal(lg, rl) and torch.equal(idx, ri) and torch.equal(val, rv)
        ref, absacc = oracle.logits(np_input(xs[-1], xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                    nthreads=4)
        assert_logits_close(to_f64(outs[-1][0]), ref, absacc, f"static m={m}")


@pytest.mark.parametrize("m", [9, 16])
def test_logits_long_rows_many_tokens(m):
    """k = 5120 with up to 16 bf16 token rows: X for 16 rows (160 KB) does
    not fit in shared memory next to the rings, so the rows run as balanced
    slices (8 + 8, or 5 + 4)."""
    n, k, K = 4099, 5120, 8
    scheme = (4, 128, oracle.BF16, oracle.BF16, oracle.BF16, 0)
    bits, group, sdt, wdt, xdt, clip = scheme
    w, qw, o_qw, o_s = _make(n, k, scheme, seed=31)
    x = synth.activations(m, k, xdt, seed=700 + m)
    n0 = wql.wql_launch_count()
    logits, idx, val = wql.wql_logits(x.to(DEV), qw, topk=K)
    torch.cuda.synchronize()
    assert wql.wql_launch_count() - n0 == (1 if m <= 15 else 2), "balanced decode slices"
    ref, absacc = oracle.logits(np_input(x, xdt), xdt, o_qw, bits, o_s, sdt, group, n, k,
                                nthreads=8)
    assert_logits_close(to_f64(logits), ref, absacc, f"long rows m={m}")
    g_idx, g_val = idx.cpu().numpy(), val.cpu().numpy()
    ties = sum(check_topk(g_idx[r], g_val[r], ref[r], absacc[r], K) for r in range(m))
    report_ties(f"long rows m={m}", ties, m)
