"""Pins for the CPU oracle: each test ties it to something other than itself.

* IEEE conversions against numpy (binary16) and torch (bfloat16) rounding;
* the packed layout against hand-written worked examples (tests/golden);
* the quantiser against a hand-worked example, a brute-force nearest-integer
  search in exact rational arithmetic, library fp16/bf16 rounding of the
  scale, closed-form invariants and exact-arithmetic MSE minimality;
* logits against a dense numpy fp64 product built before packing, and closed
  forms (unit vectors, zero weight, one live group, constant codes);
* top-K against a numpy lexsort brute force; rescoring against numpy dots;
* the tied-embedding gather against a hand-worked word, numpy / torch
  rounding of products formed from the codes before packing, and its
  out-of-range and overflow cases.
"""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import F32, F16, BF16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@np.errstate(over="ignore")
def _f16_bits(a):
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def _bf16_bits(a):
    t = torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _edge_floats():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9,
            2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26,
            2.0 ** -126, 2.0 ** -133, 2.0 ** -134, 1e-8, -1e-8, 3.4e38, 1.0009765625,
            1.00048828125, 1.00146484375, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 255.5, 256.5]
    return np.array(vals, dtype=np.float32)


def _random_floats(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(-2.0, 2.0, n)
    ex = rng.integers(-30, 20, n)
    v = (mant * np.exp2(ex)).astype(np.float32)
    # exact binary16 / bfloat16 ties: halfway between two neighbours
    base = rng.uniform(-100, 100, n // 8).astype(np.float16).astype(np.float32)
    ties16 = base + np.abs(base) * np.float32(2.0 ** -11)
    return np.concatenate([v, ties16.astype(np.float32)])


# --------------------------------------------------------------------------
# conversions
# --------------------------------------------------------------------------

def test_f16_rounding_matches_numpy(oracle_mod):
    v = np.concatenate([_edge_floats(), _random_floats(20000, 0)])
    np.testing.assert_array_equal(oracle.f32_to_f16_bits(v), _f16_bits(v))


def test_bf16_rounding_matches_torch(oracle_mod):
    v = np.concatenate([_edge_floats(), _random_floats(20000, 1)])
    np.testing.assert_array_equal(oracle.f32_to_bf16_bits(v), _bf16_bits(v))


def test_f16_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_bf16_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_bits_to_f64(bits)
    ref = torch.tensor(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


# --------------------------------------------------------------------------
# packing
# --------------------------------------------------------------------------

def _read_pack_golden():
    cases = []
    with open(os.path.join(GOLDEN, "pack_int4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            cases.append(([int(t) for t in lhs.split()], int(rhs.strip(), 16)))
    return cases


def test_pack_worked_examples(oracle_mod):
    cases = _read_pack_golden()
    assert len(cases) >= 5
    nib = np.array([c[0] for c in cases], dtype=np.uint8)
    words = oracle.pack_int4(nib).view(np.uint32)[:, 0]
    np.testing.assert_array_equal(words, np.array([c[1] for c in cases], dtype=np.uint32))


def test_pack_every_value_every_position(oracle_mod):
    rows = []
    expect = []
    for j in range(8):
        for v in range(16):
            r = [0] * 8
            r[j] = v
            rows.append(r)
            expect.append(v << (4 * (4 * (j % 2) + j // 2)))
    words = oracle.pack_int4(np.array(rows, dtype=np.uint8)).view(np.uint32)[:, 0]
    np.testing.assert_array_equal(words, np.array(expect, dtype=np.uint32))


def test_pack_unpack_roundtrip(oracle_mod):
    rng = np.random.default_rng(3)
    nib = rng.integers(0, 16, (37, 96), dtype=np.uint8)
    packed = oracle.pack_int4(nib)
    assert packed.shape == (37, 12) and packed.dtype == np.int32
    np.testing.assert_array_equal(oracle.unpack_int4(packed, 96), nib)


# --------------------------------------------------------------------------
# quantiser
# --------------------------------------------------------------------------

def test_quantize_worked_example(oracle_mod):
    lines = {}
    with open(os.path.join(GOLDEN, "quant_rtn_worked.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, val = line.split(":", 1)
            lines[key.strip()] = val.split()
    w = np.array([float(t) for t in lines["w"]], dtype=np.float32)[None, :]
    q, s, _ = oracle.quantize(w, F32, 4, 8, F16, 0)
    assert int(s[0, 0]) == int(lines["scale_f16_hex"][0], 16)
    np.testing.assert_array_equal(q[0], np.array([int(t) for t in lines["q"]]))
    np.testing.assert_array_equal((q[0].astype(np.int32) + 8),
                                  np.array([int(t) for t in lines["nibbles"]]))


def _nearest_int_half_even(t: Fraction, lo: int, hi: int) -> int:
    """Brute force: the integer in [lo, hi] nearest to t, ties to the even one."""
    best = None
    for q in range(lo, hi + 1):
        d = abs(Fraction(q) - t)
        if best is None or d < best[0] or (d == best[0] and q % 2 == 0):
            best = (d, q)
    return best[1]


def _scale_lib(amax: np.float32, r: float, qmax: int, sdt: int) -> np.float32:
    prod = np.float32(amax) * np.float32(r / qmax)     # numpy fp32 multiply (IEEE)
    prod = max(prod, np.float32(1e-8))
    if sdt == F16:
        return np.float32(np.float16(prod))
    return np.float32(torch.tensor(float(prod), dtype=torch.float32).to(torch.bfloat16).item())


@pytest.mark.parametrize("bits,group,sdt,wdt", [(4, 64, F16, F32), (4, 128, BF16, BF16),
                                                (8, 128, F16, F32), (8, 0, F16, F16)])
def test_quantize_rtn_brute_force(oracle_mod, bits, group, sdt, wdt):
    rng = np.random.default_rng(10 + bits)
    n, k = 6, 256
    w32 = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    w32[2, :] = 0.0                                    # an all-zero (padded) row
    wt = torch.tensor(w32)
    if wdt == F16:
        warr = wt.half().numpy()
        wval = warr.astype(np.float32)
    elif wdt == BF16:
        wb = wt.to(torch.bfloat16)
        warr = wb.view(torch.int16).numpy().view(np.uint16)
        wval = wb.float().numpy()
    else:
        warr = w32
        wval = w32
    q, s, _ = oracle.quantize(warr, wdt, bits, group, sdt, 0)
    g = k if group == 0 else group
    qmax = 7 if bits == 4 else 127
    qmin = -8 if bits == 4 else -127
    sv = oracle.scales_to_f64(s, sdt)
    for r in range(n):
        for gi in range(k // g):
            blk = wval[r, gi * g:(gi + 1) * g]
            amax = np.float32(np.max(np.abs(blk)))
            s_lib = _scale_lib(amax, 1.0, qmax, sdt)
            assert sv[r, gi] == float(s_lib), (r, gi)
            for j in range(g):
                if s_lib == 0:
                    assert q[r, gi * g + j] == 0
                    continue
                t = Fraction(float(np.float32(blk[j]) / np.float32(s_lib)))  # IEEE fp32 divide
                assert q[r, gi * g + j] == _nearest_int_half_even(t, qmin, qmax)
            if amax > 0:
                j = int(np.argmax(np.abs(blk)))
                assert abs(int(q[r, gi * g + j])) == qmax      # RTN maps amax to +-qmax
    assert np.all(q[2] == 0)                                     # zero group -> zero codes
    assert q.min() >= qmin and q.max() <= qmax


def _exact_err(q, s, w):
    return sum((Fraction(int(qi)) * Fraction(float(s)) - Fraction(float(wi))) ** 2
               for qi, wi in zip(q, w))


def test_quantize_mse_is_minimal_over_clip_grid(oracle_mod):
    rng = np.random.default_rng(7)
    n, k, g = 4, 256, 128
    w32 = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    w32[1, :5] *= 12.0                                  # outliers make clipping pay
    wb = torch.tensor(w32).to(torch.bfloat16)
    warr = wb.view(torch.int16).numpy().view(np.uint16)
    wval = wb.float().numpy()
    q, s, ridx = oracle.quantize(warr, BF16, 4, g, BF16, 1)
    q_rtn, s_rtn, _ = oracle.quantize(warr, BF16, 4, g, BF16, 0)
    sv = oracle.scales_to_f64(s, BF16)
    chose_clipped = 0
    for r in range(n):
        for gi in range(k // g):
            blk = wval[r, gi * g:(gi + 1) * g]
            amax = np.float32(np.max(np.abs(blk)))
            errs = []
            for ratio in oracle.CLIP_RATIOS:
                s_r = _scale_lib(amax, ratio, 7, BF16)
                q_r = [_nearest_int_half_even(Fraction(float(np.float32(b) / s_r)), -8, 7)
                       for b in blk]
                errs.append(_exact_err(q_r, s_r, blk))
            best = min(range(5), key=lambda i: (errs[i], i))
            assert ridx[r, gi] == best
            assert sv[r, gi] == float(_scale_lib(amax, oracle.CLIP_RATIOS[best], 7, BF16))
            chosen = _exact_err(q[r, gi * g:(gi + 1) * g], sv[r, gi], blk)
            assert chosen == errs[best]
            assert chosen <= _exact_err(q_rtn[r, gi * g:(gi + 1) * g],
                                        oracle.scales_to_f64(s_rtn, BF16)[r, gi], blk)
            chose_clipped += best > 0
    assert chose_clipped > 0


def test_quantize_fp16_scale_underflow_gives_zero_codes(oracle_mod):
    w = np.zeros((1, 64), dtype=np.float32)
    w[0, 3] = 1e-9                       # amax/7 underflows in binary16
    q, s, _ = oracle.quantize(w, F32, 4, 64, F16, 0)
    assert int(s[0, 0]) == 0 and np.all(q == 0)
    qb, sb, _ = oracle.quantize(w, F32, 4, 64, BF16, 0)
    assert oracle.scales_to_f64(sb, BF16)[0, 0] > 0     # 1e-8 survives in bf16


def test_quantize_int8_range(oracle_mod):
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    q, _, _ = oracle.quantize(w, F32, 8, 0, F16, 0)
    assert q.min() >= -127 and q.max() <= 127
    assert set(np.abs(q).max(axis=1).tolist()) == {127}


# --------------------------------------------------------------------------
# logits
# --------------------------------------------------------------------------

def _quantized(n, k, bits, group, sdt, seed=0):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    q, s, _ = oracle.quantize(w, F32, bits, group, sdt, 0)
    if bits == 4:
        qw = oracle.pack_int4((q.astype(np.int16) + 8).astype(np.uint8))
    else:
        qw = q
    return q, s, qw


def _dense(q, s, group, sdt):
    n, k = q.shape
    g = k if group == 0 else group
    sv = oracle.scales_to_f64(s, sdt)
    return q.astype(np.float64) * np.repeat(sv, g, axis=1)


@pytest.mark.parametrize("bits,group,sdt,xdt", [(4, 64, F16, F16), (4, 128, BF16, BF16),
                                                (8, 128, F16, F16), (8, 0, F16, F16)])
def test_logits_match_dense_product(oracle_mod, bits, group, sdt, xdt):
    n, k, m = 45, 256, 3
    q, s, qw = _quantized(n, k, bits, group, sdt)
    rng = np.random.default_rng(1)
    x32 = rng.standard_normal((m, k)).astype(np.float32)
    if xdt == F16:
        xarr = x32.astype(np.float16)
        xval = xarr.astype(np.float64)
    else:
        xb = torch.tensor(x32).to(torch.bfloat16)
        xarr = xb.view(torch.int16).numpy().view(np.uint16)
        xval = xb.double().numpy()
    out, absacc = oracle.logits(xarr, xdt, qw, bits, s, sdt, group, n, k)
    wd = _dense(q, s, group, sdt)
    ref = xval @ wd.T
    refabs = np.abs(xval) @ np.abs(wd).T
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * refabs.max())
    np.testing.assert_allclose(absacc, refabs, rtol=1e-12)
    rows = np.array([44, 0, 7, 7], dtype=np.int64)
    sub, _ = oracle.logits(xarr, xdt, qw, bits, s, sdt, group, n, k, rows=rows, nthreads=3)
    np.testing.assert_array_equal(sub, out[:, rows])


def test_logits_closed_forms(oracle_mod):
    n, k, g = 16, 128, 64
    q, s, qw = _quantized(n, k, 4, g, F16, seed=2)
    sv = oracle.scales_to_f64(s, F16)
    # x = e_kk picks column kk of the dequantised weight, exactly
    for kk in (0, 5, 63, 64, 127):
        x = np.zeros((1, k), dtype=np.float16)
        x[0, kk] = 1.0
        out, _ = oracle.logits(x, F16, qw, 4, s, F16, g, n, k)
        np.testing.assert_array_equal(out[0], q[:, kk] * sv[:, kk // g])
    # all-zero codes (nibble 8) give zero logits
    zero = oracle.pack_int4(np.full((n, k), 8, dtype=np.uint8))
    x = np.ones((2, k), dtype=np.float16)
    out, absacc = oracle.logits(x, F16, zero, 4, s, F16, g, n, k)
    assert np.all(out == 0) and np.all(absacc == 0)
    # constant code c with x = 1 over one live group: c * s * 64
    nib = np.full((n, k), 8, dtype=np.uint8)
    nib[:, 64:] = 8 + 3
    out, _ = oracle.logits(x, F16, oracle.pack_int4(nib), 4, s, F16, g, n, k)
    np.testing.assert_array_equal(out[0], 3 * sv[:, 1] * 64)
    # bias is added once
    b = np.linspace(-1, 1, n).astype(np.float16)
    outb, _ = oracle.logits(x, F16, oracle.pack_int4(nib), 4, s, F16, g, n, k, bias=b)
    np.testing.assert_array_equal(outb[0], out[0] + b.astype(np.float64))


# --------------------------------------------------------------------------
# top-K and rescoring
# --------------------------------------------------------------------------

def test_topk_matches_lexsort(oracle_mod):
    rng = np.random.default_rng(11)
    vals = rng.integers(-20, 20, (5, 300)).astype(np.float64)   # many exact ties
    vals[2, :] = 1.0
    for K in (1, 4, 8, 16):
        idx, val = oracle.topk(vals, K)
        for r in range(vals.shape[0]):
            order = np.lexsort((np.arange(vals.shape[1]), -vals[r]))[:K]
            np.testing.assert_array_equal(idx[r], order)
            np.testing.assert_array_equal(val[r], vals[r, order])
    small, _ = oracle.topk(vals[:, :3], 5)
    assert np.all(small[:, 3:] == -1)


def test_rescore_matches_numpy_dot(oracle_mod):
    rng = np.random.default_rng(12)
    n, k, m, K = 50, 64, 3, 8
    wref = (rng.standard_normal((n, k)) * 0.02).astype(np.float16)
    x = rng.standard_normal((m, k)).astype(np.float16)
    idx = rng.integers(0, n, (m, K)).astype(np.int32)
    out, absacc = oracle.rescore(x, F16, wref, F16, idx)
    for r in range(m):
        for t in range(K):
            ref = np.dot(x[r].astype(np.float64), wref[idx[r, t]].astype(np.float64))
            assert abs(out[r, t] - ref) <= 1e-13
    # a planted large row wins the argmax
    wref[17] = 1.0
    x = np.abs(x)
    idx[:, 0] = 17
    out, _ = oracle.rescore(x, F16, wref, F16, idx)
    assert np.all(np.argmax(out, axis=1) == 0)


# --------------------------------------------------------------------------
# tied-embedding gather
# --------------------------------------------------------------------------

def test_embed_gather_worked_example(oracle_mod):
    # codes -8..-1 in elements 0..7: nibbles 0..7, even elements in the low
    # half (0x6420), odd in the high half (0x7531); scale 0.5
    word = np.array([[0x75316420]], dtype=np.uint32).view(np.int32)
    scale = np.array([[0x3800]], dtype=np.uint16)            # fp16 0.5
    out = oracle.embed_gather(np.array([0]), word, 4, scale, F16, 8, 1, 8, F16)
    want = [0xC400, 0xC300, 0xC200, 0xC100, 0xC000, 0xBE00, 0xBC00, 0xB800]   # -4 .. -0.5
    assert out[0].tolist() == want


@pytest.mark.parametrize("bits,group,sdt,odt", [(4, 64, F16, F16), (4, 128, BF16, BF16),
                                                (4, 0, F16, BF16), (8, 64, BF16, F16),
                                                (8, 0, F16, F16)])
def test_embed_gather_matches_library_rounding(oracle_mod, bits, group, sdt, odt):
    rng = np.random.default_rng(bits + group + 3 * sdt + odt)
    n, k = 37, 256
    g = k if group == 0 else group
    if bits == 4:
        q = rng.integers(-8, 8, (n, k)).astype(np.int8)
        qw = oracle.pack_int4((q + 8).astype(np.uint8))
    else:
        q = rng.integers(-127, 128, (n, k)).astype(np.int8)
        qw = q
    s32 = (rng.standard_normal((n, k // g)) * 0.05).astype(np.float32)
    sbits = _f16_bits(s32) if sdt == F16 else _bf16_bits(s32)
    sval = (sbits.view(np.float16).astype(np.float64) if sdt == F16 else
            torch.tensor(sbits.view(np.int16)).view(torch.bfloat16).double().numpy())
    ids = np.array([0, 36, 5, 5, -1, 37, 1000, 12], dtype=np.int32)
    out = oracle.embed_gather(ids, qw, bits, sbits, sdt, group, n, k, odt)
    for i, r in enumerate(ids):
        if 0 <= r < n:
            exact = q[r].astype(np.float64) * np.repeat(sval[r], g)    # exact in fp32 too
            want = _f16_bits(exact.astype(np.float32)) if odt == F16 else \
                _bf16_bits(exact.astype(np.float32))
            np.testing.assert_array_equal(out[i], want)
        else:
            assert not out[i].any()                                   # +0 rows


def test_embed_gather_overflow_and_int8_extremes(oracle_mod):
    q = np.array([[127, -127, 1, 0, 0, 0, 0, 0]], dtype=np.int8)
    fmax = np.array([[0x7BFF]], dtype=np.uint16)                      # fp16 65504
    out16 = oracle.embed_gather(np.array([0]), q, 8, fmax, F16, 8, 1, 8, F16)
    assert out16[0, :3].tolist() == [0x7C00, 0xFC00, 0x7BFF]          # +inf, -inf, 65504
    outbf = oracle.embed_gather(np.array([0]), q, 8, fmax, F16, 8, 1, 8, BF16)
    np.testing.assert_array_equal(outbf[0, :3], _bf16_bits([127 * 65504.0, -127 * 65504.0,
                                                            65504.0]))


# --------------------------------------------------------------------------
# fp8 e4m3 per-row head
# --------------------------------------------------------------------------

def _torch_e4m3_decode(bits):
    return torch.tensor(np.asarray(bits, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_all_patterns(oracle_mod):
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(bits)
    want = _torch_e4m3_decode(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2       # 0x7F, 0xFF
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_rounding(oracle_mod):
    rng = np.random.default_rng(4)
    finite = _torch_e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = np.unique(finite[~np.isnan(finite)])
    mids = (finite[:-1] + finite[1:]) / 2                                 # exact ties
    v = np.concatenate([finite, mids, -mids, rng.uniform(-448, 448, 4000),
                        rng.uniform(-1, 1, 2000) * 2.0 ** rng.integers(-12, 2, 2000)])
    v = v.astype(np.float32)                                              # one rounding each
    v = v[np.abs(v) <= 448]
    got = oracle.f64_to_e4m3(v.astype(np.float64))
    want = torch.tensor(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, want)


def test_e4m3_encode_saturates(oracle_mod):
    # reading: beyond the largest finite value the code saturates at +-448
    got = oracle.f64_to_e4m3([449.0, 480.0, 1e30, -465.0, -1e30])
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


@pytest.mark.parametrize("sdt", [F16, BF16])
def test_quantize_fp8_is_nearest_and_hits_the_range(oracle_mod, sdt):
    rng = np.random.default_rng(sdt)
    n, k = 6, 96
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    w[2] = 0.0                                                            # zero row
    w[3, 7] = -0.5                                                        # outlier
    q, s = oracle.quantize_fp8(w, F32, sdt)
    sval = (s.view(np.float16).astype(np.float64) if sdt == F16 else
            torch.tensor(s.view(np.int16)).view(torch.bfloat16).double().numpy())
    finite = _torch_e4m3_decode(np.arange(256, dtype=np.uint8))
    codes = [c for c in range(256) if not np.isnan(finite[c])]
    for r in range(n):
        if sval[r] == 0.0:
            assert not q[r].any()
            continue
        amax_col = int(np.argmax(np.abs(w[r])))
        if np.abs(w[r]).max() > 0:
            assert abs(finite[q[r, amax_col]]) == 448.0                   # the row's amax
        for c in range(k):
            t = Fraction(float(np.float32(np.float32(w[r, c]) / np.float32(sval[r]))))
            t = max(Fraction(-448), min(Fraction(448), t))
            best = min(abs(Fraction(float(finite[cd])) - t) for cd in codes)
            ties = [cd for cd in codes if abs(Fraction(float(finite[cd])) - t) == best]
            chosen = int(q[r, c])
            assert chosen in ties or (finite[chosen] == 0.0 and any(finite[cd] == 0.0 for cd in ties))
            if len({float(finite[cd]) for cd in ties}) > 1:               # exact tie: even mantissa
                assert chosen & 1 == 0


def test_logits_fp8_match_dense_product(oracle_mod):
    rng = np.random.default_rng(8)
    n, k, m = 40, 128, 3
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    q, s = oracle.quantize_fp8(w, F32, F16)
    x = rng.standard_normal((m, k)).astype(np.float16)
    dense = _torch_e4m3_decode(q) * s.view(np.float16).astype(np.float64)[:, None]
    want = x.astype(np.float64) @ dense.T
    got, absacc = oracle.logits_fp8(x.view(np.uint16), F16, q, s, F16)
    assert np.all(np.abs(got - want) <= 1e-12 * absacc + 1e-300)
    np.testing.assert_allclose(absacc, np.abs(x.astype(np.float64)) @ np.abs(dense).T, rtol=1e-12)


# --------------------------------------------------------------------------
# zero-point (asymmetric) int4
# --------------------------------------------------------------------------

def test_asym_int4_worked_example(oracle_mod):
    # min -0.3, max 0.45: s = RN_fp16(0.75 / 15) = 0x2A66 (0.049988...), z = rint(0.3 / s) = 6,
    # q = rint(w / s) + 6: -0.3 -> 0, 0 -> 6, 0.2 -> 10, 0.45 -> 15, -0.1 -> 4, 0.05 -> 7,
    # 0.3 -> 12, 0.15 -> 9 (worked by hand)
    w = np.array([[-0.3, 0.0, 0.2, 0.45, -0.1, 0.05, 0.3, 0.15]], dtype=np.float32)
    q, s, z = oracle.quantize_asym_int4(w, F32, 8, F16)
    assert q[0].tolist() == [0, 6, 10, 15, 4, 7, 12, 9]
    assert s[0, 0] == 0x2A66 and z[0, 0] == 6


@pytest.mark.parametrize("sdt", [F16, BF16])
def test_asym_int4_codes_are_nearest(oracle_mod, sdt):
    rng = np.random.default_rng(10 + sdt)
    n, k, g = 5, 128, 32
    w = (rng.standard_normal((n, k)) * 0.02 + rng.uniform(-0.01, 0.01, (n, 1))).astype(np.float32)
    w[1, :g] = 0.0                                        # zero group
    w[2, g:2 * g] = np.abs(w[2, g:2 * g])                 # one-signed group: min is 0
    q, s, z = oracle.quantize_asym_int4(w, F32, g, sdt)
    sval = (s.view(np.float16).astype(np.float64) if sdt == F16 else
            torch.tensor(s.view(np.int16)).view(torch.bfloat16).double().numpy())
    assert q.max() <= 15 and z.max() <= 15
    for r in range(n):
        for c in range(k):
            gi = c // g
            if sval[r, gi] == 0.0:
                assert q[r, c] == 0 and z[r, gi] == 0
                continue
            t = Fraction(float(np.float32(w[r, c]) / np.float32(sval[r, gi])))
            zz = int(z[r, gi])
            dist = {qq: abs(Fraction(qq - zz) - t) for qq in range(16)}
            best = min(dist.values())
            ties = [qq for qq, d in dist.items() if d == best]
            assert int(q[r, c]) in ties
            if len(ties) > 1:
                assert (int(q[r, c]) - zz) % 2 == 0         # halfway: rint to even
            if w[r, c] == 0.0:
                assert q[r, c] == zz                      # zero is exact
    # the group's zero point reproduces its minimum within half a step
    for r in range(n):
        for gi in range(k // g):
            if sval[r, gi] == 0.0:
                continue
            lo = min(0.0, float(w[r, gi * g:(gi + 1) * g].min()))
            assert abs(-int(z[r, gi]) * sval[r, gi] - lo) <= sval[r, gi] / 2 + 1e-12


def test_asym_int4_logits_match_dense_product(oracle_mod):
    rng = np.random.default_rng(12)
    n, k, g, m = 30, 256, 64, 2
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_asym_int4(w, F32, g, F16)
    x = rng.standard_normal((m, k)).astype(np.float16)
    sv = np.repeat(s.view(np.float16).astype(np.float64), g, axis=1)
    dense = (q.astype(np.float64) - np.repeat(z.astype(np.float64), g, axis=1)) * sv
    want = x.astype(np.float64) @ dense.T
    got, absacc = oracle.logits_asym_int4(x.view(np.uint16), F16, q, s, z, F16, g)
    assert np.all(np.abs(got - want) <= 1e-12 * absacc + 1e-300)
