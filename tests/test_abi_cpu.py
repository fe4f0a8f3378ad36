"""The C ABI without a GPU: the library loads, exports every entry point that
include/wql.h declares, and rejects bad arguments on the host before any CUDA
call (so these checks run anywhere).  No compute call is made here."""
import ctypes
import os
import re

import pytest

import weight_only_quantized_wql_gb300 as wql

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wql.h")
OK, EINVAL, EUNSUPPORTED, ECUDA, EWORKSPACE = 0, 1, 2, 3, 4
A = 0x7F0000100000  # an aligned fake device address: never dereferenced by the checks


@pytest.fixture(scope="module")
def lib():
    return wql.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wql_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("wql_quantize", "wql_pack", "wql_unpack", "wql_workspace_size",
                     "wql_logits", "wql_topk_rescore", "wql_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libwql.so does not export {name}"


def test_status_strings(lib):
    for code, tag in [(OK, "WQL_OK"), (EINVAL, "WQL_EINVAL"), (EUNSUPPORTED, "WQL_EUNSUPPORTED"),
                      (ECUDA, "WQL_ECUDA"), (EWORKSPACE, "WQL_EWORKSPACE")]:
        assert wql.wql_status_string(code).startswith(tag)


def test_workspace_size_arithmetic():
    assert wql.wql_workspace_size(1, 1000, 0) == 256
    s = wql.wql_workspace_size(3, 1000, 8)
    assert s >= 256 + 1024 + 3 * wql.MAX_CTAS * 8 * 8 and s % 256 == 0
    # the need does not grow with the vocab size
    assert wql.wql_workspace_size(3, 10 ** 9, 8) == s
    assert wql.wql_workspace_size(-1, 10, 8) == 0
    assert wql.wql_workspace_size(1, 10, wql.MAX_TOPK + 1) == 0


def _weight(bits=4, group=64, sdt=1, n=1000, k=512, fmt=0, q=A, s=A, z=None):
    return wql._WqlWeight(bits, group, sdt, fmt, n, k, q, s, z)


def _logits(lib, w, x=A, xdt=1, m=2, bias=None, out=A, topk=0, idx=None, val=None, ws=None,
            wsb=0):
    return lib.wql_logits(x, xdt, m, ctypes.byref(w) if w is not None else None, bias, out,
                          topk, idx, val, ws, wsb, None)


def test_logits_argument_checks(lib):
    before = wql.wql_launch_count()
    assert _logits(lib, None) == EINVAL
    assert _logits(lib, _weight(), m=-1) == EINVAL
    assert _logits(lib, _weight(fmt=7)) == EINVAL                # unknown format
    assert _logits(lib, _weight(fmt=0x200)) == EINVAL            # unknown flag
    assert _logits(lib, _weight(fmt=0x100), m=0) == OK           # static-weights flag
    assert _logits(lib, _weight(), x=None) == EINVAL
    assert _logits(lib, _weight(), out=None) == EINVAL           # no logits and no top-K
    assert _logits(lib, _weight(q=None)) == EINVAL
    assert _logits(lib, _weight(), topk=wql.MAX_TOPK + 1) == EINVAL
    assert _logits(lib, _weight(n=4), topk=5, idx=A, val=A) == EINVAL
    assert _logits(lib, _weight(), topk=8) == EINVAL            # no idx/val buffers
    assert _logits(lib, _weight(bits=3)) == EUNSUPPORTED
    assert _logits(lib, _weight(group=96)) == EUNSUPPORTED
    assert _logits(lib, _weight(group=64, k=96)) == EUNSUPPORTED
    assert _logits(lib, _weight(k=520, group=0)) == EUNSUPPORTED
    assert _logits(lib, _weight(sdt=0)) == EUNSUPPORTED
    assert _logits(lib, _weight(), xdt=0) == EUNSUPPORTED
    assert _logits(lib, _weight(), x=A + 2) == EUNSUPPORTED     # x not 16-byte aligned
    assert _logits(lib, _weight(q=A + 8)) == EUNSUPPORTED
    assert _logits(lib, _weight(), topk=8, idx=A, val=A) == EWORKSPACE
    # candidates alone: logits_out NULL with top-K on passes the checks
    assert _logits(lib, _weight(), out=None, topk=8, idx=A, val=A) == EWORKSPACE
    # fp8 e4m3: bits 8 with one scale per row only
    assert _logits(lib, _weight(fmt=1, bits=4, group=0)) == EUNSUPPORTED
    assert _logits(lib, _weight(fmt=1, bits=8, group=64)) == EUNSUPPORTED
    # zero points: int4, a group that is a multiple of 128, a zero-point table
    assert _logits(lib, _weight(fmt=2, group=128)) == EINVAL          # no zeros
    assert _logits(lib, _weight(fmt=2, group=64, z=A)) == EUNSUPPORTED
    assert _logits(lib, _weight(fmt=2, bits=8, group=128, z=A)) == EUNSUPPORTED
    assert _logits(lib, _weight(fmt=2, group=0, z=A)) == EUNSUPPORTED
    need = wql.wql_workspace_size(2, 1000, 8)
    assert _logits(lib, _weight(), topk=8, idx=A, val=A, ws=A, wsb=need - 1) == EWORKSPACE
    assert _logits(lib, _weight(), m=0) == OK                    # empty: nothing launched
    assert _logits(lib, _weight(n=0)) == OK
    assert wql.wql_launch_count() == before


def test_quantize_pack_rescore_argument_checks(lib):
    before = wql.wql_launch_count()
    q = lib.wql_quantize
    assert q(A, 0, -1, 512, 4, 64, 1, 0, A, A, None) == EINVAL
    assert q(A, 0, 10, 512, 4, 64, 1, 2, A, A, None) == EINVAL      # clip mode
    assert q(None, 0, 10, 512, 4, 64, 1, 0, A, A, None) == EINVAL
    assert q(A, 0, 10, 512, 3, 64, 1, 0, A, A, None) == EUNSUPPORTED
    assert q(A, 0, 10, 512, 4, 64, 0, 0, A, A, None) == EUNSUPPORTED  # fp32 scales
    assert q(A, 0, 10, 500, 4, 64, 1, 0, A, A, None) == EUNSUPPORTED
    assert q(A, 0, 0, 512, 4, 64, 1, 0, A, A, None) == OK
    qx = lib.wql_quantize_ex
    assert qx(A, 0, 10, 512, 7, 4, 64, 1, 0, A, A, None, None) == EINVAL          # format
    assert qx(A, 0, 10, 512, 1, 8, 64, 1, 0, A, A, None, None) == EUNSUPPORTED    # e4m3 group
    assert qx(A, 0, 10, 512, 1, 8, 0, 1, 1, A, A, None, None) == EUNSUPPORTED     # e4m3 MSE
    assert qx(A, 0, 10, 512, 1, 4, 0, 1, 0, A, A, None, None) == EUNSUPPORTED     # e4m3 bits
    assert qx(A, 0, 10, 512, 2, 4, 128, 1, 0, A, A, None, None) == EINVAL         # no zeros
    assert qx(A, 0, 10, 512, 2, 4, 64, 1, 0, A, A, A, None) == EUNSUPPORTED       # group 64
    assert qx(A, 0, 10, 512, 2, 8, 128, 1, 0, A, A, A, None) == EUNSUPPORTED      # bits 8
    assert qx(A, 0, 0, 512, 2, 4, 128, 1, 0, A, A, A, None) == OK
    assert lib.wql_pack(A, 4, 12, A, None) == EUNSUPPORTED
    assert lib.wql_pack(None, 4, 16, A, None) == EINVAL
    assert lib.wql_unpack(A, 0, 16, A, None) == OK
    r = lib.wql_topk_rescore
    assert r(A, 1, 2, A, 2, 100, 256, None, 8, A, A, A, None) == EUNSUPPORTED  # dtype mismatch
    assert r(A, 1, 2, A, 1, 100, 252, None, 8, A, A, A, None) == EUNSUPPORTED  # k % 8
    assert r(A, 1, 2, A, 1, 4, 256, None, 8, A, A, A, None) == EINVAL          # topk > n
    assert r(A, 1, 2, A, 1, 100, 256, None, 0, A, A, A, None) == OK            # nothing to do
    assert wql.wql_launch_count() == before


def test_embed_gather_argument_checks(lib):
    before = wql.wql_launch_count()
    e = lib.wql_embed_gather

    def call(w, ids=A, t=4, odt=1, out=A):
        return e(ids, t, ctypes.byref(w) if w is not None else None, odt, out, None)

    assert call(None) == EINVAL
    assert call(_weight(), t=-1) == EINVAL
    assert call(_weight(fmt=7)) == EINVAL
    assert call(_weight(fmt=1, bits=8, group=0)) == EUNSUPPORTED  # fp8 rows: not gathered
    assert call(_weight(), ids=None) == EINVAL
    assert call(_weight(), out=None) == EINVAL
    assert call(_weight(s=None)) == EINVAL
    assert call(_weight(bits=2)) == EUNSUPPORTED
    assert call(_weight(), odt=0) == EUNSUPPORTED                # fp32 output
    assert call(_weight(sdt=0)) == EUNSUPPORTED
    assert call(_weight(k=260, group=0)) == EUNSUPPORTED         # k % 8
    assert call(_weight(group=24, k=512)) == EUNSUPPORTED        # k % group
    assert call(_weight(), out=A + 8) == EUNSUPPORTED            # out not 16-byte aligned
    assert call(_weight(q=A + 4)) == EUNSUPPORTED                # qweight not 8-byte aligned
    assert call(_weight(), ids=A + 2) == EUNSUPPORTED
    assert call(_weight(), t=0) == OK                            # nothing launched
    assert call(_weight(), t=0, ids=None, out=None) == OK
    assert wql.wql_launch_count() == before


def test_binding_refuses_host_tensors(lib):
    """There is no CPU path: every entry point raises on host tensors before
    any library call (nothing is launched, nothing falls back)."""
    before = wql.wql_launch_count()
    import torch
    n, k = 64, 128
    qw = wql.QuantizedWeight(torch.zeros(n, k // 8, dtype=torch.int32),
                             torch.zeros(n, k // 64, dtype=torch.float16), 4, 64, n, k)
    x = torch.zeros(2, k, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wql.wql_quantize(torch.zeros(n, k), 4, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wql.wql_logits(x, qw, topk=0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wql.wql_embed_gather(torch.zeros(3, dtype=torch.int32), qw)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wql.wql_topk_rescore(x, torch.zeros(n, k, dtype=torch.float16),
                             torch.zeros(2, 8, dtype=torch.int32),
                             torch.zeros(2, 8), torch.zeros(2, n, dtype=torch.float16))
    assert wql.wql_launch_count() == before


def test_missing_library_raises(monkeypatch):
    """A missing libwql.so is an error, not a fallback."""
    from weight_only_quantized_wql_gb300 import _build
    monkeypatch.setattr(wql, "_lib", None)
    monkeypatch.setattr(_build, "LIB", "/nonexistent/libwql.so")
    with pytest.raises(RuntimeError, match="libwql.so not found"):
        wql.load(build_if_missing=False)


def test_debug_set_waits_rejects_bad_arguments(lib):
    assert lib.wql_debug_set_waits(-1, 0) == EINVAL
    assert lib.wql_debug_set_waits(0, 2) == EINVAL
    assert lib.wql_debug_set_waits(0, 0) == OK
