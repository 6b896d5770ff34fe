"""The C-ABI library loads, exports every symbol include/cpdr.h declares, and
validates on the host before touching the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

from context_merge_gb300 import cpdr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cpdr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpdr_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(cpdr_lib):
    names = declared_symbols()
    assert "cpdr_preprocess" in names and "cpdr_merge" in names and "cpdr_fwd" in names
    for name in names:
        assert hasattr(cpdr_lib, name), name
    assert set(cpdr.EXPORTED) >= set(names)


def test_version(cpdr_lib):
    assert b"sm_103a" in cpdr_lib.cpdr_version()


def make(**kw):
    base = dict(B=1, T=1024, H=2, d=64, R=4, gate="gdn", dtype="fp32", host_only=True)
    base.update(kw)
    return cpdr.Context(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(T=1000, R=3), cpdr.ERR_INVALID),            # not divisible
    (dict(T=2, R=4), cpdr.ERR_INVALID),               # fewer tokens than segments
    (dict(d=96), cpdr.ERR_UNSUPPORTED),
    (dict(B=2, T=100, cu_seqlens=[0, 50, 100], R=2), cpdr.ERR_INVALID),   # packed needs B == 1
    (dict(T=100, cu_seqlens=[0, 60, 50, 100], R=2), cpdr.ERR_INVALID),   # non-monotone
    (dict(T=100, cu_seqlens=[0, 60, 90], R=2), cpdr.ERR_INVALID),        # does not end at T
    (dict(R=0), cpdr.ERR_INVALID),
])
def test_create_validation(cpdr_lib, kw, status):
    with pytest.raises(cpdr.CpdrError) as ei:
        make(**kw)
    assert ei.value.status == status
    assert cpdr_lib.cpdr_last_error()


def test_host_only_context_rejects_launches(cpdr_lib):
    ctx = make()
    rc = cpdr_lib.cpdr_merge(ctx._h, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert rc == cpdr.ERR_INVALID
    assert b"HOST_ONLY" in cpdr_lib.cpdr_last_error()


def test_null_descriptor(cpdr_lib):
    h = ctypes.c_void_p()
    assert cpdr_lib.cpdr_ctx_create(None, ctypes.byref(h)) == cpdr.ERR_INVALID
    assert not h.value


def test_buffer_sizes(cpdr_lib):
    ctx = make(B=2, T=512, H=3, d=128, R=8, dtype="bf16")
    se, m, si, fin = ctx.buffer_sizes()
    assert se == si == 8 * 2 * 3 * 128 * 128 * 4
    assert m == se
    assert fin == 2 * 3 * 128 * 128 * 4
    ws = ctx.host_workspace_bytes()
    assert ws >= 3 * 2 * 512 * 3 * 128 * 2 + se + m + si + fin


@pytest.mark.parametrize("kw", [
    dict(B=1, T=4096, H=4, d=128, R=4, dtype="bf16"),
    dict(B=2, T=1000, H=3, d=128, R=5, dtype="bf16"),
    dict(B=1, T=2048, H=16, d=128, R=2, dtype="bf16", cu_seqlens=[0, 700, 1800, 2048]),
])
def test_wy_workspace_covers_every_chunk_of_every_fragment(cpdr_lib, kw):
    """24 KiB of WY tiles per (64-token chunk of a fragment, head) on the
    tensor-core path; nothing on the CUDA-core path."""
    ctx = make(**kw)
    chunks = sum((f[1] + 63) // 64 for f in ctx.fragments())
    assert ctx.counts()["tc"] == 1
    assert ctx.wy_bytes() == chunks * kw["H"] * 3 * 8192
    simt = make(**kw, force_simt=True)
    assert simt.wy_bytes() == 0
    assert make(**dict(kw, dtype="fp32")).wy_bytes() == 0
    # per-dim gate: the WY tiles plus the pre-gated operand tiles, 113 KiB
    kda = make(**dict(kw, gate="kda"))
    assert kda.counts()["tc"] == 1 and kda.wy_bytes() == chunks * kw["H"] * 113 * 1024
    # grouped query heads with the per-dim gate: query heads past each
    # state's first keep their Qg and P (24 KiB) after the units
    for G in (2, 3):
        gq = make(**dict(kw, gate="kda", Hq=G * kw["H"]))
        assert gq.counts()["tc"] == 1
        assert gq.wy_bytes() == chunks * kw["H"] * (113 + (G - 1) * 24) * 1024


def test_selftest_rejects_host_only_context(cpdr_lib):
    ctx = make()
    rc = cpdr_lib.cpdr_selftest_wait_timeout(ctx._h, ctypes.c_longlong(1000), None)
    assert rc == cpdr.ERR_INVALID
    assert b"HOST_ONLY" in cpdr_lib.cpdr_last_error()
