"""C-ABI checks that need no GPU: the library loads, exports every function
include/mla.h declares, and refuses bad arguments on the host before any
launch (fake, aligned device addresses are never dereferenced on these paths).
"""
import ctypes
import os
import re

import pytest

import mla_latent_kv_07_gb300 as mla
from mla_latent_kv_07_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")

FAKE = 0x7F0000000000  # 16-byte aligned, never touched


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return mla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("mla_cache_append", "mla_decode", "mla_decode_sparse", "mla_workspace_size",
                 "mla_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_only_the_abi_is_exported():
    out = os.popen(f"nm -D --defined-only {mla.LIB_PATH}").read()
    syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {s for s in syms if s.startswith("mla_")}
    assert ours == set(declared_functions())


def test_status_strings(L):
    for code, name in mla.STATUS.items():
        assert L.mla_status_string(code).decode() == name


def _cache(fmt=0, B=2, S=64, scale=True):
    return mla._CCache(fmt, B, S, FAKE, FAKE + 4096 if (fmt in (1, 2) and scale) else None, FAKE + 8192)


def test_append_rejects_bad_arguments(L):
    c = _cache()
    pos = (ctypes.c_int32 * 2)(0, 63)
    ok_args = (ctypes.byref(c), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), pos, 2, None)
    assert L.mla_cache_append(None, *ok_args[1:]) == 1
    bad = (ctypes.c_int32 * 2)(0, 64)                      # == max_seq_len
    assert L.mla_cache_append(ctypes.byref(c), ok_args[1], ok_args[2], bad, 2, None) == 2
    neg = (ctypes.c_int32 * 2)(-1, 3)
    assert L.mla_cache_append(ctypes.byref(c), ok_args[1], ok_args[2], neg, 2, None) == 2
    assert L.mla_cache_append(ctypes.byref(c), ok_args[1], ok_args[2], pos, 3, None) == 1  # B > max_batch
    assert L.mla_cache_append(ctypes.byref(c), ctypes.c_void_p(FAKE + 8), ok_args[2], pos, 2, None) == 1
    c8 = _cache(fmt=1, scale=False)                        # FP8 without scales
    assert L.mla_cache_append(ctypes.byref(c8), ok_args[1], ok_args[2], pos, 2, None) == 1
    c82 = _cache(fmt=2, scale=False)                       # power-of-two FP8 without scales
    assert L.mla_cache_append(ctypes.byref(c82), ok_args[1], ok_args[2], pos, 2, None) == 1
    cx = _cache(fmt=7)
    assert L.mla_cache_append(ctypes.byref(cx), ok_args[1], ok_args[2], pos, 2, None) == 3
    wide = _cache(B=4096)                                  # more rows than one call may write
    many = (ctypes.c_int32 * 2049)(*([0] * 2049))
    assert L.mla_cache_append(ctypes.byref(wide), ok_args[1], ok_args[2], many, 2049, None) == 1


def test_decode_rejects_bad_arguments(L):
    c = _cache()
    f = ctypes.c_void_p(FAKE)

    def dec(B=2, H=128, max_end=64, cache=c, q=f, out=f, scale=0.1):
        return L.mla_decode(ctypes.byref(cache), q, f, f, max_end, B, H, scale, out, None, f, 1 << 30, None)

    assert dec(H=48) == 3                                   # unsupported head count
    assert dec(B=3) == 1                                    # B > max_batch
    assert dec(max_end=65) == 2                             # past max_seq_len
    assert dec(max_end=0) == 2
    assert dec(q=ctypes.c_void_p(FAKE + 2)) == 1            # misaligned
    assert dec(out=None) == 1
    assert dec(scale=float("nan")) == 1


def test_decode_append_rejects_bad_arguments(L):
    c = _cache(fmt=1)
    f = ctypes.c_void_p(FAKE)

    def da(kv=f, pe=f, B=2, H=128, max_end=64):
        return L.mla_decode_append(ctypes.byref(c), kv, pe, f, f, f, max_end, B, H, 0.1, f, None, f,
                                   1 << 30, None)

    assert da(kv=None) == 1
    assert da(pe=None) == 1
    assert da(kv=ctypes.c_void_p(FAKE + 8)) == 1            # misaligned new rows
    assert da(B=3) == 1                                     # B > max_batch
    assert da(H=48) == 3
    assert da(max_end=65) == 2


def test_sparse_rejects_bad_arguments(L):
    c = _cache(fmt=1)
    f = ctypes.c_void_p(FAKE)

    def sp(K=2048, topk=f, kv_new=None, pe_new=None):
        return L.mla_decode_sparse(ctypes.byref(c), f, f, f, 64, 2, 128, 0.1, topk, K, kv_new, pe_new,
                                   f, None, None, None, f, 1 << 30, None)

    assert sp(K=0) == 1
    assert sp(K=8193) == 1
    assert sp(topk=None) == 1
    assert sp(kv_new=f, pe_new=None) == 1                   # one of the pair only
    big = _cache(fmt=1, B=2, S=1 << 30)                     # row index b * S + pos past int32
    assert L.mla_decode_sparse(ctypes.byref(big), f, f, f, 64, 2, 128, 0.1, f, 2048, None, None,
                               f, None, None, None, f, 1 << 30, None) == 3


def test_topk_select_rejects_bad_arguments(L):
    f = ctypes.c_void_p(FAKE)
    assert L.mla_topk_select(None, f, 2, 64, 8, f, None) == 1
    assert L.mla_topk_select(f, f, 2, 64, 8, None, None) == 1
    assert L.mla_topk_select(ctypes.c_void_p(FAKE + 2), f, 2, 64, 8, f, None) == 1   # misaligned
    assert L.mla_topk_select(f, f, 0, 64, 8, f, None) == 1
    assert L.mla_topk_select(f, f, 2, 0, 8, f, None) == 1
    assert L.mla_topk_select(f, f, 2, 64, 0, f, None) == 1
    assert L.mla_topk_select(f, f, 2, 64, 8193, f, None) == 1


def test_workspace_size_rejects_bad_arguments(L):
    assert L.mla_workspace_size(0, 128, 64, 0) == 0
    assert L.mla_workspace_size(4, 24, 64, 0) == 0
    assert L.mla_workspace_size(4, 128, 64, -1) == 0
    assert L.mla_workspace_size(4, 128, 64, 9000) == 0


def test_trace_counts_launches_without_events(L):
    # max_records = 0 only counts launches: no events are created, so this
    # needs no GPU; a second begin while tracing is on, and a negative count,
    # are refused
    assert L.mla_trace_begin(-1) == 1
    assert L.mla_trace_begin(0) == 0
    try:
        assert L.mla_trace_begin(0) == 1
    finally:
        ms, n, k = ctypes.c_float(1.0), ctypes.c_int32(1), ctypes.c_int32(1)
        assert L.mla_trace_end(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(k)) == 0
    assert (ms.value, n.value, k.value) == (0.0, 0, 0)
    assert L.mla_trace_end(None, None, None) == 1   # not tracing


def test_read_ceiling_rejects_bad_arguments(L):
    f = ctypes.c_void_p(FAKE)
    assert L.mla_read_ceiling(None, 1024, f, None) == 1
    assert L.mla_read_ceiling(f, 0, f, None) == 1
    assert L.mla_read_ceiling(f, 1000, f, None) == 1          # not a multiple of 16
    assert L.mla_read_ceiling(ctypes.c_void_p(FAKE + 8), 1024, f, None) == 1
    assert L.mla_read_ceiling(f, 1024, None, None) == 1


def test_multi_token_decode_rejects_bad_arguments(L):
    c = _cache(fmt=0, B=2, S=64)
    f = ctypes.c_void_p(FAKE)

    def mtp(B=2, s=2, H=128):
        return L.mla_decode_mtp(ctypes.byref(c), f, f, f, 64, B, s, H, 0.1, f, None, f, 1 << 30, None)

    assert mtp(s=0) == 1
    assert mtp(s=1025) == 1
    assert mtp(B=3) == 1                                    # more slots than the cache holds
    assert mtp(H=24) == 3


def test_absorb_and_project_reject_bad_arguments(L):
    f = ctypes.c_void_p(FAKE)
    odd = ctypes.c_void_p(FAKE + 8)
    for fn in (L.mla_absorb_q, L.mla_project_out):
        assert fn(None, f, 4, 8, f, None, None) == 1
        assert fn(f, odd, 4, 8, f, None, None) == 1          # misaligned weights
        assert fn(f, f, 0, 8, f, None, None) == 1
        assert fn(f, f, 4, 0, f, None, None) == 1
        assert fn(f, f, 4, 8, f, ctypes.c_void_p(FAKE + 2), None) == 1   # misaligned status
