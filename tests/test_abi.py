"""The C-ABI library builds, loads and exports every symbol include/kvc.h declares.

Host-side argument validation is exercised too: these calls return before
any CUDA call, so they run without a GPU.
"""

import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_135_gb300 as kvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kvc.build()
    return kvc.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("kvc_build_slot_mapping", "kvc_reshape_and_cache", "kvc_paged_decode"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exported_symbols_are_c_linkage():
    out = subprocess.run(["nm", "-D", "--defined-only", kvc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (kvc_[a-z0-9_]+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_version_and_status_strings(lib):
    assert lib.kvc_version() >= 100
    assert lib.kvc_status_string(0) == b"KVC_OK"
    assert lib.kvc_status_string(4) == b"KVC_ERR_WORKSPACE"
    assert lib.kvc_status_string(99) == b"KVC_UNKNOWN_STATUS"


P = 0x1000  # any non-null pointer value: rejected calls never dereference it


def decode_call(lib, **kw):
    a = dict(q=P, kc=P, vc=P, bt=P, sl=P, out=P, B=2, Hq=8, Hkv=2, D=128, bs=16, maxb=4, NB=8,
             scale=0.125, dtype=1, ctas=0, ws=P, wsb=1 << 20, flag=None, stream=None)
    a.update(kw)
    return lib.kvc_paged_decode(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["out"], a["B"],
                                a["Hq"], a["Hkv"], a["D"], a["bs"], a["maxb"], a["NB"],
                                a["scale"], a["dtype"], a["ctas"], a["ws"], a["wsb"], a["flag"],
                                a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), kvc.KVC_ERR_INVALID_ARG),        # Hq % Hkv != 0
    (dict(Hkv=0), kvc.KVC_ERR_INVALID_ARG),
    (dict(scale=float("nan")), kvc.KVC_ERR_INVALID_ARG),  # no silent default scale
    (dict(dtype=7), kvc.KVC_ERR_INVALID_ARG),
    (dict(q=None), kvc.KVC_ERR_INVALID_ARG),
    (dict(q=P + 2), kvc.KVC_ERR_INVALID_ARG),             # misaligned
    (dict(D=96), kvc.KVC_ERR_UNSUPPORTED),
    (dict(bs=12), kvc.KVC_ERR_UNSUPPORTED),
    (dict(bs=4), kvc.KVC_ERR_UNSUPPORTED),
    (dict(Hq=64, Hkv=2), kvc.KVC_ERR_UNSUPPORTED),        # group 32 > 16
    (dict(B=2000), kvc.KVC_ERR_UNSUPPORTED),
    (dict(B=0), kvc.KVC_OK),                              # nothing to do
])
def test_decode_host_validation(lib, kw, status):
    assert decode_call(lib, **kw) == status


def test_write_host_validation(lib):
    f = lib.kvc_reshape_and_cache
    # value without value_cache
    assert f(P, P, P, None, P, 4, 2, 64, 64, 16, 8, 0, None, None) == kvc.KVC_ERR_INVALID_ARG
    # head dim not a multiple of 8 elements
    assert f(P, None, P, None, P, 4, 2, 60, 0, 16, 8, 0, None, None) == kvc.KVC_ERR_UNSUPPORTED
    assert f(P, None, P, None, P, 0, 2, 64, 0, 16, 8, 0, None, None) == kvc.KVC_OK
    g = lib.kvc_build_slot_mapping
    # decode form needs one token per sequence
    assert g(P, 4, None, P, 2, 3, 16, 8, P, None, None) == kvc.KVC_ERR_INVALID_ARG
    assert g(P, 4, None, P, 2, 0, 16, 8, P, None, None) == kvc.KVC_OK
    assert g(P, 4, None, P, 2, 2, 0, 8, P, None, None) == kvc.KVC_ERR_INVALID_ARG


def test_workspace_query_rejects_bad_shapes(lib):
    assert lib.kvc_paged_decode_workspace_size(6, 4, 128, 10) == 0
    assert lib.kvc_paged_decode_workspace_size(8, 2, 96, 10) == 0
    # explicit CTA count: no device query needed
    # 10 CTAs: counters (padded to 256 B) + 2 shares x 4 rows x (128 + 2) floats each
    assert lib.kvc_paged_decode_workspace_size(8, 2, 128, 10) == 256 + 10 * 2 * 4 * 130 * 4


def test_block_manager_calls_reject_a_null_handle(lib):
    inv = 1  # KVC_ERR_INVALID_ARG
    buf = (ctypes.c_int32 * 8)()
    ids = (ctypes.c_int64 * 2)(0, 1)
    p = ctypes.addressof(buf)
    assert lib.kvc_bm_create(0, 16, 4, ctypes.byref(ctypes.c_void_p())) == inv
    assert lib.kvc_bm_create(4, 16, 4, None) == inv
    lib.kvc_bm_destroy(None)                      # no-op
    assert lib.kvc_bm_num_free(None) == -1
    assert lib.kvc_bm_ref_count(None, 0) == -1
    assert lib.kvc_bm_seq_len(None, 0) == -1
    assert lib.kvc_bm_add(None, 0, 4, None) == inv
    assert lib.kvc_bm_fork(None, 0, 1) == inv
    assert lib.kvc_bm_append(None, 0, p, None, None) == inv
    assert lib.kvc_bm_free(None, 0) == inv
    assert lib.kvc_bm_tables(None, ctypes.addressof(ids), 2, 0, p, None) == inv
    assert lib.kvc_bm_step(None, ctypes.addressof(ids), 2, 0, p, p, p, None, None) == inv
    assert lib.kvc_status_string(5) == b"KVC_ERR_OUT_OF_BLOCKS"
