"""The C-ABI library loads and exports every function include/vg.h declares,
and host-side argument checks return their status without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "self_speculative_sparse_vg_gb300", "libvg.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from self_speculative_sparse_vg_gb300 import build
        build.build()
    return ctypes.CDLL(LIB)


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(vg_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_exports_match_header():
    from self_speculative_sparse_vg_gb300 import vg
    assert sorted(vg.EXPORTED) == _declared_functions()


def test_status_strings_and_version(lib):
    lib.vg_status_string.restype = ctypes.c_char_p
    lib.vg_version.restype = ctypes.c_char_p
    assert lib.vg_status_string(0) == b"VG_OK"
    assert lib.vg_status_string(3) == b"VG_ERR_WORKSPACE_TOO_SMALL"
    assert lib.vg_version().decode().count(".") == 2


def _kv(head_dim=128, page_size=16, k=0x1000, v=0x2000, table=0x3000):
    from self_speculative_sparse_vg_gb300.vg import PagedKVStruct
    return PagedKVStruct(k, v, table, 100, page_size, 64, 8, head_dim)


def test_host_argument_checks_without_gpu():
    """Every call below is rejected by host validation before any CUDA call."""
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.vg import PagedKVStruct
    L = vg._lib
    fake = ctypes.c_void_p(0x4000)
    # null KV struct / null pointers
    assert L.vg_verify_attention(None, fake, fake, 1, 6, 32, 100, 0.1, fake, 1, fake, 0, None, 0,
                                 None, None) == 1
    kv = _kv()
    assert L.vg_verify_attention(ctypes.byref(kv), None, fake, 1, 6, 32, 100, 0.1, fake, 1, fake,
                                 0, None, 0, None, None) == 1
    # unsupported head_dim and page size
    assert L.vg_verify_attention(ctypes.byref(_kv(head_dim=96)), fake, fake, 1, 6, 32, 100, 0.1,
                                 fake, 1, fake, 0, None, 0, None, None) == 2
    assert L.vg_verify_attention(ctypes.byref(_kv(page_size=32)), fake, fake, 1, 6, 32, 100, 0.1,
                                 fake, 1, fake, 0, None, 0, None, None) == 2
    # misaligned pool base
    assert L.vg_verify_attention(ctypes.byref(_kv(k=0x1004)), fake, fake, 1, 6, 32, 100, 0.1,
                                 fake, 1, fake, 0, None, 0, None, None) == 1
    # group too large (g = 16), too many rows
    assert L.vg_verify_attention(ctypes.byref(kv), fake, fake, 1, 2, 128, 100, 0.1, fake, 1, fake,
                                 0, None, 0, None, None) == 2
    assert L.vg_verify_attention(ctypes.byref(kv), fake, fake, 1, 17, 32, 100, 0.1, fake, 1, fake,
                                 0, None, 0, None, None) == 2
    # capture requested without a buffer; bad capture mode
    assert L.vg_verify_attention(ctypes.byref(kv), fake, fake, 1, 6, 32, 100, 0.1, fake, 1, None,
                                 0, None, 0, None, None) == 1
    assert L.vg_verify_attention(ctypes.byref(kv), fake, fake, 1, 6, 32, 100, 0.1, fake, 9, fake,
                                 0, None, 0, None, None) == 1
    # cache too small for max_prefix + rows (64 pages * 16 = 1024 positions)
    assert L.vg_verify_attention(ctypes.byref(kv), fake, fake, 1, 6, 32, 1020, 0.1, fake, 1, fake,
                                 0, None, 0, None, None) == 1
    # missing workspace when the plan needs split partials (20 forced splits:
    # more than one cluster holds, so they merge through the workspace)
    kv2 = PagedKVStruct(0x1000, 0x2000, 0x3000, 400, 16, 400, 8, 128)
    assert L.vg_verify_workspace_bytes(1, 6, 32, 8, 128, 5000, 24) > 0
    assert L.vg_verify_attention(ctypes.byref(kv2), fake, fake, 1, 6, 32, 5000, 0.1, fake, 1, fake,
                                 24, None, 0, None, None) == 3
    # select: cap too small, bad mode, non-divisible heads
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 5000, 100, 4, 16, 0, fake, fake, 50, None,
                          None, None, 0, None, None) == 1
    assert L.vg_select_kv(fake, 0, fake, 1, 32, 8, 5000, 100, 4, 16, 0, fake, fake, 200, None,
                          None, None, 0, None, None) == 1
    assert L.vg_select_kv(fake, 1, fake, 1, 30, 8, 5000, 100, 4, 16, 0, fake, fake, 200, None,
                          None, None, 0, None, None) == 1
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 300000, 100, 4, 16, 0, fake, fake, 200, None,
                          None, None, 0, None, None) == 2
    # select: launch count of an invalid or unsupported shape (no device needed)
    assert L.vg_select_launches(0, 0, 8, 5000, 0) == 0
    assert L.vg_select_launches(0, 1, 8, 300000, 0) == 0
    assert L.vg_select_launches(7, 1, 8, 5000, 0) == 0
    # select: the score-key workspace is missing or too small
    assert L.vg_select_workspace_bytes(1, 8, 5000, 0) >= 5000 * 4
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 5000, 100, 4, 16, 0, fake, fake, 200, None,
                          None, None, 0, None, None) == 3
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 5000, 100, 4, 16, 1, fake, fake, 200, None,
                          None, fake, 5000 * 4, None, None) == 3
    # select: slots without the cache, or a page table too short for max_prefix
    ws = L.vg_select_workspace_bytes(1, 8, 5000, 0)
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 5000, 100, 4, 16, 0, fake, fake, 200, None,
                          fake, fake, ws, None, None) == 1
    assert L.vg_select_kv(fake, 1, fake, 1, 32, 8, 5000, 100, 4, 16, 0, fake, fake, 200,
                          ctypes.byref(kv), fake, fake, ws, None, None) == 1
    # sparse draft: g > 8; a list longer than 65536 entries; no workspace is needed
    assert L.vg_sparse_draft_attention(ctypes.byref(kv), fake, fake, None, fake, 0, 200, fake,
                                       fake, 1, 80, 5, 0.1, fake, None, 0, None, None) == 2
    assert L.vg_sparse_draft_workspace_bytes(1, 32, 8, 128, 200, 5) == 0
    assert L.vg_sparse_draft_attention(ctypes.byref(kv), fake, fake, fake, fake, 0, 70000, fake,
                                       fake, 1, 32, 5, 0.1, fake, fake, 1 << 30, None, None) == 2
    assert L.vg_sparse_draft_attention(ctypes.byref(kv), fake, None, None, fake, 0, 200, fake,
                                       fake, 1, 32, 5, 0.1, fake, None, 0, None, None) == 1
