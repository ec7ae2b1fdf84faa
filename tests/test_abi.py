"""The C-ABI library builds, loads, exports every entry point that
include/sparse_engine.h declares, and rejects bad arguments on the host
(these calls return before any CUDA call, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

from kv_cache_decode_quest_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "sparse_engine.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(se_\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.endswith("_t")))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_four_hot_path_calls():
    names = declared_functions()
    for n in ("se_quest_select", "se_sparse_decode", "se_snapkv_compact", "se_h2o_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_status_strings_and_version(lib):
    assert lib.se_version() == 1
    for rc in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(lib.se_status_str(rc), bytes)


def test_sync_status_validates_before_touching_the_device(lib):
    lib.se_sync_status.restype = ctypes.c_int
    assert lib.se_sync_status(None, None) == -1             # SE_ERR_INVALID_ARG
    assert lib.se_sync_status(ctypes.c_void_p((1 << 20) + 4), None) == -3   # not 256-aligned
    assert lib.se_sync_status(ctypes.c_void_p((1 << 20) + 128), None) == -3


def test_workspace_sizes(lib):
    assert lib.se_small_workspace() == 256
    assert lib.se_quest_select_workspace(16, 4, 2052) >= 16 * 4 * 2052 * 4
    assert lib.se_quest_select_workspace(16, 4, 2052) % 256 == 0
    d = lib.se_sparse_decode_workspace(64, 8, 128, 64)
    assert d >= 64 * 64 * 8 * 128 * 4 and d % 256 == 0


def _paged(head_dim=128, page_size=16, nulls=False):
    fake = None if nulls else 1 << 20       # never dereferenced: validation fails first
    return binding.PagedKVC(fake, fake, fake, fake, fake, 10, 4, 4, head_dim, page_size)


def test_host_validation_rejects_bad_arguments(lib):
    ws = ctypes.c_void_p(1 << 20)
    # null cache pointers
    assert lib.se_page_meta_build(ctypes.byref(_paged(nulls=True)), 1, ws, 256, None) == -1
    # unsupported head_dim / page size
    assert lib.se_page_meta_build(ctypes.byref(_paged(head_dim=96)), 1, ws, 256, None) == -2
    assert lib.se_page_meta_build(ctypes.byref(_paged(page_size=32)), 1, ws, 256, None) == -2
    # workspace too small / misaligned
    assert lib.se_page_meta_build(ctypes.byref(_paged()), 1, ws, 16, None) == -3
    assert lib.se_page_meta_build(ctypes.byref(_paged()), 1, ctypes.c_void_p((1 << 20) + 8),
                                  256, None) == -3
    # decode: unsupported group size (Hq/Hkv = 3) and head_dim
    view = binding.ViewC(1 << 20, 1 << 20, 4, 8)
    args = [ctypes.c_void_p(1 << 20)] * 2
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 1, 12,
                                4, 128, 0.1, None, ctypes.c_void_p(1 << 20), None, ws,
                                1 << 30, None) == -2
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 1, 32,
                                4, 80, 0.1, None, ctypes.c_void_p(1 << 20), None, ws,
                                1 << 30, None) == -2
    # decode: view unit count mismatch
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 2, 32,
                                4, 128, 0.1, None, ctypes.c_void_p(1 << 20), None, ws,
                                1 << 30, None) == -1
    # decode: max_splits out of range
    opts = binding.DecodeOptsC(0, 65, None, 0, None, None)
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 1, 32,
                                4, 128, 0.1, ctypes.byref(opts), ctypes.c_void_p(1 << 20), None,
                                ws, 1 << 30, None) == -1
    # decode: workspace too small for the split count
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 1, 32,
                                4, 128, 0.1, None, ctypes.c_void_p(1 << 20), None, ws,
                                1024, None) == -3
    # quest select: view too small for the block table width
    small_view = binding.ViewC(1 << 20, 1 << 20, 4, 2)
    assert lib.se_quest_select(ctypes.byref(_paged()), ctypes.c_void_p(1 << 20), 1, 32,
                               ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 20),
                               ctypes.c_void_p(1 << 20), ctypes.byref(small_view), ws,
                               1 << 30, None) == -5


def test_zero_batch_is_a_no_op(lib):
    view = binding.ViewC(None, None, 0, 0)
    assert lib.se_sparse_decode(None, None, 0, ctypes.byref(view), None, 0, 32, 4, 128, 0.1,
                                None, None, None, None, 0, None) == 0


def test_quest_step_workspace_and_host_validation(lib):
    """se_quest_step: workspace size, and every argument error caught on the
    host before a launch (fake, never dereferenced pointers)."""
    w = lib.se_quest_step_workspace(16, 4, 32, 128, 2052, 64)
    assert w % 256 == 0
    assert w >= 16 * 4 * 2052 * 4 + 16 * 4 * 64 * 8 * 128 * 4     # keys + decode partials
    assert lib.se_quest_step_workspace(16, 4, 30, 128, 2052, 64) == 0   # Hq not a multiple of Hkv
    P = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 20)
    kv = _paged()                                   # 4 KV heads, 4 pages per sequence
    view = binding.ViewC(1 << 20, 1 << 20, 4, 8)

    def call(k_new=P, v_new=P, batch=1, hq=32, view_=view, opts=None, ws_bytes=1 << 30, kv_=kv):
        return lib.se_quest_step(ctypes.byref(kv_), k_new, v_new, P, batch, hq, P, 0.1,
                                 None if opts is None else ctypes.byref(opts), P, P,
                                 ctypes.byref(view_), P, None, ws, ws_bytes, None)

    assert call(v_new=None) == -1                   # k_new without v_new
    assert call(hq=12) == -2                        # group size 3
    assert call(kv_=_paged(head_dim=96)) == -2
    assert call(batch=2) == -1                      # view unit count mismatch
    assert call(view_=binding.ViewC(1 << 20, 1 << 20, 4, 2)) == -5   # view narrower than the table
    big = binding.ViewC(1 << 20, 1 << 20, 1025 * 4, 8)
    assert call(batch=1025, view_=big) == -2        # batch limit
    O = binding.QuestStepOptsC
    assert call(opts=O(0, 65, None, None, 0)) == -1                  # max_splits
    assert call(opts=O(2, 0, None, None, 0)) == -1                   # out_dtype
    assert call(opts=O(0, 0, None, None, -5)) == -1                  # wait_limit_ns
    many = binding.ViewC(1 << 20, 1 << 20, 1024 * 8, 8)
    kv8 = binding.PagedKVC(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 10, 4, 8, 128, 16)
    assert call(batch=1024, hq=64, view_=many, kv_=kv8) == -2        # more than 4096 units
    assert call(ws_bytes=1024) == -3                # workspace too small
    # no append (k_new and v_new both NULL) is accepted up to the workspace check
    assert call(k_new=None, v_new=None, ws_bytes=1024) == -3
    # zero batch: nothing to do
    assert lib.se_quest_step(ctypes.byref(kv), None, None, None, 0, 32, None, 0.1, None, None,
                             None, None, None, None, ws, 1 << 30, None) == 0


def test_decode_view_chunk_limit(lib):
    """The split-K plan's 32-bit products bound view->max_chunks at 2^20."""
    args = [ctypes.c_void_p(1 << 20)] * 2
    view = binding.ViewC(1 << 20, 1 << 20, 4, (1 << 20) + 1)
    assert lib.se_sparse_decode(*args, 100, ctypes.byref(view), ctypes.c_void_p(1 << 20), 1, 32,
                                4, 128, 0.1, None, ctypes.c_void_p(1 << 20), None,
                                ctypes.c_void_p(1 << 20), 1 << 30, None) == -2
