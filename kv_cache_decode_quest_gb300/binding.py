"""Thin ctypes binding of libsparse_engine.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
CUDA tensors, passes their device pointers and the current CUDA stream, and
raises ``SparseEngineError`` on a negative status.  All computation happens in
the library's kernels; there is no Python or CPU fallback: if the library is
not built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

from . import build as _build

c_i32p = ctypes.c_void_p  # device pointers are passed as raw addresses


class SparseEngineError(RuntimeError):
    pass


class PagedKVC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32)]


class ViewC(ctypes.Structure):
    _fields_ = [("chunk_row", ctypes.c_void_p), ("n_tokens", ctypes.c_void_p),
                ("num_units", ctypes.c_int32), ("max_chunks", ctypes.c_int32)]


class VarlenKVC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("score", ctypes.c_void_p), ("seg_off", ctypes.c_void_p),
                ("seg_len", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("seg_cap", ctypes.c_int32), ("total_rows", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class H2OStateC(ctypes.Structure):
    _fields_ = [("kv", VarlenKVC), ("budget", ctypes.c_int32), ("recent", ctypes.c_int32)]


class DecodeOptsC(ctypes.Structure):
    _fields_ = [("out_dtype", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("logits_out", ctypes.c_void_p), ("logits_stride", ctypes.c_int32),
                ("ev_kernel_begin", ctypes.c_void_p), ("ev_kernel_end", ctypes.c_void_p)]


class SelectOptsC(ctypes.Structure):
    _fields_ = [("group_agg", ctypes.c_int32)]


SE_AGG_SUM, SE_AGG_MAX = 0, 1


class QuestStepOptsC(ctypes.Structure):
    _fields_ = [("out_dtype", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("ev_kernel_begin", ctypes.c_void_p), ("ev_kernel_end", ctypes.c_void_p),
                ("wait_limit_ns", ctypes.c_int32)]


# C entry points: name -> (restype, argtypes)
_VP, _I, _SZ, _F, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_int64
SIGNATURES = {
    "se_status_str": (ctypes.c_char_p, [_I]),
    "se_version": (_I, []),
    "se_sync_status": (_I, [_VP, _VP]),
    "se_small_workspace": (_SZ, []),
    "se_quest_select_workspace": (_SZ, [_I, _I, _I]),
    "se_sparse_decode_workspace": (_SZ, [_I, _I, _I, _I]),
    "se_quest_step_workspace": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "se_snapkv_workspace": (_SZ, [_I, _I, _I, _I, _I]),
    "se_h2o_workspace": (_SZ, [_I, _I, _I, _I, _I]),
    "se_page_meta_build": (_I, [_VP, _I, _VP, _SZ, _VP]),
    "se_kv_append": (_I, [_VP, _VP, _VP, _I, _VP, _SZ, _VP]),
    "se_quest_select": (_I, [_VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "se_quest_select_append": (_I, [_VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _SZ,
                                    _VP]),
    "se_quest_step": (_I, [_VP, _VP, _VP, _VP, _I, _I, _VP, _F, _VP, _VP, _VP, _VP, _VP, _VP,
                           _VP, _SZ, _VP]),
    "se_view_from_segments": (_I, [_VP, _I, _VP, _VP, _SZ, _VP]),
    "se_quest_select_ex": (_I, [_VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                                _VP]),
    "se_sparse_decode": (_I, [_VP, _VP, _I64, _VP, _VP, _I, _I, _I, _I, _F, _VP, _VP, _VP,
                              _VP, _SZ, _VP]),
    "se_sparse_decode_noalloc": (_I, [_VP, _VP, _I64, _VP, _VP, _I, _I, _I, _I, _F, _I, _VP,
                                      _VP, _VP, _VP]),
    "se_varlen_append": (_I, [_VP, _VP, _VP, _I, _VP, _SZ, _VP]),
    "se_varlen_append_view": (_I, [_VP, _VP, _VP, _I, _VP, _VP, _SZ, _VP]),
    "se_snapkv_compact": (_I, [_VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _SZ, _VP]),
    "se_h2o_step": (_I, [_VP, _VP, _VP, _VP, _I, _I, _F, _I, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "se_chain_snapshot_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "se_chain_save": (_I, [_VP, _VP, _I, _I, _VP, _SZ, _VP, _SZ, _VP]),
    "se_chain_restore": (_I, [_VP, _SZ, _I, _I, _VP, _VP, _VP, _SZ, _VP]),
    "se_chain_index_create": (_VP, []),
    "se_chain_index_destroy": (None, [_VP]),
    "se_chain_index_put": (_I, [_VP, _VP, _I64, _I64]),
    "se_chain_index_match": (_I64, [_VP, _VP, _I64, _VP]),
    "se_chain_index_erase": (_I, [_VP, _I64]),
    "se_chain_index_size": (_I64, [_VP]),
    "se_span_prune": (_I, [_VP, _VP, _I, _I, _I, _I, _VP, _VP, _F, _VP, _VP, _SZ, _VP]),
    "se_view_sink_recent": (_I, [_VP, _I, _I, _I, _VP, _VP, _SZ, _VP]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise SparseEngineError(
            f"{path} is missing: build it first (kv_cache_decode_quest_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().se_status_str(rc).decode()
        raise SparseEngineError(f"{what} failed: {msg} ({rc})")


def _p(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ref(x):
    return ctypes.byref(x) if x is not None else None


# ---------------------------------------------------------------------------
# holders: keep the tensors alive next to the C struct that points at them
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class PagedKV:
    k: torch.Tensor            # bf16 [num_pages][Hkv][16][D]
    v: torch.Tensor
    meta: torch.Tensor         # bf16 [B][max_pages][Hkv][2][D], logical page order
    block_table: torch.Tensor  # int32 [B][max_pages]
    ctx_len: torch.Tensor      # int32 [B]

    @property
    def c(self) -> PagedKVC:
        P, H, S, D = self.k.shape
        return PagedKVC(_p(self.k), _p(self.v), _p(self.meta), _p(self.block_table),
                        _p(self.ctx_len), P, self.block_table.shape[1], H, D, S)


@dataclasses.dataclass
class View:
    chunk_row: torch.Tensor    # int32 [units][max_chunks]
    n_tokens: torch.Tensor     # int32 [units]

    @property
    def c(self) -> ViewC:
        return ViewC(_p(self.chunk_row), _p(self.n_tokens), self.chunk_row.shape[0],
                     self.chunk_row.shape[1])

    @staticmethod
    def empty(units: int, max_chunks: int, device="cuda") -> "View":
        return View(torch.zeros(units, max_chunks, dtype=torch.int32, device=device),
                    torch.zeros(units, dtype=torch.int32, device=device))


@dataclasses.dataclass
class VarlenKV:
    k: torch.Tensor            # bf16 [rows][D]
    v: torch.Tensor
    pos: torch.Tensor          # int32 [rows]
    score: torch.Tensor | None # fp32 [rows]
    seg_off: torch.Tensor      # int32 [units]
    seg_len: torch.Tensor      # int32 [units]
    seq_len: torch.Tensor      # int32 [B]
    seg_cap: int
    num_kv_heads: int

    @property
    def c(self) -> VarlenKVC:
        return VarlenKVC(_p(self.k), _p(self.v), _p(self.pos), _p(self.score), _p(self.seg_off),
                         _p(self.seg_len), _p(self.seq_len), self.seg_cap, self.k.shape[0],
                         self.num_kv_heads, self.k.shape[1])

    @staticmethod
    def empty(batch: int, num_kv_heads: int, seg_cap: int, head_dim: int, with_score=False,
              device="cuda") -> "VarlenKV":
        units = batch * num_kv_heads
        rows = units * seg_cap
        return VarlenKV(
            torch.zeros(rows, head_dim, dtype=torch.bfloat16, device=device),
            torch.zeros(rows, head_dim, dtype=torch.bfloat16, device=device),
            torch.full((rows,), -1, dtype=torch.int32, device=device),
            torch.zeros(rows, dtype=torch.float32, device=device) if with_score else None,
            torch.arange(units, dtype=torch.int32, device=device) * seg_cap,
            torch.zeros(units, dtype=torch.int32, device=device),
            torch.zeros(batch, dtype=torch.int32, device=device),
            seg_cap, num_kv_heads)


@dataclasses.dataclass
class H2OState:
    kv: VarlenKV               # with score
    budget: int
    recent: int

    @property
    def c(self) -> H2OStateC:
        return H2OStateC(self.kv.c, self.budget, self.recent)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace (status word cleared)."""
    return torch.zeros(max(256, int(nbytes)), dtype=torch.uint8, device=device)


def se_sync_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the SE_DEV_* bits of the workspace's
    status word (raises on a negative status)."""
    rc = load().se_sync_status(_p(ws), _stream(stream))
    if rc < 0:
        _check(rc, "se_sync_status")
    return rc


def status_word(ws: torch.Tensor) -> int:
    """The device status word of a workspace, read through se_sync_status."""
    return se_sync_status(ws)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def se_version() -> int:
    return load().se_version()


def se_small_workspace() -> int:
    return load().se_small_workspace()


def se_quest_select_workspace(batch, num_kv_heads, max_pages_per_seq) -> int:
    return load().se_quest_select_workspace(batch, num_kv_heads, max_pages_per_seq)


def se_sparse_decode_workspace(num_units, group_size, head_dim, max_splits=64) -> int:
    return load().se_sparse_decode_workspace(num_units, group_size, head_dim, max_splits)


def se_quest_step_workspace(batch, num_kv_heads, num_q_heads, head_dim, max_pages_per_seq,
                            max_splits=64) -> int:
    return load().se_quest_step_workspace(batch, num_kv_heads, num_q_heads, head_dim,
                                          max_pages_per_seq, max_splits)


def se_snapkv_workspace(batch, num_kv_heads, num_q_heads, window, max_ctx) -> int:
    return load().se_snapkv_workspace(batch, num_kv_heads, num_q_heads, window, max_ctx)


def se_h2o_workspace(batch, num_kv_heads, num_q_heads, head_dim, seg_cap) -> int:
    return load().se_h2o_workspace(batch, num_kv_heads, num_q_heads, head_dim, seg_cap)


def se_page_meta_build(kv: PagedKV, batch: int, ws, stream=None):
    c = kv.c
    _check(load().se_page_meta_build(ctypes.byref(c), batch, _p(ws), ws.numel(), _stream(stream)),
           "se_page_meta_build")


def se_kv_append(kv: PagedKV, k_new, v_new, batch: int, ws, stream=None):
    c = kv.c
    _check(load().se_kv_append(ctypes.byref(c), _p(k_new), _p(v_new), batch, _p(ws), ws.numel(),
                               _stream(stream)), "se_kv_append")


def se_quest_select(kv: PagedKV, q, batch: int, num_q_heads: int, budget_tokens, sel_pages,
                    n_sel, view: View, ws, stream=None):
    c, vc = kv.c, view.c
    _check(load().se_quest_select(ctypes.byref(c), _p(q), batch, num_q_heads, _p(budget_tokens),
                                  _p(sel_pages), _p(n_sel), ctypes.byref(vc), _p(ws), ws.numel(),
                                  _stream(stream)), "se_quest_select")


def se_quest_select_append(kv: PagedKV, k_new, v_new, q, batch: int, num_q_heads: int,
                           budget_tokens, sel_pages, n_sel, view: View, ws, stream=None):
    c, vc = kv.c, view.c
    _check(load().se_quest_select_append(ctypes.byref(c), _p(k_new), _p(v_new), _p(q), batch,
                                         num_q_heads, _p(budget_tokens), _p(sel_pages),
                                         _p(n_sel), ctypes.byref(vc), _p(ws), ws.numel(),
                                         _stream(stream)), "se_quest_select_append")


def se_quest_select_ex(kv: PagedKV, k_new, v_new, q, batch: int, num_q_heads: int,
                       budget_tokens, sel_pages, n_sel, view: View, ws, group_agg: int = 0,
                       stream=None):
    """Quest selection (with the append when k_new/v_new are given) with
    options: group_agg SE_AGG_SUM or SE_AGG_MAX."""
    c, vc = kv.c, view.c
    opts = SelectOptsC(group_agg)
    _check(load().se_quest_select_ex(ctypes.byref(c), _p(k_new), _p(v_new), _p(q), batch,
                                     num_q_heads, _p(budget_tokens), ctypes.byref(opts),
                                     _p(sel_pages), _p(n_sel), ctypes.byref(vc), _p(ws),
                                     ws.numel(), _stream(stream)), "se_quest_select_ex")


def se_quest_step(kv: PagedKV, k_new, v_new, q, batch: int, num_q_heads: int, budget_tokens,
                  scale: float, sel_pages, n_sel, view: View, out, lse, ws, out_dtype: int = 0,
                  max_splits: int = 64, wait_limit_ns: int = 0, ev_begin=None, ev_end=None,
                  stream=None):
    """One Quest decode step (append when k_new/v_new are given, select, decode)
    in one kernel."""
    c, vc = kv.c, view.c
    opts = QuestStepOptsC(out_dtype, max_splits,
                          ev_begin.cuda_event if ev_begin is not None else None,
                          ev_end.cuda_event if ev_end is not None else None,
                          wait_limit_ns)
    _check(load().se_quest_step(ctypes.byref(c), _p(k_new), _p(v_new), _p(q), batch, num_q_heads,
                                _p(budget_tokens), scale, ctypes.byref(opts), _p(sel_pages),
                                _p(n_sel), ctypes.byref(vc), _p(out), _p(lse), _p(ws), ws.numel(),
                                _stream(stream)), "se_quest_step")


def se_view_from_segments(kv: VarlenKV, batch: int, view: View, ws, stream=None):
    c, vc = kv.c, view.c
    _check(load().se_view_from_segments(ctypes.byref(c), batch, ctypes.byref(vc), _p(ws),
                                        ws.numel(), _stream(stream)), "se_view_from_segments")


def se_sparse_decode(k_rows, v_rows, view: View, q, batch: int, num_q_heads: int,
                     num_kv_heads: int, head_dim: int, scale: float, out, lse, ws,
                     out_dtype: int = 0, max_splits: int = 64, logits_out=None,
                     logits_stride: int = 0, ev_begin=None, ev_end=None, stream=None):
    vc = view.c
    opts = DecodeOptsC(out_dtype, max_splits, _p(logits_out), logits_stride,
                       ev_begin.cuda_event if ev_begin is not None else None,
                       ev_end.cuda_event if ev_end is not None else None)
    total_rows = k_rows.numel() // head_dim
    _check(load().se_sparse_decode(_p(k_rows), _p(v_rows), total_rows, ctypes.byref(vc), _p(q),
                                   batch, num_q_heads, num_kv_heads, head_dim, scale,
                                   ctypes.byref(opts), _p(out), _p(lse), _p(ws), ws.numel(),
                                   _stream(stream)), "se_sparse_decode")


def se_sparse_decode_noalloc(k_rows, v_rows, view: View, q, batch: int, num_q_heads: int,
                             num_kv_heads: int, head_dim: int, scale: float, out, lse,
                             out_dtype: int = 0, status_out=None, stream=None):
    """se_sparse_decode without a workspace (scratch inside the library)."""
    vc = view.c
    total_rows = k_rows.numel() // head_dim
    _check(load().se_sparse_decode_noalloc(_p(k_rows), _p(v_rows), total_rows, ctypes.byref(vc),
                                           _p(q), batch, num_q_heads, num_kv_heads, head_dim,
                                           scale, out_dtype, _p(out), _p(lse), _p(status_out),
                                           _stream(stream)), "se_sparse_decode_noalloc")


def se_varlen_append(kv: VarlenKV, k_new, v_new, batch: int, ws, stream=None):
    c = kv.c
    _check(load().se_varlen_append(ctypes.byref(c), _p(k_new), _p(v_new), batch, _p(ws),
                                   ws.numel(), _stream(stream)), "se_varlen_append")


def se_varlen_append_view(kv: VarlenKV, k_new, v_new, batch: int, view: View, ws, stream=None):
    c, vc = kv.c, view.c
    _check(load().se_varlen_append_view(ctypes.byref(c), _p(k_new), _p(v_new), batch,
                                        ctypes.byref(vc), _p(ws), ws.numel(), _stream(stream)),
           "se_varlen_append_view")


def se_snapkv_compact(prefill: PagedKV, q_win, batch: int, num_q_heads: int, window: int,
                      pool_kernel: int, keep: int, recent: int, scale: float, out: VarlenKV, ws,
                      stream=None):
    c, oc = prefill.c, out.c
    _check(load().se_snapkv_compact(ctypes.byref(c), _p(q_win), batch, num_q_heads, window,
                                    pool_kernel, keep, recent, scale, ctypes.byref(oc), _p(ws),
                                    ws.numel(), _stream(stream)), "se_snapkv_compact")


def se_h2o_step(st: H2OState, q, k_new, v_new, batch: int, num_q_heads: int, scale: float,
                out, lse, evicted_pos, ws, out_dtype: int = 0, stream=None):
    c = st.c
    _check(load().se_h2o_step(ctypes.byref(c), _p(q), _p(k_new), _p(v_new), batch, num_q_heads,
                              scale, out_dtype, _p(out), _p(lse), _p(evicted_pos), _p(ws),
                              ws.numel(), _stream(stream)), "se_h2o_step")


def se_span_prune(prefix: PagedKV, q_win, batch: int, num_q_heads: int, window: int,
                  pool_kernel: int, span, keep_tokens, scale: float, out: VarlenKV, ws,
                  stream=None):
    """Prune each sequence's span [span[b,0], span[b,1]) to its best
    keep_tokens[b] tokens by window score; everything else is kept."""
    c, oc = prefix.c, out.c
    _check(load().se_span_prune(ctypes.byref(c), _p(q_win), batch, num_q_heads, window,
                                pool_kernel, _p(span), _p(keep_tokens), scale, ctypes.byref(oc),
                                _p(ws), ws.numel(), _stream(stream)), "se_span_prune")


def se_view_sink_recent(kv: PagedKV, batch: int, sink_pages: int, recent_pages: int, view: View,
                        ws, stream=None):
    """The sink + recent pages view of a paged cache."""
    c, vc = kv.c, view.c
    _check(load().se_view_sink_recent(ctypes.byref(c), batch, sink_pages, recent_pages,
                                      ctypes.byref(vc), _p(ws), ws.numel(), _stream(stream)),
           "se_view_sink_recent")


def se_chain_snapshot_bytes(num_seqs: int, num_kv_heads: int, head_dim: int, rows: int,
                            with_score: bool) -> int:
    return load().se_chain_snapshot_bytes(num_seqs, num_kv_heads, head_dim, rows, int(with_score))


def se_chain_save(kv: VarlenKV, seqs, rows: int, snap, ws, stream=None):
    """Copy the retained segments of sequences `seqs` (int32 device) into `snap`."""
    c = kv.c
    _check(load().se_chain_save(ctypes.byref(c), _p(seqs), seqs.numel(), rows, _p(snap),
                                snap.numel(), _p(ws), ws.numel(), _stream(stream)),
           "se_chain_save")


def se_chain_restore(snap, rows: int, seqs, kv: VarlenKV, ws, stream=None):
    """Copy a snapshot's slots into the segments of sequences `seqs` of `kv`."""
    c = kv.c
    _check(load().se_chain_restore(_p(snap), snap.numel(), seqs.numel(), rows, _p(seqs),
                                   ctypes.byref(c), _p(ws), ws.numel(), _stream(stream)),
           "se_chain_restore")


class ChainIndex:
    """The host ChainCacheIndex: logical token prefix -> session id."""

    def __init__(self):
        self._h = load().se_chain_index_create()
        if not self._h:
            raise SparseEngineError("se_chain_index_create failed")

    def close(self):
        if self._h:
            load().se_chain_index_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _tok(tokens):
        import numpy as np
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return t, t.ctypes.data_as(ctypes.c_void_p), t.size

    def put(self, tokens, sid: int):
        t, ptr, n = self._tok(tokens)
        _check(load().se_chain_index_put(self._h, ptr, n, sid), "se_chain_index_put")

    def match(self, tokens):
        """(id, matched tokens) of the longest stored prefix, (-1, 0) if none."""
        t, ptr, n = self._tok(tokens)
        m = ctypes.c_int64(0)
        sid = load().se_chain_index_match(self._h, ptr, n, ctypes.byref(m))
        if sid < -1:
            _check(int(sid), "se_chain_index_match")
        return int(sid), int(m.value)

    def erase(self, sid: int):
        _check(load().se_chain_index_erase(self._h, sid), "se_chain_index_erase")

    def __len__(self):
        return int(load().se_chain_index_size(self._h))
