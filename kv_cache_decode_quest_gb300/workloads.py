"""Device-side set-up and decode-step drivers for the synthetic workloads.

A driver owns the caller-side buffers of one workload (caches, views,
workspaces, per-step inputs) and issues the library's entry points for one
decode step.  Set-up (placing the prefill cache into pages, building page
summaries) happens once, outside any timed region.  All arithmetic of the
path runs in the library's kernels; this module only moves bytes.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import binding as se
from . import synth

PAGE = synth.PAGE_SIZE


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload bf16 bit patterns (uint16) as a bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device, non_blocking=False).view(torch.bfloat16)


def paged_layout(seqs_k, seqs_v, lengths, block_table, num_pages, num_kv_heads, head_dim):
    """Scatter per-sequence logical K/V ([Hkv][T][D] bf16 bits, first `lengths[b]`
    tokens) into physical pages [num_pages][Hkv][16][D] by the block table."""
    K = np.zeros((num_pages, num_kv_heads, PAGE, head_dim), dtype=np.uint16)
    V = np.zeros_like(K)
    for b, L in enumerate(lengths):
        n = -(-int(L) // PAGE)
        if n == 0:
            continue
        for src, dst in ((seqs_k[b], K), (seqs_v[b], V)):
            blk = np.zeros((num_kv_heads, n * PAGE, head_dim), dtype=np.uint16)
            blk[:, :L] = src[:, :L]
            dst[block_table[b, :n]] = blk.reshape(num_kv_heads, n, PAGE, head_dim).transpose(1, 0, 2, 3)
    return K, V


class QuestRun:
    """Paged KV + Quest selection + split-K decode, one appended token per step.

    mode: "fused"    -- se_quest_select_append, then se_sparse_decode (the
                        default here; the faster path for a single query);
          "step"     -- se_quest_step: append, select and decode in one kernel
                        (the faster path on the multi-sequence workloads);
          "separate" -- se_kv_append, se_quest_select, se_sparse_decode.
    step_tuning: se_quest_step_opts fields (mode "step"): wait_limit_ns."""

    MODES = ("step", "fused", "separate")

    def __init__(self, w: synth.QuestWorkload, inputs: dict, out_dtype: int = 0,
                 max_splits: int | None = None, device="cuda", mode: str = "fused",
                 step_tuning: dict | None = None):
        if mode not in self.MODES:
            raise ValueError(f"mode {mode!r} not in {self.MODES}")
        self.w = w
        self.mode = mode
        self.step_tuning = dict(step_tuning or {})
        B, Hq, Hkv, D, S = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.steps
        self.B, self.Hq, self.Hkv, self.D, self.S = B, Hq, Hkv, D, S
        self.G = Hq // Hkv
        self.scale = 1.0 / math.sqrt(D)
        self.out_dtype = out_dtype
        self.max_splits = max_splits or w.max_splits
        ctx = np.asarray(w.ctx, dtype=np.int64)
        pages = -(-(ctx + S) // PAGE)
        bt, num_pages = synth.block_table(w.seed, w.name + "/block_table", pages)
        self.block_table_np = bt
        K, V = paged_layout(inputs["k"], inputs["v"], ctx, bt, num_pages, Hkv, D)
        self.kv = se.PagedKV(
            k=to_dev_bf16(K, device), v=to_dev_bf16(V, device),
            meta=torch.zeros(B, bt.shape[1], Hkv, 2, D, dtype=torch.bfloat16, device=device),
            block_table=torch.from_numpy(bt).to(device),
            ctx_len=torch.from_numpy(ctx.astype(np.int32)).to(device))
        del K, V
        # per-step inputs
        # per-step inputs, one contiguous row per step: q [B][Hq][D], then the
        # appended k and v [B][Hkv][D] (a caller feeding the step from host
        # memory copies one row per step)
        kn = np.stack([np.stack([inputs["k"][b][:, ctx[b] + s] for b in range(B)]) for s in range(S)])
        vn = np.stack([np.stack([inputs["v"][b][:, ctx[b] + s] for b in range(B)]) for s in range(S)])
        nq, nk = B * Hq * D, B * Hkv * D
        rows = np.concatenate([np.asarray(inputs["q"]).reshape(S, nq), kn.reshape(S, nk),
                               vn.reshape(S, nk)], axis=1)
        self.step_inputs = to_dev_bf16(rows, device)                             # [S][nq + 2 nk]
        self.q = self.step_inputs[:, :nq].view(S, B, Hq, D)
        self.k_new = self.step_inputs[:, nq:nq + nk].view(S, B, Hkv, D)
        self.v_new = self.step_inputs[:, nq + nk:].view(S, B, Hkv, D)
        self.budget = torch.tensor([min(b, 2 ** 31 - 1) for b in w.budget], dtype=torch.int32,
                                   device=device)
        units = B * Hkv
        maxp = bt.shape[1]
        self.sel = torch.zeros(units, maxp, dtype=torch.int32, device=device)
        self.n_sel = torch.zeros(units, dtype=torch.int32, device=device)
        self.view = se.View.empty(units, maxp, device)
        self.ws_small = se.workspace(se.se_small_workspace(), device)
        self.ws_sel = se.workspace(se.se_quest_select_workspace(B, Hkv, maxp), device)
        self.ws_dec = se.workspace(se.se_sparse_decode_workspace(units, self.G, D, self.max_splits),
                                   device)
        self.ws_step = se.workspace(se.se_quest_step_workspace(B, Hkv, Hq, D, maxp, self.max_splits),
                                    device)
        odt = torch.float32 if out_dtype == 1 else torch.bfloat16
        self.out = torch.zeros(B, Hq, D, dtype=odt, device=device)
        self.lse = torch.zeros(B, Hq, dtype=torch.float32, device=device)
        se.se_page_meta_build(self.kv, B, self.ws_small)

    def append(self, s: int):
        se.se_kv_append(self.kv, self.k_new[s], self.v_new[s], self.B, self.ws_small)

    def select(self, s: int):
        se.se_quest_select(self.kv, self.q[s], self.B, self.Hq, self.budget, self.sel, self.n_sel,
                           self.view, self.ws_sel)

    group_agg = se.SE_AGG_SUM

    def append_select(self, s: int):
        """The step's append fused into the selection (one kernel fewer)."""
        if self.group_agg != se.SE_AGG_SUM:
            se.se_quest_select_ex(self.kv, self.k_new[s], self.v_new[s], self.q[s], self.B,
                                  self.Hq, self.budget, self.sel, self.n_sel, self.view,
                                  self.ws_sel, group_agg=self.group_agg)
            return
        se.se_quest_select_append(self.kv, self.k_new[s], self.v_new[s], self.q[s], self.B,
                                  self.Hq, self.budget, self.sel, self.n_sel, self.view,
                                  self.ws_sel)

    def decode(self, s: int, out=None, lse=None, ev_begin=None, ev_end=None):
        se.se_sparse_decode(self.kv.k, self.kv.v, self.view, self.q[s], self.B, self.Hq, self.Hkv,
                            self.D, self.scale, self.out if out is None else out,
                            self.lse if lse is None else lse, self.ws_dec,
                            out_dtype=self.out_dtype, max_splits=self.max_splits,
                            ev_begin=ev_begin, ev_end=ev_end)

    def one_kernel_step(self, s: int, out=None, lse=None, ev_begin=None, ev_end=None):
        """Append, select and decode in one kernel (se_quest_step)."""
        se.se_quest_step(self.kv, self.k_new[s], self.v_new[s], self.q[s], self.B, self.Hq,
                         self.budget, self.scale, self.sel, self.n_sel, self.view,
                         self.out if out is None else out, self.lse if lse is None else lse,
                         self.ws_step, out_dtype=self.out_dtype, max_splits=self.max_splits,
                         ev_begin=ev_begin, ev_end=ev_end, **self.step_tuning)

    def step(self, s: int, out=None, lse=None, ev_begin=None, ev_end=None):
        """One decode step: append the step's token, select pages, attend."""
        if self.mode == "step":
            self.one_kernel_step(s, out, lse, ev_begin, ev_end)
            return
        if self.mode == "fused":
            self.append_select(s)
        else:
            self.append(s)
            self.select(s)
        self.decode(s, out, lse, ev_begin, ev_end)

    def status(self) -> int:
        return se.status_word(self.ws_small) | se.status_word(self.ws_sel) | \
            se.status_word(self.ws_dec) | se.status_word(self.ws_step)

    def algorithmic_bytes(self, ctx_now: np.ndarray) -> dict:
        """Bytes one step must move at least, given each sequence's length after
        the append: page summaries of every candidate page of a sequence that is
        not wholly selected (2*D*2 bytes per page and KV head), K and V of every
        selected token (2*D*2 bytes per token and KV head), q, the appended k/v,
        and the output."""
        D, Hkv, Hq = self.D, self.Hkv, self.Hq
        meta = sel = 0
        for b, L in enumerate(ctx_now):
            n = -(-int(L) // PAGE)
            k = max(1, min(self.w.budget[b], 2 ** 31 - 1) // PAGE)
            if n > k:                                  # every page selected: nothing scored
                meta += (n - 1) * Hkv * 2 * D * 2
            if n <= k:
                toks = int(L)
            else:
                toks = (k - 1) * PAGE + (int(L) - PAGE * (n - 1))
            sel += toks * Hkv * 2 * D * 2
        outb = 4 if self.out_dtype == 1 else 2
        small = self.B * (Hq * D * 2 + 2 * Hkv * D * 2 + Hq * D * outb)
        return {"meta": meta, "kv": sel, "small": small, "total": meta + sel + small}


class OmniRun:
    """Cross-layer selection reuse over `layers` attention layers of one model:
    every layer keeps its own paged K/V (one block table for all), the filter
    layers keep page summaries and select with se_quest_select_append, the
    other layers append with se_kv_append (no summaries) and every layer
    decodes with se_sparse_decode through the view of the latest filter layer
    at or before it."""

    def __init__(self, w: synth.OmniKVWorkload, inputs: list, device="cuda", out_dtype: int = 0):
        self.w = w
        B, Hq, Hkv, D, S, L = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.steps, w.layers
        self.B, self.Hq, self.Hkv, self.D, self.S, self.L = B, Hq, Hkv, D, S, L
        self.G = Hq // Hkv
        self.scale = 1.0 / math.sqrt(D)
        self.out_dtype = out_dtype
        self.filters = tuple(sorted(w.filters))
        if not self.filters or self.filters[0] != 0:
            raise ValueError("layer 0 must be a filter layer")
        ctx = np.asarray(w.ctx, dtype=np.int64)
        pages = -(-(ctx + S) // PAGE)
        bt, num_pages = synth.block_table(w.seed, w.name + "/block_table", pages)
        maxp = bt.shape[1]
        units = B * Hkv
        block_table = torch.from_numpy(bt).to(device)
        self.kv, self.q, self.k_new, self.v_new = [], [], [], []
        self.sel, self.n_sel, self.view, self.ws_sel = {}, {}, {}, {}
        for layer in range(L):
            inp = inputs[layer]
            K, V = paged_layout(inp["k"], inp["v"], ctx, bt, num_pages, Hkv, D)
            meta = (torch.zeros(B, maxp, Hkv, 2, D, dtype=torch.bfloat16, device=device)
                    if layer in self.filters else None)
            self.kv.append(se.PagedKV(k=to_dev_bf16(K, device), v=to_dev_bf16(V, device), meta=meta,
                                      block_table=block_table,
                                      ctx_len=torch.from_numpy(ctx.astype(np.int32)).to(device)))
            del K, V
            self.q.append(to_dev_bf16(np.asarray(inp["q"]), device))
            kn = np.stack([np.stack([inp["k"][b][:, ctx[b] + s] for b in range(B)]) for s in range(S)])
            vn = np.stack([np.stack([inp["v"][b][:, ctx[b] + s] for b in range(B)]) for s in range(S)])
            self.k_new.append(to_dev_bf16(kn, device))
            self.v_new.append(to_dev_bf16(vn, device))
            if layer in self.filters:
                self.sel[layer] = torch.zeros(units, maxp, dtype=torch.int32, device=device)
                self.n_sel[layer] = torch.zeros(units, dtype=torch.int32, device=device)
                self.view[layer] = se.View.empty(units, maxp, device)
                self.ws_sel[layer] = se.workspace(se.se_quest_select_workspace(B, Hkv, maxp), device)
        self.budget = torch.tensor([min(b, 2 ** 31 - 1) for b in w.budget], dtype=torch.int32,
                                   device=device)
        self.ws_small = se.workspace(se.se_small_workspace(), device)
        self.ws_dec = se.workspace(se.se_sparse_decode_workspace(units, self.G, D, w.max_splits),
                                   device)
        odt = torch.float32 if out_dtype == 1 else torch.bfloat16
        self.out = [torch.zeros(B, Hq, D, dtype=odt, device=device) for _ in range(L)]
        self.lse = [torch.zeros(B, Hq, dtype=torch.float32, device=device) for _ in range(L)]
        for layer in self.filters:
            se.se_page_meta_build(self.kv[layer], B, self.ws_small)

    def source(self, layer: int) -> int:
        return max(f for f in self.filters if f <= layer)

    def step(self, s: int, ev_begin=None, ev_end=None):
        """One decode step through every layer, in layer order."""
        for layer in range(self.L):
            kv = self.kv[layer]
            if layer in self.filters:
                se.se_quest_select_append(kv, self.k_new[layer][s], self.v_new[layer][s],
                                          self.q[layer][s], self.B, self.Hq, self.budget,
                                          self.sel[layer], self.n_sel[layer], self.view[layer],
                                          self.ws_sel[layer])
            else:
                se.se_kv_append(kv, self.k_new[layer][s], self.v_new[layer][s], self.B,
                                self.ws_small)
            timed = ev_begin is not None and layer == self.L - 1
            se.se_sparse_decode(kv.k, kv.v, self.view[self.source(layer)], self.q[layer][s], self.B,
                                self.Hq, self.Hkv, self.D, self.scale, self.out[layer],
                                self.lse[layer], self.ws_dec, out_dtype=self.out_dtype,
                                max_splits=self.w.max_splits, ev_begin=ev_begin if timed else None,
                                ev_end=ev_end if timed else None)

    def status(self) -> int:
        st = se.status_word(self.ws_small) | se.status_word(self.ws_dec)
        for ws in self.ws_sel.values():
            st |= se.status_word(ws)
        return st

    def algorithmic_bytes(self, ctx_now: np.ndarray) -> dict:
        """Bytes one step must move at least: the filter layers' page summaries
        of every candidate page, every layer's K and V of the selected tokens,
        and each layer's q, appended k/v and output."""
        D, Hkv, Hq = self.D, self.Hkv, self.Hq
        meta = kv = 0
        for b, L in enumerate(ctx_now):
            n = -(-int(L) // PAGE)
            k = max(1, min(self.w.budget[b], 2 ** 31 - 1) // PAGE)
            meta += max(0, n - 1) * Hkv * 2 * D * 2 if n > k else 0
            toks = int(L) if n <= k else (k - 1) * PAGE + (int(L) - PAGE * (n - 1))
            kv += toks * Hkv * 2 * D * 2
        outb = 4 if self.out_dtype == 1 else 2
        small = self.B * (Hq * D * 2 + 2 * Hkv * D * 2 + Hq * D * outb)
        total = len(self.filters) * meta + self.L * (kv + small)
        return {"meta": len(self.filters) * meta, "kv": self.L * kv, "total": total}


class SnapKVRun:
    """SnapKV compaction of `groups` prefill batches into one per-(sequence, KV
    head) varlen cache, then decode over it with one appended token per step."""

    def __init__(self, w: synth.SnapKVWorkload, groups=None, device="cuda", max_splits=None,
                 keep_inputs=False, with_score=False):
        self.w = w
        self.groups = w.groups if groups is None else groups
        B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
        self.B, self.Hq, self.Hkv, self.D = B, Hq, Hkv, D
        self.Bt = B * self.groups
        self.G = Hq // Hkv
        self.scale = 1.0 / math.sqrt(D)
        self.max_splits = max_splits or w.max_splits
        self.device = device
        L = w.ctx
        kept = min(w.keep, max(0, L - w.window)) + min(w.window, L)
        self.seg_cap = kept + w.steps
        self.cache = se.VarlenKV.empty(self.Bt, Hkv, self.seg_cap, D, with_score=with_score,
                                       device=device)
        self.inputs = [] if keep_inputs else None
        self.prefill = None
        pages = -(-L // PAGE)
        self.ws_snap = se.workspace(se.se_snapkv_workspace(B, Hkv, Hq, w.window, L), device)
        for g in range(self.groups):
            inp = synth.snapkv_inputs(w, g)
            if keep_inputs:
                self.inputs.append(inp)
            bt, num_pages = synth.block_table(w.seed, f"{w.name}/g{g}/block_table",
                                              np.full(B, pages))
            K, V = paged_layout(list(inp["k"]), list(inp["v"]), np.full(B, L), bt, num_pages,
                                Hkv, D)
            pre = se.PagedKV(k=to_dev_bf16(K, device), v=to_dev_bf16(V, device),
                             meta=torch.zeros(1, dtype=torch.bfloat16, device=device),
                             block_table=torch.from_numpy(bt).to(device),
                             ctx_len=torch.full((B,), L, dtype=torch.int32, device=device))
            del K, V
            q_win = to_dev_bf16(inp["q_win"], device)
            self.compact_group(g, pre, q_win)
            if g == self.groups - 1:
                self.prefill, self.q_win = pre, q_win      # last group kept for timing
            torch.cuda.synchronize()
        dec = synth.snapkv_decode_inputs(w)
        self.q = to_dev_bf16(dec["q"], device)
        self.k_new = to_dev_bf16(dec["k_new"], device)
        self.v_new = to_dev_bf16(dec["v_new"], device)
        self.dec_inputs = dec if keep_inputs else None
        units = self.Bt * Hkv
        self.view = se.View.empty(units, -(-self.seg_cap // PAGE), device)
        self.ws_small = se.workspace(se.se_small_workspace(), device)
        self.ws_dec = se.workspace(se.se_sparse_decode_workspace(units, self.G, D, self.max_splits),
                                   device)
        self.out = torch.zeros(self.Bt, Hq, D, dtype=torch.bfloat16, device=device)
        self.lse = torch.zeros(self.Bt, Hq, dtype=torch.float32, device=device)

    def group_slice(self, g) -> se.VarlenKV:
        """The varlen cache restricted to compaction group g's units."""
        c, B, H = self.cache, self.B, self.Hkv
        return se.VarlenKV(c.k, c.v, c.pos, c.score, c.seg_off[g * B * H:(g + 1) * B * H],
                           c.seg_len[g * B * H:(g + 1) * B * H], c.seq_len[g * B:(g + 1) * B],
                           c.seg_cap, H)

    def compact_group(self, g, prefill, q_win):
        w = self.w
        se.se_snapkv_compact(prefill, q_win, self.B, self.Hq, w.window, w.pool_kernel, w.keep,
                             w.window, self.scale, self.group_slice(g), self.ws_snap)

    def step(self, s, ev_begin=None, ev_end=None, fused=True):
        if fused:
            se.se_varlen_append_view(self.cache, self.k_new[s], self.v_new[s], self.Bt, self.view,
                                     self.ws_small)
        else:
            se.se_varlen_append(self.cache, self.k_new[s], self.v_new[s], self.Bt, self.ws_small)
            se.se_view_from_segments(self.cache, self.Bt, self.view, self.ws_small)
        se.se_sparse_decode(self.cache.k, self.cache.v, self.view, self.q[s], self.Bt, self.Hq,
                            self.Hkv, self.D, self.scale, self.out, self.lse, self.ws_dec,
                            max_splits=self.max_splits, ev_begin=ev_begin, ev_end=ev_end)

    def status(self) -> int:
        return se.status_word(self.ws_small) | se.status_word(self.ws_snap) | \
            se.status_word(self.ws_dec)


class H2ORun:
    """H2O decode: the prefill's window column scores (pool 1) seed the scores
    and the initial retained set (recent + best budget-recent), then one
    se_h2o_step per decode step."""

    def __init__(self, w: synth.H2OWorkload, device="cuda", keep_inputs=False, out_dtype=0):
        self.w = w
        B, Hq, Hkv, D, L = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.ctx
        self.B, self.Hq, self.Hkv, self.D = B, Hq, Hkv, D
        self.G = Hq // Hkv
        self.scale = 1.0 / math.sqrt(D)
        self.out_dtype = out_dtype
        inp = synth.h2o_inputs(w)
        self.inputs = inp if keep_inputs else None
        pages = -(-L // PAGE)
        bt, num_pages = synth.block_table(w.seed, w.name + "/block_table", np.full(B, pages))
        K, V = paged_layout(list(inp["k"]), list(inp["v"]), np.full(B, L), bt, num_pages, Hkv, D)
        pre = se.PagedKV(k=to_dev_bf16(K, device), v=to_dev_bf16(V, device),
                         meta=torch.zeros(1, dtype=torch.bfloat16, device=device),
                         block_table=torch.from_numpy(bt).to(device),
                         ctx_len=torch.full((B,), L, dtype=torch.int32, device=device))
        del K, V
        self.cap = w.budget + 1
        cache = se.VarlenKV.empty(B, Hkv, self.cap, D, with_score=True, device=device)
        ws = se.workspace(se.se_snapkv_workspace(B, Hkv, Hq, w.window, L), device)
        se.se_snapkv_compact(pre, to_dev_bf16(inp["q_win"], device), B, Hq, w.window, 1,
                             max(0, w.budget - w.recent), w.recent, self.scale, cache, ws)
        torch.cuda.synchronize()
        self.init_status = se.status_word(ws)
        del pre, ws
        self.state = se.H2OState(cache, w.budget, w.recent)
        self.q = to_dev_bf16(inp["q"], device)
        self.k_new = to_dev_bf16(inp["k_new"], device)
        self.v_new = to_dev_bf16(inp["v_new"], device)
        units = B * Hkv
        self.ws = se.workspace(se.se_h2o_workspace(B, Hkv, Hq, D, self.cap), device)
        odt = torch.float32 if out_dtype == 1 else torch.bfloat16
        self.out = torch.zeros(B, Hq, D, dtype=odt, device=device)
        self.lse = torch.zeros(B, Hq, dtype=torch.float32, device=device)
        self.evicted = torch.zeros(units, dtype=torch.int32, device=device)

    def step(self, s, ev_begin=None, ev_end=None):
        se.se_h2o_step(self.state, self.q[s], self.k_new[s], self.v_new[s], self.B, self.Hq,
                       self.scale, self.out, self.lse, self.evicted, self.ws,
                       out_dtype=self.out_dtype)

    def status(self) -> int:
        return self.init_status | se.status_word(self.ws)
