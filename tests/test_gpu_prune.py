"""GPU parity: span-restricted prefix pruning (se_span_prune) and the sink +
recent page view (se_view_sink_recent + se_sparse_decode) through the C ABI
against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.quest import selected_tokens
from kv_cache_decode_quest_gb300 import binding as se
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import PAGE, QuestRun, paged_layout, to_dev_bf16
from tests.parity import TOL_BF16, TOL_F32, check_topk, max_abs
from tests.test_gpu_snapkv import score_close

pytestmark = pytest.mark.gpu


def run_prune(lengths, spans, keeps, Hq=16, Hkv=2, D=128, W=16, pool=7, seed=0):
    g = np.random.default_rng(seed)
    B = len(lengths)
    k = [synth.f32_to_bf16_bits(g.standard_normal((Hkv, L, D)).astype(np.float32)) for L in lengths]
    v = [synth.f32_to_bf16_bits(g.standard_normal((Hkv, L, D)).astype(np.float32)) for L in lengths]
    q_win = synth.f32_to_bf16_bits(g.standard_normal((B, W, Hq, D)).astype(np.float32))
    pages = np.array([-(-L // PAGE) for L in lengths])
    bt, num_pages = synth.block_table(seed, "prune_test_bt", pages)
    K, V = paged_layout(k, v, lengths, bt, num_pages, Hkv, D)
    pre = se.PagedKV(to_dev_bf16(K), to_dev_bf16(V), None, torch.from_numpy(bt).cuda(),
                     torch.tensor(lengths, dtype=torch.int32, device="cuda"))
    out = se.VarlenKV.empty(B, Hkv, max(lengths), D, with_score=True)
    ws = se.workspace(se.se_snapkv_workspace(B, Hkv, Hq, W, max(lengths)))
    span = torch.tensor(np.asarray(spans, dtype=np.int32).reshape(B, 2), device="cuda")
    keep = torch.tensor(keeps, dtype=torch.int32, device="cuda")
    se.se_span_prune(pre, to_dev_bf16(q_win), B, Hq, W, pool, span, keep, 1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    assert se.status_word(ws) == 0
    G = Hq // Hkv
    pos_all = out.pos.cpu().numpy()
    kd = out.k.view(torch.int16).cpu().numpy().view(np.uint16)
    sc = out.score.cpu().numpy()
    seg_len, seg_off = out.seg_len.cpu().numpy(), out.seg_off.cpu().numpy()
    assert out.seq_len.cpu().numpy().tolist() == list(lengths)
    for u in range(B * Hkv):
        b, h = divmod(u, Hkv)
        L = lengths[b]
        A = oracle.window_scores(oracle.widen(q_win[b][:, h * G:(h + 1) * G]),
                                 oracle.widen(k[b][h]), 1 / math.sqrt(D))
        s0, s1 = spans[b]
        ref = oracle.span_keep_positions(A, L, s0, s1, keeps[b], pool)
        n, off = int(seg_len[u]), int(seg_off[u])
        assert n == len(ref), (u, n, len(ref))
        got = pos_all[off:off + n]
        assert np.all(np.diff(got) > 0)
        lo, hi = max(0, min(s0, L)), max(max(0, min(s0, L)), min(s1, L))
        kk = min(keeps[b], hi - lo)
        assert np.array_equal(got[:lo], np.arange(lo))
        assert np.array_equal(got[lo + kk:], np.arange(hi, L))
        if 0 < kk < hi - lo:
            pooled = oracle.max_pool(A[lo:hi], pool)
            boundary = pooled[oracle.rank_order(pooled)[kk - 1]]
            check_topk(got[lo:lo + kk] - lo, ref[lo:lo + kk] - lo, pooled, boundary,
                       what=f"unit {u}")
        else:
            assert np.array_equal(got, ref)
        assert np.array_equal(kd[off:off + n], k[b][h][got])
        score_close(sc[off:off + n], A[got])


def test_span_prune_ragged_spans():
    lengths = [1200, 3000, 700, 64]
    spans = [(100, 900), (0, 2990), (650, 10 ** 6), (-5, 30)]
    keeps = [160, 600, 10, 0]
    run_prune(lengths, spans, keeps)


def test_span_prune_edges():
    # empty span, keep more than the span, span past the end, pool 1
    lengths = [500, 333, 900]
    spans = [(200, 200), (10, 300), (950, 1000)]
    keeps = [5, 10 ** 6, 3]
    run_prune(lengths, spans, keeps, pool=1, D=64, Hq=8, Hkv=2, W=8, seed=4)


@pytest.mark.parametrize("sink,recent", [(1, 3), (4, 60), (0, 1), (2, 0), (200, 200)])
def test_sink_recent_view_decode(sink, recent):
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="streaming", batch=3, ctx=(1000, 2053, 17),
                     budget=(synth.UNBOUNDED_BUDGET,) * 3,
                     steps=2)
    inputs = synth.quest_inputs(w)
    run = QuestRun(w, inputs, out_dtype=1)
    G, Hkv = run.G, run.Hkv
    view = se.View.empty(run.B * Hkv, run.sel.shape[1])
    for s in range(w.steps):
        run.append(s)
        se.se_view_sink_recent(run.kv, run.B, sink, recent, view, run.ws_small)
        se.se_sparse_decode(run.kv.k, run.kv.v, view, run.q[s], run.B, run.Hq, Hkv, run.D,
                            run.scale, run.out, run.lse, run.ws_dec, out_dtype=1)
        torch.cuda.synchronize()
        out = run.out.double().cpu().numpy()
        for u in range(run.B * Hkv):
            b, h = divmod(u, Hkv)
            L = w.ctx[b] + s + 1
            pages = oracle.sink_recent_pages(L, sink, recent)
            tok = selected_tokens(pages, L)
            K = oracle.widen(inputs["k"][b][h, :L])
            V = oracle.widen(inputs["v"][b][h, :L])
            q = oracle.widen(inputs["q"][s, b, h * G:(h + 1) * G])
            o_ref, _ = oracle.attend(q, K[tok], V[tok], run.scale)
            assert int(view.n_tokens[u]) == len(tok)
            assert max_abs(out[b, h * G:(h + 1) * G], o_ref) <= TOL_F32, (u, s)
    assert run.status() == 0
