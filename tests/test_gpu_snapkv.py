"""GPU parity: SnapKV compaction (window scores, max-pool, per-head top-k,
varlen compaction) through the C ABI against the oracle, then decode over the
compacted caches; small ragged cases, the edge cases, and the full-size
32K-context workload."""
import math

import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_quest_gb300 import binding as se
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import PAGE, SnapKVRun, paged_layout, to_dev_bf16
from tests.parity import TOL_BF16, bf16_tensor_to_f64, check_topk, max_abs

pytestmark = pytest.mark.gpu


def score_close(gpu, ref):
    gpu, ref = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    assert np.all(err <= 1e-5 + 1e-4 * np.abs(ref)), f"max err {err.max()}"


def run_compaction(B, Hq, Hkv, D, lengths, W, pool, keep, recent, seed=0, extra_cap=0):
    """Compaction of random inputs; returns (logical inputs, varlen cache, status)."""
    g = np.random.default_rng(seed)
    G = Hq // Hkv
    Lmax = max(lengths)
    k = [synth.f32_to_bf16_bits(g.standard_normal((Hkv, L, D)).astype(np.float32)) for L in lengths]
    v = [synth.f32_to_bf16_bits(g.standard_normal((Hkv, L, D)).astype(np.float32)) for L in lengths]
    q_win = synth.f32_to_bf16_bits(g.standard_normal((B, W, Hq, D)).astype(np.float32))
    pages = np.array([-(-L // PAGE) for L in lengths])
    bt, num_pages = synth.block_table(seed, "snap_test_bt", pages)
    K, V = paged_layout(k, v, lengths, bt, num_pages, Hkv, D)
    pre = se.PagedKV(to_dev_bf16(K), to_dev_bf16(V), torch.zeros(1, dtype=torch.bfloat16,
                                                                   device="cuda"),
                     torch.from_numpy(bt).cuda(), torch.tensor(lengths, dtype=torch.int32,
                                                               device="cuda"))
    cap = Lmax + extra_cap
    out = se.VarlenKV.empty(B, Hkv, cap, D, with_score=True)
    ws = se.workspace(se.se_snapkv_workspace(B, Hkv, Hq, W, Lmax))
    se.se_snapkv_compact(pre, to_dev_bf16(q_win), B, Hq, W, pool, keep, recent, 1 / math.sqrt(D),
                         out, ws)
    torch.cuda.synchronize()
    return {"k": k, "v": v, "q_win": q_win, "G": G}, out, se.status_word(ws)


def check_units(inp, out, B, Hkv, D, lengths, W, pool, keep, recent):
    pos_all = out.pos.cpu().numpy()
    kd = out.k.view(torch.int16).cpu().numpy().view(np.uint16)
    vd = out.v.view(torch.int16).cpu().numpy().view(np.uint16)
    sc = out.score.cpu().numpy()
    seg_len = out.seg_len.cpu().numpy()
    seg_off = out.seg_off.cpu().numpy()
    assert out.seq_len.cpu().numpy().tolist() == list(lengths)
    G = inp["G"]
    for u in range(B * Hkv):
        b, h = divmod(u, Hkv)
        L = lengths[b]
        q = oracle.widen(inp["q_win"][b][:, h * G:(h + 1) * G])          # [W][G][D]
        K = oracle.widen(inp["k"][b][h])
        A = oracle.window_scores(q, K, 1 / math.sqrt(D))
        R = min(recent, L)
        ref_pos = oracle.keep_positions(A, L, R, keep, pool)
        n = int(seg_len[u])
        assert n == len(ref_pos)
        off = int(seg_off[u])
        gpos = pos_all[off:off + n]
        assert np.all(np.diff(gpos) > 0)
        assert gpos[len(gpos) - R:].tolist() == list(range(L - R, L))
        ncand = L - R
        K_ = min(keep, ncand)
        if 0 < K_ < ncand:
            pooled = oracle.max_pool(A[:ncand], pool)
            boundary = pooled[oracle.rank_order(pooled)[K_ - 1]]
            check_topk(gpos[:K_], ref_pos[:K_], pooled, boundary, what=f"unit {u}")
        else:
            assert np.array_equal(gpos, ref_pos)
        # compaction: bit-exact rows, scores of the kept tokens
        assert np.array_equal(kd[off:off + n], inp["k"][b][h][gpos])
        assert np.array_equal(vd[off:off + n], inp["v"][b][h][gpos])
        score_close(sc[off:off + n], A[gpos])


def test_keep_everything_exposes_window_scores():
    B, Hq, Hkv, D, W = 2, 8, 2, 64, 8
    lengths = [300, 517]
    inp, out, st = run_compaction(B, Hq, Hkv, D, lengths, W, pool=7, keep=10 ** 6, recent=W)
    assert st == 0
    check_units(inp, out, B, Hkv, D, lengths, W, 7, 10 ** 6, W)


@pytest.mark.parametrize("pool", [1, 3, 7])
def test_ragged_selection_and_compaction(pool):
    B, Hq, Hkv, D, W = 3, 32, 4, 128, 32
    lengths = [1000, 4133, 2056]
    inp, out, st = run_compaction(B, Hq, Hkv, D, lengths, W, pool=pool, keep=256, recent=W, seed=pool)
    assert st == 0
    check_units(inp, out, B, Hkv, D, lengths, W, pool, 256, W)


def test_h2o_style_seeding_recent_larger_than_window():
    B, Hq, Hkv, D, W = 2, 16, 2, 128, 16
    lengths = [1500, 900]
    inp, out, st = run_compaction(B, Hq, Hkv, D, lengths, W, pool=1, keep=200, recent=96, seed=5)
    assert st == 0
    check_units(inp, out, B, Hkv, D, lengths, W, 1, 200, 96)


def test_context_not_longer_than_recent():
    B, Hq, Hkv, D, W = 2, 8, 2, 64, 4
    lengths = [4, 30]
    inp, out, st = run_compaction(B, Hq, Hkv, D, lengths, W, pool=7, keep=5, recent=30, seed=3)
    assert st == 0
    check_units(inp, out, B, Hkv, D, lengths, W, 7, 5, 30)


def _decode_check(run, s, units):
    """Oracle attention over the GPU's compacted segment after step s."""
    c = run.cache
    seg_off = c.seg_off.cpu().numpy()
    seg_len = c.seg_len.cpu().numpy()
    kd = c.k.view(torch.int16).cpu().numpy().view(np.uint16)
    vd = c.v.view(torch.int16).cpu().numpy().view(np.uint16)
    out = bf16_tensor_to_f64(run.out)
    q = run.dec_inputs["q"]
    G = run.G
    for u in units:
        b, h = divmod(u, run.Hkv)
        o, n = int(seg_off[u]), int(seg_len[u])
        ref, _ = oracle.attend(oracle.widen(q[s, b, h * G:(h + 1) * G]), oracle.widen(kd[o:o + n]),
                               oracle.widen(vd[o:o + n]), run.scale)
        err = max_abs(out[b, h * G:(h + 1) * G], ref)
        assert err <= TOL_BF16, (s, u, err)


def test_decode_over_compacted_caches_small():
    base = synth.workloads()["snapkv_32k"]
    w = synth.scaled(base, name="snap_small", batch=2, groups=2, ctx=2000, keep=300, steps=3)
    run = SnapKVRun(w, keep_inputs=True, with_score=True)
    for g in range(run.groups):
        inp = dict(run.inputs[g], G=run.G)
        sl = run.group_slice(g)
        check_units(inp, sl, w.batch, w.num_kv_heads, w.head_dim, [w.ctx] * w.batch, w.window,
                    w.pool_kernel, w.keep, w.window)
    seg_len0 = run.cache.seg_len.clone()
    for s in range(w.steps):
        run.step(s)
        torch.cuda.synchronize()
        assert torch.equal(run.cache.seg_len, seg_len0 + s + 1)
        # the appended token's position is the next logical position
        _decode_check(run, s, range(run.Bt * run.Hkv))
    assert run.status() == 0


def test_fused_varlen_append_view_matches_separate_calls():
    """se_varlen_append_view == se_varlen_append + se_view_from_segments, bit
    for bit: cache rows, positions, scores, lengths and the view, step by step."""
    base = synth.workloads()["snapkv_32k"]
    w = synth.scaled(base, name="snap_fused", batch=3, groups=1, ctx=700, keep=100, steps=18)
    a = SnapKVRun(w, with_score=True)
    b = SnapKVRun(w, with_score=True)
    for s in range(w.steps):
        a.step(s, fused=True)
        b.step(s, fused=False)
        torch.cuda.synchronize()
        assert torch.equal(a.cache.seg_len.cpu(), b.cache.seg_len.cpu()), s
        assert torch.equal(a.cache.seq_len.cpu(), b.cache.seq_len.cpu()), s
        assert torch.equal(a.view.n_tokens.cpu(), b.view.n_tokens.cpu()), s
        nt = b.view.n_tokens.cpu()
        for u in range(len(nt)):
            nc = -(-int(nt[u]) // 16)
            assert torch.equal(a.view.chunk_row[u, :nc].cpu(), b.view.chunk_row[u, :nc].cpu())
        assert torch.equal(a.out.cpu(), b.out.cpu()), s
    for name in ("k", "v", "pos", "score"):
        assert torch.equal(getattr(a.cache, name).cpu(), getattr(b.cache, name).cpu()), name
    assert a.status() == 0 and b.status() == 0


@pytest.mark.slow
def test_full_size_snapkv_32k():
    """Compaction of 8 x 32K-context prefills (every unit checked), then all 64
    decode steps of the 64-request batch with steps 0 and 63 checked."""
    w = synth.workloads()["snapkv_32k"]
    run = SnapKVRun(w, groups=8, keep_inputs=True, with_score=True)
    inp = dict(run.inputs[0], G=run.G)
    check_units(inp, run.group_slice(0), w.batch, w.num_kv_heads, w.head_dim, [w.ctx] * w.batch,
                w.window, w.pool_kernel, w.keep, w.window)
    for s in range(w.steps):
        run.step(s)
        if s in (0, w.steps - 1):
            torch.cuda.synchronize()
            _decode_check(run, s, range(0, run.Bt * run.Hkv, 7))
    torch.cuda.synchronize()
    assert run.status() == 0
