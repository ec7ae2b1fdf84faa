"""GPU parity: Quest selection + split-K decode (through the C ABI) against the
oracle, step by step, on seeded inputs: the tiny single-query case, ragged
multi-step cases across group sizes and head dims, the edge cases (k = 1,
budget >= context, empty prefill, one split vs many), and the full-size
32K-context and ragged 64K-128K workloads on sampled (step, unit) pairs."""
import math

import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import QuestRun
from tests.parity import TOL_BF16, TOL_F32, bf16_tensor_to_f64, check_topk, max_abs

pytestmark = pytest.mark.gpu
U32 = synth.UNBOUNDED_BUDGET
# int32 words of the one-kernel step's workspace head: status header, sync
# words, 1024 per-sequence and 4096 per-unit counters
CTL_WORDS = (256 + 256 + 1024 * 4 + 4096 * 4) // 4


def oracle_unit(w, inputs, b, h, s, gpu_pages=None, agg=0):
    """Oracle for unit (b, h) at step s (after that step's append).  Returns
    (U, oracle pages, k, out [G][D], lse [G]) where the attention uses the
    GPU's page set when given (after it passed the selection check); agg 1
    takes the max-aggregation bound."""
    G = w.num_q_heads // w.num_kv_heads
    L = w.ctx[b] + s + 1
    K = oracle.widen(inputs["k"][b][h, :L])
    V = oracle.widen(inputs["v"][b][h, :L])
    q = oracle.widen(inputs["q"][s, b, h * G:(h + 1) * G])
    kmin, kmax = oracle.page_minmax(K)
    U = (oracle.quest_bound_max if agg else oracle.quest_bound)(q, kmin, kmax)
    k = oracle.quest_k_pages(min(w.budget[b], U32))
    pages = oracle.quest_select(U, k)
    use = pages if gpu_pages is None else np.asarray(gpu_pages)
    tok = oracle.quest.selected_tokens(use, L)
    out, lse = oracle.attend(q, K[tok], V[tok], 1.0 / math.sqrt(w.head_dim))
    return U, pages, k, out, lse


def check_step(run, inputs, s, units=None):
    w = run.w
    G, Hkv = run.G, run.Hkv
    sel = run.sel.cpu().numpy()
    n_sel = run.n_sel.cpu().numpy()
    out = bf16_tensor_to_f64(run.out)
    lse = run.lse.cpu().numpy().astype(np.float64)
    tol = TOL_F32 if run.out_dtype == 1 else TOL_BF16
    worst = 0.0
    allowed = 0
    for u in (range(run.B * Hkv) if units is None else units):
        b, h = divmod(u, Hkv)
        gpu_pages = sel[u, :n_sel[u]]
        assert np.all(np.diff(gpu_pages) > 0), "pages not ascending"
        U, pages, k, _, _ = oracle_unit(w, inputs, b, h, s, agg=run.group_agg)
        n = len(U)
        if n > k:
            cand = U[:n - 1]
            boundary = cand[oracle.rank_order(cand)[k - 2]] if k >= 2 else np.inf
            assert gpu_pages[-1] == n - 1, "last page not forced"
            if k >= 2:
                allowed += check_topk(gpu_pages[:-1], pages[:-1], cand, boundary,
                                      what=f"step {s} unit {u}")
            else:
                assert len(gpu_pages) == 1
        else:
            assert np.array_equal(gpu_pages, pages)
        _, _, _, o_ref, l_ref = oracle_unit(w, inputs, b, h, s, gpu_pages, agg=run.group_agg)
        err = max_abs(out[b, h * G:(h + 1) * G], o_ref)
        worst = max(worst, err)
        assert err <= tol, f"step {s} unit {u}: max-abs {err} > {tol}"
        assert max_abs(lse[b, h * G:(h + 1) * G], l_ref) <= 1e-3
    return worst, allowed


def run_and_check(w, out_dtype=0, max_splits=None, steps=None, units=None, mode="step",
                  step_tuning=None, group_agg=0):
    inputs = synth.quest_inputs(w)
    run = QuestRun(w, inputs, out_dtype=out_dtype, max_splits=max_splits, mode=mode,
                   step_tuning=step_tuning)
    run.group_agg = group_agg
    worst = 0.0
    for s in range(w.steps):
        run.step(s)
        if steps is None or s in steps:
            torch.cuda.synchronize()
            e, _ = check_step(run, inputs, s, units)
            worst = max(worst, e)
    torch.cuda.synchronize()
    assert run.status() == 0, f"device status word {run.status()}"
    return worst


@pytest.mark.parametrize("mode", QuestRun.MODES)
def test_tiny_quest_single_query(mode):
    w = synth.workloads()["tiny_quest"]
    run_and_check(w, mode=mode)
    run_and_check(w, out_dtype=1, mode=mode)


def test_fused_append_select_matches_separate_calls():
    """se_quest_select_append == se_kv_append + se_quest_select, bit for bit:
    selections, view, lengths, cache rows, page summaries and the attention
    output, over steps that open new pages (contexts 15, 16, 31 and 1000 tokens
    at the start) and a sequence whose pages are all selected."""
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_fused", batch=5, ctx=(15, 16, 31, 1000, 2047),
                     budget=(64, 64, 256, 128, U32), steps=20)
    inputs = synth.quest_inputs(w)
    a = QuestRun(w, inputs, mode="fused")
    b = QuestRun(w, inputs, mode="separate")
    for s in range(w.steps):
        a.step(s)
        b.step(s)
        torch.cuda.synchronize()
        n = b.n_sel.cpu()
        assert torch.equal(a.n_sel.cpu(), n), f"step {s}"
        for u in range(len(n)):
            k = int(n[u])
            assert torch.equal(a.sel[u, :k].cpu(), b.sel[u, :k].cpu()), f"step {s} unit {u}"
            assert torch.equal(a.view.chunk_row[u, :k].cpu(), b.view.chunk_row[u, :k].cpu())
        assert torch.equal(a.view.n_tokens.cpu(), b.view.n_tokens.cpu())
        assert torch.equal(a.kv.ctx_len.cpu(), b.kv.ctx_len.cpu())
        assert torch.equal(a.out.cpu(), b.out.cpu())
    assert torch.equal(a.kv.k.cpu(), b.kv.k.cpu())
    assert torch.equal(a.kv.v.cpu(), b.kv.v.cpu())
    assert torch.equal(a.kv.meta.cpu(), b.kv.meta.cpu())
    assert a.status() == 0 and b.status() == 0


@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("mode", ["step", "fused"])
def test_ragged_multi_step_outliers(out_dtype, mode):
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_ragged_small", batch=4, ctx=(1000, 2053, 300, 0),
                     budget=(256, 512, 4096, 64), steps=5)
    run_and_check(w, out_dtype=out_dtype, mode=mode)


def test_one_kernel_step_matches_two_calls():
    """se_quest_step == se_quest_select_append + se_sparse_decode: selections,
    view, lengths, cache rows and page summaries bit for bit, outputs within
    the rounding of their different split pieces; steps open new pages
    (contexts 15, 16, 31, 1000 and 2047 tokens at the start, one sequence with
    every page selected), and the split limit of the step's decode plan is
    varied from step to step."""
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_step_eq", batch=5, ctx=(15, 16, 31, 1000, 2047),
                     budget=(64, 64, 256, 128, U32), steps=12)
    inputs = synth.quest_inputs(w)
    a = QuestRun(w, inputs, mode="step", out_dtype=1)
    b = QuestRun(w, inputs, mode="fused", out_dtype=1)
    top = a.max_splits                                   # the workspace's split count
    splits = [top, 1, 3, 7, 2, top, 5]
    for s in range(w.steps):
        a.max_splits = min(top, splits[s % len(splits)])
        a.step(s)
        b.step(s)
        torch.cuda.synchronize()
        n = b.n_sel.cpu()
        assert torch.equal(a.n_sel.cpu(), n), f"step {s}"
        for u in range(len(n)):
            k = int(n[u])
            assert torch.equal(a.sel[u, :k].cpu(), b.sel[u, :k].cpu()), f"step {s} unit {u}"
            assert torch.equal(a.view.chunk_row[u, :k].cpu(), b.view.chunk_row[u, :k].cpu())
        assert torch.equal(a.view.n_tokens.cpu(), b.view.n_tokens.cpu())
        assert torch.equal(a.kv.ctx_len.cpu(), b.kv.ctx_len.cpu())
        assert max_abs(a.out.double().cpu().numpy(), b.out.double().cpu().numpy()) <= 1e-4
        assert max_abs(a.lse.cpu().numpy(), b.lse.cpu().numpy()) <= 1e-4
    assert torch.equal(a.kv.k.cpu(), b.kv.k.cpu())
    assert torch.equal(a.kv.v.cpu(), b.kv.v.cpu())
    assert torch.equal(a.kv.meta.cpu(), b.kv.meta.cpu())
    assert a.status() == 0 and b.status() == 0
    # the control words (finished blocks, abort word, scored pages per
    # sequence, split arrival counters) sit right after the status header,
    # and every call leaves them at zero
    assert int(a.ws_step.view(torch.int32)[64:CTL_WORDS].abs().sum().item()) == 0, "not reset"


# (hkv 8 at d 128 and hkv 3 at d 64 take the scoring path with coefficients in
# shared memory; the others keep them in registers)
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (8, 4, 64), (32, 4, 128), (32, 2, 64),
                                       (64, 4, 128), (16, 4, 64), (64, 8, 128), (6, 3, 64),
                                       (16, 1, 128)])
@pytest.mark.parametrize("mode", ["step", "fused"])
def test_group_sizes_and_head_dims(hq, hkv, d, mode):
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name=f"quest_g{hq // hkv}_d{d}", batch=2, num_q_heads=hq,
                     num_kv_heads=hkv, head_dim=d, ctx=(777, 1600), budget=(128, 256), steps=2)
    run_and_check(w, mode=mode)


@pytest.mark.parametrize("mode", ["step", "fused"])
def test_budget_of_one_page_and_full_budget(mode):
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_edges", batch=3, ctx=(500, 129, 2000),
                     budget=(16, U32, U32), steps=2)
    run_and_check(w, out_dtype=1, mode=mode)


@pytest.mark.parametrize("max_splits", [1, 3, 64])
@pytest.mark.parametrize("mode", ["step", "fused"])
def test_split_count_does_not_change_results(max_splits, mode):
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_splits", batch=2, ctx=(3000, 1234), budget=(U32, 1024),
                     steps=1)
    run_and_check(w, out_dtype=1, max_splits=max_splits, mode=mode)


def test_many_units_block_plan():
    """640 units (more than the single-warp plan takes): the block-wide plan,
    with short ragged contexts so that some units are split and some not."""
    base = synth.workloads()["quest_32k"]
    B = 160
    ctx = tuple(int(x) for x in (np.arange(B) * 37 % 900 + 20))
    w = synth.scaled(base, name="quest_many_units", batch=B, ctx=ctx, budget=(256,) * B, steps=1)
    run_and_check(w, units=range(0, B * 4, 7), mode="fused")
    run_and_check(w, units=range(0, B * 4, 7), mode="step")


def _tied_inputs(w):
    """Sequences 0 and 1: their best-scoring page (KV head 0, step 0) copied
    over pages [40, 200) and [30, 70), so that 161 and 41 candidate pages tie
    at the top score, more than the budget keeps; sequence 3: its page of the
    54th best score copied over pages [300, 320), so that the budget's
    boundary falls inside the 21 tied pages; sequence 2: one page repeated
    throughout (every score equal).  Returns the inputs and the tied page
    groups."""
    inputs = synth.quest_inputs(w)
    groups = {}
    for b, (lo, hi), nth in ((0, (40, 200), 0), (1, (30, 70), 0), (3, (300, 320), 53)):
        U = oracle_unit(w, inputs, b, 0, 0)[0]
        src = int(oracle.rank_order(U[:len(U) - 1])[nth])
        k = inputs["k"][b]
        for pg in range(lo, hi):
            k[:, pg * 16:(pg + 1) * 16] = k[:, src * 16:(src + 1) * 16]
        groups[b] = sorted(set(range(lo, hi)) | {src})
    k = inputs["k"][2]
    for pg in range(1, (w.ctx[2] + w.steps) // 16):
        k[:, pg * 16:(pg + 1) * 16] = k[:, 0:16]
    return inputs, groups


@pytest.mark.parametrize("mode", ["step", "fused"])
def test_tied_scores_keep_page_order(mode):
    """Exact ties at the selection boundary are broken by page order: 161 tied
    pages at the top (more than one boundary bin holds, so the radix passes
    decide), 41 tied pages at the top (ranked inside the boundary bin), 21
    tied pages across the boundary of a 750-page sequence, and all-equal
    scores."""
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="quest_ties", batch=4, ctx=(4000, 3000, 2500, 12000),
                     budget=(1024, 512, 256, 1024), steps=1)
    inputs, groups = _tied_inputs(w)
    run = QuestRun(w, inputs, mode=mode, out_dtype=1)
    run.step(0)
    torch.cuda.synchronize()
    assert run.status() == 0
    check_step(run, inputs, 0)
    Hkv = w.num_kv_heads
    sel = run.sel.cpu().numpy()
    n_sel = run.n_sel.cpu().numpy()
    for b, grp in groups.items():
        u = b * Hkv                                       # head 0: the group's scores
        pages = set(sel[u, :n_sel[u]].tolist())
        k = w.budget[b] // 16
        taken = [pg for pg in grp if pg in pages]
        if b < 2:                                         # the group is the top
            assert taken == grp[:k - 1], f"sequence {b}: tied pages not taken in page order"
        else:                                             # the boundary is inside it
            assert 0 < len(taken) < len(grp), f"sequence {b}: boundary not inside the group"
            assert taken == grp[:len(taken)], f"sequence {b}: tied pages not taken in page order"
    n = (w.ctx[2] + 1 + 15) // 16
    k = w.budget[2] // 16
    for h in range(Hkv):
        u = 2 * Hkv + h
        assert sel[u, :n_sel[u]].tolist() == list(range(k - 1)) + [n - 1]


def test_more_sequences_than_blocks():
    """1024 sequences x 4 KV heads (the step's batch and unit limits), more
    sequences than resident blocks: each block scores several whole
    sequences; short ragged contexts, a 4-page budget."""
    base = synth.workloads()["quest_32k"]
    B = 1024
    ctx = tuple(int(x) for x in (np.arange(B) * 53 % 700 + 5))
    w = synth.scaled(base, name="quest_max_batch", batch=B, ctx=ctx, budget=(64,) * B, steps=1)
    run_and_check(w, units=range(0, B * 4, 37), mode="step")
    run_and_check(w, units=range(3, B * 4, 41), mode="fused")


def test_stream_k_plan():
    """One 30K-token sequence among 99 short ones, every page attended: the
    proportional one-piece-per-CTA plan does not fit the grid, so the units
    are cut stream-K (equal chunk ranges per CTA, pieces merged by LSE)."""
    base = synth.workloads()["quest_32k"]
    B = 100
    w = synth.scaled(base, name="quest_streamk", batch=B, ctx=(30000,) + (40,) * (B - 1),
                     budget=(U32,) * B, steps=1)
    run_and_check(w, out_dtype=1, units=[0, 1, 2, 3, 4, 5, 100, 399], mode="fused")
    run_and_check(w, out_dtype=1, units=[0, 1, 2, 3, 4, 5, 100, 399], mode="step")


def test_ragged_long_scaled():
    base = synth.workloads()["ragged_quest_128k"]
    w = synth.scaled(base, name="ragged_small", batch=4, ctx=(2300, 4100, 3333, 2900),
                     budget=(U32, 512, U32, 512), steps=3)
    run_and_check(w, mode="fused")
    run_and_check(w, mode="step")


@pytest.mark.slow
def test_full_size_quest_32k_sampled():
    """The 16 x 32K-context workload, all 64 steps on the GPU with the bench's
    launch configuration; the oracle checks steps 0, 31, 63 on every unit."""
    w = synth.workloads()["quest_32k"]
    run_and_check(w, steps={0, 31, 63})
    run_and_check(w, steps={0, 63}, mode="fused")


@pytest.mark.slow
def test_full_size_ragged_128k_sampled():
    """The ragged 64K-128K workload (half dense-equivalent), all 32 steps on
    the GPU; the oracle checks steps 0 and 31 on units of every sequence."""
    w = synth.workloads()["ragged_quest_128k"]
    run_and_check(w, steps={0, 31}, units=list(range(0, 32, 3)), mode="fused")
    run_and_check(w, steps={0, 31}, units=list(range(0, 32, 3)), mode="step")


def test_step_wait_that_runs_out_reports_timeout_and_resets():
    """A bounded wait that runs out sets SE_DEV_TIMEOUT, leaves ctx_len
    unchanged and the control words at zero; the next call, with the default
    limit and the status word cleared, matches the oracle.  The wait is made
    to run out by a limit of 1 ns and a skewed batch: 40 sequences take an
    equal share of the blocks each, so the blocks that score one page of a
    20-token sequence reach the pieces of the 30000-token one long before the
    few blocks that score it are done."""
    base = synth.workloads()["quest_32k"]
    B = 40
    w = synth.scaled(base, name="quest_timeout", batch=B, ctx=(30000,) + (20,) * (B - 1),
                     budget=(2048,) + (16,) * (B - 1), steps=2)
    inputs = synth.quest_inputs(w)
    run = QuestRun(w, inputs, mode="step", step_tuning={"wait_limit_ns": 1})
    ctx0 = run.kv.ctx_len.clone()
    run.step(0)
    st = se_status(run.ws_step)
    assert st & 8, f"status {st}: expected SE_DEV_TIMEOUT"
    assert torch.equal(run.kv.ctx_len, ctx0), "lengths committed after an abort"
    assert int(run.ws_step.view(torch.int32)[64:CTL_WORDS].abs().sum().item()) == 0
    run.ws_step.zero_()
    run.step_tuning = {}
    run.step(0)
    torch.cuda.synchronize()
    assert run.status() == 0
    check_step(run, inputs, 0)


def se_status(ws):
    from kv_cache_decode_quest_gb300 import binding
    return binding.se_sync_status(ws)


@pytest.mark.parametrize("hq,hkv,d", [(32, 4, 128), (16, 2, 64), (8, 8, 128), (4, 1, 64),
                                       (16, 8, 128), (2, 2, 64)])
def test_max_aggregation_bound(hq, hkv, d):
    """se_quest_select_ex with SE_AGG_MAX (the largest of the query heads'
    bounds): selections against the oracle's max bound, outputs against the
    oracle attention, with the append fused, over ragged contexts."""
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name=f"quest_max_g{hq // hkv}_d{d}", batch=3, num_q_heads=hq,
                     num_kv_heads=hkv, head_dim=d, ctx=(777, 3000, 40), budget=(128, 512, 64),
                     steps=3)
    run_and_check(w, mode="fused", group_agg=1)


def test_max_aggregation_full_size_sampled():
    """The 16 x 32K workload with the max bound, steps 0 and 3."""
    w = synth.scaled(synth.workloads()["quest_32k"], steps=4)
    run_and_check(w, mode="fused", group_agg=1, steps={0, 3}, units=list(range(0, 64, 5)))
