"""GPU parity: cross-layer selection reuse (OmniKV-style) through the C ABI.

The filter layers select pages with se_quest_select_append; every layer
appends its own token (se_kv_append without page summaries for the others)
and decodes with se_sparse_decode through the view of the latest filter layer
at or before it.  Each (layer, unit) is compared with the oracle: the filter
layers' selections exactly (up to the boundary allowance), the outputs within
the bf16 / fp32 tolerance, with the oracle attending over the GPU's pages."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.quest import selected_tokens
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import OmniRun
from tests.parity import TOL_BF16, TOL_F32, check_topk, max_abs

pytestmark = pytest.mark.gpu
U32 = synth.UNBOUNDED_BUDGET


def check_omni_step(run, inputs, s, units=None):
    w = run.w
    G, Hkv, L = run.G, run.Hkv, run.L
    tol = TOL_F32 if run.out_dtype == 1 else TOL_BF16
    sel = {f: run.sel[f].cpu().numpy() for f in run.filters}
    nsel = {f: run.n_sel[f].cpu().numpy() for f in run.filters}
    outs = [o.double().cpu().numpy() for o in run.out]
    lses = [x.double().cpu().numpy() for x in run.lse]
    scale = 1.0 / math.sqrt(w.head_dim)
    for u in (range(run.B * Hkv) if units is None else units):
        b, h = divmod(u, Hkv)
        T = w.ctx[b] + s + 1
        qs = [oracle.widen(inputs[x]["q"][s, b, h * G:(h + 1) * G]) for x in range(L)]
        ks = [oracle.widen(inputs[x]["k"][b][h, :T]) for x in range(L)]
        vs = [oracle.widen(inputs[x]["v"][b][h, :T]) for x in range(L)]
        ref = oracle.omnikv_layers(qs, ks, vs, run.filters, min(w.budget[b], U32), scale)
        for f in run.filters:
            gpu_pages = sel[f][u, :nsel[f][u]]
            pages = ref[f][0]
            U = oracle.quest_bound(qs[f], *oracle.page_minmax(ks[f]))
            k = oracle.quest_k_pages(min(w.budget[b], U32))
            n = len(U)
            if n > k and k >= 2:
                cand = U[:n - 1]
                boundary = cand[oracle.rank_order(cand)[k - 2]]
                assert gpu_pages[-1] == n - 1
                check_topk(gpu_pages[:-1], pages[:-1], cand, boundary, what=f"layer {f} unit {u}")
            else:
                assert np.array_equal(gpu_pages, pages), (f, u)
        for layer in range(L):
            f = oracle.source_layer(layer, run.filters)
            tok = selected_tokens(sel[f][u, :nsel[f][u]], T)
            o_ref, l_ref = oracle.attend(qs[layer], ks[layer][tok], vs[layer][tok], scale)
            err = max_abs(outs[layer][b, h * G:(h + 1) * G], o_ref)
            assert err <= tol, f"step {s} layer {layer} unit {u}: max-abs {err}"
            assert max_abs(lses[layer][b, h * G:(h + 1) * G], l_ref) <= 1e-3


def run_omni(w, out_dtype=0, steps=None, units=None):
    inputs = synth.omnikv_inputs(w)
    run = OmniRun(w, inputs, out_dtype=out_dtype)
    for s in range(w.steps):
        run.step(s)
        if steps is None or s in steps:
            torch.cuda.synchronize()
            check_omni_step(run, inputs, s, units)
    torch.cuda.synchronize()
    assert run.status() == 0, run.status()
    # every layer appended every step
    for kv in run.kv:
        assert np.array_equal(kv.ctx_len.cpu().numpy(), np.asarray(w.ctx) + w.steps)


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_reuse_small_ragged(out_dtype):
    base = synth.workloads()["omnikv_32k"]
    w = synth.scaled(base, name="omni_small", batch=3, ctx=(1000, 2053, 300),
                     budget=(256, 512, U32), steps=3, layers=4, filters=(0, 2))
    run_omni(w, out_dtype)


def test_reuse_single_filter_group_sizes():
    base = synth.workloads()["omnikv_32k"]
    w = synth.scaled(base, name="omni_g", batch=2, num_q_heads=16, num_kv_heads=2, head_dim=64,
                     ctx=(777, 1600), budget=(128, 64), steps=2, layers=3, filters=(0,))
    run_omni(w)


@pytest.mark.slow
def test_full_size_omnikv_32k_sampled():
    """The 16 x 32K workload through 4 layers (filter layer 0) in the bench's
    launch configuration; the oracle checks steps 0 and the last on units of
    every sequence."""
    w = synth.workloads()["omnikv_32k"]
    run_omni(w, steps={0, w.steps - 1}, units=list(range(0, 64, 5)))
