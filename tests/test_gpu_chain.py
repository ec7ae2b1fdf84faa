"""GPU: Chain Cache save / restore of retained state (se_chain_save,
se_chain_restore).  A restored state decodes exactly as the saved one: H2O
steps after a restore into another segment layout match, bit for bit, the
steps of the original state continued; restored rows, positions and scores
equal the saved bytes; a restore into other sequence slots matches the oracle
(teacher forced); SnapKV decode resumes bit for bit; a snapshot of another
shape is refused by the kernel (status bit, cache left as is)."""
import math

import numpy as np
import pytest
import torch

from kv_cache_decode_quest_gb300 import binding as se
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import H2ORun, SnapKVRun
from tests.test_gpu_h2o import check_step, gpu_unit_state

pytestmark = pytest.mark.gpu


def _h2o_workload():
    base = synth.workloads()["h2o_16k"]
    return synth.scaled(base, name="chain_h2o", batch=3, num_q_heads=8, num_kv_heads=2,
                        head_dim=64, ctx=700, budget=200, recent=24, window=8, steps=12)


def _fresh_like(kv: se.VarlenKV, batch, reverse=True):
    """An empty cache of the same shape whose segments sit in another order,
    one row apart (a different physical layout)."""
    H, cap, D = kv.num_kv_heads, kv.seg_cap, kv.k.shape[1]
    units = batch * H
    rows = units * (cap + 1)
    order = torch.arange(units, dtype=torch.int32, device="cuda")
    if reverse:
        order = units - 1 - order
    return se.VarlenKV(
        torch.zeros(rows, D, dtype=torch.bfloat16, device="cuda"),
        torch.zeros(rows, D, dtype=torch.bfloat16, device="cuda"),
        torch.full((rows,), -1, dtype=torch.int32, device="cuda"),
        None if kv.score is None else torch.zeros(rows, dtype=torch.float32, device="cuda"),
        order * (cap + 1) + 1, torch.zeros(units, dtype=torch.int32, device="cuda"),
        torch.zeros(batch, dtype=torch.int32, device="cuda"), cap, H)


def _snapshot(kv, seqs, rows, ws):
    snap = torch.zeros(se.se_chain_snapshot_bytes(len(seqs), kv.num_kv_heads, kv.k.shape[1], rows,
                                                  kv.score is not None),
                       dtype=torch.uint8, device="cuda")
    se.se_chain_save(kv, torch.tensor(seqs, dtype=torch.int32, device="cuda"), rows, snap, ws)
    return snap


def test_h2o_resume_is_bit_exact():
    w = _h2o_workload()
    run = H2ORun(w, keep_inputs=True)
    s1 = 5
    for s in range(s1):
        run.step(s)
    torch.cuda.synchronize()
    units = w.batch * w.num_kv_heads
    saved = [gpu_unit_state(run, u) for u in range(units)]
    ws = se.workspace(se.se_small_workspace())
    snap = _snapshot(run.state.kv, list(range(w.batch)), run.cap, ws)
    # the original continues
    outs, evs = [], []
    for s in range(s1, w.steps):
        run.step(s)
        outs.append(run.out.clone())
        evs.append(run.evicted.clone())
    torch.cuda.synchronize()
    final = [gpu_unit_state(run, u) for u in range(units)]
    # a restore into another layout, then the same steps
    fresh = _fresh_like(run.state.kv, w.batch)
    se.se_chain_restore(snap, run.cap, torch.arange(w.batch, dtype=torch.int32, device="cuda"),
                        fresh, ws)
    torch.cuda.synchronize()
    assert se.status_word(ws) == 0
    run2 = H2ORun.__new__(H2ORun)
    run2.__dict__.update(run.__dict__)
    run2.state = se.H2OState(fresh, w.budget, w.recent)
    run2.ws = se.workspace(se.se_h2o_workspace(w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim,
                                               run.cap))
    run2.out = torch.zeros_like(run.out)
    run2.evicted = torch.zeros_like(run.evicted)
    for u in range(units):
        got = gpu_unit_state(run2, u)
        for a, b in zip(got, saved[u]):
            assert np.array_equal(a, b)
    assert fresh.seq_len.cpu().tolist() == [w.ctx + s1] * w.batch
    for i, s in enumerate(range(s1, w.steps)):
        run2.step(s)
        assert torch.equal(run2.out, outs[i]), s
        assert torch.equal(run2.evicted, evs[i]), s
    torch.cuda.synchronize()
    for u in range(units):
        for a, b in zip(gpu_unit_state(run2, u), final[u]):
            assert np.array_equal(a, b)
    assert se.status_word(run2.ws) == 0 and run.status() == 0


def test_h2o_restore_into_other_sequences_matches_oracle():
    w = _h2o_workload()
    run = H2ORun(w, keep_inputs=True)
    for s in range(4):
        run.step(s)
    ws = se.workspace(se.se_small_workspace())
    snap = _snapshot(run.state.kv, [2, 0], run.cap, ws)        # sequences 2 and 0
    # a two-sequence state: slot 0 <- sequence 2, slot 1 <- sequence 0
    w2 = synth.scaled(w, batch=2)
    fresh = _fresh_like(run.state.kv, 2, reverse=False)
    se.se_chain_restore(snap, run.cap, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                        fresh, ws)
    torch.cuda.synchronize()
    assert se.status_word(ws) == 0
    run2 = H2ORun.__new__(H2ORun)
    run2.__dict__.update(run.__dict__)
    run2.w, run2.B = w2, 2
    run2.state = se.H2OState(fresh, w.budget, w.recent)
    run2.ws = se.workspace(se.se_h2o_workspace(2, w.num_kv_heads, w.num_q_heads, w.head_dim,
                                               run.cap))
    perm = [2, 0]
    run2.inputs = dict(run.inputs)
    for key in ("q", "k_new", "v_new"):
        run2.inputs[key] = run.inputs[key][:, perm]
    run2.q, run2.k_new, run2.v_new = run.q[:, perm].contiguous(), run.k_new[:, perm].contiguous(), \
        run.v_new[:, perm].contiguous()
    run2.out = torch.zeros(2, w.num_q_heads, w.head_dim, dtype=run.out.dtype, device="cuda")
    run2.lse = torch.zeros(2, w.num_q_heads, dtype=torch.float32, device="cuda")
    run2.evicted = torch.zeros(2 * w.num_kv_heads, dtype=torch.int32, device="cuda")
    units = list(range(2 * w.num_kv_heads))
    for s in (4, 5):
        torch.cuda.synchronize()
        seq = fresh.seq_len.cpu().numpy()
        before = {u: gpu_unit_state(run2, u) + (int(seq[u // w.num_kv_heads]),) for u in units}
        run2.step(s)
        torch.cuda.synchronize()
        check_step(run2, s, units, before)
    assert se.status_word(run2.ws) == 0


def test_snapkv_decode_resumes_bit_exact():
    base = synth.workloads()["snapkv_32k"]
    w = synth.scaled(base, name="chain_snap", batch=2, groups=1, num_q_heads=8, num_kv_heads=2,
                     head_dim=128, ctx=3000, window=16, keep=512, steps=8)
    run = SnapKVRun(w)
    for s in range(3):
        run.step(s)
    ws = se.workspace(se.se_small_workspace())
    snap = _snapshot(run.cache, list(range(run.Bt)), run.seg_cap, ws)
    outs = []
    for s in range(3, w.steps):
        run.step(s)
        outs.append(run.out.clone())
    fresh = _fresh_like(run.cache, run.Bt)
    se.se_chain_restore(snap, run.seg_cap, torch.arange(run.Bt, dtype=torch.int32, device="cuda"),
                        fresh, ws)
    run.cache = fresh
    for i, s in enumerate(range(3, w.steps)):
        run.step(s)
        assert torch.equal(run.out, outs[i]), s
    torch.cuda.synchronize()
    assert se.status_word(ws) == 0 and run.status() == 0


def test_snapshot_of_another_shape_is_refused():
    w = _h2o_workload()
    run = H2ORun(w)
    ws = se.workspace(se.se_small_workspace())
    snap = _snapshot(run.state.kv, [0], run.cap, ws)
    before = run.state.kv.seg_len.clone()
    # restore with a smaller row count than the snapshot was written with
    se.se_chain_restore(snap, run.cap - 1, torch.tensor([1], dtype=torch.int32, device="cuda"),
                        run.state.kv, ws)
    torch.cuda.synchronize()
    assert se.status_word(ws) & 1                     # SE_DEV_BAD_INDEX
    assert torch.equal(run.state.kv.seg_len, before)
