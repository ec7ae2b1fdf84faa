"""GPU parity: the H2O step through the C ABI against the oracle, teacher
forced (each checked step starts the oracle from the GPU's state), plus the
initial heavy-hitter/recent state; small and config-shaped cases, the
not-yet-full cache, and the full-size 64 x 16K workload on sampled steps."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import H2ORun
from tests.parity import TOL_BF16, TOL_F32, bf16_tensor_to_f64, max_abs

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_unit_state(run, u):
    c = run.state.kv
    off = int(c.seg_off[u])
    n = int(c.seg_len[u])
    return (c.pos[off:off + n].cpu().numpy().astype(np.int64),
            _u16(c.k[off:off + n]), _u16(c.v[off:off + n]),
            c.score[off:off + n].cpu().numpy().astype(np.float64))


def scores_close(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert np.all(np.abs(a - b) <= 1e-5 + 1e-4 * np.abs(b)), float(np.max(np.abs(a - b)))


def check_init(run, units):
    w, G = run.w, run.G
    for u in units:
        b, h = divmod(u, run.Hkv)
        pos, k, v, sc = gpu_unit_state(run, u)
        q = oracle.widen(run.inputs["q_win"][b][:, h * G:(h + 1) * G])
        K = oracle.widen(run.inputs["k"][b][h])
        A = oracle.window_scores(q, K, run.scale)
        ref = oracle.h2o_init(q, K, oracle.widen(run.inputs["v"][b][h]), w.budget, w.recent,
                              run.scale)
        order = np.argsort(pos)
        gp = pos[order]
        assert len(gp) == len(ref.pos)
        diff = set(gp.tolist()) ^ set(ref.pos.tolist())
        if diff:
            older = A[:w.ctx - w.recent]
            boundary = older[oracle.rank_order(older)[w.budget - w.recent - 1]]
            assert all(abs(A[p] - boundary) <= 1e-5 * abs(boundary) for p in diff), diff
        assert np.array_equal(k[order], run.inputs["k"][b][h][gp])
        scores_close(sc[order], A[gp])


def check_step(run, s, units, before):
    """Compare GPU step s (already run) against the oracle started from the
    GPU state `before` (captured before the step)."""
    w, G = run.w, run.G
    out = bf16_tensor_to_f64(run.out)
    ev = run.evicted.cpu().numpy()
    tol = TOL_F32 if run.out_dtype == 1 else TOL_BF16
    for u in units:
        b, h = divmod(u, run.Hkv)
        pos0, k0, v0, sc0, new_pos = before[u]
        st = oracle.H2OState(pos=pos0, k=oracle.widen(k0), v=oracle.widen(v0), score=sc0)
        q = oracle.widen(run.inputs["q"][s, b, h * G:(h + 1) * G])
        kn = oracle.widen(run.inputs["k_new"][s, b, h])
        vn = oracle.widen(run.inputs["v_new"][s, b, h])
        new, o_ref, l_ref, ev_ref = oracle.h2o_step(st, q, kn, vn, new_pos, w.budget, w.recent,
                                                    run.scale)
        err = max_abs(out[b, h * G:(h + 1) * G], o_ref)
        assert err <= tol, (s, u, err)
        # the scores after the update, for every token (before the eviction)
        p = np.exp(oracle.logits(q, np.vstack([st.k, kn[None]]), run.scale) - l_ref[:, None])
        upd = dict(zip(np.concatenate([pos0, [new_pos]]).tolist(),
                       (np.concatenate([sc0, [0.0]]) + p.sum(axis=0)).tolist()))
        if ev[u] != ev_ref:
            assert ev[u] >= 0 and ev_ref >= 0, (s, u, ev[u], ev_ref)
            assert abs(upd[int(ev[u])] - upd[ev_ref]) <= 1e-5 * abs(upd[ev_ref]), \
                (s, u, ev[u], ev_ref, upd[int(ev[u])], upd[ev_ref])
        pos1, k1, _, sc1 = gpu_unit_state(run, u)
        expect = set(upd) - ({int(ev[u])} if ev[u] >= 0 else set())
        assert set(pos1.tolist()) == expect
        scores_close(sc1, [upd[x] for x in pos1.tolist()])


def run_and_check(w, steps=None, units=None, out_dtype=0):
    run = H2ORun(w, keep_inputs=True, out_dtype=out_dtype)
    all_units = list(range(w.batch * w.num_kv_heads)) if units is None else units
    check_init(run, all_units)
    for s in range(w.steps):
        check = steps is None or s in steps
        if check:
            torch.cuda.synchronize()
            seq = run.state.kv.seq_len.cpu().numpy()
            before = {u: gpu_unit_state(run, u) + (int(seq[u // w.num_kv_heads]),)
                      for u in all_units}
        run.step(s)
        if check:
            torch.cuda.synchronize()
            check_step(run, s, all_units, before)
    torch.cuda.synchronize()
    assert run.status() == 0, run.status()
    return run


def test_small_h2o_steps():
    base = synth.workloads()["h2o_16k"]
    w = synth.scaled(base, name="h2o_small", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=64,
                     ctx=700, budget=200, recent=24, window=8, steps=12)
    run_and_check(w)


def test_config_shaped_h2o_steps_fp32():
    base = synth.workloads()["h2o_16k"]
    w = synth.scaled(base, name="h2o_mid", batch=3, ctx=3000, budget=512, recent=64, steps=16)
    run_and_check(w, out_dtype=1)


def test_large_budget_unstaged_eviction():
    """A budget of 12300 tokens: the segment (12301 slots) is too large for the
    shared-memory staging of the eviction, which then works on the cache in
    global memory."""
    base = synth.workloads()["h2o_16k"]
    w = synth.scaled(base, name="h2o_large", batch=1, num_q_heads=8, num_kv_heads=2, head_dim=64,
                     ctx=14000, budget=12300, recent=64, window=8, steps=4)
    run_and_check(w)


def test_cache_not_full_yet_then_evicting():
    base = synth.workloads()["h2o_16k"]
    w = synth.scaled(base, name="h2o_fill", batch=2, ctx=100, budget=110, recent=8, window=8,
                     steps=20)
    run = run_and_check(w)
    ev = run.evicted.cpu().numpy()
    assert np.all(ev >= 0)        # full after 10 steps: the last step evicts


@pytest.mark.slow
def test_full_size_h2o_16k_sampled():
    """64 x 16K context -> 4096 retained, all 256 steps on the GPU; the oracle
    checks steps 0, 128 and 255 on every fifth unit, teacher forced."""
    w = synth.workloads()["h2o_16k"]
    run_and_check(w, steps={0, 128, 255}, units=list(range(0, 256, 5)))
