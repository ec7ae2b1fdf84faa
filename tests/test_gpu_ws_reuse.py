"""One workspace reused across calls of different batch sizes.

The words a call needs at zero (split-K arrival counters, the one-kernel
step's queue words and counters) sit at fixed offsets of the workspace, so a
workspace sized for the largest call serves smaller and larger calls in any
order.  Batch 4 -> 16 -> 4 on the self-planned decode path (units <= 512),
each call checked against the oracle, the status word 0 after each; the same
for the allocation-free decode (whose fixed scratch every call shares) and for
the one-kernel Quest step."""
import pytest
import torch

from kv_cache_decode_quest_gb300 import binding as se
from kv_cache_decode_quest_gb300 import synth
from kv_cache_decode_quest_gb300.workloads import QuestRun
from tests.test_gpu_quest import check_step

pytestmark = pytest.mark.gpu
U32 = synth.UNBOUNDED_BUDGET


def _runs(mode, out_dtype):
    base = synth.workloads()["quest_32k"]
    shapes = [(4, (3000, 1500, 4100, 700), (1024, U32, 512, 256)),
              (16, tuple(500 + 211 * i for i in range(16)), tuple([U32, 256, 512, 1024] * 4)),
              (4, (2222, 4000, 90, 3333), (512, 2048, U32, 128))]
    runs = []
    for i, (B, ctx, bud) in enumerate(shapes):
        w = synth.scaled(base, name=f"ws_reuse_{i}", batch=B, ctx=ctx, budget=bud, steps=1)
        inputs = synth.quest_inputs(w)
        runs.append((QuestRun(w, inputs, out_dtype=out_dtype, mode=mode), inputs))
    return runs


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_decode_workspace_reused_across_batch_sizes(out_dtype):
    runs = _runs("fused", out_dtype)
    big = max(r.B * r.Hkv for r, _ in runs)
    ws = se.workspace(se.se_sparse_decode_workspace(big, runs[0][0].G, runs[0][0].D, 64))
    for r, inputs in runs:
        r.ws_dec = ws
        r.step(0)
        assert se.se_sync_status(ws) == 0
        check_step(r, inputs, 0)
        assert r.status() == 0


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_noalloc_decode_across_batch_sizes(out_dtype):
    runs = _runs("fused", out_dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r, inputs in runs:
        r.append_select(0)
        r.out.fill_(float("nan"))
        se.se_sparse_decode_noalloc(r.kv.k, r.kv.v, r.view, r.q[0], r.B, r.Hq, r.Hkv, r.D,
                                    r.scale, r.out, r.lse, out_dtype=out_dtype, status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_step(r, inputs, 0)
        assert r.status() == 0


def test_quest_step_workspace_reused_across_batch_sizes():
    runs = _runs("step", 1)
    r0 = runs[1][0]
    ws = se.workspace(se.se_quest_step_workspace(r0.B, r0.Hkv, r0.Hq, r0.D,
                                                 max(r.sel.shape[1] for r, _ in runs), 64))
    for r, inputs in runs:
        r.ws_step = ws
        r.step(0)
        assert se.se_sync_status(ws) == 0
        check_step(r, inputs, 0)
