"""The allocation-free decode entry point against the workspace one.

se_sparse_decode_noalloc exists for callers that cannot allocate device
memory (code inside another framework's memory pool, hot loops that must not
pay cudaMalloc's synchronisation, hosts that own every allocation): it keeps
its scratch in a fixed array inside the library.  Its results must match
se_sparse_decode on the same view, on two calls in a row (the second call
reuses the array the first one left behind).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from kv_cache_decode_quest_gb300 import binding, build, synth
from kv_cache_decode_quest_gb300.workloads import QuestRun
from tests.parity import TOL_BF16, TOL_F32, max_abs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_noalloc_matches_workspace_decode_twice(out_dtype):
    build.build()
    base = synth.workloads()["quest_32k"]
    w = synth.scaled(base, name="noalloc", batch=4, ctx=(3000, 1500, 4100, 700),
                     budget=(1024, synth.UNBOUNDED_BUDGET, 512, 256), steps=2)
    run = QuestRun(w, synth.quest_inputs(w), out_dtype=out_dtype)
    tol = TOL_F32 if out_dtype == 1 else TOL_BF16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(2):                      # two calls in a row, different queries
        run.append(s)
        run.select(s)
        run.decode(s)                        # the workspace entry point
        ref_out, ref_lse = run.out.clone(), run.lse.clone()
        out = torch.full_like(run.out, float("nan"))
        lse = torch.full_like(run.lse, float("nan"))
        binding.se_sparse_decode_noalloc(run.kv.k, run.kv.v, run.view, run.q[s], run.B, run.Hq,
                                         run.Hkv, run.D, run.scale, out, lse,
                                         out_dtype=out_dtype, status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert max_abs(out.double().cpu().numpy(), ref_out.double().cpu().numpy()) <= tol
        assert max_abs(lse.cpu().numpy(), ref_lse.cpu().numpy()) <= 1e-4
    assert run.status() == 0


def test_noalloc_rejects_a_batch_beyond_its_fixed_scratch():
    build.build()
    lib = binding.load()
    # 40000 units x 16 heads x 128 dims of fp32 partials cannot fit in 8 MiB
    # even with one piece per unit: rejected on the host, nothing launched.
    view = binding.ViewC(1 << 20, 1 << 20, 40000 * 4, 8)
    p = ctypes.c_void_p(1 << 20)
    rc = lib.se_sparse_decode_noalloc(p, p, 1000, ctypes.byref(view), p, 40000, 64, 4, 128, 0.1,
                                      0, p, None, None, None)
    assert rc == -5
    assert b"too small" in lib.se_status_str(rc)
    assert np.int32(rc) == -5
