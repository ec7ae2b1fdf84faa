"""The CUDA path on the golden fixtures (explicit small inputs, expected values
written from the oracle): Quest selection + decode, SnapKV compaction, one
H2O step."""
import json
import math
import os

import numpy as np
import pytest
import torch

from kv_cache_decode_quest_gb300 import binding as se
from kv_cache_decode_quest_gb300 import synth
from tests.parity import TOL_BF16, max_abs

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        return json.load(f)


def bf16(x):
    bits = synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def test_quest_golden():
    c = load("quest_tiny")
    D, G, T = c["head_dim"], c["group"], c["ctx"]
    k, v = np.asarray(c["k"]), np.asarray(c["v"])
    n_pages = -(-T // 16)
    K = np.zeros((n_pages, 1, 16, D), dtype=np.float32)
    V = np.zeros_like(K)
    for t in range(T):
        K[t // 16, 0, t % 16], V[t // 16, 0, t % 16] = k[t], v[t]
    kv = se.PagedKV(bf16(K), bf16(V), torch.zeros(1, n_pages, 1, 2, D, dtype=torch.bfloat16,
                                                   device="cuda"),
                    torch.arange(n_pages, dtype=torch.int32, device="cuda")[None].contiguous(),
                    torch.tensor([T], dtype=torch.int32, device="cuda"))
    ws = se.workspace(se.se_small_workspace())
    se.se_page_meta_build(kv, 1, ws)
    q = bf16(np.asarray(c["q"])[None])
    sel = torch.zeros(1, n_pages, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(1, dtype=torch.int32, device="cuda")
    view = se.View.empty(1, n_pages)
    wsq = se.workspace(se.se_quest_select_workspace(1, 1, n_pages))
    se.se_quest_select(kv, q, 1, G, torch.tensor([c["budget"]], dtype=torch.int32, device="cuda"),
                       sel, nsel, view, wsq)
    out = torch.zeros(1, G, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, G, dtype=torch.float32, device="cuda")
    wsd = se.workspace(se.se_sparse_decode_workspace(1, G, D))
    se.se_sparse_decode(kv.k, kv.v, view, q, 1, G, 1, D, 1 / math.sqrt(D), out, lse, wsd)
    torch.cuda.synchronize()
    e = c["expected"]
    assert sel[0, :int(nsel[0])].tolist() == e["pages"]
    assert max_abs(out[0].double().cpu().numpy(), e["out"]) <= TOL_BF16
    assert max_abs(lse[0].cpu().numpy(), e["lse"]) <= 1e-3
    assert se.status_word(ws) | se.status_word(wsq) | se.status_word(wsd) == 0


def test_snapkv_golden():
    c = load("snapkv_tiny")
    D, G, L, W = c["head_dim"], c["group"], c["ctx"], c["window"]
    k, v = np.asarray(c["k"]), np.asarray(c["v"])
    n_pages = -(-L // 16)
    K = np.zeros((n_pages, 1, 16, D), dtype=np.float32)
    V = np.zeros_like(K)
    for t in range(L):
        K[t // 16, 0, t % 16], V[t // 16, 0, t % 16] = k[t], v[t]
    pre = se.PagedKV(bf16(K), bf16(V), torch.zeros(1, dtype=torch.bfloat16, device="cuda"),
                     torch.arange(n_pages, dtype=torch.int32, device="cuda")[None].contiguous(),
                     torch.tensor([L], dtype=torch.int32, device="cuda"))
    out = se.VarlenKV.empty(1, 1, L, D, with_score=True)
    ws = se.workspace(se.se_snapkv_workspace(1, 1, G, W, L))
    se.se_snapkv_compact(pre, bf16(np.asarray(c["q_win"])[None]), 1, G, W, c["pool"], c["keep"], W,
                         1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    e = c["expected"]
    n = int(out.seg_len[0])
    pos = out.pos[:n].cpu().numpy()
    assert pos.tolist() == e["kept"]
    A = np.asarray(e["A"])
    got = out.score[:n].cpu().numpy()
    assert np.all(np.abs(got - A[pos]) <= 1e-5 + 1e-4 * np.abs(A[pos]))
    assert se.status_word(ws) == 0


def test_h2o_golden():
    c = load("h2o_tiny")
    D, G, budget, recent = c["head_dim"], c["group"], c["budget"], c["recent"]
    n = len(c["pos"])
    kv = se.VarlenKV.empty(1, 1, budget + 1, D, with_score=True)
    kv.k[:n] = bf16(np.asarray(c["k"]))
    kv.v[:n] = bf16(np.asarray(c["v"]))
    kv.pos[:n] = torch.tensor(c["pos"], dtype=torch.int32)
    kv.score[:n] = torch.tensor(c["score"], dtype=torch.float32)
    kv.seg_len[0] = n
    kv.seq_len[0] = c["new_pos"]
    st = se.H2OState(kv, budget, recent)
    out = torch.zeros(1, G, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, G, dtype=torch.float32, device="cuda")
    ev = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = se.workspace(se.se_h2o_workspace(1, 1, G, D, budget + 1))
    se.se_h2o_step(st, bf16(np.asarray(c["q"])[None]), bf16(np.asarray(c["k_new"])[None, None]),
                   bf16(np.asarray(c["v_new"])[None, None]), 1, G, 1 / math.sqrt(D), out, lse, ev, ws)
    torch.cuda.synchronize()
    e = c["expected"]
    assert int(ev[0]) == e["evicted"]
    assert max_abs(out[0].double().cpu().numpy(), e["out"]) <= TOL_BF16
    m = int(kv.seg_len[0])
    pos = kv.pos[:m].cpu().numpy()
    order = np.argsort(pos)
    assert pos[order].tolist() == e["pos_after"]
    sc = kv.score[:m].cpu().numpy()[order]
    assert np.all(np.abs(sc - e["score_after"]) <= 1e-5 + 1e-4 * np.abs(e["score_after"]))
    assert se.status_word(ws) == 0
