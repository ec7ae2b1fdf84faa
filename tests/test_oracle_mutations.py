"""The oracle's pins catch plausible mistakes: each case plants one mistake in
a copy of an oracle function (a wrong sign, a dropped term, a wrong index, a
transposed operand, a wrong tie rule) and checks that a pin test fails."""
import numpy as np
import pytest

import oracle.attention as att
import oracle.h2o as h2o
import oracle.quest as quest
import oracle.snapkv as snap
import oracle.topk as topk
from tests import test_oracle_attention as T_att
from tests import test_oracle_h2o as T_h2o
from tests import test_oracle_quest as T_quest
from tests import test_oracle_snapkv as T_snap
from tests import test_oracle_topk as T_topk


def fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _bound_min(q_group, kmin, kmax):            # max replaced by min
    q = np.asarray(q_group, float)
    return np.minimum(q[:, None] * kmin[None], q[:, None] * kmax[None]).sum(axis=(0, 2))


def _bound_first_head(q_group, kmin, kmax):     # group sum dropped
    q = np.asarray(q_group, float)[:1]
    return np.maximum(q[:, None] * kmin[None], q[:, None] * kmax[None]).sum(axis=(0, 2))


def _bound_kmax_only(q_group, kmin, kmax):      # sign of q ignored
    q = np.asarray(q_group, float)
    return (q[:, None] * kmax[None]).sum(axis=(0, 2))


@pytest.mark.parametrize("bad", [_bound_min, _bound_first_head, _bound_kmax_only])
def test_quest_bound_mutations_are_caught(monkeypatch, bad):
    monkeypatch.setattr(T_quest, "quest_bound", bad)
    caught = fails(T_quest.test_hand_worked_bound) or \
        any(fails(T_quest.test_bound_dominates_every_key_of_its_page, s) for s in range(3))
    assert caught


def test_quest_select_not_forcing_last_page_is_caught(monkeypatch):
    def bad(U, k):
        return np.sort(topk.top_k(np.asarray(U, float), k))
    monkeypatch.setattr(T_quest, "quest_select", bad)
    assert fails(T_quest.test_selection_rules)


def test_topk_ties_to_higher_index_is_caught(monkeypatch):
    def bad(scores, k, index=None):
        s = np.asarray(scores, float)
        order = np.lexsort((-np.arange(len(s)), -s))
        return np.sort(order[:k])
    monkeypatch.setattr(T_topk, "top_k", bad)
    assert fails(T_topk.test_topk_ties_go_to_lower_index)


def test_attention_mutations_are_caught(monkeypatch):
    # softmax without the max shift is still exact; these are real mistakes:
    def no_scale(q, k, v, scale):
        return att.attend(q, k, v, 1.0)

    def transposed_values(q, k, v, scale):
        out, lse = att.attend(q, k, v, scale)
        return out[:, ::-1], lse

    def lse_missing_max(q, k, v, scale):
        out, lse = att.attend(q, k, v, scale)
        s = att.logits(q, k, scale)
        return out, lse - s.max(axis=1)

    for bad in (no_scale, transposed_values, lse_missing_max):
        monkeypatch.setattr(T_att, "attend", bad)
        assert any(fails(T_att.test_matches_torch_sdpa_float64, s) for s in range(3)) or \
            fails(T_att.test_two_tokens_closed_form)


def test_snapkv_non_causal_window_is_caught(monkeypatch):
    def bad(q_win, k, scale):
        q, k = np.asarray(q_win, float), np.asarray(k, float)
        A = np.zeros(k.shape[0])
        for i in range(q.shape[0]):
            s = scale * (q[i] @ k.T)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            A += (e / e.sum(axis=1, keepdims=True)).sum(axis=0)
        return A
    monkeypatch.setattr(T_snap, "window_scores", bad)
    assert fails(T_snap.test_hand_worked_two_rows) or fails(T_snap.test_matches_torch_causal_softmax, 0)


def test_snapkv_pool_off_by_one_is_caught(monkeypatch):
    def bad(a, kernel):
        a = np.asarray(a, float)
        r = kernel // 2
        return np.array([a[max(0, j - r):min(len(a), j + r)].max() for j in range(len(a))])
    monkeypatch.setattr(T_snap, "max_pool", bad)
    assert fails(T_snap.test_max_pool_matches_scipy_maximum_filter, 7)


def test_h2o_mutations_are_caught(monkeypatch):
    orig = h2o.h2o_step

    def evict_highest(st, q, kn, vn, new_pos, budget, recent, scale):
        neg = h2o.H2OState(st.pos, st.k, st.v, -st.score)
        new, out, lse, ev = orig(neg, -np.asarray(q), kn, vn, new_pos, budget, recent, scale)
        return new, out, lse, ev

    def no_update(st, q, kn, vn, new_pos, budget, recent, scale):
        new, out, lse, ev = orig(st, q, kn, vn, new_pos, budget, recent, scale)
        new.score = np.concatenate([st.score, [0.0]])[:len(new.score)]
        return new, out, lse, ev

    for bad in (evict_highest, no_update):
        monkeypatch.setattr(T_h2o, "h2o_step", bad)
        assert fails(T_h2o.test_hand_worked_step) or fails(T_h2o.test_mass_conservation_and_rules, 0)


def _widen_sign_extended(bits):                # sign-extended to 64 bits, upper half of a double
    u = np.asarray(bits, dtype=np.uint16).view(np.int16).astype(np.int64) << 48
    return u.view(np.float64)


def _widen_shift_15(bits):                     # one bit short of the upper half
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
    return u.view(np.float32).astype(np.float64)


def _widen_as_float16(bits):                   # the 16 bits viewed as IEEE half
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _widen_low_half(bits):                     # placed in the low half of binary32
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("bad", [_widen_sign_extended, _widen_shift_15, _widen_as_float16,
                                 _widen_low_half])
def test_widen_mutations_are_caught(monkeypatch, bad):
    from tests import test_oracle_bf16 as T_bf16
    monkeypatch.setattr(T_bf16, "widen", bad)
    caught = any(fails(T_bf16.test_explicit_bit_patterns, b, v) for b, v in T_bf16.CASES) or \
        fails(T_bf16.test_matches_torch_bfloat16_on_random_patterns)
    assert caught


def test_omnikv_mutations_are_caught(monkeypatch):
    import oracle.omnikv as om
    from tests import test_oracle_omnikv as T_om
    good = om.omnikv_layers

    def attends_filter_kv(qs, ks, vs, filters, budget, scale):     # the filter layer's K/V reused too
        res = good(qs, ks, vs, filters, budget, scale)
        out = []
        for layer, (pages, _, _) in enumerate(res):
            f = om.source_layer(layer, filters)
            tok = om.selected_tokens(pages, len(ks[0]))
            o, l = om.attend(qs[layer], np.asarray(ks[f])[tok], np.asarray(vs[f])[tok], scale)
            out.append((pages, o, l))
        return out

    def own_selection(qs, ks, vs, filters, budget, scale):         # no reuse
        return good(qs, ks, vs, tuple(range(len(qs))), budget, scale)

    def first_filter(qs, ks, vs, filters, budget, scale):          # always layer 0's decision
        return good(qs, ks, vs, (0,), budget, scale)

    for bad, pins in ((attends_filter_kv, [(T_om.test_full_budget_is_dense_attention_per_layer, 0)]),
                      (own_selection, [(T_om.test_reuse_takes_the_filter_layers_pages_not_the_layers_own,)]),
                      (first_filter, [(T_om.test_every_layer_a_filter_is_per_layer_quest,),
                                      (T_om.test_reuse_takes_the_filter_layers_pages_not_the_layers_own,)])):
        monkeypatch.setattr(T_om, "omnikv_layers", bad)
        assert any(fails(fn, *args) for fn, *args in pins), bad.__name__
    monkeypatch.setattr(T_om, "omnikv_layers", good)


def test_span_prune_mutations_are_caught(monkeypatch):
    import oracle.prune as pr
    from tests import test_oracle_prune as T_pr

    def pool_unclipped(A, L, s0, s1, keep, kernel):             # neighbours outside the span used
        A = np.asarray(A, float)
        s0 = max(0, min(int(s0), L))
        s1 = max(s0, min(int(s1), L))
        full = snap.max_pool(A, kernel)
        cand = topk.top_k(full[s0:s1], keep) + s0
        return np.concatenate([np.arange(s0), cand, np.arange(s1, L)]).astype(np.int64)

    def drops_tail(A, L, s0, s1, keep, kernel):                 # tokens after the span lost
        got = pr.span_keep_positions(A, L, s0, s1, keep, kernel)
        return got[got < max(0, min(int(s1), L))]

    for bad in (pool_unclipped, drops_tail):
        monkeypatch.setattr(T_pr, "span_keep_positions", bad)
        assert fails(T_pr.test_span_selection_matches_brute_force_on_small_cases) or \
            fails(T_pr.test_outside_positions_untouched_and_ascending), bad.__name__


def _bound_max_by_min(q_group, kmin, kmax):     # min over the group instead of max
    q = np.asarray(q_group, float)
    return np.maximum(q[:, None] * kmin[None], q[:, None] * kmax[None]).sum(axis=2).min(axis=0)


def _bound_max_of_products(q_group, kmin, kmax):  # max taken before the channel sum
    q = np.asarray(q_group, float)
    return np.maximum(q[:, None] * kmin[None], q[:, None] * kmax[None]).max(axis=0).sum(axis=1)


@pytest.mark.parametrize("bad", [_bound_max_by_min, _bound_max_of_products, quest.quest_bound])
def test_quest_bound_max_mutations_are_caught(monkeypatch, bad):
    monkeypatch.setattr(T_quest, "quest_bound_max", bad)
    caught = fails(T_quest.test_max_bound_hand_worked) or \
        fails(T_quest.test_max_bound_page_size_one_is_the_exact_max_logit) or \
        any(fails(T_quest.test_max_bound_dominates_every_heads_logit, s) for s in range(3))
    assert caught
