"""The host ChainCacheIndex (se_chain_index_*): the longest stored logical
token prefix of a request wins, compared token by token; checked against a
brute-force search on random sessions with shared prefixes.  Host code only
(no GPU)."""
import numpy as np
import pytest

from kv_cache_decode_quest_gb300 import binding, build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load()


def test_longest_prefix_wins_and_erase():
    ix = binding.ChainIndex()
    ix.put([1, 2, 3, 4], 7)
    assert ix.match([1, 2, 3, 4, 5, 6]) == (7, 4)
    assert ix.match([1, 2, 3, 4]) == (7, 4)
    assert ix.match([1, 2, 3]) == (-1, 0)
    assert ix.match([1, 2, 9, 4, 5]) == (-1, 0)
    ix.put([1, 2, 3, 4, 5], 8)
    assert ix.match([1, 2, 3, 4, 5, 6]) == (8, 5)
    assert ix.match([1, 2, 3, 4, 9]) == (7, 4)
    ix.erase(8)
    assert ix.match([1, 2, 3, 4, 5, 6]) == (7, 4)
    ix.erase(8)                                   # absent: no error
    assert len(ix) == 1
    ix.put([9, 9], 7)                             # the id now stands for another prefix
    assert ix.match([1, 2, 3, 4]) == (-1, 0)
    assert ix.match([9, 9, 1]) == (7, 2)
    assert len(ix) == 1
    ix.close()


def test_empty_prefix_matches_everything_with_zero_tokens():
    ix = binding.ChainIndex()
    ix.put([], 3)
    assert ix.match([5, 6]) == (3, 0)
    assert ix.match([]) == (3, 0)
    ix.put([5], 4)
    assert ix.match([5, 6]) == (4, 1)


def test_random_sessions_against_brute_force():
    rng = np.random.default_rng(0)
    ix = binding.ChainIndex()
    stored = {}
    trunk = rng.integers(0, 50, size=300).astype(np.int32)
    for sid in range(60):
        cut = int(rng.integers(0, 300))
        tail = rng.integers(0, 3, size=int(rng.integers(0, 20))).astype(np.int32)
        t = np.concatenate([trunk[:cut], tail])
        stored[sid] = t
        ix.put(t, sid)
    for sid in rng.choice(60, size=10, replace=False):
        ix.erase(int(sid))
        del stored[int(sid)]
    assert len(ix) == len(stored)
    for _ in range(300):
        cut = int(rng.integers(0, 300))
        q = np.concatenate([trunk[:cut], rng.integers(0, 3, size=int(rng.integers(0, 25)))]).astype(np.int32)
        best = (-1, 0)
        for sid, t in stored.items():
            if len(t) <= len(q) and np.array_equal(q[:len(t)], t) and len(t) >= best[1]:
                if len(t) > best[1] or best[0] == -1:
                    best = (sid, len(t))
        got = ix.match(q)
        assert got[1] == best[1], (got, best)
        if best[0] != -1:
            assert np.array_equal(stored[got[0]], q[:got[1]])   # any session with that prefix
        else:
            assert got[0] == -1


def test_bad_arguments():
    lib = binding.load()
    assert lib.se_chain_index_put(None, None, 0, 1) == -1
    assert lib.se_chain_index_match(None, None, 0, None) == -1
    ix = binding.ChainIndex()
    assert lib.se_chain_index_put(ix._h, None, 3, 1) == -1      # tokens missing
    assert lib.se_chain_index_put(ix._h, None, 0, -2) == -1     # negative id
