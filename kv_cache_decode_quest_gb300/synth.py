"""Seeded synthetic inputs for the sparse-decode hot path.

This module is the one place both the CUDA path and the CPU oracle take their
inputs from.  It draws random numbers and lays them out; it holds none of the
method's arithmetic (no scores, no softmax, no selection).

Randomness: numpy's PCG64 bit generator, one independent sub-stream per
(workload, tensor, indices) label, keyed through ``numpy.random.SeedSequence``.
Normal variates are drawn in float32 and rounded to bfloat16 with
round-to-nearest-even; tensors are returned as raw bf16 bit patterns
(``numpy.uint16``) so that both sides see the exact same bytes.

The workloads stand in for the long-context agent traces that the SparseEngine
pages evaluate on (128K-token inputs, Qwen3-30B-A3B attention shape: 32 query
heads, 4 KV heads, head_dim 128; "SparseEngine 统一接入十五种稀疏注意力",
section "论文报告的吞吐量优势涵盖哪些条件").  Those traces are not available;
the shapes, distributions and length mixes below are the synthetic recipe.
"""
from __future__ import annotations

import dataclasses
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

PAGE_SIZE = 16


# ---------------------------------------------------------------------------
# random streams
# ---------------------------------------------------------------------------

def _label_words(labels) -> list[int]:
    words = []
    for lab in labels:
        if isinstance(lab, (int, np.integer)):
            words.append(int(lab) & 0xFFFFFFFF)
        else:
            words.append(zlib.crc32(str(lab).encode()) & 0xFFFFFFFF)
    return words


def stream(seed: int, *labels) -> np.random.Generator:
    """An independent PCG64 generator for the given seed and label path."""
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF] + _label_words(labels))
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_bf16(seed: int, label: str, shape, lead: int = 0,
                channel_scale: np.ndarray | None = None) -> np.ndarray:
    """N(0,1) bf16 bits of ``shape``.

    The first ``lead`` axes index independent sub-streams (one per index tuple,
    drawn in parallel); the rest is drawn from that sub-stream in C order.
    ``channel_scale`` (broadcast against the sub-array, typically [..., D])
    multiplies the float32 draw before rounding, which is how outlier channels
    are planted.  The per-sub-stream scale is ``channel_scale[idx]`` when it
    has the ``lead`` axes, else the same array for all.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    lead_shape = shape[:lead]
    sub_shape = shape[lead:]
    idxs = list(np.ndindex(*lead_shape)) if lead else [()]

    def one(idx):
        g = stream(seed, label, *idx)
        x = g.standard_normal(sub_shape, dtype=np.float32)
        if channel_scale is not None:
            cs = channel_scale[idx] if (lead and channel_scale.ndim > len(sub_shape)) else channel_scale
            x *= cs
        out[idx] = f32_to_bf16_bits(x)

    if len(idxs) == 1:
        one(idxs[0])
    else:
        with ThreadPoolExecutor(_workers()) as ex:
            list(ex.map(one, idxs))
    return out


def outlier_scale(seed: int, label: str, lead_shape, head_dim: int,
                  n_outliers: int = 4, factor: float = 8.0) -> np.ndarray:
    """Per-channel multipliers: ``n_outliers`` distinct channels (chosen per
    index of ``lead_shape``, e.g. per (sequence, KV head)) get ``factor``."""
    lead_shape = tuple(lead_shape)
    sc = np.ones(lead_shape + (head_dim,), dtype=np.float32)
    for idx in np.ndindex(*lead_shape):
        g = stream(seed, label, *idx)
        ch = g.choice(head_dim, size=n_outliers, replace=False)
        sc[idx + (slice(None),)][ch] = factor
    return sc


def block_table(seed: int, label: str, pages_per_seq: np.ndarray, num_pages: int | None = None,
                max_pages: int | None = None) -> tuple[np.ndarray, int]:
    """Block table mapping each sequence's logical pages to distinct physical
    pages, in a seeded random order (so that a reader must follow the table).
    Unused entries are -1.  Returns (table [B][max_pages] int32, num_pages)."""
    pages_per_seq = np.asarray(pages_per_seq, dtype=np.int64)
    total = int(pages_per_seq.sum())
    if num_pages is None:
        num_pages = total
    if max_pages is None:
        max_pages = int(pages_per_seq.max()) if len(pages_per_seq) else 0
    perm = stream(seed, label).permutation(num_pages)[:total].astype(np.int32)
    bt = np.full((len(pages_per_seq), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class QuestWorkload:
    """Paged-KV decode with Quest page selection."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: tuple            # per-sequence prefill context length
    budget: tuple         # per-sequence token budget (>= context means all pages)
    steps: int            # decode steps, one appended token each
    outliers: bool        # 4 outlier channels per (sequence, KV head), scaled x8
    max_splits: int = 64
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class SnapKVWorkload:
    """SnapKV compaction at the end of prefill, then decode over the result."""
    name: str
    batch: int            # requests per compaction batch
    groups: int           # independently seeded compaction batches concatenated for decode
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: int              # prefill length L
    window: int           # observation window W (last W query rows)
    pool_kernel: int
    keep: int             # per-KV-head top-k of the prefix
    steps: int            # decode steps after compaction
    max_splits: int = 64
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class H2OWorkload:
    """H2O heavy-hitter + recent-window decode."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: int              # initial context
    budget: int           # retained tokens (heavy hitters + recent)
    recent: int
    window: int           # query rows whose attention seeds the initial scores
    steps: int
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class OmniKVWorkload:
    """Multi-layer Quest decode with cross-layer selection reuse: the filter
    layers select pages with Quest; every other layer attends through the
    selection of the latest filter layer before it.  Every layer has its own
    K, V and queries (drawn like a QuestWorkload of the same shape), and all
    layers share one paging of the cache."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: tuple
    budget: tuple
    steps: int
    outliers: bool
    layers: int
    filters: tuple        # filter layers, sorted, containing 0
    max_splits: int = 64
    seed: int = 0

    def layer(self, layer: int) -> QuestWorkload:
        """Layer ``layer``'s tensors as a QuestWorkload (its own sub-streams)."""
        return QuestWorkload(f"{self.name}/L{layer}", self.batch, self.num_q_heads,
                             self.num_kv_heads, self.head_dim, self.ctx, self.budget, self.steps,
                             self.outliers, self.max_splits, self.seed)


UNBOUNDED_BUDGET = 2 ** 31 - 1


def _ragged_ctx(seed, batch, lo, hi):
    g = stream(seed, "ragged_ctx")
    return tuple(int(x) for x in g.integers(lo, hi + 1, size=batch))


def workloads(seed: int = 0) -> dict:
    """The synthetic workloads, keyed by name: the five of the hot path and the
    multi-layer cross-layer reuse workload."""
    ragged = _ragged_ctx(seed, 8, 65536, 131072)
    return {
        "tiny_quest": QuestWorkload(
            "tiny_quest", batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
            ctx=(2048,), budget=(128,), steps=1, outliers=False, seed=seed),
        "quest_32k": QuestWorkload(
            "quest_32k", batch=16, num_q_heads=32, num_kv_heads=4, head_dim=128,
            ctx=(32768,) * 16, budget=(2048,) * 16, steps=64, outliers=True, seed=seed),
        "snapkv_32k": SnapKVWorkload(
            "snapkv_32k", batch=8, groups=8, num_q_heads=32, num_kv_heads=4, head_dim=128,
            ctx=32768, window=32, pool_kernel=7, keep=4096, steps=64, seed=seed),
        "h2o_16k": H2OWorkload(
            "h2o_16k", batch=64, num_q_heads=32, num_kv_heads=4, head_dim=128,
            ctx=16384, budget=4096, recent=256, window=32, steps=256, seed=seed),
        "omnikv_32k": OmniKVWorkload(
            "omnikv_32k", batch=16, num_q_heads=32, num_kv_heads=4, head_dim=128,
            ctx=(32768,) * 16, budget=(2048,) * 16, steps=16, outliers=True, layers=4,
            filters=(0,), seed=seed),
        "ragged_quest_128k": QuestWorkload(
            "ragged_quest_128k", batch=8, num_q_heads=32, num_kv_heads=4, head_dim=128,
            ctx=ragged,
            budget=tuple(UNBOUNDED_BUDGET if b % 2 == 0 else 4096 for b in range(8)),
            steps=32, outliers=True, max_splits=64, seed=seed),
    }


# ---------------------------------------------------------------------------
# tensor sets
# ---------------------------------------------------------------------------

def quest_sequence(w: QuestWorkload, b: int, tag: str = "") -> tuple:
    """Logical k, v of sequence b: [Hkv][ctx_b + steps][D] bf16 bits (prefill,
    then the appended tokens of each step)."""
    Hkv, D, S = w.num_kv_heads, w.head_dim, w.steps
    label = w.name + tag
    T = w.ctx[b] + S
    cs = None
    if w.outliers:
        cs = outlier_scale(w.seed, label + "/outliers", (w.batch, Hkv), D)[b][:, None, :]
    k = normal_bf16(w.seed, f"{label}/k/{b}", (Hkv, T, D), lead=1, channel_scale=cs)
    v = normal_bf16(w.seed, f"{label}/v/{b}", (Hkv, T, D), lead=1)
    return k, v


def quest_queries(w: QuestWorkload, tag: str = "") -> np.ndarray:
    """q [steps][B][Hq][D] bf16 bits."""
    return normal_bf16(w.seed, w.name + tag + "/q", (w.steps, w.batch, w.num_q_heads, w.head_dim),
                       lead=2)


def quest_inputs(w: QuestWorkload, tag: str = "") -> dict:
    """Logical tensors of a Quest decode run (bf16 bits, uint16).

    k, v:   per sequence, [Hkv][ctx_b + steps][D] (prefill then the appended tokens)
    q:      [steps][B][Hq][D]
    The appended token of step s for sequence b is row ctx_b + s.
    """
    ks, vs = [], []
    for b in range(w.batch):
        k, v = quest_sequence(w, b, tag)
        ks.append(k)
        vs.append(v)
    return {"k": ks, "v": vs, "q": quest_queries(w, tag)}


def snapkv_inputs(w: SnapKVWorkload, group: int) -> dict:
    """One compaction batch: prefill k, v [B][Hkv][L][D], window queries
    q_win [B][W][Hq][D] (query rows of positions L-W .. L-1)."""
    B, Hq, Hkv, D, L, W = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.ctx, w.window
    label = f"{w.name}/g{group}"
    k = normal_bf16(w.seed, label + "/k", (B, Hkv, L, D), lead=2)
    v = normal_bf16(w.seed, label + "/v", (B, Hkv, L, D), lead=2)
    q_win = normal_bf16(w.seed, label + "/q_win", (B, W, Hq, D), lead=1)
    return {"k": k, "v": v, "q_win": q_win}


def snapkv_decode_inputs(w: SnapKVWorkload) -> dict:
    """Decode-phase tensors for the concatenated batch (groups * batch requests):
    q [steps][Bt][Hq][D], k_new/v_new [steps][Bt][Hkv][D]."""
    Bt = w.batch * w.groups
    S, Hq, Hkv, D = w.steps, w.num_q_heads, w.num_kv_heads, w.head_dim
    q = normal_bf16(w.seed, w.name + "/dec/q", (S, Bt, Hq, D), lead=1)
    kn = normal_bf16(w.seed, w.name + "/dec/k", (S, Bt, Hkv, D), lead=1)
    vn = normal_bf16(w.seed, w.name + "/dec/v", (S, Bt, Hkv, D), lead=1)
    return {"q": q, "k_new": kn, "v_new": vn}


def h2o_inputs(w: H2OWorkload) -> dict:
    """Prefill k, v [B][Hkv][ctx][D], seeding window queries q_win [B][W][Hq][D],
    decode q [steps][B][Hq][D], k_new/v_new [steps][B][Hkv][D]."""
    B, Hq, Hkv, D, L, W, S = (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                              w.ctx, w.window, w.steps)
    return {
        "k": normal_bf16(w.seed, w.name + "/k", (B, Hkv, L, D), lead=2),
        "v": normal_bf16(w.seed, w.name + "/v", (B, Hkv, L, D), lead=2),
        "q_win": normal_bf16(w.seed, w.name + "/q_win", (B, W, Hq, D), lead=1),
        "q": normal_bf16(w.seed, w.name + "/dec/q", (S, B, Hq, D), lead=1),
        "k_new": normal_bf16(w.seed, w.name + "/dec/k", (S, B, Hkv, D), lead=1),
        "v_new": normal_bf16(w.seed, w.name + "/dec/v", (S, B, Hkv, D), lead=1),
    }


def scaled(w, **changes):
    """A copy of workload ``w`` with some fields replaced (smaller test sizes)."""
    return dataclasses.replace(w, **changes)


def omnikv_inputs(w: OmniKVWorkload) -> list:
    """Per layer, the tensors of ``quest_inputs`` for that layer's sub-streams."""
    return [quest_inputs(w.layer(layer)) for layer in range(w.layers)]
