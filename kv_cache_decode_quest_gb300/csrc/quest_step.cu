// One Quest decode step in one persistent kernel: the new token's append, the
// page scoring, the per-KV-head top-k and the split-K decode over the selected
// pages.  Same results as se_quest_select_append followed by se_sparse_decode.
//
// Quest picks pages by the query's upper-bound score against each page's key
// min/max summary while the whole history stays resident (tokendh.com article on
// SparseEngine, section "历史太长,会撑爆什么"); the attention then reads only the
// rows the view exposes ("SparseEngine：稀疏优先推理引擎", section "方法 / 关键模块").
//
// Why one kernel: the step is two HBM streams (the page summaries, then the
// selected K/V rows) separated by a short, latency-bound top-k per unit.  As
// separate launches the two streams never overlap and every top-k sits on the
// critical path.  Here the step is a queue of work items taken in order from
// one global counter by persistent CTAs:
//   score tile (sequence b, a range of its candidate pages, all KV heads)
//   top-k      (unit u = (b, h)): waits until every score tile of b is done
//   decode     (a piece of unit u): waits until the top-k of u is done
// The queue is laid out in rounds r = 0, 1, ...: the score tiles of sequence r,
// then the top-k items of sequence r - lag_topk, then the decode pieces of
// sequence r - lag_dec (lag_dec >= lag_topk >= 0), so every item depends only on
// items before it.  A CTA takes items in increasing order and a taken item is
// held by a running CTA, so the earliest unfinished item always has its inputs
// and can finish: the waits cannot deadlock, whatever the grid or residency.
// Every wait is bounded (1 s, or at once when another CTA has given up); a CTA
// that gives up records SE_DEV_TIMEOUT and raises a global abort word that the
// others poll.
//
// CTA layout (160 threads): warp 4 is the producer; it takes the items, publishes
// each one to the consumers through a 4-slot descriptor ring (mbarriers), and
// streams the item's data into one shared-memory stage ring: 1-D bulk copies of
// page summaries for a score tile, 2-D TMA boxes of K and V chunks for a decode
// piece.  Warps 0-3 consume: stage s is handled by warp (stage sequence % 4).
// Score tiles turn summaries into order-preserving keys in global memory; the
// top-k runs on the four consumer warps (10-bit radix threshold, ballot emit)
// and writes the view and the new token's row; decode pieces run the mma.sync
// decode of decode_core.cuh with its last-piece LSE merge.
//
// The last CTA to finish resets the queue counters and commits ctx_len + 1 of
// every sequence whose token was appended, after every CTA has read the old
// lengths.
#include <algorithm>

#include "append.cuh"
#include "common.cuh"
#include "decode_core.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kItemSlots = 4;
constexpr int kDigit = 10, kStepBins = 1 << kDigit;   // 10-bit radix digits: 8 bins per consumer thread
constexpr int kCThreads = kConsumerWarps * 32;

enum : int { kItemScore = 0, kItemTopk = 1, kItemDecode = 2, kItemEnd = 3, kItemFold = 4 };

// score: a0..a1 = candidate pages; decode: a0..a1 = chunks, a2 = partial slot
// (-1: the piece is the whole unit), a3 = the unit's first slot, a4 = its pieces
struct StepItem {
    int type, b, h, a0, a1, a2, a3, a4;
};

struct StepParams {
    se_paged_kv kv;
    const uint16_t* q;
    int Hq, G, batch;
    const int32_t* budget;
    const uint4* k_new;                 // null: no append
    const uint4* v_new;
    int32_t* sel_pages;
    int32_t* n_sel;
    se_view view;
    float scale, scale_log2;
    void* out;
    int out_f32;
    float* lse_out;
    uint32_t* keys;                     // [units][max_pages_per_seq]
    float* coef;                        // [batch][H][2][D]: Q- then Q+ per KV head
    int* sync;                          // [0] item counter, [1] CTAs finished, [2] abort
    int* seq_folded;                    // [batch] coefficients written
    int* seq_scored;                    // [batch] score tiles finished
    int* unit_ready;                    // [units] top-k done
    int* counters;                      // [units] decode pieces finished
    float* o_part;                      // [units * max_splits][G][D]
    float* lse_part;                    // [units * max_splits][G]
    int tile_pages, piece_chunks, max_splits, lag_topk, lag_dec, rounds;
    int64_t total_rows;
    // dynamic shared memory offsets (bytes from the 1024-aligned base)
    int off_coef, off_union, off_sinfo, off_rstart;
    int* status;
};

template <int D>
struct StepShape {
    static constexpr int kStageBytes = DecShape<D, 1>::kStageBytes;   // 8 KB at D = 128
    static constexpr int kStages = D == 64 ? 24 : 12;                  // 96 KB ring
    static constexpr int kSumBytes = 2 * D * 2;                        // one (page, head) summary
    static constexpr int kSumsPerStage = kStageBytes / kSumBytes;      // 16
    static_assert(kStages % kConsumerWarps == 0, "stage ownership needs kStages % 4 == 0");
    // ring, full/empty, item full/empty, stage counts, items, misc ints
    static constexpr int kFixed = kStages * kStageBytes + kStages * 16 + kItemSlots * 16 +
                                  kStages * 4 + kItemSlots * (int)sizeof(StepItem) + 64;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait for *flag >= target (acquire).  False on timeout, on this CTA's
// abort, or when another CTA raised the global abort word.
__device__ bool wait_geq(const int* flagp, int target, volatile int* abort_flag, const int* gabort) {
    if (ld_acquire(flagp) >= target) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        __nanosleep(100);
        if (ld_acquire(flagp) >= target) return true;
        if (*abort_flag || *reinterpret_cast<const volatile int*>(gabort)) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// This CTA gives up: results are invalid, the kernel drains and ends.
__device__ __forceinline__ void give_up(const StepParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    flag(p.status, SE_DEV_TIMEOUT);
    atomicExch(p.sync + 2, 1);
}

// Per-sequence plan values, the same in every CTA: held = clamped ctx_len,
// ctx = held + 1 when the new token fits, n pages, k pages of budget.
struct SeqPlan {
    int held, ctx, n, k;
    int tiles, chunks, tokens, pieces;
};
__device__ SeqPlan seq_plan(const StepParams& p, int b, bool report) {
    SeqPlan s;
    const int cap = p.kv.max_pages_per_seq * kPage;
    int held = p.kv.ctx_len[b];
    if (held < 0 || held > cap) {
        if (report) flag(p.status, SE_DEV_BAD_LENGTH);
        held = held < 0 ? 0 : cap;
    }
    const bool pending = p.k_new != nullptr;
    if (pending && held >= cap && report) flag(p.status, SE_DEV_CAPACITY);
    s.held = held;
    s.ctx = (pending && held < cap) ? held + 1 : held;
    s.n = (s.ctx + kPage - 1) / kPage;
    const int bud = p.budget[b];
    s.k = max(1, (bud < 0 ? 0 : bud) / kPage);
    if (s.n <= s.k) {
        s.tiles = 0;
        s.chunks = s.n;
        s.tokens = s.ctx;
    } else {
        s.tiles = (s.n - 1 + p.tile_pages - 1) / p.tile_pages;
        s.chunks = s.k;
        s.tokens = kPage * (s.k - 1) + (s.ctx - kPage * (s.n - 1));
    }
    s.pieces = max(1, min(p.max_splits, (s.chunks + p.piece_chunks - 1) / p.piece_chunks));
    return s;
}

// Inclusive scan over the 128 consumer threads; tmp holds 4 ints.
__device__ __forceinline__ int scan128(int v, int* tmp, int warp, int lane) {
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    consumer_bar();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += tmp[i];
    consumer_bar();
    return x + before;
}

// Threshold of the top K of m order-preserving keys in shared memory, on the
// 128 consumer threads: bits above the highest bit in which the largest and
// smallest key differ are common to all keys, so the radix digits start
// there (10-bit digits: the histogram stays small beside the stage ring), and
// a pass ends the search when the boundary digit is kept whole.  On
// return: keys above *T (under *mask) are kept, and so are the first *need keys
// equal to *T.
__device__ void step_threshold(const uint32_t* sk, int m, int K, int* hist, int* tmp,
                               uint32_t* red, int* sel, uint32_t* T, uint32_t* mask, int* need,
                               int warp, int lane) {
    const int ctid = warp * 32 + lane;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int i = ctid; i < m; i += kCThreads) {
        const uint32_t k = sk[i];
        lo = min(lo, k);
        hi = max(hi, k);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        red[warp] = lo;
        red[4 + warp] = hi;
    }
    consumer_bar();
    lo = min(min(red[0], red[1]), min(red[2], red[3]));
    hi = max(max(red[4], red[5]), max(red[6], red[7]));
    const uint32_t diff = lo ^ hi;
    if (diff == 0u) {                                     // every key is equal
        *T = hi;
        *mask = 0xffffffffu;
        *need = K;
        return;
    }
    const int top = 31 - __clz(diff);                     // highest differing bit
    uint32_t msk = top == 31 ? 0u : ~((2u << top) - 1u);
    uint32_t prefix = hi & msk;
    int remaining = K;
    int low = top + 1;                                    // bits [low, 32) are decided
    constexpr int kPer = kStepBins / kCThreads;           // 8 bins per thread
    while (low > 0) {
        // thread t owns bins 1023 - 8t .. 1016 - 8t (descending)
        const int w = min(kDigit, low), shift = low - w;
        const uint32_t dm = (1u << w) - 1u;
#pragma unroll
        for (int j = 0; j < kPer; ++j) hist[ctid * kPer + j] = 0;
        consumer_bar();
        for (int i = ctid; i < m; i += kCThreads) {
            const uint32_t k = sk[i];
            if ((k & msk) == prefix) atomicAdd(&hist[(k >> shift) & dm], 1);
        }
        consumer_bar();
        int vv[kPer], v = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            vv[j] = hist[kStepBins - 1 - (ctid * kPer + j)];
            v += vv[j];
        }
        int run = scan128(v, tmp, warp, lane) - v;        // digits above this thread's
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (run < remaining && run + vv[j] >= remaining) {
                sel[0] = kStepBins - 1 - (ctid * kPer + j);
                sel[1] = run;
                sel[2] = vv[j];
            }
            run += vv[j];
        }
        consumer_bar();
        prefix |= static_cast<uint32_t>(sel[0]) << shift;
        msk |= dm << shift;
        remaining -= sel[1];
        low = shift;
        const bool whole_bin = sel[2] == remaining;
        consumer_bar();                                   // sel is rewritten by the next pass
        if (whole_bin) break;
    }
    *T = prefix;
    *mask = msk;
    *need = remaining;
}

// Top-k item of unit u = (b, h) on the consumer warps: exact top-(k-1) of the
// candidate pages 0..n-2 by (score desc, page asc), emitted in page order, plus
// the last page (always selected, never scored); the view chunk of a selected
// page is its physical page of this KV head.  With the append, head h's new
// row goes in first (its loads are issued before the selection, its stores
// after it).  `area`: the union area of shared memory.
__device__ void step_topk(const StepParams& p, int b, int h, const SeqPlan& s, uint8_t* area,
                          int warp, int lane) {
    const int ctid = warp * 32 + lane;
    const se_paged_kv& kv = p.kv;
    const int H = kv.num_kv_heads, stride = kv.max_pages_per_seq;
    const int u = b * H + h;
    int* hist = reinterpret_cast<int*>(area);                    // [2048]
    int* small = hist + kStepBins;                               // 64 ints
    int* tmp = small;                                            // [4]
    uint32_t* red = reinterpret_cast<uint32_t*>(small + 4);      // [8]
    int* sel = small + 12;                                       // [4]
    int* wgt = small + 16;                                       // [4]
    int* weq = small + 20;                                       // [4]
    uint32_t* skeys = reinterpret_cast<uint32_t*>(small + 64);   // [stride]
    const bool room = p.k_new != nullptr && s.ctx == s.held + 1;
    const int segs = kv.head_dim / 8;
    AppendRegs ar;
    if (room && ctid < segs) append_load(kv, b, h, s.held, p.k_new, p.v_new, ctid, ar);
    const int32_t* btr = kv.block_table + (int64_t)b * stride;
    int phys_new = -1;
    if (room) phys_new = btr[s.held / kPage];
    const int n = s.n, k = s.k, m = n - 1;
    if (n > k) {
        // stage the candidate keys (written by other CTAs: read through L2)
        const uint32_t* keys = p.keys + (int64_t)u * stride;
        constexpr int kU = 8;
        for (int base = ctid; base < m; base += kCThreads * kU) {
            uint32_t kv2[kU];
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int i = base + j * kCThreads;
                kv2[j] = i < m ? __ldcg(keys + i) : 0u;
            }
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int i = base + j * kCThreads;
                if (i < m) skeys[i] = kv2[j];
            }
        }
        consumer_bar();
    }
    int32_t* selp = p.sel_pages + (int64_t)u * stride;
    int32_t* crow = p.view.chunk_row + (int64_t)u * p.view.max_chunks;
    // the view chunk of selected page `page`: its physical page of head h
    auto chunk_of = [&](int page) {
        const int phys = btr[page];
        if (phys >= 0 && phys < kv.num_pages) return (phys * H + h) * kPage;
        flag(p.status, SE_DEV_BAD_INDEX);
        return -1;
    };
    if (n <= k) {
        for (int c = ctid; c < n; c += kCThreads) {
            selp[c] = c;
            crow[c] = chunk_of(c);
        }
        if (ctid == 0) {
            p.n_sel[u] = n;
            p.view.n_tokens[u] = s.tokens;
        }
    } else {
        const int K = k - 1;
        if (K > 0) {
            int need_eq = 0;
            uint32_t T = 0, msk = 0;
            step_threshold(skeys, m, K, hist, tmp, red, sel, &T, &msk, &need_eq, warp, lane);
            // pages in ascending order: warp w owns a contiguous range read with
            // a lane stride; ballots rank the kept pages inside the warp and a
            // scan over the four warps places each warp's run
            const int chunk = ((m + kConsumerWarps - 1) / kConsumerWarps + 31) & ~31;
            const int c0 = min(m, warp * chunk), c1 = min(m, c0 + chunk);
            int gt = 0, eq = 0;
            for (int i = c0 + lane; i < c1; i += 32) {
                const uint32_t kk = skeys[i] & msk;
                gt += kk > T;
                eq += kk == T;
            }
            gt = __reduce_add_sync(0xffffffffu, gt);
            eq = __reduce_add_sync(0xffffffffu, eq);
            if (lane == 0) {
                wgt[warp] = gt;
                weq[warp] = eq;
            }
            consumer_bar();
            int eq_seen = 0, out = 0;
            for (int w = 0; w < warp; ++w) {
                const int take_w = max(0, min(weq[w], need_eq - eq_seen));
                out += wgt[w] + take_w;
                eq_seen += weq[w];
            }
            const uint32_t lt = (1u << lane) - 1u;
            for (int i0 = c0; i0 < c1; i0 += 32) {
                const int i = i0 + lane;
                const uint32_t kk = i < c1 ? skeys[i] & msk : 0u;
                const bool is_eq = i < c1 && kk == T;
                const uint32_t meq = __ballot_sync(0xffffffffu, is_eq);
                const bool take =
                    (i < c1 && kk > T) || (is_eq && eq_seen + __popc(meq & lt) < need_eq);
                const uint32_t mt = __ballot_sync(0xffffffffu, take);
                if (take) selp[out + __popc(mt & lt)] = i;
                out += __popc(mt);
                eq_seen += __popc(meq);
            }
        }
        if (ctid == 0) {
            selp[K] = n - 1;
            p.n_sel[u] = k;
            p.view.n_tokens[u] = s.tokens;
        }
        // then the view rows, every block-table lookup in flight together (a
        // lookup inside the ranking loop above would serialise them)
        consumer_bar();
        for (int c = ctid; c < k; c += kCThreads) crow[c] = chunk_of(__ldcg(selp + c));
    }
    if (room && ctid < segs) {
        if (phys_new >= 0 && phys_new < kv.num_pages) {
            append_store(kv, b, h, s.held, phys_new, ctid, ar);
            fence_proxy_async_global();     // the row is read next by TMA (async proxy)
        } else if (ctid == 0) {
            flag(p.status, SE_DEV_BAD_INDEX);
        }
    }
}

// Q- / Q+ of sequence b per (KV head, d) for the page bound, on the consumer
// warps, into coef (global memory): U[p] = sum_d Q-[d] kmin[p,d] + Q+[d] kmax[p,d] with Q+ = sum_g max(q_g, 0)
// and Q- = sum_g min(q_g, 0) (kmin <= kmax picks the larger product per sign).
// coef[h][0][d] = Q-, coef[h][1][d] = Q+.  Group sums are xor-shuffles across
// the lanes of one d-block (G is a power of two).
template <int D>
__device__ __forceinline__ void step_fold(const StepParams& p, int b, float* coef, int warp,
                                          int lane) {
    const int H = p.kv.num_kv_heads, G = p.G;
    const int kNdv = 32 / G;                              // d-blocks of 8 per warp task
    const int tph = (D / 8 + kNdv - 1) / kNdv;            // warp tasks per head
    const int g = lane / kNdv, dv = lane % kNdv;
    constexpr int kPre = 4;
    uint4 qv[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
        const int task = warp + i * kConsumerWarps;
        const int hh = task / tph, d8 = (task % tph) * kNdv + dv;
        qv[i] = (task < H * tph && d8 < D / 8)
                    ? *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + hh * G + g) * D + d8 * 8)
                    : make_uint4(0, 0, 0, 0);
    }
    int i = 0;
    for (int task = warp; task < H * tph; task += kConsumerWarps, ++i) {
        const int hh = task / tph, d8 = (task % tph) * kNdv + dv;
        uint4 v = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < kPre; ++j)
            if (i == j) v = qv[j];
        if (i >= kPre && d8 < D / 8)
            v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + hh * G + g) * D + d8 * 8);
        const uint32_t a4[4] = {v.x, v.y, v.z, v.w};
        float lo[8], hi[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float f0 = bf_lo(a4[e]), f1 = bf_hi(a4[e]);
            lo[2 * e] = fminf(f0, 0.f);
            lo[2 * e + 1] = fminf(f1, 0.f);
            hi[2 * e] = fmaxf(f0, 0.f);
            hi[2 * e + 1] = fmaxf(f1, 0.f);
        }
        for (int o = kNdv; o < 32; o <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] += __shfl_xor_sync(0xffffffffu, lo[e], o);
                hi[e] += __shfl_xor_sync(0xffffffffu, hi[e], o);
            }
        }
        if (g == 0 && d8 < D / 8) {
            float4* cl = reinterpret_cast<float4*>(coef + (hh * 2) * D + d8 * 8);
            float4* ch = reinterpret_cast<float4*>(coef + (hh * 2 + 1) * D + d8 * 8);
            cl[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
            cl[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
            ch[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
            ch[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
        }
    }
}

// The consumers' wait for the next item descriptor is longer than any producer
// wait, so that a producer which gives up always publishes the end item first:
// every consumer warp then reads the same descriptors and reaches the same
// named barriers.
constexpr unsigned long long kItemWaitLimitNs = 4ull * kWaitLimitNs;

__device__ bool item_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kItemWaitLimitNs) return false;
    }
}

// A consumer warp's bounded wait on a full stage.  Every lane polls; the
// outcome is lane 0's, so that the whole warp takes one branch before the
// warp-synchronous code that reads the stage.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           const StepParams& p, int lane) {
    bool ok = !*abort_flag && mbar_wait(bar, parity, abort_flag);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok && lane == 0 && !*abort_flag) give_up(p, abort_flag);
    return ok;
}

template <int D, int NT, bool TWO_TERM, int VPL, bool REG>
__global__ void __launch_bounds__(kDecodeThreads, NT == 2 ? 2 : 0)
    quest_step_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const StepParams p) {
    using S = DecShape<D, NT>;
    using SS = StepShape<D>;
    constexpr int NS = SS::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* ring = base;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * SS::kStageBytes);
    uint64_t* empty = full + NS;
    uint64_t* ifull = empty + NS;
    uint64_t* iempty = ifull + kItemSlots;
    int* stage_ntok = reinterpret_cast<int*>(iempty + kItemSlots);
    StepItem* items = reinterpret_cast<StepItem*>(stage_ntok + NS);
    int* misc = reinterpret_cast<int*>(items + kItemSlots);   // 16 ints
    volatile int* abort_flag = misc;                          // [0]
    // [1] last-piece flag of the decode merge, [2] top-k go, [3] last CTA,
    // [4..7] scan scratch, [8] block total
    float* coef = reinterpret_cast<float*>(base + p.off_coef);
    uint8_t* area = base + p.off_union;
    int4* sinfo = reinterpret_cast<int4*>(base + p.off_sinfo);   // [2 * batch]
    int* rstart = reinterpret_cast<int*>(base + p.off_rstart);   // [rounds + 1]
    const int* gabort = p.sync + 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.kv.num_kv_heads, stride = p.kv.max_pages_per_seq;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&ifull[s], 1);
            mbar_init(&iempty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    int grab = 0;
    if (warp == kConsumerWarps && lane == 0) grab = atomicAdd(p.sync, 1);
    if (warp < kConsumerWarps) {
        // ---- per-sequence plans and the round table (consumer warps) ----
        const int ctid = threadIdx.x;
        int carry = 0;
        for (int b0 = 0; b0 < p.batch; b0 += kCThreads) {
            const int b = b0 + ctid;
            SeqPlan s = {};
            int dec = 0;
            if (b < p.batch) {
                s = seq_plan(p, b, true);
                dec = H * s.pieces;
            }
            const int incl = scan128(dec, misc + 4, warp, lane);
            if (b < p.batch) {
                sinfo[2 * b] = make_int4(s.tiles, s.pieces, s.chunks, carry + incl - dec);
                sinfo[2 * b + 1] = make_int4(s.held, s.ctx, s.n, s.k);
            }
            if (ctid == kCThreads - 1) misc[8] = incl;
            consumer_bar();
            carry += misc[8];
            consumer_bar();
        }
        carry = 0;
        for (int r0 = 0; r0 <= p.rounds; r0 += kCThreads) {
            const int r = r0 + ctid;
            int cnt = 0;
            if (r < p.rounds) {
                if (r < p.batch) cnt += sinfo[2 * r].x;
                const int bt = r - p.lag_topk;
                if (bt >= 0 && bt < p.batch) cnt += H;
                const int bd = r - p.lag_dec;
                if (bd >= 0 && bd < p.batch) cnt += H * sinfo[2 * bd].y;
            }
            const int incl = scan128(cnt, misc + 4, warp, lane);
            if (r <= p.rounds) rstart[r] = carry + incl - cnt;
            if (ctid == kCThreads - 1) misc[8] = incl;
            consumer_bar();
            carry += misc[8];
            consumer_bar();
        }
    }
    __syncthreads();
    const int total = rstart[p.rounds];

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
        }
        auto make_item = [&](int gidx) {
            StepItem it = {kItemEnd, 0, 0, 0, 0, 0, 0, 0};
            if (gidx >= p.batch + total || *abort_flag ||
                *reinterpret_cast<const volatile int*>(gabort))
                return it;
            if (gidx < p.batch) {                         // the query folds come first
                it.type = kItemFold;
                it.b = gidx;
                return it;
            }
            const int idx = gidx - p.batch;
            int lo = 0, hi = p.rounds - 1;                // last round starting at or before idx
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (rstart[mid] <= idx) lo = mid; else hi = mid - 1;
            }
            const int r = lo;
            int off = idx - rstart[r];
            if (r < p.batch) {
                const int tiles = sinfo[2 * r].x;
                if (off < tiles) {
                    const int m = sinfo[2 * r + 1].z - 1;
                    it.type = kItemScore;
                    it.b = r;
                    it.a0 = off * p.tile_pages;
                    it.a1 = min(m, it.a0 + p.tile_pages);
                    return it;
                }
                off -= tiles;
            }
            const int bt = r - p.lag_topk;
            if (bt >= 0 && bt < p.batch) {
                if (off < H) {
                    it.type = kItemTopk;
                    it.b = bt;
                    it.h = off;
                    return it;
                }
                off -= H;
            }
            const int bd = r - p.lag_dec;
            const int4 a = sinfo[2 * bd];
            const int pieces = a.y, chunks = a.z;
            const int h = off / pieces, kp = off % pieces;
            it.type = kItemDecode;
            it.b = bd;
            it.h = h;
            it.a0 = (int)((int64_t)chunks * kp / pieces);
            it.a1 = (int)((int64_t)chunks * (kp + 1) / pieces);
            it.a3 = a.w + h * pieces;
            it.a2 = pieces == 1 ? -1 : it.a3 + kp;
            it.a4 = pieces;
            return it;
        };
        uint32_t seq = 0, iseq = 0;
        int cur = grab;                                    // lane 0's
        while (true) {
            StepItem it = {kItemEnd, 0, 0, 0, 0, 0, 0, 0};
            int nxt = 0;
            if (lane == 0) {
                it = make_item(cur);
                if (it.type != kItemEnd) nxt = atomicAdd(p.sync, 1);   // the next item, early
                const int is = iseq % kItemSlots;
                // not cut short by the abort word: after an abort the consumers
                // skip their work, free the slot at once and need the end item
                volatile int never = 0;
                if (!mbar_wait(&iempty[is], ((iseq / kItemSlots) & 1) ^ 1, &never)) {
                    // the consumers stopped reading: publish nothing more
                    if (!*abort_flag) give_up(p, abort_flag);
                    it.type = kItemEnd;
                } else {
                    items[is] = it;
                    mbar_arrive(&ifull[is]);
                }
            }
            ++iseq;
            const int type = __shfl_sync(0xffffffffu, it.type, 0);
            if (type == kItemEnd) break;
            const int b = __shfl_sync(0xffffffffu, it.b, 0);
            const int a0 = __shfl_sync(0xffffffffu, it.a0, 0);
            const int a1 = __shfl_sync(0xffffffffu, it.a1, 0);
            if (type == kItemScore) {
                // the tile's summaries are one contiguous block: 1-D bulk copies
                const int64_t bytes = (int64_t)(a1 - a0) * H * SS::kSumBytes;
                const uint8_t* src = static_cast<const uint8_t*>(p.kv.meta) +
                                     ((int64_t)b * stride + a0) * H * SS::kSumBytes;
                const int nst = static_cast<int>((bytes + SS::kStageBytes - 1) / SS::kStageBytes);
                if (lane == 0) {
                    for (int j = 0; j < nst; ++j) {
                        const uint32_t sq = seq + j;
                        const int s = sq % NS;
                        if (!*abort_flag && !mbar_wait(&empty[s], ((sq / NS) & 1) ^ 1, abort_flag))
                            give_up(p, abort_flag);
                        const uint32_t sz = static_cast<uint32_t>(
                            min(static_cast<int64_t>(SS::kStageBytes), bytes - (int64_t)j * SS::kStageBytes));
                        if (!*abort_flag) {
                            mbar_arrive_expect_tx(&full[s], sz);
                            bulk_g2s(ring + s * SS::kStageBytes, src + (int64_t)j * SS::kStageBytes, sz,
                                     &full[s]);
                        } else {
                            mbar_arrive(&full[s]);
                        }
                    }
                }
                seq += nst;
            } else if (type == kItemDecode) {
                const int h = __shfl_sync(0xffffffffu, it.h, 0);
                const int u = b * H + h;
                const int4 si = sinfo[2 * b + 1];          // held, ctx, n, k
                const int tokens = si.z <= si.w ? si.y : kPage * (si.w - 1) + (si.y - kPage * (si.z - 1));
                if (a1 > a0) {
                    if (lane == 0 && !*abort_flag &&
                        !wait_geq(p.unit_ready + u, 1, abort_flag, gabort))
                        give_up(p, abort_flag);
                    __syncwarp();
                    // the view rows and the appended row were written by the CTA
                    // that ran the top-k; the row is read here by TMA
                    fence_proxy_async_global();
                }
                const int32_t* crow = p.view.chunk_row + (int64_t)u * p.view.max_chunks;
                for (int cb = a0; cb < a1; cb += 32) {
                    const int row_l = cb + lane < a1 ? __ldcg(crow + cb + lane) : -1;
                    const int nb = min(32, a1 - cb);
                    // four chunks per iteration: chunk t = lane / 4 of the group is
                    // led by lane 4t (waits for its stage, arms its barrier); then
                    // lanes 4t..4t+3 issue that chunk's K and V boxes together
                    for (int j0 = 0; j0 < nb; j0 += 4) {
                        const int t = lane >> 2, q = lane & 3;
                        const int j = j0 + t;
                        const bool mine = t < 4 && j < nb;
                        const int row = __shfl_sync(0xffffffffu, row_l, min(j, 31));
                        const uint32_t sq = seq + t;
                        const int s = sq % NS;
                        int go = 0;
                        if (mine && q == 0) {
                            const int c = cb + j;
                            if (!*abort_flag && !mbar_wait(&empty[s], ((sq / NS) & 1) ^ 1, abort_flag))
                                give_up(p, abort_flag);
                            int cnt = min(kPage, tokens - c * kPage);
                            if (*abort_flag) {
                                cnt = 0;
                            } else if (row < 0 || (int64_t)row >= p.total_rows) {
                                flag(p.status, SE_DEV_BAD_INDEX);
                                cnt = 0;
                            }
                            stage_ntok[s] = cnt;
                            go = cnt > 0;
                            if (go)
                                mbar_arrive_expect_tx(&full[s], S::kStageBytes);
                            else
                                mbar_arrive(&full[s]);
                        }
                        go = __shfl_sync(0xffffffffu, go, lane & ~3);
                        if (mine && go && q < 2 * S::kBoxes) {
                            uint8_t* dst = ring + s * SS::kStageBytes + (q & 1) * S::kChunkBytes +
                                           (q >> 1) * 2048;
                            tma_load_2d(dst, (q & 1) ? &tv : &tk, &full[s], 64 * (q >> 1), row);
                        }
                        seq += min(4, nb - j0);
                    }
                }
            }
            cur = __shfl_sync(0xffffffffu, nxt, 0);
        }
        // every copy issued by this CTA lands before the CTA may exit
        if (lane == 0) {
            const uint32_t first = seq > (uint32_t)NS ? seq - NS : 0;
            volatile int never = 0;
            for (uint32_t q2 = first; q2 < seq; ++q2)
                mbar_wait(&full[q2 % NS], (q2 / NS) & 1, &never);
        }
    } else {
        // ------------------------------ consumers ------------------------------
        const int ctid = threadIdx.x;
        DecOut dout;
        dout.out = p.out;
        dout.out_f32 = p.out_f32;
        dout.lse_out = p.lse_out;
        dout.o_part = p.o_part;
        dout.lse_part = p.lse_part;
        dout.counters = p.counters;
        dout.Hq = p.Hq;
        dout.G = p.G;
        uint32_t seq = 0, iseq = 0;
        int coef_b = -1;
        while (true) {
            const int is = iseq % kItemSlots;
            if (!item_wait(&ifull[is], (iseq / kItemSlots) & 1)) {
                // the producer is gone (it always publishes the end item when it
                // gives up, well inside this limit): stop
                if (lane == 0) give_up(p, abort_flag);
                break;
            }
            const StepItem it = items[is];
            __syncwarp();
            if (lane == 0) mbar_arrive(&iempty[is]);
            ++iseq;
            if (it.type == kItemEnd) break;
            const int b = it.b;
            if (it.type == kItemFold) {
                step_fold<D>(p, b, p.coef + (int64_t)b * H * 2 * D, warp, lane);
                consumer_bar();
                if (ctid == 0) st_release(p.seq_folded + b, 1);
            } else if (it.type == kItemScore) {
                constexpr int kU4 = D / 4;                    // 16-byte vectors per summary
                constexpr int kLps = kU4 / VPL;               // lanes per summary
                constexpr int kR = 32 / kLps;                 // summaries per warp-wide read
                const int sub = lane % kLps, slot = lane / kLps;
                const float* cg = p.coef + (int64_t)b * H * 2 * D;
                if (b != coef_b) {
                    // the sequence's coefficients, folded by its fold item
                    if (ctid == 0 && !*abort_flag &&
                        !wait_geq(p.seq_folded + b, 1, abort_flag, gabort))
                        give_up(p, abort_flag);
                    consumer_bar();
                    if (!REG) {
                        for (int i = ctid; i < H * 2 * D / 4; i += kCThreads)
                            reinterpret_cast<float4*>(coef)[i] = __ldcg(reinterpret_cast<const float4*>(cg) + i);
                        consumer_bar();
                    }
                    coef_b = b;
                }
                float cr[REG ? VPL * 8 : 1];
                if (REG) {
                    const int h = slot % H;                   // fixed: kR is a multiple of H
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const float4* c4 = reinterpret_cast<const float4*>(cg + h * 2 * D + (j * kLps + sub) * 8);
                        const float4 x0 = __ldcg(c4), x1 = __ldcg(c4 + 1);
                        cr[REG ? j * 8 + 0 : 0] = x0.x;
                        cr[REG ? j * 8 + 1 : 0] = x0.y;
                        cr[REG ? j * 8 + 2 : 0] = x0.z;
                        cr[REG ? j * 8 + 3 : 0] = x0.w;
                        cr[REG ? j * 8 + 4 : 0] = x1.x;
                        cr[REG ? j * 8 + 5 : 0] = x1.y;
                        cr[REG ? j * 8 + 6 : 0] = x1.z;
                        cr[REG ? j * 8 + 7 : 0] = x1.w;
                    }
                }
                const int nsum_all = (it.a1 - it.a0) * H;
                const int nst = (nsum_all + SS::kSumsPerStage - 1) / SS::kSumsPerStage;
                uint32_t* keys = p.keys + (int64_t)b * H * stride + it.a0;
                for (int j = 0; j < nst; ++j, ++seq) {
                    if ((seq % kConsumerWarps) != (uint32_t)warp) continue;
                    const int s = seq % NS;
                    const bool ok = stage_wait(&full[s], (seq / NS) & 1, abort_flag, p, lane);
                    const int nsum = min(SS::kSumsPerStage, nsum_all - j * SS::kSumsPerStage);
                    if (ok) {
                        const uint8_t* st = ring + s * SS::kStageBytes;
                        for (int t0 = 0; t0 < nsum; t0 += kR) {
                            const int tl = t0 + slot;
                            const int t = j * SS::kSumsPerStage + tl;   // summary within the tile
                            const int h = t % H, pl = t / H;
                            float acc = 0.f;
                            if (tl < nsum) {
                                const uint4* sv = reinterpret_cast<const uint4*>(st + tl * SS::kSumBytes);
#pragma unroll
                                for (int jj = 0; jj < VPL; ++jj) {
                                    const uint4 w = sv[jj * kLps + sub];
                                    const uint32_t a4[4] = {w.x, w.y, w.z, w.w};
                                    const float* cf = coef + h * 2 * D + (jj * kLps + sub) * 8;
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float c0 = REG ? cr[REG ? jj * 8 + 2 * e : 0] : cf[2 * e];
                                        const float c1 = REG ? cr[REG ? jj * 8 + 2 * e + 1 : 0] : cf[2 * e + 1];
                                        acc = fmaf(c0, bf_lo(a4[e]), acc);
                                        acc = fmaf(c1, bf_hi(a4[e]), acc);
                                    }
                                }
                            }
#pragma unroll
                            for (int o = kLps / 2; o >= 1; o >>= 1)
                                acc += __shfl_xor_sync(0xffffffffu, acc, o);
                            if (sub == 0 && tl < nsum) keys[(int64_t)h * stride + pl] = float_key(acc);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
                // the tile's keys are stored: count it for sequence b
                consumer_bar();
                if (ctid == 0) red_release_add(p.seq_scored + b, 1);
            } else if (it.type == kItemTopk) {
                const int4 a = sinfo[2 * b], c = sinfo[2 * b + 1];
                SeqPlan s;
                s.tiles = a.x;
                s.held = c.x;
                s.ctx = c.y;
                s.n = c.z;
                s.k = c.w;
                s.tokens = s.n <= s.k ? s.ctx : kPage * (s.k - 1) + (s.ctx - kPage * (s.n - 1));
                if (ctid == 0) {
                    int go = !*abort_flag;
                    if (go && s.tiles > 0 && !wait_geq(p.seq_scored + b, s.tiles, abort_flag, gabort)) {
                        give_up(p, abort_flag);
                        go = 0;
                    }
                    misc[2] = go;
                }
                consumer_bar();
                const int go = misc[2];
                if (go) step_topk(p, b, it.h, s, area, warp, lane);
                consumer_bar();
                if (ctid == 0 && go) st_release(p.unit_ready + b * H + it.h, 1);
            } else {
                const int h = it.h, u = b * H + h;
                DecState<D, NT> st;
                dec_begin<D, NT>(st, p.q, (int64_t)b * p.Hq + h * p.G, p.G, lane);
                for (int c = it.a0; c < it.a1; ++c, ++seq) {
                    if ((seq % kConsumerWarps) != (uint32_t)warp) continue;
                    const int s = seq % NS;
                    const bool ok = stage_wait(&full[s], (seq / NS) & 1, abort_flag, p, lane);
                    const int cnt = ok ? stage_ntok[s] : 0;
                    if (cnt > 0)
                        dec_chunk<D, NT, TWO_TERM>(st, ring + s * SS::kStageBytes, cnt, lane, p.scale,
                                                   p.scale_log2, p.G, nullptr, 0ull);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
                dec_finish<D, NT>(st, reinterpret_cast<float*>(area), misc + 1, dout, b, h, u, it.a2,
                                  make_int2(it.a3, it.a4), warp, lane);
            }
        }
    }

    // ---- the last CTA to finish resets the queue and commits the lengths ----
    __syncthreads();
    if (threadIdx.x == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(p.sync + 1)
                     : "memory");
        misc[3] = old == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (misc[3]) {
        // after an abort the appended rows are not known to be written: the
        // lengths stay as they were
        const bool commit = *reinterpret_cast<const volatile int*>(gabort) == 0;
        for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
            p.seq_scored[b] = 0;
            p.seq_folded[b] = 0;
            const int4 c = sinfo[2 * b + 1];
            if (commit && p.k_new != nullptr && c.y == c.x + 1) {
                const int phys = p.kv.block_table[(int64_t)b * stride + c.x / kPage];
                if (phys >= 0 && phys < p.kv.num_pages) p.kv.ctx_len[b] = c.y;
            }
        }
        for (int u = threadIdx.x; u < p.batch * H; u += blockDim.x) {
            p.unit_ready[u] = 0;
            p.counters[u] = 0;
        }
        if (threadIdx.x == 0) {
            p.sync[0] = 0;
            p.sync[1] = 0;
            p.sync[2] = 0;
        }
    }
}

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct StepWs {
    int* status;
    uint32_t* keys;
    float* coef;
    int* sync;
    int* seq_folded;
    int* seq_scored;
    int* unit_ready;
    int* counters;
    float* lse_part;
    float* o_part;
};

StepWs step_ws_carve(void* ws, int batch, int H, int G, int D, int max_pages, int max_splits) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t units = (size_t)batch * H, slots = units * max_splits;
    StepWs w;
    w.status = reinterpret_cast<int*>(base);
    size_t off = 256;
    w.keys = reinterpret_cast<uint32_t*>(base + off);
    off += a256(units * max_pages * sizeof(uint32_t));
    w.sync = reinterpret_cast<int*>(base + off);
    off += 256;
    w.seq_scored = reinterpret_cast<int*>(base + off);
    off += a256((size_t)batch * sizeof(int));
    w.seq_folded = reinterpret_cast<int*>(base + off);
    off += a256((size_t)batch * sizeof(int));
    w.coef = reinterpret_cast<float*>(base + off);
    off += a256(units * 2 * D * sizeof(float));
    w.unit_ready = reinterpret_cast<int*>(base + off);
    off += a256(units * sizeof(int));
    w.counters = reinterpret_cast<int*>(base + off);
    off += a256(units * sizeof(int));
    w.lse_part = reinterpret_cast<float*>(base + off);
    off += a256(slots * G * sizeof(float));
    w.o_part = reinterpret_cast<float*>(base + off);
    return w;
}

template <int D, int NT, bool TWO, int VPL, bool REG>
cudaError_t run_step(const CUtensorMap& tk, const CUtensorMap& tv, const StepParams& p, size_t smem,
                     cudaStream_t s) {
    auto kern = quest_step_kernel<D, NT, TWO, VPL, REG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem);
    if (e != cudaSuccess) return e;
    const int grid = num_sms() * max(1, per_sm);
    kern<<<grid, kDecodeThreads, smem, s>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int D, int NT, bool TWO>
cudaError_t run_step_vpl(const CUtensorMap& tk, const CUtensorMap& tv, const StepParams& p,
                         size_t smem, cudaStream_t s) {
    // register coefficients when a warp-wide read (4 summaries at D = 128 with
    // 4 vectors per lane, 8 at D = 64) is a multiple of the KV head count
    constexpr int kR = 32 / (D / 4 / 4);
    if (kR % p.kv.num_kv_heads == 0) return run_step<D, NT, TWO, 4, true>(tk, tv, p, smem, s);
    return run_step<D, NT, TWO, 1, false>(tk, tv, p, smem, s);
}

// Dynamic shared memory of the step kernel: the fixed part, the coefficients,
// the union (decode merge / top-k keys and histogram), the sequence plans and
// the round table.  Writes the offsets into p when given.
size_t step_smem(int batch, int H, int D, int G, int max_pages, int lag_dec, StepParams* p) {
    // register coefficients (no shared copy) when a warp-wide read covers a
    // multiple of the KV heads: 4 summaries at D = 128, 8 at D = 64
    const bool reg = (D == 128 ? 4 : 8) % H == 0;
    const int NT = G > 8 ? 2 : 1;
    const size_t fixed = D == 64 ? StepShape<64>::kFixed : StepShape<128>::kFixed;
    const size_t merge = (size_t)(kConsumerWarps * NT * 8 * 2 + 2 * NT * 8 * D +
                                  (kConsumerWarps + 1) * NT * 8) * 4;
    const size_t topk = (size_t)(kStepBins + 64) * 4 + (size_t)max_pages * 4;
    size_t off = (fixed + 15) & ~size_t(15);
    const size_t coef = off;
    off += reg ? 0 : (size_t)H * 2 * D * 4;
    off = (off + 15) & ~size_t(15);
    const size_t uni = off;
    off += std::max(merge, topk);
    off = (off + 15) & ~size_t(15);
    const size_t sinfo = off;
    off += (size_t)batch * 32;
    const size_t rstart = off;
    off += (size_t)(batch + lag_dec + 1) * 4;
    if (p) {
        p->off_coef = static_cast<int>(coef);
        p->off_union = static_cast<int>(uni);
        p->off_sinfo = static_cast<int>(sinfo);
        p->off_rstart = static_cast<int>(rstart);
    }
    return off + 1024;                                              // alignment slack
}

}  // namespace

size_t quest_step_ws_bytes(int batch, int H, int G, int D, int max_pages, int max_splits) {
    const size_t units = (size_t)batch * H, slots = units * max_splits;
    return 256 + a256(units * max_pages * sizeof(uint32_t)) + 256 +
           2 * a256((size_t)batch * sizeof(int)) + a256(units * 2 * D * sizeof(float)) +
           2 * a256(units * sizeof(int)) + a256(slots * G * sizeof(float)) +
           a256(slots * G * D * sizeof(float));
}

size_t quest_step_smem_bytes(int batch, int H, int D, int G, int max_pages, int lag_dec) {
    return step_smem(batch, H, D, G, max_pages, lag_dec, nullptr);
}

cudaError_t launch_quest_step(const se_paged_kv& kv, const void* k_new, const void* v_new,
                              const void* q, int batch, int num_q_heads, const int32_t* budget,
                              float scale, int out_dtype, int max_splits, const StepTuning& tune,
                              int32_t* sel_pages, int32_t* n_sel, const se_view& view, void* out,
                              float* lse, void* ws, cudaEvent_t ev_begin, cudaEvent_t ev_end,
                              cudaStream_t s) {
    const int H = kv.num_kv_heads, D = kv.head_dim, G = num_q_heads / H;
    const int units = batch * H;
    if (units == 0) return cudaSuccess;
    const int64_t total_rows = (int64_t)kv.num_pages * H * kPage;
    CUtensorMap tk, tv;
    if (!encode_rows_map(&tk, kv.k, total_rows, D) || !encode_rows_map(&tv, kv.v, total_rows, D))
        return cudaErrorInvalidValue;
    const StepWs w = step_ws_carve(ws, batch, H, G, D, kv.max_pages_per_seq, max_splits);

    StepParams p;
    p.kv = kv;
    p.q = static_cast<const uint16_t*>(q);
    p.Hq = num_q_heads;
    p.G = G;
    p.batch = batch;
    p.budget = budget;
    p.k_new = static_cast<const uint4*>(k_new);
    p.v_new = static_cast<const uint4*>(v_new);
    p.sel_pages = sel_pages;
    p.n_sel = n_sel;
    p.view = view;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.out = out;
    p.out_f32 = out_dtype == 1;
    p.lse_out = lse;
    p.keys = w.keys;
    p.coef = w.coef;
    p.sync = w.sync;
    p.seq_folded = w.seq_folded;
    p.seq_scored = w.seq_scored;
    p.unit_ready = w.unit_ready;
    p.counters = w.counters;
    p.o_part = w.o_part;
    p.lse_part = w.lse_part;
    // defaults: ~128 KB score tiles; decode pieces of 16 chunks (128 KB of K/V
    // at D = 128); the top-k of a sequence 8 rounds after its score tiles, so
    // that it mostly finds them done; every decode piece after the last score
    // tile, so that no scoring block waits behind a decode piece whose top-k
    // has not run
    const int page_bytes = H * 2 * D * 2;
    p.tile_pages = tune.tile_pages > 0 ? tune.tile_pages : std::max(1, 131072 / page_bytes);
    p.piece_chunks = tune.piece_chunks > 0 ? tune.piece_chunks : 16;
    p.max_splits = max_splits;
    p.lag_topk = tune.lag_topk > 0 ? tune.lag_topk : 8;
    p.lag_dec = std::max(p.lag_topk, tune.lag_dec > 0 ? tune.lag_dec : batch - 1);
    p.rounds = batch + p.lag_dec;
    p.total_rows = total_rows;
    p.status = w.status;
    const int NT = G > 8 ? 2 : 1;
    const size_t smem = step_smem(batch, H, D, G, kv.max_pages_per_seq, p.lag_dec, &p);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;

    auto record = [&](cudaEvent_t ev) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e2 = cudaStreamIsCapturing(s, &cs);
        if (e2 != cudaSuccess) return e2;
        return cs == cudaStreamCaptureStatusActive
                   ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                   : cudaEventRecord(ev, s);
    };
    cudaError_t e = cudaSuccess;
    if (ev_begin && (e = record(ev_begin)) != cudaSuccess) return e;
    const bool two = out_dtype == 1;
    if (D == 64) {
        e = NT == 1 ? (two ? run_step_vpl<64, 1, true>(tk, tv, p, smem, s)
                           : run_step_vpl<64, 1, false>(tk, tv, p, smem, s))
                    : (two ? run_step_vpl<64, 2, true>(tk, tv, p, smem, s)
                           : run_step_vpl<64, 2, false>(tk, tv, p, smem, s));
    } else {
        e = NT == 1 ? (two ? run_step_vpl<128, 1, true>(tk, tv, p, smem, s)
                           : run_step_vpl<128, 1, false>(tk, tv, p, smem, s))
                    : (two ? run_step_vpl<128, 2, true>(tk, tv, p, smem, s)
                           : run_step_vpl<128, 2, false>(tk, tv, p, smem, s));
    }
    if (e != cudaSuccess) return e;
    if (ev_end && (e = record(ev_end)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace se
