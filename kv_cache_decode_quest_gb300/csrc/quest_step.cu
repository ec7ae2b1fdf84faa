// One Quest decode step in one cooperative kernel: the new token's append, the
// page scoring, the per-KV-head top-k and the split-K decode over the selected
// pages.  Same results as se_quest_select_append followed by se_sparse_decode.
//
// Quest picks pages by the query's upper-bound score against each page's key
// min/max summary while the whole history stays resident (tokendh.com article on
// SparseEngine, section "历史太长,会撑爆什么"); the attention then reads only the
// rows the view exposes ("SparseEngine：稀疏优先推理引擎", section "方法 / 关键模块").
//
// Why one kernel: the step is two HBM streams (the page summaries, then the
// selected K/V rows) joined by a short, latency-bound top-k per unit.  As
// separate launches every kernel boundary, the top-k kernel and the decode's
// planning sit on the critical path.  Here every CTA of one resident wave (a
// cooperative launch, so every CTA is running) follows a static schedule that
// it computes itself:
//   score: one contiguous slice of one sequence's candidate page summaries
//     (all KV heads of each page), derived from the lengths and budgets alone
//     so that the first copy leaves at once; streamed with 1-D bulk copies
//     through the stage ring and turned into order-preserving keys in the
//     workspace; the slice's page count is then added to the sequence's
//     scored counter;
//   plan: once its own slices are scored (while the other CTAs finish
//     theirs), the decode pieces, the same split plan in every CTA;
//   decode piece: a range of chunks of one unit u = (b, h), streamed with 2-D
//     TMA into the same ring for the mma.sync decode of decode_core.cuh; split
//     units are merged by the last piece to finish.
// A piece waits (bounded) until every candidate page of b is scored, computes
// the exact top-k of u itself from the keys in L2 (every piece of u computes
// the same selection; none waits on another's), writes its ranks of the
// selection and of the view, and releases the producer.  When no unit has more
// than 2048 candidate pages, the consumers select all the CTA's pieces first,
// in shared memory, while the producer already streams the first pieces'
// chunks; otherwise each selection runs in the idle stage ring right before
// its piece.  The new token's row is written by the piece that holds the
// unit's last chunk (the forced last page), before that chunk's copy.  The
// last CTA to finish commits ctx_len + 1 of every sequence whose token was
// appended (every CTA has read the old lengths by then) and clears the
// control words.  Waits are bounded: a CTA that gives up records
// SE_DEV_TIMEOUT and raises a global abort word that the other waits poll;
// every CTA still walks the same barriers to the end.
//
// CTA layout (160 threads): warps 0-3 consume (stage s is handled by warp
// (stage sequence % 4), in both phases), warp 4 is the producer.
#include <algorithm>

#include "append.cuh"
#include "common.cuh"
#include "decode_core.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kCThreads = kConsumerWarps * 32;         // 128 consumer threads
constexpr int kProducerWarp = kConsumerWarps;          // warp 4
constexpr int kStepThreads = (kConsumerWarps + 1) * 32;
constexpr int kDigit = 10, kStepBins = 1 << kDigit;     // top-k: 10-bit radix digits
constexpr int kMaxPieces = 32;                          // decode pieces per CTA at most
constexpr int kMaxScoreItems = 8;                       // score slices per CTA at most
constexpr uint32_t kFirstFill = 2;                      // score stages issued before the first lands
// The top-k runs once per piece, so its instructions come cold from the
// instruction caches every step: its passes are short rolled loops (code
// fetched once, then reused) rather than unrolled runs.  A unit's keys sit in
// shared memory with one pad word per 32 keys, so that consumer thread t can
// walk its own kKeysPerThread consecutive keys [16t, 16t + 16) of a batch of
// kAreaKeys without bank conflicts; ranks in page order then come from block
// scans of per-thread counts.
constexpr int kKeysPerThread = 16;
constexpr int kAreaKeys = kKeysPerThread * kCThreads;   // 2048
constexpr int kSmallInts = 64;
__host__ __device__ constexpr int key_slots(int m) { return m + (m >> 5); }
__device__ __forceinline__ int kidx(int i) { return i + (i >> 5); }
// the top-k's shared memory: histogram, small ints, keys
constexpr int kSelectBytes = kStepBins * 4 + kSmallInts * 4;
constexpr int kAreaBytes = kSelectBytes + key_slots(kAreaKeys) * 4;

struct StepParams {
    se_paged_kv kv;
    const uint16_t* q;
    int Hq, G, batch, units;
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
    uint32_t* keys;                     // [units][kstride]
    int kstride;                        // max_pages_per_seq rounded up to 4 (16-byte rows)
    int* seq_scored;                    // [batch] candidate pages scored
    int* counters;                      // [units] decode pieces finished
    int* sync;                          // [0] CTAs finished, [1] abort
    float* o_part;                      // [units * max_splits][G][D]
    float* lse_part;                    // [units * max_splits][G]
    int max_splits;
    int off_union;                      // union area offset in dynamic shared memory
    int64_t total_rows;
    unsigned long long wait_ns;
    int* status;
};

template <int D, int NT>
struct StepShape {
    using S = DecShape<D, NT>;
    static constexpr int kStageBytes = S::kStageBytes;                 // 8 KB at D = 128
    static constexpr int kStages = D == 64 ? 24 : (NT == 1 ? 12 : 8);  // as the decode kernel
    static constexpr int kSumBytes = 2 * D * 2;                        // one (page, head) summary
    static constexpr int kSumsPerStage = kStageBytes / kSumBytes;      // 16
    static_assert(kStages % kConsumerWarps == 0, "stage ownership needs kStages % 4 == 0");
    // small areas after the ring: full/empty barriers, the plan barrier (and
    // 8 bytes of padding), the pieces' ready barriers, stage token counts,
    // misc ints, the CTA's pieces (item, sequence values, unit range) and its
    // score slices (the consumers' and the producer's copies)
    static constexpr int kFixed = kStages * 16 + 16 + kMaxPieces * 8 + kStages * 4 + 64 * 4 +
                                  kMaxPieces * 32 + 2 * kMaxScoreItems * 16;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// This CTA gives up: results are invalid; the kernel walks on to its end.
__device__ __forceinline__ void give_up(const StepParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    flag(p.status, SE_DEV_TIMEOUT);
    atomicExch(p.sync + 1, 1);
}

// Bounded wait (one thread) for *ctr >= target (acquire).  False on timeout,
// on this CTA's abort, or when another CTA raised the global abort word.
__device__ bool wait_count(const StepParams& p, const int* ctr, int target,
                           volatile int* abort_flag) {
    if (ld_acquire(ctr) >= target) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (ld_acquire(ctr) >= target) return true;
        if (*abort_flag || *reinterpret_cast<const volatile int*>(p.sync + 1)) return false;
        if (globaltimer() - t0 > p.wait_ns) return false;
        __nanosleep(64);
    }
}

// A sequence's step values, the same in every CTA: held = clamped ctx_len, the
// token appended when it fits, n pages, k pages of budget, m candidate pages
// to score (0 when every page is selected), the unit's chunks and tokens.
struct SeqVals {
    int held, ctx, n, k, m, chunks, tokens, room;
};
__device__ __forceinline__ SeqVals seq_vals(int held_raw, int bud, int cap, bool pending) {
    SeqVals s;
    s.held = held_raw < 0 ? 0 : (held_raw > cap ? cap : held_raw);
    s.room = pending && s.held < cap;
    s.ctx = s.room ? s.held + 1 : s.held;
    s.n = (s.ctx + kPage - 1) / kPage;
    s.k = max(1, (bud < 0 ? 0 : bud) / kPage);
    if (s.n > s.k) {
        s.m = s.n - 1;
        s.chunks = s.k;
        s.tokens = kPage * (s.k - 1) + (s.ctx - kPage * (s.n - 1));
    } else {
        s.m = 0;
        s.chunks = s.n;
        s.tokens = s.ctx;
    }
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

// The float an order-preserving key was made from (float_key inverted).
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Descending scan of a 1024-bin histogram on the 128 consumer threads (thread
// t owns bins 1023-8t .. 1016-8t): the bin holding the remaining-th largest
// key.  Writes sel[0] = that bin, sel[1] = keys in the bins above it, sel[2] =
// keys in it.
__device__ __forceinline__ void find_bin(const int* hist, int remaining, int* tmp, int* sel,
                                         int warp, int lane) {
    constexpr int NB = kStepBins;
    constexpr int kPer = NB / kCThreads;                  // 8 bins per thread
    const int ctid = warp * 32 + lane;
    int vv[kPer], v = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        vv[j] = hist[NB - 1 - (ctid * kPer + j)];
        v += vv[j];
    }
    int run = scan128(v, tmp, warp, lane) - v;            // keys in the bins above this thread's
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (run < remaining && run + vv[j] >= remaining) {
            sel[0] = NB - 1 - (ctid * kPer + j);
            sel[1] = run;
            sel[2] = vv[j];
        }
        run += vv[j];
    }
    consumer_bar();
}

// Exclusive scan over the 128 consumer threads; *total gets the sum.
__device__ __forceinline__ int scan128_excl(int v, int* tmp, int warp, int lane, int* total) {
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    consumer_bar();
    int before = 0;
#pragma unroll
    for (int i = 0; i < kConsumerWarps; ++i) before += i < warp ? tmp[i] : 0;
    *total = tmp[0] + tmp[1] + tmp[2] + tmp[3];
    consumer_bar();
    return x - v + before;
}

// Radix threshold (the general case): bits above the highest bit in which the
// largest and smallest key differ are common to all keys, so the 10-bit radix
// digits start there, and a pass ends the search when the boundary digit is
// kept whole.
__device__ void radix_threshold(const uint32_t* sk, int m, int K, uint32_t lo, uint32_t hi,
                                int* hist, int* tmp, int* sel, uint32_t* T, uint32_t* mask,
                                int* need, int warp, int lane) {
    constexpr int kPer = kStepBins / kCThreads;
    const int ctid = warp * 32 + lane;
    const int top = 31 - __clz(lo ^ hi);                  // highest differing bit
    uint32_t msk = top == 31 ? 0u : ~((2u << top) - 1u);
    uint32_t prefix = hi & msk;
    int remaining = K;
    int low = top + 1;                                    // bits [low, 32) are decided
#pragma unroll 1
    while (low > 0) {
        const int w = min(kDigit, low), shift = low - w;
        const uint32_t dm = (1u << w) - 1u;
#pragma unroll
        for (int j = 0; j < kPer; ++j) hist[ctid * kPer + j] = 0;
        consumer_bar();
#pragma unroll 2
        for (int i = ctid; i < m; i += kCThreads) {
            const uint32_t k = sk[kidx(i)];
            if ((k & msk) == prefix) atomicAdd(&hist[(k >> shift) & dm], 1);
        }
        consumer_bar();
        find_bin(hist, remaining, tmp, sel, warp, lane);
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

// Threshold of the top K of m order-preserving keys in shared memory (lo /
// hi: the smallest and largest), on the 128 consumer threads.  On return:
// keys above *T (under *mask) are kept, and so are the first *need keys equal
// to *T.  One histogram pass over 1024 equal-width bins of the score VALUES
// between the smallest and the largest (weakly monotone in the key, so every
// bin above the boundary bin is kept whole and every bin below it dropped),
// then the keys of the boundary bin, when it holds at most kBinCap, are
// gathered and ranked exactly by (key desc, page asc); a larger boundary bin
// (many equal or clustered scores, or a range that overflows) takes the
// radix passes.
constexpr int kBinCap = 128;
__device__ void step_threshold(const uint32_t* sk, int m, int K, uint32_t lo, uint32_t hi,
                               int* hist, int* tmp, int* sel, int* cnt, uint32_t* T,
                               uint32_t* mask, int* need, int warp, int lane) {
    constexpr int kPer = kStepBins / kCThreads;
    const int ctid = warp * 32 + lane;
    if (lo == hi) {                                       // every key is equal
        *T = hi;
        *mask = 0xffffffffu;
        *need = K;
        return;
    }
    const float flo = key_float(lo);
    const float scale = static_cast<float>(kStepBins) / (key_float(hi) - flo);
    auto bin_of = [&](uint32_t k) {
        const int b = static_cast<int>((key_float(k) - flo) * scale);   // NaN -> 0
        return min(kStepBins - 1, max(0, b));
    };
#pragma unroll
    for (int j = 0; j < kPer; ++j) hist[ctid * kPer + j] = 0;
    if (ctid == 0) *cnt = 0;
    consumer_bar();
#pragma unroll 2
    for (int i = ctid; i < m; i += kCThreads) atomicAdd(&hist[bin_of(sk[kidx(i)])], 1);
    consumer_bar();
    find_bin(hist, K, tmp, sel, warp, lane);
    const int bstar = sel[0], R = K - sel[1], E = sel[2];
    if (E > kBinCap) {
        consumer_bar();                                   // sel is rewritten
        radix_threshold(sk, m, K, lo, hi, hist, tmp, sel, T, mask, need, warp, lane);
        return;
    }
    // the boundary bin's keys and pages, gathered into the free histogram
    uint32_t* bk = reinterpret_cast<uint32_t*>(hist);
    int* bp = hist + kBinCap;
#pragma unroll 2
    for (int i = ctid; i < m; i += kCThreads) {
        const uint32_t k = sk[kidx(i)];
        if (bin_of(k) == bstar) {
            const int at = atomicAdd(cnt, 1);
            bk[at] = k;
            bp[at] = i;
        }
    }
    consumer_bar();
    if (ctid < E) {
        const uint32_t k = bk[ctid];
        const int pg = bp[ctid];
        int rank = 0, above = 0;
#pragma unroll 1
        for (int j = 0; j < E; ++j) {
            const uint32_t kj = bk[j];
            rank += kj > k || (kj == k && bp[j] < pg);
            above += kj > k;
        }
        if (rank == R - 1) {                              // the last kept key of the bin
            sel[3] = static_cast<int>(k);
            sel[4] = R - above;
        }
    }
    consumer_bar();
    *T = static_cast<uint32_t>(sel[3]);
    *mask = 0xffffffffu;
    *need = sel[4];
    consumer_bar();                                       // hist and sel are rewritten next
}

// The selection of unit u = (b, h) restricted to ranks [c0, c1) on the four
// consumer warps: exact top-(k-1) of the candidate pages 0..n-2 by (score
// desc, page asc) in ascending page order, then the last page (always
// selected, never scored) at rank k-1; all pages when n <= k.  Writes
// sel_pages[u][rank] for the ranks of the range.  The keys were written by
// the scoring slices of other CTAs (read through L2); `area` holds the
// histogram, small ints and the keys (key_slots(m) words).  Returns where in
// the area the range's pages are also left (page of rank c at [c - c0]), or
// null.
__device__ const int* piece_select(const StepParams& p, int u, const SeqVals& s, int c0, int c1,
                                   uint8_t* area, int warp, int lane) {
    const int ctid = warp * 32 + lane;
    const int stride = p.kv.max_pages_per_seq;
    int32_t* selp = p.sel_pages + (int64_t)u * stride;
    int* hist = reinterpret_cast<int*>(area);                    // [1024]
    int* small = hist + kStepBins;                               // kSmallInts
    int* tmp = small;                                            // [4]
    uint32_t* red = reinterpret_cast<uint32_t*>(small + 4);      // [8]
    int* sel = small + 12;                                       // [8]
    int* cnt = small + 20;                                       // [1]
    uint32_t* sk = reinterpret_cast<uint32_t*>(small + kSmallInts);   // [key_slots(m)]
    int* spage = hist;                                           // [c1 - c0] at the end
    const bool keep = c1 - c0 <= kStepBins;
    if (s.m == 0) {
#pragma unroll 1
        for (int c = c0 + ctid; c < c1; c += kCThreads) {
            selp[c] = c;
            if (keep) spage[c - c0] = c;
        }
        return keep ? spage : nullptr;
    }
    const int m = s.m, K = s.k - 1;
    if (K > 0 && c0 < K) {
        // the keys into shared memory, with their smallest and largest
        const uint32_t* keys = p.keys + (int64_t)u * p.kstride;
        uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll 1
        for (int base = ctid; base < m; base += kCThreads * 4) {
            uint32_t kk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = base + j * kCThreads;
                kk[j] = i < m ? __ldcg(keys + i) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = base + j * kCThreads;
                if (i < m) {
                    sk[kidx(i)] = kk[j];
                    lo = min(lo, kk[j]);
                    hi = max(hi, kk[j]);
                }
            }
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
        int need = 0;
        uint32_t T = 0, msk = 0;
        step_threshold(sk, m, K, lo, hi, hist, tmp, sel, cnt, &T, &msk, &need, warp, lane);
        // ranks in page order: thread t walks its keys [16t, 16t + 16) of each
        // batch of kAreaKeys, so block scans of the per-thread counts of
        // equal and of kept keys place each kept key
        int eq_carry = 0, take_carry = 0;
#pragma unroll 1
        for (int base = 0; base < m && take_carry < c1; base += kAreaKeys) {
            const int first = base + ctid * kKeysPerThread;
            const int nv = max(0, min(kKeysPerThread, m - first));
            int gt = 0, eq = 0;
#pragma unroll 2
            for (int t = 0; t < nv; ++t) {
                const uint32_t x = sk[kidx(first + t)] & msk;
                gt += x > T;
                eq += x == T;
            }
            int eq_tot = 0, take_tot = 0;
            const int eq_before = eq_carry + scan128_excl(eq, tmp, warp, lane, &eq_tot);
            const int take_eq = max(0, min(eq, need - eq_before));
            int rank = take_carry + scan128_excl(gt + take_eq, tmp, warp, lane, &take_tot);
            int used = 0;
#pragma unroll 2
            for (int t = 0; t < nv; ++t) {
                const uint32_t x = sk[kidx(first + t)] & msk;
                const bool is_eq = x == T;
                const bool tk = x > T || (is_eq && used < take_eq);
                used += is_eq;
                if (tk) {
                    if (rank >= c0 && rank < c1) {
                        selp[rank] = first + t;
                        if (keep) spage[rank - c0] = first + t;
                    }
                    ++rank;
                }
            }
            eq_carry += eq_tot;
            take_carry += take_tot;
        }
    }
    if (c1 == s.k && ctid == 0) {                       // the last page
        selp[K] = s.n - 1;
        if (keep) spage[K - c0] = s.n - 1;
    }
    return keep ? spage : nullptr;
}

__device__ __forceinline__ int warp_excl_scan(int v, int lane) {
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x - v;
}

// The view rows of ranks [c0, c1) of unit u: the physical chunk of each
// selected page (from spage when not null, page of rank c at [c - c0], else
// from sel_pages, written by the calling threads), `nt` threads t = 0..nt-1,
// eight block-table lookups of a thread in flight together.
__device__ void view_rows(const StepParams& p, int u, int c0, int c1, const int* spage, int t,
                          int nt) {
    const int H = p.kv.num_kv_heads, h = u % H, b = u / H;
    const int stride = p.kv.max_pages_per_seq;
    const int32_t* selp = p.sel_pages + (int64_t)u * stride;
    int32_t* crow = p.view.chunk_row + (int64_t)u * p.view.max_chunks;
    const int32_t* btr = p.kv.block_table + (int64_t)b * stride;
    for (int c00 = c0; c00 < c1; c00 += nt * 8) {
        int page[8], phys[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = c00 + e * nt + t;
            page[e] = c < c1 ? (spage ? spage[c - c0] : __ldcg(selp + c)) : -1;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) phys[e] = (page[e] >= 0 && page[e] < stride) ? btr[page[e]] : -1;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = c00 + e * nt + t;
            if (c < c1) {
                if (phys[e] >= 0 && phys[e] < p.kv.num_pages) {
                    crow[c] = (phys[e] * H + h) * kPage;
                } else {
                    crow[c] = -1;
                    flag(p.status, SE_DEV_BAD_INDEX);
                }
            }
        }
    }
}

// Q- / Q+ of sequence b per (KV head, d) for the page bound, into coef (shared
// memory): U[p] = sum_d Q-[d] kmin[p,d] + Q+[d] kmax[p,d] with Q+ = sum_g
// max(q_g, 0) and Q- = sum_g min(q_g, 0) (kmin <= kmax picks the larger
// product per sign).  coef[h][0][d] = Q-, coef[h][1][d] = Q+.  One (head,
// 8-channel block) per consumer thread, its group's loads in flight together.
template <int D>
__device__ __forceinline__ void step_fold(const StepParams& p, int b, float* coef, int ctid) {
    const int H = p.kv.num_kv_heads, G = p.G;
    for (int task = ctid; task < H * (D / 8); task += kCThreads) {
        const int h = task / (D / 8), d8 = task % (D / 8);
        const uint16_t* qb = p.q + ((int64_t)b * p.Hq + h * G) * D + d8 * 8;
        float lo[8], hi[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) lo[e] = hi[e] = 0.f;
#pragma unroll 4
        for (int g = 0; g < G; ++g) {
            const uint4 v = *reinterpret_cast<const uint4*>(qb + (int64_t)g * D);
            const uint32_t a4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float f0 = bf_lo(a4[e]), f1 = bf_hi(a4[e]);
                lo[2 * e] += fminf(f0, 0.f);
                lo[2 * e + 1] += fminf(f1, 0.f);
                hi[2 * e] += fmaxf(f0, 0.f);
                hi[2 * e + 1] += fmaxf(f1, 0.f);
            }
        }
        float4* cl = reinterpret_cast<float4*>(coef + (h * 2) * D + d8 * 8);
        float4* ch = reinterpret_cast<float4*>(coef + (h * 2 + 1) * D + d8 * 8);
        cl[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
        cl[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
        ch[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
        ch[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
    }
}

// One consumer warp scores one stage of `nsum` summaries (all KV heads of a
// page together; summary t of the slice is page p0 + t / H, head t % H): each
// summary is read by kLps lanes, 4 16-byte vectors each (vector j of lane
// `sub` is vector j*kLps + sub of the summary: conflict-free shared-memory
// reads), and becomes the key of its (unit, page).
template <int D>
__device__ __forceinline__ void score_stage(const StepParams& p, const uint8_t* st, int nsum,
                                            int t0, int b, int p0, const float* coef, int lane) {
    constexpr int kU4 = D / 4;                            // 16-byte vectors per summary
    constexpr int kLps = kU4 / 4;                         // lanes per summary
    constexpr int kR = 32 / kLps;                         // summaries per warp-wide read
    constexpr int kSum = 2 * D * 2;
    const int H = p.kv.num_kv_heads;
    const int sub = lane % kLps, slot = lane / kLps;
    for (int r = 0; r < nsum; r += kR) {
        const int tl = r + slot;
        const int t = t0 + tl;
        const int h = t % H, pl = t / H;
        float acc = 0.f;
        if (tl < nsum) {
            const uint4* sv = reinterpret_cast<const uint4*>(st + tl * kSum);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 w = sv[j * kLps + sub];
                const float4* cf =
                    reinterpret_cast<const float4*>(coef + h * 2 * D + (j * kLps + sub) * 8);
                const float4 c0 = cf[0], c1 = cf[1];
                acc = fmaf(c0.x, bf_lo(w.x), acc);
                acc = fmaf(c0.y, bf_hi(w.x), acc);
                acc = fmaf(c0.z, bf_lo(w.y), acc);
                acc = fmaf(c0.w, bf_hi(w.y), acc);
                acc = fmaf(c1.x, bf_lo(w.z), acc);
                acc = fmaf(c1.y, bf_hi(w.z), acc);
                acc = fmaf(c1.z, bf_lo(w.w), acc);
                acc = fmaf(c1.w, bf_hi(w.w), acc);
            }
        }
#pragma unroll
        for (int o = kLps / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (sub == 0 && tl < nsum)
            p.keys[((int64_t)b * H + h) * p.kstride + p0 + pl] = float_key(acc);
    }
}

// score_stage with the lane's coefficients in registers (kPerStage summaries
// per full stage).  When H (a power of two) divides the summaries of one
// warp-wide read, lane (slot, sub) always reads head slot % H and the same
// channel vectors j*kLps + sub, so its 32 coefficients are loaded once per
// slice (coef_regs) and a stage costs shared memory nothing but the
// summaries' own bytes.  The stage's kPerStage / kR reads are independent
// chains, computed together with no branch between them (a partial last stage
// reads stale bytes past nsum and stores no key for them); each chain sums in
// the order of score_stage.  krow: the lane's key row at the stage's first
// page, (b*H + slot%H)*kstride + p0 + t0/H + slot/H.
template <int D>
__device__ __forceinline__ bool coef_in_regs(int H) {
    return (H & (H - 1)) == 0 && (32 / (D / 16)) % H == 0;
}
template <int D>
__device__ __forceinline__ void coef_regs(const float* coef, int H, int lane, float (&cr)[32]) {
    constexpr int kLps = D / 16;
    const int sub = lane % kLps, h = (lane / kLps) % H;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4* cf = reinterpret_cast<const float4*>(coef + h * 2 * D + (j * kLps + sub) * 8);
        const float4 c0 = cf[0], c1 = cf[1];
        cr[j * 8 + 0] = c0.x;
        cr[j * 8 + 1] = c0.y;
        cr[j * 8 + 2] = c0.z;
        cr[j * 8 + 3] = c0.w;
        cr[j * 8 + 4] = c1.x;
        cr[j * 8 + 5] = c1.y;
        cr[j * 8 + 6] = c1.z;
        cr[j * 8 + 7] = c1.w;
    }
}
template <int D, int kPerStage>
__device__ __forceinline__ void score_stage_regs(const uint8_t* st, int nsum, uint32_t* krow,
                                                 int lgH, const float (&cr)[32], int lane) {
    constexpr int kLps = D / 16;
    constexpr int kR = 32 / kLps;
    constexpr int kSum = 2 * D * 2;
    constexpr int kIt = kPerStage / kR;
    const int sub = lane % kLps, slot = lane / kLps;
    float acc[kIt];
#pragma unroll
    for (int r = 0; r < kIt; ++r) acc[r] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 w[kIt];
#pragma unroll
        for (int r = 0; r < kIt; ++r)
            w[r] = reinterpret_cast<const uint4*>(st + (r * kR + slot) * kSum)[j * kLps + sub];
#pragma unroll
        for (int r = 0; r < kIt; ++r) {
            acc[r] = fmaf(cr[j * 8 + 0], bf_lo(w[r].x), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 1], bf_hi(w[r].x), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 2], bf_lo(w[r].y), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 3], bf_hi(w[r].y), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 4], bf_lo(w[r].z), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 5], bf_hi(w[r].z), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 6], bf_lo(w[r].w), acc[r]);
            acc[r] = fmaf(cr[j * 8 + 7], bf_hi(w[r].w), acc[r]);
        }
    }
#pragma unroll
    for (int o = kLps / 2; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < kIt; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
    if (sub == 0) {
#pragma unroll
        for (int r = 0; r < kIt; ++r)
            if (r * kR + slot < nsum) krow[(r * kR) >> lgH] = float_key(acc[r]);
    }
}

// This CTA's scoring slices, from the lengths and budgets alone (no plan
// step, so the first copy goes out at once); one warp, v = (ctx_len, budget)
// of sequence `lane` when batch <= 32.  Up to 32 sequences share the grid in
// proportion to their candidate pages m_b: sequence b owns the consecutive
// CTAs from start_b = b + floor((grid - batch) * (m_0 + ... + m_{b-1}) / M)
// (at least one each), which split its pages evenly.  Up to `grid` sequences
// own grid / batch CTAs each (+1 for the first grid % batch); with more
// sequences than CTAs, CTA c scores sequences c, c + grid, ... whole.  Lane 0
// writes (b, first page, end page) of each non-empty slice; returns their
// count (at most kMaxScoreItems, which the launch guarantees).
__device__ int my_slices(const StepParams& p, int lane, int2 v, int4* items) {
    const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int cap = p.kv.max_pages_per_seq * kPage;
    const bool pending = p.k_new != nullptr;
    int cnt = 0;
    if (p.batch <= 32 && p.batch <= grid) {
        const int m = lane < p.batch ? seq_vals(v.x, v.y, cap, pending).m : 0;
        const long long pre = warp_excl_scan(m, lane);
        const long long M = __reduce_add_sync(0xffffffffu, m);
        const int start = lane + (M > 0 ? (int)((long long)(grid - p.batch) * pre / M) : 0);
        const unsigned own = __ballot_sync(0xffffffffu, lane < p.batch && start <= c);
        const int b = 31 - __clz(own);                   // start_0 = 0 <= c
        const int sb = __shfl_sync(0xffffffffu, start, b);
        const int nx = __shfl_sync(0xffffffffu, start, min(b + 1, 31));
        const int mb = __shfl_sync(0xffffffffu, m, b);
        const int nb = (b + 1 < p.batch ? nx : grid) - sb, j = c - sb;
        const int p0 = (int)((long long)mb * j / nb), p1 = (int)((long long)mb * (j + 1) / nb);
        if (lane == 0 && p1 > p0) items[0] = make_int4(b, p0, p1, 0);
        cnt = p1 > p0;
    } else if (p.batch <= grid) {
        const int per = grid / p.batch, extra = grid % p.batch;
        const int b = c < extra * (per + 1) ? c / (per + 1) : extra + (c - extra * (per + 1)) / per;
        const int sb = b < extra ? b * (per + 1) : extra * (per + 1) + (b - extra) * per;
        const int nb = per + (b < extra ? 1 : 0), j = c - sb;
        const int m = seq_vals(p.kv.ctx_len[b], p.budget[b], cap, pending).m;
        const int p0 = (int)((long long)m * j / nb), p1 = (int)((long long)m * (j + 1) / nb);
        if (lane == 0 && p1 > p0) items[0] = make_int4(b, p0, p1, 0);
        cnt = p1 > p0;
    } else {
        // lane i looks at sequence c + i * grid
        const int b = c + lane * grid;
        const int m = lane < kMaxScoreItems && b < p.batch
                          ? seq_vals(p.kv.ctx_len[b], p.budget[b], cap, pending).m
                          : 0;
        const unsigned has = __ballot_sync(0xffffffffu, m > 0);
        if (m > 0) items[__popc(has & ((1u << lane) - 1))] = make_int4(b, 0, m, 0);
        cnt = __popc(has);
    }
    __syncwarp();
    return cnt;
}

// Sequence b's step values from its ctx_len and budget (L1-cached loads: both
// stay unchanged until the last CTA commits the new lengths).
__device__ __forceinline__ SeqVals seq_of(const StepParams& p, int b) {
    return seq_vals(p.kv.ctx_len[b], p.budget[b], p.kv.max_pages_per_seq * kPage,
                    p.k_new != nullptr);
}

// Where a unit's top-k keeps its keys: in the union area of shared memory when
// no unit has more than kAreaKeys candidate pages (every selection of the CTA
// then runs before its decodes, while the ring streams), else in the idle
// stage ring, right before each piece's decode.  One warp.
__device__ int keys_in_area(const StepParams& p, int lane) {
    int mx = 0;
#pragma unroll 1
    for (int b = lane; b < p.batch; b += 32) mx = max(mx, seq_of(p, b).m);
    return __reduce_max_sync(0xffffffffu, mx) <= kAreaKeys;
}

// Decode pieces, the same in every CTA (one warp): unit u gets pieces_u =
// max(1, min(max_splits, nc_u, floor(nc_u * share / total))) pieces of
// nc_u * k / pieces_u chunks, share lowered from slots = grid * ceil(units /
// grid) until the pieces fit the slots; piece t (in unit order) is run by CTA
// t % grid and owns the partial slot t.  Writes this CTA's pieces (unit, first
// chunk, end chunk, partial slot or -1) and their units' (first slot, pieces),
// and returns their count.
__device__ int plan_decode(const StepParams& p, int lane, int4* items, int2* uitems) {
    const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int H = p.kv.num_kv_heads, units = p.units;
    auto nc_of = [&](int u) { return seq_of(p, u / H).chunks; };
    int total = 0;
#pragma unroll 1
    for (int base = 0; base < units; base += 32)
        total += __reduce_add_sync(0xffffffffu, base + lane < units ? nc_of(base + lane) : 0);
    const int tot = max(1, total);
    const int slots = grid * ((units + grid - 1) / grid);
    auto pieces_of = [&](int nc, int share) {
        return nc == 0 ? 1
                       : max(1, min(p.max_splits, min(nc, (int)((long long)nc * share / tot))));
    };
    int share = slots, run = 0;
#pragma unroll 1
    for (int iter = 0; iter < 6; ++iter) {
        run = 0;
#pragma unroll 1
        for (int base = 0; base < units; base += 32) {
            const int u = base + lane;
            const int nc = u < units ? nc_of(u) : 0;
            const int pc = u < units ? pieces_of(nc, share) : 0;
            const int off = run + warp_excl_scan(pc, lane);
            if (u < units) {
                for (int t = c; t < off + pc; t += grid) {
                    if (t >= off && (t - c) / grid < kMaxPieces) {
                        const int j = (t - c) / grid, k = t - off;
                        items[j] = make_int4(u, (int)((long long)nc * k / pc),
                                             (int)((long long)nc * (k + 1) / pc), pc == 1 ? -1 : t);
                        uitems[j] = make_int2(off, pc);
                    }
                }
            }
            run += __reduce_add_sync(0xffffffffu, pc);
        }
        __syncwarp();
        if (run <= slots || share == 0) break;            // share 0: one piece per unit
        share = iter == 4 ? 0 : max(0, share - (run - slots));
    }
    return min(kMaxPieces, run > c ? (run - c + grid - 1) / grid : 0);
}

template <int D, int NT, bool TWO_TERM>
__global__ void __launch_bounds__(kStepThreads, 2)
    quest_step_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const StepParams p) {
    using S = DecShape<D, NT>;
    using SS = StepShape<D, NT>;
    constexpr int NS = SS::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* ring = base;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * SS::kStageBytes);
    uint64_t* empty = full + NS;
    uint64_t* planbar = empty + NS;                            // the pieces (+ 8 bytes pad)
    uint64_t* pready = planbar + 2;                            // [kMaxPieces] view rows written
    int* stage_ntok = reinterpret_cast<int*>(pready + kMaxPieces);
    int* misc = stage_ntok + NS;                               // 64 ints
    volatile int* abort_flag = misc;                           // [0]
    // [1] last-piece flag of the merge, [3] last CTA, [4] score slices,
    // [5] pieces, [6] top-k in the union area
    int4* pitem = reinterpret_cast<int4*>(misc + 64);          // [kMaxPieces]
    int2* pseq = reinterpret_cast<int2*>(pitem + kMaxPieces);  // [kMaxPieces] held, budget
    int2* puit = pseq + kMaxPieces;                            // [kMaxPieces]
    int4* sitem = reinterpret_cast<int4*>(puit + kMaxPieces);  // [kMaxScoreItems] consumers'
    int4* psitem = sitem + kMaxScoreItems;                     // [kMaxScoreItems] producer's
    // the union area, in turn: the query coefficients, the top-k, the merge
    uint8_t* uni = base + p.off_union;
    float* coef = reinterpret_cast<float*>(uni);               // [H][2][D]
    float* merge = reinterpret_cast<float*>(uni);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.kv.num_kv_heads, stride = p.kv.max_pages_per_seq;
    const int cap = stride * kPage;
    const bool pending = p.k_new != nullptr;
    const int segs = D / 8;
    // (ctx_len, budget) of sequence `lane` (producer) or `threadIdx.x`
    // (consumers), loaded before anything waits on them
    const int vb = warp == kProducerWarp ? lane : static_cast<int>(threadIdx.x);
    const int2 v = vb < p.batch ? make_int2(p.kv.ctx_len[vb], p.budget[vb]) : make_int2(0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&planbar[0], 1);
        for (int j = 0; j < kMaxPieces; ++j) mbar_init(&pready[j], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
        }
        const int nscore = my_slices(p, lane, v, psitem);
        uint32_t seq = 0;
        // the score slices: each one contiguous block of summaries, 1-D bulk copies
        for (int i = 0; i < nscore; ++i) {
            const int4 it = psitem[i];
            const int64_t bytes = (int64_t)(it.z - it.y) * H * SS::kSumBytes;
            const uint8_t* src = static_cast<const uint8_t*>(p.kv.meta) +
                                 ((int64_t)it.x * stride + it.y) * H * SS::kSumBytes;
            const int nst = static_cast<int>((bytes + SS::kStageBytes - 1) / SS::kStageBytes);
            if (lane == 0) {
                for (int j = 0; j < nst; ++j) {
                    const uint32_t sq = seq + j;
                    const int s = sq % NS;
                    // the ring's first fill: two stages, then the rest once the
                    // first has landed.  Every block asking for its whole ring
                    // at once had each block's first stage land only with the
                    // rest (~6 us after the first copy); this way the scoring
                    // warps start ~1.2 us earlier and the step ends ~1.5 us
                    // earlier on 16 x 32K.
                    if (sq == kFirstFill && !*abort_flag && !mbar_wait(&full[0], 0, abort_flag))
                        give_up(p, abort_flag);
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
        }
        // the decode pieces, each once the consumers have written its view
        // rows (and the new token's row)
        if (lane == 0 && !*abort_flag && !mbar_wait(&planbar[0], 0, abort_flag)) give_up(p, abort_flag);
        __syncwarp();
        const int npieces = *abort_flag ? 0 : misc[5];
        const uint64_t kv_policy = l2_evict_first();
        for (int j = 0; j < npieces; ++j) {
            if (lane == 0 && !*abort_flag && !mbar_wait(&pready[j], 0, abort_flag))
                give_up(p, abort_flag);
            __syncwarp();
            const int4 it = pitem[j];
            const int u = it.x, c0 = it.y, c1 = it.z;
            const int ntok = seq_vals(pseq[j].x, pseq[j].y, cap, pending).tokens;
            const int32_t* crow = p.view.chunk_row + (int64_t)u * p.view.max_chunks;
            int row_next = c0 + lane < c1 ? __ldcg(crow + c0 + lane) : -1;
            for (int cb = c0; cb < c1; cb += 32) {
                const int row_l = row_next;
                row_next = cb + 32 + lane < c1 ? __ldcg(crow + cb + 32 + lane) : -1;
                const int nb = min(32, c1 - cb);
                // four chunks per iteration: chunk t = lane / 4 of the group is
                // led by lane 4t (waits for its stage, arms its barrier); then
                // lanes 4t..4t+3 issue that chunk's K and V boxes together
                for (int j0 = 0; j0 < nb; j0 += 4) {
                    const int t = lane >> 2, qq = lane & 3;
                    const int jj = j0 + t;
                    const bool mine = t < 4 && jj < nb;
                    const int row = __shfl_sync(0xffffffffu, row_l, min(jj, 31));
                    const uint32_t sq = seq + t;
                    const int s = sq % NS;
                    int go = 0;
                    if (mine && qq == 0) {
                        const int c = cb + jj;
                        if (!*abort_flag && !mbar_wait(&empty[s], ((sq / NS) & 1) ^ 1, abort_flag))
                            give_up(p, abort_flag);
                        int cnt = min(kPage, ntok - c * kPage);
                        if (!*abort_flag && (row < 0 || (int64_t)row >= p.total_rows)) {
                            flag(p.status, SE_DEV_BAD_INDEX);
                            cnt = 0;
                        }
                        stage_ntok[s] = cnt;
                        go = cnt > 0 && !*abort_flag;
                        if (go)
                            mbar_arrive_expect_tx(&full[s], S::kStageBytes);
                        else
                            mbar_arrive(&full[s]);
                    }
                    go = __shfl_sync(0xffffffffu, go, lane & ~3);
                    if (mine && go && qq < 2 * S::kBoxes) {
                        uint8_t* dst = ring + s * S::kStageBytes + (qq & 1) * S::kChunkBytes +
                                       (qq >> 1) * 2048;
                        tma_load_2d_hint(dst, (qq & 1) ? &tv : &tk, &full[s], 64 * (qq >> 1), row,
                                         kv_policy);
                    }
                    seq += min(4, nb - j0);
                }
            }
        }
        // Drain: every copy issued by this CTA lands before the CTA may exit.
        if (lane == 0) {
            const uint32_t first = seq > (uint32_t)NS ? seq - NS : 0;
            volatile int never = 0;
            for (uint32_t q2 = first; q2 < seq; ++q2)
                mbar_wait(&full[q2 % NS], (q2 / NS) & 1, &never);
        }
    } else {
        // -------------------------------- consumers --------------------------------
        const int ctid = threadIdx.x;
        // the plans, while the first summaries are on their way: the score
        // slices by warp 0, the decode pieces by warp 1 (published to the
        // producer through the plan barrier)
        if (warp == 0) {
            const int n = my_slices(p, lane, v, sitem);
            if (lane == 0) misc[4] = n;
        } else if (warp == 1) {
            const int in_area = keys_in_area(p, lane);
            const int n = plan_decode(p, lane, pitem, puit);
            __syncwarp();
            for (int j = lane; j < n; j += 32) {
                const int b = pitem[j].x / H;
                pseq[j] = make_int2(p.kv.ctx_len[b], p.budget[b]);
            }
            __syncwarp();
            if (lane == 0) {
                misc[5] = n;
                misc[6] = in_area;
                mbar_arrive(&planbar[0]);
            }
            // the block-table rows the pieces' view rows will read, into L2
            // while the summaries stream
            for (int j = 0; j < n; ++j) {
                const int b = pitem[j].x / H;
                const int np = min(stride, seq_vals(pseq[j].x, pseq[j].y, cap, pending).n);
                const int32_t* row = p.kv.block_table + (int64_t)b * stride;
                for (int e = lane * 32; e < np; e += 32 * 32) prefetch_l2(row + e);
            }
        }
        if (blockIdx.x == 0) {
            for (int b = ctid; b < p.batch; b += kCThreads) {
                const int held = b == ctid ? v.x : p.kv.ctx_len[b];
                if (held < 0 || held > cap) flag(p.status, SE_DEV_BAD_LENGTH);
                else if (pending && held >= cap) flag(p.status, SE_DEV_CAPACITY);
            }
        }
        consumer_bar();
        const int nscore = misc[4];
        const bool regs = coef_in_regs<D>(H);
        const int lgH = 31 - __clz(H);
        uint32_t seq = 0;
        int folded = -1;
        float cr[32];
        for (int si = 0; si < nscore; ++si) {
            const int4 it = sitem[si];
            const int b = it.x;
            if (b != folded) {
                consumer_bar();                          // the previous reads of the union area
                step_fold<D>(p, b, coef, ctid);
                consumer_bar();
                if (regs) coef_regs<D>(coef, H, lane, cr);
                folded = b;
            }
            const int nsum_all = (it.z - it.y) * H;
            const int nst = (nsum_all + SS::kSumsPerStage - 1) / SS::kSumsPerStage;
            for (int j = 0; j < nst; ++j, ++seq) {
                if ((seq % kConsumerWarps) != (uint32_t)warp) continue;
                const int s = seq % NS;
                if (lane == 0 && !*abort_flag && !mbar_wait(&full[s], (seq / NS) & 1, abort_flag))
                    give_up(p, abort_flag);
                __syncwarp();
                if (!*abort_flag) {
                    const uint8_t* stg = ring + s * SS::kStageBytes;
                    const int ns = min(SS::kSumsPerStage, nsum_all - j * SS::kSumsPerStage);
                    if (regs) {
                        const int t0 = j * SS::kSumsPerStage, sl = lane / (D / 16);
                        uint32_t* krow = p.keys + ((int64_t)b * H + (sl & (H - 1))) * p.kstride +
                                         it.y + (t0 >> lgH) + (sl >> lgH);
                        score_stage_regs<D, SS::kSumsPerStage>(stg, ns, krow, lgH, cr, lane);
                    } else
                        score_stage<D>(p, stg, ns, j * SS::kSumsPerStage, b, it.y, coef, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // every key of the slice is written: publish the slice's pages
            consumer_bar();
            if (ctid == 0) {
                __threadfence();
                atomicAdd(p.seq_scored + b, it.z - it.y);
            }
        }
        const int npieces = misc[5];
        const bool in_area = misc[6] != 0;
        // the top-k of piece j (its ranks of the selection, its view rows, the
        // new token's row), then the producer is released for it
        auto select_piece = [&](int j, uint8_t* area) {
            const int4 it = pitem[j];
            const int u = it.x, c0 = it.y, c1 = it.z;
            const int b = u / H, h = u % H;
            const SeqVals sv = seq_vals(pseq[j].x, pseq[j].y, cap, pending);
            const bool app = sv.room && c1 == sv.chunks;     // the piece of the last page
            AppendRegs ar;
            if (app && ctid < segs) append_load(p.kv, b, h, sv.held, p.k_new, p.v_new, ctid, ar);
            const int phys_new = app ? p.kv.block_table[(int64_t)b * stride + sv.held / kPage] : -1;
            consumer_bar();
            if (ctid == 0 && sv.m > 0 && !*abort_flag &&
                !wait_count(p, p.seq_scored + b, sv.m, abort_flag))
                give_up(p, abort_flag);
            consumer_bar();
            const int* spage = piece_select(p, u, sv, c0, c1, area, warp, lane);
            consumer_bar();
            view_rows(p, u, c0, c1, spage, ctid, kCThreads);
            if (c0 == 0 && ctid == 0) {
                p.n_sel[u] = sv.chunks;
                p.view.n_tokens[u] = sv.tokens;
            }
            if (app && ctid < segs) {
                if (phys_new >= 0 && phys_new < p.kv.num_pages) {
                    append_store(p.kv, b, h, sv.held, phys_new, ctid, ar);
                    fence_proxy_async_global();              // read next by TMA (async proxy)
                } else if (ctid == 0) {
                    flag(p.status, SE_DEV_BAD_INDEX);
                }
            }
            consumer_bar();
            if (ctid == 0) mbar_arrive(&pready[j]);
        };
        // every selection of the CTA up front, in the union area, while the
        // producer streams the first pieces' chunks; else each one in the idle
        // ring right before its piece
        if (in_area)
            for (int j = 0; j < npieces; ++j) select_piece(j, uni);
        DecOut dout;
        dout.out = p.out;
        dout.out_f32 = p.out_f32;
        dout.lse_out = p.lse_out;
        dout.o_part = p.o_part;
        dout.lse_part = p.lse_part;
        dout.counters = p.counters;
        dout.Hq = p.Hq;
        dout.G = p.G;
        for (int j = 0; j < npieces; ++j) {
            if (!in_area) select_piece(j, ring);
            const int4 it = pitem[j];
            const int u = it.x, c0 = it.y, c1 = it.z;
            const int b = u / H, h = u % H;
            DecState<D, NT> st;
            dec_begin<D, NT>(st, p.q, (int64_t)b * p.Hq + h * p.G, p.G, lane);
            for (int c = c0; c < c1; ++c, ++seq) {
                if ((seq % kConsumerWarps) != (uint32_t)warp) continue;
                const int s = seq % NS;
                const uint32_t ph = (seq / NS) & 1;
                if (!*abort_flag && !mbar_wait(&full[s], ph, abort_flag)) give_up(p, abort_flag);
                const int cnt = *abort_flag ? 0 : stage_ntok[s];
                if (cnt > 0)
                    dec_chunk<D, NT, TWO_TERM>(st, ring + s * S::kStageBytes, cnt, lane, p.scale,
                                               p.scale_log2, p.G, nullptr, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            consumer_bar();                              // the union area -> merge
            dec_finish<D, NT>(st, merge, misc + 1, dout, b, h, u, it.w, puit[j], warp, lane);
        }
    }
    // ---- end: the last CTA commits the lengths and clears the control words ----
    __syncthreads();
    if (threadIdx.x == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(p.sync)
                     : "memory");
        misc[3] = old == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (misc[3]) {
        const bool aborted = *reinterpret_cast<const volatile int*>(p.sync + 1) != 0;
        for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
            if (pending && !aborted) {
                const int held = __ldcg(p.kv.ctx_len + b);
                if (held >= 0 && held < cap) {
                    const int phys = p.kv.block_table[(int64_t)b * stride + held / kPage];
                    if (phys >= 0 && phys < p.kv.num_pages) p.kv.ctx_len[b] = held + 1;
                }
            }
            p.seq_scored[b] = 0;
        }
        for (int u = threadIdx.x; u < p.units; u += blockDim.x) p.counters[u] = 0;
        __syncthreads();
        if (threadIdx.x == 0) {
            p.sync[1] = 0;
            p.sync[0] = 0;
        }
    }
}

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct StepWs {
    int* status;
    int* sync;
    int* seq_scored;
    int* counters;
    uint32_t* keys;
    float* lse_part;
    float* o_part;
};

// Workspace layout.  Every word the kernel needs at zero when it starts -- the
// finished-CTA count and the abort word, the per-sequence scored counters and
// the per-unit arrival counters -- sits in one control block right after the
// 256-byte header, each array at an offset fixed by the largest supported
// shape (kStepMaxBatch sequences, kStepMaxUnits units), so that no call's
// zero words ever land on another call's data; every call leaves them at zero.
size_t step_ctl_bytes() {
    return 256 + 256 + a256((size_t)kStepMaxBatch * sizeof(int)) +
           a256((size_t)kStepMaxUnits * sizeof(int));
}

int key_stride(int max_pages) { return (max_pages + 3) & ~3; }

StepWs step_ws_carve(void* ws, int batch, int H, int G, int max_pages, int max_splits) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t units = (size_t)batch * H, slots = units * max_splits;
    StepWs w;
    w.status = reinterpret_cast<int*>(base);
    size_t off = 256;
    w.sync = reinterpret_cast<int*>(base + off);
    off += 256;
    w.seq_scored = reinterpret_cast<int*>(base + off);
    off += a256((size_t)kStepMaxBatch * sizeof(int));
    w.counters = reinterpret_cast<int*>(base + off);
    off += a256((size_t)kStepMaxUnits * sizeof(int));
    w.keys = reinterpret_cast<uint32_t*>(base + off);
    off += a256(units * key_stride(max_pages) * sizeof(uint32_t));
    w.lse_part = reinterpret_cast<float*>(base + off);
    off += a256(slots * G * sizeof(float));
    w.o_part = reinterpret_cast<float*>(base + off);
    return w;
}

// Dynamic shared memory: the stage ring, the small areas, then the union area
// (the query coefficients, the top-k, the decode merge area).
template <int D, int NT>
size_t step_smem(int H, int* off_union) {
    using SS = StepShape<D, NT>;
    const size_t ring = (size_t)SS::kStages * SS::kStageBytes;
    const size_t uni_off = (ring + SS::kFixed + 15) & ~static_cast<size_t>(15);
    const size_t uni = std::max({(size_t)DecShape<D, NT>::kMergeFloats * 4, (size_t)H * 2 * D * 4,
                                 (size_t)kAreaBytes});
    if (off_union) *off_union = static_cast<int>(uni_off);
    return 1024 + uni_off + uni;
}

template <int D, int NT, bool TWO>
cudaError_t run_step(const CUtensorMap& tk, const CUtensorMap& tv, StepParams p, cudaStream_t s) {
    auto kern = quest_step_kernel<D, NT, TWO>;
    const size_t smem = step_smem<D, NT>(p.kv.num_kv_heads, &p.off_union);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStepThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = std::min(2048, num_sms() * per_sm);
    // a CTA's pieces and score slices must fit its lists
    if ((p.units + grid - 1) / grid > kMaxPieces || (p.batch + grid - 1) / grid > kMaxScoreItems)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;     // every CTA resident: the waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

size_t quest_step_ws_bytes(int batch, int H, int G, int D, int max_pages, int max_splits) {
    (void)D;
    const size_t units = (size_t)batch * H, slots = units * max_splits;
    return step_ctl_bytes() + a256(units * key_stride(max_pages) * sizeof(uint32_t)) +
           a256(slots * G * sizeof(float)) + a256(slots * G * (size_t)D * sizeof(float));
}

size_t quest_step_smem_bytes(int H, int D, int G) {
    const int NT = G > 8 ? 2 : 1;
    if (D == 64) return NT == 1 ? step_smem<64, 1>(H, nullptr) : step_smem<64, 2>(H, nullptr);
    return NT == 1 ? step_smem<128, 1>(H, nullptr) : step_smem<128, 2>(H, nullptr);
}

// A unit with more than kAreaKeys candidate pages keeps its keys in the idle
// stage ring, after the top-k's histogram and small ints.
int quest_step_max_pages(int D, int G) {
    const size_t ring =
        D == 64 ? (size_t)StepShape<64, 1>::kStages * StepShape<64, 1>::kStageBytes
        : G > 8 ? (size_t)StepShape<128, 2>::kStages * StepShape<128, 2>::kStageBytes
                : (size_t)StepShape<128, 1>::kStages * StepShape<128, 1>::kStageBytes;
    // the largest m with key_slots(m) words after the histogram and small ints
    size_t words = (ring - kSelectBytes) / 4, m = words * 32 / 33;
    while (m > 0 && (size_t)key_slots(static_cast<int>(m)) > words) --m;
    return static_cast<int>(std::min<size_t>(16384, m + 1));
}

cudaError_t launch_quest_step(const se_paged_kv& kv, const void* k_new, const void* v_new,
                              const void* q, int batch, int num_q_heads, const int32_t* budget,
                              float scale, int out_dtype, int max_splits,
                              unsigned long long wait_ns, int32_t* sel_pages, int32_t* n_sel,
                              const se_view& view, void* out, float* lse, void* ws,
                              cudaEvent_t ev_begin, cudaEvent_t ev_end, cudaStream_t s) {
    const int H = kv.num_kv_heads, D = kv.head_dim, G = num_q_heads / H;
    const int units = batch * H;
    if (units == 0) return cudaSuccess;
    const int64_t total_rows = (int64_t)kv.num_pages * H * kPage;
    CUtensorMap tk, tv;
    if (!encode_rows_map(&tk, kv.k, total_rows, D) || !encode_rows_map(&tv, kv.v, total_rows, D))
        return cudaErrorInvalidValue;
    const StepWs w = step_ws_carve(ws, batch, H, G, kv.max_pages_per_seq, max_splits);

    StepParams p;
    p.kv = kv;
    p.q = static_cast<const uint16_t*>(q);
    p.Hq = num_q_heads;
    p.G = G;
    p.batch = batch;
    p.units = units;
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
    p.kstride = key_stride(kv.max_pages_per_seq);
    p.seq_scored = w.seq_scored;
    p.counters = w.counters;
    p.sync = w.sync;
    p.o_part = w.o_part;
    p.lse_part = w.lse_part;
    p.max_splits = max_splits;
    p.off_union = 0;
    p.total_rows = total_rows;
    p.wait_ns = wait_ns;
    p.status = w.status;
    const int NT = G > 8 ? 2 : 1;

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
        e = NT == 1 ? (two ? run_step<64, 1, true>(tk, tv, p, s) : run_step<64, 1, false>(tk, tv, p, s))
                    : (two ? run_step<64, 2, true>(tk, tv, p, s) : run_step<64, 2, false>(tk, tv, p, s));
    } else {
        e = NT == 1 ? (two ? run_step<128, 1, true>(tk, tv, p, s) : run_step<128, 1, false>(tk, tv, p, s))
                    : (two ? run_step<128, 2, true>(tk, tv, p, s) : run_step<128, 2, false>(tk, tv, p, s));
    }
    if (e != cudaSuccess) return e;
    if (ev_end && (e = record(ev_end)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace se
