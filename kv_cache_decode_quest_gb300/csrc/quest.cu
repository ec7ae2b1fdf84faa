// Quest query-aware page selection: per-page upper-bound scores from the
// channel-wise key min/max summaries, an exact per-KV-head top-k under a token
// budget (last page forced, ties to the lower page), and the AttentionView of
// the selected pages.
//
// Quest selects pages by the query while the full history stays resident
// (tokendh.com article on SparseEngine, section "历史太长,会撑爆什么"); the view
// exposes the selected positions to the attention kernel in one format
// ("SparseEngine：稀疏优先推理引擎", section "方法 / 关键模块").
//
// Bound: U[p] = sum_g sum_d max(q_g[d]*kmin[p,d], q_g[d]*kmax[p,d]).  Because
// kmin <= kmax, max(q*kmin, q*kmax) is q*kmax for q >= 0 and q*kmin for q < 0,
// so U[p] = sum_d Q+[d]*kmax[p,d] + Q-[d]*kmin[p,d] with Q+ = sum_g max(q_g,0)
// and Q- = sum_g min(q_g,0): one 2*D-long dot product per (page, KV head),
// which keeps the scoring a pure stream over the 2*D*2-byte page summaries.
#include "append.cuh"
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kSelWarps = 8;               // scoring warps
constexpr int kSelThreads = (kSelWarps + 1) * 32;   // + the copy warp
constexpr int kSelChunk = 16384;           // bytes per ring stage
constexpr int kSelStages = 4;
constexpr int kSelMinBlocks = 2;           // resident scoring CTAs per SM
constexpr int kTopkThreads = 256;
constexpr size_t kSelSmemFixed = 128 /* alignment slack */ + (size_t)kSelStages * kSelChunk +
                                 (size_t)kSelStages * 16 /* full, empty */ + 16 /* abort */;

template <int D>
struct SelShape {
    static constexpr int kSumBytes = 2 * D * 2;        // one (page, head) summary: kmin then kmax
};

__device__ __forceinline__ int clamp_ctx(int ctx, int cap, int* status, bool report) {
    if (ctx < 0 || ctx > cap) {
        if (report) flag(status, SE_DEV_BAD_LENGTH);
        return ctx < 0 ? 0 : cap;
    }
    return ctx;
}

// grid (CTAs per sequence, batch), one resident wave.  The page summaries of a
// sequence are stored in logical page order, all KV heads of a page together,
// so a CTA's range of candidate pages is one contiguous block of bytes: its
// copy warp streams the block through a ring of shared-memory stages with 1-D
// bulk copies (mbarrier completion, no block-table indirection) while the
// scoring warps first fold the queries into Q-/Q+ and then turn each
// (page, head) summary into U = sum_d Q-[d]*kmin[d] + Q+[d]*kmax[d] and an
// order-preserving key in keys[unit][page].
template <int D, int VPL, bool REG>
__global__ void __launch_bounds__(kSelThreads, kSelMinBlocks)
    quest_score_kernel(se_paged_kv kv, const uint16_t* __restrict__ q, int Hq,
                       const int32_t* __restrict__ budget, uint32_t* __restrict__ keys_ws,
                       int pending, int32_t* __restrict__ tickets, int* status) {
    using S = SelShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                               ~static_cast<uintptr_t>(127));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kSelStages * kSelChunk);
    uint64_t* empty = full + kSelStages;
    volatile int* abort_flag = reinterpret_cast<int*>(empty + kSelStages);
    float* coef = reinterpret_cast<float*>(empty + kSelStages) + 4;   // [H][2][D]: Q- then Q+
    const int b = blockIdx.y, x = blockIdx.x;
    const int H = kv.num_kv_heads, G = Hq / H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    // The query loads of the Q-/Q+ fold are the first memory requests of the
    // kernel, ahead of every CTA's stage copies.  lane = g * kNdv + dv loads 8
    // query values of group member g for d-block (task % tph) * kNdv + dv.
    const int kNdv = 32 / G;                              // d-blocks of 8 per warp task
    const int tph = (D / 8 + kNdv - 1) / kNdv;            // warp tasks per head
    constexpr int kQPre = 4;                              // tasks per warp loaded up front
    uint4 qv[kQPre];
    auto q_load = [&](int task) {
        const int h = task / tph, d8 = (task % tph) * kNdv + lane % kNdv, g = lane / kNdv;
        return d8 < D / 8 ? *reinterpret_cast<const uint4*>(q + ((int64_t)b * Hq + h * G + g) * D + d8 * 8)
                          : make_uint4(0, 0, 0, 0);
    };
#pragma unroll
    for (int i = 0; i < kQPre; ++i) {
        const int task = warp + i * kSelWarps;
        qv[i] = (warp < kSelWarps && task < H * tph) ? q_load(task) : make_uint4(0, 0, 0, 0);
    }
    const int stride = kv.max_pages_per_seq;
    int ctx = clamp_ctx(kv.ctx_len[b], stride * kPage, status, threadIdx.x == 0 && x == 0);
    // a pending append (written by the top-k kernel) counts when it fits; its
    // page is the last one, which is never scored
    if (pending) {
        if (ctx < stride * kPage) ++ctx;
        if (x == 0 && tid == 0) tickets[b] = 0;
    }
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    if (n <= k) return;                                   // all pages selected: nothing to score
    const int m = n - 1;                                  // candidates: pages 0..n-2
    const int per = (m + gridDim.x - 1) / gridDim.x;
    const int p_begin = x * per, p_end = min(m, p_begin + per);
    if (p_begin >= p_end) return;
    const int64_t bytes = (int64_t)(p_end - p_begin) * H * S::kSumBytes;
    const uint8_t* src = static_cast<const uint8_t*>(kv.meta) +
                         ((int64_t)b * stride + p_begin) * H * S::kSumBytes;
    const int nchunks = static_cast<int>((bytes + kSelChunk - 1) / kSelChunk);
    if (warp == kSelWarps) {
        // ------------------------------ copy warp ------------------------------
        // It initialises the barriers, releases the scoring warps (named barrier
        // 2, arrive only) and starts copying without waiting for them.
        if (lane == 0) {
            for (int s = 0; s < kSelStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kSelWarps);
            }
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"r"(kSelThreads) : "memory");
        if (lane == 0) {
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kSelStages;
                const uint32_t ph = (c / kSelStages) & 1;
                if (!*abort_flag && !mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    flag(status, SE_DEV_TIMEOUT);
                }
                const uint32_t sz = static_cast<uint32_t>(min(static_cast<int64_t>(kSelChunk), bytes - (int64_t)c * kSelChunk));
                if (!*abort_flag) {
                    mbar_arrive_expect_tx(&full[s], sz);
                    bulk_g2s(ring + s * kSelChunk, src + (int64_t)c * kSelChunk, sz, &full[s]);
                } else {
                    mbar_arrive(&full[s]);
                }
            }
            // every copy lands before the CTA may exit
            const int first = max(0, nchunks - kSelStages);
            volatile int never = 0;
            for (int c = first; c < nchunks; ++c)
                mbar_wait(&full[c % kSelStages], (c / kSelStages) & 1, &never);
        }
        return;
    }

    // ------------------------------ scoring warps ------------------------------
    asm volatile("bar.sync 2, %0;" ::"r"(kSelThreads) : "memory");   // barriers initialised
    // Q- / Q+ per (head, d): the sums over the group are xor-shuffles across
    // the lanes of one d-block.
    {
        const int g = lane / kNdv, dv = lane % kNdv;
        int i = 0;
        for (int task = warp; task < H * tph; task += kSelWarps, ++i) {
            const int h = task / tph, d8 = (task % tph) * kNdv + dv;
            uint4 v = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < kQPre; ++j)
                if (i == j) v = qv[j];
            if (i >= kQPre) v = q_load(task);
            const uint32_t a4[4] = {v.x, v.y, v.z, v.w};
            float lo[8], hi[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float f0 = bf_lo(a4[i]), f1 = bf_hi(a4[i]);
                lo[2 * i] = fminf(f0, 0.f);
                lo[2 * i + 1] = fminf(f1, 0.f);
                hi[2 * i] = fmaxf(f0, 0.f);
                hi[2 * i + 1] = fmaxf(f1, 0.f);
            }
            for (int o = kNdv; o < 32; o <<= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    lo[e] += __shfl_xor_sync(0xffffffffu, lo[e], o);
                    hi[e] += __shfl_xor_sync(0xffffffffu, hi[e], o);
                }
            }
            if (g == 0 && d8 < D / 8) {
                float4* cl = reinterpret_cast<float4*>(coef + (h * 2) * D + d8 * 8);
                float4* ch = reinterpret_cast<float4*>(coef + (h * 2 + 1) * D + d8 * 8);
                cl[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
                cl[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
                ch[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
                ch[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kSelWarps * 32) : "memory");
    // Each summary is read by kLps lanes, kVpl 16-byte vectors each; vector j
    // of lane `sub` is vector j*kLps + sub of the summary (conflict-free
    // shared-memory reads).  One warp-wide read covers kR summaries.
    constexpr int kU4 = D / 4;                            // 16-byte vectors per summary
    constexpr int kLps = kU4 / VPL;
    constexpr int kR = 32 / kLps;
    constexpr int kPerChunk = kSelChunk / S::kSumBytes;   // summaries per full stage
    const int sub = lane % kLps, slot = lane / kLps;
    // vector v of a summary multiplies coef[h][0][v*8..] (v < D/8: kmin by Q-)
    // or coef[h][1][(v-D/8)*8..] (kmax by Q+): coef + h*2*D + v*8 in both cases
    float cr[REG ? VPL * 8 : 1];
    if (REG) {
        const int h = slot % H;                           // fixed: kR is a multiple of H
#pragma unroll
        for (int j = 0; j < VPL; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) cr[REG ? j * 8 + e : 0] = coef[h * 2 * D + (j * kLps + sub) * 8 + e];
    }
    int32_t abort_seen = 0;
    for (int c = 0; c < nchunks; ++c) {
        const int s = c % kSelStages;
        const uint32_t ph = (c / kSelStages) & 1;
        if (lane == 0) {
            abort_seen = *abort_flag;
            if (!abort_seen && !mbar_wait(&full[s], ph, abort_flag)) {
                *abort_flag = 1;
                flag(status, SE_DEV_TIMEOUT);
                abort_seen = 1;
            }
        }
        abort_seen = __shfl_sync(0xffffffffu, abort_seen, 0);
        const int nsum = static_cast<int>(min(static_cast<int64_t>(kSelChunk),
                                              bytes - (int64_t)c * kSelChunk)) /
                         S::kSumBytes;
        if (!abort_seen) {
            const uint8_t* st = ring + s * kSelChunk;
            for (int t0 = warp * kR; t0 < nsum; t0 += kSelWarps * kR) {
                const int tl = t0 + slot;                  // summary within the stage
                const int t = c * kPerChunk + tl;          // summary within the CTA's range
                const int h = t % H, pl = t / H;
                float acc = 0.f;
                if (tl < nsum) {
                    const uint4* sv = reinterpret_cast<const uint4*>(st + tl * S::kSumBytes);
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const uint4 w = sv[j * kLps + sub];
                        const uint32_t a4[4] = {w.x, w.y, w.z, w.w};
                        const float* cf = coef + h * 2 * D + (j * kLps + sub) * 8;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float c0 = REG ? cr[REG ? j * 8 + 2 * i : 0] : cf[2 * i];
                            const float c1 = REG ? cr[REG ? j * 8 + 2 * i + 1 : 0] : cf[2 * i + 1];
                            acc = fmaf(c0, bf_lo(a4[i]), acc);
                            acc = fmaf(c1, bf_hi(a4[i]), acc);
                        }
                    }
                }
#pragma unroll
                for (int o = kLps / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (sub == 0 && tl < nsum)
                    keys_ws[((int64_t)b * H + h) * stride + p_begin + pl] = float_key(acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// The max-aggregation variant of the bound (flag SE_AGG_MAX):
//   U[p] = max_g sum_d max(q_g[d]*kmin[p,d], q_g[d]*kmax[p,d])
// is G dot products of length 2*D per (page, KV head) instead of one, so it is
// computed without the shared-memory ring: grid (CTAs per sequence, batch),
// 8 warps per CTA; every warp of a sequence owns one KV head h (8 % H == 0,
// G <= 8) and a stride of its candidate pages, and each lane keeps, for the 8
// channels of its 16-byte vector of a summary, the coefficients of all G query
// heads in registers (min(q, 0) for the kmin vectors, max(q, 0) for the kmax
// ones).  A summary is read by kVec = D/4 lanes (one coalesced 16-byte load
// each, kU summaries in flight per lane); the G partial sums are reduced over
// those lanes by a halving butterfly (each level keeps half of the values:
// G - 1 shuffles, then the plain levels), and their maximum over g (the lanes
// of the G partial results) is the page's key.
template <int D, int G>
__global__ void __launch_bounds__(256)
    quest_score_max_kernel(se_paged_kv kv, const uint16_t* __restrict__ q, int Hq,
                           const int32_t* __restrict__ budget, uint32_t* __restrict__ keys_ws,
                           int pending, int32_t* __restrict__ tickets, int* status) {
    constexpr int kVec = D / 4;                           // 16-byte vectors per summary
    constexpr int kSpr = 32 / kVec;                       // summaries per warp-wide read
    constexpr int kU = 8;                                 // reads in flight per lane
    static_assert(G <= kVec, "the halving reduction needs G <= lanes per summary");
    const int b = blockIdx.y, x = blockIdx.x;
    const int H = kv.num_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int stride = kv.max_pages_per_seq;
    int ctx = clamp_ctx(kv.ctx_len[b], stride * kPage, status, threadIdx.x == 0 && x == 0);
    if (pending) {
        if (ctx < stride * kPage) ++ctx;
        if (x == 0 && threadIdx.x == 0) tickets[b] = 0;
    }
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    if (n <= k) return;
    const int m = n - 1;
    const int gw = x * 8 + warp, W = gridDim.x * 8;
    const int h = gw % H, wp = gw / H, WP = W / H;
    const int v = lane % kVec, sub = lane / kVec;
    const bool upper_part = v >= D / 8;                   // a kmax vector
    const int d0 = (v % (D / 8)) * 8;
    float c[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 w = *reinterpret_cast<const uint4*>(q + ((int64_t)b * Hq + h * G + g) * D + d0);
        const uint32_t a4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float f0 = bf_lo(a4[e]), f1 = bf_hi(a4[e]);
            c[g][2 * e] = upper_part ? fmaxf(f0, 0.f) : fminf(f0, 0.f);
            c[g][2 * e + 1] = upper_part ? fmaxf(f1, 0.f) : fminf(f1, 0.f);
        }
    }
    const uint4* M = static_cast<const uint4*>(kv.meta) + (int64_t)b * stride * H * kVec;
    const int slots = (m + kSpr - 1) / kSpr;              // page groups of one warp-wide read
    uint32_t* keys = keys_ws + ((int64_t)b * H + h) * stride;
    for (int j0 = wp; j0 < slots; j0 += WP * kU) {
        uint4 xv[kU];
#pragma unroll
        for (int t = 0; t < kU; ++t) {
            const int page = (j0 + t * WP) * kSpr + sub;
            xv[t] = page < m ? M[((int64_t)page * H + h) * kVec + v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int t = 0; t < kU; ++t) {
            const int page = (j0 + t * WP) * kSpr + sub;
            const uint32_t a4[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
            float acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s0 = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s0 = fmaf(c[g][2 * e], bf_lo(a4[e]), s0);
                    s0 = fmaf(c[g][2 * e + 1], bf_hi(a4[e]), s0);
                }
                acc[g] = s0;
            }
            // halving butterfly over the kVec lanes of the summary
            int off = kVec / 2;
#pragma unroll
            for (int lvl = G; lvl > 1; lvl >>= 1) {
                const bool up = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < lvl / 2; ++i) {
                    const float send = up ? acc[i] : acc[i + lvl / 2];
                    const float keep = up ? acc[i + lvl / 2] : acc[i];
                    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
                off >>= 1;
            }
#pragma unroll
            for (int o = off; o >= 1; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
            // acc[0] is one head's bound; the G heads sit on the lanes that
            // differ in the halving bits
            float mx = acc[0];
#pragma unroll
            for (int o = kVec / 2; o >= kVec / G && o >= 1; o >>= 1)
                if (G > 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (v == 0 && page < m) keys[page] = float_key(mx);
        }
    }
}

// Threshold of the top K of m order-preserving keys in shared memory (256
// threads).  Bits above the highest bit in which the largest and smallest key
// differ are common to all keys, so the 11-bit radix digits start there; a pass
// ends the search early when every key of the boundary digit is kept.  On
// return, under *mask: keys above *T are kept, and so are the first *need keys
// equal to *T.
constexpr int kDigitBits = 11, kDigitBins = 1 << kDigitBits;   // 8 bins per thread of 256
__device__ void topk_threshold(const uint32_t* sk, int m, int K, int* hist, int* tmp,
                               uint32_t* red, int* sel, uint32_t* T, uint32_t* mask, int* need) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int i = tid; i < m; i += blockDim.x) {
        const uint32_t k = sk[i];
        lo = min(lo, k);
        hi = max(hi, k);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        red[wid] = lo;
        red[8 + wid] = hi;
    }
    __syncthreads();
    lo = red[0];
    hi = red[8];
#pragma unroll
    for (int w = 1; w < kTopkThreads / 32; ++w) {
        lo = min(lo, red[w]);
        hi = max(hi, red[8 + w]);
    }
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
    while (low > 0) {
        // 11-bit digits: thread t owns bins 2047-8t .. 2040-8t (descending)
        const int w = min(kDigitBits, low), shift = low - w;
        const uint32_t dm = (1u << w) - 1u;
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[tid * 8 + j] = 0;
        __syncthreads();
        for (int i = tid; i < m; i += blockDim.x) {
            const uint32_t k = sk[i];
            if ((k & msk) == prefix) atomicAdd(&hist[(k >> shift) & dm], 1);
        }
        __syncthreads();
        int v8[8], v = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v8[j] = hist[kDigitBins - 1 - (tid * 8 + j)];
            v += v8[j];
        }
        int run = scan256(v, tmp) - v;                    // digits above this thread's
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (run < remaining && run + v8[j] >= remaining) {
                sel[0] = kDigitBins - 1 - (tid * 8 + j);
                sel[1] = run;
                sel[2] = v8[j];
            }
            run += v8[j];
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sel[0]) << shift;
        msk |= dm << shift;
        remaining -= sel[1];
        low = shift;
        const bool whole_bin = sel[2] == remaining;
        __syncthreads();                                  // sel is rewritten by the next pass
        if (whole_bin) break;
    }
    *T = prefix;
    *mask = msk;
    *need = remaining;
}

// One CTA (256 threads) per unit: exact top-(k-1) of pages 0..n-2 by
// (score desc, page asc) -- 11-bit radix passes over the unit's keys
// staged in shared memory -- then the pages in page order (ballots rank them
// inside a warp, a scan over the warps places each warp's run), plus the last
// page, which is always selected and never scored; the AttentionView chunk of
// each selected page is its physical page of this KV head.
__global__ void __launch_bounds__(kTopkThreads)
    quest_topk_kernel(se_paged_kv kv, const int32_t* __restrict__ budget,
                      const uint32_t* __restrict__ keys_ws, int32_t* __restrict__ sel_pages,
                      int32_t* __restrict__ n_sel, se_view view, const uint4* __restrict__ k_new,
                      const uint4* __restrict__ v_new, int32_t* __restrict__ tickets, int* status) {
    extern __shared__ uint32_t skeys[];                   // [max_pages_per_seq] keys, then block table
    __shared__ int hist[kDigitBins];
    __shared__ int tmp[33];
    __shared__ int stat[3];
    __shared__ uint32_t red[16];
    __shared__ int wgt[32], weq[32];
    const int u = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int H = kv.num_kv_heads;
    const int b = u / H, h = u % H;
    const int stride = kv.max_pages_per_seq;
    const int held = clamp_ctx(kv.ctx_len[b], stride * kPage, status, tid == 0 && h == 0);
    // fused append (k_new given): this CTA writes head h's new row at position
    // `held`, the sequence's last CTA to finish commits ctx_len = held + 1
    const bool pending = k_new != nullptr;
    const bool room = pending && held < stride * kPage;
    if (pending && !room && tid == 0 && h == 0) flag(status, SE_DEV_CAPACITY);
    const int ctx = room ? held + 1 : held;
    // the append's loads go out now; its stores come last
    AppendRegs ar;
    const int segs = kv.head_dim / 8;
    if (room && tid < segs) append_load(kv, b, h, held, k_new, v_new, tid, ar);
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    int32_t* bts = reinterpret_cast<int32_t*>(skeys + stride);   // block-table row in shared memory
    const uint32_t* keys = keys_ws + (int64_t)u * stride;
    const int m = n - 1;
    // the block-table row and the candidate keys are staged with all loads
    // of a thread in flight together
    {
        constexpr int kU = 8;
        const int32_t* btr = kv.block_table + (int64_t)b * stride;
        for (int base = tid; base < n; base += kTopkThreads * kU) {
            int32_t bv[kU];
            uint32_t kv2[kU];
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int i = base + j * kTopkThreads;
                bv[j] = i < n ? btr[i] : 0;
                kv2[j] = (i < m && n > k) ? keys[i] : 0u;
            }
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int i = base + j * kTopkThreads;
                if (i < n) bts[i] = bv[j];
                if (i < m && n > k) skeys[i] = kv2[j];
            }
        }
    }
    __syncthreads();
    bool appended = false;
    const int phys_new = room ? bts[held / kPage] : -1;
    if (room) {
        appended = phys_new >= 0 && phys_new < kv.num_pages;
        if (!appended && tid == 0 && h == 0) flag(status, SE_DEV_BAD_INDEX);
    }
    // The ticket is taken as soon as this CTA has read ctx_len (every CTA of
    // sequence b takes one after its read, so the last taker stores the new
    // length after all reads); its result is only used at the end, so the
    // atomic's round trip overlaps the selection.
    int ticket = -1;
    if (pending && tid == 0) {
        __threadfence();
        ticket = atomicAdd(&tickets[b], 1);
    }
    auto commit = [&]() {
        if (appended && tid < segs) append_store(kv, b, h, held, phys_new, tid, ar);
        if (ticket == H - 1) {
            tickets[b] = 0;
            if (appended) kv.ctx_len[b] = held + 1;
        }
    };
    int32_t* sel = sel_pages + (int64_t)u * stride;
    int32_t* crow = view.chunk_row + (int64_t)u * view.max_chunks;
    auto emit = [&](int c, int page) {
        sel[c] = page;
        const int phys = bts[page];
        if (phys >= 0 && phys < kv.num_pages) {
            crow[c] = (phys * H + h) * kPage;
        } else {
            crow[c] = -1;
            flag(status, SE_DEV_BAD_INDEX);
        }
    };
    if (n <= k) {
        for (int c = tid; c < n; c += blockDim.x) emit(c, c);
        if (tid == 0) {
            n_sel[u] = n;
            view.n_tokens[u] = ctx;
        }
        commit();
        return;
    }
    const int K = k - 1;
    if (K > 0) {
        int need_eq = 0;
        uint32_t T = 0, msk = 0;
        topk_threshold(skeys, m, K, hist, tmp, red, stat, &T, &msk, &need_eq);
        // pages in ascending order: warp w owns a contiguous chunk read with a
        // lane stride; ballots rank the kept pages inside the warp and a scan
        // over the warps places each warp's run
        const int nw = blockDim.x >> 5, wid = tid >> 5, lane = tid & 31;
        const int chunk = ((m + nw - 1) / nw + 31) & ~31;
        const int c0 = min(m, wid * chunk), c1 = min(m, c0 + chunk);
        int gt = 0, eq = 0;
        for (int i = c0 + lane; i < c1; i += 32) {
            const uint32_t kk = skeys[i] & msk;
            gt += kk > T;
            eq += kk == T;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            gt += __shfl_xor_sync(0xffffffffu, gt, o);
            eq += __shfl_xor_sync(0xffffffffu, eq, o);
        }
        if (lane == 0) {
            wgt[wid] = gt;
            weq[wid] = eq;
        }
        __syncthreads();
        const int g_l = lane < nw ? wgt[lane] : 0, e_l = lane < nw ? weq[lane] : 0;
        int e_incl = e_l;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, e_incl, o);
            if (lane >= o) e_incl += y;
        }
        const int take_l = max(0, min(e_l, need_eq - (e_incl - e_l)));
        int o_incl = g_l + take_l;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, o_incl, o);
            if (lane >= o) o_incl += y;
        }
        int eq_seen = __shfl_sync(0xffffffffu, e_incl - e_l, wid);
        int out = __shfl_sync(0xffffffffu, o_incl - g_l - take_l, wid);
        const uint32_t lt = (1u << lane) - 1u;
        for (int i0 = c0; i0 < c1; i0 += 32) {
            const int i = i0 + lane;
            const uint32_t kk = i < c1 ? skeys[i] & msk : 0u;
            const bool is_eq = i < c1 && kk == T;
            const uint32_t meq = __ballot_sync(0xffffffffu, is_eq);
            const bool take = (i < c1 && kk > T) || (is_eq && eq_seen + __popc(meq & lt) < need_eq);
            const uint32_t mt = __ballot_sync(0xffffffffu, take);
            if (take) emit(out + __popc(mt & lt), i);
            out += __popc(mt);
            eq_seen += __popc(meq);
        }
    }
    if (tid == 0) {
        emit(K, n - 1);
        n_sel[u] = k;
        view.n_tokens[u] = kPage * (k - 1) + (ctx - kPage * (n - 1));
    }
    commit();
}

}  // namespace

// Workspace: status header | keys [units][max_pages] | append tickets [units]
size_t quest_ws_bytes(int units, int max_pages) {
    return 256 + (((size_t)units * max_pages * sizeof(uint32_t) + 255) & ~(size_t)255) +
           (((size_t)units * sizeof(int32_t) + 255) & ~(size_t)255);
}

cudaError_t launch_quest_select(const se_paged_kv& kv, const void* q, int batch, int num_q_heads,
                                const int32_t* budget, int32_t* sel_pages, int32_t* n_sel,
                                const se_view& view, const void* k_new, const void* v_new,
                                void* ws, int* status, cudaStream_t s, int group_agg) {
    const int units = batch * kv.num_kv_heads;
    if (units == 0) return cudaSuccess;
    uint32_t* keys = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 256);
    int32_t* tickets = reinterpret_cast<int32_t*>(
        static_cast<uint8_t*>(ws) + 256 +
        (((size_t)units * kv.max_pages_per_seq * sizeof(uint32_t) + 255) & ~(size_t)255));
    const int pending = k_new != nullptr;
    // scoring: one resident wave of kSelMinBlocks CTAs per SM shared by the sequences
    const int per_seq = max(1, min((num_sms() * kSelMinBlocks) / batch, kv.max_pages_per_seq));
    dim3 grid(per_seq, batch);
    const int smem = static_cast<int>(kSelSmemFixed) + kv.num_kv_heads * 2 * kv.head_dim * 4;
    // register coefficients when a warp-wide read (4 summaries at D=128 with 4
    // vectors per lane, 8 at D=64) is a multiple of the KV head count
    const int H = kv.num_kv_heads;
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e2 != cudaSuccess) return e2;
        kern<<<grid, kSelThreads, smem, s>>>(kv, static_cast<const uint16_t*>(q), num_q_heads,
                                             budget, keys, pending, tickets, status);
        return cudaSuccess;
    };
    cudaError_t e = cudaSuccess;
    if (group_agg == SE_AGG_MAX) {
        // the max of the group: 8 warps per CTA, a few CTAs per SM
        const int per = max(1, min((num_sms() * 4) / batch, kv.max_pages_per_seq));
        const int G = num_q_heads / H;
        auto gm = [&](auto kern) {
            kern<<<dim3(per, batch), 256, 0, s>>>(kv, static_cast<const uint16_t*>(q), num_q_heads,
                                                 budget, keys, pending, tickets, status);
        };
        if (kv.head_dim == 128) {
            switch (G) {
                case 1: gm(quest_score_max_kernel<128, 1>); break;
                case 2: gm(quest_score_max_kernel<128, 2>); break;
                case 4: gm(quest_score_max_kernel<128, 4>); break;
                default: gm(quest_score_max_kernel<128, 8>); break;
            }
        } else {
            switch (G) {
                case 1: gm(quest_score_max_kernel<64, 1>); break;
                case 2: gm(quest_score_max_kernel<64, 2>); break;
                case 4: gm(quest_score_max_kernel<64, 4>); break;
                default: gm(quest_score_max_kernel<64, 8>); break;
            }
        }
    } else if (kv.head_dim == 128) {
        e = (4 % H == 0) ? go(quest_score_kernel<128, 4, true>) : go(quest_score_kernel<128, 1, false>);
    } else {
        e = (8 % H == 0) ? go(quest_score_kernel<64, 4, true>) : go(quest_score_kernel<64, 1, false>);
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int topk_smem = kv.max_pages_per_seq * 8;
    e = cudaFuncSetAttribute(quest_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             topk_smem);
    if (e != cudaSuccess) return e;
    quest_topk_kernel<<<units, kTopkThreads, topk_smem, s>>>(
        kv, budget, keys, sel_pages, n_sel, view, static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), tickets, status);
    return cudaGetLastError();
}

}  // namespace se
