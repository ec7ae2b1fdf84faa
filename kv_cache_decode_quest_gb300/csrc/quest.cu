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
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kSelWarps = 8;
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSelUnroll = 8;              // 16-byte loads in flight per lane
constexpr int kSelMinBlocks = 4;           // resident scoring CTAs per SM
constexpr int kTopkThreads = 256;

template <int D>
struct SelShape {
    static constexpr int kLpp = D / 4;                 // lanes per page-head summary (512 B at D=128)
    static constexpr int kPpw = 32 / kLpp;             // summaries per warp-wide load
    static constexpr int kPerIter = kSelWarps * kPpw * kSelUnroll;   // summaries per CTA iteration
};

__device__ __forceinline__ int clamp_ctx(int ctx, int cap, int* status, bool report) {
    if (ctx < 0 || ctx > cap) {
        if (report) flag(status, SE_DEV_BAD_LENGTH);
        return ctx < 0 ? 0 : cap;
    }
    return ctx;
}

// grid (CTAs per sequence, batch), 256 threads, one resident wave.  The page
// summaries of a sequence are stored in logical page order, all KV heads of a
// page together, so a CTA's range of candidate pages is one contiguous block
// that it streams with coalesced 16-byte loads (kSelUnroll in flight per lane)
// -- no block-table indirection.  Each (page, head) bound
// U = sum_d Q-[d]*kmin[d] + Q+[d]*kmax[d] becomes an order-preserving key in
// keys[unit][page].
template <int D>
__global__ void __launch_bounds__(kSelThreads, kSelMinBlocks)
    quest_score_kernel(se_paged_kv kv, const uint16_t* __restrict__ q, int Hq,
                       const int32_t* __restrict__ budget, uint32_t* __restrict__ keys_ws,
                       int* status) {
    using S = SelShape<D>;
    extern __shared__ float coef[];                       // [H][2][D]: Q- then Q+
    const int b = blockIdx.y, x = blockIdx.x;
    const int H = kv.num_kv_heads, G = Hq / H;
    const int stride = kv.max_pages_per_seq;
    const int ctx = clamp_ctx(kv.ctx_len[b], stride * kPage, status, threadIdx.x == 0 && x == 0);
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    if (n <= k) return;                                   // all pages selected: nothing to score
    const int m = n - 1;                                  // candidates: pages 0..n-2
    const int per = (m + gridDim.x - 1) / gridDim.x;
    const int p_begin = x * per, p_end = min(m, p_begin + per);
    if (p_begin >= p_end) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < H * D; i += blockDim.x) {
        const int h = i / D, d = i % D;
        float lo = 0.f, hi = 0.f;
        for (int g = 0; g < G; ++g) {
            const uint16_t v = q[((int64_t)b * Hq + h * G + g) * D + d];
            const float f = __uint_as_float(static_cast<uint32_t>(v) << 16);
            lo += fminf(f, 0.f);
            hi += fmaxf(f, 0.f);
        }
        coef[(h * 2) * D + d] = lo;
        coef[(h * 2 + 1) * D + d] = hi;
    }
    __syncthreads();
    const int sub = lane % S::kLpp;                       // 16-byte segment of the summary
    const int items = (p_end - p_begin) * H;              // page-head summaries, page-major
    const uint4* src = static_cast<const uint4*>(kv.meta) +
                       ((int64_t)b * stride + p_begin) * H * (D / 4);
    for (int t0 = warp * S::kPpw * kSelUnroll; t0 < items; t0 += S::kPerIter) {
        uint4 w[kSelUnroll];
#pragma unroll
        for (int j = 0; j < kSelUnroll; ++j) {
            const int t = t0 + j * S::kPpw + lane / S::kLpp;
            w[j] = t < items ? __ldg(src + (int64_t)t * (D / 4) + sub) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kSelUnroll; ++j) {
            const int t = t0 + j * S::kPpw + lane / S::kLpp;
            const int h = t % H, pl = t / H;
            const float* c = coef + h * 2 * D + sub * 8;  // segments 0..D/8-1 = kmin, then kmax
            const uint32_t a[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(c[2 * i], bf_lo(a[i]), acc);
                acc = fmaf(c[2 * i + 1], bf_hi(a[i]), acc);
            }
#pragma unroll
            for (int o = S::kLpp / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (sub == 0 && t < items)
                keys_ws[((int64_t)b * H + h) * stride + p_begin + pl] = float_key(acc);
        }
    }
}

// One CTA (256 threads) per unit: exact top-(k-1) of pages 0..n-2 by
// (score desc, page asc) -- four 8-bit radix passes over the unit's keys
// staged in shared memory -- then the pages in page order (each thread owns a
// contiguous run of candidates: two block scans place them), plus the last
// page, which is always selected and never scored; the AttentionView chunk of
// each selected page is its physical page of this KV head.
__global__ void __launch_bounds__(kTopkThreads)
    quest_topk_kernel(se_paged_kv kv, const int32_t* __restrict__ budget,
                      const uint32_t* __restrict__ keys_ws, int32_t* __restrict__ sel_pages,
                      int32_t* __restrict__ n_sel, se_view view, int* status) {
    extern __shared__ uint32_t skeys[];                   // [max_pages_per_seq] keys, then block table
    __shared__ int hist[256];
    __shared__ int tmp[33];
    __shared__ int stat[2];
    const int u = blockIdx.x, tid = threadIdx.x;
    const int H = kv.num_kv_heads;
    const int b = u / H, h = u % H;
    const int stride = kv.max_pages_per_seq;
    const int ctx = clamp_ctx(kv.ctx_len[b], stride * kPage, status, tid == 0 && h == 0);
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    int32_t* bts = reinterpret_cast<int32_t*>(skeys + stride);   // block-table row in shared memory
    for (int i = tid; i < n; i += blockDim.x) bts[i] = kv.block_table[(int64_t)b * stride + i];
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
        __syncthreads();
        for (int c = tid; c < n; c += blockDim.x) emit(c, c);
        if (tid == 0) {
            n_sel[u] = n;
            view.n_tokens[u] = ctx;
        }
        return;
    }
    const int m = n - 1, K = k - 1;
    const uint32_t* keys = keys_ws + (int64_t)u * stride;
    for (int i = tid; i < m; i += blockDim.x) skeys[i] = keys[i];
    __syncthreads();
    if (K > 0) {
        int need_eq = 0;
        const uint32_t T = block_radix_select([&](int i) { return skeys[i]; }, m, K, hist, tmp,
                                              stat, &need_eq);
        const int per = (m + blockDim.x - 1) / blockDim.x;
        const int i0 = min(m, tid * per), i1 = min(m, i0 + per);
        int gt = 0, eq = 0;
        for (int i = i0; i < i1; ++i) {
            gt += skeys[i] > T;
            eq += skeys[i] == T;
        }
        int t1, t2;
        int eq_before = block_exclusive_scan(eq, tmp, &t1);
        const int take_eq = max(0, min(eq, need_eq - eq_before));
        int out = block_exclusive_scan(gt + take_eq, tmp, &t2);
        for (int i = i0; i < i1; ++i) {
            const uint32_t kk = skeys[i];
            if (kk > T || (kk == T && eq_before++ < need_eq)) emit(out++, i);
        }
    }
    if (tid == 0) {
        emit(K, n - 1);
        n_sel[u] = k;
        view.n_tokens[u] = kPage * (k - 1) + (ctx - kPage * (n - 1));
    }
}

}  // namespace

size_t quest_ws_bytes(int units, int max_pages) {
    return 256 + (((size_t)units * max_pages * sizeof(uint32_t) + 255) & ~(size_t)255);
}

cudaError_t launch_quest_select(const se_paged_kv& kv, const void* q, int batch, int num_q_heads,
                                const int32_t* budget, int32_t* sel_pages, int32_t* n_sel,
                                const se_view& view, void* ws, int* status, cudaStream_t s) {
    const int units = batch * kv.num_kv_heads;
    if (units == 0) return cudaSuccess;
    uint32_t* keys = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 256);
    // scoring: one resident wave of kSelMinBlocks CTAs per SM shared by the sequences
    const int per_seq = max(1, min((num_sms() * kSelMinBlocks) / batch, kv.max_pages_per_seq));
    dim3 grid(per_seq, batch);
    const int kScoreDyn = kv.num_kv_heads * 2 * kv.head_dim * 4;
    cudaError_t e;
    if (kv.head_dim == 128) {
        e = cudaFuncSetAttribute(quest_score_kernel<128>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreDyn);
        if (e != cudaSuccess) return e;
        quest_score_kernel<128><<<grid, kSelThreads, kScoreDyn, s>>>(
            kv, static_cast<const uint16_t*>(q), num_q_heads, budget, keys, status);
    } else {
        e = cudaFuncSetAttribute(quest_score_kernel<64>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreDyn);
        if (e != cudaSuccess) return e;
        quest_score_kernel<64><<<grid, kSelThreads, kScoreDyn, s>>>(
            kv, static_cast<const uint16_t*>(q), num_q_heads, budget, keys, status);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int topk_smem = kv.max_pages_per_seq * 8;
    e = cudaFuncSetAttribute(quest_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             topk_smem);
    if (e != cudaSuccess) return e;
    quest_topk_kernel<<<units, kTopkThreads, topk_smem, s>>>(kv, budget, keys, sel_pages, n_sel,
                                                            view, status);
    return cudaGetLastError();
}

}  // namespace se
