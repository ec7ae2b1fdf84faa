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

constexpr int kScoreWarps = 8;
constexpr int kScoreUnroll = 8;

template <int D>
struct ScoreShape {
    static constexpr int kLpp = D / 4;                 // lanes per page (min half, max half)
    static constexpr int kPpw = 32 / kLpp;             // pages per warp-wide load
    static constexpr int kPagesPerCta = kScoreWarps * kPpw * kScoreUnroll;
};

__device__ __forceinline__ int clamp_ctx(int ctx, int cap, int* status, bool report) {
    if (ctx < 0 || ctx > cap) {
        if (report) flag(status, SE_DEV_BAD_LENGTH);
        return ctx < 0 ? 0 : cap;
    }
    return ctx;
}

// grid (page blocks, units); 256 threads.  scores[u][p] for p < n-1.
template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32)
    quest_score_kernel(se_paged_kv kv, const uint16_t* __restrict__ q, int Hq,
                       float* __restrict__ scores, int* status) {
    using S = ScoreShape<D>;
    const int u = blockIdx.y;
    const int H = kv.num_kv_heads, G = Hq / H;
    const int b = u / H, h = u % H;
    const int ctx = clamp_ctx(kv.ctx_len[b], kv.max_pages_per_seq * kPage, status, false);
    const int n = (ctx + kPage - 1) / kPage;
    const int ncand = n - 1;                           // the last page is forced
    const int p_cta = blockIdx.x * S::kPagesPerCta;
    if (p_cta >= ncand) return;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % S::kLpp;
    const bool is_max = sub >= S::kLpp / 2;
    const int seg = sub % (S::kLpp / 2);               // 8-channel segment

    // coefficients for this lane's 8 channels: Q+ (kmax half) or Q- (kmin half)
    float c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = 0.f;
    const uint4* q4 = reinterpret_cast<const uint4*>(q);
    for (int g = 0; g < G; ++g) {
        const uint4 w = q4[(((int64_t)b * Hq + h * G + g) * D) / 8 + seg];
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = bf_lo(a[i]), x1 = bf_hi(a[i]);
            c[2 * i] += is_max ? fmaxf(x0, 0.f) : fminf(x0, 0.f);
            c[2 * i + 1] += is_max ? fmaxf(x1, 0.f) : fminf(x1, 0.f);
        }
    }

    const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
    const uint4* meta = static_cast<const uint4*>(kv.meta);
    const int p_warp = p_cta + warp * S::kPpw * kScoreUnroll + lane / S::kLpp;

    uint4 w[kScoreUnroll];
    bool ok[kScoreUnroll];
#pragma unroll
    for (int j = 0; j < kScoreUnroll; ++j) {
        const int p = p_warp + j * S::kPpw;
        ok[j] = false;
        w[j] = make_uint4(0, 0, 0, 0);
        if (p < ncand) {
            const int phys = bt[p];
            if (phys >= 0 && phys < kv.num_pages) {
                ok[j] = true;
                w[j] = meta[((((int64_t)phys * H + h) * 2 + (is_max ? 1 : 0)) * D) / 8 + seg];
            } else if (sub == 0) {
                flag(status, SE_DEV_BAD_INDEX);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kScoreUnroll; ++j) {
        const uint32_t a[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(c[2 * i], bf_lo(a[i]), acc);
            acc = fmaf(c[2 * i + 1], bf_hi(a[i]), acc);
        }
#pragma unroll
        for (int o = S::kLpp / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const int p = p_warp + j * S::kPpw;
        if (sub == 0 && p < ncand)
            scores[(int64_t)u * kv.max_pages_per_seq + p] = ok[j] ? acc : -INFINITY;
    }
}

// One CTA (1024 threads) per unit: exact top-(k-1) of pages 0..n-2 by
// (score desc, page asc) via a 4-pass 8-bit radix select on order-preserving
// keys, then an index-ordered emit, plus the forced last page.
__global__ void __launch_bounds__(1024)
    quest_topk_kernel(se_paged_kv kv, const int32_t* __restrict__ budget,
                      const float* __restrict__ scores, int32_t* __restrict__ sel_pages,
                      int32_t* __restrict__ n_sel, se_view view, int* status) {
    __shared__ int hist[256];
    __shared__ int tmp[33];
    __shared__ int s_digit, s_above;

    const int u = blockIdx.x, tid = threadIdx.x;
    const int H = kv.num_kv_heads;
    const int b = u / H, h = u % H;
    const int stride = kv.max_pages_per_seq;
    const int ctx = clamp_ctx(kv.ctx_len[b], stride * kPage, status, tid == 0 && h == 0);
    const int n = (ctx + kPage - 1) / kPage;
    const int bud = budget[b];
    const int k = max(1, (bud < 0 ? 0 : bud) / kPage);
    const float* sc = scores + (int64_t)u * stride;
    int32_t* sel = sel_pages + (int64_t)u * stride;
    int32_t* crow = view.chunk_row + (int64_t)u * view.max_chunks;
    const int32_t* bt = kv.block_table + (int64_t)b * stride;

    auto emit = [&](int c, int page) {
        sel[c] = page;
        const int phys = bt[page];
        if (phys >= 0 && phys < kv.num_pages) {
            crow[c] = (phys * H + h) * kPage;
        } else {
            crow[c] = -1;
            flag(status, SE_DEV_BAD_INDEX);
        }
    };

    int count;
    if (n <= k) {
        for (int c = tid; c < n; c += blockDim.x) emit(c, c);
        count = n;
    } else {
        const int K = k - 1, m = n - 1;
        uint32_t prefix = 0, mask = 0;
        int remaining = K;
        if (K > 0) {
            for (int shift = 24; shift >= 0; shift -= 8) {
                if (tid < 256) hist[tid] = 0;
                __syncthreads();
                for (int i = tid; i < m; i += blockDim.x) {
                    const uint32_t key = float_key(sc[i]);
                    if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
                }
                __syncthreads();
                // cnt_ge[d] = number of matching keys whose digit is >= d
                const int v = tid < 256 ? hist[255 - tid] : 0;
                const int incl = scan256(v, tmp);
                if (tid < 256) {
                    const int excl = incl - v;
                    if (excl < remaining && incl >= remaining) {
                        s_digit = 255 - tid;
                        s_above = excl;
                    }
                }
                __syncthreads();
                prefix |= static_cast<uint32_t>(s_digit) << shift;
                mask |= 255u << shift;
                remaining -= s_above;
                __syncthreads();
            }
        }
        // keys > T all taken; the first `remaining` keys == T (by page) taken.
        const uint32_t T = prefix;
        const int need_eq = K > 0 ? remaining : 0;
        int run_eq = 0, run_out = 0;
        for (int base = 0; base < m; base += blockDim.x) {
            const int i = base + tid;
            uint32_t key = 0;
            if (i < m) key = float_key(sc[i]);
            const int gt = (K > 0 && i < m && key > T) ? 1 : 0;
            const int eq = (K > 0 && i < m && key == T) ? 1 : 0;
            int eq_tot, take_tot;
            const int eq_before = block_exclusive_scan(eq, tmp, &eq_tot);
            const int take = gt || (eq && run_eq + eq_before < need_eq);
            const int pos = block_exclusive_scan(take, tmp, &take_tot);
            if (take) emit(run_out + pos, i);
            run_eq += eq_tot;
            run_out += take_tot;
        }
        if (tid == 0) emit(run_out, n - 1);
        count = run_out + 1;
    }
    if (tid == 0) {
        n_sel[u] = count;
        view.n_tokens[u] = count == 0 ? 0 : kPage * (count - 1) + (ctx - kPage * (n - 1));
    }
}

}  // namespace

cudaError_t launch_quest_select(const se_paged_kv& kv, const void* q, int batch, int num_q_heads,
                                const int32_t* budget, int32_t* sel_pages, int32_t* n_sel,
                                const se_view& view, float* scores, int* status,
                                cudaStream_t s) {
    const int units = batch * kv.num_kv_heads;
    if (units == 0) return cudaSuccess;
    const int max_cand = kv.max_pages_per_seq;             // upper bound on n-1 candidates
    if (kv.head_dim == 128) {
        const int ppc = ScoreShape<128>::kPagesPerCta;
        dim3 grid((max_cand + ppc - 1) / ppc, units);
        quest_score_kernel<128><<<grid, kScoreWarps * 32, 0, s>>>(
            kv, static_cast<const uint16_t*>(q), num_q_heads, scores, status);
    } else {
        const int ppc = ScoreShape<64>::kPagesPerCta;
        dim3 grid((max_cand + ppc - 1) / ppc, units);
        quest_score_kernel<64><<<grid, kScoreWarps * 32, 0, s>>>(
            kv, static_cast<const uint16_t*>(q), num_q_heads, scores, status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    quest_topk_kernel<<<units, 1024, 0, s>>>(kv, budget, scores, sel_pages, n_sel, view, status);
    return cudaGetLastError();
}

}  // namespace se
