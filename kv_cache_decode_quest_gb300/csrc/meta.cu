// Cache maintenance kernels: Quest page summaries (channel-wise key min/max per
// (page, KV head)), the decode-step appends for the paged and the
// variable-length caches, and the AttentionView of whole varlen segments.
//
// The page summary is Quest's "summary index" kept beside the full history
// (tokendh.com article on SparseEngine, section "历史太长,会撑爆什么");
// pages of 16 tokens with a token->page table follow the paged KV layout of
// "长程 agent 把显存撑爆以后", section "四、为什么进不了 vLLM 一类的引擎".
#include "append.cuh"
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

__global__ void page_meta_build_kernel(se_paged_kv kv, int* status) {
    const int b = blockIdx.y, p = blockIdx.x;
    const int H = kv.num_kv_heads, D = kv.head_dim, segs = D / 8;
    int ctx = kv.ctx_len[b];
    const int cap = kv.max_pages_per_seq * kPage;
    if (ctx < 0 || ctx > cap) {
        if (p == 0 && threadIdx.x == 0) flag(status, SE_DEV_BAD_LENGTH);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int n = (ctx + kPage - 1) / kPage;
    if (p >= n) return;
    const int phys = kv.block_table[(int64_t)b * kv.max_pages_per_seq + p];
    if (phys < 0 || phys >= kv.num_pages) {
        if (threadIdx.x == 0) flag(status, SE_DEV_BAD_INDEX);
        return;
    }
    const int valid = min(kPage, ctx - p * kPage);
    const uint4* K = static_cast<const uint4*>(kv.k);
    uint4* M = static_cast<uint4*>(kv.meta);
    for (int t = threadIdx.x; t < H * segs; t += blockDim.x) {
        const int h = t / segs, sg = t % segs;
        const int64_t row0 = ((int64_t)phys * H + h) * kPage;
        Bf8 mn = unpack8(K[row0 * segs + sg]), mx = mn;
        for (int r = 1; r < valid; ++r) {
            const Bf8 x = unpack8(K[(row0 + r) * segs + sg]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mn.x[i] = fminf(mn.x[i], x.x[i]);
                mx.x[i] = fmaxf(mx.x[i], x.x[i]);
            }
        }
        const int64_t m0 = (((int64_t)b * kv.max_pages_per_seq + p) * H + h) * 2;
        M[m0 * segs + sg] = pack8(mn);
        M[(m0 + 1) * segs + sg] = pack8(mx);
    }
}

__global__ void kv_append_kernel(se_paged_kv kv, const uint4* k_new, const uint4* v_new,
                                 int* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int H = kv.num_kv_heads;
    __shared__ int s_pos;
    if (threadIdx.x == 0) s_pos = kv.ctx_len[b];
    __syncthreads();
    const int pos = s_pos;
    const int p = pos / kPage;
    bool ok = pos >= 0 && p < kv.max_pages_per_seq;
    int phys = -1;
    if (ok) {
        phys = kv.block_table[(int64_t)b * kv.max_pages_per_seq + p];
        if (phys < 0 || phys >= kv.num_pages) {
            if (threadIdx.x == 0) flag(status, SE_DEV_BAD_INDEX);
            ok = false;
        }
    } else if (threadIdx.x == 0) {
        flag(status, pos < 0 ? SE_DEV_BAD_LENGTH : SE_DEV_CAPACITY);
    }
    if (ok) {
        // each head's vectors are split over blockDim / H threads
        const int nthr = static_cast<int>(blockDim.x);
        const int per_head = max(1, nthr / H), heads_at_once = nthr / per_head;
        for (int h = threadIdx.x / per_head; h < H; h += heads_at_once)
            append_head(kv, b, h, pos, phys, k_new, v_new, threadIdx.x % per_head, per_head);
    }
    __syncthreads();
    if (threadIdx.x == 0 && ok) kv.ctx_len[b] = pos + 1;
}

// One block per sequence b: the new row of every KV head of b, then (with_view)
// the AttentionView of b's whole segments, then seq_len[b] -- one block reads
// and writes b's lengths, so there is no race between blocks.
__global__ void varlen_append_kernel(se_varlen_kv kv, const uint4* k_new, const uint4* v_new,
                                     se_view view, int with_view, int* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int H = kv.num_kv_heads, D = kv.head_dim, segs = D / 8;
    __shared__ int s_pos;
    if (threadIdx.x == 0) s_pos = kv.seq_len[b];
    __syncthreads();
    const int pos = s_pos;
    uint4* K = static_cast<uint4*>(kv.k);
    uint4* V = static_cast<uint4*>(kv.v);
    for (int t = threadIdx.x; t < H * segs; t += blockDim.x) {
        const int h = t / segs, sg = t % segs;
        const int u = b * H + h;
        const int len = kv.seg_len[u];
        const int off = kv.seg_off[u];
        if (len < 0 || len >= kv.seg_cap) {
            if (sg == 0) flag(status, len < 0 ? SE_DEV_BAD_LENGTH : SE_DEV_CAPACITY);
            continue;
        }
        const int64_t row = (int64_t)off + len;
        if (off < 0 || row >= kv.total_rows) {
            if (sg == 0) flag(status, SE_DEV_BAD_INDEX);
            continue;
        }
        K[row * segs + sg] = k_new[((int64_t)b * H + h) * segs + sg];
        V[row * segs + sg] = v_new[((int64_t)b * H + h) * segs + sg];
        if (sg == 0) {
            kv.pos[row] = pos;
            if (kv.score) kv.score[row] = 0.0f;
        }
    }
    __syncthreads();
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const int u = b * H + h;
        const int len = kv.seg_len[u];
        const int64_t row = (int64_t)kv.seg_off[u] + len;
        if (len >= 0 && len < kv.seg_cap && kv.seg_off[u] >= 0 && row < kv.total_rows)
            kv.seg_len[u] = len + 1;
    }
    if (with_view) {
        __syncthreads();                       // this block's seg_len updates are visible
        const int lim = min(kv.seg_cap, view.max_chunks * kPage);
        for (int h = 0; h < H; ++h) {
            const int u = b * H + h;
            int len = kv.seg_len[u];
            if (len < 0 || len > lim) {
                if (threadIdx.x == 0) flag(status, SE_DEV_BAD_LENGTH);
                len = len < 0 ? 0 : lim;
            }
            const int off = kv.seg_off[u];
            const int nc = (len + kPage - 1) / kPage;
            for (int c = threadIdx.x; c < nc; c += blockDim.x)
                view.chunk_row[(int64_t)u * view.max_chunks + c] = off + c * kPage;
            if (threadIdx.x == 0) view.n_tokens[u] = len;
        }
    }
    if (threadIdx.x == 0) kv.seq_len[b] = pos + 1;
}

__global__ void view_segments_kernel(se_varlen_kv kv, se_view view, int* status) {
    pdl_wait();
    pdl_trigger();
    const int u = blockIdx.x;
    int len = kv.seg_len[u];
    const int lim = min(kv.seg_cap, view.max_chunks * kPage);
    if (len < 0 || len > lim) {
        if (threadIdx.x == 0) flag(status, SE_DEV_BAD_LENGTH);
        len = len < 0 ? 0 : lim;
    }
    const int off = kv.seg_off[u];
    const int nc = (len + kPage - 1) / kPage;
    for (int c = threadIdx.x; c < nc; c += blockDim.x)
        view.chunk_row[(int64_t)u * view.max_chunks + c] = off + c * kPage;
    if (threadIdx.x == 0) view.n_tokens[u] = len;
}

// The sink + recent view of unit u = (b, h) of a paged cache (StreamingLLM:
// the first tokens and a recent window, here at page granularity): pages
// [0, sink) and [n - recent, n) of the sequence's n pages, each page once;
// its chunk is the page's physical rows of head h.  Only the newest page can
// be partial, and it is the view's last chunk when it is selected.
__global__ void view_sink_recent_kernel(se_paged_kv kv, int sink, int recent, se_view view,
                                        int* status) {
    pdl_wait();
    pdl_trigger();
    const int H = kv.num_kv_heads;
    const int u = blockIdx.x, b = u / H, h = u % H;
    const int cap = kv.max_pages_per_seq * kPage;
    int L = kv.ctx_len[b];
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && h == 0) flag(status, SE_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : cap;
    }
    const int n = (L + kPage - 1) / kPage;
    const int first = min(sink, n);                       // pages [0, first)
    const int tail0 = max(first, n - recent);             // then pages [tail0, n)
    const int np = first + (n - tail0);
    const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
    for (int c = threadIdx.x; c < np && c < view.max_chunks; c += blockDim.x) {
        const int page = c < first ? c : tail0 + (c - first);
        const int phys = bt[page];
        if (phys >= 0 && phys < kv.num_pages) {
            view.chunk_row[(int64_t)u * view.max_chunks + c] = (phys * H + h) * kPage;
        } else {
            view.chunk_row[(int64_t)u * view.max_chunks + c] = -1;
            flag(status, SE_DEV_BAD_INDEX);
        }
    }
    if (threadIdx.x == 0) {
        // tokens: every selected page is full except the newest (page n - 1)
        const bool last_in = np > 0 && (tail0 < n || first == n);
        view.n_tokens[u] = last_in ? kPage * (np - 1) + (L - kPage * (n - 1)) : kPage * np;
    }
}

}  // namespace

cudaError_t launch_view_sink_recent(const se_paged_kv& kv, int batch, int sink_pages,
                                    int recent_pages, const se_view& view, int* status,
                                    cudaStream_t s) {
    const int units = batch * kv.num_kv_heads;
    if (units == 0) return cudaSuccess;
    view_sink_recent_kernel<<<units, 128, 0, s>>>(kv, sink_pages, recent_pages, view, status);
    return cudaGetLastError();
}

cudaError_t launch_page_meta_build(const se_paged_kv& kv, int batch, int* status,
                                   cudaStream_t s) {
    if (batch == 0 || kv.max_pages_per_seq == 0) return cudaSuccess;
    dim3 grid(kv.max_pages_per_seq, batch);
    page_meta_build_kernel<<<grid, 128, 0, s>>>(kv, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const se_paged_kv& kv, const void* k_new, const void* v_new,
                             int batch, int* status, cudaStream_t s) {
    if (batch == 0) return cudaSuccess;
    kv_append_kernel<<<batch, 128, 0, s>>>(kv, static_cast<const uint4*>(k_new),
                                           static_cast<const uint4*>(v_new), status);
    return cudaGetLastError();
}

cudaError_t launch_varlen_append(const se_varlen_kv& kv, const void* k_new, const void* v_new,
                                 int batch, int* status, cudaStream_t s) {
    if (batch == 0) return cudaSuccess;
    se_view none = {};
    varlen_append_kernel<<<batch, 128, 0, s>>>(kv, static_cast<const uint4*>(k_new),
                                               static_cast<const uint4*>(v_new), none, 0, status);
    return cudaGetLastError();
}

cudaError_t launch_varlen_append_view(const se_varlen_kv& kv, const void* k_new,
                                      const void* v_new, int batch, const se_view& view,
                                      int* status, cudaStream_t s) {
    if (batch == 0) return cudaSuccess;
    varlen_append_kernel<<<batch, 128, 0, s>>>(kv, static_cast<const uint4*>(k_new),
                                               static_cast<const uint4*>(v_new), view, 1, status);
    return cudaGetLastError();
}

cudaError_t launch_view_from_segments(const se_varlen_kv& kv, int batch, const se_view& view,
                                      int* status, cudaStream_t s) {
    const int units = batch * kv.num_kv_heads;
    if (units == 0) return cudaSuccess;
    view_segments_kernel<<<units, 128, 0, s>>>(kv, view, status);
    return cudaGetLastError();
}

}  // namespace se
