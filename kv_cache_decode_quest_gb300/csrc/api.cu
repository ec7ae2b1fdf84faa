// C ABI of libsparse_engine: host-side validation, workspace layout and kernel
// launches.  Every entry point validates its arguments on the host, returns a
// negative status without launching when they are wrong, and otherwise
// enqueues its kernels on the caller's stream.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "cudaTypedefs.h"

namespace se {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 1;
        g_sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int head_dim) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode || rows <= 0) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace se

using namespace se;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

int check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (!ws || !aligned(ws, 256) || ws_bytes < need) return SE_ERR_WORKSPACE;
    return SE_OK;
}

int check_paged(const se_paged_kv* kv, bool need_meta) {
    if (!kv || !kv->k || !kv->v || !kv->block_table || !kv->ctx_len) return SE_ERR_INVALID_ARG;
    if (need_meta && !kv->meta) return SE_ERR_INVALID_ARG;
    if (kv->page_size != SE_PAGE_SIZE || !head_dim_ok(kv->head_dim)) return SE_ERR_UNSUPPORTED;
    if (kv->num_kv_heads <= 0 || kv->num_pages <= 0 || kv->max_pages_per_seq <= 0)
        return SE_ERR_INVALID_ARG;
    if (!aligned(kv->k, 16) || !aligned(kv->v, 16) || (kv->meta && !aligned(kv->meta, 16)))
        return SE_ERR_INVALID_ARG;
    if ((int64_t)kv->num_pages * kv->num_kv_heads * SE_PAGE_SIZE > INT32_MAX)
        return SE_ERR_UNSUPPORTED;
    return SE_OK;
}

int check_varlen(const se_varlen_kv* kv) {
    if (!kv || !kv->k || !kv->v || !kv->pos || !kv->seg_off || !kv->seg_len || !kv->seq_len)
        return SE_ERR_INVALID_ARG;
    if (!head_dim_ok(kv->head_dim)) return SE_ERR_UNSUPPORTED;
    if (kv->num_kv_heads <= 0 || kv->seg_cap < 0 || kv->total_rows <= 0) return SE_ERR_INVALID_ARG;
    if (!aligned(kv->k, 16) || !aligned(kv->v, 16)) return SE_ERR_INVALID_ARG;
    return SE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SE_OK : SE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* se_status_str(int status) {
    switch (status) {
        case SE_OK: return "ok";
        case SE_ERR_INVALID_ARG: return "invalid argument (null pointer, bad size or stride)";
        case SE_ERR_UNSUPPORTED: return "unsupported shape";
        case SE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SE_ERR_CUDA: return "CUDA runtime error";
        case SE_ERR_CAPACITY: return "output buffer too small";
        default: return "unknown status";
    }
}

int se_version(void) { return 1; }

int se_sync_status(const void* ws, se_stream_t stream) {
    if (!ws) return SE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return SE_ERR_WORKSPACE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SE_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SE_ERR_CUDA;
    return word & (SE_DEV_BAD_INDEX | SE_DEV_CAPACITY | SE_DEV_BAD_LENGTH | SE_DEV_TIMEOUT);
}

size_t se_small_workspace(void) { return 256; }

size_t se_quest_select_workspace(int batch, int num_kv_heads, int max_pages_per_seq) {
    if (batch < 0 || num_kv_heads <= 0 || max_pages_per_seq < 0) return 0;
    return quest_ws_bytes(batch * num_kv_heads, max_pages_per_seq);
}

size_t se_sparse_decode_workspace(int num_units, int group_size, int head_dim, int max_splits) {
    if (num_units < 0 || group_size <= 0 || head_dim <= 0 || max_splits <= 0) return 0;
    return decode_ws_bytes(num_units, group_size, head_dim, max_splits);
}

int se_page_meta_build(const se_paged_kv* kv, int batch, void* ws, size_t ws_bytes,
                       se_stream_t stream) {
    int rc = check_paged(kv, true);
    if (rc) return rc;
    if (batch < 0) return SE_ERR_INVALID_ARG;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_page_meta_build(*kv, batch, static_cast<int*>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

int se_kv_append(const se_paged_kv* kv, const void* k_new, const void* v_new, int batch, void* ws,
                 size_t ws_bytes, se_stream_t stream) {
    int rc = check_paged(kv, false);
    if (rc) return rc;
    if (batch < 0 || (batch > 0 && (!k_new || !v_new))) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_kv_append(*kv, k_new, v_new, batch, static_cast<int*>(ws),
                                        static_cast<cudaStream_t>(stream)));
}

int se_quest_select(const se_paged_kv* kv, const void* q, int batch, int num_q_heads,
                    const int32_t* budget_tokens, int32_t* sel_pages, int32_t* n_sel,
                    const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_paged(kv, true);
    if (rc) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % kv->num_kv_heads || !group_ok(num_q_heads / kv->num_kv_heads))
        return SE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !budget_tokens || !sel_pages || !n_sel || !view || !view->chunk_row ||
                      !view->n_tokens))
        return SE_ERR_INVALID_ARG;
    if (!aligned(q, 16)) return SE_ERR_INVALID_ARG;
    if (view && view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if (view && view->max_chunks < kv->max_pages_per_seq) return SE_ERR_CAPACITY;
    // the top-k keeps one key and one block-table entry per page of a sequence
    // in shared memory (at most 26624 pages)
    if (kv->max_pages_per_seq > 26624) return SE_ERR_UNSUPPORTED;
    if ((rc = check_ws(ws, ws_bytes,
                       se_quest_select_workspace(batch, kv->num_kv_heads, kv->max_pages_per_seq))))
        return rc;
    return cuda_status(launch_quest_select(*kv, q, batch, num_q_heads, budget_tokens, sel_pages,
                                           n_sel, *view, nullptr, nullptr, ws,
                                           static_cast<int*>(ws),
                                           static_cast<cudaStream_t>(stream)));
}

int se_quest_select_append(const se_paged_kv* kv, const void* k_new, const void* v_new,
                           const void* q, int batch, int num_q_heads,
                           const int32_t* budget_tokens, int32_t* sel_pages, int32_t* n_sel,
                           const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream) {
    if (batch > 0 && (!k_new || !v_new)) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    int rc = check_paged(kv, true);
    if (rc) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % kv->num_kv_heads || !group_ok(num_q_heads / kv->num_kv_heads))
        return SE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !budget_tokens || !sel_pages || !n_sel || !view || !view->chunk_row ||
                      !view->n_tokens))
        return SE_ERR_INVALID_ARG;
    if (!aligned(q, 16)) return SE_ERR_INVALID_ARG;
    if (view && view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if (view && view->max_chunks < kv->max_pages_per_seq) return SE_ERR_CAPACITY;
    if (kv->max_pages_per_seq > 26624) return SE_ERR_UNSUPPORTED;
    if ((rc = check_ws(ws, ws_bytes,
                       se_quest_select_workspace(batch, kv->num_kv_heads, kv->max_pages_per_seq))))
        return rc;
    return cuda_status(launch_quest_select(*kv, q, batch, num_q_heads, budget_tokens, sel_pages,
                                           n_sel, *view, k_new, v_new, ws, static_cast<int*>(ws),
                                           static_cast<cudaStream_t>(stream)));
}

int se_quest_select_ex(const se_paged_kv* kv, const void* k_new, const void* v_new,
                       const void* q, int batch, int num_q_heads, const int32_t* budget_tokens,
                       const se_select_opts* opts, int32_t* sel_pages, int32_t* n_sel,
                       const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream) {
    if ((k_new == nullptr) != (v_new == nullptr)) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    const int agg = opts ? opts->group_agg : SE_AGG_SUM;
    if (agg != SE_AGG_SUM && agg != SE_AGG_MAX) return SE_ERR_INVALID_ARG;
    int rc = check_paged(kv, true);
    if (rc) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % kv->num_kv_heads || !group_ok(num_q_heads / kv->num_kv_heads))
        return SE_ERR_UNSUPPORTED;
    if (agg == SE_AGG_MAX &&
        (num_q_heads / kv->num_kv_heads > 8 || 8 % kv->num_kv_heads != 0))
        return SE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !budget_tokens || !sel_pages || !n_sel || !view || !view->chunk_row ||
                      !view->n_tokens))
        return SE_ERR_INVALID_ARG;
    if (!aligned(q, 16)) return SE_ERR_INVALID_ARG;
    if (view && view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if (view && view->max_chunks < kv->max_pages_per_seq) return SE_ERR_CAPACITY;
    if (kv->max_pages_per_seq > 26624) return SE_ERR_UNSUPPORTED;
    if ((rc = check_ws(ws, ws_bytes,
                       se_quest_select_workspace(batch, kv->num_kv_heads, kv->max_pages_per_seq))))
        return rc;
    return cuda_status(launch_quest_select(*kv, q, batch, num_q_heads, budget_tokens, sel_pages,
                                           n_sel, *view, k_new, v_new, ws, static_cast<int*>(ws),
                                           static_cast<cudaStream_t>(stream), agg));
}

size_t se_quest_step_workspace(int batch, int num_kv_heads, int num_q_heads, int head_dim,
                               int max_pages_per_seq, int max_splits) {
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 ||
        max_pages_per_seq < 0 || max_splits <= 0 || num_q_heads % num_kv_heads)
        return 0;
    return quest_step_ws_bytes(batch, num_kv_heads, num_q_heads / num_kv_heads, head_dim,
                               max_pages_per_seq, max_splits);
}

int se_quest_step(const se_paged_kv* kv, const void* k_new, const void* v_new, const void* q,
                  int batch, int num_q_heads, const int32_t* budget_tokens, float scale,
                  const se_quest_step_opts* opts, int32_t* sel_pages, int32_t* n_sel,
                  const se_view* view, void* out, float* lse, void* ws, size_t ws_bytes,
                  se_stream_t stream) {
    if ((k_new == nullptr) != (v_new == nullptr)) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    int rc = check_paged(kv, true);
    if (rc) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % kv->num_kv_heads || !group_ok(num_q_heads / kv->num_kv_heads))
        return SE_ERR_UNSUPPORTED;
    if (batch > 0 && (!q || !budget_tokens || !sel_pages || !n_sel || !view || !view->chunk_row ||
                      !view->n_tokens || !out))
        return SE_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16)) return SE_ERR_INVALID_ARG;
    if (view && view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if (view && view->max_chunks < kv->max_pages_per_seq) return SE_ERR_CAPACITY;
    if (batch > kStepMaxBatch || batch * kv->num_kv_heads > kStepMaxUnits ||
        kv->max_pages_per_seq > 16384)
        return SE_ERR_UNSUPPORTED;
    se_quest_step_opts o = {0, SE_MAX_SPLITS, nullptr, nullptr, 0};
    if (opts) {
        o = *opts;
        if (o.max_splits == 0) o.max_splits = SE_MAX_SPLITS;
    }
    if (o.out_dtype != 0 && o.out_dtype != 1) return SE_ERR_INVALID_ARG;
    if (o.max_splits < 1 || o.max_splits > SE_MAX_SPLITS) return SE_ERR_INVALID_ARG;
    if (o.wait_limit_ns < 0) return SE_ERR_INVALID_ARG;
    const int G = num_q_heads / kv->num_kv_heads;
    if (quest_step_smem_bytes(kv->num_kv_heads, kv->head_dim, G) > 227 * 1024)
        return SE_ERR_UNSUPPORTED;
    if (kv->max_pages_per_seq > quest_step_max_pages(kv->head_dim, G)) return SE_ERR_UNSUPPORTED;
    if ((rc = check_ws(ws, ws_bytes,
                       se_quest_step_workspace(batch, kv->num_kv_heads, num_q_heads, kv->head_dim,
                                               kv->max_pages_per_seq, o.max_splits))))
        return rc;
    if (batch == 0) return SE_OK;
    const unsigned long long wait_ns =
        o.wait_limit_ns > 0 ? (unsigned long long)o.wait_limit_ns : 1000000000ull;
    return cuda_status(launch_quest_step(
        *kv, k_new, v_new, q, batch, num_q_heads, budget_tokens, scale, o.out_dtype, o.max_splits,
        wait_ns, sel_pages, n_sel, *view, out, lse, ws,
        static_cast<cudaEvent_t>(o.ev_kernel_begin), static_cast<cudaEvent_t>(o.ev_kernel_end),
        static_cast<cudaStream_t>(stream)));
}

int se_view_from_segments(const se_varlen_kv* kv, int batch, const se_view* view, void* ws,
                          size_t ws_bytes, se_stream_t stream) {
    int rc = check_varlen(kv);
    if (rc) return rc;
    if (batch < 0 || !view || !view->chunk_row || !view->n_tokens) return SE_ERR_INVALID_ARG;
    if (view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if ((int64_t)view->max_chunks * SE_PAGE_SIZE < kv->seg_cap) return SE_ERR_CAPACITY;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_view_from_segments(*kv, batch, *view, static_cast<int*>(ws),
                                                 static_cast<cudaStream_t>(stream)));
}

int se_sparse_decode(const void* k_rows, const void* v_rows, int64_t total_rows, const se_view* view,
                     const void* q, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                     float scale, const se_decode_opts* opts, void* out, float* lse, void* ws,
                     size_t ws_bytes, se_stream_t stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0) return SE_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim)) return SE_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads || !group_ok(num_q_heads / num_kv_heads))
        return SE_ERR_UNSUPPORTED;
    if (batch == 0) return SE_OK;
    if (!k_rows || !v_rows || !view || !view->chunk_row || !view->n_tokens || !q || !out)
        return SE_ERR_INVALID_ARG;
    if (total_rows <= 0 || total_rows > INT32_MAX) return SE_ERR_INVALID_ARG;
    if (!aligned(k_rows, 16) || !aligned(v_rows, 16) || !aligned(q, 16) || !aligned(out, 16))
        return SE_ERR_INVALID_ARG;
    if (view->num_units != batch * num_kv_heads || view->max_chunks <= 0) return SE_ERR_INVALID_ARG;
    if (view->max_chunks > (1 << 20)) return SE_ERR_UNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    se_decode_opts o = {0, SE_MAX_SPLITS, nullptr, 0, nullptr, nullptr};
    if (opts) {
        o = *opts;
        if (o.max_splits == 0) o.max_splits = SE_MAX_SPLITS;
    }
    if (o.out_dtype != 0 && o.out_dtype != 1) return SE_ERR_INVALID_ARG;
    if (o.max_splits < 1 || o.max_splits > SE_MAX_SPLITS) return SE_ERR_INVALID_ARG;
    if (o.logits_out && o.logits_stride < (int64_t)view->max_chunks * SE_PAGE_SIZE)
        return SE_ERR_CAPACITY;
    const int units = batch * num_kv_heads;
    int rc = check_ws(ws, ws_bytes, decode_ws_bytes(units, G, head_dim, o.max_splits));
    if (rc) return rc;
    const DecodeWs w = decode_ws_carve(ws, units, G, head_dim, o.max_splits);
    return cuda_status(launch_sparse_decode(
        k_rows, v_rows, total_rows, *view, q, batch, num_q_heads, num_kv_heads, head_dim, scale,
        o.out_dtype, o.max_splits, o.logits_out, o.logits_stride,
        static_cast<cudaEvent_t>(o.ev_kernel_begin), static_cast<cudaEvent_t>(o.ev_kernel_end), out,
        lse, w, static_cast<cudaStream_t>(stream)));
}

int se_varlen_append_view(const se_varlen_kv* kv, const void* k_new, const void* v_new, int batch,
                          const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_varlen(kv);
    if (rc) return rc;
    if (batch < 0 || (batch > 0 && (!k_new || !v_new))) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    if (!view || !view->chunk_row || !view->n_tokens) return SE_ERR_INVALID_ARG;
    if (view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if ((int64_t)view->max_chunks * SE_PAGE_SIZE < kv->seg_cap) return SE_ERR_CAPACITY;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_varlen_append_view(*kv, k_new, v_new, batch, *view,
                                                 static_cast<int*>(ws),
                                                 static_cast<cudaStream_t>(stream)));
}

int se_varlen_append(const se_varlen_kv* kv, const void* k_new, const void* v_new, int batch,
                     void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_varlen(kv);
    if (rc) return rc;
    if (batch < 0 || (batch > 0 && (!k_new || !v_new))) return SE_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return SE_ERR_INVALID_ARG;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_varlen_append(*kv, k_new, v_new, batch, static_cast<int*>(ws),
                                            static_cast<cudaStream_t>(stream)));
}

size_t se_snapkv_workspace(int batch, int num_kv_heads, int num_q_heads, int window,
                           int max_ctx) {
    (void)num_q_heads;
    (void)window;
    if (batch < 0 || num_kv_heads <= 0 || max_ctx < 0) return 0;
    return snapkv_ws_bytes(batch * num_kv_heads, max_ctx);
}

int se_snapkv_compact(const se_paged_kv* prefill, const void* q_win, int batch, int num_q_heads,
                      int window, int pool_kernel, int keep, int recent, float scale,
                      const se_varlen_kv* out, void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_paged(prefill, false);
    if (rc) return rc;
    if ((rc = check_varlen(out))) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % prefill->num_kv_heads) return SE_ERR_UNSUPPORTED;
    const int G = num_q_heads / prefill->num_kv_heads;
    if (!group_ok(G)) return SE_ERR_UNSUPPORTED;
    if (out->num_kv_heads != prefill->num_kv_heads || out->head_dim != prefill->head_dim)
        return SE_ERR_INVALID_ARG;
    if (window < 1 || window > 64 || window * G > 256) return SE_ERR_UNSUPPORTED;
    if (pool_kernel < 1 || pool_kernel > 63 || pool_kernel % 2 == 0) return SE_ERR_UNSUPPORTED;
    if (keep < 0 || recent < 1) return SE_ERR_INVALID_ARG;
    if (batch == 0) return SE_OK;
    if (!q_win || !aligned(q_win, 16)) return SE_ERR_INVALID_ARG;
    // the workspace fixes the longest context it can score
    const size_t base = se_snapkv_workspace(batch, prefill->num_kv_heads, num_q_heads, window, 0);
    const size_t per_ctx = (size_t)batch * prefill->num_kv_heads * 8;
    if (!ws || !aligned(ws, 256) || ws_bytes < base) return SE_ERR_WORKSPACE;
    int64_t max_ctx = (int64_t)((ws_bytes - base) / per_ctx);
    max_ctx = std::min<int64_t>(max_ctx, (int64_t)prefill->max_pages_per_seq * SE_PAGE_SIZE);
    while (max_ctx > 0 &&
           se_snapkv_workspace(batch, prefill->num_kv_heads, num_q_heads, window, (int)max_ctx) >
               ws_bytes)
        --max_ctx;
    if (max_ctx <= 0) return SE_ERR_WORKSPACE;
    return cuda_status(launch_snapkv_compact(*prefill, q_win, batch, num_q_heads, window,
                                             pool_kernel, keep, recent, scale, *out, ws,
                                             (int)max_ctx, static_cast<cudaStream_t>(stream)));
}

int se_span_prune(const se_paged_kv* prefix, const void* q_win, int batch, int num_q_heads,
                  int window, int pool_kernel, const int32_t* span, const int32_t* keep_tokens,
                  float scale, const se_varlen_kv* out, void* ws, size_t ws_bytes,
                  se_stream_t stream) {
    int rc = check_paged(prefix, false);
    if (rc) return rc;
    if ((rc = check_varlen(out))) return rc;
    if (batch < 0 || num_q_heads <= 0) return SE_ERR_INVALID_ARG;
    if (num_q_heads % prefix->num_kv_heads) return SE_ERR_UNSUPPORTED;
    const int G = num_q_heads / prefix->num_kv_heads;
    if (!group_ok(G)) return SE_ERR_UNSUPPORTED;
    if (out->num_kv_heads != prefix->num_kv_heads || out->head_dim != prefix->head_dim)
        return SE_ERR_INVALID_ARG;
    if (window < 1 || window > 64 || window * G > 256) return SE_ERR_UNSUPPORTED;
    if (pool_kernel < 1 || pool_kernel > 63 || pool_kernel % 2 == 0) return SE_ERR_UNSUPPORTED;
    if (batch == 0) return SE_OK;
    if (!q_win || !aligned(q_win, 16) || !span || !keep_tokens) return SE_ERR_INVALID_ARG;
    const size_t base = se_snapkv_workspace(batch, prefix->num_kv_heads, num_q_heads, window, 0);
    const size_t per_ctx = (size_t)batch * prefix->num_kv_heads * 8;
    if (!ws || !aligned(ws, 256) || ws_bytes < base) return SE_ERR_WORKSPACE;
    int64_t max_ctx = (int64_t)((ws_bytes - base) / per_ctx);
    max_ctx = std::min<int64_t>(max_ctx, (int64_t)prefix->max_pages_per_seq * SE_PAGE_SIZE);
    while (max_ctx > 0 &&
           se_snapkv_workspace(batch, prefix->num_kv_heads, num_q_heads, window, (int)max_ctx) >
               ws_bytes)
        --max_ctx;
    if (max_ctx <= 0) return SE_ERR_WORKSPACE;
    return cuda_status(launch_snapkv_compact(*prefix, q_win, batch, num_q_heads, window,
                                             pool_kernel, 0, 0, scale, *out, ws, (int)max_ctx,
                                             static_cast<cudaStream_t>(stream), span,
                                             keep_tokens));
}

int se_view_sink_recent(const se_paged_kv* kv, int batch, int sink_pages, int recent_pages,
                        const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_paged(kv, false);
    if (rc) return rc;
    if (batch < 0 || sink_pages < 0 || recent_pages < 0) return SE_ERR_INVALID_ARG;
    if (!view || !view->chunk_row || !view->n_tokens) return SE_ERR_INVALID_ARG;
    if (view->num_units != batch * kv->num_kv_heads) return SE_ERR_INVALID_ARG;
    if (view->max_chunks < std::min<int64_t>((int64_t)sink_pages + recent_pages,
                                             kv->max_pages_per_seq))
        return SE_ERR_CAPACITY;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_view_sink_recent(*kv, batch, sink_pages, recent_pages, *view,
                                               static_cast<int*>(ws),
                                               static_cast<cudaStream_t>(stream)));
}

int se_chain_save(const se_varlen_kv* kv, const int32_t* seqs, int num_seqs, int rows, void* snap,
                  size_t snap_bytes, void* ws, size_t ws_bytes, se_stream_t stream) {
    int rc = check_varlen(kv);
    if (rc) return rc;
    if (num_seqs < 0 || rows < 0) return SE_ERR_INVALID_ARG;
    if (num_seqs == 0) return SE_OK;
    if (!seqs || !snap || !aligned(snap, 256)) return SE_ERR_INVALID_ARG;
    if (snap_bytes < chain_snapshot_bytes(num_seqs, kv->num_kv_heads, kv->head_dim, rows,
                                          kv->score != nullptr))
        return SE_ERR_CAPACITY;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_chain_copy(true, *kv, seqs, num_seqs, rows, snap,
                                         static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

int se_chain_restore(const void* snap, size_t snap_bytes, int num_seqs, int rows,
                     const int32_t* seqs, const se_varlen_kv* kv, void* ws, size_t ws_bytes,
                     se_stream_t stream) {
    int rc = check_varlen(kv);
    if (rc) return rc;
    if (num_seqs < 0 || rows < 0) return SE_ERR_INVALID_ARG;
    if (num_seqs == 0) return SE_OK;
    if (!seqs || !snap || !aligned(snap, 256)) return SE_ERR_INVALID_ARG;
    if (snap_bytes < chain_snapshot_bytes(num_seqs, kv->num_kv_heads, kv->head_dim, rows,
                                          kv->score != nullptr))
        return SE_ERR_CAPACITY;
    if ((rc = check_ws(ws, ws_bytes, se_small_workspace()))) return rc;
    return cuda_status(launch_chain_copy(false, *kv, seqs, num_seqs, rows,
                                         const_cast<void*>(snap), static_cast<int*>(ws),
                                         static_cast<cudaStream_t>(stream)));
}

size_t se_h2o_workspace(int batch, int num_kv_heads, int num_q_heads, int head_dim, int seg_cap) {
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads ||
        seg_cap < 0 || !head_dim_ok(head_dim))
        return 0;
    return h2o_ws_bytes(batch, num_kv_heads, num_q_heads, head_dim, seg_cap);
}

int se_h2o_step(const se_h2o_state* st, const void* q, const void* k_new, const void* v_new,
                int batch, int num_q_heads, float scale, int out_dtype, void* out, float* lse,
                int32_t* evicted_pos, void* ws, size_t ws_bytes, se_stream_t stream) {
    if (!st) return SE_ERR_INVALID_ARG;
    int rc = check_varlen(&st->kv);
    if (rc) return rc;
    const se_varlen_kv& kv = st->kv;
    if (!kv.score) return SE_ERR_INVALID_ARG;
    if (batch < 0 || num_q_heads <= 0 || num_q_heads % kv.num_kv_heads) return SE_ERR_INVALID_ARG;
    if (!group_ok(num_q_heads / kv.num_kv_heads)) return SE_ERR_UNSUPPORTED;
    if (st->budget < 1 || st->recent < 1 || st->recent > st->budget) return SE_ERR_INVALID_ARG;
    if (kv.seg_cap < st->budget + 1) return SE_ERR_CAPACITY;
    if (out_dtype != 0 && out_dtype != 1) return SE_ERR_INVALID_ARG;
    if (batch == 0) return SE_OK;
    if (!q || !k_new || !v_new || !out || !evicted_pos) return SE_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16))
        return SE_ERR_INVALID_ARG;
    if ((rc = check_ws(ws, ws_bytes, se_h2o_workspace(batch, kv.num_kv_heads, num_q_heads,
                                                      kv.head_dim, kv.seg_cap))))
        return rc;
    return cuda_status(launch_h2o_step(*st, q, k_new, v_new, batch, num_q_heads, scale, out_dtype,
                                       out, lse, evicted_pos, ws,
                                       static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
