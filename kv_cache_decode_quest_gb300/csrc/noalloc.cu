// se_sparse_decode_noalloc: the split-K decode of se_sparse_decode for callers
// that cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: code that runs inside
// another runtime's memory pool and may not call cudaMalloc itself, hot loops
// that must not pay cudaMalloc's implicit device synchronisation, or plugins
// whose host framework owns every allocation.  For them this entry point takes
// its scratch (work list, per-piece partial outputs) from one file-scope
// device array of fixed size instead of a caller buffer.
//
// The array is reserved in every GPU that loads the library, for the life of
// the process.  All calls share it, so calls whose kernels overlap on the GPU
// (different streams without ordering) race; calls on one stream are safe.
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (host code cannot use the symbol itself: on the host it
// names a stand-in, not device memory); make that first call before any
// stream capture.  The call allocates nothing: no cudaMalloc, no cudaFree.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 8u << 20;   // 8 MiB per device
constexpr int kMaxDev = 64;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDev] = {};

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return SE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SE_OK;
}

}  // namespace

extern "C" {

int se_sparse_decode_noalloc(const void* k_rows, const void* v_rows, int64_t total_rows,
                             const se_view* view, const void* q, int batch, int num_q_heads,
                             int num_kv_heads, int head_dim, float scale, int out_dtype, void* out,
                             float* lse, int32_t* status_out, se_stream_t stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0) return SE_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return SE_ERR_UNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (num_q_heads % num_kv_heads || !(G == 1 || G == 2 || G == 4 || G == 8 || G == 16))
        return SE_ERR_UNSUPPORTED;
    if (batch == 0) return SE_OK;
    if (!k_rows || !v_rows || !view || !view->chunk_row || !view->n_tokens || !q || !out)
        return SE_ERR_INVALID_ARG;
    if (out_dtype != 0 && out_dtype != 1) return SE_ERR_INVALID_ARG;
    if (total_rows <= 0 || total_rows > INT32_MAX) return SE_ERR_INVALID_ARG;
    const uintptr_t a = reinterpret_cast<uintptr_t>(k_rows) | reinterpret_cast<uintptr_t>(v_rows) |
                        reinterpret_cast<uintptr_t>(q);
    if ((a & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return SE_ERR_INVALID_ARG;
    const int units = batch * num_kv_heads;
    if (view->num_units != units || view->max_chunks <= 0) return SE_ERR_INVALID_ARG;
    if (view->max_chunks > (1 << 20)) return SE_ERR_UNSUPPORTED;

    // The most split-K pieces per unit whose partials fit the fixed scratch.
    int max_splits = SE_MAX_SPLITS;
    while (max_splits > 0 && se::decode_ws_bytes(units, G, head_dim, max_splits) > kScratchBytes)
        --max_splits;
    if (max_splits == 0) return SE_ERR_CAPACITY;   // too many units for the fixed scratch

    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every word that must start at zero -- the status header and the split-K
    // arrival counters, which sit at a fixed place right after it -- is
    // cleared by each call, whatever the previous call's shape or outcome
    if (cudaMemsetAsync(scratch, 0, se::decode_ctl_bytes(units), s) != cudaSuccess)
        return SE_ERR_CUDA;
    se::DecodeWs w = se::decode_ws_carve(scratch, units, G, head_dim, max_splits);
    if (status_out) w.status = status_out;
    const cudaError_t e = se::launch_sparse_decode(
        k_rows, v_rows, total_rows, *view, q, batch, num_q_heads, num_kv_heads, head_dim, scale,
        out_dtype, max_splits, nullptr, 0, nullptr, nullptr, out, lse, w, s);
    return e == cudaSuccess ? SE_OK : SE_ERR_CUDA;
}

}  // extern "C"
