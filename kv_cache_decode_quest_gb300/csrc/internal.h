// Host-side launch interface between the C ABI layer (api.cu) and the kernel
// translation units.  Every launcher enqueues on `stream` and returns the
// launch's cudaError_t; arguments were validated by the caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_engine.h"

namespace se {

// Launches `kern` with programmatic stream serialization: its blocks may
// become resident while the previous kernel in the stream runs, and wait in
// pdl_wait() (which every kernel launched this way calls before touching
// global memory) for that kernel to complete.  Used for the decode plan and
// the decode kernel, small enough or resident late enough not to crowd the
// kernel ahead of them (early-resident top-k blocks slowed the page scoring).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

int num_sms();

// ---- meta.cu ----
cudaError_t launch_page_meta_build(const se_paged_kv& kv, int batch, int* status, cudaStream_t s);
cudaError_t launch_kv_append(const se_paged_kv& kv, const void* k_new, const void* v_new,
                             int batch, int* status, cudaStream_t s);
cudaError_t launch_varlen_append(const se_varlen_kv& kv, const void* k_new, const void* v_new,
                                 int batch, int* status, cudaStream_t s);
// the varlen append and the segment view in one kernel (one block per sequence)
cudaError_t launch_varlen_append_view(const se_varlen_kv& kv, const void* k_new,
                                      const void* v_new, int batch, const se_view& view,
                                      int* status, cudaStream_t s);
cudaError_t launch_view_sink_recent(const se_paged_kv& kv, int batch, int sink_pages,
                                    int recent_pages, const se_view& view, int* status,
                                    cudaStream_t s);
cudaError_t launch_view_from_segments(const se_varlen_kv& kv, int batch, const se_view& view,
                                      int* status, cudaStream_t s);

// ---- quest.cu ----
size_t quest_ws_bytes(int units, int max_pages);
// k_new / v_new non-null: the decode-step append of the new token is fused in
// (same result as launch_kv_append followed by the selection).
cudaError_t launch_quest_select(const se_paged_kv& kv, const void* q, int batch, int num_q_heads,
                                const int32_t* budget, int32_t* sel_pages, int32_t* n_sel,
                                const se_view& view, const void* k_new, const void* v_new,
                                void* ws, int* status, cudaStream_t s, int group_agg = SE_AGG_SUM);

// ---- quest_step.cu ----
// se_quest_step's fixed control block holds the counters of at most this many
// sequences and units.
constexpr int kStepMaxBatch = 1024;
constexpr int kStepMaxUnits = 4096;
size_t quest_step_ws_bytes(int batch, int H, int G, int D, int max_pages, int max_splits);
size_t quest_step_smem_bytes(int H, int D, int G);
int quest_step_max_pages(int D, int G);
cudaError_t launch_quest_step(const se_paged_kv& kv, const void* k_new, const void* v_new,
                              const void* q, int batch, int num_q_heads, const int32_t* budget,
                              float scale, int out_dtype, int max_splits,
                              unsigned long long wait_ns, int32_t* sel_pages,
                              int32_t* n_sel,
                              const se_view& view, void* out, float* lse, void* ws,
                              cudaEvent_t ev_begin, cudaEvent_t ev_end, cudaStream_t s);

// ---- chain.cu ----
size_t chain_snapshot_bytes(int num_seqs, int H, int D, int rows, bool with_score);
cudaError_t launch_chain_copy(bool save, const se_varlen_kv& kv, const int32_t* seqs, int n,
                              int rows, void* snap, int* status, cudaStream_t s);

// ---- decode.cu ----
struct DecodeWs {
    int* status;
    int* n_items;
    int4* items;          // [num_units * max_splits]
    int* gstart;          // [num_units * max_splits]: global first chunk of each item
    int* cta_first;       // [grid + 1]: first item of each decode CTA
    int2* unit_items;     // [num_units]: (first item, item count)
    int* counters;        // [num_units]: pieces finished; at a fixed offset (256), left at
                          // zero by every call (the plan kernel also clears them)
    float* lse_part;      // [num_units * max_splits][G]   (log2 domain)
    float* o_part;        // [num_units * max_splits][G][D] (normalised)
};
// Bytes of the workspace head that must be zero before a call: the status
// header and the arrival counters (fixed offset, independent of G, D and splits).
size_t decode_ctl_bytes(int num_units);
size_t decode_ws_bytes(int num_units, int G, int D, int max_splits);
DecodeWs decode_ws_carve(void* ws, int num_units, int G, int D, int max_splits);
cudaError_t launch_sparse_decode(const void* k_rows, const void* v_rows, int64_t total_rows,
                                 const se_view& view, const void* q, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, float scale, int out_dtype,
                                 int max_splits, float* logits_out, int logits_stride,
                                 cudaEvent_t ev_begin, cudaEvent_t ev_end, void* out, float* lse,
                                 const DecodeWs& w, cudaStream_t s);

// ---- snapkv.cu / snapkv_tc.cu ----
constexpr int kSnapMaxSplits = 64;      // key ranges per unit at most (partials workspace)
constexpr int kSnapMaxSplitsTc = kSnapMaxSplits;
// Both scoring passes on tcgen05 (head_dim 128, W*G <= 256): per-row partials
// into part [units][splits][256] and column scores into colsum [units][max_ctx].
cudaError_t launch_snapkv_scores_tc(const se_paged_kv& kv, const void* q_win, int batch, int Hq,
                                    int W, float scale, float2* part, float* colsum, int max_ctx,
                                    int* status, cudaStream_t s);
size_t snapkv_ws_bytes(int units, int max_ctx);
cudaError_t launch_snapkv_compact(const se_paged_kv& kv, const void* q_win, int batch, int Hq,
                                  int W, int pool_kernel, int keep, int recent, float scale,
                                  const se_varlen_kv& out, void* ws, int max_ctx, cudaStream_t s,
                                  const int32_t* span = nullptr, const int32_t* keep_seq = nullptr);

// ---- h2o.cu ----
size_t h2o_ws_bytes(int batch, int Hkv, int Hq, int D, int seg_cap);
cudaError_t launch_h2o_step(const se_h2o_state& st, const void* q, const void* k_new,
                            const void* v_new, int batch, int Hq, float scale, int out_dtype,
                            void* out, float* lse, int32_t* evicted_pos, void* ws,
                            cudaStream_t s);

// ---- tensor maps (api.cu) ----
// 2-D bf16 map over [rows][head_dim] with 16-row x 64-column boxes, 128B swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int head_dim);

}  // namespace se
