/*
 * sparse_engine.h -- C ABI of libsparse_engine.so, the GB300 (sm_103a) hot path
 * of sparse-first KV-cache decoding: Quest page selection, split-K GQA decode
 * attention over an AttentionView, SnapKV compaction and the H2O step.
 *
 * Sources: the SparseEngine pages --
 *   [tokendh] tokendh.com news article on SparseEngine, sections
 *             "历史太长,会撑爆什么" (method families; Quest picks pages by the
 *             query, H2O keeps an accumulated attention score and deletes) and
 *             "把边界划在'生命周期'上" (per-method cache managers; SnapKV reads
 *             the last few tokens' attention and physically deletes; H2O
 *             updates scores each decode step; AttentionView turns every
 *             method's cache into one format the attention reads);
 *   [card]    "SparseEngine：稀疏优先推理引擎" (ai-feeds.com paper card),
 *             section "方法 / 关键模块" (AttentionView exposes the selected
 *             positions uniformly, so methods need no kernel changes);
 *   [jetabc]  "长程 agent 把显存撑爆以后" (jetabc.cn explainer), section
 *             "四、为什么进不了 vLLM 一类的引擎" (fixed-size pages + a table
 *             mapping tokens to pages).
 * The pages give no formulas; each entry point states the definition it computes.
 *
 * Conventions shared by every entry point
 *   - Every pointer in a struct or argument is a DEVICE pointer unless marked
 *     "host".  The caller owns and allocates all memory; the library never
 *     allocates, never frees, and never synchronises the stream (except
 *     se_sync_status, whose purpose is to).
 *   - bf16 = IEEE bfloat16 bit patterns (uint16 in memory).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *     Calls are reentrant; the library's only global state is a per-device
 *     cache of device attributes.
 *   - Host-side validation failures return a negative status and launch
 *     nothing.  A failed CUDA launch returns SE_ERR_CUDA.
 *   - Workspace (`ws`, `ws_bytes`): a caller-provided device buffer, 256-byte
 *     aligned, of at least the size its *_workspace() function returns.  Its
 *     first 4 bytes are the DEVICE STATUS WORD (int32): kernels OR in SE_DEV_*
 *     bits when they meet inconsistent device data (an index outside its
 *     buffer, a full segment, a wait that ran out of time); the offending
 *     access is skipped, nothing traps.  The word is sticky: clear it (a
 *     4-byte memset) to reset; read it after synchronising the stream.
 *     Calls that share one workspace must not overlap on the GPU.
 *   - Supported shapes: head_dim in {64, 128}; page size 16; group size
 *     G = num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}.
 *   - A "unit" is one (sequence b, KV head h) pair, u = b*num_kv_heads + h.
 */
#ifndef SPARSE_ENGINE_H
#define SPARSE_ENGINE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ------------------------------------- */
#define SE_OK               0
#define SE_ERR_INVALID_ARG (-1)  /* null pointer, bad size or stride */
#define SE_ERR_UNSUPPORTED (-2)  /* shape outside the supported set */
#define SE_ERR_WORKSPACE   (-3)  /* workspace missing, misaligned or too small */
#define SE_ERR_CUDA        (-4)  /* a CUDA runtime call or launch failed */
#define SE_ERR_CAPACITY    (-5)  /* an output buffer is too small for the request */

/* ---- device status word bits (workspace bytes 0..3) -------------------- */
#define SE_DEV_BAD_INDEX   1     /* block-table entry / row / position outside its buffer */
#define SE_DEV_CAPACITY    2     /* append past the last page or a full segment: dropped */
#define SE_DEV_BAD_LENGTH  4     /* a device length outside [0, capacity]: clamped */
#define SE_DEV_TIMEOUT     8     /* an intra-CTA wait ran past its limit; results invalid */

#define SE_PAGE_SIZE 16
#define SE_MAX_SPLITS 64

/* How a KV head's page bound combines its query heads (se_select_opts). */
#define SE_AGG_SUM 0             /* sum of the query heads' bounds (default) */
#define SE_AGG_MAX 1             /* largest of the query heads' bounds */

typedef void* se_stream_t;       /* cudaStream_t */

/* Paged KV cache with Quest page summaries ([jetabc] paging; [tokendh] the
 * "summary index" of dynamic-sparse methods).
 *   k, v   bf16 [num_pages][num_kv_heads][page_size][head_dim]: one (page, head)
 *          chunk is page_size contiguous rows of head_dim elements.  Viewed as
 *          [rows][head_dim], a token is row (page*num_kv_heads + h)*16 + slot.
 *   meta   bf16 [batch][max_pages_per_seq][num_kv_heads][2][head_dim]: per
 *          (sequence, LOGICAL page, head) the channel-wise min over the page's valid
 *          tokens, then the max.  Summaries are kept in logical page order per
 *          sequence (not by physical page) so that Quest scoring, which reads every
 *          summary of a sequence, is one sequential stream.
 *   block_table int32 [batch][max_pages_per_seq]: physical page of each logical
 *          page (entries past a sequence's pages are never read).
 *   ctx_len int32 [batch]: tokens held per sequence (se_kv_append increments it). */
typedef struct se_paged_kv {
    void* k;
    void* v;
    void* meta;
    const int32_t* block_table;
    int32_t* ctx_len;
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
} se_paged_kv;

/* AttentionView ([card] "exposes the selected positions in one format";
 * [tokendh] AttentionView): for each unit u, the rows it attends, as chunks of
 * 16 consecutive rows of a row-addressed K/V base ([rows][head_dim] bf16).
 *   chunk_row int32 [num_units][max_chunks]: first row of each chunk.
 *   n_tokens  int32 [num_units]: tokens of unit u; chunk c holds
 *             min(16, n_tokens - 16c) valid rows (only the last may be partial).
 * Token order = chunk order, then row order within a chunk. */
typedef struct se_view {
    int32_t* chunk_row;
    int32_t* n_tokens;
    int32_t num_units;
    int32_t max_chunks;
} se_view;

/* Per-(sequence, KV head) variable-length cache: the physical home of evicted
 * caches ([tokendh] SnapKV/H2O delete physically; retained tokens keep their
 * logical positions, section "聊天记录也能'续命':Chain Cache").
 *   k, v    bf16 [total_rows][head_dim]
 *   pos     int32 [total_rows]: logical position of each held row
 *   score   float [total_rows] or NULL: per-token accumulated score (H2O)
 *   seg_off int32 [num_units]: first row of unit u's segment
 *   seg_len int32 [num_units]: rows held
 *   seq_len int32 [batch]: logical tokens seen per sequence (= next position)
 *   seg_cap rows available to each segment (seg_off[u] + seg_cap <= total_rows). */
typedef struct se_varlen_kv {
    void* k;
    void* v;
    int32_t* pos;
    float* score;
    const int32_t* seg_off;
    int32_t* seg_len;
    int32_t* seq_len;
    int32_t seg_cap;
    int32_t total_rows;
    int32_t num_kv_heads;
    int32_t head_dim;
} se_varlen_kv;

/* H2O state: a varlen cache with scores.  Unit u holds its tokens in slots
 * [0, seg_len[u]) of its segment, in no particular order (an eviction moves the
 * segment's last token into the freed slot); seg_cap must be >= budget + 1. */
typedef struct se_h2o_state {
    se_varlen_kv kv;          /* score != NULL */
    int32_t budget;           /* tokens kept after each step */
    int32_t recent;           /* newest positions never evicted (1 <= recent <= budget) */
} se_h2o_state;

/* Decode options (optional; NULL means all defaults). */
typedef struct se_decode_opts {
    int32_t out_dtype;        /* 0 = bf16 output (default), 1 = fp32 output */
    int32_t max_splits;       /* split-K pieces per unit, 1..64 (0 = default 64) */
    float* logits_out;        /* NULL, or fp32 [num_units][logits_stride][G]:
                                 scale*q.k of every attended token, view order */
    int32_t logits_stride;    /* tokens per unit in logits_out */
    void* ev_kernel_begin;    /* NULL or a cudaEvent_t recorded right before / */
    void* ev_kernel_end;      /* right after the attention kernel (timing only;
                                 during a stream capture they are captured as
                                 external event-record nodes of the graph) */
} se_decode_opts;

/* Options of se_quest_step (optional; NULL means all defaults). */
typedef struct se_quest_step_opts {
    int32_t out_dtype;        /* 0 = bf16 output (default), 1 = fp32 output */
    int32_t max_splits;       /* decode pieces per unit at most, 1..64 (0 = 64) */
    void* ev_kernel_begin;    /* NULL or a cudaEvent_t recorded right before / */
    void* ev_kernel_end;      /* right after the step kernel (timing only; captured
                                 as external event-record nodes in a graph) */
    int32_t wait_limit_ns;    /* bound of each wait of one block on another
                                 (0: 1 s); a wait that runs out sets
                                 SE_DEV_TIMEOUT and the step's results, its
                                 append included, are invalid */
} se_quest_step_opts;

/* ---- library ------------------------------------------------------------ */
const char* se_status_str(int status);      /* static string, never NULL */
int se_version(void);                       /* ABI version, currently 1 */

/* Waits for every piece of work enqueued on `stream` and returns the SE_DEV_*
 * bits of the device status word at byte 0 of workspace `ws` (0 when no
 * kernel met inconsistent device data): the host-side reading of the status
 * word that the conventions above describe.  It does not clear the word.
 * Returns SE_ERR_INVALID_ARG for a NULL ws, SE_ERR_WORKSPACE for a ws that is
 * not 256-byte aligned (neither launches nor waits), and SE_ERR_CUDA when the
 * synchronisation or the 4-byte device-to-host copy fails (a failed kernel of
 * the stream included).  This is the one entry point that synchronises. */
int se_sync_status(const void* ws, se_stream_t stream);

/* ---- workspace sizes (bytes, multiples of 256) --------------------------- */
size_t se_small_workspace(void);            /* ops that need only the status word */
size_t se_quest_select_workspace(int batch, int num_kv_heads, int max_pages_per_seq);
size_t se_sparse_decode_workspace(int num_units, int group_size, int head_dim, int max_splits);
size_t se_quest_step_workspace(int batch, int num_kv_heads, int num_q_heads, int head_dim,
                               int max_pages_per_seq, int max_splits);
size_t se_snapkv_workspace(int batch, int num_kv_heads, int num_q_heads, int window, int max_ctx);
size_t se_h2o_workspace(int batch, int num_kv_heads, int num_q_heads, int head_dim, int seg_cap);

/* ---- page summaries ----------------------------------------------------- */
/* Rebuilds meta for every valid (page, head) of the first `batch` sequences:
 * kmin/kmax over tokens [16p, min(16p+16, ctx_len[b])).  Called once after
 * prefill.  Bad block-table entries set SE_DEV_BAD_INDEX and are skipped.
 * Workspace: se_small_workspace(). */
int se_page_meta_build(const se_paged_kv* kv, int batch,
                       void* ws, size_t ws_bytes, se_stream_t stream);

/* Decode-step append: writes k_new/v_new (bf16 [batch][num_kv_heads][head_dim])
 * at position ctx_len[b], folds the key into its page's min/max (a page's first
 * token sets both), then increments ctx_len[b].  block_table[b][ctx_len[b]/16]
 * must name a page; past max_pages_per_seq: SE_DEV_CAPACITY, token dropped.
 * kv->meta may be NULL: the rows are written and no summary is kept (a layer
 * that attends through the pages another layer selects, as in cross-layer
 * selection reuse; see se_sparse_decode).  Workspace: se_small_workspace(). */
int se_kv_append(const se_paged_kv* kv, const void* k_new, const void* v_new, int batch,
                 void* ws, size_t ws_bytes, se_stream_t stream);

/* ---- (a) Quest page selection ([tokendh] Quest picks pages by the query) ----
 * For unit u = (b, h) with query heads g of KV head h and n = ceil(ctx_len[b]/16):
 *   U[p] = sum_g sum_d max(q[b,hG+g,d]*kmin[p,h,d], q[b,hG+g,d]*kmax[p,h,d])
 *   k    = max(1, budget_tokens[b] / 16)   (integer division)
 *   selected = all pages if n <= k, else the last page n-1 plus the k-1 best of
 *   pages 0..n-2 under (U desc, page asc); written in ascending order.
 * q         bf16 [batch][num_q_heads][head_dim]
 * budget_tokens int32 [batch]
 * sel_pages int32 [num_units][max_pages_per_seq]: logical page ids (first n_sel[u])
 * n_sel     int32 [num_units]
 * view      filled for the paged K/V viewed as rows: chunk c of unit u is page
 *           block_table[b][sel[c]] of head h; n_tokens counts valid tokens.
 *           Needs view->num_units == batch*num_kv_heads and
 *           view->max_chunks >= max_pages_per_seq.
 * U is evaluated in fp32 as sum_d (Q+[d]*kmax[d] + Q-[d]*kmin[d]) with
 * Q+ = sum_g max(q_g, 0), Q- = sum_g min(q_g, 0): the same value in exact
 * arithmetic.  Limit: max_pages_per_seq <= 26624 (425984 tokens), else
 * SE_ERR_UNSUPPORTED.  Workspace: se_quest_select_workspace(). */
int se_quest_select(const se_paged_kv* kv, const void* q, int batch, int num_q_heads,
                    const int32_t* budget_tokens, int32_t* sel_pages, int32_t* n_sel,
                    const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream);

/* The decode step's append fused into the selection: the same effect as
 * se_kv_append(kv, k_new, v_new, batch) followed by se_quest_select(...) on the
 * same stream, in one kernel fewer.  The new token belongs to the last page,
 * which is always selected and never scored, so the scoring only needs the
 * new length; each top-k block writes its KV head's row and summary fold, and
 * the last block of a sequence to finish stores ctx_len[b] + 1.
 * k_new, v_new bf16 [batch][num_kv_heads][head_dim], 16-byte aligned; the other
 * arguments, limits and workspace are those of se_quest_select.  No token room
 * (ctx_len = max_pages_per_seq*16): SE_DEV_CAPACITY and nothing is appended.
 * A block-table entry that names no page for the new token: SE_DEV_BAD_INDEX,
 * nothing is appended and the selection for that sequence is unspecified. */
int se_quest_select_append(const se_paged_kv* kv, const void* k_new, const void* v_new,
                           const void* q, int batch, int num_q_heads,
                           const int32_t* budget_tokens, int32_t* sel_pages, int32_t* n_sel,
                           const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream);

/* Options of se_quest_select_ex (NULL means all defaults). */
typedef struct se_select_opts {
    int32_t group_agg;        /* SE_AGG_SUM (0, default) or SE_AGG_MAX */
} se_select_opts;

/* se_quest_select (k_new, v_new NULL) or se_quest_select_append (both given)
 * with options.  group_agg = SE_AGG_MAX takes the other reading of how a KV
 * head's query heads combine in the page bound:
 *   U[p] = max_g sum_d max(q[b,hG+g,d]*kmin[p,h,d], q[b,hG+g,d]*kmax[p,h,d]),
 * the largest of the heads' own bounds (an upper bound of every head's logit
 * over the page) instead of their sum; everything else is the same.  It needs
 * G <= 8 query heads per KV head and num_kv_heads in {1, 2, 4, 8}, else
 * SE_ERR_UNSUPPORTED.  Arguments, limits and workspace: se_quest_select's. */
int se_quest_select_ex(const se_paged_kv* kv, const void* k_new, const void* v_new,
                       const void* q, int batch, int num_q_heads, const int32_t* budget_tokens,
                       const se_select_opts* opts, int32_t* sel_pages, int32_t* n_sel,
                       const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream);

/* View of whole varlen segments: chunk c of unit u starts at row seg_off[u] + 16c;
 * n_tokens[u] = seg_len[u].  Needs view->max_chunks >= ceil(seg_cap / 16).
 * Workspace: se_small_workspace(). */
int se_view_from_segments(const se_varlen_kv* kv, int batch, const se_view* view,
                          void* ws, size_t ws_bytes, se_stream_t stream);

/* ---- (b) split-K GQA decode attention over a view ----------------------------
 * For unit u = (b, h), each query head g of the group, over the view's T tokens t:
 *   s[g,t] = scale * q[b,hG+g] . k_rows[row(t)]
 *   out[b,hG+g] = sum_t softmax_t(s[g,:]) v_rows[row(t)];  lse = log sum_t exp(s[g,t])
 * Each unit is cut into at most max_splits pieces of whole chunks; the pieces are
 * merged by their log-sum-exp.  T = 0 gives out = 0, lse = -inf.
 * k_rows, v_rows bf16 [total_rows][head_dim]; q bf16 [batch][num_q_heads][head_dim];
 * out bf16 or fp32 [batch][num_q_heads][head_dim]; lse fp32 [batch][num_q_heads] or NULL.
 * A chunk row outside [0, total_rows) sets SE_DEV_BAD_INDEX and counts as empty.
 * view->max_chunks <= 2^20 (16M tokens per unit), else SE_ERR_UNSUPPORTED.
 * Cross-layer selection reuse ([tokendh] "把边界划在'生命周期'上": OmniKV decides
 * in some layers which history matters and later layers reuse that decision):
 * the view holds row numbers of a row-addressed base, and caches that share one
 * paging (the layers of a model with one block table) share row numbers, so
 * the view a filter layer's se_quest_select filled may be passed with another
 * layer's k_rows/v_rows and q: that layer attends over its own keys and values
 * of the same pages, with no selection of its own.
 * Workspace: se_sparse_decode_workspace(num_units, G, head_dim, max_splits),
 * zero-filled before its first use: it holds the arrival counters of split
 * units, which every call leaves at zero (clear it again after a call that set
 * a device error bit).  The counters sit at a fixed offset whatever the shape,
 * so one workspace serves calls of any shape whose size it covers. */
int se_sparse_decode(const void* k_rows, const void* v_rows, int64_t total_rows,
                     const se_view* view, const void* q, int batch, int num_q_heads,
                     int num_kv_heads, int head_dim, float scale, const se_decode_opts* opts,
                     void* out, float* lse, void* ws, size_t ws_bytes, se_stream_t stream);

/* se_sparse_decode for callers that cannot allocate device memory (no
 * counterpart in the pages: this is a library-usage addition).  Callers that run
 * inside another framework's memory pool, that must not pay cudaMalloc's device
 * synchronisation, or whose host application owns every allocation cannot pass
 * a workspace; this variant takes its scratch from a fixed 8 MiB device array
 * inside the library (held by every GPU that loads it until the process exits)
 * and allocates nothing.  Same arguments and results as se_sparse_decode with
 * default options, except:
 *   - no workspace; out_dtype as in se_decode_opts; the split-K piece count is
 *     the largest (<= 64) whose partials fit the array, and a batch whose single
 *     piece per unit does not fit returns SE_ERR_CAPACITY;
 *   - status_out: NULL or a device int32 that receives the SE_DEV_* bits;
 *   - all calls share the array: calls that overlap on the GPU race (order them
 *     on one stream); each call clears the part that must start at zero;
 *   - the first call on a device looks up the array's device address; make it
 *     before any stream capture. */
int se_sparse_decode_noalloc(const void* k_rows, const void* v_rows, int64_t total_rows,
                             const se_view* view, const void* q, int batch, int num_q_heads,
                             int num_kv_heads, int head_dim, float scale, int out_dtype, void* out,
                             float* lse, int32_t* status_out, se_stream_t stream);

/* One Quest decode step in one kernel: se_quest_select_append (or
 * se_quest_select when k_new and v_new are NULL) followed by se_sparse_decode
 * over the view it fills, with the same selection, view, n_sel, ctx_len update
 * and outputs (up to the rounding order of the decode's split pieces).
 *   q, budget_tokens, sel_pages, n_sel, view: as in se_quest_select;
 *   k_new, v_new: as in se_quest_select_append, or both NULL (no append);
 *   scale, out, lse: as in se_sparse_decode (out bf16 or fp32 by opts->out_dtype).
 * The kernel is one cooperative launch (every block resident at once).  Each
 * block scores a slice of one sequence's page summaries (up to 32 sequences
 * share the blocks in proportion to their candidate pages), then decodes
 * pieces of units; a piece's top-k is computed by the block itself, once
 * every page of that sequence is scored, while its copy engine keeps
 * streaming the next data.  The waits of one block on the others are bounded
 * (opts->wait_limit_ns): one that runs out sets SE_DEV_TIMEOUT, leaves ctx_len
 * unchanged and the results invalid.  The last block to finish commits the new
 * lengths and clears the workspace's control words.
 * Limits: batch <= 1024, batch * num_kv_heads <= 4096, max_pages_per_seq <=
 * 16384 (14833 with 16 query heads per KV head at head_dim 128), else
 * SE_ERR_UNSUPPORTED.  A device that cannot hold the whole grid at once fails
 * the launch (SE_ERR_CUDA).
 * Workspace: se_quest_step_workspace(batch, num_kv_heads, num_q_heads, head_dim,
 * max_pages_per_seq, max_splits), zero-filled before its first use: it holds
 * control words (finished blocks, scored pages per sequence, split arrival
 * counters), which every call leaves at zero, at fixed offsets whatever the
 * shape, so one workspace serves calls of any shape whose size it covers.
 * Clear it again after a call that set a device error bit. */
int se_quest_step(const se_paged_kv* kv, const void* k_new, const void* v_new, const void* q,
                  int batch, int num_q_heads, const int32_t* budget_tokens, float scale,
                  const se_quest_step_opts* opts, int32_t* sel_pages, int32_t* n_sel,
                  const se_view* view, void* out, float* lse, void* ws, size_t ws_bytes,
                  se_stream_t stream);

/* Varlen append for decode over compacted caches: writes k_new/v_new (bf16
 * [batch][num_kv_heads][head_dim]) at row seg_off[u] + seg_len[u] with
 * pos = seq_len[b], then increments seg_len[u] and seq_len[b].  A full segment
 * sets SE_DEV_CAPACITY and drops the token.  Workspace: se_small_workspace(). */
int se_varlen_append(const se_varlen_kv* kv, const void* k_new, const void* v_new, int batch,
                     void* ws, size_t ws_bytes, se_stream_t stream);

/* se_varlen_append followed by se_view_from_segments on the same stream, in one
 * kernel (one block per sequence appends every KV head's row, then writes the
 * view of that sequence's whole segments).  Arguments, limits and errors are
 * those of the two calls.  Workspace: se_small_workspace(). */
int se_varlen_append_view(const se_varlen_kv* kv, const void* k_new, const void* v_new, int batch,
                          const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream);

/* ---- (c) SnapKV compaction ([tokendh] SnapKV: the last few tokens' attention
 * over the history decides what is kept; the rest is deleted physically) ------------
 * For unit (b, h), L = ctx_len[b]: window row i = 0..window-1 (position L-window+i,
 * queries q_win[b][i][hG+g]) attends causally to keys j <= L-window+i and
 *   A[j] = sum_i sum_g softmax_j(scale * q_win[b,i,hG+g] . k[j]).
 * Candidates are positions [0, L-recent); their A is max-pooled with the odd window
 * `pool_kernel` (stride 1, same length, clipped borders); the best `keep` under
 * (pooled desc, position asc) plus positions [L-recent, L) are kept, ascending.
 * SnapKV proper uses recent = window; recent > window with pool_kernel 1 seeds H2O.
 * Output rows seg_off[u] .. seg_off[u]+n_kept-1 of out->k/v, out->pos, out->score
 * (the unpooled A of each kept token) when non-NULL; seg_len[u] = n_kept;
 * seq_len[b] = L.  n_kept = min(keep, L-recent) + recent must fit seg_cap.
 * prefill: paged K/V (meta unused); q_win bf16 [batch][window][num_q_heads][head_dim].
 * Limits: 1 <= window <= 64, window*G <= 256, 1 <= recent <= L, L <= max_ctx of the
 * workspace query, pool_kernel odd and <= 63.
 * Workspace: se_snapkv_workspace(batch, num_kv_heads, num_q_heads, window, max_ctx). */
int se_snapkv_compact(const se_paged_kv* prefill, const void* q_win, int batch, int num_q_heads,
                      int window, int pool_kernel, int keep, int recent, float scale,
                      const se_varlen_kv* out, void* ws, size_t ws_bytes, se_stream_t stream);

/* ---- prefix-cache pruning over a caller span ([tokendh] "该删哪段历史,让应用自己说了算:
 * 可控前缀裁剪": the application names a region of the history and how much of it
 * to keep; a scorer keeps the tokens of the region that matter and the logical
 * prefix stays whole for prefix matching) ---------------------------------------
 * For unit (b, h), L = ctx_len[b]: the candidates are the positions
 * [span[2b], span[2b+1]) clipped to [0, L).  Their scores are the window
 * column scores A[j] of se_snapkv_compact (window rows L-window .. L-1, the
 * scorer the pages name, KVzip, being undescribed there), max-pooled over the
 * span with `pool_kernel` (neighbours outside the span ignored).  The best
 * keep_tokens[b] candidates under (pooled desc, position asc) are kept, and so
 * is every position outside the span.  Output as se_snapkv_compact: rows in
 * ascending position, pos = the logical positions (so a logical prefix still
 * matches), score = the unpooled A of each kept token, seg_len[u] = rows kept,
 * seq_len[b] = L; rows past seg_cap: SE_DEV_CAPACITY.
 * span int32 [batch][2], keep_tokens int32 [batch]: device.
 * Limits and workspace: those of se_snapkv_compact. */
int se_span_prune(const se_paged_kv* prefix, const void* q_win, int batch, int num_q_heads,
                  int window, int pool_kernel, const int32_t* span, const int32_t* keep_tokens,
                  float scale, const se_varlen_kv* out, void* ws, size_t ws_bytes,
                  se_stream_t stream);

/* StreamingLLM-style view of a paged cache (the first tokens as attention
 * sinks plus a recent window; "SparseEngine 统一接入十五种稀疏注意力", section
 * "哪些情况下加速幅度会缩小"), at page granularity: unit u = (b, h) attends the
 * pages [0, sink_pages) and the last recent_pages pages of its n =
 * ceil(ctx_len[b]/16) pages, each page once (all pages when they overlap), in
 * page order; n_tokens counts their valid tokens.  Needs view->max_chunks >=
 * min(sink_pages + recent_pages, max_pages_per_seq).  Feed the view to
 * se_sparse_decode.  Workspace: se_small_workspace(). */
int se_view_sink_recent(const se_paged_kv* kv, int batch, int sink_pages, int recent_pages,
                        const se_view* view, void* ws, size_t ws_bytes, se_stream_t stream);

/* ---- Chain Cache: retained state carried across turns ([tokendh] "聊天记录也能
 * '续命':Chain Cache": a method that deleted history physically resumes from the
 * state it kept when a new turn continues the same logical prefix; [netics]
 * "部署长上下文 Agent 的团队可以从中得到什么": the ChainCacheIndex links a session
 * to its retained per-layer KV, its method metadata and its logical token
 * prefix).  The device part copies state; the host part is a prefix index.
 *
 * Snapshot: a caller-owned device buffer (256-byte aligned) of
 * se_chain_snapshot_bytes(num_seqs, num_kv_heads, head_dim, rows, with_score)
 * bytes: a format header, then one slot per (saved sequence i, KV head h) of
 * `rows` rows: the unit's seg_len retained rows of K and V, their logical
 * positions, their scores when the cache keeps scores (with_score = score !=
 * NULL), and the sequence's seq_len.  A cache's method metadata that is not
 * per token (H2O's budget and recent window) stays with the caller.
 *
 * se_chain_save: slot (i, h) <- unit (seqs[i], h) of kv, rows [0, seg_len) in
 * their order.  se_chain_restore: unit (seqs[i], h) of kv <- slot (i, h),
 * written at that unit's seg_off with seg_len and seq_len set; the target
 * cache may place its segments anywhere (its seg_off), need not be the saved
 * one, and must have the same num_kv_heads, head_dim and score presence.  A
 * restored cache decodes exactly as the saved one would have (the rows, their
 * order, positions and scores are the same bytes).
 * seqs int32 [num_seqs] device.  A segment longer than `rows`, or a slot
 * longer than the target's seg_cap: SE_DEV_CAPACITY (truncated).  A snapshot
 * written for another shape, or seqs[i] < 0: SE_DEV_BAD_INDEX, unit left as is.
 * Workspace: se_small_workspace(). */
size_t se_chain_snapshot_bytes(int num_seqs, int num_kv_heads, int head_dim, int rows,
                               int with_score);
int se_chain_save(const se_varlen_kv* kv, const int32_t* seqs, int num_seqs, int rows, void* snap,
                  size_t snap_bytes, void* ws, size_t ws_bytes, se_stream_t stream);
int se_chain_restore(const void* snap, size_t snap_bytes, int num_seqs, int rows,
                     const int32_t* seqs, const se_varlen_kv* kv, void* ws, size_t ws_bytes,
                     se_stream_t stream);

/* The ChainCacheIndex (host): maps the logical token prefix a saved session
 * stands for -- every token of the conversation so far, the physically
 * deleted ones included -- to the caller's id for that session (for instance
 * a snapshot buffer).  A new request whose tokens begin with a stored prefix
 * matches it; the longest stored prefix wins, compared token by token.
 * Tokens are host int32 arrays.  The index is the one object the library
 * allocates (host memory, freed by se_chain_index_destroy); its calls are
 * thread-safe.
 *   create: NULL when out of memory.
 *   put: stores (tokens, id) -- an existing entry with that id is replaced.
 *   match: the id of the longest stored prefix of tokens (-1 when none), its
 *          length in *matched_tokens (may be NULL).
 *   erase: forgets id (no error when absent).  size: entries stored. */
typedef struct se_chain_index se_chain_index;
se_chain_index* se_chain_index_create(void);
void se_chain_index_destroy(se_chain_index* ix);
int se_chain_index_put(se_chain_index* ix, const int32_t* tokens, int64_t n_tokens, int64_t id);
int64_t se_chain_index_match(se_chain_index* ix, const int32_t* tokens, int64_t n_tokens,
                             int64_t* matched_tokens);
int se_chain_index_erase(se_chain_index* ix, int64_t id);
int64_t se_chain_index_size(se_chain_index* ix);

/* ---- (d) H2O decode step ([tokendh] H2O: accumulated attention scores updated
 * every decode step, then a physical deletion) -----------------------------------
 * For each unit u = (b, h):
 *   1. the new token (k_new/v_new bf16 [batch][num_kv_heads][head_dim]) goes to slot
 *      seg_len[u] with pos = seq_len[b] and score 0;
 *   2. decode attention of q (bf16 [batch][num_q_heads][head_dim]) over all held
 *      tokens -> out (bf16 or fp32 per out_dtype), lse (fp32, NULL allowed);
 *   3. score[t] += sum_g exp(s[g,t] - lse[g]) for every held token t;
 *   4. if more than `budget` tokens are held: among tokens whose position is not
 *      one of the `recent` largest, the last under (score desc, position asc) --
 *      the lowest score, the higher position on equal scores -- is evicted: its
 *      position goes to evicted_pos[u] (else -1) and the segment's last token
 *      moves into its slot.
 * seq_len[b] is incremented.  Positions must be unique per unit.
 * Workspace: se_h2o_workspace(batch, num_kv_heads, num_q_heads, head_dim, seg_cap),
 * zero-filled before its first use (it contains a decode workspace). */
int se_h2o_step(const se_h2o_state* st, const void* q, const void* k_new, const void* v_new,
                int batch, int num_q_heads, float scale, int out_dtype, void* out, float* lse,
                int32_t* evicted_pos, void* ws, size_t ws_bytes, se_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPARSE_ENGINE_H */
