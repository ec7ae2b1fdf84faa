// Split-K GQA decode attention over an AttentionView, and its log-sum-exp merge.
//
// The attention reads only the rows the view exposes ("SparseEngine：稀疏优先推理
// 引擎", section "方法 / 关键模块": AttentionView exposes the selected
// positions in one format, so methods need no kernel changes; tokendh.com
// article on SparseEngine, section "把边界划在'生命周期'上").
//
// Design (sm_103a):
//  * plan_kernel (1 CTA) cuts every unit's chunk list into pieces of about equal
//    size (at most max_splits per unit) and writes a work list.
//  * decode_kernel is persistent: one producer warp streams each 16-row K and V
//    chunk into a ring of shared-memory stages with 2-D TMA loads (128B swizzle,
//    mbarrier completion); consumer warp w owns the stages s with s % 4 == w.  Per
//    16-token chunk a warp computes S^T = K Q^T (tokens as M=16, the GQA group
//    as N=8) with ldmatrix + mma.sync.m16n8k16 (bf16 -> fp32), an online
//    softmax in the exp2 domain, transposes P in registers (movmatrix) and
//    accumulates O^T = V^T P^T (head_dim as M) with ldmatrix.trans + mma.
//    At the end of a piece the four warps merge through shared memory; a unit
//    cut into one piece is written directly, others go to fp32 partials.
//  * A unit cut into several pieces is merged by the last of its pieces to
//    finish (an arrival counter per unit; nobody waits on another CTA).
#include "common.cuh"
#include "decode_core.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kMaxGrid = 2048;              // persistent decode CTAs at most

// The decode kernel's shared-memory ring and layout.
template <int D, int NT>
struct DecRing {
    using S = DecShape<D, NT>;
    // Stage s is always consumed by warp s % 4 (kStages is a multiple of 4), so a
    // warp never waits on a stage more than one phase ahead of its own use.
    // 192 KB of stages in flight per SM at two CTAs per SM (96 KB at G = 16,
    // head_dim 128, where the merge area is twice as large)
    static constexpr int kStages = D == 64 ? 24 : (NT == 1 ? 12 : 8);
    static_assert(kStages % kConsumerWarps == 0, "stage ownership needs kStages % 4 == 0");
    static constexpr size_t kSmem = 1024 /* alignment slack */ + (size_t)kStages * S::kStageBytes +
                                    (size_t)kStages * 16 /* full, empty */ +
                                    (size_t)kStages * 4 /* ntok */ + 16 /* abort */ +
                                    (size_t)S::kMergeFloats * 4;
};

struct DecodeParams {
    const int32_t* chunk_row;
    const int32_t* n_tokens;
    int max_chunks;
    const uint16_t* q;
    int Hq, Hkv, G;
    float scale, scale_log2;
    const int4* items;
    const int* cta_first;     // [grid+1]: CTA c runs items cta_first[c] .. cta_first[c+1]-1
    const int2* unit_items;
    // self_plan: no plan kernel ran; each CTA derives its one piece (units <= grid)
    int self_plan, num_units, max_splits;
    int* counters;
    float* o_part;
    float* lse_part;
    void* out;
    int out_f32;
    float* lse_out;
    float* logits_out;
    int logits_stride;
    int64_t total_rows;
    int* status;
};

// Up to this many units (and no more than the grid) the decode CTAs plan for
// themselves; above it the block-wide plan kernel runs first.
constexpr int kSelfPlanUnits = 512;

// One piece per CTA, computed by one warp of every CTA (no plan kernel): unit
// u gets pieces_u = max(1, min(max_splits, nc_u, floor(nc_u * share / total)))
// pieces of nc_u * k / pieces_u chunks, with share = grid lowered until the
// pieces fit the grid (share 0 gives one piece per unit, which fits since
// units <= grid).  Piece k of unit u is item off_u + k, run by CTA off_u + k.
// tok: every unit's clamped token count, staged in shared memory by the whole
// CTA in one round trip.  The loops stay rolled: the plan runs once per launch,
// right after the previous kernel, when its instructions are not cached.
// Writes this CTA's item (unit, first chunk, end chunk, partial slot or -1),
// its unit's (first item, pieces) and token count; *has = 0 when the CTA runs
// none.
__device__ __noinline__ void plan_own_piece(const DecodeParams& p, const int* tok, int lane,
                                            int4* item, int2* uitem, int* ntok, int* has) {
    const int units = p.num_units, grid = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    int total = 0;
#pragma unroll 1
    for (int base = 0; base < units; base += 32)
        total += __reduce_add_sync(0xffffffffu,
                                   base + lane < units ? (tok[base + lane] + kPage - 1) / kPage : 0);
    // 32-bit products: nc <= max_chunks <= 2^20 (a host-side limit) and
    // share, k <= 2048 keep nc * share and nc * k below 2^31
    const int tot = max(1, total);
    auto pieces_of = [&](int nc, int share) {
        return nc == 0 ? 1 : max(1, min(p.max_splits, min(nc, nc * share / tot)));
    };
    // one pass per share: the scan over the pieces both finds this CTA's piece
    // and totals them; a share whose pieces do not fit the grid is lowered
    int share = grid;
#pragma unroll 1
    for (int iter = 0; iter < 5; ++iter) {
        if (lane == 0) *has = 0;
        __syncwarp();
        int run = 0;
#pragma unroll 1
        for (int base = 0; base < units; base += 32) {
            const int u = base + lane;
            const int n = u < units ? tok[u] : 0;
            const int nc = (n + kPage - 1) / kPage;
            const int pc = u < units ? pieces_of(nc, share) : 0;
            int x = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int off = run + x - pc;
            if (u < units && c >= off && c < off + pc) {
                const int k = c - off;
                *item = make_int4(u, nc * k / pc, nc * (k + 1) / pc, pc == 1 ? -1 : c);
                *uitem = make_int2(off, pc);
                *ntok = n;
                *has = 1;
            }
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        __syncwarp();                                   // *has / *item settled before a retry
        if (run <= grid || share == 0) break;          // share 0: one piece per unit
        share = iter == 3 ? 0 : max(0, share - (run - grid));
    }
}

__device__ __forceinline__ int unit_tokens(const DecodeParams& p, int u) {
    int n = p.n_tokens[u];
    const int lim = p.max_chunks * kPage;
    if (n < 0 || n > lim) {
        flag(p.status, SE_DEV_BAD_LENGTH);
        n = n < 0 ? 0 : lim;
    }
    return n;
}

// TWO_TERM: P is fed to the PV product as bf16 hi + bf16 lo (about 16
// mantissa bits) for the fp32-output mode; otherwise P is rounded once to bf16.
template <int D, int NT, bool TWO_TERM>
__global__ void __launch_bounds__(kDecodeThreads, NT == 2 ? 2 : 0)
    decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const DecodeParams p) {
    using S = DecShape<D, NT>;
    constexpr int NS = DecRing<D, NT>::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + NS * S::kStageBytes);
    uint64_t* empty = full + NS;
    int* stage_ntok = reinterpret_cast<int*>(empty + NS);
    volatile int* abort_flag = stage_ntok + NS;
    float* merge = reinterpret_cast<float*>(stage_ntok + NS + 4);   // 16-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    pdl_wait();
    pdl_trigger();
    // this CTA's items: [it_begin, it_end) of the plan's list, or its own
    // piece (item index blockIdx.x) when it plans for itself
    __shared__ int4 s_item;
    __shared__ int2 s_uitem;
    __shared__ int s_ntok, s_has;
    __shared__ int s_tok[kSelfPlanUnits];
    if (p.self_plan) {
        // every unit's token count, one load per thread (clamped: the
        // consumers flag a bad length)
        const int lim = p.max_chunks * kPage;
        for (int u = threadIdx.x; u < p.num_units; u += blockDim.x) {
            const int n = p.n_tokens[u];
            s_tok[u] = n < 0 ? 0 : (n > lim ? lim : n);
        }
        __syncthreads();
        if (warp == kConsumerWarps) plan_own_piece(p, s_tok, lane, &s_item, &s_uitem, &s_ntok, &s_has);
    }
    __syncthreads();
    int it_begin, it_end;
    if (p.self_plan) {
        it_begin = static_cast<int>(blockIdx.x);
        it_end = it_begin + s_has;
    } else {
        it_begin = p.cta_first[blockIdx.x];
        it_end = p.cta_first[blockIdx.x + 1];
    }

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        // The whole warp walks the chunk sequence; each lane loads one chunk row
        // of a 32-chunk block (one coalesced load, the next block prefetched),
        // lane 0 waits for the stage to be free and issues the TMA copies.
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
        }
        uint32_t seq = 0;
        // the next item's descriptor, token count and first 32 chunk rows are
        // fetched while the current item streams, so an item boundary costs no
        // dependent round trips
        int4 nitem = make_int4(0, 0, 0, 0);
        int nntok = 0, nrow = -1;
        // item blockIdx.x is this CTA's first item whenever cta_first says so
        // (the one-piece-per-CTA plan): it is loaded alongside cta_first, which
        // saves a dependent round trip before the first copy (the items array
        // holds at least grid entries, so the read stays in bounds)
        const int4 spec = p.self_plan ? s_item : p.items[blockIdx.x];
        const uint64_t kv_policy = l2_evict_first();
        auto fetch = [&](int it) {
            if (it >= it_end) return;
            nitem = it == static_cast<int>(blockIdx.x) ? spec : p.items[it];
            // the chunk rows go out first; the planned piece's token count is
            // already in shared memory (no second dependent round trip)
            const int32_t* c = p.chunk_row + (int64_t)nitem.x * p.max_chunks;
            nrow = nitem.y + lane < nitem.z ? c[nitem.y + lane] : -1;
            nntok = (p.self_plan && it == static_cast<int>(blockIdx.x)) ? s_ntok
                                                                          : unit_tokens(p, nitem.x);
        };
        fetch(it_begin);
        for (int it = it_begin; it < it_end; ++it) {
            const int4 item = nitem;
            const int u = item.x;
            const int ntok = nntok;
            const int32_t* crow = p.chunk_row + (int64_t)u * p.max_chunks;
            int row_next = nrow;
            fetch(it + 1);
            for (int cb = item.y; cb < item.z; cb += 32) {
                const int row_l = row_next;
                row_next = cb + 32 + lane < item.z ? crow[cb + 32 + lane] : -1;
                const int nb = min(32, item.z - cb);
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
                        const uint32_t ph = (sq / NS) & 1;
                        if (!*abort_flag && !mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                            *abort_flag = 1;
                            flag(p.status, SE_DEV_TIMEOUT);
                        }
                        int cnt = min(kPage, ntok - c * kPage);
                        if (row < 0 || (int64_t)row >= p.total_rows) {
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
                    if (mine && go && q < 2 * S::kBoxes) {
                        uint8_t* dst = stages + s * S::kStageBytes + (q & 1) * S::kChunkBytes +
                                       (q >> 1) * 2048;
                        // with logits saved, K/V (read once) leave L2 first so
                        // that the logits stay there for the next kernel
                        if (p.logits_out != nullptr)
                            tma_load_2d_hint(dst, (q & 1) ? &tv : &tk, &full[s], 64 * (q >> 1),
                                             row, kv_policy);
                        else
                            tma_load_2d(dst, (q & 1) ? &tv : &tk, &full[s], 64 * (q >> 1), row);
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
        return;
    }

    // -------------------------------- consumers --------------------------------
    DecOut dout;
    dout.out = p.out;
    dout.out_f32 = p.out_f32;
    dout.lse_out = p.lse_out;
    dout.o_part = p.o_part;
    dout.lse_part = p.lse_part;
    dout.counters = p.counters;
    dout.Hq = p.Hq;
    dout.G = p.G;
    uint32_t seq = 0;
    const int4 spec_c = p.self_plan ? s_item : p.items[blockIdx.x];   // as in the producer
    const uint64_t logit_policy = l2_evict_last();
    for (int it = it_begin; it < it_end; ++it) {
        const int4 item = it == static_cast<int>(blockIdx.x) ? spec_c : p.items[it];
        const int u = item.x;
        const int b = u / p.Hkv, h = u % p.Hkv;
        unit_tokens(p, u);                                  // flags a bad length
        DecState<D, NT> st;
        dec_begin<D, NT>(st, p.q, (int64_t)b * p.Hq + h * p.G, p.G, lane);
        for (int c = item.y; c < item.z; ++c, ++seq) {
            if ((seq % kConsumerWarps) != (uint32_t)warp) continue;
            const int s = seq % NS;
            const uint32_t ph = (seq / NS) & 1;
            if (!*abort_flag && !mbar_wait(&full[s], ph, abort_flag)) {
                *abort_flag = 1;
                flag(p.status, SE_DEV_TIMEOUT);
            }
            const int cnt = *abort_flag ? 0 : stage_ntok[s];
            if (cnt > 0) {
                float* lg = p.logits_out != nullptr
                                ? p.logits_out + ((int64_t)u * p.logits_stride + c * kPage) * p.G
                                : nullptr;
                dec_chunk<D, NT, TWO_TERM>(st, stages + s * S::kStageBytes, cnt, lane, p.scale,
                                           p.scale_log2, p.G, lg, logit_policy);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        const int slot = item.w;
        const int2 ui = slot < 0 ? make_int2(0, 1) : (p.self_plan ? s_uitem : p.unit_items[u]);
        dec_finish<D, NT>(st, merge, stage_ntok + NS + 1, dout, b, h, u, slot, ui, warp, lane);
    }
}

// One CTA.  Stream-K plan: the units' chunks are laid end to end (unit u owns
// global chunks [P_u, P_u + nc_u)); CTA c owns the global range
// [c*per, (c+1)*per) with per = ceil(total / grid), so every CTA streams the
// same number of chunks.  A unit is cut at range boundaries into pieces
// (items); per is raised when needed so that no unit has more than max_splits
// pieces.  With max_splits < 3 a unit is cut into at most max_splits equal
// pieces instead.  Outputs: items (unit, first chunk, end chunk, partial slot
// or -1 when the piece is the whole unit), per-unit (first item, count), and
// cta_first[c] = first item of CTA c (items whose global start lies in its range).
__global__ void __launch_bounds__(1024)
    plan_kernel(const int32_t* __restrict__ n_tokens, int units, int max_chunks, int max_splits,
                int grid, int4* __restrict__ items, int* __restrict__ gstart,
                int2* __restrict__ unit_items, int* __restrict__ cta_first,
                int* __restrict__ n_items, int* __restrict__ counters, int* status) {
    __shared__ int tmp[33];
    __shared__ int s_max;
    pdl_wait();
    pdl_trigger();
    const int lim = max_chunks * kPage;
    auto chunks_of = [&](int u) {
        int n = n_tokens[u];
        if (n < 0 || n > lim) {
            flag(status, SE_DEV_BAD_LENGTH);
            n = n < 0 ? 0 : lim;
        }
        return (n + kPage - 1) / kPage;
    };
    if (threadIdx.x == 0) s_max = 0;
    for (int u = threadIdx.x; u < units; u += blockDim.x) counters[u] = 0;
    __syncthreads();
    int total = 0;
    for (int base = 0; base < units; base += blockDim.x) {
        const int u = base + threadIdx.x;
        const int nc = u < units ? chunks_of(u) : 0;
        if (nc > 0) atomicMax(&s_max, nc);
        int t;
        block_exclusive_scan(nc, tmp, &t);
        total += t;
    }
    __syncthreads();
    // One piece per CTA when possible: unit u gets max(1, floor(nc_u*grid/total))
    // pieces (at most max_splits); if that fits the grid, every CTA streams one
    // piece and no CTA pays a second piece's epilogue in mid-stream.
    int fit_pieces = 0;
    for (int base = 0; base < units; base += blockDim.x) {
        const int u = base + threadIdx.x;
        int pc = 0;
        if (u < units) {
            const int nc = chunks_of(u);
            pc = nc == 0 ? 1
                         : max(1, min(max_splits, min(nc, (int)((int64_t)nc * grid / max(1, total)))));
        }
        int t;
        block_exclusive_scan(pc, tmp, &t);
        fit_pieces += t;
    }
    const bool one_each = fit_pieces <= grid;
    const bool streamk = !one_each && max_splits >= 3;
    int per = max(1, (total + grid - 1) / max(1, grid));
    if (streamk) per = max(per, (s_max + max_splits - 3) / (max_splits - 2));

    int run_items = 0, run_chunks = 0;
    for (int base = 0; base < units; base += blockDim.x) {
        const int u = base + threadIdx.x;
        int nc = 0, pieces = 0;
        if (u < units) {
            nc = chunks_of(u);
        }
        int t_chunks;
        const int P = run_chunks + block_exclusive_scan(nc, tmp, &t_chunks);
        if (u < units) {
            if (nc == 0)
                pieces = 1;
            else if (one_each)
                pieces = max(1, min(max_splits, min(nc, (int)((int64_t)nc * grid / max(1, total)))));
            else if (streamk)
                pieces = (P + nc - 1) / per - P / per + 1;
            else
                pieces = min(max_splits, nc);
        }
        int t_items;
        const int off = run_items + block_exclusive_scan(pieces, tmp, &t_items);
        if (u < units) {
            unit_items[u] = make_int2(off, pieces);
            for (int k = 0; k < pieces; ++k) {
                int c0, c1;
                if (nc == 0) {
                    c0 = c1 = 0;
                } else if (one_each) {
                    c0 = (int)((int64_t)nc * k / pieces);
                    c1 = (int)((int64_t)nc * (k + 1) / pieces);
                } else if (streamk) {
                    const int g0 = k == 0 ? P : (P / per + k) * per;
                    const int g1 = min(P + nc, (P / per + k + 1) * per);
                    c0 = g0 - P;
                    c1 = g1 - P;
                } else {
                    c0 = (int)((int64_t)nc * k / pieces);
                    c1 = (int)((int64_t)nc * (k + 1) / pieces);
                }
                items[off + k] = make_int4(u, c0, c1, pieces == 1 ? -1 : off + k);
                gstart[off + k] = P + c0;
            }
        }
        run_items += t_items;
        run_chunks += t_chunks;
    }
    __syncthreads();
    const int n = run_items;
    // CTA c takes the items whose global start lies in [c*per, (c+1)*per);
    // the last CTA also takes anything past the end.
    for (int c = threadIdx.x; c <= grid; c += blockDim.x) {
        if (one_each) {                                   // CTA c runs piece c (if any)
            cta_first[c] = min(c, n);
            continue;
        }
        int lo = 0, hi = n;
        if (c == grid) {
            lo = n;
        } else {
            const int64_t key = (int64_t)c * per;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (gstart[mid] < key) lo = mid + 1; else hi = mid;
            }
        }
        cta_first[c] = (c == 0) ? 0 : lo;
    }
    if (threadIdx.x == 0) *n_items = n;
}

template <int D, int NT, bool TWO>
cudaError_t run_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                       int grid, cudaStream_t s) {
    using S = DecRing<D, NT>;
    auto kern = decode_kernel<D, NT, TWO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(S::kSmem));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kDecodeThreads), S::kSmem, s, tk, tv, p);
}

template <int D, int NT>
int ctas_per_sm() {
    using S = DecRing<D, NT>;
    // dynamic ring + the kernel's static shared memory (plan staging), and the
    // 1 KB the hardware reserves per CTA
    return (S::kSmem + kSelfPlanUnits * 4 + 64) * 2 + 2048 <= 228 * 1024 ? 2 : 1;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Workspace layout.  The words every call must find at zero -- the split-K
// arrival counters, one per unit -- come first, right after the 256-byte
// header, in a block of at least kSelfPlanUnits words.  Their place does not
// depend on the call's shape, so a workspace that served one call serves any
// other whose size it covers: up to kSelfPlanUnits units the decode plans
// for itself and relies on the counters being zero, and those words are
// never anything but counters (every call leaves them at zero); above that
// the plan kernel clears the counters it uses at the start of the call.
size_t decode_ctl_bytes(int num_units) {
    return 256 + align256((size_t)max(num_units, kSelfPlanUnits) * sizeof(int));
}

size_t decode_ws_bytes(int num_units, int G, int D, int max_splits) {
    const size_t items = (size_t)num_units * max_splits;
    return decode_ctl_bytes(num_units) + align256(items * sizeof(int4)) +
           align256(items * sizeof(int)) + align256((size_t)num_units * sizeof(int2)) +
           align256((kMaxGrid + 1) * sizeof(int)) + align256(items * G * sizeof(float)) +
           align256(items * G * D * sizeof(float));
}

DecodeWs decode_ws_carve(void* ws, int num_units, int G, int D, int max_splits) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t items = (size_t)num_units * max_splits;
    DecodeWs w;
    w.status = reinterpret_cast<int*>(base);
    w.n_items = reinterpret_cast<int*>(base + 16);
    w.counters = reinterpret_cast<int*>(base + 256);
    size_t off = decode_ctl_bytes(num_units);
    w.items = reinterpret_cast<int4*>(base + off);
    off += align256(items * sizeof(int4));
    w.gstart = reinterpret_cast<int*>(base + off);
    off += align256(items * sizeof(int));
    w.unit_items = reinterpret_cast<int2*>(base + off);
    off += align256((size_t)num_units * sizeof(int2));
    w.cta_first = reinterpret_cast<int*>(base + off);
    off += align256((kMaxGrid + 1) * sizeof(int));
    w.lse_part = reinterpret_cast<float*>(base + off);
    off += align256(items * G * sizeof(float));
    w.o_part = reinterpret_cast<float*>(base + off);
    return w;
}

cudaError_t launch_sparse_decode(const void* k_rows, const void* v_rows, int64_t total_rows,
                                 const se_view& view, const void* q, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, float scale, int out_dtype,
                                 int max_splits, float* logits_out, int logits_stride,
                                 cudaEvent_t ev_begin, cudaEvent_t ev_end, void* out, float* lse,
                                 const DecodeWs& w, cudaStream_t s) {
    const int units = batch * num_kv_heads;
    if (units == 0) return cudaSuccess;
    if (view.max_chunks > (1 << 20)) return cudaErrorInvalidValue;   // the plan's 32-bit products
    const int G = num_q_heads / num_kv_heads;
    const int NT = G > 8 ? 2 : 1;
    CUtensorMap tk, tv;
    if (!encode_rows_map(&tk, k_rows, total_rows, head_dim) ||
        !encode_rows_map(&tv, v_rows, total_rows, head_dim))
        return cudaErrorInvalidValue;

    const int cps = head_dim == 64 ? ctas_per_sm<64, 1>()
                                   : (NT == 1 ? ctas_per_sm<128, 1>() : ctas_per_sm<128, 2>());
    const int max_items = units * max_splits;
    const int grid = max(1, min(kMaxGrid, min(max_items, num_sms() * cps)));

    // up to kSelfPlanUnits units (and no more than the grid), every decode CTA
    // derives its own piece and no plan kernel runs
    const bool self_plan = units <= kSelfPlanUnits && units <= grid;
    cudaError_t e = cudaSuccess;
    if (!self_plan) {
        e = launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s,
                       static_cast<const int32_t*>(view.n_tokens), units, view.max_chunks,
                       max_splits, grid, w.items, w.gstart, w.unit_items, w.cta_first, w.n_items,
                       w.counters, w.status);
        if (e != cudaSuccess) return e;
    }

    DecodeParams p;
    p.chunk_row = view.chunk_row;
    p.n_tokens = view.n_tokens;
    p.max_chunks = view.max_chunks;
    p.q = static_cast<const uint16_t*>(q);
    p.Hq = num_q_heads;
    p.Hkv = num_kv_heads;
    p.G = G;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.items = w.items;
    p.cta_first = w.cta_first;
    p.unit_items = w.unit_items;
    p.self_plan = self_plan ? 1 : 0;
    p.num_units = units;
    p.max_splits = max_splits;
    p.counters = w.counters;
    p.o_part = w.o_part;
    p.lse_part = w.lse_part;
    p.out = out;
    p.out_f32 = out_dtype == 1;
    p.lse_out = lse;
    p.logits_out = logits_out;
    p.logits_stride = logits_stride;
    p.total_rows = total_rows;
    p.status = w.status;

    // Inside a stream capture the timing events become event-record nodes of
    // the graph (external records), so a replayed graph times its own kernel.
    auto record = [&](cudaEvent_t ev) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e2 = cudaStreamIsCapturing(s, &cs);
        if (e2 != cudaSuccess) return e2;
        return cs == cudaStreamCaptureStatusActive
                   ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                   : cudaEventRecord(ev, s);
    };
    if (ev_begin) {
        e = record(ev_begin);
        if (e != cudaSuccess) return e;
    }
    const bool two = out_dtype == 1;
    if (head_dim == 64) {
        e = NT == 1 ? (two ? run_decode<64, 1, true>(tk, tv, p, grid, s)
                           : run_decode<64, 1, false>(tk, tv, p, grid, s))
                    : (two ? run_decode<64, 2, true>(tk, tv, p, grid, s)
                           : run_decode<64, 2, false>(tk, tv, p, grid, s));
    } else {
        e = NT == 1 ? (two ? run_decode<128, 1, true>(tk, tv, p, grid, s)
                           : run_decode<128, 1, false>(tk, tv, p, grid, s))
                    : (two ? run_decode<128, 2, true>(tk, tv, p, grid, s)
                           : run_decode<128, 2, false>(tk, tv, p, grid, s));
    }
    if (e != cudaSuccess) return e;
    if (ev_end) {
        e = record(ev_end);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace se
