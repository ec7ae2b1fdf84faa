// SnapKV compaction at the end of prefill: observation-window attention
// scores, 1-D max-pool, per-KV-head top-k, and compaction of the survivors
// into a per-(sequence, KV head) variable-length cache.
//
// SnapKV inspects how the last few query rows attend over the history, keeps
// the important part and physically deletes the rest (tokendh.com article on
// SparseEngine, section "把边界划在'生命周期'上"); kept tokens keep their
// logical positions (same article, section "聊天记录也能'续命':Chain Cache").
//
// Definitions (unit u = (b, h), L = ctx_len[b], window rows i = 0..W-1 at
// positions L-W+i, G query heads per KV head, M = W*G rows r = i*G + g):
//   s[r,j] = scale * q_win[b,i,hG+g] . k[j]          for j <= L-W+i (causal)
//   A[j]   = sum_r exp(s[r,j] - lse_r),  lse_r = log sum_j exp(s[r,j])
//   candidates [0, L-recent): pooled A (odd window, clipped), best `keep` kept
//   under (pooled desc, position asc), plus [L-recent, L).
//
// Kernels:
//   snapkv_score_kernel<PASS 1>: per (unit, key range) the per-row running
//     (max, sum) of exp2 over the range -> partials;
//   snapkv_score_kernel<PASS 2>: merges the partials into lse_r, recomputes S
//     and writes the column sums A[j] of its key range;
//   snapkv_select_kernel: per unit, pool -> keys, exact radix top-k, emit the
//     kept positions ascending, gather their K/V rows into the varlen cache.
// S = Q K^T is the one dense contraction of the path (M = W*G rows): Q rows
// sit in registers as mma.sync A fragments, 64-key blocks of K are staged by
// TMA from the paged cache (producer warp + mbarriers), B fragments come from
// ldmatrix on the 128B-swizzled boxes.
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kSkWarps = 8;                 // consumer warps (16*MT rows each)
constexpr int kSkThreads = (kSkWarps + 1) * 32;
constexpr int kSkBlockKeys = 64;            // keys per stage (4 pages)
constexpr int kSkStages = 4;
constexpr float kLog2eF = 1.4426950408889634f;

template <int D, int MT>
struct SkShape {
    static constexpr int kRows = kSkWarps * 16 * MT;          // padded M
    static constexpr int kQStride = D + 8;                     // bf16 elems per smem row
    static constexpr int kPageBytes = (D / 64) * 2048;
    static constexpr int kStageBytes = 4 * kPageBytes;         // 64 keys of K
    static constexpr size_t kSmem = 1024 + (size_t)kSkStages * kStageBytes +
                                    (size_t)kRows * kQStride * 2 + kSkStages * 8 * 2 + 64 +
                                    (size_t)kRows * 4 + kSkBlockKeys * 4 * kSkWarps;
};

struct SkParams {
    se_paged_kv kv;
    const uint16_t* q_win;   // [B][W][Hq][D]
    int W, Hq, G, M;          // M = W*G real rows
    int splits;               // key ranges per unit
    float scale_log2;
    float2* part;             // [units][splits][kRows] (max, sum) in the exp2 domain
    float* colsum;            // [units][max_ctx]
    int max_ctx;
    int* status;
};

template <int D, int MT, int PASS>
__global__ void __launch_bounds__(kSkThreads, 1)
    snapkv_score_kernel(const __grid_constant__ CUtensorMap tk, const SkParams p) {
    using S = SkShape<D, MT>;
    constexpr int KSTEPS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint16_t* qs = reinterpret_cast<uint16_t*>(stages + kSkStages * S::kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(qs + S::kRows * S::kQStride);
    uint64_t* empty = full + kSkStages;
    volatile int* abort_flag = reinterpret_cast<int*>(empty + kSkStages);
    float* lse2 = reinterpret_cast<float*>(empty + kSkStages) + 16;   // [kRows]
    float* wsum = lse2 + S::kRows;                                    // [warps][64]

    const int H = p.kv.num_kv_heads;
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / H, h = u % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = p.kv.ctx_len[b];
    if (L < 0 || L > min(p.max_ctx, p.kv.max_pages_per_seq * kPage)) {
        if (threadIdx.x == 0 && split == 0) flag(p.status, SE_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : min(p.max_ctx, p.kv.max_pages_per_seq * kPage);
    }
    const int nblk = (L + kSkBlockKeys - 1) / kSkBlockKeys;
    const int per = (nblk + p.splits - 1) / p.splits;
    const int blk0 = min(nblk, split * per), blk1 = min(nblk, blk0 + per);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSkWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // window queries -> shared memory (rows past M are zero)
    for (int i = threadIdx.x; i < S::kRows * (D / 8); i += blockDim.x) {
        const int r = i / (D / 8), sg = i % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < p.M) {
            const int wi = r / p.G, g = r % p.G;
            v = reinterpret_cast<const uint4*>(
                p.q_win + (((int64_t)b * p.W + wi) * p.Hq + h * p.G + g) * D)[sg];
        }
        *reinterpret_cast<uint4*>(qs + r * S::kQStride + sg * 8) = v;
    }
    if (PASS == 2) {
        // merge the pass-1 partials of every row into lse (exp2 domain)
        for (int r = threadIdx.x; r < S::kRows; r += blockDim.x) {
            float m = -INFINITY, l = 0.f;
            for (int s2 = 0; s2 < p.splits; ++s2) {
                const float2 x = p.part[((int64_t)u * p.splits + s2) * S::kRows + r];
                if (x.y <= 0.f) continue;
                const float mn = fmaxf(m, x.x);
                l = l * exp2f(m - mn) + x.y * exp2f(x.x - mn);
                m = mn;
            }
            lse2[r] = (r < p.M && l > 0.f) ? m + log2f(l) : INFINITY;
        }
    }
    __syncthreads();

    if (warp == kSkWarps) {
        // ---------------- producer: one 64-key block (4 pages) per stage ----------------
        if (lane == 0) {
            prefetch_tmap(&tk);
            const int32_t* bt = p.kv.block_table + (int64_t)b * p.kv.max_pages_per_seq;
            uint32_t seq = 0;
            for (int blk = blk0; blk < blk1; ++blk, ++seq) {
                const int s = seq % kSkStages;
                const uint32_t ph = (seq / kSkStages) & 1;
                if (!*abort_flag && !mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    flag(p.status, SE_DEV_TIMEOUT);
                }
                int rows[4];
                int n = 0;
                for (int pg = 0; pg < 4; ++pg) {
                    const int page = blk * 4 + pg;
                    rows[pg] = -1;
                    if (page * kPage < L) {
                        const int phys = bt[page];
                        if (phys >= 0 && phys < p.kv.num_pages) {
                            rows[pg] = (phys * H + h) * kPage;
                            ++n;
                        } else {
                            flag(p.status, SE_DEV_BAD_INDEX);
                        }
                    }
                }
                if (n > 0 && !*abort_flag) {
                    mbar_arrive_expect_tx(&full[s], n * S::kPageBytes);
                    for (int pg = 0; pg < 4; ++pg) {
                        if (rows[pg] < 0) continue;
#pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_load_2d(stages + s * S::kStageBytes + pg * S::kPageBytes + bx * 2048,
                                        &tk, &full[s], 64 * bx, rows[pg]);
                    }
                } else {
                    mbar_arrive(&full[s]);
                }
            }
            const uint32_t first = seq > (uint32_t)kSkStages ? seq - kSkStages : 0;
            volatile int never = 0;
            for (uint32_t q2 = first; q2 < seq; ++q2)
                mbar_wait(&full[q2 % kSkStages], (q2 / kSkStages) & 1, &never);
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    constexpr int NG = 4;                         // n-tiles (8 keys) per group
    const int r4 = lane >> 2, cq = lane & 3;
    uint32_t qa[MT][KSTEPS][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const int row = warp * 16 * MT + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = kk * 16 + (lane >> 4) * 8;
            ldsm_x4(smem_u32(qs + row * S::kQStride + col), qa[mt][kk][0], qa[mt][kk][1],
                    qa[mt][kk][2], qa[mt][kk][3]);
        }
    // rows of this thread: [mt][half] -> row index, last visible key, lse
    int last_key[MT][2];
    float lrow[MT][2];
    float m[MT][2], l[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int row = warp * 16 * MT + mt * 16 + r4 + hf * 8;
            last_key[mt][hf] = row < p.M ? L - p.W + row / p.G : -1;
            lrow[mt][hf] = PASS == 2 ? lse2[row] : 0.f;
            m[mt][hf] = -INFINITY;
            l[mt][hf] = 0.f;
        }
    const int lj = lane >> 3, lr = lane & 7;

    uint32_t seq = 0;
    for (int blk = blk0; blk < blk1; ++blk, ++seq) {
        const int s = seq % kSkStages;
        const uint32_t ph = (seq / kSkStages) & 1;
        if (!*abort_flag && !mbar_wait(&full[s], ph, abort_flag)) {
            *abort_flag = 1;
            flag(p.status, SE_DEV_TIMEOUT);
        }
        const uint8_t* kb = stages + s * S::kStageBytes;
        const uint32_t kbase = smem_u32(kb);
        float colp[kSkBlockKeys / 8][2];
#pragma unroll
        for (int grp = 0; grp < kSkBlockKeys / 8 / NG; ++grp) {
            float sacc[NG][MT][4];
#pragma unroll
            for (int n = 0; n < NG; ++n)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[n][mt][e] = 0.f;
#pragma unroll
            for (int n = 0; n < NG; ++n) {
                const int nt = grp * NG + n;
                const int keyrow = (nt & 1) * 8 + lr;
#pragma unroll
                for (int k2 = 0; k2 < KSTEPS / 2; ++k2) {
                    const int d = k2 * 32 + lj * 8;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + (nt >> 1) * S::kPageBytes + (d >> 6) * 2048 +
                                swz128(keyrow, (d & 63) >> 3),
                            b0, b1, b2, b3);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        mma_16816(sacc[n][mt], qa[mt][2 * k2][0], qa[mt][2 * k2][1],
                                  qa[mt][2 * k2][2], qa[mt][2 * k2][3], b0, b1);
                        mma_16816(sacc[n][mt], qa[mt][2 * k2 + 1][0], qa[mt][2 * k2 + 1][1],
                                  qa[mt][2 * k2 + 1][2], qa[mt][2 * k2 + 1][3], b2, b3);
                    }
                }
            }
            // mask (causal, past-the-end, padding rows) and scale to the exp2 domain
#pragma unroll
            for (int n = 0; n < NG; ++n)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = blk * kSkBlockKeys + (grp * NG + n) * 8 + 2 * cq + (e & 1);
                        const bool ok = key <= last_key[mt][e >> 1];
                        sacc[n][mt][e] = ok ? sacc[n][mt][e] * p.scale_log2 : -INFINITY;
                    }
            if (PASS == 1) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float mx = m[mt][hf];
#pragma unroll
                        for (int n = 0; n < NG; ++n)
                            mx = fmaxf(mx, fmaxf(sacc[n][mt][2 * hf], sacc[n][mt][2 * hf + 1]));
                        if (mx == -INFINITY) continue;
                        float acc = l[mt][hf] * exp2f(m[mt][hf] - mx);
#pragma unroll
                        for (int n = 0; n < NG; ++n)
                            acc += exp2f(sacc[n][mt][2 * hf] - mx) + exp2f(sacc[n][mt][2 * hf + 1] - mx);
                        l[mt][hf] = acc;
                        m[mt][hf] = mx;
                    }
            } else {
#pragma unroll
                for (int n = 0; n < NG; ++n) {
                    float c0 = 0.f, c1 = 0.f;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        c0 += exp2f(sacc[n][mt][0] - lrow[mt][0]) + exp2f(sacc[n][mt][2] - lrow[mt][1]);
                        c1 += exp2f(sacc[n][mt][1] - lrow[mt][0]) + exp2f(sacc[n][mt][3] - lrow[mt][1]);
                    }
                    colp[grp * NG + n][0] = c0;
                    colp[grp * NG + n][1] = c1;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        if (PASS == 2) {
            // column sums: over this warp's rows (lanes sharing cq), then over warps
#pragma unroll
            for (int nt = 0; nt < kSkBlockKeys / 8; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float x = colp[nt][j];
                    x += __shfl_xor_sync(0xffffffffu, x, 4);
                    x += __shfl_xor_sync(0xffffffffu, x, 8);
                    x += __shfl_xor_sync(0xffffffffu, x, 16);
                    if (r4 == 0) wsum[warp * kSkBlockKeys + nt * 8 + 2 * cq + j] = x;
                }
            asm volatile("bar.sync 1, %0;" ::"r"(kSkWarps * 32) : "memory");
            if (threadIdx.x < kSkBlockKeys) {
                const int key = blk * kSkBlockKeys + threadIdx.x;
                float a = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kSkWarps; ++w2) a += wsum[w2 * kSkBlockKeys + threadIdx.x];
                if (key < L) p.colsum[(int64_t)u * p.max_ctx + key] = a;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kSkWarps * 32) : "memory");
        }
    }
    if (PASS == 1) {
        // merge the four lanes that share each row, then store (max, sum)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float mm = m[mt][hf], ll = l[mt][hf];
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
                    const float l2 = __shfl_xor_sync(0xffffffffu, ll, o);
                    const float mn = fmaxf(mm, m2);
                    if (mn != -INFINITY) {
                        ll = ll * exp2f(mm - mn) + l2 * exp2f(m2 - mn);
                        mm = mn;
                    }
                }
                if (cq == 0) {
                    const int row = warp * 16 * MT + mt * 16 + r4 + hf * 8;
                    p.part[((int64_t)u * p.splits + split) * S::kRows + row] = make_float2(mm, ll);
                }
            }
    }
}

struct SkSelParams {
    se_paged_kv kv;
    se_varlen_kv out;
    const float* colsum;     // [units][max_ctx]
    uint32_t* keys;          // [units][max_ctx], used when the keys do not fit shared memory
    int max_ctx, recent, keep, pool_kernel;
    // span pruning (null: SnapKV, candidates [0, L - recent)): per sequence
    // the candidate span [span[2b], span[2b+1]) and the candidates to keep
    const int32_t* span;
    const int32_t* keep_seq;
    int keys_in_smem;
    int* status;
};
constexpr int kGatherRows = 128;                // kept rows per gather CTA
constexpr int kSelSmemMax = 200 * 1024;         // shared-memory key budget of the select
constexpr int kPoolRegs = 32;                    // scores per thread of the one-round pooling

// The float an order-preserving key was made from (float_key inverted).
__device__ __forceinline__ float sel_key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Threshold of the top K of m keys in ky (lo / hi: the smallest and largest),
// one block of 1024 threads: one histogram pass over kValBins equal-width
// bins of the key VALUES between the smallest and the largest (weakly
// monotone in the key, so every bin above the boundary bin is kept whole and
// every bin below it dropped), then the boundary bin's keys are gathered and
// ranked exactly by (key desc, position asc).  Returns the K-th largest key T
// and in *need_eq how many keys equal to T belong to the top K; a boundary bin
// of more than kValCap keys (many equal or clustered values) takes the radix
// passes instead.  vh: kValBins ints of shared memory.
constexpr int kValBins = 2048, kValCap = 1024;
template <typename KeyAt>
__device__ uint32_t value_select(KeyAt key_at, int m, int K, uint32_t lo, uint32_t hi, int* vh,
                                 int* hist, int* tmp, int* sel, int* need_eq) {
    if (lo == hi) {                                       // every key is equal
        *need_eq = K;
        return hi;
    }
    const int tid = threadIdx.x;
    const float flo = sel_key_float(lo);
    const float scale = static_cast<float>(kValBins) / (sel_key_float(hi) - flo);
    auto bin_of = [&](uint32_t k) {
        const int b = static_cast<int>((sel_key_float(k) - flo) * scale);   // NaN -> 0
        return min(kValBins - 1, max(0, b));
    };
    constexpr int kPer = kValBins / 1024;                 // bins per thread
#pragma unroll
    for (int j = 0; j < kPer; ++j) vh[tid * kPer + j] = 0;
    if (tid == 0) sel[0] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += blockDim.x) atomicAdd(&vh[bin_of(key_at(i))], 1);
    __syncthreads();
    // the boundary bin, scanning from the top (thread t owns bins
    // kValBins-1-kPer*t ..)
    int vv[kPer], v = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        vv[j] = vh[kValBins - 1 - (tid * kPer + j)];
        v += vv[j];
    }
    int total = 0;
    int run = block_exclusive_scan(v, tmp, &total);
    __shared__ int s_bin[3];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (run < K && run + vv[j] >= K) {
            s_bin[0] = kValBins - 1 - (tid * kPer + j);
            s_bin[1] = run;
            s_bin[2] = vv[j];
        }
        run += vv[j];
    }
    __syncthreads();
    const int bstar = s_bin[0], R = K - s_bin[1], E = s_bin[2];
    if (E > kValCap) return block_radix_select(key_at, m, K, hist, tmp, sel, need_eq);
    // the boundary bin's keys and positions, gathered into the free histogram
    uint32_t* bk = reinterpret_cast<uint32_t*>(vh);
    int* bp = vh + kValCap;
    for (int i = tid; i < m; i += blockDim.x) {
        const uint32_t k = key_at(i);
        if (bin_of(k) == bstar) {
            const int at = atomicAdd(&sel[0], 1);
            bk[at] = k;
            bp[at] = i;
        }
    }
    __syncthreads();
    __shared__ uint32_t s_T;
    __shared__ int s_need;
    for (int t = tid; t < E; t += blockDim.x) {
        const uint32_t k = bk[t];
        const int ps = bp[t];
        int rank = 0, above = 0;
        for (int j = 0; j < E; ++j) {
            const uint32_t kj = bk[j];
            rank += kj > k || (kj == k && bp[j] < ps);
            above += kj > k;
        }
        if (rank == R - 1) {                              // the last kept key of the bin
            s_T = k;
            s_need = R - above;
        }
    }
    __syncthreads();
    *need_eq = s_need;
    return s_T;
}

// One CTA (1024 threads) per unit (candidates: SnapKV's prefix before the
// recent window, or a caller's span with every position outside it kept):
// max-pooled candidate scores -> keys (in
// shared memory when they fit), exact top-`keep` by (pooled desc, position
// asc) from one value histogram and the boundary bin's ranks (value_select),
// then the kept positions in ascending
// order (each thread owns a contiguous run of candidates: two block scans
// place them) followed by the recent window.  The rows are gathered by
// snapkv_gather_kernel.
__global__ void __launch_bounds__(1024) snapkv_select_kernel(const SkSelParams p) {
    extern __shared__ uint32_t skeys[];                   // [max_ctx] when keys_in_smem
    __shared__ int hist[256];
    __shared__ int tmp[33];
    __shared__ int sel[2];
    __shared__ int wgt[32], weq[32];
    __shared__ int vh[kValBins];
    __shared__ uint32_t s_lo[32], s_hi[32];
    const int H = p.kv.num_kv_heads;
    const int u = blockIdx.x, b = u / H, h = u % H;
    int L = p.kv.ctx_len[b];
    const int lim = min(p.max_ctx, p.kv.max_pages_per_seq * kPage);
    if (L < 0 || L > lim) {
        if (threadIdx.x == 0 && h == 0) flag(p.status, SE_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : lim;
    }
    // candidates [s0, s1): SnapKV's [0, L - recent), or the caller's span;
    // the positions before and after them are all kept
    int s0 = 0, s1 = L - min(p.recent, L), K = 0;
    if (p.span != nullptr) {
        s0 = min(max(p.span[2 * b], 0), L);
        s1 = min(max(p.span[2 * b + 1], s0), L);
        K = min(max(p.keep_seq[b], 0), s1 - s0);
    } else {
        K = min(p.keep, s1);
    }
    const int ncand = s1 - s0, R = L - s1;
    const int rad = p.pool_kernel / 2;
    const float* A = p.colsum + (int64_t)u * p.max_ctx + s0;
    uint32_t* ky = p.keys_in_smem ? skeys : p.keys + (int64_t)u * p.max_ctx;
    const int nw = blockDim.x >> 5, wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // max-pool over [j-rad, j+rad] clipped to the candidates (rad <= 31)
    uint32_t klo = 0xffffffffu, khi = 0u;         // the keys' smallest and largest
    if (p.keys_in_smem && ncand <= kPoolRegs * 1024) {
        // every score of the unit in flight at once (32 coalesced loads per
        // thread, one latency round), staged in the key area; each thread
        // pools its positions from there into registers, then the keys
        // overwrite the scores in place
        float* sa = reinterpret_cast<float*>(skeys);
        float v[kPoolRegs];
#pragma unroll
        for (int q = 0; q < kPoolRegs; ++q) {
            const int j = q * 1024 + threadIdx.x;
            v[q] = j < ncand ? A[j] : -INFINITY;
        }
#pragma unroll
        for (int q = 0; q < kPoolRegs; ++q) {
            const int j = q * 1024 + threadIdx.x;
            if (j < ncand) sa[j] = v[q];
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kPoolRegs; ++q) {
            const int j = q * 1024 + threadIdx.x;
            float mx = v[q];
            const int t0 = max(0, j - rad), t1 = min(ncand - 1, j + rad);
            for (int t = t0; t <= t1; ++t) mx = fmaxf(mx, sa[t]);
            v[q] = mx;
        }
        __syncthreads();                                  // every window is read
#pragma unroll
        for (int q = 0; q < kPoolRegs; ++q) {
            const int j = q * 1024 + threadIdx.x;
            if (j < ncand) {
                const uint32_t k = float_key(v[q]);
                ky[j] = k;
                klo = min(klo, k);
                khi = max(khi, k);
            }
        }
    } else {
        // a warp takes 32 consecutive positions, one per lane, and its 2*rad
        // neighbours by shuffle (lanes < rad also hold the halo on either side)
        constexpr int kPB = 8;                    // chunks whose loads are in flight together
        for (int jb = wid * 32; jb < ncand; jb += nw * 32 * kPB) {
            float x[kPB], hl[kPB], hr[kPB];
#pragma unroll
            for (int q = 0; q < kPB; ++q) {
                const int j0 = jb + q * nw * 32, j = j0 + lane;
                x[q] = j < ncand ? A[j] : -INFINITY;
                hl[q] = -INFINITY;
                hr[q] = -INFINITY;
                if (lane < rad) {
                    const int jl = j0 - rad + lane, jr = j0 + 32 + lane;
                    if (jl >= 0 && jl < ncand) hl[q] = A[jl];
                    if (jr < ncand) hr[q] = A[jr];
                }
            }
#pragma unroll
            for (int q = 0; q < kPB; ++q) {
                const int j = jb + q * nw * 32 + lane;
                float mx = x[q];
                for (int t = 1; t <= rad; ++t) {
                    const float li = __shfl_sync(0xffffffffu, x[q], (lane - t) & 31);
                    const float lh = __shfl_sync(0xffffffffu, hl[q], (lane - t + rad) & 31);
                    const float ri = __shfl_sync(0xffffffffu, x[q], (lane + t) & 31);
                    const float rh = __shfl_sync(0xffffffffu, hr[q], (lane + t - 32) & 31);
                    mx = fmaxf(mx, fmaxf(lane >= t ? li : lh, lane + t < 32 ? ri : rh));
                }
                if (j < ncand) {
                    const uint32_t k = float_key(mx);
                    ky[j] = k;
                    klo = min(klo, k);
                    khi = max(khi, k);
                }
            }
        }
    }
    klo = __reduce_min_sync(0xffffffffu, klo);
    khi = __reduce_max_sync(0xffffffffu, khi);
    if (lane == 0) {
        s_lo[wid] = klo;
        s_hi[wid] = khi;
    }
    __syncthreads();
    if (wid == 0) {
        klo = __reduce_min_sync(0xffffffffu, lane < nw ? s_lo[lane] : 0xffffffffu);
        khi = __reduce_max_sync(0xffffffffu, lane < nw ? s_hi[lane] : 0u);
        if (lane == 0) {
            s_lo[0] = klo;
            s_hi[0] = khi;
        }
    }
    __syncthreads();
    klo = s_lo[0];
    khi = s_hi[0];

    const int off = p.out.seg_off[u];
    const int cap = p.out.seg_cap;
    const int n_kept = s0 + K + R;
    const int n = min(n_kept, cap);
    if (threadIdx.x == 0 && n_kept > cap) flag(p.status, SE_DEV_CAPACITY);
    const bool off_ok = off >= 0 && (int64_t)off + n <= p.out.total_rows;
    if (threadIdx.x == 0 && !off_ok) flag(p.status, SE_DEV_BAD_INDEX);
    int32_t* pos = p.out.pos + off;
    if (off_ok) {
        for (int j = threadIdx.x; j < s0 && j < cap; j += blockDim.x) pos[j] = j;
        pos += s0;                                        // the candidates' ranks start here
        if (K == ncand) {
            for (int j = threadIdx.x; j < ncand && j + s0 < cap; j += blockDim.x) pos[j] = s0 + j;
        } else if (K > 0) {
            int need_eq;
            const uint32_t T = value_select([&](int i) { return ky[i]; }, ncand, K, klo, khi, vh,
                                            hist, tmp, sel, &need_eq);
            // emit in ascending position: warp w owns a contiguous chunk read
            // with a lane stride; ballots rank the kept keys inside the warp and
            // a scan over the warps places each warp's run.
            const int chunk = ((ncand + nw - 1) / nw + 31) & ~31;
            const int c0 = min(ncand, wid * chunk), c1 = min(ncand, c0 + chunk);
            int gt = 0, eq = 0;
            for (int i = c0 + lane; i < c1; i += 32) {
                const uint32_t kk = ky[i];
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
            // lane l summarises warp l: equal keys before it, then its output offset
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
            int o = __shfl_sync(0xffffffffu, o_incl - g_l - take_l, wid);
            const uint32_t lt = (1u << lane) - 1u;
            for (int i0 = c0; i0 < c1; i0 += 32) {
                const int i = i0 + lane;
                const uint32_t kk = i < c1 ? ky[i] : 0u;
                const bool is_eq = i < c1 && kk == T;
                const uint32_t meq = __ballot_sync(0xffffffffu, is_eq);
                const bool take = (i < c1 && kk > T) ||
                                  (is_eq && eq_seen + __popc(meq & lt) < need_eq);
                const uint32_t mt = __ballot_sync(0xffffffffu, take);
                if (take) {
                    const int at = o + __popc(mt & lt);
                    if (at + s0 < cap) pos[at] = s0 + i;
                }
                o += __popc(mt);
                eq_seen += __popc(meq);
            }
        }
        for (int t = threadIdx.x; t < R; t += blockDim.x)
            if (s0 + K + t < cap) pos[K + t] = s1 + t;
    }
    if (threadIdx.x == 0) {
        p.out.seg_len[u] = off_ok ? n : 0;
        if (h == 0) p.out.seq_len[b] = L;
    }
}

// grid (row blocks, units): copies the kept rows of K and V (and their
// unpooled scores) into the unit's varlen segment, in kept order.  The block's
// rows are resolved first (position, then its physical page: two dependent
// round trips per block, not per copy) into shared memory; then each thread
// issues all of its 16-byte K and V loads before its stores.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads) snapkv_gather_kernel(const SkSelParams p) {
    __shared__ int64_t s_src[kGatherRows];                // source row, -1 when invalid
    const int H = p.kv.num_kv_heads, D = p.kv.head_dim, segs = D / 8;
    const int u = blockIdx.y, b = u / H, h = u % H;
    const int n = p.out.seg_len[u];
    const int off = p.out.seg_off[u];
    const int r0 = blockIdx.x * kGatherRows;
    if (r0 >= n) return;
    const int r1 = min(n, r0 + kGatherRows);
    const int32_t* bt = p.kv.block_table + (int64_t)b * p.kv.max_pages_per_seq;
    const int32_t* pos = p.out.pos + off;
    const float* A = p.colsum + (int64_t)u * p.max_ctx;
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        const int ps = pos[r];
        const int page = ps / kPage;
        const int phys = (ps >= 0 && page < p.kv.max_pages_per_seq) ? bt[page] : -1;
        int64_t src = -1;
        if (phys < 0 || phys >= p.kv.num_pages) {
            flag(p.status, SE_DEV_BAD_INDEX);
        } else {
            src = ((int64_t)phys * H + h) * kPage + ps % kPage;
            if (p.out.score) p.out.score[(int64_t)off + r] = A[ps];
        }
        s_src[r - r0] = src;
    }
    __syncthreads();
    const uint4* Ks = static_cast<const uint4*>(p.kv.k);
    const uint4* Vs = static_cast<const uint4*>(p.kv.v);
    uint4* Kd = static_cast<uint4*>(p.out.k);
    uint4* Vd = static_cast<uint4*>(p.out.v);
    const int total = (r1 - r0) * segs;
    constexpr int kU = 4;                                 // copies of a thread in flight together
    for (int i0 = threadIdx.x; i0 < total; i0 += kGatherThreads * kU) {
        uint4 kv4[kU], vv4[kU];
        int64_t dst[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int i = i0 + q * kGatherThreads;
            dst[q] = -1;
            if (i < total) {
                const int r = i / segs, sg = i % segs;
                const int64_t src = s_src[r];
                if (src >= 0) {
                    kv4[q] = Ks[src * segs + sg];
                    vv4[q] = Vs[src * segs + sg];
                    dst[q] = ((int64_t)off + r0 + r) * segs + sg;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            if (dst[q] >= 0) {
                Kd[dst[q]] = kv4[q];
                Vd[dst[q]] = vv4[q];
            }
        }
    }
}

template <int D, int MT, int PASS>
cudaError_t run_score(const CUtensorMap& tk, const SkParams& p, int units, cudaStream_t s) {
    using S = SkShape<D, MT>;
    auto kern = snapkv_score_kernel<D, MT, PASS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(S::kSmem));
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.splits, units), kSkThreads, S::kSmem, s>>>(tk, p);
    return cudaGetLastError();
}

template <int D, int MT>
cudaError_t run_both(const CUtensorMap& tk, const SkParams& p, int units, cudaStream_t s) {
    cudaError_t e = run_score<D, MT, 1>(tk, p, units, s);
    if (e != cudaSuccess) return e;
    return run_score<D, MT, 2>(tk, p, units, s);
}

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t snapkv_ws_bytes(int units, int max_ctx) {
    return 256 + al256((size_t)units * kSnapMaxSplits * 256 * sizeof(float2)) +
           2 * al256((size_t)units * max_ctx * sizeof(float));
}

cudaError_t launch_snapkv_compact(const se_paged_kv& kv, const void* q_win, int batch, int Hq,
                                  int W, int pool_kernel, int keep, int recent, float scale,
                                  const se_varlen_kv& out, void* ws, int max_ctx, cudaStream_t s,
                                  const int32_t* span, const int32_t* keep_seq) {
    const int H = kv.num_kv_heads, units = batch * H, G = Hq / H, D = kv.head_dim;
    if (units == 0) return cudaSuccess;
    uint8_t* base = static_cast<uint8_t*>(ws);
    SkParams p;
    p.kv = kv;
    p.q_win = static_cast<const uint16_t*>(q_win);
    p.W = W;
    p.Hq = Hq;
    p.G = G;
    p.M = W * G;
    const int nblk = (max_ctx + kSkBlockKeys - 1) / kSkBlockKeys;
    p.splits = max(1, min(kSnapMaxSplits, min(nblk, (num_sms() * 4 + units / 2) / units)));
    p.scale_log2 = scale * kLog2eF;
    p.status = reinterpret_cast<int*>(base);
    size_t off = 256;
    p.part = reinterpret_cast<float2*>(base + off);
    off += al256((size_t)units * kSnapMaxSplits * 256 * sizeof(float2));
    p.colsum = reinterpret_cast<float*>(base + off);
    off += al256((size_t)units * max_ctx * sizeof(float));
    uint32_t* keys = reinterpret_cast<uint32_t*>(base + off);
    p.max_ctx = max_ctx;
    cudaError_t e;
    if (D == 128) {
        // the window-score contraction on the 5th-generation tensor cores
        e = launch_snapkv_scores_tc(kv, q_win, batch, Hq, W, scale, p.part, p.colsum, max_ctx,
                                    p.status, s);
    } else {
        CUtensorMap tk;
        if (!encode_rows_map(&tk, kv.k, (int64_t)kv.num_pages * H * kPage, D))
            return cudaErrorInvalidValue;
        e = p.M <= 128 ? run_both<64, 1>(tk, p, units, s) : run_both<64, 2>(tk, p, units, s);
    }
    if (e != cudaSuccess) return e;
    SkSelParams q;
    q.kv = kv;
    q.out = out;
    q.colsum = p.colsum;
    q.keys = keys;
    q.max_ctx = max_ctx;
    q.recent = recent;
    q.keep = keep;
    q.pool_kernel = pool_kernel;
    q.span = span;
    q.keep_seq = keep_seq;
    q.status = p.status;
    const size_t key_bytes = (size_t)max_ctx * sizeof(uint32_t);
    q.keys_in_smem = key_bytes <= kSelSmemMax;
    const int smem = q.keys_in_smem ? (int)key_bytes : 0;
    e = cudaFuncSetAttribute(snapkv_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    snapkv_select_kernel<<<units, 1024, smem, s>>>(q);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int max_rows = min(out.seg_cap, max_ctx);
    dim3 g((max_rows + kGatherRows - 1) / kGatherRows, units);
    snapkv_gather_kernel<<<g, kGatherThreads, 0, s>>>(q);
    return cudaGetLastError();
}

}  // namespace se
