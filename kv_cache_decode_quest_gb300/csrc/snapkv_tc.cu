// SnapKV window scoring on the 5th-generation tensor cores (head_dim 128).
//
// The observation-window scores are the one dense contraction of the path:
// S = Q K^T with Q the W*G window rows (<= 256) of a KV head and K its prefill
// keys (SnapKV reads how the last query rows attend to the history; tokendh.com
// article on SparseEngine, section "把边界划在'生命周期'上").  Two passes:
//   pass 1: S = Q K^T (M = window rows, N = 128 keys per tile): each epilogue
//           thread owns window rows and keeps their running max / sum of exp2
//           thread-locally -> per-(row, key range) partials;
//   pass 2: S^T = K Q^T (M = 128 keys, N = 256 rows): each epilogue thread owns
//           one key and sums exp2(s - lse_row) over the rows thread-locally ->
//           the column score A[key].
// Dataflow per CTA (one unit, a range of 128-key tiles): a producer warp
// streams the tile's 8 pages with 2-D TMA (128B swizzle) into a 3-stage ring
// laid out as two K-major swizzled regions (head_dim 0..63, 64..127); one
// thread of the MMA warp issues tcgen05.mma (kind::f16, bf16 in, fp32 out)
// into a double-buffered accumulator in tensor memory (2 x 256 columns) and
// commits to mbarriers; eight epilogue warps read the accumulator with
// tcgen05.ld.  Every wait is bounded; tensor memory is freed on every path.
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kTcRows = 256;                       // window rows, padded
constexpr int kTcKeys = 128;                       // keys per tile (8 pages)
constexpr int kTcStages = 4;
constexpr int kTcEpiWarps = 16;                    // 4 per TMEM lane quadrant
constexpr int kTcThreads = (kTcEpiWarps + 2) * 32;  // + TMA producer warp + MMA warp
constexpr int kQRegion = kTcRows * 128;             // one 64-column region of Q (bytes)
constexpr int kKRegion = kTcKeys * 128;             // one 64-column region of a K tile
constexpr int kQBytes = 2 * kQRegion;               // 64 KB
constexpr int kTileBytes = 2 * kKRegion;            // 32 KB
constexpr uint32_t kTmemCols = 512;                 // 2 accumulators x 256 columns
constexpr int kCtrlBytes = 1024;                    // barriers, TMEM slot, flags
constexpr size_t kTcSmem = 1024 + kQBytes + (size_t)kTcStages * kTileBytes + kCtrlBytes +
                           kTcRows * 4 /* lse */ + 4096 /* partial-merge buffer */;
constexpr float kLog2e = 1.4426950408889634f;

struct TcParams {
    se_paged_kv kv;
    const uint16_t* q_win;   // [B][W][Hq][128]
    int W, Hq, G, M;
    int splits;
    float scale_log2;
    float2* part;            // [units][splits][kTcRows] (max, sum) in the exp2 domain
    float* colsum;           // [units][max_ctx]
    int max_ctx;
    int* status;
};

__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"r"(kTcEpiWarps * 32) : "memory");
}

template <int PASS>
__global__ void __launch_bounds__(kTcThreads, 1)
    snapkv_score_tc_kernel(const __grid_constant__ CUtensorMap tk, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* qs = smem;
    uint8_t* kst = smem + kQBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(kst + kTcStages * kTileBytes);
    uint64_t* empty = full + kTcStages;
    uint64_t* tfull = empty + kTcStages;               // [2]
    uint64_t* tempty = tfull + 2;                       // [2]
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    float* nlse2 = reinterpret_cast<float*>(kst + kTcStages * kTileBytes + kCtrlBytes);
    float* halfbuf = nlse2 + kTcRows;                   // 1024 floats

    const int H = p.kv.num_kv_heads;
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / H, h = u % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = p.kv.ctx_len[b];
    const int lim = min(p.max_ctx, p.kv.max_pages_per_seq * kPage);
    if (L < 0 || L > lim) {
        if (threadIdx.x == 0 && split == 0) flag(p.status, SE_DEV_BAD_LENGTH);
        L = L < 0 ? 0 : lim;
    }
    const int ntile = (L + kTcKeys - 1) / kTcKeys;
    const int per = (ntile + p.splits - 1) / p.splits;
    const int t0 = min(ntile, split * per), t1 = min(ntile, t0 + per);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kTcEpiWarps);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // window queries -> the two 128B-swizzled regions (rows past M are zero)
    const uint4* q4 = reinterpret_cast<const uint4*>(p.q_win);
    const int lg = __ffs(p.G) - 1;                      // G is a power of two
    for (int i = threadIdx.x; i < kTcRows * 16; i += blockDim.x) {
        const int r = i >> 4, c16 = i & 15;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < p.M) {
            const int wi = r >> lg, g = r & (p.G - 1);
            v = q4[((((int64_t)b * p.W + wi) * p.Hq + h * p.G + g) * 128) / 8 + c16];
        }
        *reinterpret_cast<uint4*>(qs + (c16 >> 3) * kQRegion + r * 128 +
                                  (((c16 & 7) ^ (r & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();                           // visible to the tensor cores
    if (PASS == 2) {
        for (int r = threadIdx.x; r < kTcRows; r += blockDim.x) {
            float m = -INFINITY, l = 0.f;
            for (int s2 = 0; s2 < p.splits; ++s2) {
                const float2 x = p.part[((int64_t)u * p.splits + s2) * kTcRows + r];
                if (x.y <= 0.f) continue;
                const float mn = fmaxf(m, x.x);
                l = l * exp2f(m - mn) + x.y * exp2f(x.x - mn);
                m = mn;
            }
            // minus the row's log2-sum-exp2; padding rows get -inf (weight 0)
            nlse2[r] = (r < p.M && l > 0.f) ? -(m + log2f(l)) : -INFINITY;
        }
    }
    if (warp == kTcEpiWarps + 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcEpiWarps) {
        // ------------------------------ TMA producer ------------------------------
        // Lane pg < 8 owns page pg of a tile: its block-table entry is read two
        // tiles ahead, and lanes 0..15 issue the tile's 16 boxes (page lane&7,
        // head_dim half lane>>3) together.
        if (lane == 0) prefetch_tmap(&tk);
        const int32_t* bt = p.kv.block_table + (int64_t)b * p.kv.max_pages_per_seq;
        auto fetch = [&](int kb) -> int {              // -2: no page (past the tile range or L)
            const int page = kb * 8 + (lane & 7);
            return (kb < t1 && page * kPage < L) ? bt[page] : -2;
        };
        int nxt1 = fetch(t0), nxt2 = fetch(t0 + 1);
        uint32_t seq = 0;
        for (int kb = t0; kb < t1; ++kb, ++seq) {
            const int s = seq % kTcStages;
            const int cur = nxt1;
            nxt1 = nxt2;
            nxt2 = fetch(kb + 2);
            int row = -1;
            if (cur != -2) {
                if (cur >= 0 && cur < p.kv.num_pages) {
                    row = (cur * H + h) * kPage;
                } else if (lane < 8) {
                    flag(p.status, SE_DEV_BAD_INDEX);
                }
            }
            const int n = __popc(__ballot_sync(0xffffffffu, lane < 8 && row >= 0));
            int go = 0;
            if (lane == 0) {
                go = !*abort_flag;
                if (go && !mbar_wait(&empty[s], ((seq / kTcStages) & 1) ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    flag(p.status, SE_DEV_TIMEOUT);
                    go = 0;
                }
                if (go && n > 0) mbar_arrive_expect_tx(&full[s], n * 4096);
                else mbar_arrive(&full[s]);
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            const int rowpg = __shfl_sync(0xffffffffu, row, lane & 7);
            if (go && lane < 16 && rowpg >= 0) {
                const int half = lane >> 3;
                tma_load_2d(kst + s * kTileBytes + half * kKRegion + (lane & 7) * 2048, &tk,
                            &full[s], half * 64, rowpg);
            }
        }
        if (lane == 0) {
            // the last stages' copies have landed before the block exits
            const uint32_t first = seq > (uint32_t)kTcStages ? seq - kTcStages : 0;
            volatile int never = 0;
            for (uint32_t q2 = first; q2 < seq; ++q2)
                mbar_wait(&full[q2 % kTcStages], (q2 / kTcStages) & 1, &never);
        }
        __syncwarp();
    } else if (warp == kTcEpiWarps + 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(qs);
            uint32_t seq = 0;
            for (int kb = t0; kb < t1; ++kb, ++seq) {
                const int s = seq % kTcStages, buf = seq & 1;
                if (!*abort_flag && !mbar_wait(&full[s], (seq / kTcStages) & 1, abort_flag)) {
                    *abort_flag = 1;
                    flag(p.status, SE_DEV_TIMEOUT);
                }
                if (!*abort_flag && !mbar_wait(&tempty[buf], ((seq >> 1) & 1) ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    flag(p.status, SE_DEV_TIMEOUT);
                }
                tc_fence_after();
                if (!*abort_flag) {
                    const uint32_t k_addr = smem_u32(kst + s * kTileBytes);
                    const uint32_t acc = tmem + buf * 256;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t koff = (ks >> 2) * kKRegion + (ks & 3) * 32;
                        const uint32_t qoff = (ks >> 2) * kQRegion + (ks & 3) * 32;
                        if (PASS == 1) {
#pragma unroll
                            for (int t = 0; t < 2; ++t)
                                umma_bf16(acc + t * 128, umma_desc_sw128(q_addr + qoff + t * 128 * 128),
                                          umma_desc_sw128(k_addr + koff),
                                          umma_idesc_bf16_f32(128, 128), ks > 0);
                        } else {
                            umma_bf16(acc, umma_desc_sw128(k_addr + koff),
                                      umma_desc_sw128(q_addr + qoff),
                                      umma_idesc_bf16_f32(128, 256), ks > 0);
                        }
                    }
                }
                umma_commit(&empty[s]);                 // the K stage is free once read
                umma_commit(&tfull[buf]);               // the accumulator is ready
            }
            umma_commit(done);                          // every MMA of this CTA has finished
            volatile int never = 0;
            mbar_wait(done, 0, &never);
        }
    } else {
        // ------------------------------ epilogue warps ------------------------------
        // warp w reads TMEM lanes 32*(w%4) .. +31 (its lane quadrant); the four
        // warps of a quadrant split the accumulator's 256 columns four ways.
        const int qd = warp & 3, part = warp >> 2;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        // pass 1: row t*128 + 32*qd + lane, keys hf*64 .. hf*64+63 of the tile
        const int t = part >> 1, hf = part & 1;
        const int row1 = t * 128 + 32 * qd + lane;
        const int last1 = row1 < p.M ? L - p.W + (row1 >> lg) : -1;
        float m1 = -INFINITY, l1 = 0.f;
        uint32_t seq = 0;
        for (int kb = t0; kb < t1; ++kb, ++seq) {
            const int buf = seq & 1;
            if (!*abort_flag && !mbar_wait(&tfull[buf], (seq >> 1) & 1, abort_flag)) {
                *abort_flag = 1;
                flag(p.status, SE_DEV_TIMEOUT);
            }
            tc_fence_after();
            const bool live = !*abort_flag;
            // every window row sees every key of the tile: no per-element mask
            // (keys <= L-W are visible to all rows, and L-W < L)
            const bool full_tile = (kb + 1) * kTcKeys - 1 <= L - p.W;
            float v[64];
            if (live) {
                tmem_ld64(lane_base + buf * 256 + (PASS == 1 ? t * 128 + hf * 64 : part * 64), v);
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) v[j] = 0.f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);   // the accumulator is in registers
            if (PASS == 1) {
                float mx;
                if (full_tile && p.scale_log2 > 0.f) {
                    // max over the raw logits (the scale is positive), four chains
                    float r4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
                    for (int j = 4; j < 64; ++j) r4[j & 3] = fmaxf(r4[j & 3], v[j]);
                    mx = fmaxf(m1, fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3])) * p.scale_log2);
                    const float nmx = -mx;
                    float a4[4] = {l1 * ex2_approx(m1 - mx), 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 64; ++j) a4[j & 3] += ex2_approx(fmaf(v[j], p.scale_log2, nmx));
                    l1 = (a4[0] + a4[1]) + (a4[2] + a4[3]);
                    m1 = mx;
                } else {
                    // masked tile (or a non-positive scale): scale first, then mask
                    const int key0 = kb * kTcKeys + hf * 64;
                    float r4[4] = {m1, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        v[j] = (full_tile || key0 + j <= last1) ? v[j] * p.scale_log2 : -INFINITY;
                        r4[j & 3] = fmaxf(r4[j & 3], v[j]);
                    }
                    mx = fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3]));
                    if (mx != -INFINITY) {
                        float a4[4] = {l1 * ex2_approx(m1 - mx), 0.f, 0.f, 0.f};
#pragma unroll
                        for (int j = 0; j < 64; ++j) a4[j & 3] += ex2_approx(v[j] - mx);
                        l1 = (a4[0] + a4[1]) + (a4[2] + a4[3]);
                        m1 = mx;
                    }
                }
            } else {
                // key kb*128 + 32*qd + lane against rows part*64 .. part*64+63
                const int key = kb * kTcKeys + 32 * qd + lane;
                const float4* nl4 = reinterpret_cast<const float4*>(nlse2 + part * 64);
                float acc = 0.f;
                if (full_tile) {
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        const float4 nl = nl4[j4];
                        acc += ex2_approx(fmaf(v[4 * j4], p.scale_log2, nl.x));
                        acc += ex2_approx(fmaf(v[4 * j4 + 1], p.scale_log2, nl.y));
                        acc += ex2_approx(fmaf(v[4 * j4 + 2], p.scale_log2, nl.z));
                        acc += ex2_approx(fmaf(v[4 * j4 + 3], p.scale_log2, nl.w));
                    }
                } else {
                    // row r sees this key iff key <= L-W + r/G, i.e. r >= G*max(0, key-(L-W))
                    const int min_row = key < L ? max(0, key - (L - p.W)) << lg : kTcRows;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const int row = part * 64 + j;
                        const float e = ex2_approx(fmaf(v[j], p.scale_log2, nlse2[row]));
                        acc += row >= min_row ? e : 0.f;
                    }
                }
                // the four row quarters meet in shared memory (double-buffered by
                // tile parity, so one barrier per tile suffices)
                float* hb = halfbuf + buf * 512;
                if (part != 0) hb[part * 128 + 32 * qd + lane] = acc;
                epi_bar();
                if (part == 0 && key < L) {
                    const int i = 32 * qd + lane;
                    p.colsum[(int64_t)u * p.max_ctx + key] = acc + hb[128 + i] + hb[256 + i] + hb[384 + i];
                }
            }
        }
        if (PASS == 1) {
            // merge the two key halves of each row, then store (max, sum)
            if (hf == 1) {
                halfbuf[2 * row1] = m1;
                halfbuf[2 * row1 + 1] = l1;
            }
            epi_bar();
            if (hf == 0) {
                const float m2 = halfbuf[2 * row1], l2 = halfbuf[2 * row1 + 1];
                float mm = m1, ll = l1;
                const float mn = fmaxf(mm, m2);
                if (mn != -INFINITY) {
                    ll = ll * exp2f(mm - mn) + l2 * exp2f(m2 - mn);
                    mm = mn;
                }
                p.part[((int64_t)u * p.splits + split) * kTcRows + row1] = make_float2(mm, ll);
            }
        }
    }
    // every role is done (producer drained, MMAs completed, loads finished)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcEpiWarps + 1) tmem_dealloc(tmem, kTmemCols);
}

template <int PASS>
cudaError_t run_tc(const CUtensorMap& tk, const TcParams& p, int units, cudaStream_t s) {
    auto kern = snapkv_score_tc_kernel<PASS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kTcSmem));
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.splits, units), kTcThreads, kTcSmem, s>>>(tk, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_snapkv_scores_tc(const se_paged_kv& kv, const void* q_win, int batch, int Hq,
                                    int W, float scale, float2* part, float* colsum, int max_ctx,
                                    int* status, cudaStream_t s) {
    const int H = kv.num_kv_heads, units = batch * H;
    if (units == 0) return cudaSuccess;
    TcParams p;
    p.kv = kv;
    p.q_win = static_cast<const uint16_t*>(q_win);
    p.W = W;
    p.Hq = Hq;
    p.G = Hq / H;
    p.M = W * p.G;
    const int ntile = (max_ctx + kTcKeys - 1) / kTcKeys;
    p.splits = max(1, min(ntile, min(kSnapMaxSplitsTc, num_sms() / units)));
    p.scale_log2 = scale * kLog2e;
    p.part = part;
    p.colsum = colsum;
    p.max_ctx = max_ctx;
    p.status = status;
    CUtensorMap tk;
    if (!encode_rows_map(&tk, kv.k, (int64_t)kv.num_pages * H * kPage, 128))
        return cudaErrorInvalidValue;
    cudaError_t e = run_tc<1>(tk, p, units, s);
    if (e != cudaSuccess) return e;
    return run_tc<2>(tk, p, units, s);
}

}  // namespace se
