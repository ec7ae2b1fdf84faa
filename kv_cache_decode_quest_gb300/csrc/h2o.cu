// H2O decode step: accumulated-attention score update and heavy-hitter +
// recent-window eviction.
//
// H2O keeps a running accumulated attention score per retained token, updates
// it at every decode step and then decides which token to delete, physically
// (tokendh.com article on SparseEngine, sections "历史太长,会撑爆什么" and
// "把边界划在'生命周期'上").
//
// One step for unit u = (b, h), held tokens in slots [0, n) of its segment:
//   1. append: the new token goes to slot n with pos = seq_len[b], score 0
//      (the varlen append kernel);
//   2. decode attention over the n+1 slots, with every token's logits
//      s[g,t] saved (the split-K decode kernel, logits mode);
//   3. h2o_evict_kernel: score[t] += sum_g exp(s[g,t] - lse[g]); if more than
//      `budget` tokens are held, the token ranked last under (score desc,
//      position asc) among those whose position is not one of the `recent`
//      largest is evicted, and the last slot's token moves into its slot, so
//      the held tokens stay contiguous.
#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

struct EvictParams {
    se_varlen_kv kv;
    int budget, recent, G, Hq;
    const float* logits;      // [units][stride][G]
    int stride;
    const float* lse;         // [B][Hq]
    int32_t* evicted_pos;     // [units]
    int* status;
};

// 512 threads: two blocks per SM, so one block per unit runs in a single wave.
// STAGED: the unit's positions and scores are read once into shared memory
// (all loads in flight), every later pass reads them there, and the updated
// scores go back in one pass; used when 8 * seg_cap bytes fit kEvictStageMax.
constexpr int kEvictThreads = 512;
constexpr int kEvictStageMax = 96 * 1024;
// G4 = G / 4 (a compile-time count of 16-byte logit vectors per token, so a
// thread's loads for several tokens are issued together), or 0 for G = 1, 2.
template <bool STAGED, int G4>
__global__ void __launch_bounds__(kEvictThreads) h2o_evict_kernel(const EvictParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t stage[];                  // STAGED: [seg_cap] pos, [seg_cap] score
    __shared__ float s_lse[16];
    __shared__ int hist[256];
    __shared__ int tmp[33];
    __shared__ int sel[2];
    __shared__ unsigned long long s_best[32];
    __shared__ int s_cnt;
    const int H = p.kv.num_kv_heads, segs = p.kv.head_dim / 8;
    const int u = blockIdx.x, b = u / H, h = u % H;
    const int G = p.G;
    int n = p.kv.seg_len[u];
    const int off = p.kv.seg_off[u];
    if (n < 0 || n > p.kv.seg_cap || off < 0 || (int64_t)off + n > p.kv.total_rows) {
        if (threadIdx.x == 0) {
            flag(p.status, SE_DEV_BAD_LENGTH);
            p.evicted_pos[u] = -1;
        }
        return;
    }
    if (threadIdx.x < G) s_lse[threadIdx.x] = p.lse[(int64_t)b * p.Hq + h * G + threadIdx.x];
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();

    float* gscore = p.kv.score + off;
    int32_t* gpos = p.kv.pos + off;
    int32_t* pos = STAGED ? stage : gpos;
    float* score = STAGED ? reinterpret_cast<float*>(stage + p.kv.seg_cap) : gscore;
    // 1. score update with this step's normalised probabilities (a token's G
    //    logits as 16-byte vectors when G % 4 == 0), positions staged alongside
    const float* lg = p.logits + (int64_t)u * p.stride * G;
#pragma unroll 4
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        float pr = 0.f;
        if (G4 > 0) {
            const float4* l4 = reinterpret_cast<const float4*>(lg + (int64_t)t * G);
#pragma unroll
            for (int j = 0; j < G4; ++j) {
                const float4 x = l4[j];
                pr += __expf(x.x - s_lse[4 * j]) + __expf(x.y - s_lse[4 * j + 1]) +
                      __expf(x.z - s_lse[4 * j + 2]) + __expf(x.w - s_lse[4 * j + 3]);
            }
        } else {
            for (int g = 0; g < G; ++g) pr += __expf(lg[(int64_t)t * G + g] - s_lse[g]);
        }
        score[t] = gscore[t] + pr;
        if (STAGED) pos[t] = gpos[t];
    }
    __syncthreads();
    // the updated scores go back to the cache (STAGED), after any move
    auto write_back = [&](int count) {
        if (STAGED)
            for (int t = threadIdx.x; t < count; t += blockDim.x) gscore[t] = score[t];
    };
    if (n <= p.budget) {
        write_back(n);
        if (threadIdx.x == 0) p.evicted_pos[u] = -1;
        return;
    }
    // 2. the recent window: positions above new_pos - recent when the newest
    //    `recent` positions are all held (the usual case), else an exact
    //    selection of the `recent` largest positions.
    const int new_pos = p.kv.seq_len[b] - 1;
    int thr = new_pos - p.recent;            // candidates: pos <= thr
    int c = 0;
#pragma unroll 4
    for (int t = threadIdx.x; t < n; t += blockDim.x) c += pos[t] > thr;
    atomicAdd(&s_cnt, c);
    __syncthreads();
    if (s_cnt != p.recent) {
        int need_eq;
        const uint32_t T = block_radix_select(
            [&](int i) { return static_cast<uint32_t>(pos[i]) ^ 0x80000000u; }, n,
            min(p.recent, n), hist, tmp, sel, &need_eq);
        thr = static_cast<int>(T ^ 0x80000000u) - 1;   // positions are unique
    }
    // 3. victim: lowest score, then the higher position
    unsigned long long best = ~0ull;
#pragma unroll 4
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const int ps = pos[t];
        if (ps > thr) continue;
        const unsigned long long key =
            (static_cast<unsigned long long>(float_key(score[t])) << 32) |
            static_cast<unsigned long long>(0x7fffffffu - static_cast<uint32_t>(ps));
        best = key < best ? key : best;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
        best = y < best ? y : best;
    }
    if ((threadIdx.x & 31) == 0) s_best[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        best = threadIdx.x < (blockDim.x >> 5) ? s_best[threadIdx.x] : ~0ull;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
            best = y < best ? y : best;
        }
        if (threadIdx.x == 0) s_best[0] = best;
    }
    __syncthreads();
    best = s_best[0];
    if (best == ~0ull) {   // no candidate (recent >= n): nothing can be evicted
        write_back(n);
        if (threadIdx.x == 0) p.evicted_pos[u] = -1;
        return;
    }
    const int victim_pos = static_cast<int>(0x7fffffffu - static_cast<uint32_t>(best & 0xffffffffu));
    // 4. find the victim's slot, then move the last slot into it
    __shared__ int s_slot;
#pragma unroll 4
    for (int t = threadIdx.x; t < n; t += blockDim.x)
        if (pos[t] == victim_pos) s_slot = t;
    __syncthreads();
    const int v = s_slot, last = n - 1;
    if (v != last) {
        uint4* K = static_cast<uint4*>(p.kv.k) + (int64_t)off * segs;
        uint4* V = static_cast<uint4*>(p.kv.v) + (int64_t)off * segs;
        for (int i = threadIdx.x; i < segs; i += blockDim.x) {
            K[(int64_t)v * segs + i] = K[(int64_t)last * segs + i];
            V[(int64_t)v * segs + i] = V[(int64_t)last * segs + i];
        }
        if (threadIdx.x == 0) {
            pos[v] = pos[last];
            score[v] = score[last];
            if (STAGED) gpos[v] = pos[last];
        }
    }
    __syncthreads();
    write_back(n - 1);
    if (threadIdx.x == 0) {
        p.evicted_pos[u] = victim_pos;
        p.kv.seg_len[u] = n - 1;
    }
}

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Workspace: the decode workspace first (its header, with the status word at
// byte 0, and its arrival counters stay at fixed offsets whatever the shape),
// then logits [units][stride][G] | lse [B][Hq] | view chunk_row [units][chunks]
// | view n_tokens [units].
size_t h2o_ws_bytes(int batch, int Hkv, int Hq, int D, int seg_cap) {
    const int units = batch * Hkv, G = Hq / Hkv;
    const int chunks = (seg_cap + kPage - 1) / kPage;
    const size_t stride = (size_t)chunks * kPage;
    return decode_ws_bytes(units, G, D, SE_MAX_SPLITS) +
           al256((size_t)units * stride * G * sizeof(float)) +
           al256((size_t)batch * Hq * sizeof(float)) + al256((size_t)units * chunks * sizeof(int)) +
           al256((size_t)units * sizeof(int));
}

cudaError_t launch_h2o_step(const se_h2o_state& st, const void* q, const void* k_new,
                            const void* v_new, int batch, int Hq, float scale, int out_dtype,
                            void* out, float* lse, int32_t* evicted_pos, void* ws,
                            cudaStream_t s) {
    const se_varlen_kv& kv = st.kv;
    const int Hkv = kv.num_kv_heads, D = kv.head_dim, units = batch * Hkv, G = Hq / Hkv;
    if (units == 0) return cudaSuccess;
    const int chunks = (kv.seg_cap + kPage - 1) / kPage;
    const int stride = chunks * kPage;
    uint8_t* base = static_cast<uint8_t*>(ws);
    DecodeWs w = decode_ws_carve(base, units, G, D, SE_MAX_SPLITS);
    int* status = w.status;
    size_t off = decode_ws_bytes(units, G, D, SE_MAX_SPLITS);
    float* logits = reinterpret_cast<float*>(base + off);
    off += al256((size_t)units * stride * G * sizeof(float));
    float* lse_int = reinterpret_cast<float*>(base + off);
    off += al256((size_t)batch * Hq * sizeof(float));
    se_view view;
    view.chunk_row = reinterpret_cast<int32_t*>(base + off);
    off += al256((size_t)units * chunks * sizeof(int));
    view.n_tokens = reinterpret_cast<int32_t*>(base + off);
    view.num_units = units;
    view.max_chunks = chunks;

    cudaError_t e = launch_varlen_append_view(kv, k_new, v_new, batch, view, status, s);
    if (e != cudaSuccess) return e;
    float* lse_used = lse ? lse : lse_int;
    e = launch_sparse_decode(kv.k, kv.v, kv.total_rows, view, q, batch, Hq, Hkv, D, scale,
                             out_dtype, SE_MAX_SPLITS, logits, stride, nullptr, nullptr, out,
                             lse_used, w, s);
    if (e != cudaSuccess) return e;
    EvictParams p;
    p.kv = kv;
    p.budget = st.budget;
    p.recent = st.recent;
    p.G = G;
    p.Hq = Hq;
    p.logits = logits;
    p.stride = stride;
    p.lse = lse_used;
    p.evicted_pos = evicted_pos;
    p.status = status;
    const size_t stage_bytes = (size_t)8 * kv.seg_cap;
    const bool staged = stage_bytes <= kEvictStageMax;
    auto go = [&](auto kern) -> cudaError_t {
        const size_t smem = staged ? stage_bytes : 0;
        cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (e2 != cudaSuccess) return e2;
        kern<<<units, kEvictThreads, smem, s>>>(p);
        return cudaGetLastError();
    };
    switch (G) {
        case 4:  return staged ? go(h2o_evict_kernel<true, 1>) : go(h2o_evict_kernel<false, 1>);
        case 8:  return staged ? go(h2o_evict_kernel<true, 2>) : go(h2o_evict_kernel<false, 2>);
        case 16: return staged ? go(h2o_evict_kernel<true, 4>) : go(h2o_evict_kernel<false, 4>);
        default: return staged ? go(h2o_evict_kernel<true, 0>) : go(h2o_evict_kernel<false, 0>);
    }
}

}  // namespace se
