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
// One pass over the unit's tokens does the usual step whole: the score update
// (written in place), the count of the recent window and the victim among the
// others (lowest score, then the higher position) with its slot, reduced
// over the block once.  Only when the newest `recent` positions are not all
// held does a second, exact pass select the recent window (a radix selection
// of the `recent` largest positions) and look for the victim again.
constexpr int kEvictThreads = 512;
// G4 = G / 4 (a compile-time count of 16-byte logit vectors per token, so a
// thread's loads for several tokens are issued together), or 0 for G = 1, 2.
template <int G4>
__global__ void __launch_bounds__(kEvictThreads) h2o_evict_kernel(const EvictParams p) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_lse[16];
    __shared__ int hist[256];
    __shared__ int tmp[33];
    __shared__ int sel[2];
    __shared__ unsigned long long s_best[32];
    __shared__ int s_slot[32], s_cnt[32];
    const int H = p.kv.num_kv_heads, segs = p.kv.head_dim / 8;
    const int u = blockIdx.x, b = u / H, h = u % H;
    const int G = p.G;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
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
    __syncthreads();

    float* score = p.kv.score + off;
    int32_t* pos = p.kv.pos + off;
    const bool evict = n > p.budget;
    // the recent window when its newest `recent` positions are all held (the
    // usual case): positions above new_pos - recent
    const int new_pos = p.kv.seq_len[b] - 1;
    int thr = new_pos - p.recent;
    // the victim key: float_key(score) high, then the higher position first
    auto victim_key = [](float sc, int ps) {
        return (static_cast<unsigned long long>(float_key(sc)) << 32) |
               static_cast<unsigned long long>(0x7fffffffu - static_cast<uint32_t>(ps));
    };
    // 1. score update with this step's normalised probabilities (a token's G
    //    logits as 16-byte vectors when G % 4 == 0), the recent count and the
    //    thread's victim candidate, all in one pass
    const float* lg = p.logits + (int64_t)u * p.stride * G;
    int c = 0, best_slot = -1;
    unsigned long long best = ~0ull;
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
        const float sc = score[t] + pr;
        score[t] = sc;
        if (evict) {
            const int ps = pos[t];
            c += ps > thr;
            if (ps <= thr) {
                const unsigned long long key = victim_key(sc, ps);
                if (key < best) {
                    best = key;
                    best_slot = t;
                }
            }
        }
    }
    if (!evict) {
        if (threadIdx.x == 0) p.evicted_pos[u] = -1;
        return;
    }
    // the block's recent count and victim (key, slot)
    auto reduce = [&](int cnt) {
        cnt = __reduce_add_sync(0xffffffffu, cnt);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
            const int ys = __shfl_xor_sync(0xffffffffu, best_slot, o);
            if (y < best) {
                best = y;
                best_slot = ys;
            }
        }
        if (lane == 0) {
            s_best[wid] = best;
            s_slot[wid] = best_slot;
            s_cnt[wid] = cnt;
        }
        __syncthreads();                                  // every score is written too
        if (wid == 0) {
            best = lane < nw ? s_best[lane] : ~0ull;
            best_slot = lane < nw ? s_slot[lane] : -1;
            cnt = __reduce_add_sync(0xffffffffu, lane < nw ? s_cnt[lane] : 0);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
                const int ys = __shfl_xor_sync(0xffffffffu, best_slot, o);
                if (y < best) {
                    best = y;
                    best_slot = ys;
                }
            }
            if (lane == 0) {
                s_best[0] = best;
                s_slot[0] = best_slot;
                s_cnt[0] = cnt;
            }
        }
        __syncthreads();
        best = s_best[0];
        best_slot = s_slot[0];
        return s_cnt[0];
    };
    const int held_recent = reduce(c);
    __syncthreads();                                      // s_* are rewritten below
    if (held_recent != p.recent) {
        // 2. the exact recent window: the `recent` largest positions
        int need_eq;
        const uint32_t T = block_radix_select(
            [&](int i) { return static_cast<uint32_t>(pos[i]) ^ 0x80000000u; }, n,
            min(p.recent, n), hist, tmp, sel, &need_eq);
        thr = static_cast<int>(T ^ 0x80000000u) - 1;     // positions are unique
        best = ~0ull;
        best_slot = -1;
#pragma unroll 4
        for (int t = threadIdx.x; t < n; t += blockDim.x) {
            const int ps = pos[t];
            if (ps > thr) continue;
            const unsigned long long key = victim_key(score[t], ps);
            if (key < best) {
                best = key;
                best_slot = t;
            }
        }
        reduce(0);
    }
    if (best == ~0ull) {   // no candidate (recent >= n): nothing can be evicted
        if (threadIdx.x == 0) p.evicted_pos[u] = -1;
        return;
    }
    const int victim_pos = static_cast<int>(0x7fffffffu - static_cast<uint32_t>(best & 0xffffffffu));
    // 3. move the last slot into the victim's
    const int v = best_slot, last = n - 1;
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
        }
    }
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
    auto go = [&](auto kern) -> cudaError_t {
        kern<<<units, kEvictThreads, 0, s>>>(p);
        return cudaGetLastError();
    };
    switch (G) {
        case 4:  return go(h2o_evict_kernel<1>);
        case 8:  return go(h2o_evict_kernel<2>);
        case 16: return go(h2o_evict_kernel<4>);
        default: return go(h2o_evict_kernel<0>);
    }
}

}  // namespace se
