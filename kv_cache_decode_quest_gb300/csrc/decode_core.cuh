// The consumer side of the split-K GQA decode: per 16-token chunk in shared
// memory, S^T = K Q^T (tokens as M = 16, the GQA group as N = 8) with ldmatrix +
// mma.sync.m16n8k16 (bf16 -> fp32), an online softmax in the exp2 domain, P
// transposed in registers (movmatrix) and O^T += V^T P^T (head_dim as M); at the
// end of a piece the four consumer warps merge through shared memory, and a unit
// cut into several pieces is merged by the last of them to finish (an arrival
// counter per unit, log-sum-exp weights).  Shared by the decode kernel and the
// fused Quest step kernel.
//
// The attention reads only the rows the view exposes ("SparseEngine：稀疏优先推理
// 引擎", section "方法 / 关键模块"); the pieces of one unit are combined by their
// log-sum-exp, which is exact for softmax attention split over disjoint token sets.
#pragma once

#include "common.cuh"

namespace se {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int NT>
struct DecShape {
    static constexpr int kBoxes = D / 64;                  // 64-column TMA boxes per chunk
    static constexpr int kChunkBytes = kBoxes * 2048;      // 16 rows x D bf16
    static constexpr int kStageBytes = 2 * kChunkBytes;    // K chunk then V chunk
    static constexpr int kHeads = NT * 8;                  // padded group
    // per warp m and l; two weighted O slots (kHeads x D); per-warp head
    // weights and the LSE
    static constexpr int kMergeFloats =
        kConsumerWarps * kHeads * 2 + 2 * kHeads * D + (kConsumerWarps + 1) * kHeads;
};

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One consumer warp's running softmax state for one unit.
template <int D, int NT>
struct DecState {
    uint32_t qf[D / 16][NT][2];
    float m[NT][2], l[NT][2], o[D / 16][NT][4];
};

// Query fragments of unit (b, h) (the B operand: group member as N, d as K)
// and an empty softmax state.  qhead0 = b * Hq + h * G.
template <int D, int NT>
__device__ __forceinline__ void dec_begin(DecState<D, NT>& st, const uint16_t* q, int64_t qhead0,
                                          int G, int lane) {
    constexpr int KSTEPS = D / 16;
    const int r = lane >> 2, cq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int g = nt * 8 + r;
        const uint16_t* qrow = q + (qhead0 + min(g, G - 1)) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t x0 = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * cq);
            const uint32_t x1 = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * cq);
            st.qf[kk][nt][0] = g < G ? x0 : 0u;
            st.qf[kk][nt][1] = g < G ? x1 : 0u;
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        st.m[nt][0] = st.m[nt][1] = -INFINITY;
        st.l[nt][0] = st.l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[mt][nt][e] = 0.f;
    }
}

// One chunk of cnt (1..16) valid rows: K at kb, V at kb + kChunkBytes, both
// 16 rows x D bf16 in 64-column boxes with the 128-byte swizzle.  logits, when
// not null, receives scale * q.k of the chunk's valid rows at logits[tok * G + g]
// (stored with an L2 evict-last policy).
// TWO_TERM: P is fed to the PV product as bf16 hi + bf16 lo (about 16
// mantissa bits) for the fp32-output mode; otherwise P is rounded once to bf16.
template <int D, int NT, bool TWO_TERM>
__device__ __forceinline__ void dec_chunk(DecState<D, NT>& st, uint8_t* kb, int cnt, int lane,
                                          float scale, float scale_log2, int G, float* logits,
                                          uint64_t logit_policy) {
    using S = DecShape<D, NT>;
    constexpr int KSTEPS = D / 16;
    const int r = lane >> 2, cq = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;
    const int k_tok = (lj & 1) * 8 + lr, k_dof = (lj >> 1) * 8;   // K as A (token x d)
    const int v_tok = (lj >> 1) * 8 + lr, v_dof = (lj & 1) * 8;   // V^T as A (d x token)
    uint8_t* vb = kb + S::kChunkBytes;
    if (cnt < kPage) {
        // rows past the valid count may hold anything: zero them in V
        // (P is 0 there, but 0 * NaN would not be)
        const int per_row = S::kBoxes * 8;
        for (int idx = lane; idx < (kPage - cnt) * per_row; idx += 32) {
            const int row = cnt + idx / per_row, rem = idx % per_row;
            *reinterpret_cast<uint4*>(vb + (rem >> 3) * 2048 + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
    }
    // ---- S^T = K Q^T ----
    // two accumulators (even / odd k-steps) halve the dependent chain of
    // mma's; all K fragments are loaded up front
    float sacc[NT][4], sacc2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = sacc2[nt][e] = 0.f;
    const uint32_t kbase = smem_u32(kb);
    uint32_t kf[KSTEPS][4];
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const int d = kk * 16 + k_dof;
        ldsm_x4(kbase + (d >> 6) * 2048 + swz128(k_tok, (d & 63) >> 3), kf[kk][0], kf[kk][1],
                kf[kk][2], kf[kk][3]);
    }
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            mma_16816((kk & 1) ? sacc2[nt] : sacc[nt], kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3],
                      st.qf[kk][nt][0], st.qf[kk][nt][1]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] += sacc2[nt][e];
    // ---- mask, optional logits, online softmax (exp2 domain) ----
    float pr[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tok = r + ((e >> 1) << 3);
            sv[e] = tok < cnt ? sacc[nt][e] * scale_log2 : -INFINITY;
            if (logits != nullptr && tok < cnt) {
                const int g = nt * 8 + 2 * cq + (e & 1);
                if (g < G) st_global_hint(logits + (int64_t)tok * G + g, sacc[nt][e] * scale, logit_policy);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sv[j], sv[j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(st.m[nt][j], mx);
            const float base = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = ex2_approx(st.m[nt][j] - base);
            const float p0 = ex2_approx(sv[j] - base), p1 = ex2_approx(sv[j + 2] - base);
            st.l[nt][j] = st.l[nt][j] * alpha + p0 + p1;
            st.m[nt][j] = m_new;
            pr[nt][j] = p0;
            pr[nt][j + 2] = p1;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
                st.o[mt][nt][j] *= alpha;
                st.o[mt][nt][j + 2] *= alpha;
            }
        }
    }
    // ---- O^T += V^T P^T ----
    uint32_t pb[NT][2], pbl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint32_t x0 = pack_bf16(pr[nt][0], pr[nt][1]);
        const uint32_t x1 = pack_bf16(pr[nt][2], pr[nt][3]);
        pb[nt][0] = movmatrix_t(x0);
        pb[nt][1] = movmatrix_t(x1);
        if (TWO_TERM) {
            const uint32_t y0 = pack_bf16(pr[nt][0] - bf_lo(x0), pr[nt][1] - bf_hi(x0));
            const uint32_t y1 = pack_bf16(pr[nt][2] - bf_lo(x1), pr[nt][3] - bf_hi(x1));
            pbl[nt][0] = movmatrix_t(y0);
            pbl[nt][1] = movmatrix_t(y1);
        }
    }
    const uint32_t vbase = smem_u32(vb);
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
        const int d = mt * 16 + v_dof;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (d >> 6) * 2048 + swz128(v_tok, (d & 63) >> 3), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_16816(st.o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            if (TWO_TERM) mma_16816(st.o[mt][nt], a0, a1, a2, a3, pbl[nt][0], pbl[nt][1]);
        }
    }
}

// Where a finished piece goes: out (bf16 or fp32 [batch][Hq][D]) and lse_out
// (natural log, or null) when the piece is the whole unit, else the fp32
// partials o_part [slot][G][D] (normalised) and lse_part [slot][G] (log2) and the
// unit's arrival counter.
struct DecOut {
    void* out;
    int out_f32;
    float* lse_out;
    float* o_part;
    float* lse_part;
    int* counters;
    int Hq, G;
};

// End of a piece of unit u = (b, h) run by the four consumer warps (ctid =
// 0..127): merge the warps' states through `merge` (kMergeFloats floats of
// shared memory), then write the unit's output (slot < 0) or this piece's
// partials; the last of the unit's ui.y pieces (partial slots ui.x ..) to
// arrive merges them all.  `last` is one int of shared memory.
template <int D, int NT>
__device__ __forceinline__ void dec_finish(DecState<D, NT>& st, float* merge, volatile int* last,
                                           const DecOut& p, int b, int h, int u, int slot, int2 ui,
                                           int warp, int lane) {
    using S = DecShape<D, NT>;
    constexpr int KSTEPS = D / 16;
    const int r = lane >> 2, cq = lane & 3;
    const int ctid = warp * 32 + lane;
    const int G = p.G;
    float* mw = merge;                                      // [4][kHeads]
    float* lw = merge + kConsumerWarps * S::kHeads;         // [4][kHeads]
    float* ow = merge + 2 * kConsumerWarps * S::kHeads;     // [2][kHeads][D]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float x = st.l[nt][j];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            st.l[nt][j] = x;
        }
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mw[warp * S::kHeads + nt * 8 + 2 * cq + j] = st.m[nt][j];
                lw[warp * S::kHeads + nt * 8 + 2 * cq + j] = st.l[nt][j];
            }
    }
    consumer_bar();
    // per head: the four warps' weights exp2(m_w - M) / L and the LSE, once
    float* wf = mw + kConsumerWarps * S::kHeads * 2 + 2 * S::kHeads * D;
    if (ctid < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mw[w * S::kHeads + ctid]);
        float f[kConsumerWarps], L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            f[w] = M == -INFINITY ? 0.f : exp2f(mw[w * S::kHeads + ctid] - M);
            L += lw[w * S::kHeads + ctid] * f[w];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) wf[w * S::kHeads + ctid] = f[w] * inv;
        const float lse2 = L > 0.f ? M + log2f(L) : -INFINITY;
        wf[kConsumerWarps * S::kHeads + ctid] = lse2;
        const int64_t hq = (int64_t)b * p.Hq + h * G + ctid;
        if (slot < 0) {
            if (p.lse_out) p.lse_out[hq] = lse2 * kLn2;
        } else {
            p.lse_part[(int64_t)slot * G + ctid] = lse2;
        }
    }
    consumer_bar();
    // weighted O in two rounds through two slots: warps 2 and 3 store theirs,
    // warps 0 and 1 add theirs in place (half the merge area)
    {
        float f[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) f[nt][j] = wf[warp * S::kHeads + nt * 8 + 2 * cq + j];
        for (int round = 0; round < 2; ++round) {
            if ((warp >> 1) == 1 - round) {
                float* dst = ow + (warp & 1) * S::kHeads * D;
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int head = nt * 8 + 2 * cq + (e & 1);
                            const int d = mt * 16 + r + ((e >> 1) << 3);
                            const float v = st.o[mt][nt][e] * f[nt][e & 1];
                            float* at = dst + head * D + d;
                            *at = round == 0 ? v : *at + v;
                        }
            }
            consumer_bar();
        }
    }
    for (int idx = ctid; idx < G * D / 4; idx += kConsumerWarps * 32) {
        const int g = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const float4 x0 = *reinterpret_cast<const float4*>(ow + g * D + d);
        const float4 x1 = *reinterpret_cast<const float4*>(ow + (S::kHeads + g) * D + d);
        const float4 acc = make_float4(x0.x + x1.x, x0.y + x1.y, x0.z + x1.z, x0.w + x1.w);
        const int64_t hq = (int64_t)b * p.Hq + h * G + g;
        if (slot < 0) {
            if (p.out_f32) {
                *reinterpret_cast<float4*>(static_cast<float*>(p.out) + hq * D + d) = acc;
            } else {
                uint2 o2;
                o2.x = pack_bf16(acc.x, acc.y);
                o2.y = pack_bf16(acc.z, acc.w);
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + hq * D + d) = o2;
            }
        } else {
            *reinterpret_cast<float4*>(p.o_part + ((int64_t)slot * G + g) * D + d) = acc;
        }
    }
    consumer_bar();
    if (slot >= 0) {
        // The last piece of unit u to finish merges all of u's pieces by their
        // LSE (an arrival counter, no waiting on other CTAs).
        if (ctid == 0) {
            // the CTA barrier above orders the other threads' partial writes
            // before this thread's release; the acquire half orders the last
            // piece's reads of the other pieces after it (both cumulative)
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(p.counters + u)
                         : "memory");
            *last = old == ui.y - 1;
            if (old == ui.y - 1) atomicExch(&p.counters[u], 0);
        }
        consumer_bar();
        if (*last) {
            // each thread recomputes its head's piece weights from the LSEs (n
            // is small) while its partial rows are in flight
            const int n = min(ui.y, SE_MAX_SPLITS);
            for (int idx = ctid; idx < G * D / 4; idx += kConsumerWarps * 32) {
                const int g = idx / (D / 4), d = (idx % (D / 4)) * 4;
                const float* lsrc = p.lse_part + (int64_t)ui.x * G + g;
                const float4* src =
                    reinterpret_cast<const float4*>(p.o_part + ((int64_t)ui.x * G + g) * D + d);
                const int64_t step = (int64_t)G * D / 4;
                // one pass with a running maximum: each piece's LSE and rows
                // are loaded together (four pieces in flight)
                float M = -INFINITY, L = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int i = 0; i < n; ++i) {
                    const float x2 = __ldcg(lsrc + (int64_t)i * G);
                    const float4 x = __ldcg(src + i * step);
                    if (x2 == -INFINITY) continue;            // an empty piece
                    const float mn = fmaxf(M, x2);
                    const float a = exp2f(M - mn), f = exp2f(x2 - mn);
                    L = L * a + f;
                    acc.x = acc.x * a + f * x.x;
                    acc.y = acc.y * a + f * x.y;
                    acc.z = acc.z * a + f * x.z;
                    acc.w = acc.w * a + f * x.w;
                    M = mn;
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const int64_t hq = (int64_t)b * p.Hq + h * G + g;
                if (p.out_f32) {
                    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + hq * D + d) =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                } else {
                    uint2 o2;
                    o2.x = pack_bf16(acc.x * inv, acc.y * inv);
                    o2.y = pack_bf16(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + hq * D + d) = o2;
                }
                if (d == 0 && p.lse_out)
                    p.lse_out[hq] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
            }
        }
        consumer_bar();
    }
}

}  // namespace se
