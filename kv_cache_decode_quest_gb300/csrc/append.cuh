// One KV head's share of a decode-step append into the paged cache: the new
// key/value row at position `pos` of sequence b (physical page `phys`, slot
// pos % 16) and, when the cache keeps page summaries (meta not null), the key
// folded into that page's channel-wise min/max summary, the page's first
// token setting both (Quest's page summary kept beside the
// full history: tokendh.com article on SparseEngine, section
// "历史太长,会撑爆什么").  Threads t = 0..nt-1 share the head_dim/8 vectors.
#pragma once

#include "common.cuh"

namespace se {

struct Bf8 {
    float x[8];
};
__device__ __forceinline__ Bf8 unpack8(uint4 w) {
    Bf8 r;
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.x[2 * i] = bf_lo(a[i]);
        r.x[2 * i + 1] = bf_hi(a[i]);
    }
    return r;
}
__device__ __forceinline__ uint4 pack8(const Bf8& v) {
    // Values are bf16-representable (min/max of bf16 inputs): rounding is exact.
    return make_uint4(pack_bf16(v.x[0], v.x[1]), pack_bf16(v.x[2], v.x[3]),
                      pack_bf16(v.x[4], v.x[5]), pack_bf16(v.x[6], v.x[7]));
}

// The same append split in two for one 16-byte vector sg of head h: the loads
// (new key/value, the page's current min/max; none of them needs the physical
// page) can be issued early and the stores done later.
struct AppendRegs {
    uint4 k, v, mn, mx;
};
__device__ __forceinline__ void append_load(const se_paged_kv& kv, int b, int h, int pos,
                                            const uint4* k_new, const uint4* v_new, int sg,
                                            AppendRegs& r) {
    const int H = kv.num_kv_heads, segs = kv.head_dim / 8;
    const int p = pos / kPage, slot = pos % kPage;
    const uint4* M = static_cast<const uint4*>(kv.meta);
    const int64_t m0 = (((int64_t)b * kv.max_pages_per_seq + p) * H + h) * 2;
    r.k = k_new[((int64_t)b * H + h) * segs + sg];
    r.v = v_new[((int64_t)b * H + h) * segs + sg];
    if (slot != 0 && M != nullptr) {
        r.mn = M[m0 * segs + sg];
        r.mx = M[(m0 + 1) * segs + sg];
    }
}
__device__ __forceinline__ void append_store(const se_paged_kv& kv, int b, int h, int pos,
                                             int phys, int sg, const AppendRegs& r) {
    const int H = kv.num_kv_heads, segs = kv.head_dim / 8;
    const int p = pos / kPage, slot = pos % kPage;
    uint4* K = static_cast<uint4*>(kv.k);
    uint4* V = static_cast<uint4*>(kv.v);
    uint4* M = static_cast<uint4*>(kv.meta);
    const int64_t row = ((int64_t)phys * H + h) * kPage + slot;
    const int64_t m0 = (((int64_t)b * kv.max_pages_per_seq + p) * H + h) * 2;
    K[row * segs + sg] = r.k;
    V[row * segs + sg] = r.v;
    if (M == nullptr) return;                 // a cache kept without page summaries
    if (slot == 0) {
        M[m0 * segs + sg] = r.k;
        M[(m0 + 1) * segs + sg] = r.k;
    } else {
        Bf8 mn = unpack8(r.mn), mx = unpack8(r.mx);
        const Bf8 x = unpack8(r.k);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mn.x[i] = fminf(mn.x[i], x.x[i]);
            mx.x[i] = fmaxf(mx.x[i], x.x[i]);
        }
        M[m0 * segs + sg] = pack8(mn);
        M[(m0 + 1) * segs + sg] = pack8(mx);
    }
}

__device__ __forceinline__ void append_head(const se_paged_kv& kv, int b, int h, int pos, int phys,
                                            const uint4* k_new, const uint4* v_new, int t,
                                            int nt) {
    for (int sg = t; sg < kv.head_dim / 8; sg += nt) {
        AppendRegs r;
        append_load(kv, b, h, pos, k_new, v_new, sg, r);
        append_store(kv, b, h, pos, phys, sg, r);
    }
}

}  // namespace se
