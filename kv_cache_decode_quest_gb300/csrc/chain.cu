// Chain Cache: the retained state of evicting methods carried across turns.
//
// A method that deletes history physically (SnapKV, H2O) keeps, per sequence
// and KV head, a segment of retained rows with their logical positions (and,
// for H2O, accumulated scores).  Chain Cache keeps that state and the logical
// token prefix it stands for, so that a later request that continues the
// same logical prefix resumes from the retained state instead of rebuilding
// it (tokendh.com article on SparseEngine, section "聊天记录也能'续命':Chain
// Cache"; "SparseEngine 统一接入十五种稀疏注意力", section "部署长上下文 Agent
// 的团队可以从中得到什么": the ChainCacheIndex links a session to its retained
// per-layer KV, its method metadata and its logical token prefix).
//
// Device side (this file's kernels): se_chain_save copies the segments of
// chosen sequences into a snapshot buffer, one fixed slot per (sequence, KV
// head); se_chain_restore copies a snapshot's slots into the segments of
// chosen sequences of any varlen cache (any segment offsets), with their
// lengths.  Both are pure copies: one CTA per (slot, block of rows), 16-byte
// vectors.  Host side: a prefix index from logical token sequences to
// snapshot ids (longest stored prefix wins, exact token comparison).
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace se {
namespace {

constexpr int kChainRows = 64;             // rows per CTA
constexpr uint32_t kSnapMagic = 0x43484e31u;   // snapshot format tag

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Snapshot layout: a 256-byte header (format tag, slots, heads, head_dim,
// rows per slot, score flag), per slot (seg_len, seq_len) pairs, then per slot
// `rows` rows of K, of V (bf16 [D]), of logical positions and of scores.
struct SnapLayout {
    size_t lens, k, v, pos, score, total;
};
SnapLayout snap_layout(int n_slots, int D, int rows, bool with_score) {
    SnapLayout L;
    const size_t r = (size_t)n_slots * rows;
    size_t off = 256;
    L.lens = off;
    off += a256((size_t)n_slots * 2 * sizeof(int32_t));
    L.k = off;
    off += a256(r * D * 2);
    L.v = off;
    off += a256(r * D * 2);
    L.pos = off;
    off += a256(r * sizeof(int32_t));
    L.score = off;
    off += with_score ? a256(r * sizeof(float)) : 0;
    L.total = off;
    return L;
}

struct ChainParams {
    se_varlen_kv kv;
    const int32_t* seqs;          // [n] sequences of kv (save: sources, restore: targets)
    int n, rows;
    uint8_t* snap;
    SnapLayout lay;
    int* status;
};

// grid (row blocks, n * H): slot i = (seqs[i / H]'s head i % H).
__global__ void __launch_bounds__(128) chain_save_kernel(const ChainParams p) {
    const int H = p.kv.num_kv_heads, D = p.kv.head_dim, segs = D / 8;
    const int slot = blockIdx.y, i = slot / H, h = slot % H;
    const int b = p.seqs[i];
    int32_t* lens = reinterpret_cast<int32_t*>(p.snap + p.lay.lens);
    if (b < 0) {                                       // no such sequence: an empty slot
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            flag(p.status, SE_DEV_BAD_INDEX);
            lens[2 * slot] = 0;
            lens[2 * slot + 1] = 0;
        }
        return;
    }
    const int u = b * H + h;
    int len = p.kv.seg_len[u];
    const int off = p.kv.seg_off[u];
    if (len < 0 || len > p.kv.seg_cap || off < 0 || (int64_t)off + len > p.kv.total_rows) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, SE_DEV_BAD_LENGTH);
        len = 0;
    }
    if (len > p.rows) {                                // the slot holds fewer rows
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, SE_DEV_CAPACITY);
        len = p.rows;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        lens[2 * slot] = len;
        lens[2 * slot + 1] = p.kv.seq_len[b];
        if (slot == 0) {
            uint32_t* hdr = reinterpret_cast<uint32_t*>(p.snap);
            hdr[0] = kSnapMagic;
            hdr[1] = gridDim.y;
            hdr[2] = H;
            hdr[3] = D;
            hdr[4] = p.rows;
            hdr[5] = p.kv.score != nullptr;
        }
    }
    const int r0 = blockIdx.x * kChainRows, r1 = min(len, r0 + kChainRows);
    const int64_t dst0 = (int64_t)slot * p.rows;
    const uint4* Ks = static_cast<const uint4*>(p.kv.k);
    const uint4* Vs = static_cast<const uint4*>(p.kv.v);
    uint4* Kd = reinterpret_cast<uint4*>(p.snap + p.lay.k);
    uint4* Vd = reinterpret_cast<uint4*>(p.snap + p.lay.v);
    for (int x = threadIdx.x; x < (r1 - r0) * segs; x += blockDim.x) {
        const int r = r0 + x / segs, sg = x % segs;
        Kd[(dst0 + r) * segs + sg] = Ks[((int64_t)off + r) * segs + sg];
        Vd[(dst0 + r) * segs + sg] = Vs[((int64_t)off + r) * segs + sg];
    }
    int32_t* pos = reinterpret_cast<int32_t*>(p.snap + p.lay.pos);
    float* score = reinterpret_cast<float*>(p.snap + p.lay.score);
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        pos[dst0 + r] = p.kv.pos[off + r];
        if (p.kv.score) score[dst0 + r] = p.kv.score[off + r];
    }
}

// grid (row blocks, n * H): slot i goes to (seqs[i / H], head i % H).
__global__ void __launch_bounds__(128) chain_restore_kernel(const ChainParams p) {
    const int H = p.kv.num_kv_heads, D = p.kv.head_dim, segs = D / 8;
    const int slot = blockIdx.y, i = slot / H, h = slot % H;
    const uint32_t* hdr = reinterpret_cast<const uint32_t*>(p.snap);
    // the snapshot must have been written for this shape
    const bool fmt_ok = hdr[0] == kSnapMagic && hdr[1] == gridDim.y && hdr[2] == (uint32_t)H &&
                        hdr[3] == (uint32_t)D && hdr[4] == (uint32_t)p.rows &&
                        hdr[5] == (uint32_t)(p.kv.score != nullptr);
    const int b = p.seqs[i];
    if (!fmt_ok || b < 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, SE_DEV_BAD_INDEX);
        return;
    }
    const int u = b * H + h;
    const int32_t* lens = reinterpret_cast<const int32_t*>(p.snap + p.lay.lens);
    int len = lens[2 * slot];
    const int off = p.kv.seg_off[u];
    if (len < 0 || len > p.rows || off < 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, SE_DEV_BAD_LENGTH);
        len = 0;
    }
    if (len > p.kv.seg_cap || (int64_t)off + len > p.kv.total_rows) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, SE_DEV_CAPACITY);
        len = max(0, min(p.kv.seg_cap, p.kv.total_rows - off));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.kv.seg_len[u] = len;
        if (h == 0) p.kv.seq_len[b] = lens[2 * slot + 1];
    }
    const int r0 = blockIdx.x * kChainRows, r1 = min(len, r0 + kChainRows);
    const int64_t src0 = (int64_t)slot * p.rows;
    const uint4* Ks = reinterpret_cast<const uint4*>(p.snap + p.lay.k);
    const uint4* Vs = reinterpret_cast<const uint4*>(p.snap + p.lay.v);
    uint4* Kd = static_cast<uint4*>(p.kv.k);
    uint4* Vd = static_cast<uint4*>(p.kv.v);
    for (int x = threadIdx.x; x < (r1 - r0) * segs; x += blockDim.x) {
        const int r = r0 + x / segs, sg = x % segs;
        Kd[((int64_t)off + r) * segs + sg] = Ks[(src0 + r) * segs + sg];
        Vd[((int64_t)off + r) * segs + sg] = Vs[(src0 + r) * segs + sg];
    }
    const int32_t* pos = reinterpret_cast<const int32_t*>(p.snap + p.lay.pos);
    const float* score = reinterpret_cast<const float*>(p.snap + p.lay.score);
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        p.kv.pos[off + r] = pos[src0 + r];
        if (p.kv.score) p.kv.score[off + r] = score[src0 + r];
    }
}

}  // namespace

size_t chain_snapshot_bytes(int num_seqs, int H, int D, int rows, bool with_score) {
    return snap_layout(num_seqs * H, D, rows, with_score).total;
}

cudaError_t launch_chain_copy(bool save, const se_varlen_kv& kv, const int32_t* seqs, int n,
                              int rows, void* snap, int* status, cudaStream_t s) {
    const int H = kv.num_kv_heads;
    if (n == 0 || rows == 0) return cudaSuccess;
    ChainParams p;
    p.kv = kv;
    p.seqs = seqs;
    p.n = n;
    p.rows = rows;
    p.snap = static_cast<uint8_t*>(snap);
    p.lay = snap_layout(n * H, kv.head_dim, rows, kv.score != nullptr);
    p.status = status;
    dim3 grid((rows + kChainRows - 1) / kChainRows, n * H);
    if (save)
        chain_save_kernel<<<grid, 128, 0, s>>>(p);
    else
        chain_restore_kernel<<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace se

// ---- the host prefix index -----------------------------------------------------

struct se_chain_index {
    std::mutex mu;
    // id -> the logical token prefix it stands for
    std::unordered_map<int64_t, std::vector<int32_t>> tokens;
    // (prefix length, prefix hash) -> ids
    std::map<std::pair<int64_t, uint64_t>, std::vector<int64_t>> by_key;
    std::multiset<int64_t> lengths;
};

namespace {

// Polynomial hash of every prefix of `t` (h[i] = hash of t[0..i)), modulo 2^64.
std::vector<uint64_t> prefix_hashes(const int32_t* t, int64_t n) {
    std::vector<uint64_t> h(static_cast<size_t>(n) + 1);
    const uint64_t base = 0x9E3779B97F4A7C15ull;
    h[0] = 0x2545F4914F6CDD1Dull;
    for (int64_t i = 0; i < n; ++i)
        h[i + 1] = h[i] * base + static_cast<uint32_t>(t[i]) + 0x632BE59BD9B4E019ull;
    return h;
}

void erase_locked(se_chain_index* ix, int64_t id) {
    auto it = ix->tokens.find(id);
    if (it == ix->tokens.end()) return;
    const auto& t = it->second;
    const int64_t n = static_cast<int64_t>(t.size());
    const auto key = std::make_pair(n, prefix_hashes(t.data(), n)[n]);
    auto& ids = ix->by_key[key];
    ids.erase(std::remove(ids.begin(), ids.end(), id), ids.end());
    if (ids.empty()) ix->by_key.erase(key);
    ix->lengths.erase(ix->lengths.find(n));
    ix->tokens.erase(it);
}

}  // namespace

extern "C" {

size_t se_chain_snapshot_bytes(int num_seqs, int num_kv_heads, int head_dim, int rows,
                               int with_score) {
    if (num_seqs < 0 || num_kv_heads <= 0 || (head_dim != 64 && head_dim != 128) || rows < 0)
        return 0;
    return se::chain_snapshot_bytes(num_seqs, num_kv_heads, head_dim, rows, with_score != 0);
}

se_chain_index* se_chain_index_create(void) { return new (std::nothrow) se_chain_index(); }

void se_chain_index_destroy(se_chain_index* ix) { delete ix; }

int se_chain_index_put(se_chain_index* ix, const int32_t* tokens, int64_t n_tokens, int64_t id) {
    if (!ix || n_tokens < 0 || (n_tokens > 0 && !tokens) || id < 0) return SE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(ix->mu);
    erase_locked(ix, id);
    std::vector<int32_t> t(tokens, tokens + n_tokens);
    const uint64_t h = prefix_hashes(t.data(), n_tokens)[n_tokens];
    ix->by_key[std::make_pair(n_tokens, h)].push_back(id);
    ix->lengths.insert(n_tokens);
    ix->tokens.emplace(id, std::move(t));
    return SE_OK;
}

int64_t se_chain_index_match(se_chain_index* ix, const int32_t* tokens, int64_t n_tokens,
                             int64_t* matched_tokens) {
    if (matched_tokens) *matched_tokens = 0;
    if (!ix || n_tokens < 0 || (n_tokens > 0 && !tokens)) return SE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(ix->mu);
    const std::vector<uint64_t> h = prefix_hashes(tokens, n_tokens);
    // the longest stored prefix first; a hash match is confirmed token by token
    for (auto it = ix->lengths.rbegin(); it != ix->lengths.rend(); ++it) {
        const int64_t n = *it;
        if (n > n_tokens) continue;
        auto f = ix->by_key.find(std::make_pair(n, h[n]));
        if (f == ix->by_key.end()) continue;
        for (int64_t id : f->second) {
            const auto& t = ix->tokens[id];
            if (n == 0 || std::memcmp(t.data(), tokens, n * sizeof(int32_t)) == 0) {
                if (matched_tokens) *matched_tokens = n;
                return id;
            }
        }
    }
    return -1;
}

int se_chain_index_erase(se_chain_index* ix, int64_t id) {
    if (!ix) return SE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(ix->mu);
    erase_locked(ix, id);
    return SE_OK;
}

int64_t se_chain_index_size(se_chain_index* ix) {
    if (!ix) return SE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(ix->mu);
    return static_cast<int64_t>(ix->tokens.size());
}

}  // extern "C"
