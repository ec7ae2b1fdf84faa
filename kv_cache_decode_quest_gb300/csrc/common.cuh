// Device helpers shared by the kernels of libsparse_engine: bf16 packing,
// order-preserving float keys, block scans, and thin inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor), ldmatrix, mma.sync and movmatrix.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_engine.h"

namespace se {

constexpr int kPage = 16;
// A wait on an mbarrier that has not completed after this long means
// something is wrong; the kernel records SE_DEV_TIMEOUT and drains.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;   // 1 s

__device__ __forceinline__ void flag(int* status, int bits) {
    if (status) atomicOr(status, bits);
}

// ---- bf16 ---------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Order-preserving key: larger float -> larger unsigned key; -0 == +0.
__device__ __forceinline__ uint32_t float_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---- block-wide exclusive scan of one int per thread ----------------------
// `tmp` needs 33 ints of shared memory (blockDim.x <= 1024).  Returns the exclusive
// prefix; *total receives the block sum.  All threads must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nwarps) tmp[lane] = w;          // inclusive warp totals
        if (lane == nwarps - 1) tmp[32] = w;
    }
    __syncthreads();
    int before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
    int t = tmp[32];
    __syncthreads();
    *total = t;
    return before;
}

// ---- shared-memory addresses, timers --------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: true when the phase of `parity` completed; false when the
// CTA-wide abort flag is raised or the time limit passed (the caller then
// raises the abort flag and records SE_DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// ---- TMA ----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- cp.async (16-byte asynchronous global -> shared copies) ---------------------
// src_bytes < 16 zero-fills the rest (0 reads nothing: a zero vector).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- warp-level matrix ops -----------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Byte offset of 16-byte unit `u` of row `r` inside a TMA box written with
// CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, buffer 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(int r, int u) {
    return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

// Inclusive scan over the first 256 threads of the block (all threads call it);
// `tmp` holds 8 ints of shared memory.
__device__ __forceinline__ int scan256(int v, int* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (threadIdx.x < 256 && lane == 31) tmp[warp] = x;
    __syncthreads();
    int before = 0;
    if (threadIdx.x < 256)
        for (int i = 0; i < warp; ++i) before += tmp[i];
    __syncthreads();
    return x + before;
}

// Exact selection threshold for the K largest of m unsigned keys (1 <= K <= m),
// block-wide (blockDim.x >= 256): four 8-bit MSB-first radix passes.  Returns
// the K-th largest key T; *need_eq receives how many keys equal to T belong to
// the top K (every key > T does).  key_at(i) must be callable by any thread.
// Shared memory: hist[256], tmp[33], sel[2].
template <typename KeyAt>
__device__ uint32_t block_radix_select(KeyAt key_at, int m, int K, int* hist, int* tmp, int* sel,
                                       int* need_eq) {
    uint32_t prefix = 0, mask = 0;
    int remaining = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (threadIdx.x < 256) hist[threadIdx.x] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < m; i += blockDim.x) {
            const uint32_t key = key_at(i);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        const int v = threadIdx.x < 256 ? hist[255 - threadIdx.x] : 0;
        const int incl = scan256(v, tmp);
        if (threadIdx.x < 256) {
            const int excl = incl - v;
            if (excl < remaining && incl >= remaining) {
                sel[0] = 255 - threadIdx.x;
                sel[1] = excl;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sel[0]) << shift;
        mask |= 255u << shift;
        remaining -= sel[1];
        __syncthreads();
    }
    *need_eq = remaining;
    return prefix;
}

}  // namespace se
