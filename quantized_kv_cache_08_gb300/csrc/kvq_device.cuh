// Device helpers shared by the decode kernels: inline PTX for mbarriers, bulk
// copies and shared-memory loads, and the mapping of work items to rows.
#pragma once

#include "kvq_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace kvq {
namespace dev {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLazy = 8.0f;            // log2 units a score may exceed the reference max
constexpr int kWaitIters = 1 << 22;      // bounded mbarrier wait

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// L2 policy for bytes read once per decode (the K and V rows): they are the
// first to go when L2 needs room, so the stream does not push out what every
// launch reads again (code, lengths, queries, partial records)
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(evict_first_policy())
        : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread until the phase completes or about
// `ns` nanoseconds pass, instead of returning at once
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// bounded wait; false when it ran out
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kWaitIters; ++i)
        if (mbar_try(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ float load_q(const void* q, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
    return reinterpret_cast<const float*>(q)[idx];
}

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// ---------------------------------------------------------- work mapping

struct Item {
    int b, split, qs, pidx;
};

// visible-row window of sequence b for a T-row step: rows [lo, len)
__device__ __forceinline__ void visible_rows(const SplitParams& p, int len, int& lo) {
    lo = 0;
    if (p.window > 0) lo = max(0, len - p.T + 1 - p.window);
}

__device__ __forceinline__ Item item_of(int idx, const int* prefix, int B, int nqs) {
    Item it;
    const int pi = idx / nqs;
    it.qs = idx - pi * nqs;
    int lo = 0, hi = B;  // largest b with prefix[b] <= pi
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= pi) lo = mid;
        else hi = mid;
    }
    it.b = lo;
    it.split = pi - prefix[lo];
    it.pidx = pi;
    return it;
}

// rows of the item: [row0, row0 + n), tiles of kTileRows
struct ItemRows {
    int row0, n, base, len;
};

__device__ __forceinline__ ItemRows item_rows(const SplitParams& p, const int* lens, const int* bases,
                                              const Item& it) {
    ItemRows r;
    r.len = lens[it.b];
    r.base = bases[it.b];
    int lo;
    visible_rows(p, r.len, lo);
    r.row0 = lo + it.split * p.C;
    r.n = min(p.C, r.len - r.row0);
    return r;
}


// Per-sequence split counts from the device lengths, exclusive prefix into
// prefix[0..B] (warp 0 of the CTA; the caller synchronises afterwards).
// A sequence whose counters are out of range gets no split and sets the
// error word.
__device__ __forceinline__ void plan_splits(const SplitParams& p, const int* lens, const int* bases, int* prefix,
                                            int lane) {
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int ns = 0;
        if (b < p.B) {
            const int len = lens[b];
            int lo;
            visible_rows(p, len, lo);
            const bool bad = len < p.T || len - bases[b] > p.max_rows || lo < bases[b];
            if (bad) {
                if (blockIdx.x == 0) atomicExch(p.err_d, kErrCounter);
            } else {
                ns = (len - lo + p.C - 1) / p.C;
            }
        }
        int x = ns;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (b < p.B) prefix[b] = carry + x - ns;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) prefix[p.B] = carry;
}

}  // namespace dev
}  // namespace kvq
