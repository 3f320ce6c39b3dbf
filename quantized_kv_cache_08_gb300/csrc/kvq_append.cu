// Quantised append (q8_0 K, q5_1 V, or FP8 E4M3 K and V) and the small
// counter kernels.
//
// Formats and row placement: memra-engine "Struct KvLayer" (type
// description): a token row keeps the [token, kv_head, dim] element order, so
// element e = kv_head*head_dim + d of the row lands in 32-element block e/32
// at lane e%32; K blocks are q8_0 (34 B), V blocks q5_1 (24 B).  The append
// writes at the device slot len_d (the length before this append) and then
// adds T, in the same launch (fields len_d / base_d, the
// append_kv_quantized_dc and inc_seqlen steps); the physical row is
// slot + t - base_d.
//
// Rounding.  The fp16 scale of a block is the fp64 quotient rounded to fp16
// with round-to-nearest-even (one fp64 division per block).  A code is
// round-half-away-from-zero of x/d (q8_0) or (x-m)/d (q5_1) taken against the
// stored fp16 d and m.  The kernel estimates the quotient in fp32, whose error
// is below 2e-5 of a code step; only when the estimate lies within 1e-3 of a
// rounding boundary does it recompute the quotient in fp64 exactly as the
// definition reads, so every code equals the fp64 decision.
//
// FP8 E4M3 (memra-engine "Module cache", items gkv_on and kv_fp8_on:
// K/V held in e4m3): each element becomes one byte on its own, with no scale,
// by the hardware conversion that rounds to nearest even and saturates to
// +-448 (cvt.rn.satfinite); byte e of a token row is element e.
#include "kvq_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

namespace kvq {
namespace {

__device__ __forceinline__ float load_elem(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_min(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// round-half-away-from-zero of an fp64 value, exact
__device__ __forceinline__ double rha64(double t) {
    double a = fabs(t);
    double f = floor(a);
    double n = f + ((a - f) >= 0.5 ? 1.0 : 0.0);
    return t < 0.0 ? -n : n;
}

__device__ __forceinline__ bool near_boundary(float a) {
    // a = |t| + 0.5 (or t + 0.5): a code boundary is an integer value of a
    float fr = a - floorf(a);
    return fr < 1e-3f || fr > 0.999f || fabsf(a) >= 4194304.0f;
}

// q8_0 code of x for stored scale d (d > 0), inv = 1/d
__device__ __forceinline__ int q8_code(float x, float d, float inv) {
    float t = x * inv;
    float a = fabsf(t) + 0.5f;
    if (near_boundary(a)) {
        double n = rha64((double)x / (double)d);
        n = fmin(fmax(n, -127.0), 127.0);
        return (int)n;
    }
    int n = min((int)floorf(a), 127);
    return t < 0.f ? -n : n;
}

// q5_1 code of x for stored min m and scale d (d > 0), inv = 1/d
__device__ __forceinline__ int q5_code(float x, float m, float d, float inv) {
    float t = (x - m) * inv;
    float a = t + 0.5f;
    if (near_boundary(a)) {
        double n = rha64(((double)x - (double)m) / (double)d);
        n = fmin(fmax(n, 0.0), 31.0);
        return (int)n;
    }
    float f = floorf(a);
    f = fminf(fmaxf(f, 0.f), 31.f);
    return (int)f;
}

// One warp per (entry, row t, block j); lane = element of the block.
__device__ __forceinline__ void append_block(const AppendParams& p, const SeqIds& ids, long long w, int lane) {
    const int j = (int)(w % p.kb);
    const long long rest = w / p.kb;
    const int t = (int)(rest % p.T);
    const int i = (int)(rest / p.T);
    const int b = ids.identity ? ids.first + i : ids.id[i];
    const int slot = p.len_d[b];                 // this launch's own commit changes len_d later
    const int base = p.base_d[b];
    const int phys = slot + t - base;
    if (phys < 0 || phys >= p.max_rows) {
        if (lane == 0) atomicExch(p.err_d, kErrCounter);
        return;
    }
    const long long kvd = (long long)p.kb * kQK;
    const long long src = ((p.entry_offset + i) * p.T + t) * kvd + (long long)j * kQK + lane;
    const float xk = load_elem(p.k, src, p.bf16);
    const float xv = load_elem(p.v, src, p.bf16);
    const long long row = (long long)b * p.max_rows + phys;

    if (p.fp8) {
        const long long e = (long long)j * kQK + lane;
        p.k_plane[row * p.k_tok + e] = __nv_cvt_float_to_fp8(xk, __NV_SATFINITE, __NV_E4M3);
        p.v_plane[row * p.v_tok + e] = __nv_cvt_float_to_fp8(xv, __NV_SATFINITE, __NV_E4M3);
        return;
    }

    // ---- K: q8_0 ----
    {
        const float amax = warp_max(fabsf(xk));
        unsigned short dbits = 0;
        if (lane == 0) dbits = __half_as_ushort(__double2half((double)amax / 127.0));
        dbits = (unsigned short)__shfl_sync(0xffffffffu, (int)dbits, 0);
        const float d = __half2float(__ushort_as_half(dbits));
        int c = 0;
        if (d > 0.f) c = q8_code(xk, d, 1.0f / d);
        uint8_t* blk = p.k_plane + row * p.k_tok + (long long)j * kQ8Bytes;
        blk[2 + lane] = (uint8_t)(int8_t)c;
        if (lane == 0) *reinterpret_cast<unsigned short*>(blk) = dbits;
    }
    // ---- V: q5_1 ----
    {
        const float mn = warp_min(xv);
        const float mx = warp_max(xv);
        unsigned int dm = 0;
        if (lane == 0) {
            unsigned short db = __half_as_ushort(__double2half(((double)mx - (double)mn) / 31.0));
            unsigned short mb = __half_as_ushort(__float2half_rn(mn));
            dm = (unsigned int)db | ((unsigned int)mb << 16);
        }
        dm = __shfl_sync(0xffffffffu, dm, 0);
        const float d = __half2float(__ushort_as_half((unsigned short)(dm & 0xffffu)));
        const float m = __half2float(__ushort_as_half((unsigned short)(dm >> 16)));
        int u = 0;
        if (d > 0.f) u = q5_code(xv, m, d, 1.0f / d);
        const unsigned int qh = __ballot_sync(0xffffffffu, (u >> 4) & 1);
        const int hi = __shfl_down_sync(0xffffffffu, u, 16);
        uint8_t* blk = p.v_plane + row * p.v_tok + (long long)j * kQ5Bytes;
        if (lane < 16) blk[8 + lane] = (uint8_t)((u & 15) | ((hi & 15) << 4));
        if (lane == 0) *reinterpret_cast<unsigned int*>(blk) = dm;
        if (lane == 1) *reinterpret_cast<unsigned int*>(blk + 4) = qh;
    }
}

// The append of one launch, then its commit (len_d += T for the launch's
// sequences, the inc_seqlen step): every CTA counts itself done on the
// completion counter once its warps have read len_d, and the last one, which
// resets the counter for the next launch, commits.
__global__ void __launch_bounds__(256) append_kernel(AppendParams p, SeqIds ids, long long n_work) {
    // a decode launched next may start now: it waits for this grid (and its
    // writes) before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (w < n_work) append_block(p, ids, w, lane);
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(p.done_d, 1) == (int)gridDim.x - 1;
        if (s_last) {
            *p.done_d = 0;
            __threadfence();
        }
    }
    __syncthreads();
    if (s_last) {
        for (int i = threadIdx.x; i < ids.n; i += blockDim.x) {
            const int b = ids.identity ? ids.first + i : ids.id[i];
            p.len_d[b] += p.T;
        }
    }
}

__global__ void set_len_kernel(int* len_d, SeqIds ids, SeqIds vals) {
    for (int i = threadIdx.x; i < ids.n; i += blockDim.x) {
        const int b = ids.identity ? ids.first + i : ids.id[i];
        len_d[b] = vals.id[i];
    }
}

__global__ void set_base_kernel(int* base_d, int seq, int value) { base_d[seq] = value; }

// Rollback with the accepted count on the device ("Struct Cache", fn rollback,
// item C.1: len = snapshot_len + accept_len, where snapshot_len = len - T for
// a T-row draft step): of the last T rows the first accept_d[b] stay.  A
// sequence whose accept count is outside [0, T], that holds fewer than T rows,
// or (ring) whose new window start would fall below its base keeps its length
// and sets the error word.
__global__ void truncate_accept_kernel(int* len_d, const int* base_d, int* err_d, const int* accept_d, int n,
                                       int T, int window, int ring) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n) return;
    const int a = accept_d[b];
    const int len = len_d[b];
    const int nl = len - T + a;
    bool ok = a >= 0 && a <= T && T <= len;
    if (ok && ring) ok = max(0, nl + 1 - window) >= base_d[b];
    if (ok)
        len_d[b] = nl;
    else
        atomicExch(err_d, kErrCounter);
}

// Byte copy of two non-overlapping ranges (ring rebase legs, unaligned rows).
__global__ void __launch_bounds__(256) ring_copy_bytes_kernel(const uint8_t* __restrict__ sk,
                                                             const uint8_t* __restrict__ sv,
                                                             uint8_t* __restrict__ dk, uint8_t* __restrict__ dv,
                                                             size_t nk, size_t nv) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nk + nv; i += stride) {
        if (i < nk) dk[i] = sk[i];
        else dv[i - nk] = sv[i - nk];
    }
}

// 16-byte copy of two non-overlapping ranges (ring rebase legs).
__global__ void __launch_bounds__(256) ring_copy_kernel(const uint4* __restrict__ sk, const uint4* __restrict__ sv,
                                 uint4* __restrict__ dk, uint4* __restrict__ dv, size_t nk, size_t nv) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nk + nv; i += stride) {
        if (i < nk) dk[i] = sk[i];
        else dv[i - nk] = sv[i - nk];
    }
}

// Ring rebase in one pass: logical rows [new_base, len) of a sequence move
// to physical row 0 ("Struct KvLayer", field base_d: physical = row - base;
// "Module cache", fn swa_ring_rows).  The destination overlaps the source, so
// every CTA first reads its share of the live bytes of both planes into shared
// memory, all CTAs meet at a grid barrier (the launch is cooperative, so they
// are all resident), then write; CTA 0 then sets base_d.  A barrier that does
// not complete within ~1 s sets the error word and nothing is written.
__global__ void __launch_bounds__(256) rebase_kernel(const uint4* sk, uint4* dk, size_t nk16, const uint4* sv,
                                                     uint4* dv, size_t nv16, int* base_d, int seq, int new_base,
                                                     int* arrive, int* gen, int* err_d) {
    extern __shared__ uint4 buf[];
    const size_t total = nk16 + nv16;
    const size_t per = (total + gridDim.x - 1) / gridDim.x;
    const size_t lo = (size_t)blockIdx.x * per;
    const size_t hi = lo + per < total ? lo + per : total;
    for (size_t i = lo + threadIdx.x; i < hi; i += blockDim.x) buf[i - lo] = i < nk16 ? sk[i] : sv[i - nk16];
    __syncthreads();
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        // sense-reversing grid barrier: the last arrival opens the next generation
        const int g0 = *(volatile int*)gen;
        __threadfence();
        if (atomicAdd(arrive, 1) == (int)gridDim.x - 1) {
            *arrive = 0;
            __threadfence();
            atomicAdd(gen, 1);
            s_ok = 1;
        } else {
            const long long t0 = clock64();
            s_ok = 1;
            while (*(volatile int*)gen == g0) {
                if (clock64() - t0 > (1LL << 31)) {
                    atomicExch(err_d, kErrWait);
                    s_ok = 0;
                    break;
                }
                __nanosleep(200);
            }
        }
        __threadfence();
    }
    __syncthreads();
    if (!s_ok) return;
    for (size_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        if (i < nk16) dk[i] = buf[i - lo];
        else dv[i - nk16] = buf[i - lo];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) base_d[seq] = new_base;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, const SeqIds& ids, cudaStream_t s) {
    const long long n_work = (long long)ids.n * p.T * p.kb;
    if (n_work == 0) return cudaSuccess;
    const long long grid = (n_work + 7) / 8;
    append_kernel<<<(unsigned)grid, 256, 0, s>>>(p, ids, n_work);
    return cudaGetLastError();
}

cudaError_t launch_set_len(int* len_d, const SeqIds& ids, const int* values, cudaStream_t s) {
    SeqIds vals;
    vals.n = ids.n;
    vals.identity = 0;
    vals.first = 0;
    for (int i = 0; i < ids.n; ++i) vals.id[i] = values[i];
    set_len_kernel<<<1, 256, 0, s>>>(len_d, ids, vals);
    return cudaGetLastError();
}

cudaError_t launch_ring_copy(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                             size_t k_bytes, size_t v_bytes, cudaStream_t s) {
    const bool aligned = ((k_bytes | v_bytes | (size_t)src_k | (size_t)src_v | (size_t)dst_k | (size_t)dst_v) & 15) == 0;
    if (!aligned) {
        const size_t n = k_bytes + v_bytes;
        if (n == 0) return cudaSuccess;
        size_t grid = (n + 255) / 256;
        if (grid > 1184) grid = 1184;
        ring_copy_bytes_kernel<<<(unsigned)grid, 256, 0, s>>>(src_k, src_v, dst_k, dst_v, k_bytes, v_bytes);
        return cudaGetLastError();
    }
    const size_t nk = k_bytes / 16, nv = v_bytes / 16;
    const size_t n = nk + nv;
    if (n == 0) return cudaSuccess;
    size_t grid = (n + 255) / 256;
    if (grid > 1184) grid = 1184;
    ring_copy_kernel<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src_k),
                                                     reinterpret_cast<const uint4*>(src_v),
                                                     reinterpret_cast<uint4*>(dst_k),
                                                     reinterpret_cast<uint4*>(dst_v), nk, nv);
    return cudaGetLastError();
}

cudaError_t launch_truncate_accept(int* len_d, const int* base_d, int* err_d, const int* accept_d, int n, int T,
                                   int window, int ring, cudaStream_t s) {
    truncate_accept_kernel<<<(n + 255) / 256, 256, 0, s>>>(len_d, base_d, err_d, accept_d, n, T, window, ring);
    return cudaGetLastError();
}

bool launch_rebase_one_pass(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                            size_t k_bytes, size_t v_bytes, int* base_d, int seq, int new_base, int* arrive,
                            int* gen, int* err_d, int num_sms, cudaStream_t s, cudaError_t* err) {
    *err = cudaSuccess;
    if (((k_bytes | v_bytes | (size_t)src_k | (size_t)src_v | (size_t)dst_k | (size_t)dst_v) & 15) != 0)
        return false;
    const size_t total = (k_bytes + v_bytes) / 16;
    if (total == 0) return false;
    const int grid = (int)std::min<size_t>((size_t)num_sms, (total + 255) / 256);
    const size_t per = (total + grid - 1) / grid;
    const size_t smem = per * 16;
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(rebase_kernel, attrs, true);
    if (e != cudaSuccess) {
        *err = e;
        return true;
    }
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (smem + 1024 > (size_t)optin) return false;      // too large for one pass
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, rebase_kernel, reinterpret_cast<const uint4*>(src_k), reinterpret_cast<uint4*>(dst_k),
                           k_bytes / 16, reinterpret_cast<const uint4*>(src_v), reinterpret_cast<uint4*>(dst_v),
                           v_bytes / 16, base_d, seq, new_base, arrive, gen, err_d);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        return false;
    }
    *err = e != cudaSuccess ? e : cudaGetLastError();
    return true;
}

cudaError_t launch_set_base(int* base_d, int seq, int value, cudaStream_t s) {
    set_base_kernel<<<1, 1, 0, s>>>(base_d, seq, value);
    return cudaGetLastError();
}

}  // namespace kvq
