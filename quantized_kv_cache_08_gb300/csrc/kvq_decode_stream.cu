// Stream-K split decode for q8_0 / q5_1 and FP8 E4M3 caches whose token rows
// are 16-byte multiples.  Same semantics as the generic split kernel
// (kvq_decode.cu): cortiq-engine "Struct LayerKvCache" fn attend_group_upto
// (window, causal upto, sinks, GQA) over memra-engine "Struct KvLayer" rows.
//
// Work.  The visible rows of all sequences, repeated once per query slice,
// form one work space of W rows; CTA c takes rows [c W / G, (c + 1) W / G),
// so every CTA streams the same number of rows whatever the lengths are.  The
// part of a CTA's range inside one (slice, sequence) pair is a fragment; it
// is cut into tiles of 32 rows, and fragment (c, key = slice * B + sequence)
// writes its partial (max, sum, o) records to slot c + key (consecutive
// fragments in the work space differ by one in c or in key, so slots never
// collide).  A CTA needs no atomics and no work queue.
//
// A CTA has 16 warps.  A unit is (KV head, group of 4 queries); a tile's rows
// are split RS ways, and warp w owns unit w / RS and row slice w % RS of every
// tile.  Each warp computes the scores of its rows, runs the online softmax
// and accumulates p * v_hat itself, so no warp waits for another inside a
// tile.  K and V bytes of a tile arrive by per-row bulk copies
// (cp.async.bulk, one row per lane of the refilling warp) into rows padded to
// a stride that puts consecutive rows in different bank groups, in two rings
// of NS stages with an mbarrier each.  The last of the working warps to
// release a stage (an acquire-release shared counter decides) refills it with
// the tile NS ahead, whose coordinates it takes from a shared cursor over the
// CTA's range.
//
// K phase: lane = (row, part); the KP = 4 / QPL parts of a row take QPL of
// the unit's 4 queries each and read the whole head row.  The pre-scaled
// queries (scale * log2 e) are quantised per (query, head) to 16 bits and
// kept as pairs of 16-bit values; dp2a multiplies a pair by two int8 codes
// and accumulates in int32, so codes are never converted to float and the
// 2-byte misalignment of every other q8_0 block only selects the low or the
// high half of a code word.  With 24-bit queries a dp4a of the low bytes
// against the code words adds the rest.  Per block the sums are scaled by the
// block's d.
// Softmax: the reference maximum of each query moves only when a score
// exceeds it by more than 8 (log2 units); a warp vote finds that rare case,
// and since the same warp holds the value accumulators it rescales them in
// registers.  p goes to a small per-warp buffer in shared memory.
// V phase: lane = (row group, half block); a lane rebuilds the 16 5-bit codes
// of its half block with byte arithmetic, places each in the mantissa of 0.5
// (value 0.5 + u/256), so v_hat = 256 d F + (m - 128 d), and accumulates
// o += (256 p d) F with packed FMAs and sum p (m - 128 d) per block.
// E4M3 rows: this file compiled with KVQ_STREAM_F8 (kvq_decode_stream_f8.cu)
// gives stream_kernel_f8, whose queries stay f32; each code word of K and V
// becomes four exact floats (an E4M3 pair converts to a half pair, then to
// floats) and both phases multiply with packed FMAs; a V lane takes 16
// contiguous dims.  Everything else is shared line for line, and the q8_0 /
// q5_1 build of the file sees none of the E4M3 code.
#define KVQ_STREAM_TU 1
#include "kvq_device.cuh"

#include <type_traits>

#if KVQ_STREAM_F8
#include <cuda_fp8.h>
#define KVQ_STREAM_KERNEL stream_kernel_f8
#define KVQ_LAYOUT stream_layout_f8
#define KVQ_X2 8
#else
#define KVQ_STREAM_KERNEL stream_kernel
#define KVQ_LAYOUT stream_layout
#define KVQ_X2 16
#endif

namespace kvq {
namespace {

using namespace dev;

constexpr int kThreads = kStreamThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kRows = kStreamRows;
constexpr long long kWaitCycles = 1LL << 31;   // ~1 s bound on any mbarrier wait

template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<I + 1, N>(f);
    }
}

// d = c + a.h0 * b.byte0 + a.h1 * b.byte1 (lo) or bytes 2, 3 (hi); a: two
// signed 16-bit values, b: four signed 8-bit values
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// a: four signed 8-bit codes, b: four unsigned 8-bit query bytes
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t release_count(int* counter) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(counter)) : "memory");
    return old;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait; false once any wait of the CTA has run out (error word set).
// A waiting warp sleeps in try_wait (up to 20 us a try) instead of spinning,
// so it takes no issue slots from the warps still working; the clock and the
// abort flag are read between tries.
__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err_d) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicExch(err_d, kErrWait);
            *abort_flag = 1;
            return false;
        }
    }
}

// ------------------------------------------------------------ the walk

// floor(W c / G) for 0 <= W < 2^31 and 0 <= c <= G <= 2^16, in 32-bit
// arithmetic: W = q G + r gives q c + floor(r c / G)
__device__ __forceinline__ int range_bound(int W, int c, int G) {
    const unsigned q = (unsigned)W / (unsigned)G, r = (unsigned)W - q * (unsigned)G;
    return (int)(q * (unsigned)c + (r * (unsigned)c) / (unsigned)G);
}

// floor(n / d) for 0 <= n < 2^47 and 0 < d < 2^31 when the quotient is below
// 2^16: a float estimate, then exact integer corrections
__device__ __forceinline__ int small_quotient(long long n, long long d) {
    int q = (int)((float)n / (float)d);
    q = max(q, 0);
    while ((long long)q * d > n) --q;
    while ((long long)(q + 1) * d <= n) ++q;
    return q;
}

// Cursor over the CTA's range of the work space: the current fragment is
// key (qs, b), logical rows [row, end) with `start` its first row, and xrem
// rows of the range follow it.  Only one thread at a time touches it.
struct Walk {
    long long xrem;
    int qs, b, row, end, start, done;
};

struct Tables {
    const int* len;
    const int* base;
    const int* lo;     // first visible logical row
    const int* vis;    // visible rows (0: none or counters out of range)
    const int* pre;    // prefix of vis, [B + 1]
};

__device__ __forceinline__ Tables tables(const uint8_t* tabs, int B) {
    const int* t = reinterpret_cast<const int*>(tabs);
    Tables tb;
    tb.len = t;
    tb.base = t + (B + 1);
    tb.lo = t + 2 * (B + 1);
    tb.vis = t + 3 * (B + 1);
    tb.pre = t + 4 * (B + 1);
    return tb;
}

__device__ __forceinline__ void walk_init(Walk* w, const Tables& t, int B, long long R, long long x0, long long x1) {
    w->done = 0;
    if (x0 >= x1 || R <= 0) {
        w->b = -1;
        return;
    }
    const int qs = (int)((unsigned)x0 / (unsigned)R);        // both below 2^31
    const int xr = (int)(x0 - (long long)qs * R);
    int lo = 0, hi = B;                            // largest b with pre[b] <= xr
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (t.pre[mid] <= xr) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const int off = xr - t.pre[b];
    const int n = (int)min((long long)(t.vis[b] - off), x1 - x0);
    w->qs = qs;
    w->b = b;
    w->row = w->start = t.lo[b] + off;
    w->end = w->row + n;
    w->xrem = x1 - x0 - n;
}

// Take the next tile: {b, qs, first row, rows | last << 8 | first << 9};
// b = -1 marks the end (returned once), b = -2 nothing more.
constexpr int kTileLast = 256, kTileFirst = 512;

__device__ __forceinline__ int4 walk_take(Walk* w, const Tables& t, int B) {
    if (w->b < 0) {
        if (w->done) return make_int4(-2, 0, 0, 0);
        w->done = 1;
        return make_int4(-1, 0, 0, 0);
    }
    const int row = w->row;
    const int nr = min(kRows, w->end - row);
    const bool last = row + kRows >= w->end;
    const int4 tile = make_int4(w->b, w->qs, row, nr | (last ? kTileLast : 0) | (row == w->start ? kTileFirst : 0));
    if (!last) {
        w->row = row + kRows;
    } else if (w->xrem <= 0) {
        w->b = -1;
    } else {
        int b = w->b, qs = w->qs;
        do {
            if (++b == B) {
                b = 0;
                ++qs;
            }
        } while (t.vis[b] == 0);
        const int n = (int)min((long long)t.vis[b], w->xrem);
        w->b = b;
        w->qs = qs;
        w->row = w->start = t.lo[b];
        w->end = w->row + n;
        w->xrem -= n;
    }
    return tile;
}

// 32 rows from row y of a plane by one 2-D TMA tensor copy.  The map's element
// is 8 bytes and its box row is the padded stage row: the part past the token
// row lies outside the tensor and is filled with zeros, so rows land at the
// padded stride.  The rows are read once per decode: evict-first in L2.
__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap* map, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(bar), "l"(evict_first_policy())
        : "memory");
}

// ------------------------------------------------------- query preparation

// Quantise the 4 queries of unit (g, qg) of sequence b into this warp's
// words: query n = lane / 8, dims [(lane % 8) D / 8, +D / 8).  x' = x * scale
// * log2 e; q = rint(x' / sq) with sq = max |x'| over the head / QMAX.
// 16-bit words: W[block][pair of pairs][query][2], each word two dims; with
// 24 bits the 16-bit words hold the high part and LW[block][9][query] the
// low bytes, laid on the code words' byte grid of the block.
template <int NBH, int NQB>
__device__ __forceinline__ void prep_queries(const StreamParams& p, int b, int g, int qg, uint32_t* W, uint8_t* LW,
                                             float* SQ, int lane) {
    constexpr int D = NBH * 32;
    constexpr int PL = D / 8;
    const int n = lane >> 3, c8 = lane & 7;
    const int qi = 4 * qg + n;
    const bool valid = qi < p.Qh;
    const int t = valid ? qi / p.hpk : 0, hr = valid ? qi - t * p.hpk : 0;
    const int h = g * p.hpk + hr;
    const long long src = ((long long)(b * p.T + t) * p.Hq + h) * D + c8 * PL;
    auto load8 = [&](int k, float (&x)[8]) {
        if (!valid) {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
            return;
        }
        if (p.q_bf16) {
            const uint4 r = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + src + k);
            const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = __uint_as_float(w4[e] << 16);
                x[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
        } else {
            const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.q) + src + k);
            const float4 c = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.q) + src + k + 4);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
        }
    };
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < PL; k += 8) {
        float x[8];
        load8(k, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    constexpr float QMAX = NQB == 24 ? 8388607.f : 32767.f;
    const float am = amax * p.qscale;
    const float inv = am > 0.f ? QMAX / am : 0.f;
    if (c8 == 0) SQ[n] = am / QMAX;
    if (NQB == 24) {
        // zero this warp's low bytes (unused bytes stay zero)
        uint32_t* lw = reinterpret_cast<uint32_t*>(LW);
        for (int i = lane; i < NBH * 9 * 4; i += 32) lw[i] = 0u;
        __syncwarp();
    }
#pragma unroll
    for (int k = 0; k < PL; k += 8) {
        float x[8];
        load8(k, x);
        int v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int r = __float2int_rn(x[e] * p.qscale * inv);
            v[e] = max(-(int)QMAX, min((int)QMAX, r));
        }
        const int d0 = c8 * PL + k;                 // multiple of 8
        const int i = d0 >> 5, m0 = (d0 & 31) >> 1;   // block, first pair (multiple of 4)
        uint32_t w16[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int a = NQB == 24 ? (v[2 * j] >> 8) : v[2 * j];
            const int c = NQB == 24 ? (v[2 * j + 1] >> 8) : v[2 * j + 1];
            w16[j] = ((uint32_t)a & 0xffffu) | ((uint32_t)c << 16);
        }
        // pairs m0..m0+3 = pair-of-pairs m0/2 and m0/2 + 1, two words each
        *reinterpret_cast<uint2*>(W + ((i * 8 + (m0 >> 1)) * 4 + n) * 2) = make_uint2(w16[0], w16[1]);
        *reinterpret_cast<uint2*>(W + ((i * 8 + (m0 >> 1) + 1) * 4 + n) * 2) = make_uint2(w16[2], w16[3]);
        if (NQB == 24) {
            const bool mis = ((NBH * g + i) & 1) == 0;   // codes start 2 bytes into a word
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int pos = (mis ? 2 : 0) + (d0 & 31) + e;
                LW[((i * 9 + (pos >> 2)) * 4 + n) * 4 + (pos & 3)] = (uint8_t)(v[e] & 0xff);
            }
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------- K phase

// Score contributions of one q8_0 block whose d sits at byte O of the lane's
// 16-byte aligned head base kc; qw: this block's 16-bit query words of the
// lane's queries, lw: its low bytes (24-bit queries).
template <int QPL, int NQB, int O>
__device__ __forceinline__ void block_scores(const uint4* __restrict__ kc, const uint8_t* __restrict__ qw,
                                             const uint8_t* __restrict__ lw, float (&s)[QPL]) {
    constexpr int C0 = O >> 4;
    constexpr int NC = ((O + 35) >> 4) - C0 + 1;
    uint4 c[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) c[k] = kc[C0 + k];
    auto word = [&](int byte) -> uint32_t {
        const int rel = byte - C0 * 16;
        const uint4& ch = c[rel >> 4];
        const int w = (rel >> 2) & 3;
        return w == 0 ? ch.x : w == 1 ? ch.y : w == 2 ? ch.z : ch.w;
    };
    int acc[QPL];
#pragma unroll
    for (int j = 0; j < QPL; ++j) acc[j] = 0;
#pragma unroll
    for (int mp = 0; mp < 8; ++mp) {
        uint32_t w[QPL][2];
        if constexpr (QPL == 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(qw + mp * 32);
            const uint4 b = *reinterpret_cast<const uint4*>(qw + mp * 32 + 16);
            w[0][0] = a.x; w[0][1] = a.y; w[1][0] = a.z; w[1][1] = a.w;
            w[2][0] = b.x; w[2][1] = b.y; w[3][0] = b.z; w[3][1] = b.w;
        } else if constexpr (QPL == 2) {
            const uint4 a = *reinterpret_cast<const uint4*>(qw + mp * 32);
            w[0][0] = a.x; w[0][1] = a.y; w[1][0] = a.z; w[1][1] = a.w;
        } else {
            const uint2 a = *reinterpret_cast<const uint2*>(qw + mp * 32);
            w[0][0] = a.x; w[0][1] = a.y;
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int pos = O + 2 + 2 * (2 * mp + h2);   // byte of the code pair
            const uint32_t cw = word(pos);
#pragma unroll
            for (int j = 0; j < QPL; ++j)
                acc[j] = ((pos >> 1) & 1) ? dp2a_hi(w[j][h2], cw, acc[j]) : dp2a_lo(w[j][h2], cw, acc[j]);
        }
    }
    float tot[QPL];
    if constexpr (NQB == 24) {
        constexpr bool mis = (O & 3) == 0;
        constexpr int NW = mis ? 9 : 8;
        constexpr int B0 = mis ? O : O + 2;
        int accl[QPL];
#pragma unroll
        for (int j = 0; j < QPL; ++j) accl[j] = 0;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const uint32_t cw = word(B0 + 4 * k);
#pragma unroll
            for (int j = 0; j < QPL; ++j)
                accl[j] = dp4a_su(cw, *reinterpret_cast<const uint32_t*>(lw + k * 16 + 4 * j), accl[j]);
        }
#pragma unroll
        for (int j = 0; j < QPL; ++j) tot[j] = fmaf(256.f, (float)acc[j], (float)accl[j]);
    } else {
#pragma unroll
        for (int j = 0; j < QPL; ++j) tot[j] = (float)acc[j];
    }
    const uint32_t dw = word(O);
    const float d = h2f(((O >> 1) & 1) ? (dw >> 16) : (dw & 0xffffu));
#pragma unroll
    for (int j = 0; j < QPL; ++j) s[j] = fmaf(d, tot[j], s[j]);
}

template <int NBH, int QPL, int NQB, int PH>
__device__ __forceinline__ void head_scores(const uint4* kc, const uint8_t* qw, const uint8_t* lw, float (&s)[QPL]) {
    static_for<0, NBH>([&](auto I) {
        constexpr int i = decltype(I)::value;
        block_scores<QPL, NQB, PH + 34 * i>(kc, qw + i * 256, lw + i * 144, s);
    });
}

// The same scores read in 8-byte chunks from the head's first byte (8-byte
// aligned for head_dim 128: 136 g), so every head runs one code path: with
// 16-byte reads the heads of odd g start 8 bytes into a chunk and need their
// own unrolled path, and both paths are live at once, doubling the hot code.
template <int QPL, int NQB, int O>
__device__ __forceinline__ void block_scores8(const uint2* __restrict__ kc, const uint8_t* __restrict__ qw,
                                              const uint8_t* __restrict__ lw, float (&s)[QPL]) {
    constexpr int C0 = O >> 3;
    constexpr int NC = ((O + 35) >> 3) - C0 + 1;
    uint2 c[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) c[k] = kc[C0 + k];
    auto word = [&](int byte) -> uint32_t {
        const int rel = byte - C0 * 8;
        const uint2& ch = c[rel >> 3];
        return ((rel >> 2) & 1) ? ch.y : ch.x;
    };
    int acc[QPL];
#pragma unroll
    for (int j = 0; j < QPL; ++j) acc[j] = 0;
#pragma unroll
    for (int mp = 0; mp < 8; ++mp) {
        uint32_t w[QPL][2];
        if constexpr (QPL == 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(qw + mp * 32);
            const uint4 b = *reinterpret_cast<const uint4*>(qw + mp * 32 + 16);
            w[0][0] = a.x; w[0][1] = a.y; w[1][0] = a.z; w[1][1] = a.w;
            w[2][0] = b.x; w[2][1] = b.y; w[3][0] = b.z; w[3][1] = b.w;
        } else if constexpr (QPL == 2) {
            const uint4 a = *reinterpret_cast<const uint4*>(qw + mp * 32);
            w[0][0] = a.x; w[0][1] = a.y; w[1][0] = a.z; w[1][1] = a.w;
        } else {
            const uint2 a = *reinterpret_cast<const uint2*>(qw + mp * 32);
            w[0][0] = a.x; w[0][1] = a.y;
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int pos = O + 2 + 2 * (2 * mp + h2);
            const uint32_t cw = word(pos);
#pragma unroll
            for (int j = 0; j < QPL; ++j)
                acc[j] = ((pos >> 1) & 1) ? dp2a_hi(w[j][h2], cw, acc[j]) : dp2a_lo(w[j][h2], cw, acc[j]);
        }
    }
    float tot[QPL];
    if constexpr (NQB == 24) {
        constexpr bool mis = (O & 3) == 0;
        constexpr int NW = mis ? 9 : 8;
        constexpr int B0 = mis ? O : O + 2;
        int accl[QPL];
#pragma unroll
        for (int j = 0; j < QPL; ++j) accl[j] = 0;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const uint32_t cw = word(B0 + 4 * k);
#pragma unroll
            for (int j = 0; j < QPL; ++j)
                accl[j] = dp4a_su(cw, *reinterpret_cast<const uint32_t*>(lw + k * 16 + 4 * j), accl[j]);
        }
#pragma unroll
        for (int j = 0; j < QPL; ++j) tot[j] = fmaf(256.f, (float)acc[j], (float)accl[j]);
    } else {
#pragma unroll
        for (int j = 0; j < QPL; ++j) tot[j] = (float)acc[j];
    }
    const uint32_t dw = word(O);
    const float d = h2f(((O >> 1) & 1) ? (dw >> 16) : (dw & 0xffffu));
#pragma unroll
    for (int j = 0; j < QPL; ++j) s[j] = fmaf(d, tot[j], s[j]);
}

template <int NBH, int QPL, int NQB>
__device__ __forceinline__ void head_scores8(const uint2* kc, const uint8_t* qw, const uint8_t* lw, float (&s)[QPL]) {
    static_for<0, NBH>([&](auto I) {
        constexpr int i = decltype(I)::value;
        block_scores8<QPL, NQB, 34 * i>(kc, qw + i * 256, lw + i * 144, s);
    });
}

// PH = (34 * NBH * g) mod 16, the offset of the head's first block in its
// 16-byte chunk: 0 for NBH = 8, {0, 8} for NBH = 4, {0, 4, 8, 12} for NBH = 2
template <int NBH, int QPL, int NQB>
__device__ __forceinline__ void head_scores_ph(int ph, const uint4* kc, const uint8_t* qw, const uint8_t* lw,
                                               float (&s)[QPL]) {
    if constexpr (NBH == 8) {
        head_scores<NBH, QPL, NQB, 0>(kc, qw, lw, s);
    } else if constexpr (NBH == 4) {
        if (ph == 0) head_scores<NBH, QPL, NQB, 0>(kc, qw, lw, s);
        else head_scores<NBH, QPL, NQB, 8>(kc, qw, lw, s);
    } else {
        static_assert(NBH == 2, "head_dim 64, 128 or 256");
        switch (ph) {
            case 0: head_scores<NBH, QPL, NQB, 0>(kc, qw, lw, s); break;
            case 4: head_scores<NBH, QPL, NQB, 4>(kc, qw, lw, s); break;
            case 8: head_scores<NBH, QPL, NQB, 8>(kc, qw, lw, s); break;
            default: head_scores<NBH, QPL, NQB, 12>(kc, qw, lw, s); break;
        }
    }
}

// ------------------------------------------------------------- V phase

// One staged row for a V lane: its half block h (16 elements) of the block at
// vb, weighted by the row's 4 probabilities p4.  o2[n][2c + k] holds elements
// 2k, 2k + 1 of the lane's code word c: words 0, 1 are elements 8h + 0..7,
// words 2, 3 elements 16 + 8h + 0..7 of the block.
__device__ __forceinline__ void v_row(const uint8_t* vb, int h, uint32_t sel_lo, uint32_t sel_hi, const float4 p4,
                                      float2 (&o2)[4][8], float (&pm)[4]) {
    const uint2 dmqh = *reinterpret_cast<const uint2*>(vb);
    const uint2 qs = *reinterpret_cast<const uint2*>(vb + 8 + 8 * h);
    const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&dmqh.x));
    const float mp = fmaf(-128.f, dm.x, dm.y);
    const float pr[4] = {p4.x, p4.y, p4.z, p4.w};   // 256 p
    float2 t2[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        const float t = pr[n] * dm.x;
        t2[n] = make_float2(t, t);
        pm[n] = fmaf(pr[n], mp, pm[n]);
    }
    // fifth bits of the lane's elements: qh byte h (elements 8h..) and byte
    // h + 2 (elements 16 + 8h..), replicated; bit k of a byte moved to bit 4
    // of byte k by masking and adding (no carries between bytes)
    const uint32_t xl = __byte_perm(dmqh.y, 0, sel_lo);
    const uint32_t xh = __byte_perm(dmqh.y, 0, sel_hi);
    const uint32_t s0 = (xl & 0x08040201u) + 0x080C0E0Fu;
    const uint32_t s1 = ((xl >> 4) & 0x08040201u) + 0x080C0E0Fu;
    const uint32_t s2 = (xh & 0x08040201u) + 0x080C0E0Fu;
    const uint32_t s3 = ((xh >> 4) & 0x08040201u) + 0x080C0E0Fu;
    uint32_t u[4];
    u[0] = (qs.x & 0x0F0F0F0Fu) | (s0 & 0xF0F0F0F0u);
    u[1] = (qs.y & 0x0F0F0F0Fu) | (s1 & 0xF0F0F0F0u);
    u[2] = ((qs.x >> 4) & 0x0F0F0F0Fu) | (s2 & 0xF0F0F0F0u);
    u[3] = ((qs.y >> 4) & 0x0F0F0F0Fu) | (s3 & 0xF0F0F0F0u);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // code byte k into bits 16..23 under the exponent of 0.5
        const float2 fa = make_float2(__uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7044u)),
                                      __uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7144u)));
        const float2 fb = make_float2(__uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7244u)),
                                      __uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7344u)));
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            o2[n][2 * c] = __ffma2_rn(t2[n], fa, o2[n][2 * c]);
            o2[n][2 * c + 1] = __ffma2_rn(t2[n], fb, o2[n][2 * c + 1]);
        }
    }
}

#if KVQ_STREAM_F8
// ------------------------------------------------------------ FP8 E4M3 rows

// Two E4M3 bytes (element order: low byte first) as two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_float2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The 4 queries of unit (g, qg) of sequence b, pre-scaled (scale * log2 e)
// and kept as f32: Wf[block][word of 4 codes][query][4], so a lane reads the
// 4 values of a code word for its queries with one 16-byte load each.
template <int NBH>
__device__ __forceinline__ void prep_queries_f8(const StreamParams& p, int b, int g, int qg, float* Wf, float* SQ,
                                                int lane) {
    constexpr int D = NBH * 32;
    constexpr int PL = D / 8;
    const int n = lane >> 3, c8 = lane & 7;
    const int qi = 4 * qg + n;
    const bool valid = qi < p.Qh;
    const int t = valid ? qi / p.hpk : 0, hr = valid ? qi - t * p.hpk : 0;
    const int h = g * p.hpk + hr;
    const long long src = ((long long)(b * p.T + t) * p.Hq + h) * D + c8 * PL;
#pragma unroll
    for (int k = 0; k < PL; k += 4) {
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            if (p.q_bf16) {
                const uint2 r = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.q) + src + k);
                x[0] = __uint_as_float(r.x << 16);
                x[1] = __uint_as_float(r.x & 0xffff0000u);
                x[2] = __uint_as_float(r.y << 16);
                x[3] = __uint_as_float(r.y & 0xffff0000u);
            } else {
                const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.q) + src + k);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            }
        }
        const int d0 = c8 * PL + k;
        const int i = d0 >> 5, w = (d0 & 31) >> 2;
        *reinterpret_cast<float4*>(Wf + ((i * 8 + w) * 4 + n) * 4) =
            make_float4(x[0] * p.qscale, x[1] * p.qscale, x[2] * p.qscale, x[3] * p.qscale);
    }
    if (c8 == 0) SQ[n] = 1.f;
    __syncwarp();
}

// Scores of one E4M3 head row (D bytes at kc) for the lane's QPL queries:
// each code word becomes 4 floats, multiplied into two partial sums per query
// with packed FMAs.
template <int NBH, int QPL>
__device__ __forceinline__ void head_scores_f8(const uint4* __restrict__ kc, const float* __restrict__ qw,
                                               float (&s)[QPL]) {
    float2 acc[QPL];
#pragma unroll
    for (int j = 0; j < QPL; ++j) acc[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NBH; ++i) {
        const uint4 c0 = kc[2 * i], c1 = kc[2 * i + 1];
        const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float2 k01 = e4m3x2_float2(wv[w]), k23 = e4m3x2_float2(wv[w] >> 16);
#pragma unroll
            for (int j = 0; j < QPL; ++j) {
                const float4 q4 = *reinterpret_cast<const float4*>(qw + ((i * 8 + w) * 4 + j) * 4);
                acc[j] = __ffma2_rn(k01, make_float2(q4.x, q4.y), acc[j]);
                acc[j] = __ffma2_rn(k23, make_float2(q4.z, q4.w), acc[j]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < QPL; ++j) s[j] = acc[j].x + acc[j].y;
}

// One staged E4M3 row for a V lane: its 16 contiguous dims, weighted by the
// row's 4 probabilities p4 (256 p); o2[n][k] holds dims 2k, 2k + 1.
__device__ __forceinline__ void v_row_f8(const uint8_t* vb, const float4 p4, float2 (&o2)[4][8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(vb);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 fa = e4m3x2_float2(wv[c]), fb = e4m3x2_float2(wv[c] >> 16);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const float2 t2 = make_float2(pr[n], pr[n]);
            o2[n][2 * c] = __ffma2_rn(t2, fa, o2[n][2 * c]);
            o2[n][2 * c + 1] = __ffma2_rn(t2, fb, o2[n][2 * c + 1]);
        }
    }
}

#endif  // KVQ_STREAM_F8

// ------------------------------------------------------------ the kernel

template <int NBH, int KP, int NQB>
__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm) KVQ_STREAM_KERNEL(const StreamParams p,
                                                              const __grid_constant__ CUtensorMap kmap,
                                                              const __grid_constant__ CUtensorMap vmap) {
    constexpr int D = NBH * 32;
    constexpr int RW = 32 / KP;         // rows of a tile per warp: RW rows x KP lanes
    constexpr int RS = kRows / RW;      // row slices of a tile: warps per unit
    static_assert(RS >= 1 && RS <= 2 && RS * RW == kRows, "a tile splits into one or two row slices");
    constexpr int QPL = 4 / KP;         // queries per lane in the K phase
    constexpr int VH = 2 * NBH;         // half blocks per head: V lanes per row group
    constexpr int RG = 32 / VH;         // V row groups
    constexpr int VR = RW / RG;         // rows per V lane per tile
    static_assert(VR >= 1, "row slice shorter than the V row groups");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // TMA tile destinations need 128-byte alignment
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const StreamLayout L = KVQ_LAYOUT(p);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, NS = p.NS;
    int* s_tab = reinterpret_cast<int*>(smem + L.tabs);
    const Tables tb = tables(smem + L.tabs, B);
    int4* s_tinfo = reinterpret_cast<int4*>(smem + L.tinfo);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);   // one per stage: K and V bytes of a tile
    int* cnt = reinterpret_cast<int*>(smem + L.cnt);                // releases of each stage
    int* arm = cnt + NS;                                            // times each stage was armed
    Walk* s_walk = reinterpret_cast<Walk*>(smem + L.walk);
    __shared__ int s_abort;
    __shared__ int s_wsum[kWarps];
    __shared__ __align__(8) uint64_t s_pair[kWarps];   // per unit of two row slices: sums in, sums read

    if (tid == 0) s_abort = 0;
    // launched as a programmatic dependent of the kernel before it (an append
    // lets it start early): nothing that kernel may write is read before this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // ---- visible rows of every sequence from the device counters, prefix sums
    int v2[2] = {0, 0};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int b = 2 * tid + e;
        if (b < B) {
            const int len = p.len_d[b], base = p.base_d[b];
            const int lo = p.window > 0 ? max(0, len - p.T + 1 - p.window) : 0;
            const bool bad = len < p.T || base < 0 || len - base > p.max_rows || lo < base;
            if (bad && blockIdx.x == 0) atomicExch(p.err_d, kErrCounter);
            int* t = s_tab;
            t[b] = len;
            t[(B + 1) + b] = base;
            t[2 * (B + 1) + b] = lo;
            t[3 * (B + 1) + b] = bad ? 0 : len - lo;
            v2[e] = bad ? 0 : len - lo;
        }
    }
    {
        const int own = v2[0] + v2[1];
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < kWarps ? s_wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < kWarps) s_wsum[lane] = w;      // inclusive totals of warps
        }
        __syncthreads();
        const int excl = x - own + (warp > 0 ? s_wsum[warp - 1] : 0);
        int* pre = s_tab + 4 * (B + 1);
        if (2 * tid < B) pre[2 * tid] = excl;
        if (2 * tid + 1 < B) pre[2 * tid + 1] = excl + v2[0];
        if (tid == 0) pre[B] = s_wsum[kWarps - 1];
    }
    __syncthreads();
    const long long R = tb.pre[B];
    const long long Wtot = R * p.nqs;                // below 2^31 (checked on the host)
    const long long x0 = range_bound((int)Wtot, blockIdx.x, p.G), x1 = range_bound((int)Wtot, blockIdx.x + 1, p.G);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            cnt[s] = arm[s] = 0;
        }
        for (int s = 0; s < kWarps; ++s) mbar_init(smem_u32(&s_pair[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        walk_init(s_walk, tb, B, R, x0, x1);
    }
    __syncthreads();
    // let the merge grid launch; it waits for this grid before reading partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const uint32_t kst0 = smem_u32(smem + L.kst), vst0 = smem_u32(smem + L.vst);
    const uint32_t full0 = smem_u32(full);
    // one tile into stage s: both planes complete on the stage's barrier
    auto issue = [&](int s, int4 tile) {
        const uint32_t bar = full0 + 8u * (uint32_t)s;
        if (tile.x < 0) {
            mbar_arrive(bar);
            return;
        }
        const int y = tile.x * p.max_rows + (tile.z - tb.base[tile.x]);
        mbar_expect_tx(bar, L.kstage + L.vstage);
        tma_rows(kst0 + (uint32_t)s * L.kstage, &kmap, y, bar);
        tma_rows(vst0 + (uint32_t)s * L.vstage, &vmap, y, bar);
    };
    // ---- the first tile now; the next NS - 1 once warp 0 has its queries, so
    // that the query loads of every CTA do not queue behind the copy burst
    if (tid == 0) {
        const int4 tile = walk_take(s_walk, tb, B);     // a tile, or the end marker
        s_tinfo[0] = tile;
        arm[0] = 1;
        issue(0, tile);
    }
    __syncthreads();
    if (warp >= p.NA) return;

    // ---- this warp: unit (KV head g, query group qgl of a slice), row slice rs
    const int u = warp / RS, rs = warp - u * RS;
    const int g = u / p.QPS, qgl = u - g * p.QPS;
    const uint32_t w_off = (uint32_t)L.W + (uint32_t)warp * L.wwarp;
    const uint32_t lw_off = (uint32_t)L.LW + (uint32_t)warp * L.lwarp;
    // per-warp state: [0..3] reference maxima, [4..7] query scales, [8..11]
    // first visible row, [12..15] one past the last (ints), per query
    float* STw = reinterpret_cast<float*>(smem + L.SQ + (size_t)warp * 64);
    int* STi = reinterpret_cast<int*>(STw);
    const uint32_t p_off = (uint32_t)L.P + (uint32_t)warp * L.pwarp;
    volatile int* abort_flag = &s_abort;
    const bool causal = p.T > 1;                     // per-query row windows inside a fragment

    // K-phase lane: row kr of the warp's slice, part kp (queries kp*QPL..)
    const int kr = lane / KP, kp = lane - kr * KP;
    const int trow = rs * RW + kr;                  // tile row of this K lane
#if KVQ_STREAM_F8
    const int hb0 = D * g;                          // byte of the head's row in a token row
#else
    const int hb0 = 34 * NBH * g;                   // byte of the head's first K block in a row
#endif
    const int ph = hb0 & 15;
    const uint32_t k_lane_off = (uint32_t)L.kst + (uint32_t)trow * p.Sk + (uint32_t)(hb0 - ph);
    // V-phase lane: row group vg, half block vh of block vi
    const int vg = lane / VH, vhb = lane - vg * VH;
    const int vi = vhb >> 1, vh = vhb & 1;
#if KVQ_STREAM_F8
    // 16 contiguous dims of the head
    const uint32_t v_lane_off = (uint32_t)L.vst + (uint32_t)(rs * RW + vg) * p.Sv + (uint32_t)(D * g + 16 * vhb);
#else
    const uint32_t v_lane_off = (uint32_t)L.vst + (uint32_t)(rs * RW + vg) * p.Sv + (uint32_t)(24 * (NBH * g + vi));
#endif
    const uint32_t v_step = (uint32_t)RG * p.Sv;

    float lsum[QPL], sq[QPL], pm[4];
    float2 o2[4][8];
    auto reset = [&]() {
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            pm[n] = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) o2[n][c] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < QPL; ++jj) lsum[jj] = 0.f;
        if (lane < 4) STw[lane] = kNegInf;
    };
    reset();
    int key = -1;
    int nfrag = 0;                                  // records handed over between the two row slices
    // a new fragment: this warp's queries and row windows for (slice qs, sequence b)
    auto begin_fragment = [&](int b, int qs) {
        key = b * 65536 + qs;
        const int qg = qs * p.QPS + qgl;
#if KVQ_STREAM_F8
        prep_queries_f8<NBH>(p, b, g, qg, reinterpret_cast<float*>(smem + w_off), STw + 4, lane);
#else
        prep_queries<NBH, NQB>(p, b, g, qg, reinterpret_cast<uint32_t*>(smem + w_off), smem + lw_off, STw + 4,
                               lane);
#endif
        if (lane < 4) {
            const int qi = 4 * qg + lane;
            int lo = 0, hi = -1;
            if (qi < p.Qh) {
                hi = tb.len[b] - p.T + qi / p.hpk + 1;
                lo = p.window > 0 ? max(0, hi - p.window) : 0;
            }
            STi[8 + lane] = lo;
            STi[12 + lane] = hi;
        }
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < QPL; ++jj) sq[jj] = STw[4 + kp * QPL + jj];
    };
    {
        // the first fragment's queries load while the first tile is in flight
        const int4 t0 = s_tinfo[0];
        if (t0.x >= 0) begin_fragment(t0.x, t0.y);
        if (tid == 0 && t0.x >= 0) {
            for (int j = 1; j < NS; ++j) {
                const int4 tile = walk_take(s_walk, tb, B);
                if (tile.x == -2) break;
                s_tinfo[j] = tile;
                arm[j] = 1;
                issue(j, tile);
                if (tile.x < 0) break;
            }
        }
    }

    // tile j sits in stage st = j mod NS, use u = j div NS of it (phase parity
    // u & 1); its info in slot ti = j mod 2 NS, the refill's in (j + NS) mod 2 NS
    int st = 0, ti = 0;
    uint32_t use = 0;
    for (;;) {
        if (!wait_full(full0 + 8u * st, use & 1u, abort_flag, p.err_d)) break;
        const int4 tile = s_tinfo[ti];
        if (tile.x < 0) break;
        const int row0 = tile.z, nr = tile.w & 255;
        const bool full_tile = nr == kRows;
        if (tile.x * 65536 + tile.y != key) begin_fragment(tile.x, tile.y);
        // ------------------------------------------------ scores
        float sc[QPL];
#pragma unroll
        for (int jj = 0; jj < QPL; ++jj) sc[jj] = 0.f;
        if (full_tile || trow < nr) {
            const uint4* kc = reinterpret_cast<const uint4*>(smem + k_lane_off + (uint32_t)st * L.kstage);
#if KVQ_STREAM_F8
            head_scores_f8<NBH, QPL>(kc, reinterpret_cast<const float*>(smem + w_off) + kp * QPL * 4, sc);
#else
            if constexpr (NBH == 4)
                head_scores8<NBH, QPL, NQB>(reinterpret_cast<const uint2*>(smem + k_lane_off + ph + (uint32_t)st * L.kstage),
                                            smem + w_off + kp * QPL * 8, smem + lw_off + kp * QPL * 4, sc);
            else
                head_scores_ph<NBH, QPL, NQB>(ph, kc, smem + w_off + kp * QPL * 8, smem + lw_off + kp * QPL * 4, sc);
#endif
        }
        // ------------------------------------------------ online softmax
        // the lane's queries n = kp * QPL + jj: scale, visible rows, reference max
        float mr[QPL];
        {
            const bool in_tile = full_tile || trow < nr;
            const int lrow = row0 + trow;
#pragma unroll
            for (int jj = 0; jj < QPL; ++jj) {
                const int n = kp * QPL + jj;
                float s = sc[jj] * sq[jj];
                if (p.softcap_b > 0.f) s = p.softcap_b * tanhf(p.softcap_a * s);
                bool vis = in_tile;
                if (causal) vis = vis && lrow >= STi[8 + n] && lrow < STi[12 + n];
                sc[jj] = vis ? s : kNegInf;
                mr[jj] = STw[n];
            }
        }
        bool mv = false;
#pragma unroll
        for (int jj = 0; jj < QPL; ++jj) mv |= sc[jj] > mr[jj] + kLazy;
        if (__any_sync(0xffffffffu, mv)) {
            // a reference maximum moves: the tile maximum of every query
            // (uniform in the warp) rescales the warp's accumulators
            float al[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                float v = kNegInf;
#pragma unroll
                for (int jj = 0; jj < QPL; ++jj)
                    if (kp * QPL + jj == n) v = sc[jj];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                const float old = STw[n];
                al[n] = 1.f;
                if (v > old + kLazy) {
                    al[n] = (old == kNegInf) ? 0.f : exp2f(old - v);
                    pm[n] *= al[n];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        o2[n][c].x *= al[n];
                        o2[n][c].y *= al[n];
                    }
                    __syncwarp();
                    if (lane == 0) STw[n] = v;
                }
            }
#pragma unroll
            for (int jj = 0; jj < QPL; ++jj) {
                float a = al[0];
#pragma unroll
                for (int n = 1; n < 4; ++n)
                    if (kp * QPL + jj == n) a = al[n];
                lsum[jj] *= a;
            }
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < QPL; ++jj) mr[jj] = STw[kp * QPL + jj];
        }
        float pv[QPL];
#pragma unroll
        for (int jj = 0; jj < QPL; ++jj) {
            pv[jj] = sc[jj] == kNegInf ? 0.f : exp2f(sc[jj] - mr[jj] + 8.f);    // 256 p
            lsum[jj] += pv[jj];
        }
        {
            float* dst = reinterpret_cast<float*>(smem + p_off) + kr * 4 + kp * QPL;
            if constexpr (QPL == 4) *reinterpret_cast<float4*>(dst) = make_float4(pv[0], pv[1], pv[2], pv[3]);
            else if constexpr (QPL == 2) *reinterpret_cast<float2*>(dst) = make_float2(pv[0], pv[1]);
            else *dst = pv[0];
        }
        __syncwarp();
        // ------------------------------------------------ value accumulation
        {
            const uint8_t* vb = smem + v_lane_off + (uint32_t)st * L.vstage;
            const float* pw = reinterpret_cast<const float*>(smem + p_off) + vg * 4;
            const uint32_t sel_lo = vh ? 0x1111u : 0x0000u, sel_hi = vh ? 0x3333u : 0x2222u;
#if KVQ_STREAM_F8
            if (full_tile) {
#pragma unroll
                for (int k = 0; k < VR; ++k)
                    v_row_f8(vb + k * v_step, *reinterpret_cast<const float4*>(pw + k * RG * 4), o2);
            } else {
#pragma unroll
                for (int k = 0; k < VR; ++k)
                    if (rs * RW + vg + k * RG < nr)
                        v_row_f8(vb + k * v_step, *reinterpret_cast<const float4*>(pw + k * RG * 4), o2);
            }
#else
            if (full_tile) {
#pragma unroll
                for (int k = 0; k < VR; ++k)
                    v_row(vb + k * v_step, vh, sel_lo, sel_hi, *reinterpret_cast<const float4*>(pw + k * RG * 4), o2,
                          pm);
            } else {
#pragma unroll
                for (int k = 0; k < VR; ++k)
                    if (rs * RW + vg + k * RG < nr)
                        v_row(vb + k * v_step, vh, sel_lo, sel_hi, *reinterpret_cast<const float4*>(pw + k * RG * 4),
                              o2, pm);
            }
#endif
        }
        // done with the stage: the last working warp refills it with tile j + NS
        __syncwarp();
        if (lane == 0 && release_count(&cnt[st]) == (use + 1) * (uint32_t)p.NA - 1 && !*abort_flag) {
            const int4 nt = walk_take(s_walk, tb, B);
            if (nt.x != -2) {
                s_tinfo[ti < NS ? ti + NS : ti - NS] = nt;
                arm[st] += 1;
                issue(st, nt);
            }
        }
        // ------------------------------------------------ end of a fragment
        if (tile.w & kTileLast) {
            // the fragment's record: sums over the warp's rows (K lanes of a
            // part, V row groups); with two row slices the second warp's sums
            // reach the first through a shared-memory buffer of the unit (an
            // mbarrier hand-over each way: sums in, and, before the next
            // record's sums go in, sums read), and the first writes one record
            // per query.  P holds 256 p: t = P d is p (256 d), so the
            // value sum comes out unscaled, while pm and l carry the 256.
            const int b = tile.x, qs = tile.y;
            const int qg = qs * p.QPS + qgl;
#pragma unroll
            for (int jj = 0; jj < QPL; ++jj)
#pragma unroll
                for (int o = KP; o < 32; o <<= 1) lsum[jj] += __shfl_xor_sync(0xffffffffu, lsum[jj], o);
            float m4[4], l4[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                m4[n] = STw[n];
                l4[n] = __shfl_sync(0xffffffffu, lsum[n % QPL], n / QPL);
            }
#pragma unroll
            for (int n = 0; n < 4; ++n) {
#if !KVQ_STREAM_F8
                if constexpr (KP == 2) {
                    // q8_0 / q5_1 with two row slices: a rolled loop here frees
                    // registers for the whole kernel (measured: fewer spills,
                    // batch64 1.7 % faster; the other builds are faster unrolled)
#pragma unroll 1
                    for (int o = VH; o < 32; o <<= 1) {
                        pm[n] += __shfl_xor_sync(0xffffffffu, pm[n], o);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            o2[n][c] = __fadd2_rn(o2[n][c], make_float2(__shfl_xor_sync(0xffffffffu, o2[n][c].x, o),
                                                                        __shfl_xor_sync(0xffffffffu, o2[n][c].y, o)));
                    }
                } else
#endif
#pragma unroll
                for (int o = VH; o < 32; o <<= 1) {
                    pm[n] += __shfl_xor_sync(0xffffffffu, pm[n], o);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        o2[n][c] = __fadd2_rn(o2[n][c], make_float2(__shfl_xor_sync(0xffffffffu, o2[n][c].x, o),
                                                                    __shfl_xor_sync(0xffffffffu, o2[n][c].y, o)));
                }
#if KVQ_STREAM_F8
                // o = sum 256 p v / 256
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    o2[n][c].x *= 1.f / 256.f;
                    o2[n][c].y *= 1.f / 256.f;
                }
#else
                // o = sum 256 p d F + sum 256 p (m - 128 d) / 256
                const float a = pm[n] * (1.f / 256.f);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    o2[n][c].x += a;
                    o2[n][c].y += a;
                }
#endif
            }
#if KVQ_STREAM_F8
            const int dcol = 16 * vhb;                  // the lane's dims: dcol + 0..15
#else
            const int dcol = vi * 32 + 8 * vh;          // the lane's dims: dcol + 0..7, dcol + 16..23
#endif
            bool write = true;
            if constexpr (RS == 2) {
                float* so = reinterpret_cast<float*>(smem + L.CB + (size_t)u * (16 * D + 32));   // [4][D], m[4], l[4]
                float* sml = so + 4 * D;
                const uint32_t pf = smem_u32(&s_pair[2 * u]), pe = smem_u32(&s_pair[2 * u + 1]);
                if (rs == 1) {
                    // the first warp has read the previous record's sums
                    if (nfrag > 0) wait_full(pe, (uint32_t)((nfrag - 1) & 1), abort_flag, p.err_d);
                    if (lane < VH) {
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            float* d4 = so + n * D + dcol;
                            *reinterpret_cast<float4*>(d4) = make_float4(o2[n][0].x, o2[n][0].y, o2[n][1].x, o2[n][1].y);
                            *reinterpret_cast<float4*>(d4 + 4) = make_float4(o2[n][2].x, o2[n][2].y, o2[n][3].x, o2[n][3].y);
                            *reinterpret_cast<float4*>(d4 + KVQ_X2) = make_float4(o2[n][4].x, o2[n][4].y, o2[n][5].x, o2[n][5].y);
                            *reinterpret_cast<float4*>(d4 + KVQ_X2 + 4) = make_float4(o2[n][6].x, o2[n][6].y, o2[n][7].x, o2[n][7].y);
                        }
                    }
                    if (lane == 0) {
                        *reinterpret_cast<float4*>(sml) = make_float4(m4[0], m4[1], m4[2], m4[3]);
                        *reinterpret_cast<float4*>(sml + 4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(pf);
                    write = false;
                } else {
                    wait_full(pf, (uint32_t)(nfrag & 1), abort_flag, p.err_d);
                    const float4 mo = *reinterpret_cast<const float4*>(sml);
                    const float4 lo = *reinterpret_cast<const float4*>(sml + 4);
                    const float mo4[4] = {mo.x, mo.y, mo.z, mo.w}, lo4[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const float M = fmaxf(m4[n], mo4[n]);
                        const float a = m4[n] == kNegInf ? 0.f : exp2f(m4[n] - M);
                        const float c2 = mo4[n] == kNegInf ? 0.f : exp2f(mo4[n] - M);
                        m4[n] = M;
                        l4[n] = l4[n] * a + lo4[n] * c2;
                        if (lane < VH) {
                            const float* s4 = so + n * D + dcol;
                            const float4 x0 = *reinterpret_cast<const float4*>(s4);
                            const float4 x1 = *reinterpret_cast<const float4*>(s4 + 4);
                            const float4 x2 = *reinterpret_cast<const float4*>(s4 + KVQ_X2);
                            const float4 x3 = *reinterpret_cast<const float4*>(s4 + KVQ_X2 + 4);
                            const float xs[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                                  x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                o2[n][c].x = o2[n][c].x * a + xs[2 * c] * c2;
                                o2[n][c].y = o2[n][c].y * a + xs[2 * c + 1] * c2;
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(pe);
                }
                ++nfrag;
            }
            if (write) {
                // slot's records: the slice's queries, unit u's at 4 u .. 4 u + 3
                const long long slot = (long long)blockIdx.x + (long long)qs * B + b;
                const int QS = 4 * p.Hkv * p.QPS;
                float* po = p.part_o + slot * QS * D + dcol;
                float* pml = p.part_ml + slot * QS * 2;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    if (4 * qg + n >= p.Qh) continue;
                    const int off = 4 * u + n;
                    if (lane < VH) {
                        float* dst = po + (size_t)off * D;
                        *reinterpret_cast<float4*>(dst) = make_float4(o2[n][0].x, o2[n][0].y, o2[n][1].x, o2[n][1].y);
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(o2[n][2].x, o2[n][2].y, o2[n][3].x, o2[n][3].y);
                        *reinterpret_cast<float4*>(dst + KVQ_X2) = make_float4(o2[n][4].x, o2[n][4].y, o2[n][5].x, o2[n][5].y);
                        *reinterpret_cast<float4*>(dst + KVQ_X2 + 4) = make_float4(o2[n][6].x, o2[n][6].y, o2[n][7].x, o2[n][7].y);
                    }
                    if (lane == 0)
                        *reinterpret_cast<float2*>(pml + (size_t)off * 2) = make_float2(m4[n], l4[n] * (1.f / 256.f));
                }
            }
            __syncwarp();
            reset();
            __syncwarp();
        }
        if (++st == NS) {
            st = 0;
            ++use;
        }
        ti = ti + 1 == 2 * NS ? 0 : ti + 1;
    }
    if (*abort_flag && lane == 0) {
        // a wait ran out: copies still landing in this CTA's shared memory
        // must finish before it ends (bounded waits on every armed phase)
        for (int s2 = 0; s2 < NS; ++s2) {
            const int n2 = *(volatile int*)&arm[s2];
            if (n2 == 0) continue;
            const long long t0 = clock64();
            while (!mbar_try(full0 + 8u * s2, (uint32_t)((n2 - 1) & 1)) && clock64() - t0 < kWaitCycles) {
            }
        }
    }
}

#if !KVQ_STREAM_F8
// ------------------------------------------------------------- the merge

// Combine the partial records of one (sequence, query) over the fragments of
// its range with the sink (cortiq-engine "Struct LayerKvCache", fn
// attend_group_upto: the sink joins the max and the denominator and carries
// no value), in log2 units:
//   M = max(sink, m_r), L = 2^(sink - M) + sum l_r 2^(m_r - M),
//   out = sum o_r 2^(m_r - M) / L.
// The records of (b, q) are those of the CTAs whose ranges meet the rows
// [xa, xb) of key (slice of q, b): CTA c covers [c W / G, (c + 1) W / G), so
// the CTA holding row x is ((x + 1) G - 1) / W, and with fewer rows W than
// CTAs a range may be empty (no record).  The rows [xa, xb) come from the
// prefix of visible rows, which each merge CTA derives from the counters by
// the split kernel's rule while the split grid still runs (the merge is its
// programmatic dependent; the counters do not change until both end), so the
// only wait on the split is for the records.  A CTA has 16 warps; WPQ
// warps share one (sequence, query, chunk of DC = 32 * VPL dims), each
// folding every WPQ-th record with U records' loads in flight, and their
// states meet in shared memory.
template <int VPL, int U>
__global__ void __launch_bounds__(kMergeThreads) merge_stream_kernel(const MergeStreamParams p) {
    extern __shared__ float msm[];                   // [pairs][WPQ][2 + DC]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int PPC = kMergeWarps / p.WPQ;
    const int pl = warp / p.WPQ, sub = warp - pl * p.WPQ;
    const int DC = 32 * VPL;
    const int NCH = p.D / DC;
    const long long pair = (long long)blockIdx.x * PPC + pl;
    const long long npairs = (long long)p.B * p.Qtot * NCH;
    const bool live = pair < npairs;
    int b = 0, qg = 0, ch = 0;
    if (live) {
        ch = (int)(pair % NCH);
        const long long r = pair / NCH;
        qg = (int)(r % p.Qtot);
        b = (int)(r / p.Qtot);
    }
    // the prefix of visible rows, by the split kernel's rule, while the split
    // grid still runs: the counters are final once it has started
    int* spre = reinterpret_cast<int*>(msm + kMergeWarps * (2 + DC));   // [B + 1]
    {
        __shared__ int s_wsum[kMergeWarps];
        int v2[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int bb = 2 * (int)threadIdx.x + e;
            if (bb < p.B) {
                const int len = p.len_d[bb], base = p.base_d[bb];
                const int lo = p.window > 0 ? max(0, len - p.T + 1 - p.window) : 0;
                const bool bad = len < p.T || base < 0 || len - base > p.max_rows || lo < base;
                v2[e] = bad ? 0 : len - lo;
            }
        }
        const int own = v2[0] + v2[1];
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < kMergeWarps ? s_wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < kMergeWarps) s_wsum[lane] = w;
        }
        __syncthreads();
        const int excl = x - own + (warp > 0 ? s_wsum[warp - 1] : 0);
        if (2 * (int)threadIdx.x < p.B) spre[2 * threadIdx.x] = excl;
        if (2 * (int)threadIdx.x + 1 < p.B) spre[2 * threadIdx.x + 1] = excl + v2[0];
        if (threadIdx.x == 0) spre[p.B] = s_wsum[kMergeWarps - 1];
        __syncthreads();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int R = spre[p.B];
    const int t = qg / p.Hq, h = qg - t * p.Hq;
    const int qi = t * p.hpk + (h % p.hpk);
    const int qs = (qi >> 2) / p.QPS;
    // the query's record in a slot: unit (KV head, query group in the slice), member
    const int QS = 4 * (p.Hq / p.hpk) * p.QPS;
    const int qloc = ((h / p.hpk) * p.QPS + (qi >> 2) - qs * p.QPS) * 4 + (qi & 3);
    const int key = qs * p.B + b;
    const int xa = qs * R + spre[b];
    const int xb = xa + (spre[b + 1] - spre[b]);
    int c_lo = 0, nrec = 0;
    const long long W = (long long)R * p.nqs;
    if (live && xb > xa) {
        // the CTAs holding rows xa and xb - 1: CTA c starts at floor(c W / G),
        // so the CTA of row x is ((x + 1) G - 1) / W
        c_lo = small_quotient((long long)(xa + 1) * p.G - 1, W);
        const int c_hi = small_quotient((long long)xb * p.G - 1, W);
        nrec = c_hi - c_lo + 1;
    }
    // with fewer rows than CTAs some ranges are empty and wrote no record
    const bool some_empty = W < p.G;
    const int dim0 = ch * DC + lane * VPL;
    float M = kNegInf, Ls = 0.f, acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
    for (int r0 = sub; r0 < nrec; r0 += U * p.WPQ) {
        float m4[U], l4[U], o4[U][VPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * p.WPQ;
            bool ok = r < nrec;
            long long rec = 0;
            if (ok) {
                const int c = c_lo + r;
                if (some_empty) ok = range_bound((int)W, c + 1, p.G) > range_bound((int)W, c, p.G);
                rec = (long long)(c + key) * QS + qloc;
            }
            const float2 mlv = ok ? *reinterpret_cast<const float2*>(p.part_ml + rec * 2) : make_float2(kNegInf, 0.f);
            m4[u] = mlv.x;
            l4[u] = mlv.y;
            const float* src = p.part_o + rec * p.D + dim0;
            if constexpr (VPL % 4 == 0) {
#pragma unroll
                for (int v = 0; v < VPL; v += 4) {
                    const float4 x = ok ? *reinterpret_cast<const float4*>(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                    o4[u][v] = x.x;
                    o4[u][v + 1] = x.y;
                    o4[u][v + 2] = x.z;
                    o4[u][v + 3] = x.w;
                }
            } else if constexpr (VPL == 2) {
                const float2 x = ok ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
                o4[u][0] = x.x;
                o4[u][1] = x.y;
            } else {
                o4[u][0] = ok ? src[0] : 0.f;
            }
        }
        float Mr = M;
#pragma unroll
        for (int u = 0; u < U; ++u) Mr = fmaxf(Mr, m4[u]);
        if (Mr == kNegInf) continue;
        const float a = (M == kNegInf) ? 0.f : exp2f(M - Mr);
        Ls *= a;
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[v] *= a;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float w = (m4[u] == kNegInf) ? 0.f : exp2f(m4[u] - Mr);
            Ls = fmaf(l4[u], w, Ls);
#pragma unroll
            for (int v = 0; v < VPL; ++v) acc[v] = fmaf(o4[u][v], w, acc[v]);
        }
        M = Mr;
    }
    float* st = msm + (size_t)(pl * p.WPQ + sub) * (2 + DC);
    if (lane == 0) {
        st[0] = M;
        st[1] = Ls;
    }
#pragma unroll
    for (int v = 0; v < VPL; ++v) st[2 + lane * VPL + v] = acc[v];
    __syncthreads();
    if (sub == 0 && live) {
        const float sink = p.sinks ? p.sinks[h] * 1.4426950408889634f : kNegInf;
        const float* q0 = msm + (size_t)pl * p.WPQ * (2 + DC);
        float Mt = sink;
        for (int w = 0; w < p.WPQ; ++w) Mt = fmaxf(Mt, q0[w * (2 + DC)]);
        float Lt = (sink == kNegInf) ? 0.f : exp2f(sink - Mt);
        float At[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) At[v] = 0.f;
        for (int w = 0; w < p.WPQ; ++w) {
            const float* e = q0 + w * (2 + DC);
            if (e[0] == kNegInf) continue;
            const float f = exp2f(e[0] - Mt);
            Lt = fmaf(e[1], f, Lt);
#pragma unroll
            for (int v = 0; v < VPL; ++v) At[v] = fmaf(e[2 + lane * VPL + v], f, At[v]);
        }
        float* dst = p.out + ((long long)b * p.Qtot + qg) * p.D + dim0;
#pragma unroll
        for (int v = 0; v < VPL; ++v) dst[v] = At[v] / Lt;
    }
}

#endif  // !KVQ_STREAM_F8

template <int NBH, int KP, int NQB>
cudaError_t launch_stream_t(const StreamParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, size_t smem,
                            cudaStream_t s) {
    auto fn = KVQ_STREAM_KERNEL<NBH, KP, NQB>;
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(fn, attrs, true);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, p, kmap, vmap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#if !KVQ_STREAM_F8
template <int VPL, int U>
cudaError_t launch_merge_stream_t(const MergeStreamParams& p, cudaStream_t s) {
    const int PPC = kMergeWarps / p.WPQ;
    const long long npairs = (long long)p.B * p.Qtot * (p.D / (32 * VPL));
    const size_t smem = (size_t)kMergeWarps * (2 + 32 * VPL) * sizeof(float) + (size_t)(p.B + 1) * sizeof(int);
    auto fn = merge_stream_kernel<VPL, U>;
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(fn, attrs, true);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((npairs + PPC - 1) / PPC), 1, 1);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#endif  // !KVQ_STREAM_F8

}  // namespace

#if !KVQ_STREAM_F8
cudaError_t launch_split_stream(const StreamParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t s) {
    const size_t smem = stream_layout(p).total;
    const int NBH = p.D / 32;
    const int KP = p.RS * 32 / kStreamRows;       // lanes per row in the key phase
#define KVQ_CASE(nb, kp, nq) \
    if (NBH == nb && KP == kp && p.qbits == nq) return launch_stream_t<nb, kp, nq>(p, kmap, vmap, smem, s);
    KVQ_CASE(2, 1, 16) KVQ_CASE(2, 2, 16) KVQ_CASE(4, 1, 16) KVQ_CASE(4, 2, 16) KVQ_CASE(8, 1, 16) KVQ_CASE(8, 2, 16)
    KVQ_CASE(2, 1, 24) KVQ_CASE(2, 2, 24) KVQ_CASE(4, 1, 24) KVQ_CASE(4, 2, 24) KVQ_CASE(8, 1, 24) KVQ_CASE(8, 2, 24)
#undef KVQ_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge_stream(const MergeStreamParams& p, cudaStream_t s) {
    switch (p.DC / 32) {
        case 1: return launch_merge_stream_t<1, 16>(p, s);
        case 2: return launch_merge_stream_t<2, 16>(p, s);
        case 4: return launch_merge_stream_t<4, 8>(p, s);
        case 8: return launch_merge_stream_t<8, 4>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

bool make_stream_map(CUtensorMap* map, void* plane, int tok_bytes, int stride_bytes, long long rows) {
    using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Encode encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<Encode>(fn);
    }
    if (tok_bytes % 16 || stride_bytes % 16 || stride_bytes < tok_bytes || stride_bytes > 2048 || rows < 1)
        return false;
    // dims: 8-byte word of a token row, row; the box spans stride_bytes of a
    // row, past its end (zero fill, no memory read)
    const cuuint64_t dims[2] = {(cuuint64_t)(tok_bytes / 8), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)tok_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(stride_bytes / 8), (cuuint32_t)kStreamRows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, plane, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int stream_max_smem() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return v - 256;  // static shared variables
}

#else
cudaError_t launch_split_stream_f8(const StreamParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   cudaStream_t s) {
    const size_t smem = stream_layout_f8(p).total;
    const int NBH = p.D / 32;
    const int KP = p.RS * 32 / kStreamRows;       // lanes per row in the key phase
#define KVQ_CASE(nb, kp) \
    if (NBH == nb && KP == kp) return launch_stream_t<nb, kp, 16>(p, kmap, vmap, smem, s);
    KVQ_CASE(2, 1) KVQ_CASE(2, 2) KVQ_CASE(4, 1) KVQ_CASE(4, 2) KVQ_CASE(8, 1) KVQ_CASE(8, 2)
#undef KVQ_CASE
    return cudaErrorInvalidValue;
}
#endif  // !KVQ_STREAM_F8

}  // namespace kvq
