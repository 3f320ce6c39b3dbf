// Warp-specialised split-K decode for caches whose token rows are 16-byte
// multiples (n_kv_heads * head_dim % 256 == 0).  Same semantics, work items,
// partial records and merge as the generic split kernel (kvq_decode.cu):
// cortiq-engine "Struct LayerKvCache" fn attend_group_upto (window, causal
// upto, sinks, GQA) over memra-engine "Struct KvLayer" q8_0 / q5_1 rows.
//
// A CTA has 16 warps.  Warps 0-7 (K warps) only turn key rows into scores;
// warps 8-15 (V warps) issue every copy, run the online softmax and
// accumulate p * v_hat.  The two sides work on different tiles at once: the
// K warps may run two 32-row tiles ahead, with two score / probability
// buffers handed over through named barriers (bar.arrive / bar.sync).  Key
// bytes land in padded row slots through 16-byte cp.async copies tracked by
// an mbarrier (cp.async.mbarrier.arrive); value bytes of a tile arrive by one
// 1-D bulk TMA copy (cp.async.bulk) on its own mbarrier ring.
//
// K warps: lane = token row.  The swizzle puts the same 16-byte column of 8
// consecutive rows in 8 different bank groups, so the 32 lanes read their
// rows with conflict-free 16-byte loads.  The query is
// pre-scaled by scale * log2 e, quantised per (query, 32-element block) to
// NLIMB*8 bits against the block's largest magnitude (24 bits: the error is
// at the level of fp32 rounding) and split into int8 limbs held in shared
// memory; every lane reads the same limb words (broadcast).  DP4A multiplies
// four int8 codes by four limb bytes and accumulates in int32, so the codes
// are never converted to float; per block the limb sums are combined in
// float and scaled by d_k * s_q.
//
// V warps, softmax: a warp owns every 8th query of the CTA; lane = row.  The
// reference maximum moves only when a score exceeds it by more than 8 (log2
// units); a warp vote finds that rare case, otherwise p = 2^(s - m_ref) needs
// no reduction and each lane keeps a partial sum of p until the item ends.
// V warps, accumulation: a task is (query group of 4, KV head, block, half
// block); a warp holds TW consecutive tasks and 32/TW lane groups that take
// interleaved rows, so the row partial sums reduce with warp shuffles at the
// end of an item.  The 5-bit codes are rebuilt with byte arithmetic and placed
// in the mantissa of 0.5 (value 0.5 + u/256), so v_hat = 256 d F + (m - 128 d)
// and o += (256 p d) F with packed FMAs, plus sum p (m - 128 d) per block.
#include "kvq_device.cuh"

namespace kvq {
namespace {

using namespace dev;

constexpr int kThreads = kFastThreads;
constexpr int kRows = kFastRows;
constexpr int kSDepth = kFastSDepth;               // score buffers between K and V warps
constexpr int kKThreads = 256;                 // warps 0-7
constexpr int BAR_K = 1, BAR_V = 2, BAR_QLOAD = 3, BAR_FULL = 4, BAR_EMPTY = 4 + kSDepth;
constexpr long long kWaitCycles = 1LL << 31;   // ~1 s bound on any mbarrier wait

__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint4 lds128u(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
// 3-D TMA tile load of box {0, y, 0} of a tensor map into shared memory
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(bar)
        : "memory");
}

// Byte `col` of staged row `r` in a tile laid out by tma_load_rows: column
// block col / 128 holds the 32 rows at 128 bytes each, 16-byte chunk j of
// row r stored at chunk j ^ (r & 7) (the TMA 128-byte swizzle).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int col) {
    return base + (uint32_t)(col >> 7) * (kFastRows * 128) + (uint32_t)r * 128u +
           ((((uint32_t)col >> 4) & 7u) ^ ((uint32_t)r & 7u)) * 16u + ((uint32_t)col & 15u);
}
__device__ __forceinline__ int dp4a_su(unsigned a, unsigned b, int c) {   // a: 4 x s8, b: 4 x u8
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(unsigned a, unsigned b, int c) {   // a, b: 4 x s8
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Bounded wait that gives up for the whole CTA once any wait has run out: the
// error word is set, later waits return at once, and every thread still runs
// the full barrier protocol (results are then garbage but the kernel ends).
__device__ __forceinline__ void wait_stage(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err_d) {
    if (*abort_flag) return;
    if (mbar_try(bar, parity)) return;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (*abort_flag) return;
        if (clock64() - t0 > kWaitCycles) {
            atomicExch(err_d, kErrWait);
            *abort_flag = 1;
            return;
        }
    }
}

// Tile cursor over this CTA's items (blockIdx.x, +gridDim.x, ...), with the
// current item's decode cached so a tile step costs no division.
struct Cursor {
    int item, tile;
    Item it;
    int row0, n, base, len;
};

struct TileInfo {
    int b, r0, nr, base, len;
    bool first, last;
    Item it;
};

__device__ __forceinline__ void cursor_load(Cursor& c, const SplitParams& p, const int* lens, const int* bases,
                                            const int* prefix, int n_items) {
    if (c.item >= n_items) return;
    c.it = item_of(c.item, prefix, p.B, p.nqs);
    const ItemRows ir = item_rows(p, lens, bases, c.it);
    c.row0 = ir.row0;
    c.n = ir.n;
    c.base = ir.base;
    c.len = ir.len;
}

__device__ __forceinline__ Cursor cursor_begin(const SplitParams& p, const int* lens, const int* bases,
                                               const int* prefix, int n_items) {
    Cursor c;
    c.item = blockIdx.x;
    c.tile = 0;
    cursor_load(c, p, lens, bases, prefix, n_items);
    return c;
}

__device__ __forceinline__ TileInfo tile_of(const Cursor& c) {
    TileInfo ti;
    ti.it = c.it;
    ti.b = c.it.b;
    ti.base = c.base;
    ti.len = c.len;
    ti.r0 = c.row0 + c.tile * kRows;
    ti.nr = min(kRows, c.row0 + c.n - ti.r0);
    ti.first = c.tile == 0;
    ti.last = ti.r0 + ti.nr >= c.row0 + c.n;
    return ti;
}

__device__ __forceinline__ void advance(Cursor& c, const TileInfo& ti, const SplitParams& p, const int* lens,
                                        const int* bases, const int* prefix, int n_items) {
    if (ti.last) {
        c.item += gridDim.x;
        c.tile = 0;
        cursor_load(c, p, lens, bases, prefix, n_items);
    } else {
        ++c.tile;
    }
}

// Dot products of one key block against 4 queries, 32 dims, code bytes
// starting at byte O (compile-time, even) of the 48 staged bytes w[0..11].
template <int NLIMB, int O>
__device__ __forceinline__ void block_dot(const uint32_t (&w)[12], uint32_t ql_addr, uint32_t qs_addr, float (&sc)[4]) {
    int acc[NLIMB][4];
#pragma unroll
    for (int l = 0; l < NLIMB; ++l)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[l][n] = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        constexpr int dummy = 0;
        (void)dummy;
        const int byte = O + 2 + 4 * k;                    // compile-time after unrolling
        const int wi = byte >> 2;
        const uint32_t cw = (byte & 2) ? __byte_perm(w[wi], w[wi + 1], 0x5432u) : w[wi];
#pragma unroll
        for (int l = 0; l < NLIMB; ++l) {
            const uint4 qw = lds128u(ql_addr + (uint32_t)((k * NLIMB + l) * 16));
            if (l == NLIMB - 1) {
                acc[l][0] = dp4a_ss(cw, qw.x, acc[l][0]);
                acc[l][1] = dp4a_ss(cw, qw.y, acc[l][1]);
                acc[l][2] = dp4a_ss(cw, qw.z, acc[l][2]);
                acc[l][3] = dp4a_ss(cw, qw.w, acc[l][3]);
            } else {
                acc[l][0] = dp4a_su(cw, qw.x, acc[l][0]);
                acc[l][1] = dp4a_su(cw, qw.y, acc[l][1]);
                acc[l][2] = dp4a_su(cw, qw.z, acc[l][2]);
                acc[l][3] = dp4a_su(cw, qw.w, acc[l][3]);
            }
        }
    }
    const uint32_t dbits = (O & 2) ? (w[O >> 2] >> 16) : (w[O >> 2] & 0xffffu);
    const float d = h2f(dbits);
    const float4 s4 = lds128f(qs_addr);
    const float sq[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        float tot;
        if (NLIMB == 3) {
            const int c = acc[1][n] * 256 + acc[0][n];     // |c| < 2^28: no overflow
            tot = fmaf((float)acc[2][n], 65536.f, (float)c);
        } else {
            tot = (float)(acc[1][n] * 256 + acc[0][n]);
        }
        sc[n] = fmaf(d * sq[n], tot, sc[n]);
    }
}

// Scores of 4 queries for the lane's row over the NBH blocks of head g.
// G16 = (2 * g * NBH) mod 16 fixes the byte offset of every block in its
// 16-byte chunk.
// Key tile layout: box b holds bytes [128 b, 128 b + 128) of the 32 rows, row
// r at b * 4096 + r * 128, its 16-byte chunk j stored at chunk j ^ (r & 7)
// (the TMA 128-byte swizzle), so 8 consecutive rows read one column through
// 8 different bank groups.
__device__ __forceinline__ uint32_t key_chunk(uint32_t kbase, uint32_t rowoff, uint32_t sw, int chunk) {
    return kbase + (uint32_t)(chunk >> 3) * (kFastRows * 128) + rowoff + ((((uint32_t)chunk & 7u) ^ sw) << 4);
}

template <int NBH, int NLIMB, int G16>
__device__ __forceinline__ void head_scores(uint32_t kbase, uint32_t rowoff, uint32_t sw, int g, uint32_t ql_unit,
                                            uint32_t qs_unit, float (&sc)[4]) {
#pragma unroll
    for (int bi = 0; bi < NBH; ++bi) {
        constexpr int dummy = 0;
        (void)dummy;
        const int blk = g * NBH + bi;
        const int c = (34 * blk) >> 4;                   // first 16-byte chunk of the block
        const uint4 c0 = lds128u(key_chunk(kbase, rowoff, sw, c));
        const uint4 c1 = lds128u(key_chunk(kbase, rowoff, sw, c + 1));
        const uint4 c2 = lds128u(key_chunk(kbase, rowoff, sw, c + 2));
        const uint32_t w[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
        const uint32_t ql = ql_unit + (uint32_t)(bi * 8 * NLIMB * 16);
        const uint32_t qs = qs_unit + (uint32_t)(bi * 16);
        switch ((G16 + 2 * bi) & 15) {
            case 0: block_dot<NLIMB, 0>(w, ql, qs, sc); break;
            case 2: block_dot<NLIMB, 2>(w, ql, qs, sc); break;
            case 4: block_dot<NLIMB, 4>(w, ql, qs, sc); break;
            case 6: block_dot<NLIMB, 6>(w, ql, qs, sc); break;
            case 8: block_dot<NLIMB, 8>(w, ql, qs, sc); break;
            case 10: block_dot<NLIMB, 10>(w, ql, qs, sc); break;
            case 12: block_dot<NLIMB, 12>(w, ql, qs, sc); break;
            default: block_dot<NLIMB, 14>(w, ql, qs, sc); break;
        }
    }
}

template <int NBH, int NLIMB>
__device__ __forceinline__ void head_scores_dispatch(uint32_t kbase, uint32_t rowoff, uint32_t sw, int g,
                                                     uint32_t ql_unit, uint32_t qs_unit, float (&sc)[4]) {
    const int g16 = (2 * g * NBH) & 15;
    if constexpr (NBH >= 8) {
        head_scores<NBH, NLIMB, 0>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc);
    } else if constexpr (NBH == 4) {
        if (g16 == 0) head_scores<NBH, NLIMB, 0>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc);
        else head_scores<NBH, NLIMB, 8>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc);
    } else if constexpr (NBH == 2) {
        switch (g16) {
            case 0: head_scores<NBH, NLIMB, 0>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 4: head_scores<NBH, NLIMB, 4>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 8: head_scores<NBH, NLIMB, 8>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            default: head_scores<NBH, NLIMB, 12>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
        }
    } else {
        switch (g16) {
            case 0: head_scores<NBH, NLIMB, 0>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 2: head_scores<NBH, NLIMB, 2>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 4: head_scores<NBH, NLIMB, 4>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 6: head_scores<NBH, NLIMB, 6>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 8: head_scores<NBH, NLIMB, 8>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 10: head_scores<NBH, NLIMB, 10>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            case 12: head_scores<NBH, NLIMB, 12>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
            default: head_scores<NBH, NLIMB, 14>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc); break;
        }
    }
}

template <int NBH, int NQG, int NLIMB>
__global__ void __launch_bounds__(kThreads, 1) fast_kernel(const SplitParams p, const __grid_constant__ CUtensorMap kmap,
                                                            const __grid_constant__ CUtensorMap vmap) {
    constexpr int QC = 4 * NQG;
    constexpr int D = NBH * 32;
    constexpr int NQMAX = 32 * NQG;                 // CTA queries (Hkv * QC, Hkv <= 8): <= 4 * NQG per softmax warp
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // swizzled TMA boxes need a 1024-byte aligned destination
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const FastLayout L = fast_layout(p, NLIMB);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.Hkv;
    const int NQ = Hkv * QC;
    const int PS = NQ + 4;                          // row stride of the probability buffer

    uint8_t* kring = smem + L.kring;
    uint8_t* vring = smem + L.vring;
    uint32_t* qlimb = reinterpret_cast<uint32_t*>(smem + L.qlimb);
    float* qscl = reinterpret_cast<float*>(smem + L.qscale);
    float* S = reinterpret_cast<float*>(smem + L.S);            // [kSDepth][NQ][kRows]
    float* P = reinterpret_cast<float*>(smem + L.P);            // [2][kRows][PS]
    float* alpha = reinterpret_cast<float*>(smem + L.alpha);    // [2][NQ]
    int* qlo = reinterpret_cast<int*>(smem + L.mrun);           // [NQ] first visible row per CTA query
    int* qup = reinterpret_cast<int*>(smem + L.lrun);           // [NQ] one past the last (-1: no query)
    int* lens = reinterpret_cast<int*>(smem + L.lens);
    int* bases = lens + p.B;
    int* prefix = bases + p.B;
    uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* vbar = kbar + p.nstage_k;
    __shared__ int s_abort;
    __shared__ Cursor s_kc, s_vc;                   // copy producer state (V thread 0 only)
    __shared__ int s_k_issued, s_v_issued;

    for (int b = tid; b < p.B; b += kThreads) {
        lens[b] = p.len_d[b];
        bases[b] = p.base_d[b];
    }
    if (tid == 0) s_abort = 0;
    __syncthreads();
    if (warp == 0) plan_splits(p, lens, bases, prefix, lane);
    if (tid == 0) {
        for (int s2 = 0; s2 < p.nstage_k; ++s2) mbar_init(smem_u32(&kbar[s2]), 1);
        for (int s2 = 0; s2 < p.nstage_v; ++s2) mbar_init(smem_u32(&vbar[s2]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int b = tid; b <= p.B; b += kThreads) p.plan[b] = prefix[b];
    const int n_items = prefix[p.B] * p.nqs;
    // let the merge grid launch now; it waits (griddepcontrol.wait) for this
    // grid to complete before reading any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x >= n_items) return;

    if (warp < 8) {
        // ======================================================== K warps
        // lane = token row of the tile; each warp scores whole (head, query
        // group) units and hands the scores over to the V warps.
        const int kt = tid;
        Cursor c = cursor_begin(p, lens, bases, prefix, n_items);
        int jt = 0;
        while (c.item < n_items) {
            const TileInfo ti = tile_of(c);
            if (ti.first) {
                // quantise this item's pre-scaled queries into int8 limbs: one
                // thread per 4 consecutive dims of a query, the 8 threads of a
                // 32-dim block share its largest magnitude through shuffles
                bar_sync(BAR_K, kKThreads);          // previous item's scores are done
                const int nunits = NQ * (D / 4);
                constexpr int QB = 4;                // units per thread whose loads are in flight together
                for (int u0 = 0; u0 < nunits; u0 += QB * kKThreads) {
                    float xs[QB][4];
#pragma unroll
                    for (int j = 0; j < QB; ++j) {
                        const int u = u0 + j * kKThreads + kt;
                        const int qq = u / (D / 4), w4 = u % (D / 4);
                        const int g = qq / QC, ql = qq % QC;
                        const int qi = ti.it.qs * QC + ql;
#pragma unroll
                        for (int e = 0; e < 4; ++e) xs[j][e] = 0.f;
                        if (u < nunits && qi < p.hpk * p.T) {
                            const int t = qi / p.hpk, h = g * p.hpk + qi % p.hpk;
                            const long long base = ((long long)(ti.b * p.T + t) * p.Hq + h) * D + 4 * w4;
                            if (p.q_bf16) {
                                const uint2 raw = *reinterpret_cast<const uint2*>(
                                    reinterpret_cast<const __nv_bfloat16*>(p.q) + base);
                                xs[j][0] = __uint_as_float(raw.x << 16);
                                xs[j][1] = __uint_as_float(raw.x & 0xffff0000u);
                                xs[j][2] = __uint_as_float(raw.y << 16);
                                xs[j][3] = __uint_as_float(raw.y & 0xffff0000u);
                            } else {
                                const float4 f =
                                    *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.q) + base);
                                xs[j][0] = f.x;
                                xs[j][1] = f.y;
                                xs[j][2] = f.z;
                                xs[j][3] = f.w;
                            }
                        }
                    }
                    // the first item's query loads go out ahead of the tile stream:
                    // the copy producer waits for this signal before its first copies
                    if (jt == 0 && u0 == 0) bar_arrive(BAR_QLOAD, kKThreads + 32);
#pragma unroll
                    for (int j = 0; j < QB; ++j) {
                        const int u = u0 + j * kKThreads + kt;
                        const bool act = u < nunits;
                        const int qq = act ? u / (D / 4) : 0, w4 = act ? u % (D / 4) : 0;
                        const int bi = w4 >> 3, k = w4 & 7;
                        const int g = qq / QC, ql = qq % QC;
                        float x[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) x[e] = xs[j][e] * p.qscale;
                        // the 8 threads of a 32-dim block (consecutive lanes) share its maximum
                        float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
                        for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        constexpr float QMAX = NLIMB == 3 ? 8388607.f : 32767.f;
                        const float inv = mx > 0.f ? QMAX / mx : 0.f;
                        int v4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int v = __float2int_rn(x[e] * inv);
                            v4[e] = max(-(int)QMAX, min((int)QMAX, v));
                        }
                        if (act) {
                            const int qg = ql >> 2, n = ql & 3;
                            const int unit = g * NQG + qg;
                            uint32_t* dst = qlimb + (size_t)((unit * NBH + bi) * 8 + k) * NLIMB * 4;
#pragma unroll
                            for (int l = 0; l < NLIMB; ++l) {
                                uint32_t word = 0;
#pragma unroll
                                for (int e = 0; e < 4; ++e) word |= (uint32_t)((v4[e] >> (8 * l)) & 0xff) << (8 * e);
                                dst[l * 4 + n] = word;
                            }
                            if (k == 0) qscl[(unit * NBH + bi) * 4 + n] = mx / QMAX;
                        }
                    }
                }
                for (int qq = kt; qq < NQ; qq += kKThreads) {
                    const int qi = ti.it.qs * QC + qq % QC;
                    const bool valid = qi < p.hpk * p.T;
                    const int upto = ti.len - p.T + (valid ? qi / p.hpk : 0) + 1;
                    qup[qq] = valid ? upto : -1;
                    qlo[qq] = p.window > 0 ? max(0, upto - p.window) : 0;
                }
                bar_sync(BAR_K, kKThreads);          // limbs and row windows visible to every K warp
            }
            // ------------------------------------------------ scores
            const int kst = jt % p.nstage_k;
            wait_stage(smem_u32(&kbar[kst]), (uint32_t)((jt / p.nstage_k) & 1), &s_abort, p.err_d);
            const uint32_t kbase = smem_u32(kring + (size_t)kst * L.kstage);
            const uint32_t rowoff = (uint32_t)lane * 128u, sw = (uint32_t)lane & 7u;
            const int sb = jt % kSDepth;
            if (jt >= kSDepth) bar_sync(BAR_EMPTY + sb, kThreads);  // V has read the scores of tile jt-kSDepth
            float* Sb = S + sb * NQ * kRows;
            const int row = ti.r0 + lane;
#pragma unroll 1
            for (int unit = warp; unit < Hkv * NQG; unit += 8) {
                const int g = unit / NQG, qg = unit - g * NQG;
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                if (lane < ti.nr) {
                    const uint32_t ql_unit = smem_u32(qlimb + (size_t)(unit * NBH) * 8 * NLIMB * 4);
                    const uint32_t qs_unit = smem_u32(qscl + (size_t)(unit * NBH) * 4);
                    head_scores_dispatch<NBH, NLIMB>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc);
                }
                const int qq0 = g * QC + 4 * qg;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const bool vis = lane < ti.nr && row >= qlo[qq0 + n] && row < qup[qq0 + n];
                    Sb[(qq0 + n) * kRows + lane] = vis ? sc[n] : kNegInf;
                }
            }
            bar_arrive(BAR_FULL + sb, kThreads);           // scores of tile jt; K stage jt is free
            advance(c, ti, p, lens, bases, prefix, n_items);
            ++jt;
        }
        for (int j = max(kSDepth, jt); j < jt + kSDepth; ++j) bar_sync(BAR_EMPTY + j % kSDepth, kThreads);
    } else {
        // ======================================================== V warps
        // copy issue, online softmax, p * v_hat accumulation
        const int vt = tid - kKThreads;
        const int vw = warp - 8;
        // key and value tiles: one 3-D TMA box each (32 rows x all column
        // blocks, 128-byte swizzle).  V thread 0 issues; its cursors live in
        // shared memory.
        auto issue_k = [&]() {
            Cursor kc = s_kc;
            if (kc.item >= n_items) return;
            const TileInfo ti = tile_of(kc);
            const int st = s_k_issued % p.nstage_k;
            const uint32_t bar = smem_u32(&kbar[st]);
            mbar_expect_tx(bar, (uint32_t)L.kstage);
            tma_load_rows(smem_u32(kring + (size_t)st * L.kstage), &kmap, ti.b * p.max_rows + (ti.r0 - ti.base), bar);
            ++s_k_issued;
            advance(kc, ti, p, lens, bases, prefix, n_items);
            s_kc = kc;
        };
        auto issue_v = [&]() {
            Cursor vc = s_vc;
            if (vc.item >= n_items) return;
            const TileInfo ti = tile_of(vc);
            const int st = s_v_issued % p.nstage_v;
            const uint32_t bar = smem_u32(&vbar[st]);
            mbar_expect_tx(bar, (uint32_t)L.vstage);
            tma_load_rows(smem_u32(vring + (size_t)st * L.vstage), &vmap, ti.b * p.max_rows + (ti.r0 - ti.base), bar);
            ++s_v_issued;
            advance(vc, ti, p, lens, bases, prefix, n_items);
            s_vc = vc;
        };
        if (vw == 0) bar_sync(BAR_QLOAD, kKThreads + 32);
        if (vt == 0) {
            s_kc = cursor_begin(p, lens, bases, prefix, n_items);
            s_vc = s_kc;
            s_k_issued = 0;
            s_v_issued = 0;
            for (int s2 = 0; s2 < p.nstage_k; ++s2) issue_k();
            for (int s2 = 0; s2 < p.nstage_v; ++s2) issue_v();
        }

        // softmax state: this warp owns queries qq = vw + 8 i; m_ref per query
        // (warp-uniform), lane-partial sums of p
        float m_ref[NQMAX / 8], lsum[NQMAX / 8];
#pragma unroll
        for (int i = 0; i < NQMAX / 8; ++i) {
            m_ref[i] = kNegInf;
            lsum[i] = 0.f;
        }
        // accumulation task: TW tasks per warp (consecutive lanes), the warp's
        // 32 / TW lane groups take interleaved rows of the tile, so partial
        // sums over rows meet inside the warp and reduce with shuffles
        const int nV = 2 * NQG * Hkv * NBH;             // tasks per row
        const int TW = nV / 8;                          // tasks per warp
        const int RG = 32 / TW;                         // row groups (lane groups) per warp
        // lanes past TW * RG (TW not a power of two) hold no rows
        const int v_task = vw * TW + lane % TW, v_rg = lane / TW;
        const int v_hf = v_task & 1, v_bi = (v_task >> 1) % NBH, v_g = (v_task >> 1) / NBH % Hkv;
        const int v_qg = (v_task >> 1) / (NBH * Hkv);
        const int v_blk = v_g * NBH + v_bi;
        const int v_qq0 = v_g * QC + 4 * v_qg;
        const int col_dm = v_blk * kQ5Bytes;            // d, m, qh of the thread's block
        const int col_qs = col_dm + 8 + 8 * v_hf;       // its 8 bytes of qs
        float2 o2[4][8];
        float pm[4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            pm[n] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
        }
        Cursor c = cursor_begin(p, lens, bases, prefix, n_items);
        int jt = 0;
        while (c.item < n_items) {
            const TileInfo ti = tile_of(c);
            const int sb = jt % kSDepth;
            bar_sync(BAR_FULL + sb, kThreads);             // scores of tile jt are in
            // ------------------------------------------------ online softmax
            const float* Sb = S + sb * NQ * kRows;
            float* Pb = P + (jt & 1) * kRows * PS;
            float* ab = alpha + (jt & 1) * NQ;
#pragma unroll
            for (int i = 0; i < NQMAX / 8; ++i) {
                const int qq = vw + 8 * i;
                if (qq < NQ) {
                    const float s = Sb[qq * kRows + lane];
                    float al = 1.f;
                    if (__any_sync(0xffffffffu, s > m_ref[i] + kLazy)) {
                        // the reference maximum moves: full tile maximum
                        float tmax = s;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                        al = (m_ref[i] == kNegInf) ? 0.f : exp2f(m_ref[i] - tmax);
                        m_ref[i] = tmax;
                        lsum[i] *= al;
                    }
                    const float pv = (s == kNegInf) ? 0.f : exp2f(s - m_ref[i]);
                    lsum[i] += pv;
                    Pb[lane * PS + qq] = pv;
                    if (lane == 0) ab[qq] = al;
                }
            }
            bar_arrive(BAR_EMPTY + sb, kThreads);          // scores of tile jt consumed
            bar_sync(BAR_V, kKThreads);                    // p and alpha of tile jt written; V stage jt-1 free
            if (vt == 0) {
                issue_k();                                 // K stage of tile jt is free (FULL passed)
                if (jt >= 1) issue_v();                    // V stage of tile jt-1 is free (BAR_V passed)
            }
            // ------------------------------------------------ accumulate
            const int vst = jt % p.nstage_v;
            wait_stage(smem_u32(&vbar[vst]), (uint32_t)((jt / p.nstage_v) & 1), &s_abort, p.err_d);
            const uint32_t vtile = smem_u32(vring + (size_t)vst * L.vstage);
            {
                const float4 al4 = *reinterpret_cast<const float4*>(&ab[v_qq0]);
                const float alv[4] = {al4.x, al4.y, al4.z, al4.w};
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    if (alv[n] != 1.f) {
                        pm[n] *= alv[n];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o2[n][i].x *= alv[n];
                            o2[n][i].y *= alv[n];
                        }
                    }
                }
                const uint32_t pb = smem_u32(Pb);
                for (int r = v_rg < RG ? v_rg : kRows; r < ti.nr; r += RG) {
                    const uint2 dmqh = lds64(tile_addr(vtile, r, col_dm));
                    const uint2 qs = lds64(tile_addr(vtile, r, col_qs));
                    const float4 p4 = lds128f(pb + 4u * (uint32_t)(r * PS + v_qq0));
                    const float d = h2f(dmqh.x & 0xffffu);
                    const float m = h2f(dmqh.x >> 16);
                    const float d256 = d * 256.f;
                    const float mp = fmaf(-128.f, d, m);
                    const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
                    float2 pd[4];
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const float t = pr[n] * d256;
                        pd[n] = make_float2(t, t);
                        pm[n] = fmaf(pr[n], mp, pm[n]);
                    }
                    const uint32_t xl = __byte_perm(dmqh.y, 0, v_hf ? 0x1111u : 0x0000u);
                    const uint32_t xh = __byte_perm(dmqh.y, 0, v_hf ? 0x3333u : 0x2222u);
                    uint32_t u[4];
                    {
                        const uint32_t sp0 = ((xl & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp1 = (((xl >> 4) & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp2 = ((xh & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp3 = (((xh >> 4) & 0x08040201u) + 0x080C0E0Fu);
                        u[0] = (qs.x & 0x0F0F0F0Fu) | (sp0 & 0xF0F0F0F0u);
                        u[1] = (qs.y & 0x0F0F0F0Fu) | (sp1 & 0xF0F0F0F0u);
                        u[2] = ((qs.x >> 4) & 0x0F0F0F0Fu) | (sp2 & 0xF0F0F0F0u);
                        u[3] = ((qs.y >> 4) & 0x0F0F0F0Fu) | (sp3 & 0xF0F0F0F0u);
                    }
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const float2 fa = make_float2(__uint_as_float(__byte_perm(u[cc], 0x3F000000u, 0x7044u)),
                                                      __uint_as_float(__byte_perm(u[cc], 0x3F000000u, 0x7144u)));
                        const float2 fb = make_float2(__uint_as_float(__byte_perm(u[cc], 0x3F000000u, 0x7244u)),
                                                      __uint_as_float(__byte_perm(u[cc], 0x3F000000u, 0x7344u)));
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            o2[n][2 * cc] = __ffma2_rn(pd[n], fa, o2[n][2 * cc]);
                            o2[n][2 * cc + 1] = __ffma2_rn(pd[n], fb, o2[n][2 * cc + 1]);
                        }
                    }
                }
            }
            if (ti.last) {
                // row-group partial sums meet inside the warp: tree-reduce
                // down the lane groups, lane group 0 ends with the sum
                for (int st = 1; st < RG; st <<= 1) {
                    const bool take = v_rg + st < RG;
                    const int dl = st * TW;
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const float a = __shfl_down_sync(0xffffffffu, pm[n], dl);
                        if (take) pm[n] += a;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float x = __shfl_down_sync(0xffffffffu, o2[n][i].x, dl);
                            const float y = __shfl_down_sync(0xffffffffu, o2[n][i].y, dl);
                            if (take) {
                                o2[n][i].x += x;
                                o2[n][i].y += y;
                            }
                        }
                    }
                }
                if (v_rg == 0) {
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const int qi = ti.it.qs * QC + 4 * v_qg + n;
                        if (qi < p.hpk * p.T) {
                            const int t = qi / p.hpk, h = v_g * p.hpk + qi % p.hpk;
                            const long long rec = (long long)ti.it.pidx * p.Qtot + (long long)t * p.Hq + h;
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                const int dim = v_bi * 32 + 8 * v_hf + (cc & 1) * 4 + (cc >> 1) * 16;
                                *reinterpret_cast<float4*>(&p.part_o[rec * D + dim]) =
                                    make_float4(o2[n][2 * cc].x + pm[n], o2[n][2 * cc].y + pm[n],
                                                o2[n][2 * cc + 1].x + pm[n], o2[n][2 * cc + 1].y + pm[n]);
                            }
                        }
                    }
                }
                // (max, sum) of the softmax queries this warp owns
#pragma unroll
                for (int i = 0; i < NQMAX / 8; ++i) {
                    const int qq = vw + 8 * i;
                    if (qq < NQ) {
                        float l = lsum[i];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                        const int g = qq / QC, ql = qq % QC;
                        const int qi = ti.it.qs * QC + ql;
                        if (lane == 0 && qi < p.hpk * p.T) {
                            const int t = qi / p.hpk, h = g * p.hpk + qi % p.hpk;
                            const long long rec = (long long)ti.it.pidx * p.Qtot + (long long)t * p.Hq + h;
                            p.part_ml[rec * 2] = m_ref[i];
                            p.part_ml[rec * 2 + 1] = l;
                        }
                        m_ref[i] = kNegInf;
                        lsum[i] = 0.f;
                    }
                }
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    pm[n] = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
                }
            }
            advance(c, ti, p, lens, bases, prefix, n_items);
            ++jt;
        }
    }
}

template <int NBH, int NQG, int NLIMB>
cudaError_t launch_t(const SplitParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid, size_t smem,
                     cudaStream_t s) {
    auto fn = fast_kernel<NBH, NQG, NLIMB>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, s>>>(p, kmap, vmap);
    return cudaGetLastError();
}

}  // namespace

bool make_row_tensor_map(CUtensorMap* map, void* plane, int tok_bytes, long long rows) {
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
    // dims: byte within a 128-byte column block, row, column block; the last
    // block of a row may reach up to 127 bytes into the next row (or into the
    // plane padding kvq_required_bytes adds)
    const int blocks = (tok_bytes + 127) / 128;
    if (blocks > 256) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)blocks};
    const cuuint64_t strides[2] = {(cuuint64_t)tok_bytes, 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)kFastRows, (cuuint32_t)blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, plane, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_split_fast(const SplitParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                              cudaStream_t s) {
    const size_t smem = fast_layout(p, p.nlimb).total;
    const int NBH = p.D / 32, NQG = p.QC / 4;
#define KVQ_CASE(nb, nq, nl) \
    if (NBH == nb && NQG == nq && p.nlimb == nl) return launch_t<nb, nq, nl>(p, kmap, vmap, grid, smem, s);
    KVQ_CASE(1, 1, 3) KVQ_CASE(2, 1, 3) KVQ_CASE(4, 1, 3) KVQ_CASE(8, 1, 3) KVQ_CASE(16, 1, 3)
    KVQ_CASE(1, 2, 3) KVQ_CASE(2, 2, 3) KVQ_CASE(4, 2, 3) KVQ_CASE(8, 2, 3) KVQ_CASE(16, 2, 3)
    KVQ_CASE(1, 1, 2) KVQ_CASE(2, 1, 2) KVQ_CASE(4, 1, 2) KVQ_CASE(8, 1, 2) KVQ_CASE(16, 1, 2)
    KVQ_CASE(1, 2, 2) KVQ_CASE(2, 2, 2) KVQ_CASE(4, 2, 2) KVQ_CASE(8, 2, 2) KVQ_CASE(16, 2, 2)
#undef KVQ_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvq
