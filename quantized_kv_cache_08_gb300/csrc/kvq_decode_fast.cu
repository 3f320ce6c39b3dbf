// Warp-specialised split-K decode for caches whose token rows are 16-byte
// multiples (n_kv_heads * head_dim % 256 == 0).  Same semantics, partial
// records and merge as the generic split kernel (kvq_decode.cu):
// cortiq-engine "Struct LayerKvCache" fn attend_group_upto (window, causal
// upto, sinks, GQA) over memra-engine "Struct KvLayer" q8_0 / q5_1 rows.
//
// Persistent CTAs, one per SM.  A CTA's first work item is its block index;
// later items come from a device counter (the merge resets it), so CTAs that
// finish early take more.
//
// A CTA has 16 warps.  The key and the value bytes of a 32-row tile each
// arrive by one 3-D TMA copy (cp.async.bulk.tensor, 32 rows x all 128-byte
// column blocks, 128-byte swizzle) into its own ring of stages.  The last of
// the 8 warps that read a stage (an acquire-release shared counter decides)
// issues the copy that refills it, with the row coordinate from a small
// look-ahead table that one value thread keeps filled; that thread also
// reserves the CTA's next work item and publishes the CTA's item order, which
// the key warps follow.  No warp waits to issue copies.  Warps 0-7 (K warps)
// turn key rows into scores and run the online softmax; warps 8-15 (V warps)
// accumulate p * v_hat.  Probabilities pass from K to V warps through a ring
// of kPDepth buffers handed over with named barriers (bar.arrive / bar.sync),
// so the K warps may run up to kPDepth tiles ahead.
//
// K warps: lane = token row; a warp owns whole (KV head, query group of 4)
// units.  The swizzle puts the same 16-byte column of 8 consecutive rows in 8
// different bank groups, so the 32 lanes read their rows with conflict-free
// 16-byte loads.  The query is pre-scaled by scale * log2 e, quantised per
// (query, 32-element block) to NLIMB*8 bits against the block's largest
// magnitude and split into int8 limbs held in shared memory; every lane reads
// the same limb words (broadcast).  The next item's raw queries are staged in
// shared memory (cp.async) while the current item runs.  DP4A multiplies four
// int8 codes by four limb bytes and accumulates in int32, so the codes are
// never converted to float; per block the limb sums are combined in float and
// scaled by d_k * s_q.
// Softmax: the unit's scores of a tile sit one row per lane, so the reference
// maximum is a warp reduction.  It moves only when a score exceeds it by more
// than 8 (log2 units); a warp vote finds that rare case, otherwise
// p = 2^(s - m_ref) needs no reduction and each lane keeps a partial sum of p
// until the item ends.
// V warps: a task is (query group of 4, KV head, block, half block); a warp
// holds TW consecutive tasks and 32/TW lane groups that take interleaved
// rows, so the row partial sums reduce with warp shuffles at the end of an
// item.  The 5-bit codes are rebuilt with byte arithmetic and placed in the
// mantissa of 0.5 (value 0.5 + u/256), so v_hat = 256 d F + (m - 128 d) and
// o += (256 p d) F with packed FMAs, plus sum p (m - 128 d) per block.
#include "kvq_device.cuh"

namespace kvq {
namespace {

using namespace dev;

constexpr int kThreads = kFastThreads;
constexpr int kRows = kFastRows;
constexpr int kPDepth = kFastPDepth;           // probability buffers between K and V warps
constexpr int kKThreads = 256;                 // warps 0-7
constexpr int kKVThreads = 512;                // K and V warps
constexpr int kYRing = 16;                     // look-ahead table of tile row coordinates
constexpr int BAR_K = 1, BAR_FULL = 2, BAR_EMPTY = 2 + kPDepth, BAR_QLOAD = 2 + 2 * kPDepth,
              BAR_INIT = 3 + 2 * kPDepth;
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

// Quotient and remainder of 0 <= a < 2^20 by 1 <= b <= 1024 through a float
// reciprocal: (a + 0.5) / b lies at least 0.5 / b from an integer and the
// float product is off by less than 0.13 / b there, so truncation is exact.
__device__ __forceinline__ int qdiv(int a, int b, float inv_b, int& rem) {
    const int q = __float2int_rz(((float)a + 0.5f) * inv_b);
    rem = a - q * b;
    return q;
}

// One warp's release of a stage: an acquire-release add on the stage's
// shared-memory counter, so the warp's reads of the stage happen before a
// refill that the last releaser issues.
__device__ __forceinline__ uint32_t release_count(int* counter) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                 : "=r"(old) : "r"(smem_u32(counter)) : "memory");
    return old;
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
    int item, tile, k;             // k: the item's ordinal among this CTA's items
    Item it;
    int row0, n, base, len;
};

// Work items: a CTA's first item is blockIdx.x; later ones come from a
// device counter, so CTAs that finish early take more.  The copy look-ahead
// reserves item k + 1 of the CTA when it enters item k and publishes the
// CTA's item order in a small shared-memory queue that the K warps follow.
constexpr int kIRing = 16;

__device__ __forceinline__ int reserve_item(int* work_d, int n_items) {
    if (n_items <= (int)gridDim.x) return n_items;     // every item is in the first wave
    const int nx = (int)gridDim.x + atomicAdd(work_d, 1);
    return nx < n_items ? nx : n_items;
}

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
    c.k = 0;
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
                                        const int* bases, const int* prefix, int n_items, const int* items) {
    if (ti.last) {
        ++c.k;
        c.item = items[c.k % kIRing];
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
    constexpr int UPW = NQG;                        // units (KV head, query group) per K warp at most (Hkv <= 8)
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // swizzled TMA boxes need a 1024-byte aligned destination
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const FastLayout L = fast_layout(p, NLIMB);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.Hkv;
    const int NQ = Hkv * QC;
    const int PS = NQ + 4;                          // row stride of a probability buffer
    const float inv_hpk = 1.f / (float)p.hpk;

    uint8_t* kring = smem + L.kring;
    uint8_t* vring = smem + L.vring;
    uint32_t* qlimb = reinterpret_cast<uint32_t*>(smem + L.qlimb);
    float* qscl = reinterpret_cast<float*>(smem + L.qscale);
    uint8_t* qraw = smem + L.qraw;
    float* P = reinterpret_cast<float*>(smem + L.P);            // [kPDepth][kRows][PS]
    float* alpha = reinterpret_cast<float*>(smem + L.alpha);    // [kPDepth][NQ]
    int* qlo = reinterpret_cast<int*>(smem + L.qlo);            // [NQ] first visible row per CTA query
    int* qup = reinterpret_cast<int*>(smem + L.qup);            // [NQ] one past the last (-1: no query)
    int* lens = reinterpret_cast<int*>(smem + L.lens);
    int* bases = lens + p.B;
    int* prefix = bases + p.B;
    uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* vfull = kfull + p.nstage_k;
    __shared__ int s_abort;
    __shared__ int4 s_tinfo[kPDepth];               // per probability buffer: rows, last, query slice, record (-1 rows: end)
    __shared__ int s_y[kYRing];                     // row coordinate of tile j in the planes' maps (-1: no tile j)
    __shared__ int s_kcnt[4], s_vcnt[4];            // releases per key / value stage (8 per use)
    __shared__ int4 s_ahead;                        // the row table's cursor: next row, tiles left, item, ordinal
    __shared__ int s_items[kIRing];                 // item of this CTA's k-th work item (n_items: none)

    for (int b = tid; b < p.B; b += kThreads) {
        lens[b] = p.len_d[b];
        bases[b] = p.base_d[b];
    }
    if (tid == 0) s_abort = 0;
    __syncthreads();
    if (warp == 0) plan_splits(p, lens, bases, prefix, lane);
    if (tid == 0) {
        for (int s2 = 0; s2 < p.nstage_k; ++s2) mbar_init(smem_u32(&kfull[s2]), 1);
        for (int s2 = 0; s2 < p.nstage_v; ++s2) mbar_init(smem_u32(&vfull[s2]), 1);
        for (int s2 = 0; s2 < 4; ++s2) s_kcnt[s2] = s_vcnt[s2] = 0;
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

    const uint32_t kring_a = smem_u32(kring), vring_a = smem_u32(vring);
    const uint32_t kfull_a = smem_u32(kfull), vfull_a = smem_u32(vfull);
    const uint32_t kstage_b = (uint32_t)L.kstage, vstage_b = (uint32_t)L.vstage;
    const int nsk = p.nstage_k, nsv = p.nstage_v;
    const CUtensorMap* kmap_p = &kmap;
    const CUtensorMap* vmap_p = &vmap;
    auto issue_k = [=](int j, int y) {
        const uint32_t st = (uint32_t)(j % nsk);
        mbar_expect_tx(kfull_a + 8u * st, kstage_b);
        tma_load_rows(kring_a + st * kstage_b, kmap_p, y, kfull_a + 8u * st);
    };
    auto issue_v = [=](int j, int y) {
        const uint32_t st = (uint32_t)(j % nsv);
        mbar_expect_tx(vfull_a + 8u * st, vstage_b);
        tma_load_rows(vring_a + st * vstage_b, vmap_p, y, vfull_a + 8u * st);
    };
    // look-ahead of the row table: V thread 0 fills it, and the V warps may
    // trail the K warps by kPDepth + 1 tiles
    const int LA = max(p.nstage_k, p.nstage_v) + kPDepth + 1;

    if (warp < 8) {
        // ======================================================== K warps
        const int kt = tid;
        float m_ref[UPW][4], lsum[UPW][4];
#pragma unroll
        for (int u = 0; u < UPW; ++u)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                m_ref[u][n] = kNegInf;
                lsum[u][n] = 0.f;
            }
        const int nunit = Hkv * NQG;
        Cursor c = cursor_begin(p, lens, bases, prefix, n_items);
        int jt = 0;
        while (c.item < n_items) {
            const TileInfo ti = tile_of(c);
            if (ti.first) {
                // quantise this item's pre-scaled queries into int8 limbs: one
                // thread per 4 consecutive dims of a query, the 8 threads of a
                // 32-dim block share its largest magnitude through shuffles.
                // Later items read queries staged in shared memory during the
                // item before (cp.async), the first item reads global memory.
                const bool staged = p.q_stage && jt > 0;
                if (staged) asm volatile("cp.async.wait_all;" ::: "memory");
                bar_sync(BAR_K, kKThreads);          // previous item's scores are done; staged queries in
                const int nunits = NQ * (D / 4);
                // one unit = 4 consecutive dims of a query: scale, block maximum
                // over the unit's 8 lanes, int8 limbs and the block's scale
                auto quant_unit = [&](const float (&xs4)[4], int u, bool act) {
                    const int qq = act ? u / (D / 4) : 0, w4 = act ? u % (D / 4) : 0;
                    const int bi = w4 >> 3, k = w4 & 7;
                    const int g = qq / QC, ql = qq % QC;
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] = xs4[e] * p.qscale;
                    // the 8 threads of a 32-dim block (consecutive lanes) share its maximum
                    float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
                    for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    constexpr float QMAX = NLIMB == 3 ? 8388607.f : 32767.f;
                    // any scale works here: the dot products are rescaled by mx / QMAX
                    const float inv = mx > 0.f ? __fdividef(QMAX, mx) : 0.f;
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
                        if (k == 0) qscl[(unit * NBH + bi) * 4 + n] = mx * (1.f / QMAX);
                    }
                };
                constexpr int QB = 4;                // units per thread whose loads are in flight together
                if (staged) {
                    // queries already in shared memory (staged during the item before)
                    for (int u0 = 0; u0 < nunits; u0 += QB * kKThreads) {
                        float xs[QB][4];
#pragma unroll
                        for (int j = 0; j < QB; ++j) {
                            const int u = u0 + j * kKThreads + kt;
                            const int qq = u / (D / 4), w4 = u % (D / 4);
                            const int qi = ti.it.qs * QC + qq % QC;
#pragma unroll
                            for (int e = 0; e < 4; ++e) xs[j][e] = 0.f;
                            if (u < nunits && qi < p.hpk * p.T) {
                                if (p.q_bf16) {
                                    const uint2 raw =
                                        *reinterpret_cast<const uint2*>(qraw + ((size_t)qq * D + 4 * w4) * 2);
                                    xs[j][0] = __uint_as_float(raw.x << 16);
                                    xs[j][1] = __uint_as_float(raw.x & 0xffff0000u);
                                    xs[j][2] = __uint_as_float(raw.y << 16);
                                    xs[j][3] = __uint_as_float(raw.y & 0xffff0000u);
                                } else {
                                    const float4 f =
                                        *reinterpret_cast<const float4*>(qraw + ((size_t)qq * D + 4 * w4) * 4);
                                    xs[j][0] = f.x;
                                    xs[j][1] = f.y;
                                    xs[j][2] = f.z;
                                    xs[j][3] = f.w;
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < QB; ++j)
                            quant_unit(xs[j], u0 + j * kKThreads + kt, u0 + j * kKThreads + kt < nunits);
                    }
                } else {
                    // the CTA's first item (or staging off): queries from global memory
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
                                int hr;
                                const int t = qdiv(qi, p.hpk, inv_hpk, hr), h = g * p.hpk + hr;
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
                        // the first query loads are out, ahead of the tile stream:
                        // the value thread that starts the copies may go
                        if (jt == 0 && u0 == 0) bar_arrive(BAR_QLOAD, kKThreads + 32);
#pragma unroll
                        for (int j = 0; j < QB; ++j)
                            quant_unit(xs[j], u0 + j * kKThreads + kt, u0 + j * kKThreads + kt < nunits);
                    }
                }
                for (int qq = kt; qq < NQ; qq += kKThreads) {
                    const int qi = ti.it.qs * QC + qq % QC;
                    const bool valid = qi < p.hpk * p.T;
                    int hr;
                    const int upto = ti.len - p.T + (valid ? qdiv(qi, p.hpk, inv_hpk, hr) : 0) + 1;
                    qup[qq] = valid ? upto : -1;
                    qlo[qq] = p.window > 0 ? max(0, upto - p.window) : 0;
                }
                bar_sync(BAR_K, kKThreads);          // limbs and row windows visible to every K warp
                if (jt == 0) bar_sync(BAR_INIT, kKThreads + 32);   // the first copies and item 1 are set
                const int nx_item = s_items[(c.k + 1) % kIRing];
                if (p.q_stage && nx_item < n_items) {
                    // stage the next item's raw queries: 16-byte cp.async
                    // chunks of each query row (rows of absent queries skipped)
                    const Item nx = item_of(nx_item, prefix, p.B, p.nqs);
                    const int esz = p.q_bf16 ? 2 : 4;
                    const int cpr = D * esz / 16;    // chunks per query row
                    for (int ch = kt; ch < NQ * cpr; ch += kKThreads) {
                        const int qq = ch / cpr, k16 = ch - qq * cpr;
                        const int g = qq / QC, qi = nx.qs * QC + qq % QC;
                        if (qi < p.hpk * p.T) {
                            int hr;
                            const int t = qdiv(qi, p.hpk, inv_hpk, hr), h = g * p.hpk + hr;
                            const char* src = reinterpret_cast<const char*>(p.q) +
                                              (((long long)(nx.b * p.T + t) * p.Hq + h) * D) * esz + 16 * k16;
                            const uint32_t dst = smem_u32(qraw + ((size_t)qq * D) * esz + 16 * k16);
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
                        }
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                }
            }
            // ------------------------------------------------ scores
            const int kst = jt % p.nstage_k;
            wait_stage(smem_u32(&kfull[kst]), (uint32_t)((jt / p.nstage_k) & 1), &s_abort, p.err_d);
            const uint32_t kbase = smem_u32(kring + (size_t)kst * L.kstage);
            const uint32_t rowoff = (uint32_t)lane * 128u, sw = (uint32_t)lane & 7u;
            const int row = ti.r0 + lane;
            float sc[UPW][4];
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
                const int unit = warp + 8 * u;
#pragma unroll
                for (int n = 0; n < 4; ++n) sc[u][n] = 0.f;
                if (unit < nunit && lane < ti.nr) {
                    const int g = unit / NQG;
                    const uint32_t ql_unit = smem_u32(qlimb + (size_t)(unit * NBH) * 8 * NLIMB * 4);
                    const uint32_t qs_unit = smem_u32(qscl + (size_t)(unit * NBH) * 4);
                    head_scores_dispatch<NBH, NLIMB>(kbase, rowoff, sw, g, ql_unit, qs_unit, sc[u]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                // this warp is done with the key stage; the last of the 8 refills it
                if ((release_count(&s_kcnt[kst]) & 7) == 7) {
                    const int y = s_y[(jt + p.nstage_k) % kYRing];
                    if (y >= 0 && !*(volatile int*)&s_abort) issue_k(jt + p.nstage_k, y);
                }
            }
            // ------------------------------------------------ online softmax
            const int slot = jt % kPDepth;
            float pv[UPW][4], al[UPW][4];
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
                const int unit = warp + 8 * u;
                if (unit < nunit) {
                    const int g = unit / NQG, qg = unit - g * NQG;
                    const int qq0 = g * QC + 4 * qg;
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const bool vis = lane < ti.nr && row >= qlo[qq0 + n] && row < qup[qq0 + n];
                        const float s = vis ? sc[u][n] : kNegInf;
                        al[u][n] = 1.f;
                        if (__any_sync(0xffffffffu, s > m_ref[u][n] + kLazy)) {
                            // the reference maximum moves: full tile maximum
                            float tmax = s;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                            al[u][n] = (m_ref[u][n] == kNegInf) ? 0.f : exp2f(m_ref[u][n] - tmax);
                            m_ref[u][n] = tmax;
                            lsum[u][n] *= al[u][n];
                        }
                        pv[u][n] = (s == kNegInf) ? 0.f : exp2f(s - m_ref[u][n]);
                        lsum[u][n] += pv[u][n];
                    }
                }
            }
            if (jt >= kPDepth) bar_sync(BAR_EMPTY + slot, kKVThreads);   // V is done with tile jt - kPDepth
            float* Pb = P + slot * kRows * PS;
            float* ab = alpha + slot * NQ;
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
                const int unit = warp + 8 * u;
                if (unit < nunit) {
                    const int g = unit / NQG, qg = unit - g * NQG;
                    const int qq0 = g * QC + 4 * qg;
                    *reinterpret_cast<float4*>(&Pb[lane * PS + qq0]) = make_float4(pv[u][0], pv[u][1], pv[u][2], pv[u][3]);
                    if (lane == 0) *reinterpret_cast<float4*>(&ab[qq0]) = make_float4(al[u][0], al[u][1], al[u][2], al[u][3]);
                }
            }
            if (tid == 0) s_tinfo[slot] = make_int4(ti.nr, ti.last ? 1 : 0, ti.it.qs, ti.it.pidx);
            bar_arrive(BAR_FULL + slot, kKVThreads);       // probabilities of tile jt are in
            if (ti.last) {
                // (max, sum) of this warp's queries for the item's partial record
#pragma unroll
                for (int u = 0; u < UPW; ++u) {
                    const int unit = warp + 8 * u;
                    if (unit < nunit) {
                        const int g = unit / NQG, qg = unit - g * NQG;
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            float l = lsum[u][n];
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                            const int qi = ti.it.qs * QC + 4 * qg + n;
                            if (lane == 0 && qi < p.hpk * p.T) {
                                int hr;
                            const int t = qdiv(qi, p.hpk, inv_hpk, hr), h = g * p.hpk + hr;
                                const long long rec = (long long)ti.it.pidx * p.Qtot + (long long)t * p.Hq + h;
                                p.part_ml[rec * 2] = m_ref[u][n];
                                p.part_ml[rec * 2 + 1] = l;
                            }
                            m_ref[u][n] = kNegInf;
                            lsum[u][n] = 0.f;
                        }
                    }
                }
            }
            advance(c, ti, p, lens, bases, prefix, n_items, s_items);
            ++jt;
        }
        // copies still landing after a wait ran out must finish before the CTA ends
        if (tid == 0 && *(volatile int*)&s_abort)
            for (int j = max(0, jt - p.nstage_k); j < jt; ++j) {
                const long long t0 = clock64();
                while (!mbar_try(smem_u32(&kfull[j % p.nstage_k]), (uint32_t)((j / p.nstage_k) & 1)) &&
                       clock64() - t0 < kWaitCycles) {
                }
            }
        // end mark for the V warps, then their releases of the last tiles
        if (jt >= kPDepth) bar_sync(BAR_EMPTY + jt % kPDepth, kKVThreads);
        if (tid == 0) s_tinfo[jt % kPDepth] = make_int4(-1, 0, 0, 0);
        bar_arrive(BAR_FULL + jt % kPDepth, kKVThreads);
        for (int j = max(0, jt - kPDepth + 1); j < jt; ++j) bar_sync(BAR_EMPTY + j % kPDepth, kKVThreads);
    } else {
        // ======================================================== V warps
        const int vw = warp - 8;
        // accumulation task: TW tasks per warp (consecutive lanes), the warp's
        // 32 / TW lane groups take interleaved rows, so partial sums over rows
        // meet inside the warp and reduce with shuffles
        const int nV = 2 * NQG * Hkv * NBH;             // tasks per row
        const int TW = nV / 8;                          // tasks per warp
        const int RG = 32 / TW;                         // row groups (lane groups) per warp
        const int v_task = vw * TW + lane % TW, v_rg = lane / TW;
        const int v_hf = v_task & 1, v_bi = (v_task >> 1) % NBH, v_g = (v_task >> 1) / NBH % Hkv;
        const int v_qg = (v_task >> 1) / (NBH * Hkv);
        const int v_blk = v_g * NBH + v_bi;
        const int v_qq0 = v_g * QC + 4 * v_qg;
        const int col_dm = v_blk * kQ5Bytes;            // d, m, qh of the thread's block
        const int col_qs = col_dm + 8 + 8 * v_hf;       // its 8 bytes of qs
        // tile offsets of those bytes in the thread's first two rows (rows
        // 2 RG apart share the 128-byte swizzle phase when RG >= 4)
        const uint32_t v_o0dm = tile_addr(0, v_rg, col_dm), v_o0qs = tile_addr(0, v_rg, col_qs);
        const uint32_t v_o1dm = tile_addr(0, v_rg + RG, col_dm), v_o1qs = tile_addr(0, v_rg + RG, col_qs);
        const uint32_t v_p0 = 4u * (uint32_t)(v_rg * PS + v_qq0);
        float2 o2[4][8];
        float pm[4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            pm[n] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
        }
        if (vw == 0) {
            bar_sync(BAR_QLOAD, kKThreads + 32);
            if (lane == 0) {
                // the first query loads are out, ahead of the tile stream:
                // this thread fills the row table's first LA entries,
                // issues the first copies (tile 0's key and value first),
                // reserves item 1 after them (or when the walk reaches the
                // end of item 0) and keeps its cursor in shared memory for
                // the per-tile look-ahead below
                s_items[0] = blockIdx.x;
                bool have1 = false;
                Cursor ahead = cursor_begin(p, lens, bases, prefix, n_items);
                for (int j2 = 0; j2 < LA; ++j2) {
                    int y = -1;
                    const bool live = ahead.item < n_items;
                    TileInfo ta;
                    if (live) {
                        ta = tile_of(ahead);
                        y = ta.b * p.max_rows + (ta.r0 - ta.base);
                    }
                    s_y[j2] = y;
                    if (y >= 0 && j2 < p.nstage_k) issue_k(j2, y);
                    if (y >= 0 && j2 < p.nstage_v) issue_v(j2, y);
                    if (live) {
                        if (ta.last && ahead.k == 0) {
                            s_items[1] = reserve_item(p.work_d, n_items);
                            have1 = true;
                        }
                        const int k0 = ahead.k;
                        advance(ahead, ta, p, lens, bases, prefix, n_items, s_items);
                        if (ahead.k != k0 && ahead.item < n_items)
                            s_items[(ahead.k + 1) % kIRing] = reserve_item(p.work_d, n_items);
                    }
                }
                if (!have1) s_items[1] = reserve_item(p.work_d, n_items);
                // hand the cursor over as (next row, tiles left, item)
                int4 a = make_int4(0, 0, ahead.item, ahead.k);
                if (ahead.item < n_items) {
                    const TileInfo ta = tile_of(ahead);
                    a.x = ta.b * p.max_rows + (ta.r0 - ta.base);
                    a.y = (ahead.n - ahead.tile * kRows + kRows - 1) / kRows;
                }
                s_ahead = a;
            }
            __syncwarp();
            bar_arrive(BAR_INIT, kKThreads + 32);
        }
        int jt = 0;
        int pend_k = -1, pend_item = 0;                 // look-ahead thread: reservation not yet published
#pragma unroll 1
        for (;; ++jt) {
            const int slot = jt % kPDepth;
            bar_sync(BAR_FULL + slot, kKVThreads);         // probabilities of tile jt are in
            const int4 tinf = s_tinfo[slot];
            if (tinf.x < 0) break;                         // the K warps' end mark
            if (tid == kKThreads) {
                // row coordinate of tile jt + LA for the copy refills (the
                // barrier above orders it before the releases that read it):
                // next row, tiles left in its item; an item is decoded only
                // when the cursor enters it.  The item reserved on entering
                // an item is published one step later, off the atomic's
                // round trip.
                int4 a = s_ahead;                          // y, tiles left, item, ordinal
                if (pend_k >= 0) {
                    s_items[pend_k % kIRing] = pend_item;
                    pend_k = -1;
                }
                int y = -1;
                if (a.z < n_items) {
                    y = a.x;
                    if (a.y > 1) {
                        a.x += kRows;
                        a.y -= 1;
                    } else {
                        a.w += 1;
                        a.z = s_items[a.w % kIRing];
                        if (a.z < n_items) {
                            pend_item = reserve_item(p.work_d, n_items);
                            pend_k = a.w + 1;
                            const Item it = item_of(a.z, prefix, p.B, p.nqs);
                            const ItemRows ir = item_rows(p, lens, bases, it);
                            a.x = it.b * p.max_rows + (ir.row0 - ir.base);
                            a.y = (ir.n + kRows - 1) / kRows;
                        }
                    }
                }
                s_y[(jt + LA) % kYRing] = y;
                s_ahead = a;
            }
            const int t_nr = tinf.x, t_qs = tinf.z, t_pidx = tinf.w;
            const float* Pb = P + slot * kRows * PS;
            const float* ab = alpha + slot * NQ;
            const int vst = jt % p.nstage_v;
            wait_stage(smem_u32(&vfull[vst]), (uint32_t)((jt / p.nstage_v) & 1), &s_abort, p.err_d);
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
                // one row of the thread's task: d, m, qh and 8 qs bytes of its
                // block half, the row's 4 probabilities of its query group
                auto vrow = [&](uint32_t a_dm, uint32_t a_qs, uint32_t a_p) {
                    const uint2 dmqh = lds64(a_dm);
                    const uint2 qs = lds64(a_qs);
                    const float4 p4 = lds128f(a_p);
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
                };
                if (RG >= 4) {
                    // rows r and r + RG of the thread alternate between two
                    // swizzle phases, rows 2 RG apart share one
                    uint32_t base = vtile, pa = pb + v_p0;
                    const uint32_t pstep = 4u * (uint32_t)(RG * PS);
                    int r = v_rg;
                    for (; r + RG < t_nr; r += 2 * RG) {
                        vrow(base + v_o0dm, base + v_o0qs, pa);
                        vrow(base + v_o1dm, base + v_o1qs, pa + pstep);
                        base += (uint32_t)(2 * RG * 128);
                        pa += 2 * pstep;
                    }
                    if (r < t_nr) vrow(base + v_o0dm, base + v_o0qs, pa);
                } else {
                    for (int r = v_rg; r < t_nr; r += RG)
                        vrow(tile_addr(vtile, r, col_dm), tile_addr(vtile, r, col_qs),
                             pb + 4u * (uint32_t)(r * PS + v_qq0));
                }
            }
            __syncwarp();
            if (lane == 0) {
                // this warp is done with the value stage; the last of the 8 refills it
                if ((release_count(&s_vcnt[vst]) & 7) == 7) {
                    const int y = s_y[(jt + p.nstage_v) % kYRing];
                    if (y >= 0 && !*(volatile int*)&s_abort) issue_v(jt + p.nstage_v, y);
                }
            }
            bar_arrive(BAR_EMPTY + slot, kKVThreads);      // and with the probabilities of tile jt
            if (tinf.y) {
                // row-group partial sums meet inside the warp: butterfly over
                // the lane-group bits (TW is a power of two), one query at a
                // time; lane group 0 writes the partial and every lane restarts
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    for (int msk = TW; msk < 32; msk <<= 1) {
                        pm[n] += __shfl_xor_sync(0xffffffffu, pm[n], msk);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o2[n][i].x += __shfl_xor_sync(0xffffffffu, o2[n][i].x, msk);
                            o2[n][i].y += __shfl_xor_sync(0xffffffffu, o2[n][i].y, msk);
                        }
                    }
                    const int qi = t_qs * QC + 4 * v_qg + n;
                    if (v_rg == 0 && qi < p.hpk * p.T) {
                        int hr;
                            const int t = qdiv(qi, p.hpk, inv_hpk, hr), h = v_g * p.hpk + hr;
                        const long long rec = (long long)t_pidx * p.Qtot + (long long)t * p.Hq + h;
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int dim = v_bi * 32 + 8 * v_hf + (cc & 1) * 4 + (cc >> 1) * 16;
                            *reinterpret_cast<float4*>(&p.part_o[rec * D + dim]) =
                                make_float4(o2[n][2 * cc].x + pm[n], o2[n][2 * cc].y + pm[n],
                                            o2[n][2 * cc + 1].x + pm[n], o2[n][2 * cc + 1].y + pm[n]);
                        }
                    }
                    pm[n] = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
                }
            }
        }
        if (tid == kKThreads && *(volatile int*)&s_abort)
            for (int j = max(0, jt - p.nstage_v); j < jt; ++j) {
                const long long t0 = clock64();
                while (!mbar_try(smem_u32(&vfull[j % p.nstage_v]), (uint32_t)((j / p.nstage_v) & 1)) &&
                       clock64() - t0 < kWaitCycles) {
                }
            }
    }
}

template <int NBH, int NQG, int NLIMB>
cudaError_t launch_t(const SplitParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid, size_t smem,
                     cudaStream_t s) {
    auto fn = fast_kernel<NBH, NQG, NLIMB>;
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(fn, attrs, false);
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
