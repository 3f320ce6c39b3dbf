// Split-K flash-decode attention over the quantised cache, and its merge.
//
// Semantics (cortiq-engine "Struct LayerKvCache", fn attend_group_upto and
// fn o1_views; memra-engine "Struct KvLayer", fields len_d and base_d):
//   query row t of a T-row step sits at position s0 + t (s0 = len - T) and
//   sees logical rows [lstart_t, s0 + t + 1), lstart_t = max(0, s0+t+1-window)
//   for a windowed cache, else 0; Q head h reads KV group h / hpk; the score
//   is scale * <q, k_hat>; a sink logit joins the max and the denominator and
//   carries no value; logical row r lives at physical row r - base.
//
// Work decomposition.  The visible rows of each sequence are cut into splits
// of C rows; a work item is (sequence, split, query slice).  Persistent CTAs
// (one per SM) take items blockIdx.x, +gridDim.x, ...; the split count of
// every sequence comes from len_d on the device, so a captured launch replays
// correctly as lengths grow.  A CTA covers all KV heads of its rows, so every
// tile it stages is a contiguous byte range of each plane: one 1-D bulk TMA
// copy (cp.async.bulk) per plane per tile of 16 token rows, completing on an
// mbarrier, in a ring of `nstage` stages.
//
// Per tile:
//   K phase  one thread per (query group of 4, KV head, 32-element block):
//            32 int8 codes are turned into floats with a byte-permute into the
//            mantissa of 2^23 and one packed subtract, then packed FMAs against
//            the thread's 4 query vectors held in registers (pre-scaled by
//            scale*log2 e); partial dots are scaled by the block's d and
//            reduce-scattered over the head's blocks with warp shuffles.
//   softmax  per query: tile max, lazy rescale (the reference maximum moves
//            only when a score exceeds it by more than 8 in log2 units),
//            p = 2^(s - m), running sum.
//   V phase  one thread per (query group, KV head, block, half block): the
//            5-bit codes are rebuilt from the nibbles and qh with byte
//            arithmetic and placed into the mantissa of 0.5 (value 0.5+u/256),
//            so v_hat = 256 d * F + (m - 128 d) and o += (p*256d) F by packed
//            FMAs, with sum p*(m - 128 d) kept per block.
// FP8 E4M3 planes (memra-engine "Module cache", kv_fp8_on: K/V held in e4m3)
// take the same phases with one byte per element and no block fields: a byte
// moved into the sign, exponent and top fraction bits of a binary16 value is
// the E4M3 value times 2^-8 (the exponent biases are 15 and 7, and subnormals
// line up too), so both phases convert bytes in pairs through half2 and fold
// the 2^8 into the key score and the value weight.
// At the end of an item the V row groups are summed through shared memory and
// the partial (max, sum, o[D]) of every query is written out; the merge
// kernel combines the partials of a sequence with the sink by log-sum-exp.
#include "kvq_device.cuh"

namespace kvq {
namespace {

using namespace dev;

// Soft-capped score in log2 units: with s = scale * <q, k> * log2(e) and
// cap c, c * tanh(s' / c) on the natural-log score s' is b * tanh(a * s)
// with a = 1 / (c log2 e), b = c log2 e (b == 0: no cap).
__device__ __forceinline__ float softcap_score(const SplitParams& p, float s) {
    if (p.softcap_b > 0.f) s = p.softcap_b * tanhf(p.softcap_a * s);
    return s;
}

// Four E4M3 bytes of a little-endian word (elements 0..3) as floats scaled by
// 2^-8: byte b becomes the binary16 bits (b & 0x80) << 8 | (b & 0x7f) << 7.
__device__ __forceinline__ void e4m3x4_scaled(uint32_t w, float2& f01, float2& f23) {
    const uint32_t lo = __byte_perm(w, 0, 0x4140);   // byte 0 | byte 1 << 16
    const uint32_t hi = __byte_perm(w, 0, 0x4342);   // byte 2 | byte 3 << 16
    __half2_raw a, b;
    const uint32_t ha = ((lo << 8) & 0x80008000u) | ((lo << 7) & 0x3F803F80u);
    const uint32_t hb = ((hi << 8) & 0x80008000u) | ((hi << 7) & 0x3F803F80u);
    a.x = (unsigned short)(ha & 0xffffu);
    a.y = (unsigned short)(ha >> 16);
    b.x = (unsigned short)(hb & 0xffffu);
    b.y = (unsigned short)(hb >> 16);
    f01 = __half22float2(__half2(a));
    f23 = __half22float2(__half2(b));
}

// ------------------------------------------------------------ the kernel

template <int NBH, int NQG, bool F8>
__global__ void __launch_bounds__(kSplitThreads, 1) split_kernel(const SplitParams p) {
    constexpr int QC = 4 * NQG;                    // queries per KV group per slice
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int Hkv = p.Hkv;
    const int NQ = Hkv * QC;                       // CTA queries
    const int nK = NQG * Hkv * NBH;                // K tasks per row
    const int nV = 2 * nK;                         // V tasks per row
    const int rpK = kSplitThreads / nK;            // rows per K pass
    const int rpV = kSplitThreads / nV;            // rows per V pass

    // ---- shared memory carve-up
    uint8_t* stages = smem;
    size_t off = (size_t)p.nstage * p.stage_bytes;
    float* S = reinterpret_cast<float*>(smem + off);          // [2][kTileRows][NQ]
    off += sizeof(float) * 2 * kTileRows * NQ;
    float* m_run = reinterpret_cast<float*>(smem + off);
    off += sizeof(float) * NQ;
    float* l_run = reinterpret_cast<float*>(smem + off);
    off += sizeof(float) * NQ;
    float* alpha = reinterpret_cast<float*>(smem + off);
    off += sizeof(float) * NQ;
    float* red = reinterpret_cast<float*>(smem + off);        // [rpV-1][NQ][NBH*32]
    off += sizeof(float) * (size_t)(rpV - 1) * NQ * NBH * 32;
    int* lens = reinterpret_cast<int*>(smem + off);
    off += sizeof(int) * p.B;
    int* bases = reinterpret_cast<int*>(smem + off);
    off += sizeof(int) * p.B;
    int* prefix = reinterpret_cast<int*>(smem + off);         // [B+1]
    off += sizeof(int) * (p.B + 1);
    off = (off + 7) & ~size_t(7);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off);
    __shared__ int s_abort;

    // ---- plan: per-sequence split counts from the device lengths
    for (int b = tid; b < p.B; b += kSplitThreads) {
        lens[b] = p.len_d[b];
        bases[b] = p.base_d[b];
    }
    if (tid == 0) s_abort = 0;
    __syncthreads();
    if (tid < 32) plan_splits(p, lens, bases, prefix, tid);
    if (tid == 0) {
        for (int s = 0; s < p.nstage; ++s) mbar_init(smem_u32(&bars[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < NQ; i += kSplitThreads) {
        m_run[i] = kNegInf;
        l_run[i] = 0.f;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int b = tid; b <= p.B; b += kSplitThreads) p.plan[b] = prefix[b];
    const int n_items = prefix[p.B] * p.nqs;
    // let the merge grid launch now; it waits (griddepcontrol.wait) for this
    // grid to complete before reading any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x >= n_items) return;

    // ---- producer state (thread 0 only): next tile to issue
    int pr_item = blockIdx.x, pr_tile = 0;
    int issued = 0;
    auto issue_next = [&]() {
        if (pr_item >= n_items) return;
        const Item it = item_of(pr_item, prefix, p.B, p.nqs);
        const ItemRows ir = item_rows(p, lens, bases, it);
        const int r0 = ir.row0 + pr_tile * kTileRows;
        const int nr = min(kTileRows, ir.row0 + ir.n - r0);
        const int st = issued % p.nstage;
        const uint32_t bar = smem_u32(&bars[st]);
        // copy the 16-byte aligned superset of the rows' bytes; the tile then
        // starts (start mod 16) bytes into the stage
        const long long prow = (long long)it.b * p.max_rows + (r0 - ir.base);
        const long long ks = prow * p.k_tok, vs = prow * p.v_tok;
        const long long ks16 = ks & ~15LL, vs16 = vs & ~15LL;
        const uint32_t kb = (uint32_t)(((ks + (long long)nr * p.k_tok + 15) & ~15LL) - ks16);
        const uint32_t vb = (uint32_t)(((vs + (long long)nr * p.v_tok + 15) & ~15LL) - vs16);
        mbar_expect_tx(bar, kb + vb);
        uint8_t* dst = stages + (size_t)st * p.stage_bytes;
        bulk_g2s(smem_u32(dst), p.k_plane + ks16, kb, bar);
        bulk_g2s(smem_u32(dst + p.k_stage_bytes), p.v_plane + vs16, vb, bar);
        ++issued;
        if (++pr_tile * kTileRows >= ir.n) {
            pr_tile = 0;
            pr_item += gridDim.x;
        }
    };
    if (tid == 0)
        for (int s = 0; s < p.nstage - 1; ++s) issue_next();

    // ---- thread roles
    // K task: (qg, g, bi) with bi fastest
    const bool k_active = tid < rpK * nK;
    const int k_rg = tid / nK, k_task = tid % nK;
    const int k_bi = k_task % NBH, k_g = (k_task / NBH) % Hkv, k_qg = k_task / (NBH * Hkv);
    const int k_blk = k_g * NBH + k_bi;
    // V task: (qg, g, bi, half) with half fastest
    const bool v_active = tid < rpV * nV;
    const int v_rg = tid / nV, v_task = tid % nV;
    const int v_hf = v_task & 1, v_bi = (v_task >> 1) % NBH, v_g = (v_task >> 1) / NBH % Hkv;
    const int v_qg = (v_task >> 1) / (NBH * Hkv);
    const int v_blk = v_g * NBH + v_bi;
    const int v_qq0 = v_g * QC + 4 * v_qg;          // first of the thread's 4 CTA queries

    float2 qv[4][16];                               // K thread: 4 queries x 32 dims
    float2 o2[4][8];                                // V thread: 4 queries x 16 dims
    float pm[4];                                    // V thread: sum p*(m - 128 d)
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        pm[n] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
    }

    int tile_ctr = 0;                               // tiles consumed by this CTA
    for (int item_idx = blockIdx.x; item_idx < n_items; item_idx += gridDim.x) {
        const Item it = item_of(item_idx, prefix, p.B, p.nqs);
        const ItemRows ir = item_rows(p, lens, bases, it);
        const int s0 = ir.len - p.T;

        // K thread: load its 4 query vectors (32 dims of block k_bi), pre-scaled
        int kq_upto[4], kq_lo[4];
        if (k_active) {
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int qi = it.qs * QC + 4 * k_qg + n;
                const bool valid = qi < p.hpk * p.T;
                const int t = valid ? qi / p.hpk : 0;
                const int h = k_g * p.hpk + (valid ? qi % p.hpk : 0);
                const long long base = ((long long)(it.b * p.T + t) * p.Hq + h) * p.D + k_bi * 32;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a = 0.f, c = 0.f;
                    if (valid) {
                        a = load_q(p.q, base + 2 * i, p.q_bf16) * p.qscale;
                        c = load_q(p.q, base + 2 * i + 1, p.q_bf16) * p.qscale;
                    }
                    qv[n][i] = make_float2(a, c);
                }
                const int upto = s0 + t + 1;
                kq_upto[n] = valid ? upto : -1;     // invalid slot: no row visible
                kq_lo[n] = p.window > 0 ? max(0, upto - p.window) : 0;
            }
        }

        const int n_tiles = (ir.n + kTileRows - 1) / kTileRows;
        for (int tl = 0; tl < n_tiles; ++tl, ++tile_ctr) {
            const int st = tile_ctr % p.nstage;
            const uint32_t sbase = smem_u32(stages + (size_t)st * p.stage_bytes);
            const int r0 = ir.row0 + tl * kTileRows;
            const long long prow = (long long)it.b * p.max_rows + (r0 - ir.base);
            const uint32_t ktile = sbase + (uint32_t)((prow * p.k_tok) & 15);
            const uint32_t vtile = sbase + p.k_stage_bytes + (uint32_t)((prow * p.v_tok) & 15);
            const int nr = min(kTileRows, ir.row0 + ir.n - r0);
            float* Sb = S + (tile_ctr & 1) * kTileRows * NQ;

            if (!mbar_wait(smem_u32(&bars[st]), (uint32_t)((tile_ctr / p.nstage) & 1))) {
                atomicExch(p.err_d, kErrWait);
                s_abort = 1;
            }

            // ------------------------------------------------ K phase
            if (k_active) {
                const int iters = (kTileRows + rpK - 1) / rpK;
                for (int k = 0; k < iters; ++k) {
                    const int r = k_rg + k * rpK;
                    float sc[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (F8) {
                        if (r < nr) {
                            // 32 bytes of the block, 16-byte aligned (k_tok is a multiple of 32)
                            const uint32_t a = ktile + (uint32_t)(r * p.k_tok + k_blk * kF8Bytes);
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint2 t = lds64(a + 8 * i);
                                w[2 * i] = t.x;
                                w[2 * i + 1] = t.y;
                            }
                            float2 acc[4];
#pragma unroll
                            for (int n = 0; n < 4; ++n) acc[n] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                float2 f01, f23;
                                e4m3x4_scaled(w[i], f01, f23);
#pragma unroll
                                for (int n = 0; n < 4; ++n) {
                                    acc[n] = __ffma2_rn(qv[n][2 * i], f01, acc[n]);
                                    acc[n] = __ffma2_rn(qv[n][2 * i + 1], f23, acc[n]);
                                }
                            }
#pragma unroll
                            for (int n = 0; n < 4; ++n) sc[n] = (acc[n].x + acc[n].y) * 256.f;
                        }
                    } else if (r < nr) {
                        const uint32_t a = ktile + (uint32_t)(r * p.k_tok + k_blk * kQ8Bytes);
                        const uint32_t a0 = a & ~3u;
                        const bool odd = (a & 2u) != 0;          // block starts at 2 mod 4
                        uint32_t w[9];
#pragma unroll
                        for (int i = 0; i < 9; ++i) w[i] = lds32(a0 + 4 * i);
                        const float d = h2f(odd ? (w[0] >> 16) : (w[0] & 0xffffu));
                        const uint32_t sel = odd ? 0x7654u : 0x5432u;
                        float2 acc[4];
#pragma unroll
                        for (int n = 0; n < 4; ++n) acc[n] = make_float2(0.f, 0.f);
                        const float2 bias = make_float2(-8388736.f, -8388736.f);  // 2^23 + 128
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t cw = __byte_perm(w[i], w[i + 1], sel) ^ 0x80808080u;
                            const float2 f01 = __fadd2_rn(
                                make_float2(__uint_as_float(__byte_perm(cw, 0x4B000000u, 0x7440u)),
                                            __uint_as_float(__byte_perm(cw, 0x4B000000u, 0x7441u))),
                                bias);
                            const float2 f23 = __fadd2_rn(
                                make_float2(__uint_as_float(__byte_perm(cw, 0x4B000000u, 0x7442u)),
                                            __uint_as_float(__byte_perm(cw, 0x4B000000u, 0x7443u))),
                                bias);
#pragma unroll
                            for (int n = 0; n < 4; ++n) {
                                acc[n] = __ffma2_rn(qv[n][2 * i], f01, acc[n]);
                                acc[n] = __ffma2_rn(qv[n][2 * i + 1], f23, acc[n]);
                            }
                        }
#pragma unroll
                        for (int n = 0; n < 4; ++n) sc[n] = (acc[n].x + acc[n].y) * d;
                    }
                    // reduce-scatter over the NBH blocks of the head (lanes k_bi)
                    float res[4];
                    int nres = 4, qsel0 = 0;
                    if constexpr (NBH == 1) {
#pragma unroll
                        for (int n = 0; n < 4; ++n) res[n] = sc[n];
                    } else {
                        const unsigned FULL = 0xffffffffu;
                        const int mA = NBH / 2;
                        const bool hA = (k_bi & mA) != 0;
                        const float s0a = hA ? sc[0] : sc[2], s1a = hA ? sc[1] : sc[3];
                        const float k0a = hA ? sc[2] : sc[0], k1a = hA ? sc[3] : sc[1];
                        const float w0 = k0a + __shfl_xor_sync(FULL, s0a, mA);
                        const float w1 = k1a + __shfl_xor_sync(FULL, s1a, mA);
                        qsel0 = hA ? 2 : 0;
                        if constexpr (NBH == 2) {
                            res[0] = w0;
                            res[1] = w1;
                            nres = 2;
                        } else {
                            const int mB = NBH / 4;
                            const bool hB = (k_bi & mB) != 0;
                            float x = (hB ? w1 : w0) + __shfl_xor_sync(FULL, hB ? w0 : w1, mB);
#pragma unroll
                            for (int m = NBH / 8; m >= 1; m >>= 1) x += __shfl_xor_sync(FULL, x, m);
                            res[0] = x;
                            nres = 1;
                            qsel0 += hB ? 1 : 0;
                        }
                    }
                    const bool writer = (NBH < 8) || ((k_bi & (NBH / 4 - 1)) == 0);
                    if (r < nr && writer) {
                        const int row = r0 + r;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (j < nres) {
                                const int n = qsel0 + j;
                                int lo_n = kq_lo[0], up_n = kq_upto[0];
#pragma unroll
                                for (int m2 = 1; m2 < 4; ++m2)
                                    if (n == m2) {
                                        lo_n = kq_lo[m2];
                                        up_n = kq_upto[m2];
                                    }
                                const bool vis = row >= lo_n && row < up_n;
                                Sb[r * NQ + k_g * QC + 4 * k_qg + n] = vis ? softcap_score(p, res[j]) : kNegInf;
                            }
                        }
                    }
                }
            }
            // invalid rows of a partial tile
            if (nr < kTileRows)
                for (int i = tid; i < (kTileRows - nr) * NQ; i += kSplitThreads) Sb[nr * NQ + i] = kNegInf;
            __syncthreads();                                        // (A)
            if (s_abort) break;
            if (tid == 0) issue_next();                             // stage of the previous tile is free

            // ------------------------------------------------ online softmax
            for (int qq0 = 0; qq0 < NQ; qq0 += kSplitThreads / kTileRows) {
                const int qq = qq0 + tid / kTileRows;
                const int r = tid % kTileRows;
                const bool act = qq < NQ;
                const float s = act ? Sb[r * NQ + qq] : kNegInf;
                float tmax = s;
#pragma unroll
                for (int o = kTileRows / 2; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                const float mo = act ? m_run[qq] : kNegInf;
                float mn = mo, al = 1.f;
                if (tmax > mo + kLazy || (mo == kNegInf && tmax != kNegInf)) {
                    mn = tmax;
                    al = (mo == kNegInf) ? 0.f : exp2f(mo - mn);
                }
                const float pv = (s == kNegInf) ? 0.f : exp2f(s - mn);
                float sum = pv;
#pragma unroll
                for (int o = kTileRows / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (act) {
                    Sb[r * NQ + qq] = pv;
                    if (r == 0) {
                        m_run[qq] = mn;
                        l_run[qq] = l_run[qq] * al + sum;
                        alpha[qq] = al;
                    }
                }
            }
            __syncthreads();                                        // (B)

            // ------------------------------------------------ V phase
            if (v_active) {
                const float4 al4 = *reinterpret_cast<const float4*>(&alpha[v_qq0]);
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
                const uint32_t sb = smem_u32(Sb);
                if constexpr (F8) {
                    // dims 8hf..8hf+7 and 16+8hf..16+8hf+7 of the block, as in the q5_1 case
                    for (int r = v_rg; r < nr; r += rpV) {
                        const uint32_t vb = vtile + (uint32_t)(r * p.v_tok + v_blk * kF8Bytes + 8 * v_hf);
                        const uint2 x0 = lds64(vb);
                        const uint2 x1 = lds64(vb + 16);
                        const float4 p4 = lds128f(sb + 4u * (uint32_t)(r * NQ + v_qq0));
                        const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
                        const uint32_t u[4] = {x0.x, x0.y, x1.x, x1.y};
                        float2 pd[4];
#pragma unroll
                        for (int n = 0; n < 4; ++n) pd[n] = make_float2(pr[n] * 256.f, pr[n] * 256.f);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float2 fa, fb;
                            e4m3x4_scaled(u[c], fa, fb);
#pragma unroll
                            for (int n = 0; n < 4; ++n) {
                                o2[n][2 * c] = __ffma2_rn(pd[n], fa, o2[n][2 * c]);
                                o2[n][2 * c + 1] = __ffma2_rn(pd[n], fb, o2[n][2 * c + 1]);
                            }
                        }
                    }
                } else
                for (int r = v_rg; r < nr; r += rpV) {
                    const uint32_t vb = vtile + (uint32_t)(r * p.v_tok + v_blk * kQ5Bytes);
                    const uint2 dmqh = lds64(vb);
                    const uint2 qs = lds64(vb + 8 + 8 * v_hf);
                    const float4 p4 = lds128f(sb + 4u * (uint32_t)(r * NQ + v_qq0));
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
                    // 5-bit codes: nibbles from qs, bit 4 from qh
                    const uint32_t xl = __byte_perm(dmqh.y, 0, v_hf ? 0x1111u : 0x0000u);  // qh byte for dims lo
                    const uint32_t xh = __byte_perm(dmqh.y, 0, v_hf ? 0x3333u : 0x2222u);  // qh byte for dims +16
                    uint32_t u[4];
                    {
                        const uint32_t sp0 = ((xl & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp1 = (((xl >> 4) & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp2 = ((xh & 0x08040201u) + 0x080C0E0Fu);
                        const uint32_t sp3 = (((xh >> 4) & 0x08040201u) + 0x080C0E0Fu);
                        u[0] = (qs.x & 0x0F0F0F0Fu) | (sp0 & 0xF0F0F0F0u);          // dims j0..j0+3
                        u[1] = (qs.y & 0x0F0F0F0Fu) | (sp1 & 0xF0F0F0F0u);          // dims j0+4..j0+7
                        u[2] = ((qs.x >> 4) & 0x0F0F0F0Fu) | (sp2 & 0xF0F0F0F0u);   // dims j0+16..
                        u[3] = ((qs.y >> 4) & 0x0F0F0F0Fu) | (sp3 & 0xF0F0F0F0u);   // dims j0+20..
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float2 fa = make_float2(__uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7044u)),
                                                      __uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7144u)));
                        const float2 fb = make_float2(__uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7244u)),
                                                      __uint_as_float(__byte_perm(u[c], 0x3F000000u, 0x7344u)));
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            o2[n][2 * c] = __ffma2_rn(pd[n], fa, o2[n][2 * c]);
                            o2[n][2 * c + 1] = __ffma2_rn(pd[n], fb, o2[n][2 * c + 1]);
                        }
                    }
                }
            }
        }
        if (s_abort) break;

        // ---------------------------------------------------- finalize item
        __syncthreads();                                            // (C)
        const int Dh = NBH * 32;
        // thread dims: c in 0..3 covers 4 dims: base j0 = 8*hf (+4 for c odd, +16 for c >= 2)
        if (v_active && v_rg > 0) {
            float* dst = red + (size_t)(v_rg - 1) * NQ * Dh;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int qq = v_qq0 + n;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int dim = v_bi * 32 + 8 * v_hf + (c & 1) * 4 + (c >> 1) * 16;
                    float4 val = make_float4(o2[n][2 * c].x + pm[n], o2[n][2 * c].y + pm[n],
                                             o2[n][2 * c + 1].x + pm[n], o2[n][2 * c + 1].y + pm[n]);
                    *reinterpret_cast<float4*>(&dst[(size_t)qq * Dh + dim]) = val;
                }
            }
        }
        __syncthreads();                                            // (D)
        if (v_active && v_rg == 0) {
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int qq = v_qq0 + n;
                const int qi = it.qs * QC + 4 * v_qg + n;
                const bool valid = qi < p.hpk * p.T;
                const int t = valid ? qi / p.hpk : 0;
                const int h = v_g * p.hpk + (valid ? qi % p.hpk : 0);
                const long long rec = (long long)it.pidx * p.Qtot + (long long)t * p.Hq + h;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int dim = v_bi * 32 + 8 * v_hf + (c & 1) * 4 + (c >> 1) * 16;
                    float4 val = make_float4(o2[n][2 * c].x + pm[n], o2[n][2 * c].y + pm[n],
                                             o2[n][2 * c + 1].x + pm[n], o2[n][2 * c + 1].y + pm[n]);
                    for (int g2 = 0; g2 < rpV - 1; ++g2) {
                        const float4 o = *reinterpret_cast<const float4*>(&red[((size_t)g2 * NQ + qq) * Dh + dim]);
                        val.x += o.x;
                        val.y += o.y;
                        val.z += o.z;
                        val.w += o.w;
                    }
                    if (valid) *reinterpret_cast<float4*>(&p.part_o[rec * p.D + dim]) = val;
                }
                if (valid && v_bi == 0 && v_hf == 0) {
                    p.part_ml[rec * 2] = m_run[qq];
                    p.part_ml[rec * 2 + 1] = l_run[qq];
                }
            }
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            pm[n] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) o2[n][i] = make_float2(0.f, 0.f);
        }
        __syncthreads();                                            // (E)
        for (int i = tid; i < NQ; i += kSplitThreads) {
            m_run[i] = kNegInf;
            l_run[i] = 0.f;
        }
        // the next item's first tile writes S only after its K phase; m_run
        // is read after barrier (A), which orders this reset before it
    }

    if (s_abort && tid == 0) {
        // drain copies still in flight into this CTA's shared memory
        for (int s = 0; s < p.nstage; ++s) mbar_wait(smem_u32(&bars[s]), 0), mbar_wait(smem_u32(&bars[s]), 1);
    }
}

// Merge the partials of one (sequence, query) over its splits, with the sink:
// M = max(sink, m_s), L = 2^(sink-M) + sum l_s 2^(m_s-M), out = sum o_s 2^(m_s-M) / L
// (all in log2 units).  CTA = (group of QPB query records, sequence); its
// warps are QPB x SW: warp (qi, sg) folds splits sg, sg + SW, ... of query qi
// into a running (max, sum, o) with U splits' loads in flight, each lane
// holding VPL = D/32 consecutive dims (one vector load per split); the SW
// warp states of a query are then combined once through shared memory.
// largest merge CTA for VPL values per lane (registers: U splits of VPL in flight)
__host__ __device__ constexpr int merge_threads(int vpl) { return vpl <= 2 ? kMergeThreads : vpl <= 8 ? 512 : 256; }

template <int VPL, int U>
__global__ void __launch_bounds__(merge_threads(VPL)) merge_kernel(const MergeParams p, int QPB, int SW) {
    // U: splits whose loads are in flight together in a warp
    extern __shared__ float msm[];                  // [QPB][SW][2 + D]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qi = warp % QPB, sg = warp / QPB;
    const int gq = blockIdx.x * QPB + qi;           // t * Hq + h
    const int b = blockIdx.y;
    const int D = VPL * 32;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool live = gq < p.Qtot;
    const int first = p.plan[b];
    const int ns = live ? p.plan[b + 1] - first : 0;
    const float* ml = p.part_ml + ((long long)first * p.Qtot + gq) * 2;
    const float* po = p.part_o + ((long long)first * p.Qtot + gq) * D + lane * VPL;
    const long long rs = (long long)p.Qtot;        // record stride between splits
    float M = kNegInf, L = 0.f, acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
    for (int s0 = sg; s0 < ns; s0 += U * SW) {
        float m4[U], l4[U], o4[U][VPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * SW;
            const bool ok = s < ns;
            const float2 mlv = ok ? *reinterpret_cast<const float2*>(ml + s * rs * 2) : make_float2(kNegInf, 0.f);
            m4[u] = mlv.x;
            l4[u] = mlv.y;
            const float* src = po + s * rs * D;
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
        // the round's maximum first, then independent weights: one rescale
        // of the running state per round instead of a chain per split
        float Mr = M;
#pragma unroll
        for (int u = 0; u < U; ++u) Mr = fmaxf(Mr, m4[u]);
        if (Mr == kNegInf) continue;                // nothing visible in this round
        const float a = (M == kNegInf) ? 0.f : exp2f(M - Mr);
        L *= a;
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[v] *= a;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float w = (m4[u] == kNegInf) ? 0.f : exp2f(m4[u] - Mr);
            L = fmaf(l4[u], w, L);
#pragma unroll
            for (int v = 0; v < VPL; ++v) acc[v] = fmaf(o4[u][v], w, acc[v]);
        }
        M = Mr;
    }
    float* st = msm + (size_t)(qi * SW + sg) * (2 + D);
    if (lane == 0) {
        st[0] = M;
        st[1] = L;
    }
#pragma unroll
    for (int v = 0; v < VPL; ++v) st[2 + lane * VPL + v] = acc[v];
    __syncthreads();
    if (sg == 0 && live) {
        const float LOG2E = 1.4426950408889634f;
        const float sink = p.sinks ? p.sinks[gq % p.Hq] * LOG2E : kNegInf;
        const float* q0 = msm + (size_t)qi * SW * (2 + D);
        float Mt = sink;
#pragma unroll 8
        for (int w = 0; w < SW; ++w) Mt = fmaxf(Mt, q0[w * (2 + D)]);
        float Lt = (sink == kNegInf) ? 0.f : exp2f(sink - Mt);
        float At[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) At[v] = 0.f;
#pragma unroll 4
        for (int w = 0; w < SW; ++w) {
            const float* e = q0 + w * (2 + D);
            if (e[0] == kNegInf) continue;
            const float f = exp2f(e[0] - Mt);
            Lt += e[1] * f;
#pragma unroll
            for (int v = 0; v < VPL; ++v) At[v] += e[2 + lane * VPL + v] * f;
        }
        float* dst = p.out + (((long long)b * p.Qtot) + gq) * D + lane * VPL;
#pragma unroll
        for (int v = 0; v < VPL; ++v) dst[v] = At[v] / Lt;
    }
}

template <int NBH, int NQG, bool F8>
cudaError_t launch_split_t(const SplitParams& p, int grid, size_t smem, cudaStream_t s) {
    auto fn = split_kernel<NBH, NQG, F8>;
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(fn, attrs, false);
    if (e != cudaSuccess) return e;
    fn<<<grid, kSplitThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t split_smem_bytes(const SplitParams& p) {
    const int NQ = p.Hkv * p.QC;
    const int NBH = p.D / 32;
    const int nV = 2 * (p.QC / 4) * p.Hkv * NBH;
    const int rpV = kSplitThreads / nV;
    size_t off = (size_t)p.nstage * p.stage_bytes;
    off += sizeof(float) * 2 * kTileRows * NQ;
    off += sizeof(float) * 3 * NQ;
    off += sizeof(float) * (size_t)(rpV - 1) * NQ * p.D;
    off += sizeof(int) * (3 * (size_t)p.B + 1);
    off = (off + 7) & ~size_t(7);
    off += 8 * (size_t)p.nstage;
    return off;
}

int split_max_smem() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return v - 1024;  // static shared variables
}

cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t s) {
    const size_t smem = split_smem_bytes(p);
    const int NBH = p.D / 32, NQG = p.QC / 4;
#define KVQ_CASE(nb, nq)                                                                        \
    if (NBH == nb && NQG == nq)                                                                 \
        return p.fp8 ? launch_split_t<nb, nq, true>(p, grid, smem, s) : launch_split_t<nb, nq, false>(p, grid, smem, s);
    KVQ_CASE(1, 1) KVQ_CASE(2, 1) KVQ_CASE(4, 1) KVQ_CASE(8, 1) KVQ_CASE(16, 1)
    KVQ_CASE(1, 2) KVQ_CASE(2, 2) KVQ_CASE(4, 2) KVQ_CASE(8, 2) KVQ_CASE(16, 2)
#undef KVQ_CASE
    return cudaErrorInvalidValue;
}

template <int VPL, int U>
cudaError_t launch_merge_t(const MergeParams& p, int max_splits, bool pdl, cudaStream_t s) {
    // split warps per query: enough that each folds about four splits, up
    // to a whole CTA; queries per CTA fill the remaining warps
    constexpr int NW = merge_threads(VPL) / 32;
    int SW = 1;
    while (SW < NW && SW * 4 < max_splits) SW *= 2;
    int QPB = 1;
    while (QPB * 2 * SW <= NW && QPB * 2 <= p.Qtot) QPB *= 2;
    const size_t smem = (size_t)QPB * SW * (2 + VPL * 32) * sizeof(float);
    auto fn = merge_kernel<VPL, U>;
    // same shared-memory carveout as the split kernels, so merge CTAs launched
    // early (programmatic dependent launch) can wait beside the split CTAs
    static std::atomic<unsigned long long> attrs{0};
    cudaError_t e = kernel_attrs_once(fn, attrs, true);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.Qtot + QPB - 1) / QPB), (unsigned)p.B, 1);
    cfg.blockDim = dim3((unsigned)(32 * QPB * SW));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, fn, p, QPB, SW);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, int T, int max_splits, bool pdl, cudaStream_t s) {
    (void)T;
    // twice the loads in flight when one warp folds more than 8 splits, so
    // every split's record is requested in the first round (head_dim 128 or
    // 256; smaller heads run 32 warps a CTA)
    const bool deep = max_splits > 8 * (merge_threads(p.D / 32) / 32);
    switch (p.D / 32) {
        case 1: return launch_merge_t<1, 8>(p, max_splits, pdl, s);    // 32 warps: 256 splits a round
        case 2: return launch_merge_t<2, 8>(p, max_splits, pdl, s);
        case 4: return deep ? launch_merge_t<4, 16>(p, max_splits, pdl, s) : launch_merge_t<4, 8>(p, max_splits, pdl, s);
        case 8: return deep ? launch_merge_t<8, 8>(p, max_splits, pdl, s) : launch_merge_t<8, 4>(p, max_splits, pdl, s);
        case 16: return launch_merge_t<16, 4>(p, max_splits, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq
