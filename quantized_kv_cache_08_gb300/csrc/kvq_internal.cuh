// Internal declarations shared by the kvq CUDA translation units (not part of
// the public C ABI in include/kvq.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

namespace kvq {

constexpr int kQK = 32;            // elements per quantisation block
constexpr int kQ8Bytes = 34;       // q8_0 block: fp16 d + 32 int8 codes
constexpr int kQ5Bytes = 24;       // q5_1 block: fp16 d, fp16 m, u32 qh, 16 B qs
constexpr int kF8Bytes = 32;       // 32 FP8 E4M3 elements, no scale
constexpr int kMaxIdsPerLaunch = 256;
constexpr int kSplitThreads = 256; // decode split CTA size
constexpr int kTileRows = 16;      // KV rows staged per pipeline stage
constexpr int kMinSplitRows = 64;  // smallest rows-per-split the workspace allows
constexpr int kMergeThreads = 1024;

// device error word codes
constexpr int kErrCounter = 1;     // a length/base counter was out of range
constexpr int kErrWait = 2;        // a bounded wait on an mbarrier ran out

struct SeqIds {                    // host-chosen sequence indices, by value
    int n;                         // entries in this launch
    int identity;                  // 1: entry i is sequence first + i
    int first;
    int id[kMaxIdsPerLaunch];
};

struct AppendParams {
    const void* k;                 // [n][T][Hkv][D] f32 or bf16
    const void* v;
    int bf16;
    uint8_t* k_plane;              // [B][max_rows][k_tok]
    uint8_t* v_plane;              // [B][max_rows][v_tok]
    int* len_d;                    // read for the slot, then advanced by T (the launch's last CTA)
    const int* base_d;
    int* err_d;
    int* done_d;                   // completion counter of the launch's CTAs (0 between launches)
    int T, kb, k_tok, v_tok, max_rows;
    int fp8;                       // 1: both planes hold FP8 E4M3 bytes
    long long entry_offset;        // first input entry of this launch
};

struct SplitParams {
    const uint8_t* k_plane;
    const uint8_t* v_plane;
    const int* len_d;
    const int* base_d;
    int* err_d;
    const void* q;                 // [B][T][Hq][D]
    int q_bf16;
    float qscale;                  // score scale * log2(e)
    float softcap_a, softcap_b;    // score cap in log2 units: s -> b * tanh(a * s); b == 0: off
    int B, T, Hq, Hkv, hpk, D, kb, k_tok, v_tok, max_rows, window;
    int fp8;                       // 1: both planes hold FP8 E4M3 bytes (generic kernel only)
    int C;                         // rows per split (multiple of kTileRows)
    int nqs;                       // query slices per (sequence, split)
    int QC;                        // queries per KV group per slice
    int Qtot;                      // Hq * T
    float* part_o;                 // [item][Qtot][D]
    float* part_ml;                // [item][Qtot][2]  (max in log2 units, sum)
    int* plan;                     // [B+1] split prefix, written by CTA 0
    int nstage;
    uint32_t k_stage_bytes;        // kTileRows * k_tok rounded to 128
    uint32_t stage_bytes;          // k + v stage bytes
};

__host__ __device__ inline size_t fl_round(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Raise a kernel's dynamic shared-memory limit to the device's opt-in maximum
// less its static shared memory (and, when carveout is set, prefer the
// largest shared-memory carveout) once per device: `done` holds one bit per
// device for that kernel.
template <typename F>
inline cudaError_t kernel_attrs_once(F fn, std::atomic<unsigned long long>& done, bool carveout) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int smem = 0;
    e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);              // the kernel's static shared memory counts too
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    if (carveout) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
    }
    done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

// Stream-K decode (kvq_decode_stream.cu): the visible rows of all sequences,
// repeated once per query slice, form one work space cut into G equal
// contiguous ranges, one per CTA; the part of a CTA's range inside one
// (query slice, sequence) pair is a fragment, and fragment (c, key) writes its
// partials to record slot c + key, key = slice * B + sequence.
constexpr int kStreamThreads = 512;     // 16 warps, one (KV head, 4 queries) unit and row slice each
constexpr int kStreamRows = 32;         // token rows per tile
constexpr int kStreamCtasPerSm = 1;
constexpr int kStreamMaxB = 1024;       // sequences the per-CTA tables hold
constexpr int kStreamMaxGrid = 256;     // most CTAs a decode may use (record slots are sized by it)
constexpr int kStreamShortTiles = 16;   // at most this many tiles per CTA: one row slice per tile

struct StreamParams {
    const uint8_t* k_plane;
    const uint8_t* v_plane;
    const int* len_d;
    const int* base_d;
    int* err_d;
    const void* q;                 // [B][T][Hq][D]
    int q_bf16;
    float qscale;                  // score scale * log2(e)
    float softcap_a, softcap_b;    // score cap in log2 units: s -> b * tanh(a * s); b == 0: off
    int B, T, Hq, Hkv, hpk, D, k_tok, v_tok, max_rows, window;
    int Qh;                        // queries per KV head: hpk * T
    int QPS;                       // query groups of 4 per KV head in one slice
    int nqs;                       // query slices
    int RS;                        // warps per unit (1 or 2): a tile's rows split RS ways
    int NA;                        // working warps: Hkv * QPS * RS
    int Qtot;                      // Hq * T
    int G;                         // CTAs
    int NS;                        // stages of each of the K and V rings
    uint32_t Sk, Sv;               // shared-memory row strides of the K and V stages
    int qbits;                     // 16 or 24: query quantisation
    float* part_o;                 // [slot][4 Hkv QPS][D]: the slice's queries, unit-major
    float* part_ml;                // [slot][4 Hkv QPS][2]  (max in log2 units, sum)
};

struct StreamLayout {
    size_t kst, vst, P, W, LW, SQ, CB, tabs, tinfo, bars, cnt, walk, total;
    uint32_t kstage, vstage, pwarp, wwarp, lwarp;
};

__host__ __device__ inline StreamLayout stream_layout(const StreamParams& p) {
    StreamLayout L;
    const int warps = kStreamThreads / 32;
    const int RW = kStreamRows / p.RS;
    const int NBH = p.D / 32;
    L.kstage = (uint32_t)kStreamRows * p.Sk;
    L.vstage = (uint32_t)kStreamRows * p.Sv;
    L.pwarp = (uint32_t)RW * 16;                    // [RW rows][4 queries] f32
    L.wwarp = (uint32_t)NBH * 256;                  // [block][8 pairs of pairs][4 queries][2] 16-bit pairs
    L.lwarp = p.qbits == 24 ? (uint32_t)NBH * 9 * 16 : 0u;   // [block][9 words][4 queries] low bytes
    size_t off = 0;
    L.kst = off;
    off += (size_t)p.NS * L.kstage;
    L.vst = off;
    off += (size_t)p.NS * L.vstage;
    L.P = off;
    off += (size_t)warps * L.pwarp;
    L.W = off;
    off += (size_t)warps * L.wwarp;
    L.LW = off;
    off += (size_t)warps * L.lwarp;
    L.SQ = off;
    off += (size_t)warps * 64;
    L.CB = off;                                     // two row slices: per unit [4][D] sums + 8 floats
    off += p.RS == 2 ? (size_t)(warps / 2) * (16 * (size_t)p.D + 32) : 0;
    L.tabs = off;                                   // len, base, lo, vis, prefix: 5 x (B + 1) ints
    off += fl_round((size_t)5 * (p.B + 1) * 4, 16);
    L.tinfo = off;
    off += (size_t)2 * p.NS * 16;
    L.bars = off;
    off += (size_t)2 * p.NS * 8;
    L.cnt = off;                                    // release counters and armed-phase counts
    off += fl_round((size_t)4 * p.NS * 4, 16);
    L.walk = off;
    off += 64;
    L.total = off + 128;                            // slack to align the base to 128 bytes
    return L;
}

// The layout of the E4M3 kernel: per-warp areas for the working warps only
// (1 KB token rows leave no room for idle warps' areas with three stages),
// f32 query words.  Left out of the q8_0 / q5_1 kernel's translation unit.
#if !defined(KVQ_STREAM_TU) || defined(KVQ_STREAM_F8)
__host__ __device__ inline StreamLayout stream_layout_f8(const StreamParams& p) {
    StreamLayout L;
    const int warps = p.NA;
    const int RW = kStreamRows / p.RS;
    const int NBH = p.D / 32;
    L.kstage = (uint32_t)kStreamRows * p.Sk;
    L.vstage = (uint32_t)kStreamRows * p.Sv;
    L.pwarp = (uint32_t)RW * 16;                    // [RW rows][4 queries] f32
    L.wwarp = (uint32_t)NBH * 512;                  // [block][8 code words][4 queries][4] f32
    L.lwarp = 0u;
    size_t off = 0;
    L.kst = off;
    off += (size_t)p.NS * L.kstage;
    L.vst = off;
    off += (size_t)p.NS * L.vstage;
    L.P = off;
    off += (size_t)warps * L.pwarp;
    L.W = off;
    off += (size_t)warps * L.wwarp;
    L.LW = off;
    off += (size_t)warps * L.lwarp;
    L.SQ = off;
    off += (size_t)warps * 64;
    L.CB = off;                                     // two row slices: per unit [4][D] sums + 8 floats
    off += p.RS == 2 ? (size_t)(p.NA / 2) * (16 * (size_t)p.D + 32) : 0;
    L.tabs = off;                                   // len, base, lo, vis, prefix: 5 x (B + 1) ints
    off += fl_round((size_t)5 * (p.B + 1) * 4, 16);
    L.tinfo = off;
    off += (size_t)2 * p.NS * 16;
    L.bars = off;
    off += (size_t)2 * p.NS * 8;
    L.cnt = off;                                    // release counters and armed-phase counts
    off += fl_round((size_t)4 * p.NS * 4, 16);
    L.walk = off;
    off += 64;
    L.total = off + 128;                            // slack to align the base to 128 bytes
    return L;
}
#endif

struct MergeStreamParams {
    const float* part_o;
    const float* part_ml;
    const int* len_d;              // the counters: the merge derives the visible
    const int* base_d;             // rows of each sequence as the split kernel does
    int window, max_rows;
    const float* sinks;            // [Hq] or null
    float* out;                    // [B][T][Hq][D]
    int B, T, Hq, hpk, D, Qtot, QPS, nqs, G;
    int WPQ;                       // warps per (sequence, query, dim chunk)
    int DC;                        // dims per chunk (32 * dims per lane)
};

struct MergeParams {
    const float* part_o;
    const float* part_ml;
    const int* plan;               // [B+1]
    const float* sinks;            // [Hq] or null
    float* out;                    // [B][T][Hq][D]
    int B, Hq, Qtot, D;
};

// launchers (kvq_append.cu)
// quantised append of a launch's sequences, then len_d += T for them
cudaError_t launch_append(const AppendParams& p, const SeqIds& ids, cudaStream_t s);
cudaError_t launch_set_len(int* len_d, const SeqIds& ids, const int* values, cudaStream_t s);
cudaError_t launch_ring_copy(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k,
                             uint8_t* dst_v, size_t k_bytes, size_t v_bytes, cudaStream_t s);
cudaError_t launch_set_base(int* base_d, int seq, int value, cudaStream_t s);
// one-pass ring rebase (move the live rows to physical row 0, then base_d =
// new_base) when the rows are 16-byte aligned and the live bytes fit the SMs'
// shared memory: returns false (nothing launched) otherwise; *err reports a
// failed launch
bool launch_rebase_one_pass(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                            size_t k_bytes, size_t v_bytes, int* base_d, int seq, int new_base, int* arrive,
                            int* gen, int* err_d, int num_sms, cudaStream_t s, cudaError_t* err);
// len_d[b] -= T - accept_d[b] for b < n, checked on the device (error word on failure)
cudaError_t launch_truncate_accept(int* len_d, const int* base_d, int* err_d, const int* accept_d, int n, int T,
                                   int window, int ring, cudaStream_t s);

// launchers (kvq_decode.cu)
size_t split_smem_bytes(const SplitParams& p);
int split_max_smem();
cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, int T, int max_splits, bool pdl, cudaStream_t s);

// stream-K decode (kvq_decode_stream.cu): token rows must be 16-byte multiples
// the stream-K split kernel for FP8 E4M3 rows (its own translation unit)
cudaError_t launch_split_stream_f8(const StreamParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   cudaStream_t s);
cudaError_t launch_split_stream(const StreamParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t s);
// 2-D TMA map of a byte plane of `rows` token rows of tok_bytes (a multiple of
// 16) as 8-byte elements, box = 32 rows of stride_bytes (>= tok_bytes, a
// multiple of 16, at most 2048): the box part past a token row is zero-filled
bool make_stream_map(CUtensorMap* map, void* plane, int tok_bytes, int stride_bytes, long long rows);
cudaError_t launch_merge_stream(const MergeStreamParams& p, cudaStream_t s);
int stream_max_smem();

}  // namespace kvq
