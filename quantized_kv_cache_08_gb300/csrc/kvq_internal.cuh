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
constexpr int kFastThreads = 512;  // warp-specialised decode CTA size
constexpr int kFastRows = 32;      // rows per tile of the warp-specialised decode
constexpr int kFastPDepth = 4;     // probability buffers between its key and value warps

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
    const int* len_d;
    const int* base_d;
    int* err_d;
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
    int* work_d;                   // work items handed out past the first wave (reset by the merge)
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
    // warp-specialised kernel only
    int nstage_k, nstage_v;        // depths of the K and V stage rings
    uint32_t k_row_stride;         // (generic layout only) stride of a staged key row
    int k_boxes;                   // 128-byte column blocks per key row
    int v_boxes;                   // 128-byte column blocks per value row
    int nlimb;                     // int8 limbs per quantised query element (2 or 3)
    int q_stage;                   // 1: stage the next item's queries in shared memory (cp.async)
};

// Shared-memory layout of the warp-specialised decode kernel (host and device).
struct FastLayout {
    size_t kstage, vstage, kring, vring, qlimb, qscale, qraw, P, alpha, qlo, qup, lens, bars, total;
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

__host__ __device__ inline FastLayout fast_layout(const SplitParams& p, int nlimb) {
    FastLayout L;
    const size_t NQ = (size_t)p.Hkv * p.QC;
    const size_t NBH = (size_t)p.D / 32;
    // key tiles: k_boxes swizzled boxes of kFastRows x 128 bytes (1024-byte aligned)
    L.kstage = (size_t)p.k_boxes * kFastRows * 128;
    L.vstage = (size_t)p.v_boxes * kFastRows * 128;
    size_t off = 0;
    L.kring = off;
    off += (size_t)p.nstage_k * L.kstage;
    L.vring = off;
    off += (size_t)p.nstage_v * L.vstage;
    L.qlimb = off;
    off += fl_round(NQ * p.D * nlimb, 16);
    L.qscale = off;
    off += fl_round(NQ * NBH * 4, 16);
    L.qraw = off;                  // next item's raw queries [NQ][D] (bf16 or f32)
    off += p.q_stage ? fl_round(NQ * p.D * (p.q_bf16 ? 2 : 4), 16) : 0;
    L.P = off;
    off += fl_round((size_t)kFastPDepth * kFastRows * (NQ + 4) * 4, 16);
    L.alpha = off;
    off += fl_round((size_t)kFastPDepth * NQ * 4, 16);
    L.qlo = off;
    off += fl_round(NQ * 4, 16);
    L.qup = off;
    off += fl_round(NQ * 4, 16);
    L.lens = off;
    off += fl_round((3 * (size_t)p.B + 1) * 4, 16);
    L.bars = off;
    off += 8 * (size_t)(p.nstage_k + p.nstage_v);
    L.total = off + 1024;          // slack to align the base to 1024 bytes
    return L;
}

struct MergeParams {
    const float* part_o;
    const float* part_ml;
    const int* plan;               // [B+1]
    const float* sinks;            // [Hq] or null
    int* work_d;                   // the split kernel's work-item counter, reset here
    float* out;                    // [B][T][Hq][D]
    int B, Hq, Qtot, D;
};

// launchers (kvq_append.cu)
cudaError_t launch_append(const AppendParams& p, const SeqIds& ids, cudaStream_t s);
cudaError_t launch_commit(int* len_d, const SeqIds& ids, int T, cudaStream_t s);
cudaError_t launch_set_len(int* len_d, const SeqIds& ids, const int* values, cudaStream_t s);
cudaError_t launch_ring_copy(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k,
                             uint8_t* dst_v, size_t k_bytes, size_t v_bytes, cudaStream_t s);
cudaError_t launch_set_base(int* base_d, int seq, int value, cudaStream_t s);
// len_d[b] -= T - accept_d[b] for b < n, checked on the device (error word on failure)
cudaError_t launch_truncate_accept(int* len_d, const int* base_d, int* err_d, const int* accept_d, int n, int T,
                                   int window, int ring, cudaStream_t s);

// launchers (kvq_decode.cu)
size_t split_smem_bytes(const SplitParams& p);
int split_max_smem();
cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t s);
// warp-specialised decode (kvq_decode_fast.cu): token rows must be 16-byte multiples
cudaError_t launch_split_fast(const SplitParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                              cudaStream_t s);
// 3-D TMA map of a byte plane of `rows` token rows: one box = kFastRows rows x
// all 128-byte column blocks, 128-byte swizzle
bool make_row_tensor_map(CUtensorMap* map, void* plane, int tok_bytes, long long rows);
cudaError_t launch_merge(const MergeParams& p, int T, int max_splits, bool pdl, cudaStream_t s);

}  // namespace kvq
