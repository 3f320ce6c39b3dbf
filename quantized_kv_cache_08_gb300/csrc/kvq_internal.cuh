// Internal declarations shared by the kvq CUDA translation units (not part of
// the public C ABI in include/kvq.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace kvq {

constexpr int kQK = 32;            // elements per quantisation block
constexpr int kQ8Bytes = 34;       // q8_0 block: fp16 d + 32 int8 codes
constexpr int kQ5Bytes = 24;       // q5_1 block: fp16 d, fp16 m, u32 qh, 16 B qs
constexpr int kMaxIdsPerLaunch = 256;
constexpr int kSplitThreads = 256; // decode split CTA size
constexpr int kTileRows = 16;      // KV rows staged per pipeline stage
constexpr int kMinSplitRows = 64;  // smallest rows-per-split the workspace allows
constexpr int kMergeThreads = 256;

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
    int B, T, Hq, Hkv, hpk, D, kb, k_tok, v_tok, max_rows, window;
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

struct MergeParams {
    const float* part_o;
    const float* part_ml;
    const int* plan;               // [B+1]
    const float* sinks;            // [Hq] or null
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

// launchers (kvq_decode.cu)
size_t split_smem_bytes(const SplitParams& p);
int split_max_smem();
cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, int T, int max_splits, bool pdl, cudaStream_t s);

}  // namespace kvq
