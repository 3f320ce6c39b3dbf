/*
 * kvq.h - C ABI of a GPU-resident quantised KV cache for one attention layer
 * holding B sequences: K stored q8_0 and V stored q5_1 (or both stored FP8
 * E4M3, one byte per element), with quantised append,
 * truncate-based rollback and split-K flash-decode attention (GQA fan-out,
 * learned sinks, sliding window over a rebased ring, T >= 1 causal rows).
 *
 * The operations follow these passages:
 *   memra-engine "Struct KvLayer": the quantised per-layer cache (type
 *     description: q8_0 K at 34 B / 32 elements, q5_1 V at 24 B / 32 elements,
 *     [token, kv_head, dim] element order, head_dim % 32 == 0), the device
 *     mirrors len_d (append slot before the append, t_kv after it) and base_d
 *     (physical row of logical row 0 for the windowed ring view:
 *     lstart = max(0, len - window), physical = row - base), fn physical_rows.
 *   memra-engine "Struct Cache": fn new (allocate by geometry and max context),
 *     fn rollback item C.1 (len = snapshot_len + accept_len, truncate, no copy).
 *   memra-engine "Module cache": trait KvDev (every device op is ordered on the
 *     caller's stream), fn kv_blk_bytes, fn cache_bytes_per_token,
 *     fn swa_ring_rows (the ring keeps at most 31 masked rows before the live
 *     window), fn cache_ring_row_cap.
 *   cortiq-engine "Struct LayerKvCache": attention semantics of
 *     fn attend_group / fn attend_group_upto (scale 1/sqrt(head_dim), window
 *     start `first`, causal `upto = s0 + i + 1`, sink logits joining max and
 *     denominator without a value) and fn o1_views (head h reads group h/hpk).
 *
 * Ownership.  The caller allocates and owns every device buffer (the two byte
 * planes, the counters and the workspace, sized by kvq_required_bytes) and
 * every stream.  The library owns only the host handle returned by kvq_alloc.
 * It never allocates device memory, never frees caller memory and never
 * synchronises a stream except in kvq_read_device_error.  All device work is
 * enqueued on the stream passed to the call (NULL = the legacy default
 * stream); the caller keeps its buffers alive until that work completes.
 *
 * Errors.  Every call validates its arguments against the host mirror of the
 * lengths before it enqueues anything.  On error it enqueues nothing, leaves
 * the cache unchanged and returns a status; kvq_last_error() then gives a
 * one-line message (thread-local).  KVQ_ECUDA reports a failed launch; the
 * cache state is then undefined.  Kernels never trap: a kernel that finds a
 * device counter out of range, or whose bounded wait runs out, writes a
 * nonzero code to the device error word and skips its work; read it with
 * kvq_read_device_error.
 *
 * Graph capture.  kvq_append, kvq_decode and kvq_truncate read the lengths and
 * the ring base on the device, so a captured append+decode step replays
 * correctly as the lengths grow.  After replaying a captured chain of appends
 * call kvq_note_replayed so the host mirror follows; after one that contains
 * kvq_truncate_device (its accepted counts read on the device), call
 * kvq_sync_len instead.  A ring rebase is decided
 * on the host inside kvq_append: capture at most kvq_ring_headroom() appends.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,        /* bad argument or geometry                       */
    KVQ_ERANGE = 2,        /* length/capacity out of range                   */
    KVQ_ECUDA = 3,         /* a CUDA runtime call failed                     */
    KVQ_EUNSUPPORTED = 4   /* valid request this build does not implement    */
} kvq_status;

typedef enum kvq_dtype { KVQ_F32 = 0, KVQ_BF16 = 1 } kvq_dtype;

/* Block formats (memra-engine "Module cache", fn kv_blk_bytes):
 *   KVQ_Q8_0: fp16 d = amax/127 (round to nearest even), then 32 int8 codes
 *             round-half-away-from-zero(x/d) clamped to [-127,127]    34 B
 *   KVQ_Q5_1: fp16 d = (max-min)/31, fp16 m = min, u32 qh (bit i = bit 4 of
 *             code i), 16 bytes qs (byte j = code j low nibble | code j+16
 *             low nibble << 4); codes round-half-away((x-m)/d) in [0,31]
 *             against the stored m and d                                24 B
 *   KVQ_FP8_E4M3: one byte per element, no scale (memra-engine "Module
 *             cache", items gkv_on and kv_fp8_on: K/V held in e4m3).
 *             Read as OCP FP8 E4M3: sign, 4 exponent bits with bias 7, 3
 *             fraction bits, no infinities, largest finite 448; round to
 *             nearest, ties to even, magnitudes above 448 saturate to 448.
 *             A 32-element block is 32 bytes.
 * All multi-byte fields are little-endian.  Inputs must be finite. */
typedef enum kvq_fmt { KVQ_Q8_0 = 0, KVQ_Q5_1 = 1, KVQ_FP8_E4M3 = 2 } kvq_fmt;

typedef struct kvq_config {
    int n_seq;        /* B: sequences held by this layer cache (1..4096)           */
    int n_kv_heads;   /* Hkv                                                       */
    int head_dim;     /* D: multiple of 32, at most 512                            */
    int max_q_heads;  /* largest Hq a decode may pass (a multiple of Hkv)          */
    int max_t;        /* largest T of one append or decode call (1..512)           */
    int max_rows;     /* physical rows per sequence.  Flat cache: the logical      */
                      /* capacity.  Ring: 0 selects window + 30 + max_t.           */
    int window;       /* 0: full attention; > 0: each query row sees at most the   */
                      /* last `window` rows up to and including its own row        */
    int ring;         /* 1: SWA ring addressing, physical = row - base (needs      */
                      /* window > 0); 0: flat rows [0, max_rows)                   */
    kvq_fmt k_fmt;    /* KVQ_Q8_0 with v_fmt KVQ_Q5_1, or KVQ_FP8_E4M3 with        */
    kvq_fmt v_fmt;    /* v_fmt KVQ_FP8_E4M3; no other pairs                        */
} kvq_config;

/* Device bytes the caller provides (each buffer 16-byte aligned), and the
 * geometry they hold ("Module cache", fn cache_bytes_per_token and
 * fn swa_ring_rows):
 *   k_plane   [n_seq][rows][k_row_bytes], k_row_bytes = kb*34,
 *             kb = n_kv_heads*head_dim/32, plus 128 bytes of padding (the
 *             generic decode's tile copies may pass the last row), rounded up
 *             to a multiple of 256 bytes
 *   v_plane   [n_seq][rows][v_row_bytes], v_row_bytes = kb*24 (padded and
 *             rounded likewise).  With FP8 E4M3 both rows are kb*32 bytes.
 *   counters  len_d[n_seq], base_d[n_seq], error word, the append's
 *             completion counter, the ring rebase's barrier words (int32)
 *   workspace decode partials, the split plan and the ring-rebase scratch
 *   rows      physical rows per sequence: max_rows for a flat cache, and for
 *             a ring max_rows or, when it is 0, window + 30 + max_t        */
typedef struct kvq_sizes {
    size_t k_plane, v_plane, counters, workspace;
    int rows, k_row_bytes, v_row_bytes;
} kvq_sizes;

typedef struct kvq_cache kvq_cache;

/* Sizes of the four device buffers for a configuration and the rows they
 * hold (fn new of "Struct Cache" allocates by geometry and maximum context;
 * the byte counts per row are fn cache_bytes_per_token's for one layer).
 * Pure host call: KVQ_EINVAL / KVQ_EUNSUPPORTED for a bad configuration. */
kvq_status kvq_required_bytes(const kvq_config* cfg, kvq_sizes* out);

/* Build a cache over caller buffers (fn new of "Struct Cache").  Validates the
 * geometry (head_dim % 32 == 0, formats q8_0/q5_1 or e4m3/e4m3, ring needs
 * window > 0),
 * checks 16-byte alignment, and enqueues on `stream` the zeroing of the
 * counters (len = 0, base = 0, error = 0).  Byte planes are not cleared:
 * rows at or beyond a sequence's length are never read.  `*out` receives a
 * host handle to release with kvq_free.  stream: a cudaStream_t or NULL. */
kvq_status kvq_alloc(const kvq_config* cfg, void* k_plane, void* v_plane,
                     void* counters, void* workspace, void* stream,
                     kvq_cache** out);

/* Release the host handle (device buffers stay the caller's).  NULL is a
 * no-op.  No passage: the pages' cache owns its memory, this one only a
 * host handle. */
void kvq_free(kvq_cache* cache);

/* Quantised append ("Struct KvLayer": append_kv_quantized_dc[w] writes at the
 * slot len_d, inc_seqlen then adds T).  k, v: device [n][T][Hkv][D] of dtype
 * (f32 or bf16), n = n_ids, or n_seq when seq_ids is NULL.  Row t of entry i
 * is quantised into row len+t of sequence seq_ids[i] (or i).  seq_ids is a
 * HOST array of distinct indices; n_ids <= n_seq.  Flat caches return
 * KVQ_ERANGE when len + T > max_rows.  Ring caches first rebase a sequence
 * whose live rows would overflow the ring: logical rows [new_base, len) with
 * new_base = max(0, len + 1 - window) rounded down to a multiple of 32 move to
 * physical row 0 and base becomes new_base (fn swa_ring_rows: at most 31
 * masked rows precede the live window).  The move is one cooperative launch
 * through shared memory when the rows are 16-byte multiples and the live
 * bytes fit the SMs' shared memory, else two copies through the workspace.
 * Host lengths advance by T. */
kvq_status kvq_append(kvq_cache* cache, const void* k, const void* v,
                      kvq_dtype dtype, int T, const int* seq_ids, int n_ids,
                      void* stream);

/* Decode attention over the quantised rows ("Struct LayerKvCache",
 * fn attend_group_upto).  q: device [n_seq][T][n_q_heads][D] (f32 or bf16);
 * its T rows are the last T rows appended to each sequence: row t sits at
 * position s0 + t, s0 = len - T, and sees logical rows [lstart_t, s0 + t + 1)
 * with lstart_t = max(0, s0 + t + 1 - window) when window > 0, else 0.
 * Head h reads KV group h / (n_q_heads / Hkv).  Scores are scale * <q, k_hat>
 * (scale <= 0 selects 1/sqrt(D)); sinks (device [n_q_heads] f32, or NULL) are
 * unscaled logits joining the max and the denominator with no value.
 * out: device f32 [n_seq][T][n_q_heads][D].  Every sequence needs len >= T.
 * Two launches: a split kernel writes partial softmax records (running max,
 * denominator, unnormalised output) and a merge kernel combines them with the
 * sinks.  The split kernel is the stream-K kernel (its CTAs, at most one per
 * SM, each take an equal share of all sequences' visible rows in 32-row
 * tiles) or the generic kernel over (sequence, row chunk) work items; see
 * kvq_set_decode_path. */
kvq_status kvq_decode(kvq_cache* cache, const void* q, kvq_dtype dtype, int T,
                      int n_q_heads, const float* sinks, float scale,
                      float* out, void* stream);

/* Bytes of the no-alloc decode scratch (a fixed device array in the library). */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)

/* kvq_decode without the cache's workspace: the described design has no
 * counterpart of this call; it lets a caller decode without providing
 * partial-result memory.  Same arguments, semantics and results as
 * kvq_decode (the same kernels run on the same split plan), but the split
 * partials and the plan live in a file-scope device array of
 * KVQ_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library: the call allocates
 * nothing.  The decode needs R records of (head_dim + 2) * 4 bytes.  On the
 * stream-K kernel R = (G + nqs * n_seq) * 4 * Hkv * QPS, where G <= 256 is
 * the CTA count (one per SM at most), u = ceil(hpk * T / 4) four-query units per KV head (hpk =
 * n_q_heads / Hkv), QPS = max(1, min(u, 16 / Hkv)) and nqs = ceil(u / QPS):
 * 64 sequences with 8 KV heads, 32 Q heads and T = 1 need about 3.6 MB on 152
 * SMs.  On the generic kernel R = n_seq * ceil(max visible rows / split rows)
 * * n_q_heads * T, plus a plan of n_seq + 1 ints.  A call that needs more
 * returns KVQ_ERANGE (nothing launched) and says how much.  Nothing in the
 * array has to start at zero: every byte read was written earlier in the
 * same call.  The array's address is resolved (cudaGetSymbolAddress, with the
 * device current) on the first call on a device and again whenever the
 * calling thread's current CUDA context differs from the one it was resolved
 * in: make the first call in each context before any stream capture.  All
 * calls share the one array per device, so two calls whose
 * kernels may overlap (other streams, other threads, other caches) race:
 * order them on one stream or synchronise between them. */
kvq_status kvq_decode_noalloc(kvq_cache* cache, const void* q, kvq_dtype dtype, int T,
                              int n_q_heads, const float* sinks, float scale,
                              float* out, void* stream);

/* Rollback ("Struct Cache", fn rollback, item C.1): set each sequence's
 * length to new_len[b] (a HOST array of n_seq values, usually
 * snapshot_len + accept_len), no data moves.  Needs new_len[b] <= len (the
 * lower end while a kvq_truncate_device is pending); a ring
 * sequence also needs max(0, new_len + 1 - window) >= base (rewinds never
 * move the base), else KVQ_ERANGE. */
kvq_status kvq_truncate(kvq_cache* cache, const int* new_len, void* stream);

/* Rollback with the accepted counts on the device ("Struct Cache", fn
 * rollback, item C.1, len = snapshot_len + accept_len, with snapshot_len =
 * len - T for the T draft rows just appended and verified; "Struct KvLayer",
 * field base_d: rewinds move len_d only).  accept_d: DEVICE int32 [n_seq],
 * read when the kernel runs, so a captured graph replays with whatever it
 * holds then.  For each sequence, len_d -= T - accept_d[b]: the first
 * accept_d[b] of the last T rows stay.  The kernel checks 0 <= accept <= T,
 * T <= len_d and, for a ring, max(0, new_len + 1 - window) >= base; a
 * sequence that fails keeps its length and the device error word becomes 1.
 * The host does not wait, so its mirror then knows each length only within
 * [len - T, len]: appends check capacity against the upper end, a ring
 * append that would rebase returns KVQ_ERANGE, decodes need T <= the lower
 * end, and kvq_truncate takes only new_len <= the lower end (which makes the
 * length exact again), until kvq_sync_len reads the lengths back.  The host
 * refuses (KVQ_ERANGE, nothing enqueued) when a sequence may hold fewer than
 * T rows or, for a ring, when accepting nothing would drop rows below base.
 * After replaying a graph that contains this call, call kvq_sync_len before
 * any other call on the cache (kvq_note_replayed cannot know the counts). */
kvq_status kvq_truncate_device(kvq_cache* cache, const int* accept_d, int T, void* stream);

/* Synchronise `stream` and read the device lengths into the host mirror,
 * making it exact (after kvq_truncate_device).  KVQ_ERANGE if a device length
 * lies outside its sequence's resident rows (the mirror is then unchanged). */
kvq_status kvq_sync_len(kvq_cache* cache, void* stream);

/* Host mirror of the lengths and ring bases (HOST arrays of n_seq ints;
 * either pointer may be NULL): the host side of the len_d / base_d pair of
 * "Struct KvLayer".  After kvq_truncate_device and before kvq_sync_len the
 * lengths are upper bounds. */
kvq_status kvq_get_len(const kvq_cache* cache, int* len_host, int* base_host);

/* Advance the host mirror after `steps` replays of a captured graph that
 * appended T rows to every sequence per step. */
kvq_status kvq_note_replayed(kvq_cache* cache, int steps, int T);

/* Appends of T rows (to every sequence) that can run before a ring rebase is
 * due, i.e. how many steps a captured graph may replay. Flat caches: rows
 * left before max_rows, divided by T.  While a kvq_truncate_device is
 * pending it counts from the upper ends of the lengths (a safe undercount). */
kvq_status kvq_ring_headroom(const kvq_cache* cache, int T, int* steps);

/* fn physical_rows of "Struct KvLayer": map logical rows [start, end) of
 * sequence seq to physical rows; KVQ_ERANGE if any row is not resident. */
kvq_status kvq_physical_rows(const kvq_cache* cache, int seq, int start,
                             int end, int* phys_start, int* phys_end);

/* Synchronise `stream`, read the device error word into *err (0 = none;
 * 1 = a kernel saw a length or base out of range; 2 = a bounded wait ran
 * out) and clear it. */
kvq_status kvq_read_device_error(kvq_cache* cache, int* err, void* stream);

/* Choose the decode kernel: path 0 = automatic (the stream-K kernel whenever
 * it allows the cache and the call, else the generic split kernel),
 * 1 = generic, 2 = stream-K (KVQ_EUNSUPPORTED at decode time if it does not
 * allow them).  The stream-K kernel needs K and V token rows that are
 * 16-byte multiples (q8_0/q5_1: n_kv_heads * head_dim a multiple of 256;
 * E4M3: of 16) and at most 2048 bytes, head_dim 64, 128 or 256,
 * n_kv_heads <= 16, n_seq <= 1024 and its tiles within shared memory.
 * query_bits (0 = 16, or 16, or 24): on q8_0 K the stream-K kernel quantises
 * each pre-scaled query element per 32-element block to this many bits
 * against the block's largest magnitude and multiplies it with the int8 K
 * codes in integer dot products; 16 bits adds an error below 1e-4 to the
 * attention output on unit-variance data, 24 bits is at the level of fp32
 * rounding and costs half again as many dot products.  With E4M3 K the
 * queries stay f32 and query_bits does not apply. */
kvq_status kvq_set_decode_path(kvq_cache* cache, int path, int query_bits);

/* Score soft-capping for later decodes ("Struct LayerKvCache": the softcap
 * argument of fn attend_group / attend_group_upto, which the pages name
 * without defining; read as the usual logit soft-capping).  softcap > 0 maps
 * every scaled score s = scale * <q, k_hat> to softcap * tanh(s / softcap)
 * before the softmax; sink logits are not capped.  0 (the default) turns it
 * off.  Both decode kernels apply it.  KVQ_EINVAL for a negative or
 * non-finite value. */
kvq_status kvq_set_softcap(kvq_cache* cache, float softcap);

/* Row slices per 32-row tile on the stream-K kernel: 0 = automatic (two,
 * one warp per half tile, when 2 x (KV heads x four-query groups of a slice)
 * <= 16 and the CTAs have more than 16 tiles each; else one), 1, or 2 (taken
 * only where the geometry allows two; else one).  Results are the same up to
 * fp32 rounding; the choice moves speed only.  No passage: a tuning knob of
 * this implementation.  KVQ_EINVAL for another value. */
kvq_status kvq_set_row_slices(kvq_cache* cache, int slices);

/* Override the generic kernel's split size in rows (a multiple of 8, >= 64;
 * 0 = auto).  The stream-K kernel ignores it: its CTAs split the rows
 * evenly. */
kvq_status kvq_set_split_rows(kvq_cache* cache, int rows);

/* Bytes per 32-element block of a format: 34 (q8_0), 24 (q5_1) or 32
 * (FP8 E4M3); -1 if unknown ("Module cache", fn kv_blk_bytes). */
int kvq_block_bytes(kvq_fmt fmt);

/* Context-linear bytes one token occupies in this layer cache, K plus V
 * ("Module cache", fn cache_bytes_per_token, for a single layer); 0 on bad
 * input. */
size_t kvq_bytes_per_token(const kvq_config* cfg);

/* Message of the last failed call on this thread ("" if none).  No passage:
 * error reporting of this C interface. */
const char* kvq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
