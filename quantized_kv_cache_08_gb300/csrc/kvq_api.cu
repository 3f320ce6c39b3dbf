// Host side of the kvq C ABI: validation against the host mirror of the
// lengths, ring bookkeeping, workspace layout and kernel launches.  See
// include/kvq.h for the contract of every entry point.
#include "../../include/kvq.h"
#include "kvq_internal.cuh"

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

using namespace kvq;

static constexpr int kMaxDevices = 64;

struct kvq_cache {
    CUtensorMap kmap, vmap;              // 2-D TMA maps of the planes (stream-K decode)
    bool smap_ok;
    uint32_t Sk, Sv;                     // stream-K shared-memory row strides
    kvq_config cfg;
    uint8_t* k_plane;
    uint8_t* v_plane;
    int* len_d;
    int* base_d;
    int* err_d;
    uint8_t* ws;
    size_t off_part_o, off_part_ml, off_plan, off_scratch;
    int kb, k_tok, v_tok, rows;          // rows = physical rows per sequence
    int max_vis;                         // most rows one decode may read per sequence
    int num_sms;
    int split_rows;                      // 0 = automatic
    int row_slices;                      // stream-K row slices per tile: 0 = automatic, 1 or 2
    int path;                            // 0 auto, 1 generic split kernel, 2 stream-K kernel
    int qbits;                           // query bits of the stream-K kernel (16 or 24)
    int fp8;                             // 1: K and V planes hold FP8 E4M3 bytes
    float softcap;                       // score cap (0: off)
    std::vector<int> len, base;
    // lower bound of each length: equal to len except after kvq_truncate_device,
    // when len_d lies in [len_lo, len] until kvq_sync_len or kvq_truncate
    std::vector<int> len_lo;
};

namespace {

thread_local std::string g_err;

kvq_status fail(kvq_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KVQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Geometry {
    int kb, k_tok, v_tok, rows, max_vis, fp8;
};

kvq_status check_config(const kvq_config* c, Geometry* g) {
    if (!c) return fail(KVQ_EINVAL, "config is NULL");
    const bool q8q5 = c->k_fmt == KVQ_Q8_0 && c->v_fmt == KVQ_Q5_1;
    const bool f8 = c->k_fmt == KVQ_FP8_E4M3 && c->v_fmt == KVQ_FP8_E4M3;
    if (!q8q5 && !f8) return fail(KVQ_EUNSUPPORTED, "formats must be K=q8_0, V=q5_1 or K=V=fp8_e4m3");
    if (c->n_seq < 1 || c->n_seq > 4096) return fail(KVQ_EINVAL, "n_seq must be in [1, 4096]");
    if (c->n_kv_heads < 1) return fail(KVQ_EINVAL, "n_kv_heads must be >= 1");
    if (c->head_dim < 32 || c->head_dim > 512 || c->head_dim % 32)
        return fail(KVQ_EINVAL, "head_dim must be a multiple of 32 in [32, 512] (a block never straddles a head)");
    if (c->max_q_heads < c->n_kv_heads || c->max_q_heads % c->n_kv_heads)
        return fail(KVQ_EINVAL, "max_q_heads must be a positive multiple of n_kv_heads");
    if (c->max_t < 1 || c->max_t > 512) return fail(KVQ_EINVAL, "max_t must be in [1, 512]");
    if (c->window < 0) return fail(KVQ_EINVAL, "window must be >= 0");
    if (c->ring && c->window <= 0) return fail(KVQ_EINVAL, "a ring cache needs window > 0");
    const long long kvd = (long long)c->n_kv_heads * c->head_dim;
    if (kvd > 65536) return fail(KVQ_EINVAL, "n_kv_heads * head_dim too large");
    g->kb = (int)(kvd / kQK);
    g->fp8 = f8 ? 1 : 0;
    g->k_tok = g->kb * (f8 ? kF8Bytes : kQ8Bytes);
    g->v_tok = g->kb * (f8 ? kF8Bytes : kQ5Bytes);
    if (c->ring) {
        const int need = c->window + 30 + c->max_t;
        g->rows = c->max_rows == 0 ? need : c->max_rows;
        if (g->rows < need)
            return fail(KVQ_EINVAL, "ring max_rows %d below window + 30 + max_t = %d", g->rows, need);
        g->max_vis = std::min(g->rows, c->window + c->max_t - 1);
    } else {
        if (c->max_rows < 1) return fail(KVQ_EINVAL, "max_rows must be >= 1");
        g->rows = c->max_rows;
        g->max_vis = c->window > 0 ? std::min(g->rows, c->window + c->max_t - 1) : g->rows;
    }
    return KVQ_OK;
}

// Unit layout of the stream-K kernel for hpk Q heads per KV head and T query
// rows: units of 4 queries, at most 16 per CTA (one per warp and row slice),
// query slices for the rest, and rows of a tile split RS ways among the warps
// of a unit.  ok = false when the geometry or format does not allow it.
struct StreamShape {
    bool ok;
    int QPS, nqs, RS;
};

StreamShape stream_shape(const kvq_config* c, const Geometry& g, int hpk, int T) {
    StreamShape sh{false, 1, 1, 1};
    const int NBH = c->head_dim / 32;
    if (g.k_tok % 16 || g.v_tok % 16 || !(NBH == 2 || NBH == 4 || NBH == 8) || c->n_seq > kStreamMaxB ||
        c->n_kv_heads > kStreamThreads / 32)
        return sh;
    const int nQG = (hpk * T + 3) / 4;
    sh.QPS = std::max(1, std::min(nQG, (kStreamThreads / 32) / c->n_kv_heads));
    sh.nqs = (nQG + sh.QPS - 1) / sh.QPS;
    const int nU = c->n_kv_heads * sh.QPS;
    sh.RS = 2 * nU <= kStreamThreads / 32 ? 2 : 1;
    sh.ok = (long long)sh.nqs * c->n_seq * g.rows < (1LL << 31);
    return sh;
}

// Partial records of a stream-K decode on G CTAs
size_t stream_records(const kvq_config* c, const StreamShape& sh, int G) {
    return ((size_t)G + (size_t)sh.nqs * c->n_seq) * 4 * c->n_kv_heads * sh.QPS;
}

struct WsLayout {
    size_t part_o, part_ml, plan, scratch, total;
};

WsLayout ws_layout(const kvq_config* c, const Geometry& g) {
    WsLayout w;
    const size_t items = (size_t)c->n_seq * ((g.max_vis + kMinSplitRows - 1) / kMinSplitRows);
    size_t recs = items * (size_t)c->max_q_heads * c->max_t;
    // the stream-K kernel's records for every (Q heads, T) a decode may pass
    const int max_hpk = c->max_q_heads / c->n_kv_heads;
    for (int hpk = 1; hpk <= max_hpk; ++hpk)
        for (int T = 1; T <= c->max_t; ++T) {
            const StreamShape sh = stream_shape(c, g, hpk, T);
            if (sh.ok) recs = std::max(recs, stream_records(c, sh, kStreamMaxGrid));
        }
    w.part_o = 0;
    w.part_ml = round_up(w.part_o + recs * c->head_dim * sizeof(float), 256);
    w.plan = round_up(w.part_ml + recs * 2 * sizeof(float), 256);
    w.scratch = round_up(w.plan + (c->n_seq + 1) * sizeof(int), 256);
    w.total = w.scratch + (c->ring ? round_up((size_t)g.rows * (g.k_tok + g.v_tok), 256) : 0);
    return w;
}

// len_d[n], base_d[n], error word, append completion counter, rebase arrival
// counter, rebase barrier generation
size_t counters_bytes(int n_seq) { return round_up((2 * (size_t)n_seq + 4) * sizeof(int), 256); }

// visible-row start of a T-row step
int vis_lo(const kvq_cache* c, int len, int T) {
    return c->cfg.window > 0 ? std::max(0, len - T + 1 - c->cfg.window) : 0;
}

bool aligned16(const void* p) { return ((size_t)p & 15) == 0; }

}  // namespace

extern "C" {

const char* kvq_last_error(void) { return g_err.c_str(); }

int kvq_block_bytes(kvq_fmt fmt) {
    if (fmt == KVQ_Q8_0) return kQ8Bytes;
    if (fmt == KVQ_Q5_1) return kQ5Bytes;
    if (fmt == KVQ_FP8_E4M3) return kF8Bytes;
    return -1;
}

size_t kvq_bytes_per_token(const kvq_config* cfg) {
    Geometry g;
    if (check_config(cfg, &g) != KVQ_OK) return 0;
    return (size_t)g.k_tok + g.v_tok;
}

kvq_status kvq_required_bytes(const kvq_config* cfg, kvq_sizes* out) {
    Geometry g;
    kvq_status st = check_config(cfg, &g);
    if (st != KVQ_OK) return st;
    if (!out) return fail(KVQ_EINVAL, "out is NULL");
    // rounded up and padded by 128 bytes: tile copies read whole 16-byte
    // chunks and whole 128-byte column blocks, which may pass the last row
    out->k_plane = round_up((size_t)cfg->n_seq * g.rows * g.k_tok + 128, 256);
    out->v_plane = round_up((size_t)cfg->n_seq * g.rows * g.v_tok + 128, 256);
    out->counters = counters_bytes(cfg->n_seq);
    out->workspace = ws_layout(cfg, g).total;
    out->rows = g.rows;
    out->k_row_bytes = g.k_tok;
    out->v_row_bytes = g.v_tok;
    return KVQ_OK;
}

kvq_status kvq_alloc(const kvq_config* cfg, void* k_plane, void* v_plane, void* counters, void* workspace,
                     void* stream, kvq_cache** out) {
    Geometry g;
    kvq_status st = check_config(cfg, &g);
    if (st != KVQ_OK) return st;
    if (!out) return fail(KVQ_EINVAL, "out is NULL");
    *out = nullptr;
    if (!k_plane || !v_plane || !counters || !workspace) return fail(KVQ_EINVAL, "a device buffer is NULL");
    if (!aligned16(k_plane) || !aligned16(v_plane) || !aligned16(counters) || !aligned16(workspace))
        return fail(KVQ_EINVAL, "device buffers must be 16-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    kvq_cache* c = new kvq_cache();
    c->cfg = *cfg;
    c->cfg.max_rows = g.rows;
    c->k_plane = static_cast<uint8_t*>(k_plane);
    c->v_plane = static_cast<uint8_t*>(v_plane);
    c->len_d = static_cast<int*>(counters);
    c->base_d = c->len_d + cfg->n_seq;
    c->err_d = c->base_d + cfg->n_seq;
    c->ws = static_cast<uint8_t*>(workspace);
    const WsLayout w = ws_layout(cfg, g);
    c->off_part_o = w.part_o;
    c->off_part_ml = w.part_ml;
    c->off_plan = w.plan;
    c->off_scratch = w.scratch;
    c->kb = g.kb;
    c->k_tok = g.k_tok;
    c->v_tok = g.v_tok;
    c->rows = g.rows;
    c->max_vis = g.max_vis;
    c->num_sms = sms;
    c->split_rows = 0;
    c->row_slices = 0;
    // stream-K stage rows: K at an odd multiple of 16 bytes (consecutive rows
    // in different bank groups), V at 64 mod 128 bytes
    // (rows that are not 16-byte multiples cannot be tensor-copied at all)
    const bool rows16 = g.k_tok % 16 == 0 && g.v_tok % 16 == 0;
    c->Sk = (uint32_t)((g.k_tok / 16) % 2 ? g.k_tok : g.k_tok + 16);
    c->Sv = (uint32_t)g.v_tok;
    if (rows16)
        c->Sv += (uint32_t)((64 - g.v_tok % 128 + 128) % 128);
    c->smap_ok = rows16 &&
                 make_stream_map(&c->kmap, k_plane, g.k_tok, (int)c->Sk, (long long)cfg->n_seq * g.rows) &&
                 make_stream_map(&c->vmap, v_plane, g.v_tok, (int)c->Sv, (long long)cfg->n_seq * g.rows);
    c->path = 0;
    c->qbits = 16;                         // 16-bit queries unless 24 is asked for
    c->fp8 = g.fp8;
    c->softcap = 0.f;
    c->len.assign(cfg->n_seq, 0);
    c->len_lo.assign(cfg->n_seq, 0);
    c->base.assign(cfg->n_seq, 0);
    e = cudaMemsetAsync(counters, 0, counters_bytes(cfg->n_seq), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "cudaMemsetAsync(counters)");
    }
    *out = c;
    return KVQ_OK;
}

void kvq_free(kvq_cache* cache) { delete cache; }

kvq_status kvq_append(kvq_cache* c, const void* k, const void* v, kvq_dtype dtype, int T, const int* seq_ids,
                      int n_ids, void* stream) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (!k || !v) return fail(KVQ_EINVAL, "k or v is NULL");
    if (dtype != KVQ_F32 && dtype != KVQ_BF16) return fail(KVQ_EINVAL, "dtype must be f32 or bf16");
    if (T < 1 || T > c->cfg.max_t) return fail(KVQ_EINVAL, "T=%d outside [1, max_t=%d]", T, c->cfg.max_t);
    const int B = c->cfg.n_seq;
    std::vector<int> ids;
    if (seq_ids) {
        if (n_ids < 1 || n_ids > B) return fail(KVQ_EINVAL, "n_ids must be in [1, n_seq]");
        ids.assign(seq_ids, seq_ids + n_ids);
        std::vector<char> seen(B, 0);
        for (int b : ids) {
            if (b < 0 || b >= B) return fail(KVQ_EINVAL, "sequence index %d out of range", b);
            if (seen[b]) return fail(KVQ_EINVAL, "sequence index %d repeated", b);
            seen[b] = 1;
        }
    } else {
        ids.resize(B);
        for (int b = 0; b < B; ++b) ids[b] = b;
    }
    // capacity and ring decisions, all validated before anything is enqueued
    const bool ring = c->cfg.ring != 0;
    std::vector<int> new_base(ids.size());
    for (size_t i = 0; i < ids.size(); ++i) {
        const int b = ids[i];
        const long long len = c->len[b];
        int nb = c->base[b];
        if (len + T - nb > c->rows) {
            if (!ring)
                return fail(KVQ_ERANGE, "sequence %d: len %lld + T %d exceeds max_rows %d", b, len, T, c->rows);
            if (c->len_lo[b] != c->len[b])
                return fail(KVQ_ERANGE,
                            "sequence %d: a ring rebase needs the exact length, pending a device-side rollback "
                            "(call kvq_sync_len first)", b);
            nb = (int)(std::max(0LL, len + 1 - c->cfg.window) & ~31LL);
            if (len + T - nb > c->rows)
                return fail(KVQ_ERANGE, "sequence %d: T %d does not fit the ring of %d rows", b, T, c->rows);
        }
        if (len + T > 0x7fffffffLL) return fail(KVQ_ERANGE, "sequence %d: length overflows int32", b);
        new_base[i] = nb;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    // ring rebases: live rows [nb, len) move to physical row 0 through scratch
    for (size_t i = 0; i < ids.size(); ++i) {
        const int b = ids[i];
        const int nb = new_base[i];
        if (nb == c->base[b]) continue;
        const int live = c->len[b] - nb;
        const size_t src_row = (size_t)b * c->rows + (size_t)(nb - c->base[b]);
        const size_t dst_row = (size_t)b * c->rows;
        uint8_t* sk = c->ws + c->off_scratch;
        uint8_t* sv = sk + (size_t)c->rows * c->k_tok;
        const size_t kbytes = (size_t)live * c->k_tok, vbytes = (size_t)live * c->v_tok;
        // one pass through shared memory when it fits, else two copy legs
        // through the workspace scratch
        if (launch_rebase_one_pass(c->k_plane + src_row * c->k_tok, c->v_plane + src_row * c->v_tok,
                                   c->k_plane + dst_row * c->k_tok, c->v_plane + dst_row * c->v_tok, kbytes, vbytes,
                                   c->base_d, b, nb, c->err_d + 2, c->err_d + 3, c->err_d, c->num_sms, s, &e)) {
            if (e != cudaSuccess) return cuda_fail(e, "ring rebase");
            c->base[b] = nb;
            continue;
        }
        e = launch_ring_copy(c->k_plane + src_row * c->k_tok, c->v_plane + src_row * c->v_tok, sk, sv, kbytes,
                             vbytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "ring rebase copy");
        e = launch_ring_copy(sk, sv, c->k_plane + dst_row * c->k_tok, c->v_plane + dst_row * c->v_tok, kbytes,
                             vbytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "ring rebase copy back");
        e = launch_set_base(c->base_d, b, nb, s);
        if (e != cudaSuccess) return cuda_fail(e, "ring base update");
        c->base[b] = nb;
    }
    AppendParams p;
    p.k = k;
    p.v = v;
    p.bf16 = dtype == KVQ_BF16;
    p.k_plane = c->k_plane;
    p.v_plane = c->v_plane;
    p.len_d = c->len_d;
    p.base_d = c->base_d;
    p.err_d = c->err_d;
    p.done_d = c->err_d + 1;
    p.T = T;
    p.kb = c->kb;
    p.k_tok = c->k_tok;
    p.v_tok = c->v_tok;
    p.max_rows = c->rows;
    p.fp8 = c->fp8;
    SeqIds sid;
    for (size_t first = 0; first < ids.size(); first += kMaxIdsPerLaunch) {
        const int n = (int)std::min(ids.size() - first, (size_t)kMaxIdsPerLaunch);
        sid.n = n;
        sid.identity = seq_ids ? 0 : 1;
        sid.first = (int)first;
        for (int i = 0; i < n; ++i) sid.id[i] = ids[first + i];
        p.entry_offset = (long long)first;
        e = launch_append(p, sid, s);
        if (e != cudaSuccess) return cuda_fail(e, "append kernel");
    }
    for (int b : ids) {
        c->len[b] += T;
        c->len_lo[b] += T;
    }
    return KVQ_OK;
}

// Decode through the cache's workspace (scratch == nullptr) or through the
// caller-given scratch of scratch_bytes (partials, split plan).
static kvq_status decode_impl(kvq_cache* c, const void* q, kvq_dtype dtype, int T, int n_q_heads,
                              const float* sinks, float scale, float* out, void* stream, unsigned char* scratch,
                              size_t scratch_bytes) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (!q || !out) return fail(KVQ_EINVAL, "q or out is NULL");
    if (dtype != KVQ_F32 && dtype != KVQ_BF16) return fail(KVQ_EINVAL, "dtype must be f32 or bf16");
    if (T < 1 || T > c->cfg.max_t) return fail(KVQ_EINVAL, "T=%d outside [1, max_t=%d]", T, c->cfg.max_t);
    const int Hkv = c->cfg.n_kv_heads;
    if (n_q_heads < Hkv || n_q_heads % Hkv || n_q_heads > c->cfg.max_q_heads)
        return fail(KVQ_EINVAL, "n_q_heads must be a multiple of n_kv_heads and <= max_q_heads");
    const int B = c->cfg.n_seq;
    const int D = c->cfg.head_dim;
    const int hpk = n_q_heads / Hkv;
    const int Q = hpk * T;
    long long total_vis = 0;
    for (int b = 0; b < B; ++b) {
        if (c->len_lo[b] < T)
            return fail(KVQ_ERANGE, "sequence %d holds %d rows, fewer than T=%d", b, c->len_lo[b], T);
        total_vis += c->len[b] - vis_lo(c, c->len[b], T);
    }
    const float qscale = (scale > 0.f ? scale : 1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    const float cap_a = c->softcap > 0.f ? 1.0f / (c->softcap * 1.4426950408889634f) : 0.f;
    const float cap_b = c->softcap > 0.f ? c->softcap * 1.4426950408889634f : 0.f;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // ---- the stream-K kernel: 16-byte token rows, head_dim 64, 128 or 256
    Geometry g{c->kb, c->k_tok, c->v_tok, c->rows, c->max_vis, c->fp8};
    const StreamShape sh = stream_shape(&c->cfg, g, hpk, T);
    if (c->path != 1 && sh.ok && c->smap_ok) {
        StreamParams p;
        p.k_plane = c->k_plane;
        p.v_plane = c->v_plane;
        p.len_d = c->len_d;
        p.base_d = c->base_d;
        p.err_d = c->err_d;
        p.q = q;
        p.q_bf16 = dtype == KVQ_BF16;
        p.qscale = qscale;
        p.softcap_a = cap_a;
        p.softcap_b = cap_b;
        p.B = B;
        p.T = T;
        p.Hq = n_q_heads;
        p.Hkv = Hkv;
        p.hpk = hpk;
        p.D = D;
        p.k_tok = c->k_tok;
        p.v_tok = c->v_tok;
        p.max_rows = c->rows;
        p.window = c->cfg.window;
        p.Qh = Q;
        p.QPS = sh.QPS;
        p.nqs = sh.nqs;
        p.RS = sh.RS;
        p.NA = Hkv * sh.QPS * sh.RS;
        p.Qtot = n_q_heads * T;
        p.qbits = c->qbits;
        p.Sk = c->Sk;
        p.Sv = c->Sv;
        // CTAs: one per SM, fewer when there are fewer 32-row tiles of work
        const long long work = total_vis * sh.nqs;
        p.G = (int)std::max(1LL, std::min<long long>((work + kStreamRows - 1) / kStreamRows,
                                                     std::min(kStreamCtasPerSm * c->num_sms, kStreamMaxGrid)));
        // two row slices per tile pay off in the steady state (twice the warps
        // hide more latency); with few tiles per CTA one slice wins (half the
        // query preparation, no pair hand-over at a record): measured on
        // GB300 the turn is near 16 tiles per CTA
        if (p.RS == 2 && (c->row_slices == 1 ||
                          (c->row_slices == 0 && work <= kStreamShortTiles * kStreamRows * (long long)p.G))) {
            p.RS = 1;
            p.NA = Hkv * sh.QPS;
        }
        const int smem_max = stream_max_smem();
        p.NS = 3;
        auto layout_bytes = [&]() { return c->fp8 ? stream_layout_f8(p).total : stream_layout(p).total; };
        while (p.NS > 2 && layout_bytes() > (size_t)smem_max) --p.NS;
        if (layout_bytes() <= (size_t)smem_max) {
            const size_t recs = stream_records(&c->cfg, sh, p.G);
            if (scratch) {
                const size_t o_ml = round_up(recs * D * sizeof(float), 256);
                const size_t need = o_ml + recs * 2 * sizeof(float);
                if (need > scratch_bytes)
                    return fail(KVQ_ERANGE,
                                "this decode needs %zu bytes of scratch, the no-alloc entry point holds %zu", need,
                                scratch_bytes);
                p.part_o = reinterpret_cast<float*>(scratch);
                p.part_ml = reinterpret_cast<float*>(scratch + o_ml);
            } else {
                p.part_o = reinterpret_cast<float*>(c->ws + c->off_part_o);
                p.part_ml = reinterpret_cast<float*>(c->ws + c->off_part_ml);
            }
            cudaError_t e = c->fp8 ? launch_split_stream_f8(p, c->kmap, c->vmap, s)
                                   : launch_split_stream(p, c->kmap, c->vmap, s);
            if (e != cudaSuccess) return cuda_fail(e, "decode split kernel");
            MergeStreamParams m;
            m.part_o = p.part_o;
            m.part_ml = p.part_ml;
            m.len_d = c->len_d;
            m.base_d = c->base_d;
            m.window = c->cfg.window;
            m.max_rows = c->rows;
            m.sinks = sinks;
            m.out = out;
            m.B = B;
            m.T = T;
            m.Hq = n_q_heads;
            m.hpk = hpk;
            m.D = D;
            m.Qtot = p.Qtot;
            m.QPS = p.QPS;
            m.nqs = p.nqs;
            m.G = p.G;
            // records per (sequence, query): RS per CTA whose range meets it;
            // many records: 16 warps split them on 32-dim chunks, few: one
            // warp per (sequence, query) over all dims
            const long long keys = (long long)sh.nqs * B;
            const long long recs_per = (p.G + keys - 1) / keys + 2;
            int wpq = 1;
            while (wpq < 16 && wpq * 16 < recs_per) wpq *= 2;
            m.WPQ = wpq;
            m.DC = wpq >= 4 ? 32 : std::min(D, 256);
            e = launch_merge_stream(m, s);
            if (e != cudaSuccess) return cuda_fail(e, "decode merge kernel");
            return KVQ_OK;
        }
    }
    if (c->path == 2)
        return fail(KVQ_EUNSUPPORTED, "the stream-K decode does not support this geometry");

    // ---- the generic split kernel
    const int QC = Q <= 4 ? 4 : 8;
    const int NBH = D / 32;
    const int nK = (QC / 4) * Hkv * NBH;
    const bool generic_ok = 2 * nK <= kSplitThreads && kSplitThreads % (2 * nK) == 0;
    if (!generic_ok)
        return fail(KVQ_EUNSUPPORTED, "decode needs (queries/4) * n_kv_heads * head_dim/32 to divide 128");
    // rows per split: one wave of items for one sequence; otherwise about 5
    // items per CTA (an item start costs a query preparation, a partial last
    // tile costs nearly a full one)
    int C = c->split_rows;
    if (C == 0) {
        const long long per = B == 1 ? (total_vis + c->num_sms - 1) / c->num_sms
                                     : (total_vis + 5LL * c->num_sms - 1) / (5LL * c->num_sms);
        C = (int)std::max<long long>(kMinSplitRows, round_up((size_t)per, B == 1 ? 8 : 32));
    }
    const int max_splits = (c->max_vis + C - 1) / C;

    SplitParams p;
    p.k_plane = c->k_plane;
    p.v_plane = c->v_plane;
    p.len_d = c->len_d;
    p.base_d = c->base_d;
    p.err_d = c->err_d;
    p.q = q;
    p.q_bf16 = dtype == KVQ_BF16;
    p.qscale = qscale;
    p.softcap_a = cap_a;
    p.softcap_b = cap_b;
    p.B = B;
    p.T = T;
    p.Hq = n_q_heads;
    p.Hkv = Hkv;
    p.hpk = hpk;
    p.D = D;
    p.kb = c->kb;
    p.k_tok = c->k_tok;
    p.v_tok = c->v_tok;
    p.max_rows = c->rows;
    p.window = c->cfg.window;
    p.fp8 = c->fp8;
    p.C = C;
    p.QC = QC;
    p.nqs = (Q + QC - 1) / QC;
    p.Qtot = n_q_heads * T;
    if (scratch) {
        // records: at most max_splits splits per sequence, whatever the
        // device lengths are when the kernels run
        const size_t recs = (size_t)B * max_splits * p.Qtot;
        const size_t o_ml = round_up(recs * D * sizeof(float), 256);
        const size_t o_plan = round_up(o_ml + recs * 2 * sizeof(float), 256);
        const size_t need = o_plan + (B + 1) * sizeof(int);
        if (need > scratch_bytes)
            return fail(KVQ_ERANGE, "this decode needs %zu bytes of scratch, the no-alloc entry point holds %zu",
                        need, scratch_bytes);
        p.part_o = reinterpret_cast<float*>(scratch);
        p.part_ml = reinterpret_cast<float*>(scratch + o_ml);
        p.plan = reinterpret_cast<int*>(scratch + o_plan);
    } else {
        p.part_o = reinterpret_cast<float*>(c->ws + c->off_part_o);
        p.part_ml = reinterpret_cast<float*>(c->ws + c->off_part_ml);
        p.plan = reinterpret_cast<int*>(c->ws + c->off_plan);
    }
    // a tile is staged as the 16-byte aligned superset of its rows' bytes
    p.k_stage_bytes = (uint32_t)round_up((size_t)kTileRows * c->k_tok + 32, 128);
    p.stage_bytes = p.k_stage_bytes + (uint32_t)round_up((size_t)kTileRows * c->v_tok + 32, 128);
    const int smem_max = split_max_smem();
    p.nstage = 4;
    while (p.nstage > 2 && split_smem_bytes(p) > (size_t)smem_max) --p.nstage;
    if (split_smem_bytes(p) > (size_t)smem_max)
        return fail(KVQ_EUNSUPPORTED, "decode tile does not fit shared memory (%zu bytes)", split_smem_bytes(p));
    long long items = 0;
    for (int b = 0; b < B; ++b) {
        const int vis = c->len[b] - vis_lo(c, c->len[b], T);
        items += (vis + C - 1) / C;
    }
    items *= p.nqs;
    const int grid = (int)std::max(1LL, std::min<long long>(items, c->num_sms));
    cudaError_t e = launch_split(p, grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode split kernel");
    MergeParams m;
    m.part_o = p.part_o;
    m.part_ml = p.part_ml;
    m.plan = p.plan;
    m.sinks = sinks;
    m.out = out;
    m.B = B;
    m.Hq = n_q_heads;
    m.Qtot = p.Qtot;
    m.D = D;
    e = launch_merge(m, T, max_splits, true, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode merge kernel");
    return KVQ_OK;
}

kvq_status kvq_decode(kvq_cache* c, const void* q, kvq_dtype dtype, int T, int n_q_heads, const float* sinks,
                      float scale, float* out, void* stream) {
    return decode_impl(c, q, dtype, T, n_q_heads, sinks, scale, out, stream, nullptr, 0);
}

// Decode scratch of kvq_decode_noalloc: one file-scope device array per
// device (the module's copy on each device).  Its address is resolved with
// that device current the first time, and again whenever the device's current
// context is a different one (after cudaDeviceReset the module is loaded anew
// and the array may move).
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

static void* current_context() {
    using GetCurrent = CUresult (*)(CUcontext*);
    static GetCurrent get = nullptr;
    if (!get) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        get = reinterpret_cast<GetCurrent>(fn);
    }
    CUcontext ctx = nullptr;
    return get(&ctx) == CUDA_SUCCESS ? static_cast<void*>(ctx) : nullptr;
}

kvq_status kvq_decode_noalloc(kvq_cache* c, const void* q, kvq_dtype dtype, int T, int n_q_heads,
                              const float* sinks, float scale, float* out, void* stream) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static void* ctx_of[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KVQ_EUNSUPPORTED, "device %d beyond %d devices", dev, kMaxDevices);
    void* ctx = current_context();
    void* a = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!addr[dev] || ctx_of[dev] != ctx) {
            e = cudaGetSymbolAddress(&addr[dev], g_noalloc_scratch);
            if (e != cudaSuccess) {
                addr[dev] = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress of the no-alloc scratch");
            }
            ctx_of[dev] = ctx;
        }
        a = addr[dev];
    }
    return decode_impl(c, q, dtype, T, n_q_heads, sinks, scale, out, stream, static_cast<unsigned char*>(a),
                       KVQ_NOALLOC_SCRATCH_BYTES);
}

kvq_status kvq_truncate(kvq_cache* c, const int* new_len, void* stream) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (!new_len) return fail(KVQ_EINVAL, "new_len is NULL");
    const int B = c->cfg.n_seq;
    for (int b = 0; b < B; ++b) {
        const int n = new_len[b];
        if (n < 0 || n > c->len_lo[b])
            return fail(KVQ_ERANGE, "sequence %d: new length %d outside [0, %d]%s", b, n, c->len_lo[b],
                        c->len_lo[b] != c->len[b] ? " (a device-side rollback is pending: kvq_sync_len)" : "");
        if (c->cfg.ring && std::max(0, n + 1 - c->cfg.window) < c->base[b])
            return fail(KVQ_ERANGE, "sequence %d: rows below ring base %d are gone", b, c->base[b]);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    SeqIds sid;
    for (int first = 0; first < B; first += kMaxIdsPerLaunch) {
        const int n = std::min(B - first, kMaxIdsPerLaunch);
        sid.n = n;
        sid.identity = 1;
        sid.first = first;
        cudaError_t e = launch_set_len(c->len_d, sid, new_len + first, s);
        if (e != cudaSuccess) return cuda_fail(e, "truncate kernel");
    }
    for (int b = 0; b < B; ++b) c->len[b] = c->len_lo[b] = new_len[b];
    return KVQ_OK;
}

kvq_status kvq_truncate_device(kvq_cache* c, const int* accept_d, int T, void* stream) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (!accept_d) return fail(KVQ_EINVAL, "accept_d is NULL");
    if (T < 1 || T > c->cfg.max_t) return fail(KVQ_EINVAL, "T=%d outside [1, max_t=%d]", T, c->cfg.max_t);
    const int B = c->cfg.n_seq;
    for (int b = 0; b < B; ++b) {
        if (c->len_lo[b] < T)
            return fail(KVQ_ERANGE, "sequence %d may hold fewer than T=%d rows", b, T);
        // the shortest outcome (nothing accepted) must keep its window resident
        if (c->cfg.ring && std::max(0, c->len_lo[b] - T + 1 - c->cfg.window) < c->base[b])
            return fail(KVQ_ERANGE, "sequence %d: rolling back T=%d rows would reach below ring base %d", b, T,
                        c->base[b]);
    }
    cudaError_t e = launch_truncate_accept(c->len_d, c->base_d, c->err_d, accept_d, B, T, c->cfg.window,
                                           c->cfg.ring, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "device-side truncate kernel");
    for (int b = 0; b < B; ++b) c->len_lo[b] -= T;
    return KVQ_OK;
}

kvq_status kvq_sync_len(kvq_cache* c, void* stream) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    const int B = c->cfg.n_seq;
    std::vector<int> v(B);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(v.data(), c->len_d, sizeof(int) * (size_t)B, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read lengths");
    for (int b = 0; b < B; ++b)
        if (v[b] < c->base[b] || v[b] - c->base[b] > c->rows)
            return fail(KVQ_ERANGE, "sequence %d: device length %d outside its resident rows", b, v[b]);
    for (int b = 0; b < B; ++b) c->len[b] = c->len_lo[b] = v[b];
    return KVQ_OK;
}

kvq_status kvq_get_len(const kvq_cache* c, int* len_host, int* base_host) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    for (int b = 0; b < c->cfg.n_seq; ++b) {
        if (len_host) len_host[b] = c->len[b];
        if (base_host) base_host[b] = c->base[b];
    }
    return KVQ_OK;
}

kvq_status kvq_note_replayed(kvq_cache* c, int steps, int T) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (steps < 0 || T < 1 || T > c->cfg.max_t) return fail(KVQ_EINVAL, "bad steps or T");
    const long long add = (long long)steps * T;
    for (int b = 0; b < c->cfg.n_seq; ++b)
        if (c->len[b] + add - c->base[b] > c->rows)
            return fail(KVQ_ERANGE, "sequence %d would exceed its physical rows", b);
    for (int b = 0; b < c->cfg.n_seq; ++b) {
        c->len[b] += (int)add;
        c->len_lo[b] += (int)add;
    }
    return KVQ_OK;
}

kvq_status kvq_ring_headroom(const kvq_cache* c, int T, int* steps) {
    if (!c || !steps) return fail(KVQ_EINVAL, "NULL argument");
    if (T < 1 || T > c->cfg.max_t) return fail(KVQ_EINVAL, "bad T");
    long long best = 0x7fffffff;
    for (int b = 0; b < c->cfg.n_seq; ++b) {
        const long long room = (long long)c->rows - (c->len[b] - c->base[b]);
        best = std::min(best, room / T);
    }
    *steps = (int)std::max(0LL, best);
    return KVQ_OK;
}

kvq_status kvq_physical_rows(const kvq_cache* c, int seq, int start, int end, int* phys_start, int* phys_end) {
    if (!c || !phys_start || !phys_end) return fail(KVQ_EINVAL, "NULL argument");
    if (seq < 0 || seq >= c->cfg.n_seq) return fail(KVQ_EINVAL, "sequence index out of range");
    if (start < 0 || end < start) return fail(KVQ_ERANGE, "bad logical range");
    const int base = c->base[seq];
    if (start < base || end - base > c->rows)
        return fail(KVQ_ERANGE, "logical rows [%d, %d) not resident (base %d, %d physical rows)", start, end, base,
                    c->rows);
    *phys_start = start - base;
    *phys_end = end - base;
    return KVQ_OK;
}

kvq_status kvq_read_device_error(kvq_cache* c, int* err, void* stream) {
    if (!c || !err) return fail(KVQ_EINVAL, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(err, c->err_d, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    e = cudaMemset(c->err_d, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
    return KVQ_OK;
}

kvq_status kvq_set_softcap(kvq_cache* c, float softcap) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (!(softcap >= 0.f) || softcap > 3.0e38f) return fail(KVQ_EINVAL, "softcap must be finite and >= 0");
    c->softcap = softcap;
    return KVQ_OK;
}

kvq_status kvq_set_decode_path(kvq_cache* c, int path, int query_bits) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (path < 0 || path > 2) return fail(KVQ_EINVAL, "path must be 0, 1 or 2");
    if (query_bits != 0 && query_bits != 16 && query_bits != 24)
        return fail(KVQ_EINVAL, "query_bits must be 0, 16 or 24");
    c->path = path;
    c->qbits = query_bits == 24 ? 24 : 16;
    return KVQ_OK;
}

kvq_status kvq_set_row_slices(kvq_cache* c, int slices) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (slices < 0 || slices > 2) return fail(KVQ_EINVAL, "row slices must be 0, 1 or 2");
    c->row_slices = slices;
    return KVQ_OK;
}

kvq_status kvq_set_split_rows(kvq_cache* c, int rows) {
    if (!c) return fail(KVQ_EINVAL, "cache is NULL");
    if (rows != 0 && (rows < kMinSplitRows || rows % 8))
        return fail(KVQ_EINVAL, "split rows must be 0 or a multiple of 8 that is >= %d", kMinSplitRows);
    c->split_rows = rows;
    return KVQ_OK;
}

}  // extern "C"
