// api.cu -- the C ABI declared in include/gemma_attn.h: host-side validation, owner-layer
// resolution, the split plan of the decode bucket, and kernel launches. Nothing here
// allocates memory or synchronises; every launch goes to the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/gemma_attn.h"
#include "attn_internal.h"
#include "logits.h"

using gemma::RowsParams;

namespace {

constexpr int kMaxSplit = 128;
#ifndef GEMMA_MIN_CHUNK_KEYS
#define GEMMA_MIN_CHUNK_KEYS 256
#endif
#ifndef GEMMA_SPLIT_CTAS_PER_SM
#define GEMMA_SPLIT_CTAS_PER_SM 8
#endif
constexpr int kMinChunkKeys = GEMMA_MIN_CHUNK_KEYS;  // keys per split chunk when work is plentiful
// no split when the (sequence, KV head) units alone fill the GPU (at least this many per SM)
// and each attends a short key range: one CTA per unit, no partials, no combine launch
constexpr long long kNoSplitUnitsPerSm = 2;
constexpr long long kNoSplitMaxKeys = 2048;
constexpr long long kSplitCtasPerSm = GEMMA_SPLIT_CTAS_PER_SM;

// SM count of the current device, cached per device (atomics: calls may come from several
// host threads; they all store the same value)
int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }
bool group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }
long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

int check_shape(int kind, int window, int n_q, int n_kv, int head_dim, int dtype) {
    if (kind != GEMMA_SLIDING && kind != GEMMA_GLOBAL && kind != GEMMA_SLIDING_RING)
        return GEMMA_ERR_INVALID_ARG;
    if (kind != GEMMA_GLOBAL && window < 1) return GEMMA_ERR_INVALID_ARG;
    if (n_q < 1 || n_kv < 1 || n_q % n_kv != 0) return GEMMA_ERR_INVALID_ARG;
    if (dtype != GEMMA_BF16 && dtype != GEMMA_FP32) return GEMMA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim) || !group_ok(n_q / n_kv)) return GEMMA_ERR_UNSUPPORTED;
    return GEMMA_OK;
}

// Owner resolution ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", section 2.1): a
// layer reads the cache of owner_map[layer], an earlier layer that owns its cache.
int resolve_owner(const int32_t* owner_map, int n_layers, int layer, int* owner) {
    if (!owner_map || n_layers < 1 || layer < 0 || layer >= n_layers) return GEMMA_ERR_INVALID_ARG;
    const int o = owner_map[layer];
    if (o < 0 || o > layer || owner_map[o] != o) return GEMMA_ERR_INVALID_ARG;
    *owner = o;
    return GEMMA_OK;
}

struct Plan {
    int n_split;
    int chunk;
    size_t o_bytes;   // partial outputs
    size_t ws_bytes;  // total scratch
    int cluster;      // the chunks of a row tile merge inside their cluster (no scratch)
};

// Splits of at most this many chunks run as one thread-block cluster per (sequence, KV head)
// and merge through distributed shared memory; plans of up to twice as many chunks are
// coarsened to it (one launch and no scratch beat twice the CTAs plus a combine pass). When all
// CTAs of a plan of up to kMaxBigClusterSplit chunks fit on the GPU at once (one per SM), a
// latency-bound small batch, the plan keeps its chunks and runs as clusters of that many (above
// the portable cluster size; fewer keys per CTA matter more there than the wider merge).
constexpr int kMaxClusterSplit = 8;
constexpr int kMaxBigClusterSplit = 16;
// A latency-bound plan finer than the largest cluster is coarsened to one cluster of
// kMaxBigClusterSplit chunks (no combine launch) while each chunk stays at most this many keys
// (a few key tiles per CTA; longer chunks cost more per CTA than the combine pass saves).
constexpr long long kBigClusterMaxKeys = 128;

// Decode splits each (sequence, KV head) key range into chunks so that enough CTAs stream
// the cache at once: about one chunk per SM for small problems, about eight per SM (and at
// least kMinChunkKeys keys each) for large ones; not at all when the units alone fill the GPU
// over short key ranges (a sliding window across a large batch). Prefill has one row tile per 16 rows and no
// split. Depends only on the arguments and the SM count.
Plan make_plan(int batch, int kind, int window, int n_q, int n_kv, int head_dim, int max_seq_len,
               int n_tok, int n_sm, bool paged = false) {
    Plan pl{1, 1 << 30, 0, 0, 0};
    if (n_tok != 1) return pl;
    const long long T = gemma::kKeyTile;
    long long n_read = kind != GEMMA_GLOBAL && window < max_seq_len ? window : max_seq_len;
    // a ring cache's or paged pool's key tiles start at multiples of the tile (so that none wraps
    // or crosses a page): up to T - 1 keys before the window join the range
    if (kind == GEMMA_SLIDING_RING || paged) n_read += T - 1;
    if ((long long)batch * n_kv >= kNoSplitUnitsPerSm * n_sm && n_read <= kNoSplitMaxKeys) return pl;
    const long long total = (long long)batch * n_kv * n_read;
    const long long one_per_sm = round_up((total + n_sm - 1) / n_sm, T);
    const long long eight_per_sm =
        round_up((total + kSplitCtasPerSm * n_sm - 1) / (kSplitCtasPerSm * n_sm), T);
    long long chunk = one_per_sm < kMinChunkKeys ? one_per_sm : kMinChunkKeys;
    if (eight_per_sm > chunk) chunk = eight_per_sm;
    if (chunk < T) chunk = T;
    long long n_split = (n_read + chunk - 1) / chunk;
    if (n_split > kMaxSplit) {
        chunk = round_up((n_read + kMaxSplit - 1) / kMaxSplit, T);
        n_split = (n_read + chunk - 1) / chunk;
    }
    if (n_split <= 1) return pl;
    if (n_split <= kMaxBigClusterSplit && (long long)batch * n_kv * n_split <= n_sm) {
        pl.n_split = (int)n_split;
        pl.chunk = (int)chunk;
        pl.cluster = 1;
        return pl;
    }
    if (n_split > kMaxBigClusterSplit && (long long)batch * n_kv * kMaxBigClusterSplit <= n_sm &&
        n_read <= kMaxBigClusterSplit * kBigClusterMaxKeys) {
        chunk = round_up((n_read + kMaxBigClusterSplit - 1) / kMaxBigClusterSplit, T);
        n_split = (n_read + chunk - 1) / chunk;
        pl.n_split = (int)n_split;
        pl.chunk = (int)chunk;
        pl.cluster = 1;
        return pl;
    }
    if (n_split <= 2 * kMaxClusterSplit) {
        if (n_split > kMaxClusterSplit) {
            chunk = round_up((n_read + kMaxClusterSplit - 1) / kMaxClusterSplit, T);
            n_split = (n_read + chunk - 1) / chunk;
        }
        pl.n_split = (int)n_split;
        pl.chunk = (int)chunk;
        pl.cluster = 1;
        return pl;
    }
    pl.n_split = (int)n_split;
    pl.chunk = (int)chunk;
    const size_t rows = (size_t)batch * n_q * n_split;
    pl.o_bytes = (size_t)round_up((long long)(rows * head_dim * sizeof(float)), 256);
    pl.ws_bytes = pl.o_bytes + (size_t)round_up((long long)(rows * 2 * sizeof(float)), 256);
    return pl;
}

int attention(void* out, const void* q, const void* const* k_cache, const void* const* v_cache,
              const int32_t* owner_map, int n_layers, int layer, const int32_t* seq_lens,
              int max_seq_len, int n_tok, int batch, int kind, int window, int n_q, int n_kv,
              int head_dim, int k_eq_v, int kv_capacity, float scale, float softcap, int dtype,
              void* workspace, size_t workspace_bytes, uint32_t* device_error, void* stream,
              const int32_t* n_real = nullptr, const void* k_new = nullptr,
              const void* v_new = nullptr, const int32_t* write_pos = nullptr,
              const gemma::PagedLayout* pg = nullptr) {
    if (batch < 0 || n_tok < 1) return GEMMA_ERR_INVALID_ARG;
    if (pg) {  // paged pool: a multiple of 128 keys per page, so that no key tile crosses a page
        if (kind == GEMMA_SLIDING_RING || pg->page_size < 128 || pg->page_size % 128 != 0 ||
            pg->max_pages < 1 || pg->n_pages < 1)
            return pg->page_size > 0 && pg->page_size % 128 != 0 ? GEMMA_ERR_UNSUPPORTED
                                                                  : GEMMA_ERR_INVALID_ARG;
        if ((long long)pg->max_pages * pg->page_size > (1ll << 30) ||
            (long long)pg->n_pages * n_kv > (1ll << 31) - 1)
            return GEMMA_ERR_UNSUPPORTED;
        if (batch > 0 && !pg->block_table) return GEMMA_ERR_INVALID_ARG;
        kv_capacity = pg->max_pages * pg->page_size;  // logical capacity of a sequence
    }
    if (!std::isfinite(softcap) || softcap < 0.f) return GEMMA_ERR_INVALID_ARG;
    int st = check_shape(kind, window, n_q, n_kv, head_dim, dtype);
    if (st != GEMMA_OK) return st;
    int o = 0;
    st = resolve_owner(owner_map, n_layers, layer, &o);
    if (st != GEMMA_OK) return st;
    if (kv_capacity < 1 || max_seq_len < n_tok || !std::isfinite(scale) || !(scale > 0.f))
        return GEMMA_ERR_INVALID_ARG;
    const bool ring = kind == GEMMA_SLIDING_RING;
    if (ring) {
        if (kv_capacity % 128 != 0) return GEMMA_ERR_UNSUPPORTED;
        if ((long long)kv_capacity < (long long)window + n_tok - 1) return GEMMA_ERR_CAPACITY;
    } else if (max_seq_len > kv_capacity) {
        return GEMMA_ERR_CAPACITY;
    }
    if (batch > 65535) return GEMMA_ERR_UNSUPPORTED;
    if (batch == 0) return GEMMA_OK;
    if (!out || !q || !seq_lens || !k_cache || !k_cache[o]) return GEMMA_ERR_INVALID_ARG;
    const void* kc = k_cache[o];
    const void* vc = kc;
    if (!k_eq_v) {
        if (!v_cache || !v_cache[o]) return GEMMA_ERR_INVALID_ARG;
        vc = v_cache[o];
    }
    if (!aligned16(out) || !aligned16(q) || !aligned16(kc) || !aligned16(vc))
        return GEMMA_ERR_INVALID_ARG;
    const int n_sm = sm_count();
    if (n_sm < 0) return GEMMA_ERR_CUDA;
    // a padded bucket is never split over keys (pad rows have no key range to merge)
    Plan pl = n_real ? Plan{1, 1 << 30, 0, 0, 0}
                           : make_plan(batch, kind, window, n_q, n_kv, head_dim, max_seq_len,
                                       n_tok, n_sm, pg != nullptr);
    if (pl.ws_bytes > 0 &&
        (!workspace || workspace_bytes < pl.ws_bytes || !aligned16(workspace)))
        return GEMMA_ERR_WORKSPACE;

    RowsParams p{};
    p.q = q;
    p.k = kc;
    p.v = vc;
    p.seq_lens = seq_lens;
    p.n_real = n_real;
    p.k_new = k_new;
    p.v_new = v_new;
    p.write_pos = write_pos;
    p.out = out;
    p.o_part = pl.ws_bytes ? static_cast<float*>(workspace) : nullptr;
    p.ml_part = pl.ws_bytes
                    ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.o_bytes)
                    : nullptr;
    p.err = device_error;
    p.n_tok = n_tok;
    p.n_q = n_q;
    p.n_kv = n_kv;
    p.G = n_q / n_kv;
    p.cap = kv_capacity;
    p.window = window;
    p.is_sliding = kind != GEMMA_GLOBAL;
    p.ring = ring ? kv_capacity : 0;
    if (pg) {
        p.block_table = pg->block_table;
        p.page_size = pg->page_size;
        p.max_pages = pg->max_pages;
        p.n_pages = pg->n_pages;
    }
    p.k_eq_v = k_eq_v ? 1 : 0;
    p.max_seq_len = max_seq_len;
    if (pl.cluster && dtype != GEMMA_BF16) {
        // the fp32 debug path does not split a clustered plan: one pass per row
        pl.n_split = 1;
        pl.chunk = 1 << 30;
        pl.cluster = 0;
    }
    p.n_split = pl.n_split;
    p.chunk = pl.chunk;
    p.cluster = pl.cluster;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.softcap = softcap;
    p.cap_inner = softcap > 0.f ? scale / softcap : 0.f;
    p.cap_log2 = softcap * 1.4426950408889634f;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = (long long)n_tok * p.G;
    cudaError_t e;
    if (dtype == GEMMA_BF16 && (n_tok > 1 || n_real) && gemma::prefill_tc_supported(head_dim)) {
        e = gemma::launch_prefill_tc(p, head_dim, batch, s);
    } else if (dtype == GEMMA_BF16) {
        const size_t smem = gemma::rows_bf16_smem_bytes(head_dim, p.k_eq_v, &p.n_stages);
        const long long tiles = (rows + gemma::kRowTile - 1) / gemma::kRowTile;
        e = gemma::launch_rows_bf16(p, head_dim, dim3((unsigned)(tiles * pl.n_split), n_kv, batch),
                                    smem, s);
    } else {
        const long long tiles = (rows + gemma::kF32RowsPerCta - 1) / gemma::kF32RowsPerCta;
        e = gemma::launch_rows_f32(p, head_dim, dim3((unsigned)(tiles * pl.n_split), n_kv, batch),
                                   s);
    }
    if (e == cudaSuccess && pl.n_split > 1 && !pl.cluster)
        e = gemma::launch_combine(p, head_dim, batch, dtype == GEMMA_FP32, s);
    return e == cudaSuccess ? GEMMA_OK : GEMMA_ERR_CUDA;
}

int append_rows(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                int n_layers, int layer, const void* k_new, const void* v_new,
                const int32_t* write_pos, const int32_t* n_real, int ring, int batch, int n_new,
                int n_kv, int head_dim, int kv_capacity, int k_eq_v, gemma_dtype dtype,
                uint32_t* device_error, void* stream,
                const gemma::PagedLayout& pg = gemma::PagedLayout{nullptr, 0, 0, 0});

}  // namespace

extern "C" {

int gemma_abi_version(void) { return 1; }

const char* gemma_status_string(int status) {
    switch (status) {
        case GEMMA_OK: return "GEMMA_OK";
        case GEMMA_ERR_INVALID_ARG: return "GEMMA_ERR_INVALID_ARG";
        case GEMMA_ERR_UNSUPPORTED: return "GEMMA_ERR_UNSUPPORTED";
        case GEMMA_ERR_CAPACITY: return "GEMMA_ERR_CAPACITY";
        case GEMMA_ERR_WORKSPACE: return "GEMMA_ERR_WORKSPACE";
        case GEMMA_ERR_CUDA: return "GEMMA_ERR_CUDA";
    }
    return "GEMMA_UNKNOWN_STATUS";
}

int gemma_kv_append(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                    int n_layers, int layer, const void* k_new, const void* v_new,
                    const int32_t* write_pos, int batch, int n_new, int n_kv, int head_dim,
                    int kv_capacity, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                    void* stream) {
    return append_rows(k_cache, v_cache, owner_map, n_layers, layer, k_new, v_new, write_pos,
                       nullptr, 0, batch, n_new, n_kv, head_dim, kv_capacity, k_eq_v, dtype,
                       device_error, stream);
}

int gemma_kv_append_ring(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                         int n_layers, int layer, const void* k_new, const void* v_new,
                         const int32_t* write_pos, int batch, int n_new, int n_kv, int head_dim,
                         int kv_capacity, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                         void* stream) {
    return append_rows(k_cache, v_cache, owner_map, n_layers, layer, k_new, v_new, write_pos,
                       nullptr, kv_capacity, batch, n_new, n_kv, head_dim, kv_capacity, k_eq_v,
                       dtype, device_error, stream);
}

int gemma_kv_append_bucket(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                           int n_layers, int layer, const void* k_new, const void* v_new,
                           const int32_t* write_pos, const int32_t* n_real, int batch, int n_new,
                           int n_kv, int head_dim, int kv_capacity, int k_eq_v, gemma_dtype dtype,
                           uint32_t* device_error, void* stream) {
    if (!n_real && batch > 0 && n_new > 0) return GEMMA_ERR_INVALID_ARG;
    return append_rows(k_cache, v_cache, owner_map, n_layers, layer, k_new, v_new, write_pos,
                       n_real, 0, batch, n_new, n_kv, head_dim, kv_capacity, k_eq_v, dtype,
                       device_error, stream);
}

}  // extern "C"

namespace {

int append_rows(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                int n_layers, int layer, const void* k_new, const void* v_new,
                const int32_t* write_pos, const int32_t* n_real, int ring, int batch, int n_new,
                int n_kv, int head_dim, int kv_capacity, int k_eq_v, gemma_dtype dtype,
                uint32_t* device_error, void* stream, const gemma::PagedLayout& pg) {
    if (batch < 0 || n_new < 0 || n_kv < 1 || kv_capacity < 1) return GEMMA_ERR_INVALID_ARG;
    if (dtype != GEMMA_BF16 && dtype != GEMMA_FP32) return GEMMA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim)) return GEMMA_ERR_UNSUPPORTED;
    int o = 0;
    int st = resolve_owner(owner_map, n_layers, layer, &o);
    if (st != GEMMA_OK) return st;
    if (o != layer) return GEMMA_OK;  // a shared layer writes no cache
    if (n_new > kv_capacity) return GEMMA_ERR_CAPACITY;
    if (batch == 0 || n_new == 0) return GEMMA_OK;
    if (!k_cache || !k_cache[layer] || !k_new || !write_pos) return GEMMA_ERR_INVALID_ARG;
    void* vc = nullptr;
    if (!k_eq_v) {
        if (!v_cache || !v_cache[layer] || !v_new) return GEMMA_ERR_INVALID_ARG;
        vc = v_cache[layer];
    }
    if (!aligned16(k_cache[layer]) || !aligned16(k_new) ||
        (vc && (!aligned16(vc) || !aligned16(v_new))))
        return GEMMA_ERR_INVALID_ARG;
    const int n_sm = sm_count();
    if (n_sm < 0) return GEMMA_ERR_CUDA;
    const int row_bytes = head_dim * (dtype == GEMMA_BF16 ? 2 : 4);
    cudaError_t e = gemma::launch_kv_append(k_cache[layer], vc, k_new, vc ? v_new : nullptr,
                                            write_pos, n_real, ring, pg, batch, n_new, n_kv,
                                            kv_capacity,
                                            row_bytes, device_error, n_sm,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GEMMA_OK : GEMMA_ERR_CUDA;
}

}  // namespace

extern "C" {

int gemma_attn_decode(void* out, const void* q, const void* const* k_cache,
                      const void* const* v_cache, const int32_t* owner_map, int n_layers,
                      int layer, const int32_t* seq_lens, int max_seq_len, int batch,
                      gemma_layer_kind kind, int window, int n_q, int n_kv, int head_dim,
                      int k_eq_v, int kv_capacity, float scale, gemma_dtype dtype,
                      void* workspace, size_t workspace_bytes, uint32_t* device_error,
                      void* stream) {
    return attention(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens, max_seq_len,
                     1, batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale, 0.f,
                     dtype, workspace, workspace_bytes, device_error, stream);
}

int gemma_attn_prefill(void* out, const void* q, const void* const* k_cache,
                       const void* const* v_cache, const int32_t* owner_map, int n_layers,
                       int layer, const int32_t* seq_lens, int max_seq_len, int n_new,
                       int batch, gemma_layer_kind kind, int window, int n_q, int n_kv,
                       int head_dim, int k_eq_v, int kv_capacity, float scale,
                       gemma_dtype dtype, void* workspace, size_t workspace_bytes,
                       uint32_t* device_error, void* stream) {
    if (n_new == 0 && batch >= 0) return GEMMA_OK;
    return attention(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens, max_seq_len,
                     n_new, batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale,
                     0.f, dtype, workspace, workspace_bytes, device_error, stream);
}

int gemma_attn_softcap(void* out, const void* q, const void* const* k_cache,
                       const void* const* v_cache, const int32_t* owner_map, int n_layers,
                       int layer, const int32_t* seq_lens, int max_seq_len, int n_new,
                       int batch, gemma_layer_kind kind, int window, int n_q, int n_kv,
                       int head_dim, int k_eq_v, int kv_capacity, float scale, float softcap,
                       gemma_dtype dtype, void* workspace, size_t workspace_bytes,
                       uint32_t* device_error, void* stream) {
    if (n_new == 0 && batch >= 0) return GEMMA_OK;
    return attention(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens, max_seq_len,
                     n_new, batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale,
                     softcap, dtype, workspace, workspace_bytes, device_error, stream);
}

int gemma_attn_decode_append(void* out, const void* q, void* const* k_cache, void* const* v_cache,
                             const int32_t* owner_map, int n_layers, int layer, const void* k_new,
                             const void* v_new, const int32_t* write_pos,
                             const int32_t* seq_lens, int max_seq_len, int batch,
                             gemma_layer_kind kind, int window, int n_q, int n_kv, int head_dim,
                             int k_eq_v, int kv_capacity, float scale, gemma_dtype dtype,
                             void* workspace, size_t workspace_bytes, uint32_t* device_error,
                             void* stream) {
    int o = 0;
    int st = resolve_owner(owner_map, n_layers, layer, &o);
    if (st != GEMMA_OK) return st;
    const void* const* kcc = const_cast<const void* const*>(k_cache);
    const void* const* vcc = const_cast<const void* const*>(v_cache);
    if (o != layer)  // a shared layer appends nothing: plain decode against the owner's cache
        return attention(out, q, kcc, vcc, owner_map, n_layers, layer, seq_lens, max_seq_len, 1,
                         batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale,
                         0.f, dtype, workspace, workspace_bytes, device_error, stream);
    if (batch > 0 && (!k_new || !write_pos || (!k_eq_v && !v_new))) return GEMMA_ERR_INVALID_ARG;
    if (batch > 0 && (!aligned16(k_new) || (!k_eq_v && !aligned16(v_new))))
        return GEMMA_ERR_INVALID_ARG;
    if (dtype != GEMMA_BF16) {
        // the fp32 debug path keeps two launches: append, then attend
        st = append_rows(k_cache, v_cache, owner_map, n_layers, layer, k_new, v_new, write_pos,
                         nullptr, kind == GEMMA_SLIDING_RING ? kv_capacity : 0, batch, 1, n_kv,
                         head_dim, kv_capacity, k_eq_v, dtype, device_error, stream);
        if (st != GEMMA_OK) return st;
        return attention(out, q, kcc, vcc, owner_map, n_layers, layer, seq_lens, max_seq_len, 1,
                         batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale,
                         0.f, dtype, workspace, workspace_bytes, device_error, stream);
    }
    return attention(out, q, kcc, vcc, owner_map, n_layers, layer, seq_lens, max_seq_len, 1, batch,
                     kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale, 0.f, dtype,
                     workspace, workspace_bytes, device_error, stream, nullptr, k_new,
                     k_eq_v ? nullptr : v_new, write_pos);
}

namespace {
int check_paged(int max_pages, int page_size, int n_pages) {
    if (page_size > 0 && page_size % 128 != 0) return GEMMA_ERR_UNSUPPORTED;
    if (page_size < 128 || max_pages < 1 || n_pages < 1) return GEMMA_ERR_INVALID_ARG;
    if ((long long)max_pages * page_size > (1ll << 30)) return GEMMA_ERR_UNSUPPORTED;
    return GEMMA_OK;
}
}  // namespace

int gemma_kv_append_paged(void* const* k_pool, void* const* v_pool, const int32_t* owner_map,
                          int n_layers, int layer, const void* k_new, const void* v_new,
                          const int32_t* write_pos, const int32_t* block_table, int max_pages,
                          int page_size, int n_pages, int batch, int n_new, int n_kv,
                          int head_dim, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                          void* stream) {
    const int st = check_paged(max_pages, page_size, n_pages);
    if (st != GEMMA_OK) return st;
    if (batch > 0 && n_new > 0 && !block_table) return GEMMA_ERR_INVALID_ARG;
    const gemma::PagedLayout pg{block_table, max_pages, page_size, n_pages};
    return append_rows(k_pool, v_pool, owner_map, n_layers, layer, k_new, v_new, write_pos,
                       nullptr, 0, batch, n_new, n_kv, head_dim, max_pages * page_size, k_eq_v,
                       dtype, device_error, stream, pg);
}

int gemma_attn_paged(void* out, const void* q, void* const* k_pool, void* const* v_pool,
                     const int32_t* owner_map, int n_layers, int layer, const int32_t* seq_lens,
                     const int32_t* block_table, int max_pages, int page_size, int n_pages,
                     int max_seq_len, int n_new, int batch, gemma_layer_kind kind, int window,
                     int n_q, int n_kv, int head_dim, int k_eq_v, float scale, gemma_dtype dtype,
                     const void* k_new, const void* v_new, const int32_t* write_pos,
                     void* workspace, size_t workspace_bytes, uint32_t* device_error,
                     void* stream) {
    if (n_new == 0 && batch >= 0) return GEMMA_OK;
    int st = check_paged(max_pages, page_size, n_pages);
    if (st != GEMMA_OK) return st;
    const gemma::PagedLayout pg{block_table, max_pages, page_size, n_pages};
    const void* const* kcc = const_cast<const void* const*>(k_pool);
    const void* const* vcc = const_cast<const void* const*>(v_pool);
    int o = 0;
    st = resolve_owner(owner_map, n_layers, layer, &o);
    if (st != GEMMA_OK) return st;
    if (k_new && o == layer) {  // this step's rows are written by the decode launch itself
        if (n_new != 1) return GEMMA_ERR_INVALID_ARG;
        if (batch > 0 && (!write_pos || (!k_eq_v && !v_new))) return GEMMA_ERR_INVALID_ARG;
        if (batch > 0 && (!aligned16(k_new) || (!k_eq_v && !aligned16(v_new))))
            return GEMMA_ERR_INVALID_ARG;
        if (dtype != GEMMA_BF16) {  // the fp32 debug path: append, then attend
            st = append_rows(k_pool, v_pool, owner_map, n_layers, layer, k_new, v_new, write_pos,
                             nullptr, 0, batch, 1, n_kv, head_dim, max_pages * page_size, k_eq_v,
                             dtype, device_error, stream, pg);
            if (st != GEMMA_OK) return st;
        } else {
            return attention(out, q, kcc, vcc, owner_map, n_layers, layer, seq_lens, max_seq_len,
                             1, batch, kind, window, n_q, n_kv, head_dim, k_eq_v, 0, scale, 0.f,
                             dtype, workspace, workspace_bytes, device_error, stream, nullptr,
                             k_new, k_eq_v ? nullptr : v_new, write_pos, &pg);
        }
    }
    return attention(out, q, kcc, vcc, owner_map, n_layers, layer, seq_lens, max_seq_len, n_new,
                     batch, kind, window, n_q, n_kv, head_dim, k_eq_v, 0, scale, 0.f, dtype,
                     workspace, workspace_bytes, device_error, stream, nullptr, nullptr, nullptr,
                     nullptr, &pg);
}

size_t gemma_attn_workspace_size_paged(int batch, gemma_layer_kind kind, int window, int n_q,
                                       int n_kv, int head_dim, int max_seq_len, int n_new) {
    if (batch < 0 || n_new < 1 || max_seq_len < n_new || kind == GEMMA_SLIDING_RING)
        return (size_t)-1;
    if (check_shape(kind, window, n_q, n_kv, head_dim, GEMMA_BF16) != GEMMA_OK) return (size_t)-1;
    if (batch == 0) return 0;
    const int n_sm = sm_count();
    if (n_sm < 0) return (size_t)-1;
    return make_plan(batch, kind, window, n_q, n_kv, head_dim, max_seq_len, n_new, n_sm, true)
        .ws_bytes;
}

int gemma_attn_prefill_bucket(void* out, const void* q, const void* const* k_cache,
                              const void* const* v_cache, const int32_t* owner_map, int n_layers,
                              int layer, const int32_t* seq_lens, const int32_t* n_real,
                              int max_seq_len, int n_new, int batch, gemma_layer_kind kind,
                              int window, int n_q, int n_kv, int head_dim, int k_eq_v,
                              int kv_capacity, float scale, gemma_dtype dtype, void* workspace,
                              size_t workspace_bytes, uint32_t* device_error, void* stream) {
    if (n_new == 0 && batch >= 0) return GEMMA_OK;
    if (!n_real && batch > 0) return GEMMA_ERR_INVALID_ARG;
    return attention(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens, max_seq_len,
                     n_new, batch, kind, window, n_q, n_kv, head_dim, k_eq_v, kv_capacity, scale,
                     0.f, dtype, workspace, workspace_bytes, device_error, stream, n_real);
}

size_t gemma_attn_workspace_size(int batch, gemma_layer_kind kind, int window, int n_q,
                                 int n_kv, int head_dim, int max_seq_len, int n_new) {
    if (batch < 0 || n_new < 1 || max_seq_len < n_new) return (size_t)-1;
    if (check_shape(kind, window, n_q, n_kv, head_dim, GEMMA_BF16) != GEMMA_OK) return (size_t)-1;
    if (batch == 0) return 0;
    const int n_sm = sm_count();
    if (n_sm < 0) return (size_t)-1;
    return make_plan(batch, kind, window, n_q, n_kv, head_dim, max_seq_len, n_new, n_sm).ws_bytes;
}

int gemma_logit_softcap_argmax(const void* logits, int batch, int vocab, gemma_dtype dtype,
                               float softcap, void* capped_out, int32_t* argmax_out,
                               void* workspace, size_t workspace_bytes, void* stream) {
    if (batch < 0 || vocab < 1 || (dtype != GEMMA_BF16 && dtype != GEMMA_FP32))
        return GEMMA_ERR_INVALID_ARG;
    if (!std::isfinite(softcap) || softcap < 0.f) return GEMMA_ERR_INVALID_ARG;
    if (batch == 0) return GEMMA_OK;
    if (batch > 65535) return GEMMA_ERR_UNSUPPORTED;  // one grid row per batch row
    if (!logits || !argmax_out || !aligned16(logits) || (capped_out && !aligned16(capped_out)))
        return GEMMA_ERR_INVALID_ARG;
    const int n_sm = sm_count();
    if (n_sm < 0) return GEMMA_ERR_CUDA;
    const gemma::LogitPlan pl = gemma::logit_plan(batch, vocab, n_sm);
    if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes || !aligned16(workspace)))
        return GEMMA_ERR_WORKSPACE;
    const cudaError_t e = gemma::launch_logit_softcap_argmax(
        logits, capped_out, argmax_out, workspace, batch, vocab, dtype == GEMMA_FP32, softcap, pl,
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GEMMA_OK : GEMMA_ERR_CUDA;
}

size_t gemma_logit_workspace_size(int batch, int vocab) {
    if (batch < 0 || vocab < 1) return (size_t)-1;
    if (batch == 0) return 0;
    const int n_sm = sm_count();
    if (n_sm < 0) return (size_t)-1;
    return gemma::logit_plan(batch, vocab, n_sm).ws_bytes;
}

}  // extern "C"
