// attn_internal.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gemma {

// One attention launch over "rows": a row is one (query token, query head) pair. Rows are
// ordered token-major, then by the head's index inside its GQA group, so a tile of rows
// shares one KV head. Decode has one token (rows = the G heads of a group); prefill has n_tok
// tokens per sequence.
struct RowsParams {
    const void* q;            // [B][n_tok][n_q][D]
    const void* k;            // owner layer's K cache [B][n_kv][cap][D]
    const void* v;            // owner layer's V cache (== k when k_eq_v)
    const int32_t* seq_lens;  // [B], tokens in the cache after this step's append
    const int32_t* n_real;    // [B] real tokens of a padded prefill bucket, or nullptr (all real)
    // fused append (decode): this step's K/V rows [B][1][n_kv][D] written into the cache at
    // write_pos[b] by the CTA that reads that slot; k_new == nullptr: no append
    const void* k_new;
    const void* v_new;
    const int32_t* write_pos;
    void* out;                // [B][n_tok][n_q][D], written when n_split == 1
    float* o_part;            // [B][n_q][n_split][D]  unnormalised partial outputs
    float* ml_part;           // [B][n_q][n_split][2]  (running max in log2 units, sum)
    uint32_t* err;            // optional device error word
    int n_tok, n_q, n_kv, G, cap, window, is_sliding, k_eq_v;
    int max_seq_len;
    int ring;                 // ring cache of this many slots (position p at p % ring), or 0
    // paged pool [n_pages][n_kv][page_size][D] (page_size > 0): position p of sequence b lives
    // in page block_table[b][p / page_size], row p % page_size; cap = max_pages * page_size
    const int32_t* block_table;
    int page_size, max_pages, n_pages;
    int n_split;              // key chunks per row tile (1: write `out` directly)
    // the n_split chunks of a row tile run as one thread-block cluster and merge their partial
    // results through distributed shared memory (no partials in global memory, no combine
    // pass); n_split <= 8
    int cluster;
    int chunk;                // keys per chunk (multiple of the key tile)
    int n_stages;             // smem pipeline depth (bf16 kernel)
    float scale_log2;         // softmax scale * log2(e)
    float scale;              // softmax scale
    // optional attention-logit soft-cap c (0: none): a scaled score s becomes c * tanh(s / c);
    // kernels evaluate it on the raw dot product r as cap_log2 * tanh(r * cap_inner), already
    // in log2 units (cap_inner = scale / c, cap_log2 = c * log2(e))
    float softcap;
    float cap_inner;
    float cap_log2;
};

#ifdef __CUDACC__
// Row of the [rows][slots][D] view of the cache that the tensor maps and direct accesses use,
// and slot, of key `key` of sequence b and KV head kvh: row b * n_kv + kvh and slot key (key %
// ring for a ring cache); for a paged pool row page * n_kv + kvh and slot key % page_size, page
// the sequence's block-table entry. Returns false for a page index outside [0, n_pages).
__device__ __forceinline__ bool kv_place(const RowsParams& p, int b, int kvh, int key, int& row,
                                         int& slot) {
    if (p.page_size) {
        const int blk = key / p.page_size;
        const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + blk);
        row = pg * p.n_kv + kvh;
        slot = key - blk * p.page_size;
        return pg >= 0 && pg < p.n_pages;
    }
    row = b * p.n_kv + kvh;
    slot = p.ring ? key % p.ring : key;
    return true;
}
// slots per row of that view
__device__ __forceinline__ int kv_row_slots(const RowsParams& p) {
    return p.page_size ? p.page_size : p.cap;
}
#endif

// Keys per shared-memory tile of the bf16 kernel; chunks are multiples of it.
constexpr int kKeyTile = 32;
constexpr int kRowTile = 16;     // rows per CTA in the bf16 kernel (one m16 MMA tile)
constexpr int kF32RowsPerCta = 4;

size_t rows_bf16_smem_bytes(int head_dim, int k_eq_v, int* n_stages);
cudaError_t launch_rows_bf16(const RowsParams& p, int head_dim, dim3 grid, size_t smem,
                             cudaStream_t st);
cudaError_t launch_rows_f32(const RowsParams& p, int head_dim, dim3 grid, cudaStream_t st);
cudaError_t launch_combine(const RowsParams& p, int head_dim, int batch, int out_fp32,
                           cudaStream_t st);
bool prefill_tc_supported(int head_dim);
cudaError_t launch_prefill_tc(const RowsParams& p, int head_dim, int batch, cudaStream_t st);
// head_dim 256 (one CTA pair) or 512 (two pairs, one per half of head_dim) on clusters issuing
// 2-SM MMAs (called by launch_prefill_tc)
cudaError_t launch_prefill_pair(const RowsParams& p, int head_dim, int batch, cudaStream_t st);
// paged pool layout for the append (block_table == nullptr: a plain or ring cache)
struct PagedLayout {
    const int32_t* block_table;
    int max_pages, page_size, n_pages;
};
cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             const int32_t* write_pos, const int32_t* n_real, int ring,
                             const PagedLayout& pg,
                             int batch, int n_new, int n_kv,
                             int capacity, int row_bytes, uint32_t* err, int n_sm,
                             cudaStream_t st);

}  // namespace gemma
