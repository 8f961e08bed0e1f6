// kv_append.cu -- in-place write of this step's new K/V rows into an owner layer's cache.
//
//   cache[b][h][write_pos[b] + t][:] = new[b][t][h][:]     for t < n_real[b] (all n_new rows
//                                                           when n_real is null)
// and, into a ring cache of R slots, at slot (write_pos[b] + t) % R; into a paged pool
// [n_pages][n_kv][page_size][D], position p = write_pos[b] + t goes to page
// block_table[b][p / page_size], row p % page_size.
//
// "Gemma-4-E4B-it on AWS Inferentia2" ("Decode neff") keeps the KV buffers on the device and
// updates them in place each step; its one-hot masked write exists only to keep a traced
// graph free of scatters. Here each row is a direct 16-byte-vector copy: every thread moves
// one 16-byte chunk, consecutive threads cover consecutive chunks of a row, so both the read
// of the new rows and the write into the cache are fully coalesced.
#include "attn_internal.h"
#include "common.cuh"

namespace gemma {

__global__ void __launch_bounds__(256) kv_append_kernel(uint8_t* __restrict__ kc,
                                                        uint8_t* __restrict__ vc,
                                                        const uint8_t* __restrict__ kn,
                                                        const uint8_t* __restrict__ vn,
                                                        const int32_t* __restrict__ write_pos,
                                                        const int32_t* __restrict__ n_real,
                                                        int ring, const PagedLayout pg,
                                                        int batch, int n_new, int n_kv,
                                                        int capacity, int row_bytes,
                                                        uint32_t* err) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    const int chunks = row_bytes / 16;
    const long long total = (long long)batch * n_new * n_kv * chunks;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long row = idx / chunks;
        const int ch = (int)(idx - row * chunks);
        const int h = (int)(row % n_kv);
        const long long bt = row / n_kv;
        const int t = (int)(bt % n_new);
        const int b = (int)(bt / n_new);
        const int pos = __ldg(write_pos + b);
        const int nr = n_real ? __ldg(n_real + b) : n_new;  // rows of this sequence to write
        if (nr < 0 || nr > n_new) {
            if (t == 0 && h == 0 && ch == 0) report(err, GEMMA_DEVERR_N_REAL);
            continue;
        }
        if (t >= nr) continue;  // a pad row of a padded bucket
        if (pos < 0 || (!ring && (long long)pos + nr > capacity)) {
            if (t == 0 && h == 0 && ch == 0) report(err, GEMMA_DEVERR_WRITE_POS);
            continue;
        }
        size_t dst;
        if (pg.block_table) {  // capacity = max_pages * page_size
            const int p_abs = pos + t, blk = p_abs / pg.page_size;
            const int page = __ldg(pg.block_table + (size_t)b * pg.max_pages + blk);
            if (page < 0 || page >= pg.n_pages) {
                if (h == 0 && ch == 0) report(err, GEMMA_DEVERR_PAGE);
                continue;
            }
            dst = (((size_t)page * n_kv + h) * (size_t)pg.page_size +
                   (size_t)(p_abs - blk * pg.page_size)) * (size_t)row_bytes + (size_t)ch * 16;
        } else {
            const long long slot = ring ? ((long long)pos + t) % ring : (long long)pos + t;
            dst = (((size_t)b * n_kv + h) * (size_t)capacity + (size_t)slot) *
                      (size_t)row_bytes + (size_t)ch * 16;
        }
        const size_t src = (size_t)row * row_bytes + (size_t)ch * 16;
        *reinterpret_cast<uint4*>(kc + dst) = __ldg(reinterpret_cast<const uint4*>(kn + src));
        if (vc) *reinterpret_cast<uint4*>(vc + dst) = __ldg(reinterpret_cast<const uint4*>(vn + src));
    }
}

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             const int32_t* write_pos, const int32_t* n_real, int ring,
                             const PagedLayout& pg,
                             int batch, int n_new, int n_kv, int capacity, int row_bytes,
                             uint32_t* err, int n_sm, cudaStream_t st) {
    const long long total = (long long)batch * n_new * n_kv * (row_bytes / 16);
    long long blocks = (total + 255) / 256;
    const long long cap_blocks = (long long)n_sm * 8;
    if (blocks > cap_blocks) blocks = cap_blocks;
    if (blocks < 1) blocks = 1;
    return launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                      static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new),
                      write_pos, n_real, ring, pg, batch, n_new, n_kv, capacity, row_bytes, err);
}

}  // namespace gemma
