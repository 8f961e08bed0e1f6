/*
 * gemma_attn.h -- C ABI of the mixed sliding/global attention step on a device-resident
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation: one attention step of a decoder whose layers interleave sliding-window
 * and global attention ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", model family
 * table and section 2.3), with grouped-query attention (same page, section 2.2: query
 * head h reads KV head h / (n_q / n_kv)), cross-layer KV sharing (section 2.1: a shared
 * layer attends against an earlier owner layer's cache and writes none), K used as V on
 * layers with attention_k_eq_v ("Gemma-4 12B on AWS Inferentia2 - Tensor-Parallel (TP=2),
 * device prefill", text config), and a one-token decode bucket plus a multi-token prefill
 * bucket against a fixed-capacity cache that stays on the device and is updated in place
 * (first page, section 5.1; "Gemma-4-E4B-it on AWS Inferentia2", "Decode neff").
 *
 * Definition computed (per sequence b, query token i, query head h):
 *   len   = seq_lens[b]                      cache tokens after this step's append
 *   p     = len - n_tok + i                  absolute position of the query
 *   keys  = { j : j <= p, and p - j < window on a sliding layer }
 *   out   = sum_j softmax_j(scale * q . K[j]) * V[j]   over those keys,
 *   K, V  = the owner layer's cache, KV head h / (n_q / n_kv); V is K when k_eq_v.
 *
 * Conventions shared by every entry point
 *  - The caller owns all memory. The library allocates nothing, never synchronises and
 *    enqueues all work on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *    Every call can be captured in a CUDA graph.
 *  - Pointers named "device" must be device-accessible (cudaMalloc'd) memory aligned to
 *    16 bytes; arrays of pointers (k_cache, v_cache) and owner_map live in HOST memory.
 *  - Cache layout, per owner layer: [batch][n_kv][kv_capacity][head_dim], row-major.
 *    Query/output layout: [batch][n_tok][n_q][head_dim] (n_tok = 1 for decode).
 *    New K/V rows: [batch][n_new][n_kv][head_dim]. Element type: `dtype` (bf16 or fp32;
 *    fp32 is the debug build path); output has the same type.
 *  - Argument errors are detected on the host before any launch and return a negative
 *    gemma_status with nothing enqueued. A failed launch returns GEMMA_ERR_CUDA.
 *  - Data-dependent errors (a seq_lens or write_pos entry out of range, only visible on
 *    the device) never cause an out-of-bounds access: the affected sequence is skipped
 *    (its output rows are written as zeros) and, when `device_error` is not NULL, a
 *    GEMMA_DEVERR_* bit is OR-ed into that device word, which the caller reads after
 *    synchronising. Internal waits are bounded and report GEMMA_DEVERR_TIMEOUT.
 *  - Supported shapes: head_dim in {64, 128, 256, 512}; n_q / n_kv in {1, 2, 4, 8, 16};
 *    window >= 1 on sliding layers. Others return GEMMA_ERR_UNSUPPORTED.
 *  - batch == 0 or n_new == 0 is a valid empty call: GEMMA_OK, nothing enqueued.
 */
#ifndef GEMMA_ATTN_H
#define GEMMA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GEMMA_SLIDING_RING: a sliding layer whose cache is a ring of kv_capacity slots holding the
 * most recent tokens, position p at slot p % kv_capacity (the pages' fixed KV_MAX buffer sized
 * to the window rather than the context). kv_capacity must be a multiple of 128 and at least
 * window + n_new - 1 (every key a step attends is still in the ring), else
 * GEMMA_ERR_UNSUPPORTED / GEMMA_ERR_CAPACITY; seq_lens and max_seq_len may exceed it. Its rows
 * are written with gemma_kv_append_ring (or gemma_attn_decode_append, which wraps the same way). */
typedef enum { GEMMA_SLIDING = 0, GEMMA_GLOBAL = 1, GEMMA_SLIDING_RING = 2 } gemma_layer_kind;
typedef enum { GEMMA_BF16 = 0, GEMMA_FP32 = 1 } gemma_dtype;
typedef enum {
    GEMMA_OK = 0,
    GEMMA_ERR_INVALID_ARG = -1,  /* NULL/misaligned pointer, bad owner map, inconsistent sizes */
    GEMMA_ERR_UNSUPPORTED = -2,  /* head_dim or group size outside the supported set */
    GEMMA_ERR_CAPACITY = -3,     /* max_seq_len / n_new beyond kv_capacity */
    GEMMA_ERR_WORKSPACE = -4,    /* workspace NULL or smaller than gemma_attn_workspace_size */
    GEMMA_ERR_CUDA = -5          /* a CUDA runtime call or launch failed */
} gemma_status;

/* Bits OR-ed into the optional device error word. */
#define GEMMA_DEVERR_SEQ_LEN 1u    /* seq_lens[b] outside [n_tok, min(kv_capacity, max_seq_len)] */
#define GEMMA_DEVERR_WRITE_POS 2u  /* write_pos[b] < 0 or write_pos[b] + n_new > kv_capacity */
#define GEMMA_DEVERR_TIMEOUT 4u    /* an internal pipeline wait gave up */
#define GEMMA_DEVERR_N_REAL 8u     /* n_real[b] outside [0, n_new] (padded-bucket entry points) */
#define GEMMA_DEVERR_PAGE 16u      /* a block-table entry outside [0, n_pages) (paged entry points) */

/*
 * gemma_kv_append -- write this step's new K (and V) rows of an owner layer into its cache.
 *   cache[b][h][write_pos[b] + t][:] = new[b][t][h][:]   for t < n_new, h < n_kv.
 * Source: "Gemma-4-E4B-it on AWS Inferentia2" ("Decode neff": the KV buffers are updated in
 * place each step) and the first page, section 2.1 (only owner layers hold a cache; shared
 * layers never touch it). The pages' one-hot masked write is a tracing device of their
 * compiler; here it is a direct scatter of whole rows.
 *   k_cache, v_cache  HOST arrays [n_layers] of DEVICE cache pointers; entries of shared
 *                     layers are never read. v_cache (and v_cache[layer]) may be NULL when
 *                     k_eq_v, in which case v_new is ignored.
 *   owner_map         HOST int32[n_layers]; if owner_map[layer] != layer the layer is
 *                     shared and the call is a no-op returning GEMMA_OK.
 *   k_new, v_new      DEVICE [batch][n_new][n_kv][head_dim].
 *   write_pos         DEVICE int32[batch]: cache slot of the first new token of sequence b.
 *   device_error      optional DEVICE uint32 (may be NULL).
 */
int gemma_kv_append(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                    int n_layers, int layer, const void* k_new, const void* v_new,
                    const int32_t* write_pos, int batch, int n_new, int n_kv, int head_dim,
                    int kv_capacity, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                    void* stream);

/*
 * gemma_kv_append_ring -- gemma_kv_append into a ring cache (GEMMA_SLIDING_RING): row t of
 * sequence b goes to slot (write_pos[b] + t) % kv_capacity; write_pos[b] >= 0 may exceed the
 * capacity; n_new <= kv_capacity.
 */
int gemma_kv_append_ring(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                         int n_layers, int layer, const void* k_new, const void* v_new,
                         const int32_t* write_pos, int batch, int n_new, int n_kv, int head_dim,
                         int kv_capacity, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                         void* stream);

/*
 * gemma_attn_decode -- the decode bucket: one query token per sequence (n_tok = 1), whose
 * K/V were appended first, so seq_lens[b] counts it. Source: first page, section 5.1
 * ("decode: single-token forward against a fixed KV_MAX buffer").
 *   out               DEVICE [batch][1][n_q][head_dim]   (written)
 *   q                 DEVICE [batch][1][n_q][head_dim]
 *   k_cache, v_cache  HOST arrays [n_layers] of DEVICE cache pointers; the layer reads
 *                     k_cache[owner_map[layer]] (and v_cache[...] unless k_eq_v).
 *   owner_map         HOST int32[n_layers]: 0 <= owner_map[l] <= l and
 *                     owner_map[owner_map[l]] == owner_map[l]. The owner must have this
 *                     layer's kind, n_kv, head_dim and k_eq_v (the caller's contract).
 *   seq_lens          DEVICE int32[batch], 1 <= seq_lens[b] <= max_seq_len.
 *   max_seq_len       HOST bound on seq_lens, used to plan the split over keys: unsplit when
 *                     the (sequence, KV head) pairs alone fill the GPU over short key ranges;
 *                     else chunks of keys merged inside the launch when a pair's chunks form
 *                     one thread-block cluster (at most 8, or 16 when the whole grid fits one
 *                     CTA per SM), else by a second launch through the workspace.
 *   scale             softmax scale applied to q . k, finite and > 0 (1/sqrt(head_dim) in
 *                     the workloads).
 *   workspace         DEVICE scratch of at least
 *                     gemma_attn_workspace_size(batch, kind, window, n_q, n_kv, head_dim,
 *                     max_seq_len, 1) bytes (may be NULL when that size is 0). Contents on
 *                     entry are ignored; concurrent calls must not share it.
 */
int gemma_attn_decode(void* out, const void* q, const void* const* k_cache,
                      const void* const* v_cache, const int32_t* owner_map, int n_layers,
                      int layer, const int32_t* seq_lens, int max_seq_len, int batch,
                      gemma_layer_kind kind, int window, int n_q, int n_kv, int head_dim,
                      int k_eq_v, int kv_capacity, float scale, gemma_dtype dtype,
                      void* workspace, size_t workspace_bytes, uint32_t* device_error,
                      void* stream);

/*
 * gemma_attn_decode_static -- gemma_attn_decode without a caller-provided workspace. The pages
 * have no counterpart: this entry point exists for callers of this library that cannot
 * allocate device memory (code running inside an allocator or memory-pool callback, a plugin
 * whose host owns every device allocation, or a latency-critical path that must not call the
 * driver's allocator). Its split scratch is a fixed 32 MiB array compiled into the library,
 * held by every GPU that loads the library until the process exits. It allocates nothing.
 *  - Arguments and results are those of gemma_attn_decode minus workspace/workspace_bytes,
 *    with the same statuses in the same order of checks: an unsupported shape gives
 *    GEMMA_ERR_UNSUPPORTED, a bad argument GEMMA_ERR_INVALID_ARG or GEMMA_ERR_CAPACITY.
 *  - Returns GEMMA_ERR_WORKSPACE, with no launch, when the arguments are valid but
 *    gemma_attn_workspace_size(...) for them is larger than 32 MiB (e.g. batch 64 x 16 query
 *    heads of head_dim 512 split 19 ways needs about 40 MB and is refused; batch-1 plans need
 *    a few MB at most, and plans whose chunks merge inside one thread-block cluster need
 *    none).
 *  - The first call in each CUDA context (per device, and again after a device reset) looks up
 *    the array's device address with that device current; make that first call before any
 *    stream capture.
 *  - All calls share the array, which keeps the previous call's contents (nothing in it has to
 *    start at zero); calls whose kernels overlap on the GPU race on it, so the caller must
 *    order them (one stream, or events between streams).
 */
int gemma_attn_decode_static(void* out, const void* q, const void* const* k_cache,
                             const void* const* v_cache, const int32_t* owner_map, int n_layers,
                             int layer, const int32_t* seq_lens, int max_seq_len, int batch,
                             gemma_layer_kind kind, int window, int n_q, int n_kv, int head_dim,
                             int k_eq_v, int kv_capacity, float scale, gemma_dtype dtype,
                             uint32_t* device_error, void* stream);

/*
 * gemma_attn_prefill -- the prefill bucket: n_new query tokens per sequence, written to the
 * cache first (gemma_kv_append), at positions seq_lens[b] - n_new + i, attending causally
 * (and within the window on sliding layers) over the cached prefix and the new tokens.
 * Source: first page, section 5.1 ("prefill (padded prompt <= KV_BUCKET ...)") and the 12B
 * model card ("a prefill bucket (seq = 64) and a decode bucket (seq = 1)"); here the bucket
 * is exact (no pad rows) and may extend a cached prefix.
 *   out, q            DEVICE [batch][n_new][n_q][head_dim]
 *   seq_lens          DEVICE int32[batch], n_new <= seq_lens[b] <= max_seq_len.
 *   Other arguments as for gemma_attn_decode (workspace sized with n_new).
 */
int gemma_attn_prefill(void* out, const void* q, const void* const* k_cache,
                       const void* const* v_cache, const int32_t* owner_map, int n_layers,
                       int layer, const int32_t* seq_lens, int max_seq_len, int n_new,
                       int batch, gemma_layer_kind kind, int window, int n_q, int n_kv,
                       int head_dim, int k_eq_v, int kv_capacity, float scale,
                       gemma_dtype dtype, void* workspace, size_t workspace_bytes,
                       uint32_t* device_error, void* stream);

/*
 * gemma_attn_softcap -- gemma_attn_decode (n_new == 1) or gemma_attn_prefill (n_new > 1) with
 * an attention-logit soft-cap: each scaled score s = scale * q . k becomes
 * softcap * tanh(s / softcap) before the softmax. Source: "Gemma-4-E4B-it on AWS Inferentia2",
 * Architecture (the recipe keeps an explicit attention softcap; the page gives no value, so it
 * is the caller's argument).
 *   softcap           finite and >= 0; 0 applies no cap (the call then equals the entry point
 *                     without a cap). Negative or non-finite values return
 *                     GEMMA_ERR_INVALID_ARG.
 *   Other arguments, the workspace size and the results are those of gemma_attn_decode /
 *   gemma_attn_prefill for the same n_new.
 */
int gemma_attn_softcap(void* out, const void* q, const void* const* k_cache,
                       const void* const* v_cache, const int32_t* owner_map, int n_layers,
                       int layer, const int32_t* seq_lens, int max_seq_len, int n_new,
                       int batch, gemma_layer_kind kind, int window, int n_q, int n_kv,
                       int head_dim, int k_eq_v, int kv_capacity, float scale, float softcap,
                       gemma_dtype dtype, void* workspace, size_t workspace_bytes,
                       uint32_t* device_error, void* stream);

/*
 * gemma_attn_decode_append -- gemma_kv_append followed by gemma_attn_decode, in one launch:
 * the CTA of the decode kernel whose key chunk holds write_pos[b] writes this step's K (and V)
 * row of its KV head into the cache before it loads that chunk, so the step needs no separate
 * append launch. Source: first page, section 5.1 and the E4B model card ("Decode neff": the KV
 * buffers are updated in place inside the decode step itself).
 *   k_cache, v_cache  as for gemma_kv_append (written) and gemma_attn_decode (read).
 *   k_new, v_new      DEVICE [batch][1][n_kv][head_dim]; ignored on a shared layer (which
 *                     then runs gemma_attn_decode against its owner's cache).
 *   write_pos         DEVICE int32[batch]; normally seq_lens[b] - 1. A slot outside
 *                     [0, kv_capacity) is reported (GEMMA_DEVERR_WRITE_POS) and not written;
 *                     a sequence whose seq_lens[b] is invalid is skipped entirely.
 *   Other arguments, the workspace and the results as for gemma_attn_decode. The fp32 debug
 *   path runs the append and the decode as two launches.
 */
int gemma_attn_decode_append(void* out, const void* q, void* const* k_cache, void* const* v_cache,
                             const int32_t* owner_map, int n_layers, int layer, const void* k_new,
                             const void* v_new, const int32_t* write_pos,
                             const int32_t* seq_lens, int max_seq_len, int batch,
                             gemma_layer_kind kind, int window, int n_q, int n_kv, int head_dim,
                             int k_eq_v, int kv_capacity, float scale, gemma_dtype dtype,
                             void* workspace, size_t workspace_bytes, uint32_t* device_error,
                             void* stream);

/*
 * gemma_kv_append_bucket / gemma_attn_prefill_bucket -- the padded prefill bucket: every
 * sequence brings n_new query rows (and n_new new K/V rows), of which only the first
 * n_real[b] are real tokens; the rest pad the sequence to the bucket size. Source: first page,
 * section 5.1 ("prefill (padded prompt <= KV_BUCKET ...)") and the 12B model card (prefill
 * bucket of seq = 64); the pages pad and trace a fixed shape, here the pad rows are masked
 * exactly: they are neither written to the cache nor attended, and their outputs are zero.
 *   n_real            DEVICE int32[batch], 0 <= n_real[b] <= n_new (else the sequence is
 *                     skipped and GEMMA_DEVERR_N_REAL is reported).
 *   gemma_kv_append_bucket writes rows t < n_real[b] at write_pos[b] + t; other arguments as
 *   for gemma_kv_append.
 *   gemma_attn_prefill_bucket: seq_lens[b] counts the real tokens only (n_real[b] <=
 *   seq_lens[b]); the i-th real token of sequence b sits at seq_lens[b] - n_real[b] + i and
 *   attends as in gemma_attn_prefill. Other arguments and the workspace as for
 *   gemma_attn_prefill (n_new == 1 is allowed).
 */
int gemma_kv_append_bucket(void* const* k_cache, void* const* v_cache, const int32_t* owner_map,
                           int n_layers, int layer, const void* k_new, const void* v_new,
                           const int32_t* write_pos, const int32_t* n_real, int batch, int n_new,
                           int n_kv, int head_dim, int kv_capacity, int k_eq_v, gemma_dtype dtype,
                           uint32_t* device_error, void* stream);

int gemma_attn_prefill_bucket(void* out, const void* q, const void* const* k_cache,
                              const void* const* v_cache, const int32_t* owner_map, int n_layers,
                              int layer, const int32_t* seq_lens, const int32_t* n_real,
                              int max_seq_len, int n_new, int batch, gemma_layer_kind kind,
                              int window, int n_q, int n_kv, int head_dim, int k_eq_v,
                              int kv_capacity, float scale, gemma_dtype dtype, void* workspace,
                              size_t workspace_bytes, uint32_t* device_error, void* stream);

/*
 * gemma_attn_workspace_size -- bytes of scratch that gemma_attn_decode (n_new == 1) or
 * gemma_attn_prefill (n_new > 1) needs for these arguments on the current device (the split
 * plan depends on its SM count). Returns 0 when no scratch is needed and (size_t)-1 when the
 * arguments are invalid.
 */
size_t gemma_attn_workspace_size(int batch, gemma_layer_kind kind, int window, int n_q,
                                 int n_kv, int head_dim, int max_seq_len, int n_new);

/*
 * Paged KV pool -- the pages keep one fixed-capacity, device-resident KV buffer per layer,
 * updated in place (first page, section 5.1; "Gemma-4-E4B-it on AWS Inferentia2", "Decode
 * neff"). These entry points store the same logical cache of each owner layer in a shared pool
 * of fixed-size pages instead, so that a ragged batch holds only the pages its sequences use:
 *   pool        DEVICE [n_pages][n_kv][page_size][head_dim] per owner layer (k_pool[l], and
 *               v_pool[l] unless k_eq_v), caller-owned, 16-byte aligned.
 *   block_table DEVICE int32 [batch][max_pages]: position p of sequence b lives in page
 *               block_table[b * max_pages + p / page_size], row p % page_size. The same table
 *               may serve every layer. Entries are read only for the pages that hold keys a
 *               step attends or writes (from the window start rounded down to a multiple of 32
 *               keys, 64 for prefill, to the last position), so pages wholly before a sliding
 *               window may be recycled by the caller. An entry outside [0, n_pages) that is read
 *               sets GEMMA_DEVERR_PAGE; its rows read as zeros and are never written.
 *   page_size   a multiple of 128 (GEMMA_ERR_UNSUPPORTED otherwise): no key tile crosses a page.
 * The logical capacity of a sequence is max_pages * page_size; every other argument, the
 * definitions and the error behaviour are those of gemma_kv_append / gemma_attn_decode /
 * gemma_attn_prefill. Kinds GEMMA_SLIDING and GEMMA_GLOBAL only.
 */
int gemma_kv_append_paged(void* const* k_pool, void* const* v_pool, const int32_t* owner_map,
                          int n_layers, int layer, const void* k_new, const void* v_new,
                          const int32_t* write_pos, const int32_t* block_table, int max_pages,
                          int page_size, int n_pages, int batch, int n_new, int n_kv,
                          int head_dim, int k_eq_v, gemma_dtype dtype, uint32_t* device_error,
                          void* stream);

/* Attention over a paged pool: a decode step (n_new == 1) or a prefill bucket (n_new > 1).
 * With k_new != NULL (decode only, owner layers) the launch first writes this step's K (and V)
 * row [batch][1][n_kv][head_dim] at write_pos[b], as gemma_attn_decode_append does. Scratch:
 * gemma_attn_workspace_size_paged(...) bytes. */
int gemma_attn_paged(void* out, const void* q, void* const* k_pool, void* const* v_pool,
                     const int32_t* owner_map, int n_layers, int layer, const int32_t* seq_lens,
                     const int32_t* block_table, int max_pages, int page_size, int n_pages,
                     int max_seq_len, int n_new, int batch, gemma_layer_kind kind, int window,
                     int n_q, int n_kv, int head_dim, int k_eq_v, float scale, gemma_dtype dtype,
                     const void* k_new, const void* v_new, const int32_t* write_pos,
                     void* workspace, size_t workspace_bytes, uint32_t* device_error,
                     void* stream);

/* Scratch bytes of gemma_attn_paged for these arguments on the current device ((size_t)-1 for
 * invalid arguments, including GEMMA_SLIDING_RING). */
size_t gemma_attn_workspace_size_paged(int batch, gemma_layer_kind kind, int window, int n_q,
                                       int n_kv, int head_dim, int max_seq_len, int n_new);

/*
 * gemma_logit_softcap_argmax -- final-logit soft-cap and greedy argmax of each row.
 *   capped[b][i] = softcap * tanh(logits[b][i] / softcap)      (logits[b][i] when softcap == 0)
 *   argmax[b]    = the lowest i with logits[b][i] >= logits[b][j] for every non-NaN j
 * Source: "Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", family table (logit softcap 30,
 * vocabulary 262,144) and section 4.2 (the model caps its logits with softcap * tanh(x /
 * softcap); the argmax of the capped logits is the argmax of the raw ones, so greedy decoding
 * does not depend on the cap). The index is therefore taken on the raw logits: an exact
 * comparison, the same in every precision. NaN entries are never selected; a row of NaN gives
 * index 0. For bf16 logits tanh is the hardware approximation (relative error below 2^-10.9,
 * a fraction of the bf16 rounding); for fp32 logits the accurate library tanhf.
 *   logits      DEVICE [batch][vocab] of dtype, row-major, 16-byte aligned (caller-owned).
 *   capped_out  DEVICE [batch][vocab] of dtype, 16-byte aligned, or NULL to skip the capped
 *               logits; may equal logits (in place).
 *   argmax_out  DEVICE int32 [batch].
 *   softcap     >= 0 and finite.
 *   workspace   DEVICE scratch of gemma_logit_workspace_size(batch, vocab) bytes, 16-byte
 *               aligned (NULL when that is 0); holds no state between calls.
 * Returns GEMMA_ERR_INVALID_ARG (NULL or misaligned pointer, batch < 0, vocab < 1, bad softcap
 * or dtype), GEMMA_ERR_UNSUPPORTED (batch > 65535) or GEMMA_ERR_WORKSPACE before any launch;
 * batch == 0 is a no-op. Asynchronous on
 * `stream`; allocates nothing; graph-capturable.
 */
int gemma_logit_softcap_argmax(const void* logits, int batch, int vocab, gemma_dtype dtype,
                               float softcap, void* capped_out, int32_t* argmax_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of scratch gemma_logit_softcap_argmax needs on the current device ((size_t)-1 for
 * batch < 0 or vocab < 1). 0 when the batch is large enough for every row to get CTAs of its
 * own (at most 16, one thread-block cluster per row, reducing the row's index among themselves
 * in the same launch); otherwise the rows' pieces meet in the scratch and a second launch
 * reduces them. */
size_t gemma_logit_workspace_size(int batch, int vocab);

/* A static, human-readable name of a gemma_status value. */
const char* gemma_status_string(int status);

/* Version of this ABI (bumped on any signature change). */
int gemma_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMMA_ATTN_H */
