/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, double-precision CPU definition of one attention step of a
 * Gemma-4 style decoder whose layers interleave sliding-window and global
 * attention, use grouped-query attention, may read an earlier layer's KV cache
 * (cross-layer KV sharing) and may attend with V := K. Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load this library; the
 * product path (the CUDA library) never does, and the two share no code.
 *
 * Sources (page title, section):
 *  - "Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", section 2.1: a layer
 *    flagged is_kv_shared_layer computes no K/V of its own and attends against
 *    the K/V of an earlier "owner" layer; only owner layers hold a cache.
 *  - same page, section 2.2: repeat_kv hands each KV head to a contiguous group
 *    of num_key_value_groups = n_q / n_kv query heads.
 *  - same page, family table and section 2.3: sliding layers attend a local
 *    window (sliding_window = 512 or 1024), global layers the full causal
 *    context, with different KV-head counts and head_dims per layer kind.
 *  - "Gemma-4 12B on AWS Inferentia2 - Tensor-Parallel (TP=2), device prefill",
 *    text-config list: attention_k_eq_v = true, global layers reuse K as V.
 *  - first page, section 4.3: the device model runs "eager" attention, i.e.
 *    plain matmul, softmax, matmul; that definition is what is evaluated here.
 *  - first page, section 5.1 and the E4B model card ("Decode neff"): a decode
 *    bucket of one token and a prefill bucket of several tokens, both against a
 *    fixed-capacity, device-resident KV buffer updated in place at the new
 *    positions.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - window: a query at absolute position p attends key j iff j <= p and, on a
 *    sliding layer, p - j < W (W keys including itself);
 *  - the new tokens are written into the cache before attention, so the cache
 *    holds len tokens and the i-th of n_tok queries sits at p = len - n_tok + i;
 *  - the softmax scale is an explicit argument (1/sqrt(head_dim) in the
 *    workloads);
 *  - the attention-logit soft-cap ("Gemma-4-E4B-it on AWS Inferentia2",
 *    Architecture: the recipe keeps an explicit attention softcap; no value is
 *    given) is optional: with softcap c > 0 each scaled score s = scale * q.k
 *    becomes c * tanh(s / c) before the softmax; c = 0 applies none.
 *
 * Parity pins (tests): torch fp64 scaled_dot_product_attention on tiny shapes,
 * closed forms (uniform weights for K = 0, one-hot V, W = 1, two keys), and
 * invariants (W >= len equals global, K-as-V equals passing K as V, shared
 * layer equals a private copy of its owner's cache, one KV head broadcast
 * equals replicated heads, key permutation, key shift); the soft-cap by a cap
 * far above every score (no change) and by the saturated closed form (scores
 * of +-L with L >> c become exactly +-c). The scale convention of the real
 * model, and its soft-cap value, are not pinned by the pages ("parity
 * unpinned" for them).
 *
 * Final logits ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", family table and
 * section 4.2): the model caps its output logits to softcap * tanh(logits / softcap) over the
 * whole vocabulary (softcap 30, 262,144 tokens), and the page notes that the argmax of the
 * capped logits is the argmax of the raw ones, so greedy decoding does not depend on the cap.
 * Reading taken: the greedy index is the argmax of the raw logits (an exact comparison, no
 * rounding decides it), the lowest index among equal maxima, NaN entries never selected (a row
 * of NaN gives index 0). Pins: the capped value by its closed forms (a cap far above the logits
 * changes nothing, saturated logits become +-c, odd symmetry), the index against the first
 * maximum of numpy and against the argmax of the fp64 capped values (the page's statement).
 *
 * ORACLE_MUTANT, when defined, plants one deliberate mistake; the test suite
 * builds such variants to show that its pins catch each of them. The normal
 * build never defines it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ORACLE_SLIDING = 0, ORACLE_GLOBAL = 1 };
enum { ORACLE_BF16 = 0, ORACLE_FP32 = 1 };
enum { ORACLE_OK = 0, ORACLE_ERR_ARG = -1, ORACLE_ERR_CAPACITY = -3, ORACLE_ERR_ALLOC = -6 };

typedef struct {
    int32_t kind;      /* ORACLE_SLIDING or ORACLE_GLOBAL */
    int32_t window;    /* W, used by sliding layers */
    int32_t n_q;       /* query heads */
    int32_t n_kv;      /* key/value heads of this layer kind */
    int32_t head_dim;
    int32_t k_eq_v;    /* 1: V := K */
} oracle_layer;

int oracle_abi_version(void) { return 1; }
int oracle_mutant(void) { return ORACLE_MUTANT; }

/* One stored element as a double. bf16 is the upper half of an IEEE float32. */
static double load_elem(const void* base, size_t index, int dtype)
{
    if (dtype == ORACLE_FP32) return (double)((const float*)base)[index];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[index] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Owner resolution (first page, section 2.1): layer l reads the cache of
 * owner_map[l], an earlier (or the same) layer that owns a cache and has the
 * same kind, KV-head count, head_dim and K-as-V flag. Returns the owner or a
 * negative status. */
int oracle_resolve_owner(const oracle_layer* layers, const int32_t* owner_map, int n_layers,
                         int layer)
{
    if (!layers || !owner_map || layer < 0 || layer >= n_layers) return ORACLE_ERR_ARG;
    int o = owner_map[layer];
#if ORACLE_MUTANT == 5
    o = layer; /* planted mistake: the shared layer reads its own (empty) slot */
#endif
    if (o < 0 || o > layer) return ORACLE_ERR_ARG;
    if (owner_map[o] != o) return ORACLE_ERR_ARG;
    const oracle_layer* a = &layers[layer];
    const oracle_layer* b = &layers[o];
    if (a->kind != b->kind || a->n_kv != b->n_kv || a->head_dim != b->head_dim ||
        a->k_eq_v != b->k_eq_v)
        return ORACLE_ERR_ARG;
    return o;
}

/* In-place cache update (E4B model card, "Decode neff": the fixed buffer is
 * updated in place at the new position each step):
 *     cache[b][h][write_pos[b] + t][:] = rows[b][t][h][:].
 * Checks every sequence before writing anything. */
int oracle_kv_append(void* cache, const void* rows, const int32_t* write_pos, int batch,
                     int n_new, int n_kv, int head_dim, int capacity, int elem_bytes)
{
    if (!cache || !rows || !write_pos || batch < 0 || n_new < 0 || n_kv <= 0 || head_dim <= 0 ||
        capacity <= 0 || (elem_bytes != 2 && elem_bytes != 4))
        return ORACLE_ERR_ARG;
    for (int b = 0; b < batch; ++b)
        if (write_pos[b] < 0 || (int64_t)write_pos[b] + n_new > capacity) return ORACLE_ERR_CAPACITY;
    const size_t row_bytes = (size_t)head_dim * (size_t)elem_bytes;
    for (int b = 0; b < batch; ++b)
        for (int t = 0; t < n_new; ++t)
            for (int h = 0; h < n_kv; ++h) {
                size_t dst_row = ((size_t)b * n_kv + h) * (size_t)capacity + (size_t)write_pos[b] + t;
                size_t src_row = ((size_t)b * n_new + t) * (size_t)n_kv + h;
                memcpy((char*)cache + dst_row * row_bytes, (const char*)rows + src_row * row_bytes,
                       row_bytes);
            }
    return ORACLE_OK;
}

/*
 * One attention step of layer `layer` for n_tok query tokens per sequence.
 *   q        [batch][n_tok][n_q][head_dim]            (dtype)
 *   k_cache  k_cache[o] -> [batch][n_kv][capacity][head_dim] for owner layers o
 *   v_cache  likewise; unused (may be NULL) when the layer has k_eq_v
 *   seq_lens [batch] valid cache tokens after the new tokens were written
 *   out      [batch][n_tok][n_q][head_dim]            (double)
 */
int oracle_attention_softcap(const oracle_layer* layers, const int32_t* owner_map, int n_layers,
                             int layer, const void* const* k_cache, const void* const* v_cache,
                             int dtype, int capacity, const void* q, int n_tok,
                             const int32_t* seq_lens, int batch, double scale, double softcap,
                             double* out)
{
    if (!(softcap >= 0.0) || isinf(softcap)) return ORACLE_ERR_ARG;
    /* 1. which layer's cache this layer reads */
    int o = oracle_resolve_owner(layers, owner_map, n_layers, layer);
    if (o < 0) return o;
    const oracle_layer* L = &layers[layer];
    const int n_q = L->n_q, n_kv = L->n_kv, d = L->head_dim;
    if (n_q <= 0 || n_kv <= 0 || d <= 0 || d > 1024 || n_q % n_kv != 0) return ORACLE_ERR_ARG;
    if (L->kind != ORACLE_SLIDING && L->kind != ORACLE_GLOBAL) return ORACLE_ERR_ARG;
    if (L->kind == ORACLE_SLIDING && L->window < 1) return ORACLE_ERR_ARG;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP32) return ORACLE_ERR_ARG;
    if (!q || !seq_lens || !out || !k_cache || !k_cache[o] || n_tok < 1 || batch < 0)
        return ORACLE_ERR_ARG;
    if (!L->k_eq_v && (!v_cache || !v_cache[o])) return ORACLE_ERR_ARG;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[b] < n_tok || seq_lens[b] > capacity) return ORACLE_ERR_CAPACITY;

    /* 3. GQA head map (repeat_kv): query head h reads KV head h / G */
    const int G = n_q / n_kv;
    int* kv_of = (int*)malloc(sizeof(int) * (size_t)n_q);
    if (!kv_of) return ORACLE_ERR_ALLOC;
    for (int h = 0; h < n_q; ++h) {
        kv_of[h] = h / G;
#if ORACLE_MUTANT == 3
        kv_of[h] = h % n_kv; /* planted mistake: interleaved instead of grouped heads */
#endif
    }

    int status = ORACLE_OK;
    for (int b = 0; b < batch && status == ORACLE_OK; ++b) {
        const int len = seq_lens[b];
        const size_t kv_elems = (size_t)n_kv * (size_t)len * (size_t)d;
        double* K = (double*)malloc(sizeof(double) * (kv_elems ? kv_elems : 1));
        double* V = (double*)malloc(sizeof(double) * (kv_elems ? kv_elems : 1));
        unsigned char* mask = (unsigned char*)malloc((size_t)n_tok * (size_t)len + 1);
        double* s = (double*)malloc(sizeof(double) * ((size_t)len + 1));
        if (!K || !V || !mask || !s) {
            free(K); free(V); free(mask); free(s);
            status = ORACLE_ERR_ALLOC;
            break;
        }

        /* 2. the owner's keys (and values) of this sequence, as doubles;
         *    with k_eq_v, V is an explicit copy of K */
        for (int h = 0; h < n_kv; ++h)
            for (int t = 0; t < len; ++t)
                for (int c = 0; c < d; ++c) {
                    size_t src = (((size_t)b * n_kv + h) * (size_t)capacity + (size_t)t) * d + c;
                    size_t dst = ((size_t)h * len + t) * d + c;
                    K[dst] = load_elem(k_cache[o], src, dtype);
                    if (!L->k_eq_v) V[dst] = load_elem(v_cache[o], src, dtype);
                }
        if (L->k_eq_v) memcpy(V, K, sizeof(double) * kv_elems);

        /* 4. the mask: query i sits at absolute position p = len - n_tok + i */
        for (int i = 0; i < n_tok; ++i) {
            int p = len - n_tok + i;
#if ORACLE_MUTANT == 7
            p = i; /* planted mistake: position forgets the cached prefix */
#endif
            for (int j = 0; j < len; ++j) {
                int causal = j <= p;
#if ORACLE_MUTANT == 4
                causal = 1; /* planted mistake: no causal mask */
#endif
                int in_window = (L->kind == ORACLE_GLOBAL) || (p - j < L->window);
#if ORACLE_MUTANT == 1
                in_window = (L->kind == ORACLE_GLOBAL) || (p - j <= L->window); /* off by one */
#endif
                mask[(size_t)i * len + j] = (unsigned char)(causal && in_window);
            }
        }

        /* 5. masked softmax(scale * q k^T) v for every (query token, query head) */
        for (int i = 0; i < n_tok; ++i)
            for (int h = 0; h < n_q; ++h) {
                const size_t row = ((size_t)b * n_tok + i) * (size_t)n_q + h;
                const double* Kh = K + (size_t)kv_of[h] * len * d;
                const double* Vh = V + (size_t)kv_of[h] * len * d;
                const unsigned char* mrow = mask + (size_t)i * len;
                double qd[1024];
                for (int c = 0; c < d; ++c) qd[c] = load_elem(q, row * d + c, dtype);

                double m = -INFINITY;
                for (int j = 0; j < len; ++j) {
                    if (!mrow[j]) continue;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += qd[c] * Kh[(size_t)j * d + c];
                    s[j] = scale * dot;
#if ORACLE_MUTANT == 2
                    s[j] = dot; /* planted mistake: scale dropped */
#endif
                    /* 5a. optional soft-cap of the scaled score */
                    if (softcap > 0.0) {
                        s[j] = softcap * tanh(s[j] / softcap);
#if ORACLE_MUTANT == 8
                        s[j] = scale * softcap * tanh(dot / softcap); /* planted: cap before scale */
#endif
                    }
                    if (s[j] > m) m = s[j];
                }
                double denom = 0.0;
                for (int j = 0; j < len; ++j) {
#if ORACLE_MUTANT == 6
                    /* planted mistake: normaliser summed over every cached key */
                    if (!mrow[j]) {
                        double dot = 0.0;
                        for (int c = 0; c < d; ++c) dot += qd[c] * Kh[(size_t)j * d + c];
                        denom += exp(scale * dot - m);
                        continue;
                    }
#else
                    if (!mrow[j]) continue;
#endif
                    denom += exp(s[j] - m);
                }
                double* orow = out + row * d;
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                for (int j = 0; j < len; ++j) {
                    if (!mrow[j]) continue;
                    const double w = exp(s[j] - m) / denom;
                    for (int c = 0; c < d; ++c) orow[c] += w * Vh[(size_t)j * d + c];
                }
            }
        free(K); free(V); free(mask); free(s);
    }
    free(kv_of);
    return status;
}

/* oracle_attention_softcap without a soft-cap. */
int oracle_attention(const oracle_layer* layers, const int32_t* owner_map, int n_layers, int layer,
                     const void* const* k_cache, const void* const* v_cache, int dtype,
                     int capacity, const void* q, int n_tok, const int32_t* seq_lens, int batch,
                     double scale, double* out)
{
    return oracle_attention_softcap(layers, owner_map, n_layers, layer, k_cache, v_cache, dtype,
                                    capacity, q, n_tok, seq_lens, batch, scale, 0.0, out);
}

/* Final-logit soft-cap and greedy argmax of each row of logits [batch][vocab] (bf16 or fp32).
 * capped (optional, [batch][vocab]) receives c * tanh(x / c) for c > 0, x itself for c == 0;
 * index[b] receives the lowest i with x_i >= x_j for every non-NaN x_j (0 for a row of NaN). */
int oracle_logit_softcap_argmax(const void* logits, int dtype, int batch, int vocab,
                                double softcap, double* capped, int32_t* index)
{
    if (!logits || !index || batch < 0 || vocab < 1 || !(softcap >= 0.0)) return ORACLE_ERR_ARG;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP32) return ORACLE_ERR_ARG;
    for (int b = 0; b < batch; ++b) {
        int best_i = -1;
        double best = 0.0;
        for (int i = 0; i < vocab; ++i) {
            const double x = load_elem(logits, (size_t)b * vocab + i, dtype);
            if (capped) {
                double c = x;
                if (softcap > 0.0) {
#if ORACLE_MUTANT == 10
                    c = softcap * tanh(x);          /* planted: the division by the cap dropped */
#else
                    c = softcap * tanh(x / softcap);
#endif
                }
                capped[(size_t)b * vocab + i] = c;
            }
            if (isnan(x)) continue;
#if ORACLE_MUTANT == 9
            if (best_i < 0 || x >= best) {          /* planted: the last of equal maxima wins */
#else
            if (best_i < 0 || x > best) {
#endif
                best = x;
                best_i = i;
            }
        }
        index[b] = best_i < 0 ? 0 : best_i;
    }
    return ORACLE_OK;
}
