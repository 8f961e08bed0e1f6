// rows_attn.cu -- attention over a device-resident KV cache for tiles of query rows.
//
// Serves the decode bucket (one token per sequence, split over key chunks, partials merged
// by combine_kernel) and the prefill bucket (many tokens per sequence, one pass per row
// tile). Definition ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", sections 2.1-2.3
// and 4.3): query head h of a layer reads KV head h / G of the owner layer's cache; the query
// at absolute position p attends keys j <= p, and on a sliding layer only p - j < window; the
// output is softmax(scale * q k^T) v over those keys, with V = K on k_eq_v layers.
//
// bf16 kernel design (per CTA: one KV head of one sequence, 16 query rows, one key chunk):
//  - the key range is clamped to the window / causal limit before any load (no predicated
//    loads of keys the tile cannot attend);
//  - a producer warp streams 32-key K/V tiles with tiled TMA (one box per 64 columns of
//    head_dim, 128-byte swizzle) into a shared-memory ring; the ldmatrix reads below apply
//    the same swizzle, so they are bank-conflict free; every K/V tile is read from HBM once
//    and reused by all rows (all query heads of the GQA group, and all tokens of the tile);
//    rows past the chunk's last key are loaded but masked (scores) and zeroed (values) in
//    registers;
//  - eight consumer warps: (1) S = Q K^T with mma.sync m16n8k16 (warps split keys x head_dim),
//    (2) per-row online softmax in exp2 form with warp shuffles, P rounded to bf16,
//    (3) O = diag(alpha) O + P V (warps split head_dim);
//  - the producer warp starts its loads as soon as the grid may read memory, while the consumer
//    warps stage the Q rows in the ring's last stage and take their Q fragments into registers
//    (the stage is then released to the producer);
//  - fp32 accumulation throughout; partial (m, l, O) per chunk when the keys are split: merged by
//    combine_kernel, or, when a row tile's chunks form one thread-block cluster (at most 8),
//    inside the launch: each chunk sends every CTA of the cluster its part of that CTA's column
//    slice through distributed shared memory (st.async), and each CTA merges its slice.
#include <atomic>

#include "attn_internal.h"
#include "common.cuh"
#include "tc.cuh"
#include "tmap.h"

namespace gemma {

constexpr int kConsumerWarps = 8;
constexpr int kRowsThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
#ifndef GEMMA_ROWS_SMEM_BUDGET
#define GEMMA_ROWS_SMEM_BUDGET (113 * 1024)  // two CTAs per SM
#endif
#ifndef GEMMA_ROWS_MIN_BLOCKS
#define GEMMA_ROWS_MIN_BLOCKS 2
#endif
constexpr int kSmemBudget = GEMMA_ROWS_SMEM_BUDGET;
constexpr float kLazyRescaleLog2 = 8.f;  // move the softmax reference only past this growth

template <int D>
struct RowsLayout {
    static constexpr int ROW = 2 * D + 16;      // padded bytes per Q row (staged in the ring)
    static constexpr int BOX = kKeyTile * 128;  // one TMA box: 32 keys x 64 columns (swizzled)
    static constexpr int TILE = (D / 64) * BOX; // one K or V tile
    static constexpr int KSPLIT = D >= 512 ? 4 : 2;  // warps sharing one n-tile in S = QK^T
    static constexpr int S_STRIDE = kKeyTile + 8;    // fp32 words per S row
    static constexpr int P_STRIDE = kKeyTile + 8;    // bf16 elements per P row
    static constexpr int S_OFF = 0;
    static constexpr int P_OFF = S_OFF + KSPLIT * kRowTile * S_STRIDE * 4;
    static constexpr int STAT_OFF = P_OFF + kRowTile * P_STRIDE * 2;  // alpha, m, l [16] each
    static constexpr int BAR_OFF = (STAT_OFF + 3 * kRowTile * 4 + 15) / 16 * 16;
    // barriers: full[kMaxStages], empty[kMaxStages], recv (cluster merge)
    static constexpr int RING_OFF = (BAR_OFF + (2 * kMaxStages + 1) * 8 + 1023) / 1024 * 1024;
};

// Byte offset of element (key, d) in a K/V tile written by TMA with 128-byte swizzle: box
// d / 64, 128-byte row `key`, 16-byte chunk ((d / 8) % 8) ^ (key % 8).
template <int D>
GEMMA_DEVINL uint32_t tile_off(int key, int d) {
    return (uint32_t)((d >> 6) * RowsLayout<D>::BOX + key * 128 +
                      ((((d >> 3) & 7) ^ (key & 7)) << 4) + (d & 7) * 2);
}

// distributed shared memory of a cluster: a peer's copy of a local address, loads from it, and
// a full cluster barrier (release / acquire)
GEMMA_DEVINL uint32_t rows_map_peer(const void* local, uint32_t peer) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(peer));
    return r;
}
GEMMA_DEVINL float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
GEMMA_DEVINL void rows_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
GEMMA_DEVINL void rows_cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
GEMMA_DEVINL void rows_cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Column slices of the cluster merge, in column pairs: CTA c owns columns
// [merge_col(c), merge_col(c + 1)); merge_owner(col) is the CTA whose slice holds col (even).
GEMMA_DEVINL int merge_col(int c, int D, int ns) { return 2 * ((c * (D / 2)) / ns); }
GEMMA_DEVINL int merge_owner(int col, int D, int ns) { return ((col / 2 + 1) * ns - 1) / (D / 2); }

// Row geometry: local row r of tile rt is global row R = rt*16 + r, token R / G, member R % G.
struct RowInfo {
    int token, head, pos, lo;
};

GEMMA_DEVINL RowInfo row_info(const RowsParams& p, int len, int kvh, int R) {
    RowInfo ri;
    ri.token = R / p.G;
    ri.head = kvh * p.G + (R - ri.token * p.G);
    ri.pos = len - p.n_tok + ri.token;
    ri.lo = p.is_sliding ? max(0, ri.pos - p.window + 1) : 0;
    return ri;
}

template <typename OutT>
GEMMA_DEVINL void zero_rows(const RowsParams& p, int b, int kvh, int row0, int n_rows, int D) {
    const int vec = 16 / (int)sizeof(OutT);
    const int per_row = D / vec;
    for (int idx = threadIdx.x; idx < n_rows * per_row; idx += blockDim.x) {
        const int r = idx / per_row, ch = idx - r * per_row;
        const int R = row0 + r;
        const int token = R / p.G, head = kvh * p.G + (R - token * p.G);
        OutT* dst = reinterpret_cast<OutT*>(p.out) +
                    (((size_t)b * p.n_tok + token) * p.n_q + head) * (size_t)D + (size_t)ch * vec;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// CLUSTER: the chunks of a row tile merge inside their cluster (a separate instantiation, so
// that the other launches carry no code for it)
template <int D, bool CLUSTER>
__global__ void __launch_bounds__(kRowsThreads, GEMMA_ROWS_MIN_BLOCKS)
    rows_attn_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const RowsParams p) {
    pdl_launch_dependents();
    using Lay = RowsLayout<D>;
    constexpr int T = kKeyTile;
    constexpr int KSPLIT = Lay::KSPLIT;
    constexpr int NGROUPS = kConsumerWarps / KSPLIT;  // n-groups of S columns
    constexpr int NTW = (T / 8) / NGROUPS;            // 8-key n-tiles per warp in S
    constexpr int KS = D / KSPLIT / 16;               // 16-wide k-steps per warp in S
    constexpr int NB = D / 8 / 8;                     // 8-column n-tiles per warp in O
    static_assert(KS % 2 == 0 && NTW >= 1, "tile shape");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.n_split;
    const int rt = blockIdx.x / p.n_split;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int rows_total = p.n_tok * p.G;
    const int row0 = rt * kRowTile;
    const int n_rows = min(kRowTile, rows_total - row0);
    const bool direct = p.n_split == 1;
    constexpr bool clustered = CLUSTER;  // the chunks merge through their cluster

    pdl_wait();  // the previous kernel on the stream has completed
    const int len = __ldg(p.seq_lens + b);

    if (len < p.n_tok || (!p.ring && len > p.cap) || len > p.max_seq_len) {
        // (every CTA of a cluster reads the same sequence, so all of them leave here)
        if (split == 0) {
            if (threadIdx.x == 0) report(p.err, GEMMA_DEVERR_SEQ_LEN);
            if (direct || clustered) zero_rows<__nv_bfloat16>(p, b, kvh, row0, n_rows, D);
        }
        return;
    }
    // keys any row of this tile may attend, then this CTA's chunk of them
    const RowInfo first = row_info(p, len, kvh, row0);
    const RowInfo last = row_info(p, len, kvh, row0 + n_rows - 1);
    // a ring cache's or paged pool's chunks start at multiples of the key tile, so that no tile
    // wraps around the ring or crosses a page (the rows' masks drop the keys before the window)
    const int base = (p.ring || p.page_size) ? (first.lo & ~(T - 1)) : first.lo;
    const int kb = base + split * p.chunk;
    const int ke = min(last.pos + 1, kb + p.chunk);
    // an empty chunk: the combine pass skips it; in a cluster it takes part in the merge with
    // no keys (max -inf, sum 0)
    if (kb >= ke && !clustered) return;
    const int n_keys = kb >= ke ? 0 : ke - kb;
    const int n_tiles = (n_keys + T - 1) / T;
    const int nops = p.k_eq_v ? 1 : 2;
    const int stage_bytes = nops * Lay::TILE;
    const int S = p.n_stages;

    float* sS = reinterpret_cast<float*>(smem + Lay::S_OFF);
    __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(smem + Lay::P_OFF);
    float* sAlpha = reinterpret_cast<float*>(smem + Lay::STAT_OFF);
    float* sM = sAlpha + kRowTile;
    float* sL = sM + kRowTile;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFF);
    uint64_t* empty = full + kMaxStages;
    uint64_t* recv = full + 2 * kMaxStages;  // cluster merge: this CTA's column slice arrived
    uint8_t* ring = smem + Lay::RING_OFF;
    // The Q rows are staged in the ring's last stage: once every consumer warp holds its Q
    // fragments in registers it releases that stage (one extra phase of empty[S - 1]), and
    // only then does the producer load a key tile there.
    uint8_t* sQ = ring + (S - 1) * stage_bytes;
    static_assert(kRowTile * Lay::ROW <= Lay::TILE, "Q rows fit in one ring stage");

    // The producer warp initialises the ring's barriers and starts its loads at once; the
    // consumer warps meanwhile stage the Q rows, and wait for both at named barrier 2.
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int s = 0; s < S; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
            }
            if (clustered) mbar_init(recv, 1);
            fence_barrier_init();
            if (clustered) {
                // every chunk sends this CTA its rows' slice of columns and its (m, l) pairs
                const int c0 = merge_col(split, D, p.n_split), c1 = merge_col(split + 1, D, p.n_split);
                mbar_arrive_expect_tx(recv, (uint32_t)(p.n_split * n_rows * ((c1 - c0) * 4 + 8)));
            }
        }
        __syncwarp();
        named_bar_arrive(2, kRowsThreads);
    } else {
        // Q rows of the tile (zero beyond n_rows), P = 0, row statistics
        const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q);
        constexpr int CH = D / 8;
        for (int idx = threadIdx.x; idx < kRowTile * CH; idx += kConsumerWarps * 32) {
            const int r = idx / CH, ch = idx - r * CH;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < n_rows) {
                const RowInfo ri = row_info(p, len, kvh, row0 + r);
                v = __ldg(reinterpret_cast<const uint4*>(
                    q + (((size_t)b * p.n_tok + ri.token) * p.n_q + ri.head) * (size_t)D + ch * 8));
            }
            *reinterpret_cast<uint4*>(sQ + r * Lay::ROW + ch * 16) = v;
        }
        uint32_t* p32 = reinterpret_cast<uint32_t*>(sP);
        for (int idx = threadIdx.x; idx < kRowTile * Lay::P_STRIDE / 2; idx += kConsumerWarps * 32)
            p32[idx] = 0u;
        if (threadIdx.x < 3 * kRowTile) sAlpha[threadIdx.x] = 0.f;
        named_bar_sync(2, kRowsThreads);
    }

    if (warp == kConsumerWarps) {
        // ---------------- producer warp: tiled TMA loads of the K/V rows in range --------------
        if (p.k_new) {
            // fused append: the CTA whose chunk holds the new slot (split 0 when no chunk does)
            // writes this KV head's new K/V row before any TMA load reads the cache
            const int wp = __ldg(p.write_pos + b);
            const bool in_range = wp >= first.lo && wp <= last.pos;
            const bool writer = rt == 0 && (in_range ? (wp >= kb && wp < ke) : split == 0);
            if (writer) {
                int wrow = 0, wslot = 0;
                if (wp < 0 || (!p.ring && wp >= p.cap)) {
                    if (lane == 0) report(p.err, GEMMA_DEVERR_WRITE_POS);
                } else if (!kv_place(p, b, kvh, wp, wrow, wslot)) {
                    if (lane == 0) report(p.err, GEMMA_DEVERR_PAGE);
                } else {
                    const size_t src = ((size_t)b * p.n_kv + kvh) * (size_t)D;
                    const size_t dst =
                        ((size_t)wrow * (size_t)kv_row_slots(p) + wslot) * (size_t)D;
                    for (int c = lane; c < D / 8; c += 32) {
                        const uint4 kv4 = __ldg(reinterpret_cast<const uint4*>(
                            reinterpret_cast<const __nv_bfloat16*>(p.k_new) + src) + c);
                        reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(
                            reinterpret_cast<const __nv_bfloat16*>(p.k) + dst))[c] = kv4;
                        if (!p.k_eq_v) {
                            const uint4 vv4 = __ldg(reinterpret_cast<const uint4*>(
                                reinterpret_cast<const __nv_bfloat16*>(p.v_new) + src) + c);
                            reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(
                                reinterpret_cast<const __nv_bfloat16*>(p.v) + dst))[c] = vv4;
                        }
                    }
                    fence_proxy_async_global();
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            for (int t = 0; t < n_tiles; ++t) {
                const int s = t % S;
                // stage S - 1 has one extra phase: the consumers' release of the Q rows
                const int ph = t / S - (s == S - 1 ? 0 : 1);
                if (ph >= 0 && !mbar_wait(&empty[s], ph & 1, p.err)) break;
                uint8_t* dk = ring + s * stage_bytes;
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                // cache row and slot of the tile's first key (a bad page index reads zeros)
                int row3 = 0, slot0 = 0;
                if (!kv_place(p, b, kvh, kb + t * T, row3, slot0)) {
                    report(p.err, GEMMA_DEVERR_PAGE);
                    row3 = p.n_pages * p.n_kv;
                }
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_3d(dk + c * Lay::BOX, &kmap, c * 64, slot0, row3, &full[s]);
                    if (nops == 2)
                        tma_load_3d(dk + Lay::TILE + c * Lay::BOX, &vmap, c * 64, slot0, row3,
                                    &full[s]);
                }
            }
        }
        if (clustered) {  // the merge's two cluster barriers (every thread of the cluster)
            rows_cluster_sync();
            rows_cluster_arrive_release();
            rows_cluster_wait();
        }
        return;
    }

    // ---------------------------------- consumer warps ----------------------------------------
    const int ng = warp % NGROUPS;  // S columns [ng*NTW*8, +NTW*8)
    const int kp = warp / NGROUPS;  // head_dim part [kp*D/KSPLIT, +D/KSPLIT)
    const int g = lane >> 2, tq = lane & 3;

    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int d0 = kp * (D / KSPLIT) + ks * 16;
        const uint32_t addr = smem_u32(sQ + (lane & 15) * Lay::ROW + (d0 + (lane >> 4) * 8) * 2);
        ldsm_x4(addr, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[S - 1]);  // this warp's Q fragments are in registers

    // rows owned by this warp in the softmax step: warp and warp + 8
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int r_lo[2], r_hi[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = warp + 8 * rr;
        if (r < n_rows) {
            const RowInfo ri = row_info(p, len, kvh, row0 + r);
            r_lo[rr] = ri.lo;
            r_hi[rr] = ri.pos + 1;
        } else {
            r_lo[rr] = 1;
            r_hi[rr] = 0;
        }
    }

    float o[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    // A wait that gives up (recorded in the error word) makes this warp stop waiting but keep
    // walking the tile loop, so every consumer warp still reaches every named barrier.
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int s = t % S;
        if (ok) ok = mbar_wait(&full[s], (t / S) & 1, p.err);
        const uint8_t* tK = ring + s * stage_bytes;
        const uint8_t* tV = nops == 2 ? tK + Lay::TILE : tK;
        const int rows_valid = min(T, n_keys - t * T);
        // a tile-aligned chunk (ring cache, paged pool) may start before every row's window:
        // those leading keys are masked, and their values zeroed like the rows past the end
        const int rows_head = max(0, first.lo - (kb + t * T));

        // (1) partial S over this warp's head_dim part
        {
            float sacc[NTW][4];
#pragma unroll
            for (int j = 0; j < NTW; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
            for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
                const int d0 = kp * (D / KSPLIT) + ks2 * 32;
#pragma unroll
                for (int j = 0; j < NTW; ++j) {
                    const int key = (ng * NTW + j) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(tK + tile_off<D>(key, d0 + (lane >> 3) * 8)), b0, b1, b2, b3);
                    mma_bf16(sacc[j], qa[2 * ks2][0], qa[2 * ks2][1], qa[2 * ks2][2],
                             qa[2 * ks2][3], b0, b1);
                    mma_bf16(sacc[j], qa[2 * ks2 + 1][0], qa[2 * ks2 + 1][1], qa[2 * ks2 + 1][2],
                             qa[2 * ks2 + 1][3], b2, b3);
                }
            }
            float* Sk = sS + kp * kRowTile * Lay::S_STRIDE;
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int col = (ng * NTW + j) * 8 + 2 * tq;
                *reinterpret_cast<float2*>(Sk + g * Lay::S_STRIDE + col) =
                    make_float2(sacc[j][0], sacc[j][1]);
                *reinterpret_cast<float2*>(Sk + (g + 8) * Lay::S_STRIDE + col) =
                    make_float2(sacc[j][2], sacc[j][3]);
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);

        // (2) online softmax of rows warp and warp + 8: lane = key of the tile. At head_dim 512
        // (every row of the tile real: 16 query heads per KV head) the two rows go through each
        // step together, so that their shuffle and exponential latencies overlap.
        if constexpr (D >= 512) {
            float sv[2], pe[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = warp + 8 * rr;
                const int key = kb + t * T + lane;
                const bool valid = r < n_rows && lane < rows_valid && key >= r_lo[rr] && key < r_hi[rr];
                float acc = 0.f;
#pragma unroll
                for (int kq = 0; kq < KSPLIT; ++kq) acc += sS[(kq * kRowTile + r) * Lay::S_STRIDE + lane];
                if (!valid) sv[rr] = -INFINITY;
                else if (p.softcap > 0.f) sv[rr] = p.cap_log2 * tanhf(acc * p.cap_inner);
                else sv[rr] = acc * p.scale_log2;
                pe[rr] = fast_exp2(sv[rr] - (m_run[rr] == -INFINITY ? 0.f : m_run[rr]));
            }
            float mx0 = sv[0], mx1 = sv[1];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = warp + 8 * rr;
                const float mx = rr ? mx1 : mx0;
                float alpha = 1.f;
                if (mx > m_run[rr] + kLazyRescaleLog2) {  // the same decision in every lane
                    alpha = fast_exp2(m_run[rr] - mx);   // 0 while the reference is -inf
                    m_run[rr] = mx;
                    pe[rr] = fast_exp2(sv[rr] - mx);
                }
                if (r < n_rows) {
                    const __nv_bfloat16 pb = __float2bfloat16_rn(pe[rr]);
                    sP[r * Lay::P_STRIDE + lane] = pb;
                    l_run[rr] = l_run[rr] * alpha + __bfloat162float(pb);
                    if (lane == 0) sAlpha[r] = alpha;
                }
            }
        } else {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = warp + 8 * rr;
                if (r < n_rows) {
                    const int key = kb + t * T + lane;
                    const bool valid = lane < rows_valid && key >= r_lo[rr] && key < r_hi[rr];
                    float sv = 0.f;
#pragma unroll
                    for (int kq = 0; kq < KSPLIT; ++kq)
                        sv += sS[(kq * kRowTile + r) * Lay::S_STRIDE + lane];
                    // scaled score in log2 units (soft-capped when a cap is set); masked keys -inf
                    if (!valid) sv = -INFINITY;
                    else if (p.softcap > 0.f) sv = p.cap_log2 * tanhf(sv * p.cap_inner);
                    else sv *= p.scale_log2;
                    // exponentials against the running reference maximum while the tile maximum
                    // is reduced; the reference moves (and the row is recomputed) only when the
                    // tile maximum exceeds it by more than 2^8, so the result is unchanged (the
                    // final division uses the same reference) and the common tile has no
                    // maximum -> exponential dependency. l is kept per lane (every lane's share is
                    // rescaled alike) and summed over the warp once, at the end.
                    const float m_old = m_run[rr];
                    float pe = exp2f(sv - (m_old == -INFINITY ? 0.f : m_old));
                    const float mx = warp_max(sv);
                    float alpha = 1.f;
                    if (mx > m_old + kLazyRescaleLog2) {  // the same decision in every lane
                        alpha = exp2f(m_old - mx);         // 0 while the reference is -inf
                        m_run[rr] = mx;
                        pe = exp2f(sv - mx);
                    }
                    const __nv_bfloat16 pb = __float2bfloat16_rn(pe);
                    sP[r * Lay::P_STRIDE + lane] = pb;
                    l_run[rr] = l_run[rr] * alpha + __bfloat162float(pb);
                    if (lane == 0) sAlpha[r] = alpha;
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);

        // (3) O = diag(alpha) O + P V over this warp's columns [warp*D/8, +D/8)
        {
            const float a_lo = sAlpha[g], a_hi = sAlpha[g + 8];
            if (a_lo != 1.f || a_hi != 1.f) {  // the reference moved for one of these rows
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    o[j][0] *= a_lo;
                    o[j][1] *= a_lo;
                    o[j][2] *= a_hi;
                    o[j][3] *= a_hi;
                }
            }
#pragma unroll
            for (int kk = 0; kk < T / 16; ++kk) {
                uint32_t pa0, pa1, pa2, pa3;
                ldsm_x4(smem_u32(sP + (lane & 15) * Lay::P_STRIDE + kk * 16 + (lane >> 4) * 8), pa0,
                        pa1, pa2, pa3);
                // keys of this thread's B fragment halves: k0, k0+1 (low) and k0+8, k0+9 (high)
                const int k0 = kk * 16 + 2 * tq;
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (rows_valid < T || rows_head > 0) {
                    // rows past the tile's end (not loaded) or before every window: zero them
                    auto in = [&](int k) { return k >= rows_head && k < rows_valid; };
                    mlo = (in(k0) ? 0x0000ffffu : 0u) | (in(k0 + 1) ? 0xffff0000u : 0u);
                    mhi = (in(k0 + 8) ? 0x0000ffffu : 0u) | (in(k0 + 9) ? 0xffff0000u : 0u);
                }
                const int vkey = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int j = 0; j < NB; j += 2) {
                    const int col = warp * (D / 8) + j * 8 + (lane >> 4) * 8;
                    if (j + 1 < NB) {
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_t(smem_u32(tV + tile_off<D>(vkey, col)), v0, v1, v2, v3);
                        mma_bf16(o[j], pa0, pa1, pa2, pa3, v0 & mlo, v1 & mhi);
                        mma_bf16(o[j + 1], pa0, pa1, pa2, pa3, v2 & mlo, v3 & mhi);
                    } else {
                        uint32_t v0, v1;
                        const int c1 = warp * (D / 8) + j * 8;
                        asm volatile(
                            "ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                            : "=r"(v0), "=r"(v1)
                            : "r"(smem_u32(tV + tile_off<D>(vkey, c1))));
                        mma_bf16(o[j], pa0, pa1, pa2, pa3, v0 & mlo, v1 & mhi);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------- epilogue -------------------------------------------
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = warp + 8 * rr;
        if (r < n_rows) {  // the same in every lane of the warp
            const float lt = warp_sum(l_run[rr]);
            if (lane == 0) {
                sM[r] = m_run[rr];
                sL[r] = lt;
            }
        }
    }
    named_bar_sync(1, kConsumerWarps * 32);

    if (clustered) {
        // CTA c of the cluster merges the column pairs [c P / n, (c + 1) P / n) (P = D / 2) of
        // every row over the n chunks:
        //   M = max_k m_k,  w_k = 2^(m_k - M),  out = sum_k w_k O_k / sum_k w_k l_k.
        // After one cluster barrier (every chunk has consumed its tiles, so every ring is
        // free), each chunk sends each owner its rows' part of the owner's slice and its (m, l)
        // pairs with asynchronous stores that complete on the owner's recv barrier, into the
        // owner's ring: O_k as [n][16][SW] floats, then (m, l) as [n][16] pairs. The owner
        // merges from its own shared memory. The second cluster barrier's arrive (release:
        // this thread's stores have landed) comes before the wait for the slice, and its wait
        // at the end, so no CTA leaves while a store into it or from it is in flight.
        const int ns = p.n_split;
        const int SW = 2 * ((D / 2 + ns - 1) / ns);  // widest slice, in floats
        float* recvO = reinterpret_cast<float*>(ring);
        float2* recvML = reinterpret_cast<float2*>(recvO + ns * kRowTile * SW);
        rows_cluster_sync();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = g + 8 * half;
            if (r >= n_rows) continue;
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int col = warp * (D / 8) + j * 8 + 2 * tq;
                const int owner = merge_owner(col, D, ns);
                const int c0 = merge_col(owner, D, ns);
                st_async_v2(rows_map_peer(recvO + (split * kRowTile + r) * SW + (col - c0), owner),
                            o[j][2 * half], o[j][2 * half + 1], rows_map_peer(recv, owner));
            }
        }
        for (int i = threadIdx.x; i < n_rows * ns; i += kConsumerWarps * 32) {
            const int r = i / ns, dst = i - r * ns;
            st_async_v2(rows_map_peer(recvML + split * kRowTile + r, dst), sM[r], sL[r],
                        rows_map_peer(recv, dst));
        }
        rows_cluster_arrive_release();
        const bool got = mbar_wait_cluster(recv, 0, p.err);
        const int c0 = merge_col(split, D, ns), nc = merge_col(split + 1, D, ns) - c0;
        for (int idx = threadIdx.x; got && idx < n_rows * nc; idx += kConsumerWarps * 32) {
            const int r = idx / nc, c = idx - r * nc;
            float M = -INFINITY;
            for (int k = 0; k < ns; ++k) M = fmaxf(M, recvML[k * kRowTile + r].x);
            float L = 0.f, acc = 0.f;
            for (int k = 0; k < ns; ++k) {
                const float2 ml = recvML[k * kRowTile + r];
                const float wk = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
                L = fmaf(wk, ml.y, L);
                acc = fmaf(wk, recvO[(k * kRowTile + r) * SW + c], acc);
            }
            const RowInfo ri = row_info(p, len, kvh, row0 + r);
            reinterpret_cast<__nv_bfloat16*>(p.out)[(((size_t)b * p.n_tok + ri.token) * p.n_q +
                                                     ri.head) * (size_t)D + c0 + c] =
                __float2bfloat16_rn(acc / L);
        }
        rows_cluster_wait();
        return;
    }

    if constexpr (!CLUSTER) {  // the chunk's rows: final (unsplit) or a partial for the combine
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = g + 8 * half;
            if (r >= n_rows) continue;
            const RowInfo ri = row_info(p, len, kvh, row0 + r);
            if (direct) {
                const float inv = 1.f / sL[r];
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                     (((size_t)b * p.n_tok + ri.token) * p.n_q + ri.head) * (size_t)D;
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int col = warp * (D / 8) + j * 8 + 2 * tq;
                    *reinterpret_cast<uint32_t*>(dst + col) =
                        pack_bf16(o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
                }
            } else {
                const size_t pr = ((size_t)b * p.n_q + ri.head) * p.n_split + split;
                float* dst = p.o_part + pr * D;
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int col = warp * (D / 8) + j * 8 + 2 * tq;
                    *reinterpret_cast<float2*>(dst + col) = make_float2(o[j][2 * half], o[j][2 * half + 1]);
                }
                if (warp == 0 && tq == 0) {
                    p.ml_part[pr * 2 + 0] = sM[r];
                    p.ml_part[pr * 2 + 1] = sL[r];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// fp32 debug path: one warp per row, lanes split head_dim, FFMA with expf (accuracy first).
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kF32RowsPerCta * 32) rows_attn_f32_kernel(const RowsParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.n_split;
    const int rt = blockIdx.x / p.n_split;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int R = rt * kF32RowsPerCta + warp;
    if (R >= p.n_tok * p.G) return;
    const int len = __ldg(p.seq_lens + b);
    const bool direct = p.n_split == 1;
    const int token = R / p.G, head = kvh * p.G + (R - token * p.G);
    float* out_row = reinterpret_cast<float*>(p.out) +
                     (((size_t)b * p.n_tok + token) * p.n_q + head) * (size_t)D;
    // real tokens of this sequence (a padded bucket's first n_real rows; all rows otherwise)
    const int n_real = p.n_real ? __ldg(p.n_real + b) : p.n_tok;
    const bool bad_real = n_real < 0 || n_real > p.n_tok;
    const bool bad = bad_real || len < n_real || (!p.ring && len > p.cap) || len > p.max_seq_len;
    if (bad || token >= n_real) {  // a bad sequence, or a pad row: zero output
        if (split == 0) {
            if (bad && lane == 0) report(p.err, bad_real ? GEMMA_DEVERR_N_REAL : GEMMA_DEVERR_SEQ_LEN);
            if (direct)
                for (int e = 0; e < E; ++e) out_row[lane + 32 * e] = 0.f;
        }
        return;
    }
    const int pos = len - n_real + token;
    const int lo = p.is_sliding ? max(0, pos - p.window + 1) : 0;
    // chunks as in the bf16 kernel (a ring cache's start at multiples of the key tile)
    const int kb = ((p.ring || p.page_size) ? (lo & ~(kKeyTile - 1)) : lo) + split * p.chunk;
    const int ke = min(pos + 1, kb + p.chunk);
    if (kb >= ke) return;

    const float* q = reinterpret_cast<const float*>(p.q) +
                     (((size_t)b * p.n_tok + token) * p.n_q + head) * (size_t)D;
    const float* K = reinterpret_cast<const float*>(p.k);
    const float* V = reinterpret_cast<const float*>(p.v);
    const size_t rs = (size_t)kv_row_slots(p);
    float qr[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qr[e] = q[lane + 32 * e];
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int j = max(kb, lo); j < ke; ++j) {
        int krow = 0, kslot = 0;
        if (!kv_place(p, b, kvh, j, krow, kslot)) {  // a bad page index: the key is skipped
            if (lane == 0) report(p.err, GEMMA_DEVERR_PAGE);
            continue;
        }
        const size_t row = (size_t)krow * rs + (size_t)kslot;  // cache row of key j
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qr[e], K[row * D + lane + 32 * e], dot);
        float s = warp_sum(dot) * p.scale;
        if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap);
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);
        const float w = expf(s - m_new);
        l = l * alpha + w;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, V[row * D + lane + 32 * e], acc[e] * alpha);
        m = m_new;
    }
    if (direct) {
        const float inv = 1.f / l;
#pragma unroll
        for (int e = 0; e < E; ++e) out_row[lane + 32 * e] = acc[e] * inv;
    } else {
        const size_t pr = ((size_t)b * p.n_q + head) * p.n_split + split;
#pragma unroll
        for (int e = 0; e < E; ++e) p.o_part[pr * D + lane + 32 * e] = acc[e];
        if (lane == 0) {
            p.ml_part[pr * 2 + 0] = m * 1.4426950408889634f;  // natural -> log2 units
            p.ml_part[pr * 2 + 1] = l;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// split-K combine (decode): merge the per-chunk (m, l, O) of each (sequence, query head)
//   M = max_c m_c,  w_c = 2^(m_c - M),  out = sum_c w_c O_c / sum_c w_c l_c
// ---------------------------------------------------------------------------------------------
// One CTA per (query head, slice of head_dim, sequence): the whole row when the (head,
// sequence) pairs already fill the GPU, 128-column slices when they do not (small batches).
// The chunk weights w_c and their sum are computed once into shared memory; then groups of
// threads each accumulate a share of the chunks for the slice's columns (one float4 per
// thread, several L2 reads in flight), and the groups are summed through shared memory.
constexpr int kCombineThreads = 256;
constexpr int kCombineSlice = 128;  // columns per CTA when rows are sliced

template <typename OutT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const RowsParams p, int D, int n_slices) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    __shared__ float s_w[128];                                  // chunk weights (n_split <= 128)
    __shared__ float4 s_red[kCombineThreads];
    __shared__ float s_inv;
    const int SW = D / n_slices;
    const int head = blockIdx.x / n_slices, col0 = (blockIdx.x - head * n_slices) * SW;
    const int b = blockIdx.y;
    const int len = __ldg(p.seq_lens + b);
    OutT* dst = reinterpret_cast<OutT*>(p.out) + ((size_t)b * p.n_q + head) * (size_t)D + col0;
    const int tid = threadIdx.x;
    if (len < 1 || (!p.ring && len > p.cap) || len > p.max_seq_len) {
        for (int c = tid; c < SW; c += blockDim.x) dst[c] = OutT(0.f);
        return;
    }
    int lo = p.is_sliding ? max(0, len - p.window) : 0;
    if (p.ring || p.page_size) lo &= ~(kKeyTile - 1);  // chunks start at a tile boundary there
    const int nc = min(p.n_split, (len - lo + p.chunk - 1) / p.chunk);
    const size_t base = ((size_t)b * p.n_q + head) * p.n_split;
    if (tid < 32) {
        // warp 0: M = max_c m_c, w_c = 2^(m_c - M), L = sum_c w_c l_c
        float m[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = tid + 32 * i;
            m[i] = c < nc ? p.ml_part[(base + c) * 2] : -INFINITY;
            l[i] = c < nc ? p.ml_part[(base + c) * 2 + 1] : 0.f;
        }
        const float M = warp_max(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])));
        float L = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = tid + 32 * i;
            const float w = c < nc ? exp2f(m[i] - M) : 0.f;
            if (c < 128) s_w[c] = w;
            L = fmaf(w, l[i], L);
        }
        L = warp_sum(L);
        if (tid == 0) s_inv = 1.f / L;
    }
    __syncthreads();
    const int tpg = SW / 4;                      // threads per chunk group (one float4 each)
    const int n_grp = kCombineThreads / tpg;     // chunk groups
    const int grp = tid / tpg, c4 = tid - grp * tpg;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int c = grp; c < nc; c += n_grp) {
        const float w = s_w[c];
        const float4 v = *reinterpret_cast<const float4*>(p.o_part + (base + c) * D + col0 + c4 * 4);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    s_red[tid] = acc;
    __syncthreads();
    if (grp == 0) {
        float4 t = s_red[c4];
        for (int g2 = 1; g2 < n_grp; ++g2) {
            const float4 u = s_red[g2 * tpg + c4];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        const float inv = s_inv;
        dst[c4 * 4 + 0] = OutT(t.x * inv);
        dst[c4 * 4 + 1] = OutT(t.y * inv);
        dst[c4 * 4 + 2] = OutT(t.z * inv);
        dst[c4 * 4 + 3] = OutT(t.w * inv);
    }
}

// ---------------------------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------------------------
template <int D>
static size_t smem_for(int k_eq_v, int* n_stages) {
    using Lay = RowsLayout<D>;
    const int stage = (k_eq_v ? 1 : 2) * Lay::TILE;
    const int fixed = Lay::RING_OFF + 1024;  // + alignment slack of the dynamic buffer
    int s = (kSmemBudget - fixed) / stage;
    s = s < 2 ? 2 : (s > kMaxStages ? kMaxStages : s);
    if (n_stages) *n_stages = s;
    return (size_t)fixed + (size_t)s * stage;
}

size_t rows_bf16_smem_bytes(int head_dim, int k_eq_v, int* n_stages) {
    switch (head_dim) {
        case 64: return smem_for<64>(k_eq_v, n_stages);
        case 128: return smem_for<128>(k_eq_v, n_stages);
        case 256: return smem_for<256>(k_eq_v, n_stages);
        case 512: return smem_for<512>(k_eq_v, n_stages);
    }
    return 0;
}

template <int D>
static cudaError_t launch_bf16_d(const RowsParams& p, dim3 grid, size_t smem, cudaStream_t st) {
    auto kernel = p.cluster ? rows_attn_bf16_kernel<D, true> : rows_attn_bf16_kernel<D, false>;
    // attribute set once per device (the same value every time, so concurrent first calls
    // from several host threads are harmless)
    static std::atomic<bool> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(rows_attn_bf16_kernel<D, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(rows_attn_bf16_kernel<D, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        // clusters of up to 16 chunks (above the portable 8)
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(rows_attn_bf16_kernel<D, true>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_relaxed);
    }
    CUtensorMap km, vm;
    // [rows][slots][D]: rows = sequences x KV heads (pages x KV heads for a paged pool)
    const uint64_t map_slots = p.page_size ? (uint64_t)p.page_size : (uint64_t)p.cap;
    const uint64_t map_rows = p.page_size ? (uint64_t)p.n_pages * p.n_kv : (uint64_t)grid.z * p.n_kv;
    const uint64_t dims[3] = {(uint64_t)D, map_slots, map_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, map_slots * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kKeyTile, 1};
    if (!encode_bf16_sw128(&km, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&vm, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!p.cluster)
        return launch_pdl(kernel, grid, dim3(kRowsThreads), smem, st, km, vm, p);
    // the chunks of a row tile (consecutive blockIdx.x) form one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kRowsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.n_split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, km, vm, p);
}

cudaError_t launch_rows_bf16(const RowsParams& p, int head_dim, dim3 grid, size_t smem,
                             cudaStream_t st) {
    switch (head_dim) {
        case 64: return launch_bf16_d<64>(p, grid, smem, st);
        case 128: return launch_bf16_d<128>(p, grid, smem, st);
        case 256: return launch_bf16_d<256>(p, grid, smem, st);
        case 512: return launch_bf16_d<512>(p, grid, smem, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_rows_f32(const RowsParams& p, int head_dim, dim3 grid, cudaStream_t st) {
    const dim3 block(kF32RowsPerCta * 32);
    switch (head_dim) {
        case 64: return launch_pdl(rows_attn_f32_kernel<64>, grid, block, 0, st, p);
        case 128: return launch_pdl(rows_attn_f32_kernel<128>, grid, block, 0, st, p);
        case 256: return launch_pdl(rows_attn_f32_kernel<256>, grid, block, 0, st, p);
        case 512: return launch_pdl(rows_attn_f32_kernel<512>, grid, block, 0, st, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const RowsParams& p, int head_dim, int batch, int out_fp32,
                           cudaStream_t st) {
    int n_sm = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int n_slices = ((long long)p.n_q * batch >= 2LL * n_sm || head_dim <= kCombineSlice)
                             ? 1
                             : head_dim / kCombineSlice;
    const dim3 grid(p.n_q * n_slices, batch);
    const dim3 block(kCombineThreads);
    if (out_fp32)
        return launch_pdl(combine_kernel<float>, grid, block, 0, st, p, head_dim, n_slices);
    return launch_pdl(combine_kernel<__nv_bfloat16>, grid, block, 0, st, p, head_dim, n_slices);
}

}  // namespace gemma
