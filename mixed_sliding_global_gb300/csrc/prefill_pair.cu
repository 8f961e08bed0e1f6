// prefill_pair.cu -- prefill-bucket attention at head_dim 256 and 512 on CTA pairs (the 2-SM form
// of the 5th-generation tensor-core MMA, tcgen05 with cta_group::2).
//
// Computes, for tiles of 256 query rows (rows = (token, head of the GQA group) pairs, token
// major, so every row of a tile reads the same KV head), softmax(scale * Q K^T) V over the
// causal (and, on sliding layers, windowed) key range of each row, with the K/V cache of the
// owner layer ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", sections 2.1-2.3; the
// pages' "eager" matmul-softmax-matmul definition, section 4.3). The sliding layers of every
// Gemma-4 size have head_dim 256, the global layers 512.
//
// A cluster of two CTAs (one per SM) runs each MMA as one instruction of M = 256: CTA c owns
// rows 128c..128c+127 of the tile (its Q rows in its shared memory, its rows of S, P and O in
// its tensor memory), and each CTA holds half of every B operand. Per 128-key tile:
//   S = Q K^T   N = 128 keys: CTA c holds keys 64c..64c+63 of K (all 256 columns, 32 KB);
//   O += P V    N = 256 columns: CTA c holds columns 128c..128c+127 of V (all 128 keys, 32 KB).
// So a 128-key step needs 64 KB of shared memory per SM (a one-SM 128-key step needs 128 KB),
// S runs at N = 128 (an MMA of N = 64 costs as much as one of N = 128), and one step issues 24
// MMAs where one-SM 64-key steps issue 40 for the same keys.
//
// Head_dim 512 (H = 2): a 128-row O of 512 fp32 columns alone would fill one SM's tensor memory,
// so a cluster holds two pairs, pair h owning columns 256h..256h+255 of Q, K, V and O and running
// everything above on them. Its S is a partial over its half: each softmax group sends its
// columns of the partial to the partner CTA (cluster rank ^ 2) as saturating fp16 with st.async
// (bytes counted on the partner's mbarrier), and adds the partner's partial to its own fp32 one,
// so the partner's rounding moves a score by at most 2^-11 of its partial. The ring has 3 slots
// to make room for the 32 KB receive buffer.
//
// Persistent grid: each pair walks work units = (256-row tile, sequence, KV head), latest row
// tiles (longest key ranges) first; the 128-key tiles of all its units form one flat sequence.
// Warps of each CTA:
//   warps 0-7   softmax: thread r of warpgroup w owns row r (TMEM lane r) and the 64 columns
//               64w..64w+63 of each S tile, and columns 128w..128w+127 of O. The two groups
//               swap their row maxima through shared memory; the row's softmax reference moves
//               only when a tile maximum exceeds it by more than 2^8 (lazy rescaling keeps the
//               result exact: the final division uses the same reference), and O rows are
//               rescaled in TMEM when it moves. P goes to tensor memory as bf16 (two buffers,
//               so the softmax of tile t+1 does not wait for the P V of tile t).
//   warp 8      TMA producer: each unit's Q rows (once the previous unit's last S has read the
//               Q buffer) and this CTA's halves of the K and V tiles (128-byte swizzle, boxes of
//               64 keys x 64 columns) into a FIFO ring of 32 KB slots, in the MMA order.
//   warp 9      even CTA: issues S(t) = Q K(t)^T once both CTAs' softmax warps have read S(t-1),
//               so the softmax of tile t overlaps the P V of tile t-1 and the S of tile t+1.
//               Odd CTA: forwards each of its ring slots' arrivals to the even CTA's barriers
//               (an MMA reads both CTAs' halves).
//   warp 10     even CTA: issues O += P(t) V(t) once both CTAs' P(t) is in tensor memory.
// Barriers that the issuers wait on live in the even CTA and count arrivals from both CTAs;
// the issuers' commits arrive on the same barrier in both CTAs (multicast). Arrivals from the
// odd CTA are plain remote arrivals: a thread that wrote shared memory an MMA reads (zeroed V
// rows) orders those writes before the async proxy with a proxy fence first, and one that read
// or wrote tensor memory fences its tcgen05 operations before the arrival.
// TMEM (512 columns per CTA): S (128 fp32) at 0, P (2 x 64 columns of packed bf16) at 128, O
// (256 fp32) at 256. Shared memory: the ring (4 slots; 3 at head_dim 512), Q (64 KB), the
// epilogue's staging (O / l leaves in 32-column slices by TMA tensor stores).
// The Q rows of a 128-row half tile are G consecutive heads of 128 / G consecutive tokens, one
// TMA box per 64 columns; the kernel needs G to divide 128.
//
// The key range of a unit is clamped to [first row's window start, last row's position] before
// any load; rows of a V tile outside the range are zeroed in shared memory before they enter
// P V (they may hold anything, NaN included).
#include <atomic>

#include "attn_internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace gemma {

namespace {

constexpr int kPrWarps = 11;
constexpr int kPrThreads = kPrWarps * 32;
constexpr int kPrProducerWarp = 8;
constexpr int kPrSWarp = 9;     // S issuer (even CTA) / slot forwarder (odd CTA)
constexpr int kPrPvWarp = 10;   // P V issuer (even CTA)
constexpr int kPrKeys = 128;                  // keys per tile (N of S)
constexpr int kPrRows = 256;                  // rows per unit (M of the pair's MMAs)
constexpr int kPrBox = 64 * 128;              // TMA box: 64 keys x 64 columns of bf16
constexpr int kPrSlot = 4 * kPrBox;           // K half (64 keys x 256) or V half (128 x 128)
constexpr int kPrQBytes = 128 * 256 * 2;      // a CTA's Q rows: 4 boxes of 128 rows x 64 columns
constexpr int kPrQBox = 128 * 128;            // one of them
constexpr int kPrStage = 2 * 128 * 64;        // epilogue: 2 groups x 128 rows x 32 columns bf16
constexpr int kPrSmemLimit = 232448;          // max dynamic shared memory per block
constexpr int kPrListMax = 512;               // units a padded bucket's work list holds
constexpr float kPrLazyLog2 = 8.f;
constexpr int kPrSCol = 0, kPrPCol = 128, kPrOCol = 256;  // TMEM columns
// H parts of head_dim (256 columns each): a cluster of H pairs. Shared memory: ring, Q,
// staging, the partner pair's partial scores (H = 2: [2 groups][8 chunks][128 rows] x 16
// bytes), row maxima [2 tiles][2 groups][128], row sums [2][128], barriers.
template <int H>
struct PrLay {
    static constexpr int D = 256 * H;                  // head_dim
    static constexpr int SLOTS = H == 1 ? 4 : 3;       // ring slots
    static constexpr int Q_OFF = SLOTS * kPrSlot;
    static constexpr int STAGE_OFF = Q_OFF + kPrQBytes;
    static constexpr int X_OFF = STAGE_OFF + kPrStage;
    static constexpr int X_BYTES = H == 2 ? 128 * kPrKeys * 2 : 0;
    static constexpr int MX_OFF = X_OFF + X_BYTES;
    static constexpr int BAR_OFF = MX_OFF + (2 * 2 * 128 + 2 * 128) * 4;
    static constexpr int ULIST_OFF = BAR_OFF + 256;    // a padded bucket's work list
    static constexpr int SMEM = ULIST_OFF + (kPrListMax + 1) * 4 + 1024;  // + alignment slack
    static_assert(SMEM <= kPrSmemLimit, "shared memory budget");
};

struct PrParams {
    RowsParams p;
    int batch;
    int n_rt;      // 256-row tiles per (sequence, KV head)
    int n_units;   // n_rt * batch * n_kv
    int n_pairs;   // clusters walking the units (each of H pairs)
};

struct PrUnit {
    int b, kvh, rt, row0;
    int n_rows;       // rows of the bucket this unit writes
    int n_rows_real;  // rows that attend (the rest are pad rows or a bad sequence: zeros)
    int len, n_real;
    bool bad, bad_real;
    int k_begin, k_end, n_tiles;
    int n_head;       // leading keys of the first tile before every row's window (aligned start)
};

// Unit u: row tiles from the last (longest key ranges) to the first, then sequences, then KV
// heads.
__device__ __forceinline__ PrUnit pr_unit(const PrParams& fp, int u) {
    const RowsParams& p = fp.p;
    PrUnit U;
    const int per_rt = fp.batch * p.n_kv;
    const int q = u / per_rt, rem = u - q * per_rt;
    U.rt = fp.n_rt - 1 - q;
    U.b = rem / p.n_kv;
    U.kvh = rem - U.b * p.n_kv;
    const int rows_total = p.n_tok * p.G;
    U.row0 = U.rt * kPrRows;
    U.n_rows = min(kPrRows, rows_total - U.row0);
    U.len = __ldg(p.seq_lens + U.b);
    // real tokens of this sequence (a padded bucket's first n_real rows; all rows otherwise);
    // the i-th real token sits at len - n_real + i, the pad rows' outputs are zero
    U.n_real = p.n_real ? __ldg(p.n_real + U.b) : p.n_tok;
    U.bad_real = U.n_real < 0 || U.n_real > p.n_tok;
    U.bad = U.bad_real || U.len < U.n_real || (!p.ring && U.len > p.cap) || U.len > p.max_seq_len;
    U.n_rows_real = U.bad ? 0 : max(0, min(kPrRows, U.n_real * p.G - U.row0));
    // key range: from the first row's window start to the last real row's position (a ring
    // cache's or paged pool's 64-key groups start at multiples of 64, so that none wraps around
    // the ring or crosses a page; the rows' masks drop the keys before the window)
    const int tok_first = U.row0 / p.G;
    const int tok_last = (U.row0 + max(U.n_rows_real, 1) - 1) / p.G;
    const int pos_first = U.len - U.n_real + tok_first;
    const int lo_first = p.is_sliding ? max(0, pos_first - p.window + 1) : 0;
    U.k_begin = (p.ring || p.page_size) ? (lo_first & ~63) : lo_first;
    U.k_end = U.len - U.n_real + tok_last + 1;
    U.n_tiles = U.n_rows_real == 0 ? 0 : (U.k_end - U.k_begin + kPrKeys - 1) / kPrKeys;
    U.n_head = lo_first - U.k_begin;
    return U;
}

// One tile of the flat per-pair sequence, as the producer and the issuers see it.
struct PrTile {
    bool valid, first, last;
    int ord;       // ordinal of its unit among this pair's units that have tiles
    int n_valid;   // keys of the tile inside the unit's range (the rest are zeroed in V)
    int n_head;    // leading keys zeroed (first tile of an aligned-start unit)
    int key0;      // first key
    int b, kvh;
    int row0;      // the unit's first row
};

// LIST (a padded bucket): the units come from the work list in shared memory, entry j to
// worker j mod W, the units with key tiles first (so that pad rows' empty units take no
// worker's turn); otherwise worker w takes units w, w + W, w + 2W, ...
template <bool LIST>
struct PrTileIter {
    int u, stride, t, ord;
    const int* list;
    PrUnit U;
    __device__ __forceinline__ void init(const PrParams& fp, int worker, const int* ulist) {
        u = worker - fp.n_pairs;  // next() advances to the first unit
        stride = fp.n_pairs;
        list = ulist;
        t = 0;
        ord = -1;
        U.n_tiles = 0;
    }
    __device__ __forceinline__ PrTile next(const PrParams& fp) {
        PrTile T;
        T.valid = false;
        while (t >= U.n_tiles) {
            u += stride;
            if (u >= fp.n_units) return T;
            U = pr_unit(fp, LIST ? list[u] : u);
            t = 0;
            if (U.n_tiles > 0) ++ord;
        }
        T.valid = true;
        T.first = t == 0;
        T.last = t == U.n_tiles - 1;
        T.ord = ord;
        T.key0 = U.k_begin + t * kPrKeys;
        T.n_valid = min(kPrKeys, U.k_end - T.key0);
        T.n_head = t == 0 ? U.n_head : 0;
        T.b = U.b;
        T.kvh = U.kvh;
        T.row0 = U.row0;
        ++t;
        return T;
    }
};

}  // namespace

// SOFTCAP: the soft-capped variant; LIST: a padded bucket's, dealing out its units from the work
// list (separate instantiations, so that the plain kernel carries no code for either)
template <int H, bool SOFTCAP, bool LIST>
__global__ void __launch_bounds__(kPrThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap omap, const PrParams fp) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream (the append of these rows) has completed
    using Lay = PrLay<H>;
    constexpr int D = Lay::D;
    constexpr int kPrSlots = Lay::SLOTS;
    const RowsParams& p = fp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* slots = smem;
    uint8_t* sQ = smem + Lay::Q_OFF;                                  // [4][128][64] bf16
    uint8_t* sStage = smem + Lay::STAGE_OFF;                          // [2][128][32] bf16
    uint8_t* sX = smem + Lay::X_OFF;                                  // H = 2: partner's scores
    float* mxs = reinterpret_cast<float*>(smem + Lay::MX_OFF);        // [2][2][128]
    float* lxs = mxs + 2 * 2 * 128;                                   // [2][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFF);
    // ring slot s: full[s] completes when this CTA's half has landed (producer arrival +
    // transaction bytes); pfull[s] (even CTA) when the odd CTA's half has (its warp 9 forwards
    // its own full[s]); empty[s] when the MMAs that read the slot have completed (multicast).
    uint64_t* full = bars;
    uint64_t* pfull = bars + kPrSlots;
    uint64_t* empty = bars + 2 * kPrSlots;
    uint64_t* q_full = bars + 3 * kPrSlots;  // this CTA's Q rows of a unit have landed
    uint64_t* q_pfull = q_full + 1;          // even CTA: the odd CTA's have (forwarded)
    uint64_t* s_full = q_full + 2;           // S(t) is in TMEM (multicast commit)
    uint64_t* s_free = q_full + 3;           // even CTA: both CTAs' softmax warps have read S(t)
    uint64_t* p_full = q_full + 4;           // [2] even CTA: both CTAs' P(t) in TMEM buffer t % 2
    uint64_t* pv_done = q_full + 6;          // [2] P V(t) has completed (multicast commit)
    uint64_t* o_full = q_full + 8;           // a unit's last P V has completed (multicast)
    uint64_t* o_free = q_full + 9;           // even CTA: both epilogues have read O
    uint64_t* q_free = q_full + 10;          // a unit's last S has completed (multicast commit)
    uint64_t* x_full = q_full + 11;          // [2] H = 2: the partner's scores of group w landed
    uint64_t* x_free = q_full + 13;          // [2] H = 2: the partner has read what was sent
    uint32_t* tslot = reinterpret_cast<uint32_t*>(q_full + 15);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t c = rank & 1u;            // row half of the pair's tile; 0 issues its MMAs
    const uint32_t h = rank >> 1;            // H = 2: head_dim half (columns 256h..256h+255)
    const uint32_t lead = rank & ~1u;        // the pair's issuing CTA
    const uint16_t pair_mask = (uint16_t)(3u << lead);
    const int worker = blockIdx.x / (2 * H);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&pfull[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_pfull, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 16);  // 8 softmax warps per CTA
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], 16);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(o_free, 16);
        mbar_init(q_free, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&x_full[i], 1);  // one local arrival with the exchange's byte count
            mbar_init(&x_free[i], 4);  // the partner's four warps of the group have read it
        }
        fence_barrier_init();
    }
    // a padded bucket's work list: every thread evaluates units, warp 0 lists those with key
    // tiles first (in order), then the others
    int* ulist = reinterpret_cast<int*>(smem + Lay::ULIST_OFF);
    if constexpr (LIST) {
        for (int u = threadIdx.x; u < fp.n_units; u += blockDim.x)
            ulist[u] = pr_unit(fp, u).n_tiles > 0 ? 1 : 0;  // a flag first, then the entry
        __syncthreads();
        if (warp == 0) {
            // lane l owns units [16 l, 16 l + 16): its count of units with tiles, and the lanes
            // before it by a scan
            constexpr int PER = kPrListMax / 32;
            int flags = 0, cnt = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int u = PER * lane + i;
                const int f = u < fp.n_units ? ulist[u] : 0;
                flags |= f << i;
                cnt += f;
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int n_work = __shfl_sync(0xffffffffu, incl, 31);
            __syncwarp();  // every lane has read its flags before any entry is written
            int w_pos = incl - cnt;                            // next slot: a unit with tiles
            int z_pos = n_work + PER * lane - (incl - cnt);    // and one without
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int u = PER * lane + i;
                if (u < fp.n_units) {
                    if ((flags >> i) & 1) ulist[w_pos++] = u;
                    else ulist[z_pos++] = u;
                }
            }
        }
    }
    __syncthreads();
    // every CTA of the cluster runs and its barriers exist before the pair allocation, any
    // remote arrival or any multicast commit
    cluster_sync();
    if (warp == kPrSWarp) {  // one warp in each CTA, together
        tmem_alloc_pair(tslot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // rows of a V tile outside the unit's key range, zeroed (whole warp)
    auto zero_v = [&](uint8_t* tile, const PrTile& T) {
        const int n_tail = kPrKeys - T.n_valid;
        if (n_tail <= 0 && T.n_head <= 0) return;
        if (n_tail > 0) {
            for (int idx = lane; idx < 2 * n_tail * 8; idx += 32) {
                const int blk = idx / (n_tail * 8), rem = idx - blk * n_tail * 8;
                *reinterpret_cast<uint4*>(tile + blk * 2 * kPrBox + (T.n_valid + rem / 8) * 128 +
                                          (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (T.n_head > 0) {
            for (int idx = lane; idx < 2 * T.n_head * 8; idx += 32) {
                const int blk = idx / (T.n_head * 8), rem = idx - blk * T.n_head * 8;
                *reinterpret_cast<uint4*>(tile + blk * 2 * kPrBox + (rem / 8) * 128 +
                                          (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
    };

    if (warp == kPrProducerWarp) {
        // ------------------------------- TMA producer --------------------------------------
        // Loads in the MMA order: K(0), K(1), V(0), K(2), V(1), ... A slot is reused once the
        // MMAs that read its previous contents have completed. A unit's Q rows go first, once
        // the previous unit's last S (the last reader of the Q buffer) has completed.
        if (lane == 0) {
            bool ok = true;
            int L = 0;
            auto place = [&](const PrTile& T, int key, int& row3, int& slot0) {
                if (!kv_place(p, T.b, T.kvh, key, row3, slot0)) {
                    report(p.err, GEMMA_DEVERR_PAGE);  // a bad page index reads zeros
                    row3 = p.n_pages * p.n_kv;
                }
            };
            auto load = [&](const PrTile& T, bool is_v) {
                const int s = L % kPrSlots, use = L / kPrSlots;
                ++L;
                if (use > 0 && ok) ok = mbar_wait(&empty[s], (use - 1) & 1, p.err);
                mbar_arrive_expect_tx(&full[s], kPrSlot);
                if (!ok) return;
                uint8_t* dst = slots + s * kPrSlot;
                int row3 = 0, slot0 = 0;
                if (!is_v) {
                    // K: this CTA's 64 keys, the four 64-column boxes of head_dim
                    place(T, T.key0 + 64 * (int)c, row3, slot0);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_load_3d(dst + j * kPrBox, &kmap, 256 * (int)h + 64 * j, slot0, row3,
                                    &full[s]);
                } else {
                    // V: this CTA's 128 columns (two blocks of 64) of all 128 keys; block b
                    // holds keys 0-127 as 128-byte rows, the two 64-key groups one after another
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        place(T, T.key0 + 64 * g, row3, slot0);
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk)
                            tma_load_3d(dst + blk * 2 * kPrBox + g * kPrBox, &vmap,
                                        256 * (int)h + 128 * (int)c + 64 * blk, slot0, row3,
                                        &full[s]);
                    }
                }
            };
            PrTileIter<LIST> it;
            it.init(fp, worker, ulist);
            PrTile prev;
            prev.valid = false;
            int Tn = 0;
            for (;;) {
                const PrTile cur = it.next(fp);
                if (!cur.valid && !prev.valid) break;
                if (cur.valid && cur.first) {
                    // (a barrier of its own: this thread runs tiles ahead of the S MMAs, and a
                    // parity wait must not be more than one phase ahead of the barrier)
                    if (cur.ord > 0 && ok) ok = mbar_wait(q_free, (cur.ord - 1) & 1, p.err);
                    mbar_arrive_expect_tx(q_full, kPrQBytes);
                    const int tk0 = (cur.row0 + 128 * (int)c) / p.G;  // tokens past n_tok read 0
                    if (ok) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_4d(sQ + j * kPrQBox, &qmap, 256 * (int)h + 64 * j,
                                        cur.kvh * p.G, tk0, cur.b, q_full);
                    }
                }
                if (cur.valid) load(cur, false);
                if (prev.valid) load(prev, true);
                if (cur.valid) ++Tn;
                prev = cur;
            }
            // the last releases of the slots and of the Q buffer (arrivals of the MMA commits
            // on this CTA's barriers) have landed before the CTA may exit
            for (int k = 1; k <= kPrSlots && k <= L; ++k) {
                const int LL = L - k;
                if (ok) ok = mbar_wait(&empty[LL % kPrSlots], (LL / kPrSlots) & 1, p.err);
            }
            if (Tn > 0 && ok) ok = mbar_wait(q_free, it.ord & 1, p.err);
        }
    } else if (c == 0 && (warp == kPrSWarp || warp == kPrPvWarp)) {
        // ------------------ MMA issuers: S (warp 9) and P V (warp 10) -----------------------
        // An MMA is accepted only when the one before it is nearly done, so an issuing thread
        // is busy for about the tensor time of what it issues. With S and P V from separate
        // threads, one issuer's waits (for P, or for the softmax to have read S) leave the
        // tensor core to the other's MMAs. Both walk the producer's slot order.
        const bool is_s = warp == kPrSWarp;
        const uint32_t id_s = idesc_bf16(256, kPrKeys, 0, 0);
        const uint32_t id_pv = idesc_bf16(256, 256, 0, 1);
        const uint32_t tS = tmem + kPrSCol, tP = tmem + kPrPCol, tO = tmem + kPrOCol;
        bool ok = true;
        int L = 0;
        // the next slot with both CTAs' halves landed (V: its edge rows zeroed here)
        auto take = [&](const PrTile& T, bool is_v) -> int {
            const int s = L % kPrSlots;
            const uint32_t ph = (L / kPrSlots) & 1;
            ++L;
            if (ok) ok = mbar_wait(&full[s], ph, p.err);
            if (is_v) zero_v(slots + s * kPrSlot, T);
            if (ok) ok = mbar_wait(&pfull[s], ph, p.err);
            return s;
        };
        PrTileIter<LIST> it;
        it.init(fp, worker, ulist);
        PrTile prev;
        prev.valid = false;
        int Tn = 0;  // index of `cur` in the flat tile sequence
        for (;;) {
            const PrTile cur = it.next(fp);
            if (!cur.valid && !prev.valid) break;
            if (cur.valid && !is_s) {
                ++L;  // K(Tn): the S issuer's
            } else if (cur.valid) {
                // S(Tn) = Q K(Tn)^T, once both CTAs' softmax warps have read S(Tn - 1)
                const int sk = take(cur, false);
                if (cur.first && ok) {
                    ok = mbar_wait(q_full, cur.ord & 1, p.err);
                    if (ok) ok = mbar_wait(q_pfull, cur.ord & 1, p.err);
                }
                if (Tn > 0 && ok) ok = mbar_wait(s_free, (Tn - 1) & 1, p.err);
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t kd = smem_desc_sw128(smem_u32(slots + sk * kPrSlot), 0, 1024);
                    const uint64_t qd = smem_desc_sw128(smem_u32(sQ), 0, 1024);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_ss_pair(tS, qd + (uint64_t)((j * kPrQBox + ks * 32) >> 4),
                                         kd + (uint64_t)((j * kPrBox + ks * 32) >> 4), id_s,
                                         (j | ks) ? 1u : 0u);
                    umma_commit_pair(s_full, pair_mask);
                    umma_commit_pair(&empty[sk], pair_mask);
                    if (cur.last) umma_commit_pair(q_free, pair_mask);  // the Q buffer may be reloaded
                }
                __syncwarp();
            }
            if (prev.valid && is_s) {
                ++L;  // V(Tn - 1): the P V issuer's
            } else if (prev.valid) {
                // O (+)= P(Tn - 1) V(Tn - 1)
                const int Tp = Tn - 1;
                const int sv = take(prev, true);
                if (ok) ok = mbar_wait(&p_full[Tp & 1], (Tp >> 1) & 1, p.err);
                // a unit's first P V overwrites O: the previous unit's epilogues have read it
                if (prev.first && prev.ord > 0 && ok)
                    ok = mbar_wait(o_free, (prev.ord - 1) & 1, p.err);
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t vd =
                        smem_desc_sw128(smem_u32(slots + sv * kPrSlot), 2 * kPrBox, 1024);
#pragma unroll
                    for (int kk = 0; kk < kPrKeys / 16; ++kk)
                        umma_ts_pair(tO, tP + 64 * (Tp & 1) + 8 * kk,
                                     vd + (uint64_t)((kk * 2048) >> 4), id_pv,
                                     (prev.first && kk == 0) ? 0u : 1u);
                    umma_commit_pair(&pv_done[Tp & 1], pair_mask);
                    umma_commit_pair(&empty[sv], pair_mask);
                    if (prev.last) umma_commit_pair(o_full, pair_mask);
                }
                __syncwarp();
            }
            if (cur.valid) ++Tn;
            prev = cur;
        }
    } else if (c == 1 && warp == kPrSWarp) {
        // ------------------- odd CTA: forwards its slots' arrivals ---------------------------
        bool ok = true;
        int L = 0;
        const uint32_t pfull0 = map_to_peer(&pfull[0], lead);
        auto fwd = [&](const PrTile& T, bool is_v) {
            const int s = L % kPrSlots;
            const uint32_t ph = (L / kPrSlots) & 1;
            ++L;
            if (ok) ok = mbar_wait(&full[s], ph, p.err);
            if (is_v) zero_v(slots + s * kPrSlot, T);
            if (lane == 0) mbar_arrive_remote(pfull0 + 8u * (uint32_t)s);
            __syncwarp();
        };
        const uint32_t q_pfull0 = map_to_peer(q_pfull, lead);
        PrTileIter<LIST> it;
        it.init(fp, worker, ulist);
        PrTile prev;
        prev.valid = false;
        for (;;) {
            const PrTile cur = it.next(fp);
            if (!cur.valid && !prev.valid) break;
            if (cur.valid && cur.first) {
                if (ok) ok = mbar_wait(q_full, cur.ord & 1, p.err);
                if (lane == 0) mbar_arrive_remote(q_pfull0);
                __syncwarp();
            }
            if (cur.valid) fwd(cur, false);
            if (prev.valid) fwd(prev, true);
            prev = cur;
        }
    } else if (warp < 8) {
        // ------------------------------ softmax warps --------------------------------------
        const int w = warp >> 2;          // softmax group: S columns 64w.., O columns 128w..
        const int r = threadIdx.x & 127;  // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tSw = tmem + kPrSCol + 64 * w + lane_off;
        const uint32_t tOw = tmem + kPrOCol + 128 * w + lane_off;
        const uint32_t tPw = tmem + kPrPCol + 32 * w + lane_off;  // + 64 * buffer
        const uint32_t s_free0 = map_to_peer(s_free, lead), p_full0 = map_to_peer(p_full, lead),
                       o_free0 = map_to_peer(o_free, lead);
        // H = 2: this row's slot in the partner's (rank ^ 2) copy of the exchange buffer
        uint32_t peer_x = 0, peer_x_full = 0, peer_x_free = 0;
        if (H == 2) {
            peer_x = map_to_peer(sX + w * (Lay::X_BYTES / 2) + 16 * r, rank ^ 2u);
            peer_x_full = map_to_peer(&x_full[w], rank ^ 2u);
            peer_x_free = map_to_peer(&x_free[w], rank ^ 2u);
        }
        uint8_t* stage = sStage + w * (kPrStage / 2);  // this group's epilogue staging
        bool ok = true;

        auto rows_here = [&](const PrUnit& U) { return max(0, min(128, U.n_rows - 128 * (int)c)); };
        auto real_here = [&](const PrUnit& U) {
            return max(0, min(128, U.n_rows_real - 128 * (int)c));
        };
        // this group's 128 output columns of row rr of this CTA's rows
        auto out_row = [&](const PrUnit& U, int rr) -> uint4* {
            const int R = U.row0 + 128 * (int)c + rr;
            const int tk = R / p.G, hd = U.kvh * p.G + (R - tk * p.G);
            return reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                            (((size_t)U.b * p.n_tok + tk) * p.n_q + hd) * (size_t)D +
                                            256 * h + 128 * w);
        };
        auto zero_unit = [&](const PrUnit& U) {  // a unit without tiles: zeros
            if (r < rows_here(U)) {
                uint4* o = out_row(U, r);
#pragma unroll 4
                for (int j = 0; j < 16; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (U.bad && w == 0 && r == 0 && U.kvh == 0 && U.rt == 0 && rank == 0)
                report(p.err, U.bad_real ? GEMMA_DEVERR_N_REAL : GEMMA_DEVERR_SEQ_LEN);
        };
        int u = worker - fp.n_pairs;
        // finds the next unit with tiles (writing zeros for units without), or returns false
        auto next_tiled = [&](PrUnit& U) -> bool {
            for (;;) {
                u += fp.n_pairs;
                if (u >= fp.n_units) return false;
                U = pr_unit(fp, LIST ? ulist[u] : u);
                if (U.n_tiles > 0) return true;
                zero_unit(U);
            }
        };

        PrUnit cur;
        if (next_tiled(cur)) {
            int T_base = 0, ord = 0;
            for (;;) {
                const int lo_pos = cur.len - cur.n_real;  // position of the unit's token 0
                int lo = 1, hi = 0;
                if (r < real_here(cur)) {
                    const int pos = lo_pos + (cur.row0 + 128 * (int)c + r) / p.G;
                    lo = p.is_sliding ? max(0, pos - p.window + 1) : 0;
                    hi = pos + 1;
                }
                // the next unit's Q rows towards L2 while this unit runs
                if (!LIST && cur.n_tiles > 2) {
                    const int u2 = u + fp.n_pairs;
                    if (u2 < fp.n_units) {
                        const PrUnit U2 = pr_unit(fp, u2);
                        if (r < real_here(U2)) {
                            const int R = U2.row0 + 128 * (int)c + r;
                            const int tk = R / p.G, hd = U2.kvh * p.G + (R - tk * p.G);
                            const char* qrow = reinterpret_cast<const char*>(
                                reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                (((size_t)U2.b * p.n_tok + tk) * p.n_q + hd) * (size_t)D + 256 * h + 128 * w);
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow));
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + 128));
                        }
                    }
                }
                float m = -INFINITY, l_w = 0.f;  // l_w: this group's columns, relative to m
                for (int t = 0; t < cur.n_tiles; ++t) {
                    const int T = T_base + t;
                    // ---- this group's 64 columns of S(T) ----
                    if (ok) ok = mbar_wait(s_full, T & 1, p.err);
                    tc_fence_after();
                    float s[64];
                    {
                        uint32_t v0[32], v1[32];
                        tmem_ld32(tSw, v0);
                        tmem_ld32(tSw + 32, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            s[e] = __uint_as_float(v0[e]);
                            s[32 + e] = __uint_as_float(v1[e]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(s_free0);  // S(T + 1) may overwrite it

                    if (H == 2) {
                        // S over this pair's half of head_dim: send the partial to the partner
                        // (asynchronous stores that count bytes on its x_full, fp16 saturating)
                        // and add the partner's; each side keeps its own partial in fp32
                        if (r == 0) mbar_arrive_expect_tx(&x_full[w], 128 * 64 * 2);
                        if (T >= 1 && ok) ok = mbar_wait_cluster(&x_free[w], (T - 1) & 1, p.err);
                        // chunk-major layout X[c][r] (16-byte chunks of 8 fp16 scores): a warp's
                        // 32 stores of chunk c are one contiguous 512-byte write
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8)
                            st_async_v4(peer_x + c8 * (128 * 16), pack_f16_sat(s[8 * c8], s[8 * c8 + 1]),
                                        pack_f16_sat(s[8 * c8 + 2], s[8 * c8 + 3]),
                                        pack_f16_sat(s[8 * c8 + 4], s[8 * c8 + 5]),
                                        pack_f16_sat(s[8 * c8 + 6], s[8 * c8 + 7]), peer_x_full);
                        if (ok) ok = mbar_wait_cluster(&x_full[w], T & 1, p.err);
                        const uint4* xr =
                            reinterpret_cast<const uint4*>(sX + w * (Lay::X_BYTES / 2)) + r;
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const uint4 x = xr[c8 * 128];
                            const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f = unpack_f16(wd[i]);
                                const float2 t2 = f32x2_split(add_f32x2(
                                    f32x2(s[8 * c8 + 2 * i], s[8 * c8 + 2 * i + 1]), f32x2(f.x, f.y)));
                                s[8 * c8 + 2 * i] = t2.x;
                                s[8 * c8 + 2 * i + 1] = t2.y;
                            }
                        }
                        // every lane has consumed its loads of X[w]: the partner may overwrite it
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote_relaxed(peer_x_free);
                    }

                    // scores stay raw; scale > 0, so max(raw) * scale_log2 is the max of the
                    // scaled scores. With a soft-cap they are first mapped to c * tanh(scale *
                    // raw / c) in log2 units (before the mask, so masked keys stay -inf), with
                    // the SFU's tanh: one special-function instruction per score instead of an
                    // exponential and a reciprocal, and a relative error (about 2^-11) four times
                    // below the bf16 rounding that P gets before P V.
                    float sl2 = p.scale_log2;
                    if (SOFTCAP) {
                        const unsigned long long ci2 = f32x2(p.cap_inner, p.cap_inner),
                                                 cl2 = f32x2(p.cap_log2, p.cap_log2);
#pragma unroll
                        for (int e = 0; e < 64; e += 2) {
                            const float2 a = f32x2_split(mul_f32x2(f32x2(s[e], s[e + 1]), ci2));
                            const float2 o = f32x2_split(
                                mul_f32x2(f32x2(fast_tanh(a.x), fast_tanh(a.y)), cl2));
                            s[e] = o.x;
                            s[e + 1] = o.y;
                        }
                        sl2 = 1.f;
                    }
                    const int kt0 = cur.k_begin + t * kPrKeys + 64 * w;
                    if (!(kt0 >= lo && kt0 + 64 <= hi)) {
#pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            const int key = kt0 + e;
                            if (key < lo || key >= hi) s[e] = -INFINITY;
                        }
                    }
                    float mx8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3f(s[i], s[8 + i], s[16 + i]);
#pragma unroll
                    for (int e = 24; e < 56; e += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx8[i] = fmax3f(mx8[i], s[e + i], s[e + 8 + i]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[56 + i]);
                    float mx = fmax3f(fmax3f(mx8[0], mx8[1], mx8[2]), fmax3f(mx8[3], mx8[4], mx8[5]),
                                      fmaxf(mx8[6], mx8[7])) *
                               sl2;
                    // ---- the row's maximum over both groups' columns ----
                    float* mxb = mxs + (T & 1) * 256;
                    mxb[w * 128 + r] = mx;
                    named_bar_sync(1, 256);
                    mx = fmaxf(mx, mxb[(w ^ 1) * 128 + r]);
                    // ---- the row's reference: moves only by more than 2^8 ----
                    const float m_prev = m;
                    const float m_new = mx > m_prev + kPrLazyLog2 ? mx : m_prev;
                    if (m_new != m_prev) {  // references only grow; l_w follows
                        l_w = m_prev == -INFINITY ? 0.f : l_w * exp2f(m_prev - m_new);
                        m = m_new;
                    }
                    // ---- O rows whose reference moved: rescale after P V(T-1) ----
                    // (a row whose earlier keys were all masked has O = 0: nothing to rescale)
                    const bool resc = t > 0 && m_new != m_prev && m_prev != -INFINITY;
                    if (__any_sync(0xffffffffu, resc)) {
                        if (ok) ok = mbar_wait(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, p.err);
                        tc_fence_after();
                        const float alpha = resc ? exp2f(m_prev - m_new) : 1.f;
                        const unsigned long long alpha2 = f32x2(alpha, alpha);
#pragma unroll 1
                        for (int j = 0; j < 4; ++j) {
                            uint32_t v[32];
                            tmem_ld32(tOw + j * 32, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 o = f32x2_split(mul_f32x2(
                                    f32x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), alpha2));
                                v[e] = __float_as_uint(o.x);
                                v[e + 1] = __float_as_uint(o.y);
                            }
                            tmem_st32(tOw + j * 32, v);
                        }
                        tmem_st_wait();
                    }
                    // ---- P(T) = 2^(s * scale_log2 - m), this group's 64 keys ----
                    const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
                    const unsigned long long sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
                    unsigned long long sum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
                    uint32_t pw[32];
#pragma unroll
                    for (int k2 = 0; k2 < 32; ++k2) {
                        const float2 x = f32x2_split(fma_f32x2(f32x2(s[2 * k2], s[2 * k2 + 1]), sl2x2, negm2));
                        const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                        sum2[k2 & 1] = add_f32x2(sum2[k2 & 1], f32x2(p0, p1));
                        pw[k2] = pack_bf16(p0, p1);
                    }
                    const float2 sa = f32x2_split(sum2[0]), sb = f32x2_split(sum2[1]);
                    l_w += (sa.x + sa.y) + (sb.x + sb.y);
                    // P buffer T % 2 is free once P V(T-2) has completed
                    if (T >= 2 && ok) ok = mbar_wait(&pv_done[T & 1], ((T - 2) >> 1) & 1, p.err);
                    tc_fence_after();
                    tmem_st32(tPw + 64 * (T & 1), pw);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(p_full0 + 8u * (uint32_t)(T & 1));
                }

                PrUnit nxt;
                const bool more = next_tiled(nxt);

                // ---- epilogue: O / l -> bf16 for this group's 128 columns ----
                const int T_last = T_base + cur.n_tiles - 1;
                if (ok) ok = mbar_wait(o_full, ord & 1, p.err);
                if (ok) ok = mbar_wait(&pv_done[T_last & 1], (T_last >> 1) & 1, p.err);
                tc_fence_after();
                lxs[w * 128 + r] = l_w;
                named_bar_sync(2, 256);
                const float lt = l_w + lxs[(w ^ 1) * 128 + r];
                const float inv = (cur.bad || !(lt > 0.f)) ? 0.f : 1.f / lt;
                const unsigned long long inv2 = f32x2(inv, inv);
                // in slices of 32 columns: each thread converts its row's slice to bf16 into this
                // group's staging rows (64 bytes each, 16-byte chunks placed as the 64-byte TMA
                // swizzle expects), and the group's first thread stores the slice with one TMA
                // box (32 columns x G heads x 128 / G tokens; rows past the sequence's tokens
                // are not written), so no thread waits for global stores
                const bool issuer_t = r == 0;
                const int tk0 = (cur.row0 + 128 * (int)c) / p.G;
#pragma unroll 1
                for (int sl = 0; sl < 4; ++sl) {
                    if (issuer_t) bulk_wait_read_all();  // the last slice's store has read `stage`
                    named_bar_sync(3 + w, 128);
                    uint32_t v[32];
                    tmem_ld32(tOw + sl * 32, v);
                    tmem_ld_wait();
                    if (sl == 3) {  // O has been read: the next unit's first P V may overwrite it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(o_free0);
                    }
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t w4[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 o = f32x2_split(mul_f32x2(
                                f32x2(__uint_as_float(v[8 * cc + 2 * q]), __uint_as_float(v[8 * cc + 2 * q + 1])),
                                inv2));
                            w4[q] = pack_bf16(o.x, o.y);
                        }
                        *reinterpret_cast<uint4*>(stage + r * 64 + ((cc ^ ((r >> 1) & 3)) * 16)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(3 + w, 128);
                    if (issuer_t) {
                        tma_store_4d(&omap, stage, 256 * (int)h + 128 * w + 32 * sl, cur.kvh * p.G,
                                     tk0, cur.b);
                        bulk_commit_group();
                    }
                }
                if (!more) break;
                T_base += cur.n_tiles;
                cur = nxt;
                ++ord;
            }
        }
    }
    if (warp < 8 && (threadIdx.x & 127) == 0) bulk_wait_all();  // the epilogues' TMA stores
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA writes into another's shared memory or barriers any more
    if (warp == kPrSWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
template <int H>
static cudaError_t launch_pair(const RowsParams& p, int batch, cudaStream_t st) {
    using Lay = PrLay<H>;
    constexpr int D = Lay::D;
    CUtensorMap km, vm;
    // [rows][slots][D]: rows = sequences x KV heads (pages x KV heads for a paged pool)
    const uint64_t map_slots = p.page_size ? (uint64_t)p.page_size : (uint64_t)p.cap;
    const uint64_t map_rows = p.page_size ? (uint64_t)p.n_pages * p.n_kv : (uint64_t)batch * p.n_kv;
    const uint64_t dims[3] = {(uint64_t)D, map_slots, map_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, map_slots * D * 2};
    const uint32_t box[3] = {64, 64, 1};
    if (!encode_bf16_sw128(&km, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&vm, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    // Q [B][n_tok][n_q][D]: a box of 64 columns x G heads (of one KV head's group) x 128 / G
    // tokens is one 128-row half tile
    CUtensorMap qm;
    const uint64_t qdims[4] = {(uint64_t)D, (uint64_t)p.n_q, (uint64_t)p.n_tok, (uint64_t)batch};
    const uint64_t qstrides[3] = {(uint64_t)D * 2, (uint64_t)p.n_q * D * 2,
                                  (uint64_t)p.n_tok * p.n_q * D * 2};
    const uint32_t qbox[4] = {64, (uint32_t)p.G, (uint32_t)(128 / p.G), 1};
    if (p.G < 1 || 128 % p.G != 0 || !encode_bf16_sw128(&qm, p.q, 4, qdims, qstrides, qbox))
        return cudaErrorInvalidValue;
    // out, the same layout: boxes of 32 columns (64-byte rows, 64-byte swizzle)
    CUtensorMap om;
    const uint32_t obox[4] = {32, (uint32_t)p.G, (uint32_t)(128 / p.G), 1};
    if (!encode_bf16(&om, p.out, 4, qdims, qstrides, obox, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;

    // per device: the shared-memory attribute, and how many clusters fit at once
    static std::atomic<int> clusters_fit[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int n_clusters = dev >= 0 && dev < 64 ? clusters_fit[dev].load(std::memory_order_relaxed) : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * H;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kPrThreads);
    cfg.dynamicSmemBytes = Lay::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (n_clusters <= 0) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<H, false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_pair_kernel<H, true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_pair_kernel<H, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
        if (e != cudaSuccess) return e;
        int n_sm = 0;
        e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        n_clusters = n_sm / (2 * H);
        cudaLaunchConfig_t occ = cfg;
        occ.gridDim = dim3(2 * H * n_clusters);
        int fit = 0;
        e = cudaOccupancyMaxActiveClusters(&fit, prefill_pair_kernel<H, false, false>, &occ);
        if (e != cudaSuccess) return e;
        if (fit < 1) return cudaErrorInvalidConfiguration;
        if (fit < n_clusters) n_clusters = fit;
        if (dev >= 0 && dev < 64) clusters_fit[dev].store(n_clusters, std::memory_order_relaxed);
    }
    PrParams fp;
    fp.p = p;
    fp.batch = batch;
    fp.n_rt = (p.n_tok * p.G + kPrRows - 1) / kPrRows;
    fp.n_units = fp.n_rt * batch * p.n_kv;
    fp.n_pairs = fp.n_units < n_clusters ? fp.n_units : n_clusters;
    cfg.gridDim = dim3(2 * H * fp.n_pairs);
    if (p.softcap > 0.f)
        return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<H, true, false>, km, vm, qm, om, fp);
    // a padded bucket deals out its units with key tiles first (the work list) where the units
    // of a row tile divide the workers evenly, so that the plain order would give a worker the
    // same sequences in every wave (elsewhere building the list costs more than it saves)
    if (p.n_real && fp.n_units <= kPrListMax && fp.n_pairs % (batch * p.n_kv) == 0)
        return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<H, false, true>, km, vm, qm, om, fp);
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<H, false, false>, km, vm, qm, om, fp);
}

cudaError_t launch_prefill_pair(const RowsParams& p, int head_dim, int batch, cudaStream_t st) {
    if (head_dim == 256) return launch_pair<1>(p, batch, st);
    if (head_dim == 512) return launch_pair<2>(p, batch, st);
    return cudaErrorInvalidValue;
}

}  // namespace gemma
