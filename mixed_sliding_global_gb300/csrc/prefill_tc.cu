// prefill_tc.cu -- prefill-bucket attention on 5th-generation tensor cores (tcgen05 + TMEM).
//
// Computes, for tiles of 128 query rows (rows = (token, head of the GQA group) pairs, token
// major, so every row of a tile reads the same KV head), softmax(scale * Q K^T) V over the
// causal (and, on sliding layers, windowed) key range of each row, with the K/V cache of the
// owner layer ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", sections 2.1-2.3; the
// pages' "eager" matmul-softmax-matmul definition, section 4.3).
//
// This kernel runs head_dim 64 and 128; head_dim 256 and 512 run on CTA pairs issuing 2-SM
// MMAs (prefill_pair.cu).
//
// Persistent grid: one CTA per SM walks work units = (row
// tile, sequence, KV head), latest row tiles (longest key ranges) first, and within a unit
// 64-key tiles. The tiles of all its units form one flat sequence T = 0, 1, 2, ... per CTA.
// Each CTA has 10 warps:
//   warps 0-3 / 4-7   softmax warpgroups WG0 / WG1: WG (T % 2) handles tile T; thread r owns
//              row r (TMEM lane r). It reads S(T) from TMEM, masks by index, hands the row's
//              running softmax reference to the other group (the reference moves only when a
//              tile maximum exceeds it by more than 2^8: lazy rescaling keeps the result exact,
//              the final division uses the same reference), writes bf16 P to shared memory,
//              and rescales the O row in TMEM when the reference moved. The group that handles
//              a unit's first tile loads the unit's Q rows into TMEM; both groups write O / l.
//   warp 8     TMA producer: 64-key K and V tiles (128-byte swizzle, one box per 64 columns of
//              head_dim) into a FIFO ring of shared-memory slots, in the MMA warp's order.
//   warp 9     MMA issuer: step i issues S(i) = Q K(i)^T (A = Q from TMEM, B = K, K-major) into
//              TMEM buffer i % 2 and O += P(i-2) V(i-2) (A = P, K-major, B = V, MN-major), so
//              the softmax of a tile overlaps two later tiles' tensor work.
// Synchronisation is per step (rings of 8 mbarriers): step_ready[i] completes when the step's
// K/V tiles have landed and P(i-2) is written; the MMA warp commits step_done[i] after the
// step's MMAs. A tcgen05.mma is accepted only when the one before it is nearly done, so each
// wait or commit between MMA groups idles the tensor core: the MMA warp does one of each per
// step. Within a step, each 64-column block of S is preceded by one of the (longer) P V MMAs:
// the issuing thread shares its SM sub-partition with softmax warps, and a long MMA gives it
// time to be scheduled before the pipe runs dry.
// TMEM (512 columns): Q (D/2 columns of packed bf16) at 0, S buffers at 128 and 192 (64 fp32
// columns each), O (D columns) at 256.
//
// The key range of a unit is clamped to [first row's window start, last row's position] before
// any load; rows of a K/V tile outside the range are zeroed in shared memory before they enter
// P V (they may hold anything, NaN included).
#include <cuda_fp16.h>

#include <atomic>

#include "attn_internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace gemma {

constexpr int kFaWarps = 10;
constexpr int kFaThreads = kFaWarps * 32;
constexpr int kFaProducerWarp = 8;
constexpr int kFaMmaWarp = 9;
constexpr int kFaMaxSlots = 8;
constexpr int kFaSteps = 8;                   // entries of the per-step barrier rings
constexpr int kFaKeys = 64;                   // keys per tile (N of S = Q K^T)
constexpr int kFaSmemLimit = 232448;          // max dynamic shared memory per block
constexpr float kLazyRescaleLog2 = 8.f;

template <int D>
struct FaLayout {
    static constexpr int DH = D;                         // head_dim
    static constexpr int CHUNKS = DH / 64;               // 64-column boxes per K/V tile
    static constexpr int BOX = kFaKeys * 128;            // one box: 64 keys x 64 columns
    static constexpr int SLOT = CHUNKS * BOX;            // one K or V tile
    static constexpr int P_TILE = 128 * kFaKeys * 2;     // 128 rows x 64 keys bf16
    static constexpr int Q_COL = 0;                      // TMEM columns
    static constexpr int S_COL = 128;                    // + 64 * buffer
    static constexpr int O_COL = 256;
    // fixed shared memory besides the ring: P (2), reference row maxima, barriers
    static constexpr int FIXED = 2 * P_TILE + 512 + 512;
    static_assert(DH / 2 <= 128 && O_COL + DH <= 512, "TMEM budget");
    static_assert(2 * 128 * 8 <= P_TILE, "the epilogue's (m, l) exchange fits in one P buffer");
};

struct FaParams {
    RowsParams p;
    int n_slots;
    int batch;
    int n_rt;      // row tiles per (sequence, KV head)
    int n_units;   // n_rt * batch * n_kv
    int n_workers; // CTAs walking the units
};

// Non-blocking check of a phase's completion (cheaper than try_wait when it has completed).
GEMMA_DEVINL bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Adds `bytes` to the transaction count the current phase of `bar` waits for.
GEMMA_DEVINL void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// `count` arrivals on `bar` at once.
GEMMA_DEVINL void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// ---------------------------------------------------------------------------------------------
// work units
// ---------------------------------------------------------------------------------------------
struct FaUnit {
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
GEMMA_DEVINL FaUnit fa_unit(const FaParams& fp, int u) {
    const RowsParams& p = fp.p;
    FaUnit U;
    const int per_rt = fp.batch * p.n_kv;
    const int q = u / per_rt, rem = u - q * per_rt;
    U.rt = fp.n_rt - 1 - q;
    U.b = rem / p.n_kv;
    U.kvh = rem - U.b * p.n_kv;
    const int rows_total = p.n_tok * p.G;
    U.row0 = U.rt * 128;
    U.n_rows = min(128, rows_total - U.row0);
    U.len = __ldg(p.seq_lens + U.b);
    // real tokens of this sequence (a padded bucket's first n_real rows; all rows otherwise);
    // the i-th real token sits at len - n_real + i, the pad rows' outputs are zero
    U.n_real = p.n_real ? __ldg(p.n_real + U.b) : p.n_tok;
    U.bad_real = U.n_real < 0 || U.n_real > p.n_tok;
    U.bad = U.bad_real || U.len < U.n_real || (!p.ring && U.len > p.cap) || U.len > p.max_seq_len;
    U.n_rows_real = U.bad ? 0 : max(0, min(128, U.n_real * p.G - U.row0));
    // key range: from the first row's window start to the last real row's position (a ring
    // cache's or paged pool's tiles start at multiples of the tile, so that none wraps around
    // the ring or crosses a page; the rows' masks drop the keys before the window)
    const int tok_first = U.row0 / p.G;
    const int tok_last = (U.row0 + max(U.n_rows_real, 1) - 1) / p.G;
    const int pos_first = U.len - U.n_real + tok_first;
    const int lo_first = p.is_sliding ? max(0, pos_first - p.window + 1) : 0;
    U.k_begin = (p.ring || p.page_size) ? (lo_first & ~(kFaKeys - 1)) : lo_first;
    U.k_end = U.len - U.n_real + tok_last + 1;
    U.n_tiles = U.n_rows_real == 0 ? 0 : (U.k_end - U.k_begin + kFaKeys - 1) / kFaKeys;
    U.n_head = lo_first - U.k_begin;
    return U;
}

// One tile of the flat per-CTA sequence, as the producer and the MMA warp see it.
struct FaTile {
    bool valid, first, last;
    int ord;       // ordinal of its unit among this CTA's units that have tiles
    int n_valid;   // keys of the tile inside the unit's range (the rest are zeroed)
    int n_head;    // leading keys zeroed (first tile of an aligned-start unit)
    int key0;      // first key
    int b, kvh;
    int slot;      // ring slot holding it (k_eq_v: K and V)
};

// Walks this CTA's units and their tiles in order.
struct FaTileIter {
    int u, stride, t, ord;
    FaUnit U;
    GEMMA_DEVINL void init(const FaParams& fp, int worker) {
        u = worker;
        stride = fp.n_workers;
        t = 0;
        ord = -1;
        U.n_tiles = 0;
        U.b = U.kvh = 0;
        U.k_begin = 0;
        u -= stride;  // next() advances to the first unit
    }
    GEMMA_DEVINL FaTile next(const FaParams& fp) {
        FaTile T;
        T.valid = false;
        while (t >= U.n_tiles) {
            u += stride;
            if (u >= fp.n_units) return T;
            U = fa_unit(fp, u);
            t = 0;
            if (U.n_tiles > 0) ++ord;
        }
        T.valid = true;
        T.first = t == 0;
        T.last = t == U.n_tiles - 1;
        T.ord = ord;
        T.key0 = U.k_begin + t * kFaKeys;
        T.n_valid = min(kFaKeys, U.k_end - T.key0);
        T.n_head = t == 0 ? U.n_head : 0;
        T.b = U.b;
        T.kvh = U.kvh;
        T.slot = 0;
        ++t;
        return T;
    }
};

// SOFTCAP: the soft-capped variant (a separate instantiation, so that the plain kernel carries
// no code for it)
template <int D, bool SOFTCAP>
__global__ void __launch_bounds__(kFaThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const FaParams fp) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    using Lay = FaLayout<D>;
    constexpr int DH = Lay::DH;
    const RowsParams& p = fp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NS = fp.n_slots;
    uint8_t* slots = smem;
    uint8_t* sP = smem + NS * Lay::SLOT;                     // P buffers [2][128 x 64] bf16
    float* mref = reinterpret_cast<float*>(sP + 2 * Lay::P_TILE);  // [128] softmax references
    uint64_t* bars = reinterpret_cast<uint64_t*>(mref + 128);
    // Step i of the MMA warp issues S(i) and P V(i-2). step_ready[i % R] completes when the
    // step's K/V tiles have landed (producer arrival + transaction bytes) and P(i-2) is in
    // shared memory (4 warp arrivals of the softmax group; the producer arrives for them when
    // the step has no P V). step_done[i % R] is committed after the step's MMAs: S(i) is in
    // TMEM, P V(i-2) has completed (so P buffer i % 2 and the step's ring slots are free).
    uint64_t* step_ready = bars;
    uint64_t* step_done = bars + kFaSteps;
    uint64_t* o_full = bars + 2 * kFaSteps;     // a unit's last P V has completed
    uint64_t* o_free = o_full + 1;              // the epilogue has read O
    uint64_t* q_ready = o_full + 2;             // a unit's Q is in TMEM
    uint64_t* m_ready = o_full + 3;             // the reference after tile T is in mref
    uint32_t* tslot = reinterpret_cast<uint32_t*>(o_full + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int worker = blockIdx.x;

    if (warp == kFaMmaWarp) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kFaSteps; ++i) {
            mbar_init(&step_ready[i], 5);
            mbar_init(&step_done[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(o_free, 8);
        mbar_init(q_ready, 4);
        mbar_init(m_ready, 128);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tQ = tmem + Lay::Q_COL, tO = tmem + Lay::O_COL;

    if (warp == kFaProducerWarp) {
        // ------------------------------- TMA producer --------------------------------------
        // Step i loads K(i) and then (K != V) V(i-2) into the next slots of a FIFO ring. A slot
        // is reused once the step that last read it has completed (K: its S step; V, or K used
        // as V: its P V step).
        if (lane == 0) {
            bool ok = true;
            int ps = 0;
            int rel[kFaMaxSlots];  // step whose completion frees each slot (-1: free)
            for (int k = 0; k < kFaMaxSlots; ++k) rel[k] = -1;
            auto claim = [&](int release_step) -> int {
                const int s0 = ps;
                const int r0 = rel[s0];
                if (r0 >= 0 && ok) ok = mbar_wait(&step_done[r0 % kFaSteps], (r0 / kFaSteps) & 1, p.err);
                rel[s0] = release_step;
                if (++ps == NS) ps = 0;
                return s0;
            };
            auto load = [&](const CUtensorMap* map, const FaTile& T, int slot, uint64_t* bar) {
                uint8_t* dst = slots + slot * Lay::SLOT;
                // cache row and slot of the tile's first key (a bad page index reads zeros)
                int row3 = 0, slot0 = 0;
                if (!kv_place(p, T.b, T.kvh, T.key0, row3, slot0)) {
                    report(p.err, GEMMA_DEVERR_PAGE);
                    row3 = p.n_pages * p.n_kv;
                }
#pragma unroll
                for (int c = 0; c < Lay::CHUNKS; ++c)
                    tma_load_3d(dst + c * Lay::BOX, map, c * 64, slot0, row3, bar);
            };
            FaTileIter it;
            it.init(fp, worker);
            FaTile h1, h2;
            h1.valid = h2.valid = false;
            for (int i = 0;; ++i) {
                const FaTile cur = it.next(fp);
                if (!cur.valid && !h1.valid && !h2.valid) break;
                const bool pv = h2.valid;
                if (cur.valid || pv) {
                    const int sk = cur.valid ? claim(p.k_eq_v ? i + 2 : i) : -1;
                    const int sv = (!p.k_eq_v && pv) ? claim(i) : -1;
                    // the barrier entry's previous step (i - R) has completed
                    if (i >= kFaSteps && ok)
                        ok = mbar_wait(&step_done[i % kFaSteps], ((i - kFaSteps) / kFaSteps) & 1, p.err);
                    uint64_t* bar = &step_ready[i % kFaSteps];
                    const uint32_t bytes = (sk >= 0 ? Lay::SLOT : 0) + (sv >= 0 ? Lay::SLOT : 0);
                    if (bytes) mbar_expect_tx(bar, bytes);
                    mbar_arrive_cnt(bar, pv ? 1u : 5u);
                    if (ok && sk >= 0) load(&kmap, cur, sk, bar);
                    if (ok && sv >= 0) load(&vmap, h2, sv, bar);
                }
                h2 = h1;
                h1 = cur;
            }
        }
    } else if (warp == kFaMmaWarp) {
        // -------------------------------- MMA issuer ---------------------------------------
        // One wait and one commit per step: an MMA is issued only once the one before it is
        // nearly done, so every wait or commit between MMA groups idles the tensor core.
        const uint32_t id_qk = idesc_bf16(128, kFaKeys, 0, 0);
        const uint32_t id_pv = idesc_bf16(128, DH, 0, 1);
        bool ok = true;
        int ps = 0;
        // rows of a tile that must not reach P V (outside the unit's key range): zeroed
        auto zero_edges = [&](int slot, const FaTile& T) {
            const int n_tail = kFaKeys - T.n_valid;
            if (n_tail <= 0 && T.n_head <= 0) return;
            uint8_t* tile = slots + slot * Lay::SLOT;
            if (n_tail > 0) {
                for (int idx = lane; idx < Lay::CHUNKS * n_tail * 8; idx += 32) {
                    const int c = idx / (n_tail * 8), rem = idx - c * n_tail * 8;
                    *reinterpret_cast<uint4*>(tile + c * Lay::BOX + (T.n_valid + rem / 8) * 128 +
                                              (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (T.n_head > 0) {
                for (int idx = lane; idx < Lay::CHUNKS * T.n_head * 8; idx += 32) {
                    const int c = idx / (T.n_head * 8), rem = idx - c * T.n_head * 8;
                    *reinterpret_cast<uint4*>(tile + c * Lay::BOX + (rem / 8) * 128 +
                                              (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        auto issue_s = [&](const FaTile& T, int i) {  // lane 0: S(i) = Q K(i)^T
            const uint64_t kd = smem_desc_sw128(smem_u32(slots + T.slot * Lay::SLOT), 0, 1024);
            const uint32_t tS = tmem + Lay::S_COL + 64 * (i & 1);
#pragma unroll
            for (int c = 0; c < Lay::CHUNKS; ++c)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_ts(tS, tQ + c * 32 + ks * 8,
                            kd + (uint64_t)((c * Lay::BOX + ks * 32) >> 4), id_qk,
                            (c | ks) ? 1u : 0u);
        };
        auto issue_pv = [&](const FaTile& T, int i) {  // lane 0: O (+)= P(i-2) V(i-2)
            const uint64_t vd = smem_desc_sw128(smem_u32(slots + T.slot * Lay::SLOT), Lay::BOX, 1024);
            const uint64_t pd = smem_desc_sw128(smem_u32(sP + (i & 1) * Lay::P_TILE), 0, 1024);
#pragma unroll
            for (int kk = 0; kk < kFaKeys / 16; ++kk)
                umma_ss(tO, pd + (uint64_t)((kk * 32) >> 4), vd + (uint64_t)((kk * 2048) >> 4),
                        id_pv, (!T.first || kk > 0) ? 1u : 0u);
            if (T.last) umma_commit(o_full);
        };
        FaTileIter it;
        it.init(fp, worker);
        FaTile h1, h2;
        h1.valid = h2.valid = false;
        for (int i = 0;; ++i) {
            FaTile cur = it.next(fp);
            if (!cur.valid && !h1.valid && !h2.valid) break;
            if (cur.valid || h2.valid) {
                // slots in the producer's order: K(i), then (K != V) V(i-2)
                if (cur.valid) {
                    cur.slot = ps;
                    if (++ps == NS) ps = 0;
                }
                if (!p.k_eq_v && h2.valid) {
                    h2.slot = ps;
                    if (++ps == NS) ps = 0;
                }
                if (ok && !mbar_test_wait(&step_ready[i % kFaSteps], (i / kFaSteps) & 1))
                    ok = mbar_wait(&step_ready[i % kFaSteps], (i / kFaSteps) & 1, p.err);
                if (p.k_eq_v) {
                    if (cur.valid) zero_edges(cur.slot, cur);  // the slot also serves as V
                } else if (h2.valid) {
                    zero_edges(h2.slot, h2);
                }
                // the previous unit's epilogue has read O before this unit's first P V
                if (h2.valid && h2.first && h2.ord > 0 && ok)
                    ok = mbar_wait(o_free, (h2.ord - 1) & 1, p.err);
                tc_fence_after();
                if (cur.valid && cur.first) {
                    // a unit's first S: the P V goes first (the previous unit's epilogue waits
                    // for it, and the group that loads this unit's Q may have to finish that
                    // epilogue first)
                    if (h2.valid && lane == 0) issue_pv(h2, i);
                    __syncwarp();
                    if (ok) ok = mbar_wait(q_ready, cur.ord & 1, p.err);
                    tc_fence_after();
                    if (lane == 0) issue_s(cur, i);
                } else if (lane == 0) {
                    if (cur.valid && h2.valid) {
                        // S(i) and P V(i-2) interleaved: a long P V MMA before every 64 columns of S
                        const uint64_t kd = smem_desc_sw128(smem_u32(slots + cur.slot * Lay::SLOT), 0, 1024);
                        const uint32_t tS = tmem + Lay::S_COL + 64 * (i & 1);
                        const uint64_t vd = smem_desc_sw128(smem_u32(slots + h2.slot * Lay::SLOT), Lay::BOX, 1024);
                        const uint64_t pd = smem_desc_sw128(smem_u32(sP + (i & 1) * Lay::P_TILE), 0, 1024);
#pragma unroll
                        for (int c = 0; c < Lay::CHUNKS; ++c) {
                            if (c < kFaKeys / 16)
                                umma_ss(tO, pd + (uint64_t)((c * 32) >> 4), vd + (uint64_t)((c * 2048) >> 4),
                                        id_pv, (!h2.first || c > 0) ? 1u : 0u);
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_ts(tS, tQ + c * 32 + ks * 8,
                                        kd + (uint64_t)((c * Lay::BOX + ks * 32) >> 4), id_qk,
                                        (c | ks) ? 1u : 0u);
                        }
#pragma unroll
                        for (int kk = Lay::CHUNKS; kk < kFaKeys / 16; ++kk)
                            umma_ss(tO, pd + (uint64_t)((kk * 32) >> 4), vd + (uint64_t)((kk * 2048) >> 4),
                                    id_pv, (!h2.first || kk > 0) ? 1u : 0u);
                        if (h2.last) umma_commit(o_full);
                    } else {
                        if (cur.valid) issue_s(cur, i);
                        if (h2.valid) issue_pv(h2, i);
                    }
                }
                if (lane == 0) umma_commit(&step_done[i % kFaSteps]);
                __syncwarp();
            }
            h2 = h1;
            h1 = cur;
        }
    } else {
        // ------------------------------ softmax warps --------------------------------------
        const int w = warp >> 2;               // softmax group: tiles T with T % 2 == w
        const int r = threadIdx.x & 127;       // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        uint8_t* sPw = sP + w * Lay::P_TILE;
        bool ok = true;

        // this group's half of the output columns of a unit's rows
        auto out_row = [&](const FaUnit& U, int rr) -> uint4* {
            const int R = U.row0 + rr;
            const int tk = R / p.G, hd = U.kvh * p.G + (R - tk * p.G);
            return reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                            (((size_t)U.b * p.n_tok + tk) * p.n_q + hd) * (size_t)D +
                                            w * (DH / 2));
        };
        auto zero_unit = [&](const FaUnit& U) {  // a unit without tiles: zeros
            if (r < U.n_rows) {
                uint4* o = out_row(U, r);
#pragma unroll 4
                for (int j = 0; j < DH / 16; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (U.bad && w == 0 && r == 0 && U.kvh == 0 && U.rt == 0)
                report(p.err, U.bad_real ? GEMMA_DEVERR_N_REAL : GEMMA_DEVERR_SEQ_LEN);
        };
        // the unit's Q rows (this CTA's head_dim part) into TMEM, once S(T_prev) (the last S
        // MMA that reads the previous unit's Q) has completed
        auto load_q = [&](const FaUnit& U, int T_prev) {
            // in halves of at most 64 columns (16 x 16-byte loads in flight per thread); the
            // first half's loads are issued before waiting for the previous unit's last S
            constexpr int NQ = DH / 8;               // 16-byte chunks of a row's part (DH bf16)
            constexpr int HALF = NQ > 16 ? 16 : NQ;  // chunks per round
            const bool row_ok = r < U.n_rows_real;
            const int R = U.row0 + (row_ok ? r : 0);
            const int tk = R / p.G, hd = U.kvh * p.G + (R - tk * p.G);
            const uint4* qrow = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) +
                (((size_t)U.b * p.n_tok + tk) * p.n_q + hd) * (size_t)D);
#pragma unroll
            for (int hf = 0; hf < NQ / HALF; ++hf) {
                uint4 qv[HALF];
#pragma unroll
                for (int j = 0; j < HALF; ++j)
                    qv[j] = row_ok ? __ldg(qrow + hf * HALF + j) : make_uint4(0u, 0u, 0u, 0u);
                if (hf == 0) {
                    if (T_prev >= 0 && ok) ok = mbar_wait(&step_done[T_prev % kFaSteps], (T_prev / kFaSteps) & 1, p.err);
                    tc_fence_after();
                }
#pragma unroll
                for (int j = 0; j < HALF / 8; ++j) {
                    uint32_t v[32];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        v[4 * e + 0] = qv[8 * j + e].x;
                        v[4 * e + 1] = qv[8 * j + e].y;
                        v[4 * e + 2] = qv[8 * j + e].z;
                        v[4 * e + 3] = qv[8 * j + e].w;
                    }
                    tmem_st32(tQ + lane_off + (hf * HALF / 8 + j) * 32, v);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        };
        // finds the next unit with tiles (writing zeros for units without), or returns false
        int u = worker - fp.n_workers;
        auto next_tiled = [&](FaUnit& U) -> bool {
            for (;;) {
                u += fp.n_workers;
                if (u >= fp.n_units) return false;
                U = fa_unit(fp, u);
                if (U.n_tiles > 0) return true;
                zero_unit(U);
            }
        };

        FaUnit cur;
        if (next_tiled(cur)) {
            int T_base = 0, ord = 0;
            float m_w = -INFINITY, l_w = 0.f;  // this group's share of l, relative to m_w
            if (w == 0) load_q(cur, -1);
            for (;;) {
                const int lo_pos = cur.len - cur.n_real;  // position of the unit's token 0
                int lo = 1, hi = 0;
                if (r < cur.n_rows_real) {
                    const int pos = lo_pos + (cur.row0 + r) / p.G;
                    lo = p.is_sliding ? max(0, pos - p.window + 1) : 0;
                    hi = pos + 1;
                }
                // the next unit's Q rows towards L2 while this unit runs (its loader group)
                if (cur.n_tiles > 2) {
                    const int u2 = u + fp.n_workers;
                    if (u2 < fp.n_units && (((T_base + cur.n_tiles) & 1) == w)) {
                        const FaUnit U2 = fa_unit(fp, u2);
                        if (r < U2.n_rows_real) {
                            const int R = U2.row0 + r;
                            const int tk = R / p.G, hd = U2.kvh * p.G + (R - tk * p.G);
                            const char* qrow = reinterpret_cast<const char*>(
                                reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                (((size_t)U2.b * p.n_tok + tk) * p.n_q + hd) * (size_t)D);
#pragma unroll
                            for (int j = 0; j < (DH * 2) / 128; ++j)
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + j * 128));
                        }
                    }
                }
                const int t0 = ((T_base & 1) == w) ? 0 : 1;
                for (int t = t0; t < cur.n_tiles; t += 2) {
                    const int T = T_base + t;
                    const int buf = T & 1;  // == w
                    // ---- S(T) from TMEM (its step has also completed P V(T-2), so P buffer
                    // T % 2 is free) ----
                    if (ok) ok = mbar_wait(&step_done[T % kFaSteps], (T / kFaSteps) & 1, p.err);
                    tc_fence_after();
                    float s[kFaKeys];
                    {
                        uint32_t v0[32], v1[32];
                        const uint32_t tS = tmem + Lay::S_COL + 64 * buf + lane_off;
                        tmem_ld32(tS, v0);
                        tmem_ld32(tS + 32, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            s[e] = __uint_as_float(v0[e]);
                            s[32 + e] = __uint_as_float(v1[e]);
                        }
                    }

                    // scores stay raw; scale > 0, so max(raw) * scale_log2 is the max of the
                    // scaled scores. With a soft-cap they are first mapped to c * tanh(scale *
                    // raw / c) in log2 units (before the mask, so masked keys stay -inf), with
                    // the SFU's tanh (relative error about 2^-11, four times below the bf16
                    // rounding that P gets before P V).
                    float sl2 = p.scale_log2;
                    if (SOFTCAP) {
                        const unsigned long long ci2 = f32x2(p.cap_inner, p.cap_inner),
                                                 cl2 = f32x2(p.cap_log2, p.cap_log2);
#pragma unroll
                        for (int e = 0; e < kFaKeys; e += 2) {
                            const float2 a = f32x2_split(mul_f32x2(f32x2(s[e], s[e + 1]), ci2));
                            const float2 o = f32x2_split(
                                mul_f32x2(f32x2(fast_tanh(a.x), fast_tanh(a.y)), cl2));
                            s[e] = o.x;
                            s[e + 1] = o.y;
                        }
                        sl2 = 1.f;
                    }
                    const int kt0 = cur.k_begin + t * kFaKeys;
                    if (!(kt0 >= lo && kt0 + kFaKeys <= hi)) {
#pragma unroll
                        for (int e = 0; e < kFaKeys; ++e) {
                            const int key = kt0 + e;
                            if (key < lo || key >= hi) s[e] = -INFINITY;
                        }
                    }
                    // (three-input maxima and, below, packed two-lane fp32 arithmetic: fewer
                    // instructions from these warps, which share issue slots with the MMA
                    // issuer)
                    static_assert(kFaKeys == 64, "the reduction below covers 64 keys");
                    float mx8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3f(s[i], s[8 + i], s[16 + i]);
#pragma unroll
                    for (int e = 24; e < 56; e += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx8[i] = fmax3f(mx8[i], s[e + i], s[e + 8 + i]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[56 + i]);
                    const float mx = fmax3f(fmax3f(mx8[0], mx8[1], mx8[2]),
                                            fmax3f(mx8[3], mx8[4], mx8[5]),
                                            fmaxf(mx8[6], mx8[7])) *
                                     sl2;

                    // ---- the row's reference after tile T-1, then after tile T ----
                    if (T > 0 && ok) ok = mbar_wait(m_ready, (T - 1) & 1, p.err);
                    const float m_prev = t > 0 ? mref[r] : -INFINITY;
                    const float m_new = mx > m_prev + kLazyRescaleLog2 ? mx : m_prev;
                    mref[r] = m_new;
                    mbar_arrive(m_ready);
                    if (m_new != m_w) {  // references only grow; l_w follows
                        l_w = m_w == -INFINITY ? 0.f : l_w * exp2f(m_w - m_new);
                        m_w = m_new;
                    }
                    // ---- O rows whose reference moved: rescale after P V(T-1) ----
                    // (a row whose earlier keys were all masked has O = 0: nothing to rescale)
                    const bool resc = t > 0 && m_new != m_prev && m_prev != -INFINITY;
                    if (__any_sync(0xffffffffu, resc)) {
                        // P V(T-1) completes in step T + 1
                        if (ok) ok = mbar_wait(&step_done[(T + 1) % kFaSteps], ((T + 1) / kFaSteps) & 1, p.err);
                        tc_fence_after();
                        const float alpha = resc ? exp2f(m_prev - m_new) : 1.f;
#pragma unroll 1
                        for (int j = 0; j < DH / 32; ++j) {
                            uint32_t v[32];
                            tmem_ld32(tO + lane_off + j * 32, v);
                            tmem_ld_wait();
                            const unsigned long long alpha2 = f32x2(alpha, alpha);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 o = f32x2_split(mul_f32x2(
                                    f32x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), alpha2));
                                v[e] = __float_as_uint(o.x);
                                v[e + 1] = __float_as_uint(o.y);
                            }
                            tmem_st32(tO + lane_off + j * 32, v);
                        }
                        tmem_st_wait();
                    }
                    // ---- P(T) = 2^(s * scale_log2 - m) into shared memory buffer T % 2 ----
                    const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
                    const unsigned long long sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
                    unsigned long long sum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
                    uint32_t pw[kFaKeys / 2];
#pragma unroll
                    for (int k2 = 0; k2 < kFaKeys / 2; ++k2) {
                        const float2 x = f32x2_split(fma_f32x2(f32x2(s[2 * k2], s[2 * k2 + 1]), sl2x2, negm2));
                        const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                        sum2[k2 & 1] = add_f32x2(sum2[k2 & 1], f32x2(p0, p1));
                        pw[k2] = pack_bf16(p0, p1);
                    }
                    const float2 sa = f32x2_split(sum2[0]), sb = f32x2_split(sum2[1]);
                    const float sum4[4] = {sa.x, sa.y, sb.x, sb.y};
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(sPw + r * 128 + ((c ^ (r & 7)) * 16)) =
                            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                    l_w += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&step_ready[(T + 2) % kFaSteps]);  // P V(T) in step T + 2
                }

                // ---- next unit: its first tile's group loads its Q before this epilogue ----
                FaUnit nxt;
                const bool more = next_tiled(nxt);
                const int T_next = T_base + cur.n_tiles;
                if (more && (T_next & 1) == w) load_q(nxt, T_next - 1);

                // ---- epilogue: O / l -> bf16 for this group's half of the columns ----
                if (ok) ok = mbar_wait(o_full, ord & 1, p.err);
                tc_fence_after();
                {
                    // (m, l) of both groups through the first P buffer, free once the unit's
                    // last P V has completed (and until the next unit's first P is written)
                    float2* ml = reinterpret_cast<float2*>(sP);
                    ml[w * 128 + r] = make_float2(m_w, l_w);
                    named_bar_sync(1, 256);
                    const float2 o2 = ml[(w ^ 1) * 128 + r];
                    named_bar_sync(1, 256);
                    const float mf = fmaxf(m_w, o2.x);
                    float lt = 0.f;
                    if (m_w != -INFINITY) lt += l_w * exp2f(m_w - mf);
                    if (o2.x != -INFINITY) lt += o2.y * exp2f(o2.x - mf);
                    const float inv = (cur.bad || lt == 0.f) ? 0.f : 1.f / lt;
                    // O / l in slices of up to 64 columns: each thread converts its row's slice
                    // to bf16 in this group's P buffer (free until its next P: the unit's last P
                    // V has completed), then each warp writes its 32 rows' slices with whole
                    // 128-byte lines per row (rows are 2 * D bytes apart in `out`)
                    constexpr int SW = DH / 2 < 64 ? DH / 2 : 64;  // columns per slice
                    constexpr int CPR = SW / 8;                    // 16-byte chunks per row
                    uint8_t* stage = sPw;
                    const int wrow0 = (warp & 3) * 32;             // this warp's rows
#pragma unroll 1
                    for (int sl = 0; sl < (DH / 2) / SW; ++sl) {
#pragma unroll
                        for (int j = 0; j < SW / 32; ++j) {
                            uint32_t v[32];
                            tmem_ld32(tO + lane_off + w * (DH / 2) + sl * SW + j * 32, v);
                            tmem_ld_wait();
                            const unsigned long long inv2 = f32x2(inv, inv);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = j * 4 + e;
                                uint32_t w4[4];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float2 o = f32x2_split(mul_f32x2(
                                        f32x2(__uint_as_float(v[8 * e + 2 * q]), __uint_as_float(v[8 * e + 2 * q + 1])),
                                        inv2));
                                    w4[q] = pack_bf16(o.x, o.y);
                                }
                                *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) * 16)) =
                                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                        __syncwarp();
#pragma unroll
                        for (int it2 = 0; it2 < CPR; ++it2) {
                            const int idx = it2 * 32 + lane;
                            const int rr = wrow0 + idx / CPR, c = idx % CPR;
                            const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((c ^ (rr & 7)) * 16));
                            if (rr < cur.n_rows) out_row(cur, rr)[sl * CPR + c] = val;
                        }
                        __syncwarp();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
                m_w = -INFINITY;
                l_w = 0.f;
                if (!more) break;
                cur = nxt;
                T_base = T_next;
                ++ord;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kFaMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
template <int D>
static cudaError_t launch_d(const RowsParams& p, int batch, cudaStream_t st) {
    using Lay = FaLayout<D>;
    CUtensorMap km, vm;
    // [rows][slots][D]: rows = sequences x KV heads (pages x KV heads for a paged pool)
    const uint64_t map_slots = p.page_size ? (uint64_t)p.page_size : (uint64_t)p.cap;
    const uint64_t map_rows = p.page_size ? (uint64_t)p.n_pages * p.n_kv : (uint64_t)batch * p.n_kv;
    const uint64_t dims[3] = {(uint64_t)D, map_slots, map_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, map_slots * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kFaKeys, 1};
    if (!encode_bf16_sw128(&km, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&vm, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    const int fixed = Lay::FIXED + 1024;  // + alignment slack of the dynamic buffer
    int ns = (kFaSmemLimit - fixed) / Lay::SLOT;
    if (ns > kFaMaxSlots) ns = kFaMaxSlots;
    if (ns < 3) return cudaErrorInvalidValue;
    const size_t smem = (size_t)ns * Lay::SLOT + fixed;

    // per device: the shared-memory attribute, and how many CTAs fit at once
    static std::atomic<int> workers[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int n_workers = dev >= 0 && dev < 64 ? workers[dev].load(std::memory_order_relaxed) : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kFaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (n_workers <= 0) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kFaSmemLimit);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<D, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kFaSmemLimit);
        if (e != cudaSuccess) return e;
        int n_sm = 0;
        e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        n_workers = n_sm;
        if (dev >= 0 && dev < 64) workers[dev].store(n_workers, std::memory_order_relaxed);
    }
    FaParams fp;
    fp.p = p;
    fp.n_slots = ns;
    fp.batch = batch;
    fp.n_rt = (p.n_tok * p.G + 127) / 128;
    fp.n_units = fp.n_rt * batch * p.n_kv;
    fp.n_workers = fp.n_units < n_workers ? fp.n_units : n_workers;
    cfg.gridDim = dim3(fp.n_workers);
    return p.softcap > 0.f ? cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, true>, km, vm, fp)
                           : cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, false>, km, vm, fp);
}

bool prefill_tc_supported(int head_dim) {
    return head_dim == 64 || head_dim == 128 || head_dim == 256 || head_dim == 512;
}

cudaError_t launch_prefill_tc(const RowsParams& p, int head_dim, int batch, cudaStream_t st) {
    switch (head_dim) {
        case 64: return launch_d<64>(p, batch, st);
        case 128: return launch_d<128>(p, batch, st);
        case 256: return launch_prefill_pair(p, 256, batch, st);  // every supported group divides 128
        case 512: return launch_prefill_pair(p, 512, batch, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemma
