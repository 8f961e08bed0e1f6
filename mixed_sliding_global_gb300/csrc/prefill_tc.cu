// prefill_tc.cu -- prefill-bucket attention on 5th-generation tensor cores (tcgen05 + TMEM).
//
// Computes, for a tile of 128 query rows (rows = (token, head of the GQA group) pairs, token
// major, so every row of a tile reads the same KV head), softmax(scale * Q K^T) V over the
// causal (and, on sliding layers, windowed) key range of each row, with the K/V cache of the
// owner layer ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", sections 2.1-2.3; the
// pages' "eager" matmul-softmax-matmul definition, section 4.3).
//
// Each CTA has 6 warps:
//   warps 0-3  softmax: thread r owns row r (TMEM lane r): loads its Q row into TMEM, reads
//              its S row from TMEM, masks by index, keeps (m, l), writes bf16 P to shared
//              memory, rescales its O row in TMEM when the running max grows by more than
//              2^8 (lazy rescaling keeps the result exact: the final division uses the same
//              reference max), and finally writes O / l.
//   warp 4     TMA producer: streams 128-key K and V tiles (128-byte swizzle, one box per
//              64 columns of head_dim) through a ring of shared-memory slots.
//   warp 5     MMA issuer: S = Q K^T (A = Q from TMEM, B = K, K-major) and O += P V (A = P,
//              K-major, B = V, MN-major), fp32 accumulation in TMEM; tcgen05.commit signals
//              the mbarriers that order the warps.
// TMEM (512 columns): Q (DH/2 columns of packed bf16), S (128), O (DH), DH = head_dim / CL.
//
// CL = 2 (head_dim 512): a 128 x 512 fp32 O alone would fill the 512 TMEM columns of an SM,
// so a cluster of two CTAs splits head_dim: CTA h holds Q[:, 256h:256h+256] and reads only
// that half of K and V. Each computes a partial S over its half, sends it to its peer through
// distributed shared memory, and adds the peer's partial to its own; each then accumulates and
// writes its own half of O with its own P, m and l. No multiply-add is done twice. With k_eq_v
// the K half is also the V half.
// The partial scores travel as fp16 (saturating): the exchange, not the tensor core, bounds
// these clusters, and fp16 halves its bytes. Each CTA keeps its own partial in fp32; the peer's
// rounding moves a score by at most 2^-11 of its partial (for |partial| <= 128 raw, <= 0.06 raw,
// i.e. < 0.4% in exp(scale * s) at scale 1/sqrt(512)), the size of the bf16 rounding P already
// gets before P V.
//
// The key range of the tile is clamped to [first row's window start, last row's position]
// before any load; rows of the last partial key tile beyond the range are zeroed in shared
// memory before they enter P V.
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace gemma {

constexpr int kTcThreads = 192;
constexpr int kTcMaxSlots = 8;
constexpr int kTcKeys = 128;                   // keys per tile (N of S = Q K^T)
constexpr int kTcSmemLimit = 232448;           // max dynamic shared memory per block (sm_100)
constexpr float kLazyRescaleLog2 = 8.f;

struct TcParams {
    RowsParams p;
    int n_slots;
};

template <int D, int CL>
struct TcLayout {
    static constexpr int DH = D / CL;                    // head_dim columns owned by a CTA
    static constexpr int CHUNKS = DH / 64;               // 64-column boxes per K/V tile
    static constexpr int SLOT = CHUNKS * kTcKeys * 128;  // bytes of one K or V tile
    static constexpr int P_BYTES = kTcKeys * 128 * 2;    // 128 rows x 128 keys bf16
    static constexpr int X_BYTES = CL > 1 ? 128 * kTcKeys * 2 : 0;  // peer's partial S (fp16)
    static constexpr int Q_COL = 0;                      // TMEM columns
    static constexpr int S_COL = 128;
    static constexpr int O_COL = 256;
    static_assert(DH / 2 <= 128 && 256 + DH <= 512, "TMEM budget");
};

// ---------------------------------------------------------------------------------------------
// cluster helpers (distributed shared memory between the two CTAs of a cluster)
// ---------------------------------------------------------------------------------------------
GEMMA_DEVINL uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
GEMMA_DEVINL void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
GEMMA_DEVINL uint32_t map_to_peer(const void* local, uint32_t peer) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(peer));
    return r;
}
GEMMA_DEVINL void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}
// two fp32 -> packed fp16 (lo in the low half), round to nearest; values beyond the fp16
// range saturate to +-65504 instead of becoming infinite
GEMMA_DEVINL uint32_t pack_f16_sat(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
GEMMA_DEVINL float2 unpack_f16(uint32_t v) {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
}
GEMMA_DEVINL void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
GEMMA_DEVINL bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait with cluster-scope acquire (data written by the peer CTA becomes visible).
GEMMA_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
            report(err, GEMMA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// SOFTCAP: the soft-capped variant (a separate instantiation, so that the plain kernel carries
// no code for it)
template <int D, int CL, bool SOFTCAP>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcParams tp) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    using Lay = TcLayout<D, CL>;
    constexpr int DH = Lay::DH;
    const RowsParams& p = tp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NS = tp.n_slots;
    uint8_t* slots = smem;
    uint8_t* sP = smem + NS * Lay::SLOT;
    float* sX = reinterpret_cast<float*>(sP + Lay::P_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + Lay::P_BYTES + Lay::X_BYTES);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = bars + kTcMaxSlots;
    uint64_t* q_ready = bars + 2 * kTcMaxSlots;
    uint64_t* s_full = q_ready + 1;
    uint64_t* s_free = q_ready + 2;
    uint64_t* p_full = q_ready + 3;
    uint64_t* o_done = q_ready + 4;
    uint64_t* x_full = q_ready + 5;  // the peer's partial S has landed in sX
    uint64_t* x_free = q_ready + 6;  // the peer has read the partial S this CTA sent it
    uint32_t* tslot = reinterpret_cast<uint32_t*>(q_ready + 7);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t h = CL > 1 ? cluster_rank() : 0u;  // which head_dim part this CTA owns
    const int rt = blockIdx.x / CL, kvh = blockIdx.y, b = blockIdx.z;
    const int rows_total = p.n_tok * p.G;
    const int row0 = rt * 128;
    const int n_rows = min(128, rows_total - row0);  // rows of the bucket this CTA writes
    const int len = __ldg(p.seq_lens + b);
    // real tokens of this sequence (a padded bucket's first n_real rows; all rows otherwise);
    // the i-th real token sits at len - n_real + i, the pad rows' outputs are zero
    const int n_real = p.n_real ? __ldg(p.n_real + b) : p.n_tok;
    const bool bad_real = n_real < 0 || n_real > p.n_tok;
    const bool bad = bad_real || len < n_real || (!p.ring && len > p.cap) || len > p.max_seq_len;
    const int n_rows_real = bad ? 0 : max(0, min(128, n_real * p.G - row0));  // rows that attend

    // key range of the tile: from the first row's window start to the last real row's position
    const int tok_first = row0 / p.G, tok_last = (row0 + max(n_rows_real, 1) - 1) / p.G;
    const int pos_first = len - n_real + tok_first, pos_last = len - n_real + tok_last;
    // (a ring cache's tiles start at multiples of the tile, so that none wraps around the ring;
    // the rows' masks drop the keys before the window)
    const int k_begin = p.is_sliding ? (max(0, pos_first - p.window + 1) & ((p.ring || p.page_size) ? ~(kTcKeys - 1) : ~0))
                                     : 0;
    const int k_end = pos_last + 1;
    const int n_tiles = n_rows_real == 0 ? 0 : (k_end - k_begin + kTcKeys - 1) / kTcKeys;
    // K/V ring split: with K = V one ring of NS slots; otherwise NV slots for V (V is needed
    // only by P V, which comes last) and the rest for K
    const int NV = p.k_eq_v ? 0 : (NS / 3 > 1 ? NS / 3 : 1);
    const int NK = NS - NV;

    if (warp == 5) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(q_ready, 128);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(x_full, 128);
        mbar_init(x_free, 128);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tQ = tmem + Lay::Q_COL, tS = tmem + Lay::S_COL, tO = tmem + Lay::O_COL;

    if (warp == 4) {
        // ------------------------------- TMA producer --------------------------------------
        // K tiles use slots [0, NK), V tiles slots [NK, NS). K runs one tile ahead of V, so a
        // K slot is refilled as soon as its S = Q K^T finished, independently of P V.
        if (lane == 0) {
            auto load = [&](const CUtensorMap* map, int slot, int t) {
                uint8_t* dst = slots + slot * Lay::SLOT;
                mbar_arrive_expect_tx(&kv_full[slot], Lay::SLOT);
                // cache row and slot of the tile's first key (a bad page index reads zeros)
                int row3 = 0, slot0 = 0;
                if (!kv_place(p, b, kvh, k_begin + t * kTcKeys, row3, slot0)) {
                    report(p.err, GEMMA_DEVERR_PAGE);
                    row3 = p.n_pages * p.n_kv;
                }
                for (int c = 0; c < Lay::CHUNKS; ++c)
                    tma_load_3d(dst + c * kTcKeys * 128, map, (int)h * DH + c * 64, slot0, row3,
                                &kv_full[slot]);
            };
            bool ok = true;
            // ring cursors (slot, phase of the current pass, whether a pass has completed):
            // kept incrementally, no division by the runtime ring sizes
            int ks = 0, vs = 0;
            uint32_t kph = 0, vph = 0;
            bool kwrap = false, vwrap = false;
            for (int i = 0; i <= n_tiles && ok; ++i) {
                const int tk = i;          // K tile issued at step i
                const int tv = i - 1;      // V tile issued at step i
                if (tk < n_tiles) {
                    if (kwrap) ok = mbar_wait(&kv_empty[ks], kph ^ 1u, p.err);
                    if (ok) load(&kmap, ks, tk);
                    if (++ks == NK) {
                        ks = 0;
                        kph ^= 1u;
                        kwrap = true;
                    }
                }
                if (!p.k_eq_v && tv >= 0 && ok) {
                    if (vwrap) ok = mbar_wait(&kv_empty[NK + vs], vph ^ 1u, p.err);
                    if (ok) load(&vmap, NK + vs, tv);
                    if (++vs == NV) {
                        vs = 0;
                        vph ^= 1u;
                        vwrap = true;
                    }
                }
            }
        }
    } else if (warp == 5) {
        // -------------------------------- MMA issuer ---------------------------------------
        const uint32_t id_qk = idesc_bf16(128, kTcKeys, 0, 0);
        const uint32_t id_pv = idesc_bf16(128, DH, 0, 1);
        bool ok = mbar_wait(q_ready, 0, p.err);
        // rows [0, n_head) of the first tile when it starts before every row's window (a
        // tile-aligned start): masked keys whose values must not reach P V as 0 * x
        const int n_head = p.is_sliding ? max(0, max(0, pos_first - p.window + 1) - k_begin) : 0;
        auto zero_head = [&](uint8_t* tile) {
            for (int idx = lane; idx < Lay::CHUNKS * n_head * 8; idx += 32) {
                const int c = idx / (n_head * 8), rem = idx - c * n_head * 8;
                *reinterpret_cast<uint4*>(tile + c * kTcKeys * 128 + (rem / 8) * 128 +
                                          (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        auto zero_tail = [&](uint8_t* tile, int n_valid) {
            // rows [n_valid, 128) of every 64-column box: whole 128-byte rows, so the
            // swizzle does not matter
            const int n_zero = kTcKeys - n_valid;
            for (int idx = lane; idx < Lay::CHUNKS * n_zero * 8; idx += 32) {
                const int c = idx / (n_zero * 8), rem = idx - c * n_zero * 8;
                const int r = n_valid + rem / 8, q16 = rem % 8;
                *reinterpret_cast<uint4*>(tile + c * kTcKeys * 128 + r * 128 + q16 * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        // ring cursors of the consumer side: K slot and phase for S = Q K^T, V slot and phase
        // for P V, and (with K as V) the slot of the previous K tile
        int mk = 0, mv = 0, k_prev = 0;
        uint32_t mkph = 0, mvph = 0;
        auto issue_pv = [&](int j) {
            if (ok) ok = mbar_wait(p_full, j & 1, p.err);
            const int sv = p.k_eq_v ? k_prev : NK + mv;
            const uint32_t sv_phase = mvph;
            if (!p.k_eq_v && ++mv == NV) {
                mv = 0;
                mvph ^= 1u;
            }
            if (ok && !p.k_eq_v) {
                ok = mbar_wait(&kv_full[sv], sv_phase, p.err);
                const int n_valid = k_end - (k_begin + j * kTcKeys);
                if (n_valid < kTcKeys) zero_tail(slots + sv * Lay::SLOT, n_valid);
                if (j == 0 && n_head > 0) zero_head(slots + sv * Lay::SLOT);
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t vbase = smem_u32(slots + sv * Lay::SLOT);
                const uint32_t pbase = smem_u32(sP);
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(pbase + (kk / 4) * (kTcKeys * 128) +
                                                           (kk % 4) * 32, 0, 1024);
                    const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, kTcKeys * 128, 1024);
                    umma_ss(tO, a, bd, id_pv, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(o_done);
                umma_commit(&kv_empty[sv]);
            }
            __syncwarp();
        };
        for (int t = 0; t < n_tiles; ++t) {
            const int sk = mk;
            if (ok) ok = mbar_wait(&kv_full[sk], mkph, p.err);
            if (++mk == NK) {
                mk = 0;
                mkph ^= 1u;
            }
            if (p.k_eq_v) {
                const int n_valid = k_end - (k_begin + t * kTcKeys);
                if (n_valid < kTcKeys) zero_tail(slots + sk * Lay::SLOT, n_valid);
                if (t == 0 && n_head > 0) zero_head(slots + sk * Lay::SLOT);
            }
            if (t >= 1 && ok) ok = mbar_wait(s_free, (t - 1) & 1, p.err);
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kbase = smem_u32(slots + sk * Lay::SLOT);
#pragma unroll
                for (int c = 0; c < Lay::CHUNKS; ++c)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_ts(tS, tQ + c * 32 + ks * 8,
                                smem_desc_sw128(kbase + c * kTcKeys * 128 + ks * 32, 0, 1024),
                                id_qk, (c | ks) ? 1u : 0u);
                umma_commit(s_full);
                if (!p.k_eq_v) umma_commit(&kv_empty[sk]);
            }
            __syncwarp();
            if (t >= 1) issue_pv(t - 1);
            k_prev = sk;
        }
        if (n_tiles > 0) issue_pv(n_tiles - 1);
    } else {
        // ------------------------------ softmax warps --------------------------------------
        const int r = threadIdx.x;  // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const bool row_ok = r < n_rows_real;
        int token = 0, head = 0, lo = 1, hi = 0;
        if (row_ok) {
            const int R = row0 + r;
            token = R / p.G;
            head = kvh * p.G + (R - token * p.G);
            const int pos = len - n_real + token;
            lo = p.is_sliding ? max(0, pos - p.window + 1) : 0;
            hi = pos + 1;
        }
        // this CTA's part of the Q row into TMEM (zeros for rows outside the tile)
        {
            const uint4* qrow = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) +
                (((size_t)b * p.n_tok + token) * p.n_q + head) * (size_t)D + h * DH);
#pragma unroll
            for (int j = 0; j < DH / 64; ++j) {
                uint32_t v[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint4 x = row_ok ? __ldg(qrow + j * 8 + e) : make_uint4(0u, 0u, 0u, 0u);
                    v[4 * e + 0] = x.x;
                    v[4 * e + 1] = x.y;
                    v[4 * e + 2] = x.z;
                    v[4 * e + 3] = x.w;
                }
                tmem_st32(tQ + lane_off + j * 32, v);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(q_ready);

        uint32_t peer_x = 0, peer_x_full = 0, peer_x_free = 0;
        if (CL > 1) {
            peer_x = map_to_peer(sX + 4 * r, h ^ 1u);
            peer_x_full = map_to_peer(x_full, h ^ 1u);
            peer_x_free = map_to_peer(x_free, h ^ 1u);
        }

        bool ok = true;
        float m_ref = -INFINITY, l = 0.f;
        for (int t = 0; t < n_tiles; ++t) {
            if (ok) ok = mbar_wait(s_full, t & 1, p.err);
            tc_fence_after();
            float s[kTcKeys];
#pragma unroll
            for (int j = 0; j < kTcKeys / 32; ++j) {
                uint32_t v[32];
                tmem_ld32(tS + lane_off + j * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) s[j * 32 + e] = __uint_as_float(v[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);

            if (CL > 1) {
                // send this row's partial scores to the peer, then add the peer's partial
                if (t >= 1 && ok) ok = mbar_wait_cluster(x_free, (t - 1) & 1, p.err);
                // chunk-major layout X[c][r] (16-byte chunks of 8 fp16 scores): a warp's 32
                // stores of chunk c are one contiguous 512-byte write, and the local loads are
                // contiguous too
#pragma unroll
                for (int c = 0; c < kTcKeys / 8; ++c)
                    st_cluster_v4(peer_x + c * (128 * 16), pack_f16_sat(s[8 * c], s[8 * c + 1]),
                                  pack_f16_sat(s[8 * c + 2], s[8 * c + 3]),
                                  pack_f16_sat(s[8 * c + 4], s[8 * c + 5]),
                                  pack_f16_sat(s[8 * c + 6], s[8 * c + 7]));
                mbar_arrive_remote(peer_x_full);
                if (ok) ok = mbar_wait_cluster(x_full, t & 1, p.err);
                const uint4* xr = reinterpret_cast<const uint4*>(sX) + r;
#pragma unroll
                for (int e = 0; e < kTcKeys / 8; ++e) {
                    const uint4 x = xr[e * 128];
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = unpack_f16(w[i]);
                        s[8 * e + 2 * i] += f.x;
                        s[8 * e + 2 * i + 1] += f.y;
                    }
                }
                mbar_arrive_remote(peer_x_free);
            }

            // scores stay raw; scale > 0, so max(raw) * scale_log2 is the max of scaled scores.
            // With a soft-cap they are first mapped to c * tanh(scale * raw / c) in log2 units
            // (before the mask, so masked keys stay -inf).
            float sl2 = p.scale_log2;
            if (SOFTCAP) {
#pragma unroll
                for (int e = 0; e < kTcKeys; ++e) s[e] = p.cap_log2 * tanhf(s[e] * p.cap_inner);
                sl2 = 1.f;
            }
            const int kt0 = k_begin + t * kTcKeys;
            const bool full = kt0 >= lo && kt0 + kTcKeys <= hi;
            if (!full) {
#pragma unroll
                for (int e = 0; e < kTcKeys; ++e) {
                    const int key = kt0 + e;
                    if (key < lo || key >= hi) s[e] = -INFINITY;
                }
            }
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
            for (int e = 8; e < kTcKeys; e += 8)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[e + i]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                             sl2;
            const bool need = mx > m_ref + kLazyRescaleLog2;
            const float m_new = need ? mx : m_ref;
            if (t > 0 && ok) ok = mbar_wait(o_done, (t - 1) & 1, p.err);
            if (t > 0 && __any_sync(0xffffffffu, need)) {
                const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
                tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < DH / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld32(tO + lane_off + j * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(tO + lane_off + j * 32, v);
                }
                tmem_st_wait();
                l *= alpha;
            }
            m_ref = m_new;
            // p = 2^(raw * scale_log2 - m): one FFMA and one MUFU exp2 per score
            const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k0 = kb * 64 + c * 8 + 2 * e;
                        const float p0 = fast_exp2(fmaf(s[k0], sl2, neg_m));
                        const float p1 = fast_exp2(fmaf(s[k0 + 1], sl2, neg_m));
                        sum4[e] += p0 + p1;
                        w[e] = pack_bf16(p0, p1);
                    }
                    *reinterpret_cast<uint4*>(sP + kb * (kTcKeys * 128) + r * 128 +
                                              ((c ^ (r & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // epilogue: O / l -> bf16 (zeros for a sequence with a bad length)
        if (n_tiles > 0 && ok) ok = mbar_wait(o_done, (n_tiles - 1) & 1, p.err);
        tc_fence_after();
        {
            // every lane runs the collective TMEM loads; only rows of the tile store
            const int R = row0 + (r < n_rows ? r : 0);
            const int tk = R / p.G, hd = kvh * p.G + (R - tk * p.G);
            uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                   (((size_t)b * p.n_tok + tk) * p.n_q + hd) * (size_t)D +
                                                   h * DH);
            const float inv = (bad || l == 0.f) ? 0.f : 1.f / l;
#pragma unroll 1
            for (int j = 0; j < DH / 32; ++j) {
                uint32_t v[32];
                if (n_tiles > 0) {
                    tmem_ld32(tO + lane_off + j * 32, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                if (r < n_rows) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        orow[j * 4 + e] = make_uint4(
                            pack_bf16(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv),
                            pack_bf16(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv),
                            pack_bf16(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv),
                            pack_bf16(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv));
                }
            }
        }
        if (bad && r == 0 && kvh == 0 && rt == 0 && h == 0)
            report(p.err, bad_real ? GEMMA_DEVERR_N_REAL : GEMMA_DEVERR_SEQ_LEN);
    }
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync();  // the peer no longer writes into this CTA's shared memory
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
template <int D, int CL>
static cudaError_t launch_d(const RowsParams& p, int batch, cudaStream_t st) {
    using Lay = TcLayout<D, CL>;
    CUtensorMap km, vm;
    // [rows][slots][D]: rows = sequences x KV heads (pages x KV heads for a paged pool)
    const uint64_t map_slots = p.page_size ? (uint64_t)p.page_size : (uint64_t)p.cap;
    const uint64_t map_rows = p.page_size ? (uint64_t)p.n_pages * p.n_kv : (uint64_t)batch * p.n_kv;
    const uint64_t dims[3] = {(uint64_t)D, map_slots, map_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, map_slots * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kTcKeys, 1};
    if (!encode_bf16_sw128(&km, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&vm, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    TcParams tp;
    tp.p = p;
    const int fixed = Lay::P_BYTES + Lay::X_BYTES + 256 + 1024;  // P, X, barriers, alignment
    int ns = (kTcSmemLimit - fixed) / Lay::SLOT;
    if (ns > kTcMaxSlots) ns = kTcMaxSlots;
    if (ns < 2) return cudaErrorInvalidValue;
    tp.n_slots = ns;
    const size_t smem = (size_t)ns * Lay::SLOT + fixed;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, CL, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemLimit);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<D, CL, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemLimit);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    const int rows = p.n_tok * p.G;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * ((rows + 127) / 128), p.n_kv, batch);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return p.softcap > 0.f ? cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, CL, true>, km, vm, tp)
                           : cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, CL, false>, km, vm, tp);
}

bool prefill_tc_supported(int head_dim) {
    return head_dim == 64 || head_dim == 128 || head_dim == 256 || head_dim == 512;
}

cudaError_t launch_prefill_tc(const RowsParams& p, int head_dim, int batch, cudaStream_t st) {
    switch (head_dim) {
        case 64: return launch_d<64, 1>(p, batch, st);
        case 128: return launch_d<128, 1>(p, batch, st);
        case 256: return launch_d<256, 1>(p, batch, st);
        case 512: return launch_d<512, 2>(p, batch, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemma
