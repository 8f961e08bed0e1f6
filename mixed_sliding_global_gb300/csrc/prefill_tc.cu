// prefill_tc.cu -- prefill-bucket attention on 5th-generation tensor cores (tcgen05 + TMEM).
//
// Computes, for a tile of 128 query rows (rows = (token, head of the GQA group) pairs, token
// major, so every row of a tile reads the same KV head), softmax(scale * Q K^T) V over the
// causal (and, on sliding layers, windowed) key range of each row, with the K/V cache of the
// owner layer ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", sections 2.1-2.3; the
// pages' "eager" matmul-softmax-matmul definition, section 4.3).
//
// One CTA per (128-row tile, KV head, sequence); 6 warps:
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
// TMEM (512 columns): Q (head_dim/2 columns of packed bf16), S (128), O (head_dim).
// The key range of the tile is clamped to [first row's window start, last row's position]
// before any load; rows of the last partial key tile beyond the range are zeroed in shared
// memory before they enter P V.
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
    int slot_bytes;
};

template <int D>
struct TcLayout {
    static constexpr int CHUNKS = D / 64;              // 64-column boxes per K/V tile
    static constexpr int SLOT = CHUNKS * kTcKeys * 128;  // bytes of one K or V tile
    static constexpr int P_BYTES = kTcKeys * 128 * 2;   // 128 rows x 128 keys bf16
    static constexpr int Q_COL = 0;                       // TMEM columns
    static constexpr int S_COL = 128;
    static constexpr int O_COL = 256;
    static_assert(D / 2 <= 128 && 256 + D <= 512, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcParams tp) {
    using Lay = TcLayout<D>;
    const RowsParams& p = tp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NS = tp.n_slots;
    uint8_t* slots = smem;
    uint8_t* sP = smem + NS * Lay::SLOT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + Lay::P_BYTES);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = bars + kTcMaxSlots;
    uint64_t* q_ready = bars + 2 * kTcMaxSlots;
    uint64_t* s_full = q_ready + 1;
    uint64_t* s_free = q_ready + 2;
    uint64_t* p_full = q_ready + 3;
    uint64_t* o_done = q_ready + 4;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(q_ready + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int rows_total = p.n_tok * p.G;
    const int row0 = rt * 128;
    const int n_rows = min(128, rows_total - row0);
    const int len = __ldg(p.seq_lens + b);
    const bool bad = len < p.n_tok || len > p.cap || len > p.max_seq_len;

    // key range of the tile: from the first row's window start to the last row's position
    const int tok_first = row0 / p.G, tok_last = (row0 + n_rows - 1) / p.G;
    const int pos_first = len - p.n_tok + tok_first, pos_last = len - p.n_tok + tok_last;
    const int k_begin = p.is_sliding ? max(0, pos_first - p.window + 1) : 0;
    const int k_end = pos_last + 1;
    const int n_tiles = bad ? 0 : (k_end - k_begin + kTcKeys - 1) / kTcKeys;
    const int ops_per_tile = p.k_eq_v ? 1 : 2;
    const int n_ops = n_tiles * ops_per_tile;

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
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tQ = tmem + Lay::Q_COL, tS = tmem + Lay::S_COL, tO = tmem + Lay::O_COL;

    if (warp == 4) {
        // ------------------------------- TMA producer --------------------------------------
        if (lane == 0) {
            const int row3 = b * p.n_kv + kvh;
            for (int u = 0; u < n_ops; ++u) {
                const int s = u % NS;
                if (u >= NS && !mbar_wait(&kv_empty[s], ((u / NS) - 1) & 1, p.err)) break;
                const int t = u / ops_per_tile;
                const bool is_v = (u % ops_per_tile) == 1;
                const CUtensorMap* map = is_v ? &vmap : &kmap;
                uint8_t* dst = slots + s * Lay::SLOT;
                mbar_arrive_expect_tx(&kv_full[s], Lay::SLOT);
                for (int c = 0; c < Lay::CHUNKS; ++c)
                    tma_load_3d(dst + c * kTcKeys * 128, map, c * 64, k_begin + t * kTcKeys, row3,
                                &kv_full[s]);
            }
        }
    } else if (warp == 5) {
        // -------------------------------- MMA issuer ---------------------------------------
        const uint32_t id_qk = idesc_bf16(128, kTcKeys, 0, 0);
        const uint32_t id_pv = idesc_bf16(128, D, 0, 1);
        bool ok = mbar_wait(q_ready, 0, p.err);
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
        auto issue_pv = [&](int j) {
            if (ok) ok = mbar_wait(p_full, j & 1, p.err);
            const int uv = j * ops_per_tile + ops_per_tile - 1;
            const int sv = uv % NS;
            if (ok && !p.k_eq_v) {
                ok = mbar_wait(&kv_full[sv], (uv / NS) & 1, p.err);
                const int n_valid = k_end - (k_begin + j * kTcKeys);
                if (n_valid < kTcKeys) zero_tail(slots + sv * Lay::SLOT, n_valid);
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
            const int uk = t * ops_per_tile;
            const int sk = uk % NS;
            if (ok) ok = mbar_wait(&kv_full[sk], (uk / NS) & 1, p.err);
            if (p.k_eq_v) {
                const int n_valid = k_end - (k_begin + t * kTcKeys);
                if (n_valid < kTcKeys) zero_tail(slots + sk * Lay::SLOT, n_valid);
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
        }
        if (n_tiles > 0) issue_pv(n_tiles - 1);
    } else {
        // ------------------------------ softmax warps --------------------------------------
        const int r = threadIdx.x;  // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const bool row_ok = !bad && r < n_rows;
        int token = 0, head = 0, lo = 1, hi = 0;
        if (row_ok) {
            const int R = row0 + r;
            token = R / p.G;
            head = kvh * p.G + (R - token * p.G);
            const int pos = len - p.n_tok + token;
            lo = p.is_sliding ? max(0, pos - p.window + 1) : 0;
            hi = pos + 1;
        }
        // Q row into TMEM (zeros for rows outside the tile)
        {
            const uint4* qrow = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) +
                (((size_t)b * p.n_tok + token) * p.n_q + head) * (size_t)D);
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
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

            const int kt0 = k_begin + t * kTcKeys;
            const bool full = kt0 >= lo && kt0 + kTcKeys <= hi;
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < kTcKeys; ++e) {
                const int key = kt0 + e;
                const bool valid = full || (key >= lo && key < hi);
                s[e] = valid ? s[e] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[e]);
            }
            const bool need = mx > m_ref + kLazyRescaleLog2;
            const float m_new = need ? mx : m_ref;
            if (t > 0 && ok) ok = mbar_wait(o_done, (t - 1) & 1, p.err);
            if (t > 0 && __any_sync(0xffffffffu, need)) {
                const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
                tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < D / 32; ++j) {
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
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            float sum = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k0 = kb * 64 + c * 8 + 2 * e;
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(exp2f(s[k0] - m_use),
                                                                         exp2f(s[k0 + 1] - m_use));
                        const float2 back = __bfloat1622float2(pr);
                        sum += back.x + back.y;
                        w[e] = *reinterpret_cast<const uint32_t*>(&pr);
                    }
                    *reinterpret_cast<uint4*>(sP + kb * (kTcKeys * 128) + r * 128 +
                                              ((c ^ (r & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            l += sum;
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // epilogue: O / l -> bf16 rows of out (zeros for a sequence with a bad length)
        if (n_tiles > 0 && ok) ok = mbar_wait(o_done, (n_tiles - 1) & 1, p.err);
        tc_fence_after();
        {
            // every lane runs the collective TMEM loads; only rows of the tile store
            const int R = row0 + (r < n_rows ? r : 0);
            const int tk = R / p.G, hd = kvh * p.G + (R - tk * p.G);
            uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                   (((size_t)b * p.n_tok + tk) * p.n_q + hd) * (size_t)D);
            const float inv = (bad || l == 0.f) ? 0.f : 1.f / l;
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
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
        if (bad && r == 0 && kvh == 0 && rt == 0) report(p.err, GEMMA_DEVERR_SEQ_LEN);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
template <int D>
static cudaError_t launch_d(const RowsParams& p, int batch, cudaStream_t st) {
    using Lay = TcLayout<D>;
    CUtensorMap km, vm;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.cap, (uint64_t)batch * p.n_kv};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.cap * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kTcKeys, 1};
    if (!encode_bf16_sw128(&km, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&vm, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    TcParams tp;
    tp.p = p;
    tp.slot_bytes = Lay::SLOT;
    const int fixed = Lay::P_BYTES + 256 + 1024;  // P, barriers, alignment slack
    int ns = (kTcSmemLimit - fixed) / Lay::SLOT;
    if (ns > kTcMaxSlots) ns = kTcMaxSlots;
    tp.n_slots = ns;
    const size_t smem = (size_t)ns * Lay::SLOT + fixed;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemLimit);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    const int rows = p.n_tok * p.G;
    dim3 grid((rows + 127) / 128, p.n_kv, batch);
    prefill_tc_kernel<D><<<grid, kTcThreads, smem, st>>>(km, vm, tp);
    return cudaGetLastError();
}

bool prefill_tc_supported(int head_dim) { return head_dim == 64 || head_dim == 128 || head_dim == 256; }

cudaError_t launch_prefill_tc(const RowsParams& p, int head_dim, int batch, cudaStream_t st) {
    switch (head_dim) {
        case 64: return launch_d<64>(p, batch, st);
        case 128: return launch_d<128>(p, batch, st);
        case 256: return launch_d<256>(p, batch, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemma
