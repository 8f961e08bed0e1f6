// logits.cu -- final-logit soft-cap and greedy argmax over the vocabulary.
//
// "Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2" (family table and section 4.2): the
// model caps its output logits to softcap * tanh(logits / softcap) over the whole vocabulary
// (softcap 30, 262,144 tokens), and the argmax of the capped logits is the argmax of the raw
// ones (tanh is increasing), so greedy decoding does not depend on the cap. Here one pass over
// each row writes the capped logits (when asked) and finds the greedy index on the raw values:
// the lowest index of the maximum, NaN never selected, a row of NaN giving index 0.
//
// Work is HBM-bound (2 bytes read, and 2 written with the capped output, per bf16 logit). One
// wave of CTAs (as many as fit on the GPU at once) covers the flattened [batch][vocab] logits
// in equal contiguous ranges, so every SM streams the same number of bytes whatever the batch;
// CTA c owns elements [ceil(c N / C), ceil((c + 1) N / C)), i.e. element e belongs to CTA
// floor(e C / N). Each thread streams 16-byte vectors, four in flight, and keeps the best
// (key, index) of the elements it saw in increasing index order, where key is an
// order-preserving map of the float to an unsigned integer (NaN lowest, -0 taken as +0);
// (key, index) pairs pack into one 64-bit word, key high and the index's complement low, so a
// plain maximum picks the largest value and, among equal values, the lowest index. A CTA
// reduces once per row its range touches and stores the word at piece b + c (unique: pieces
// of later rows and later CTAs have larger ids); a second launch, one warp per row, reduces
// the pieces of its row. When the batch is large enough that each row can have its own CTAs
// (at most 16, filling at least half the wave), the k CTAs of a row instead form one thread-
// block cluster: each sends its word to the first CTA's shared memory and, after a cluster
// barrier, that CTA writes the row's index (one launch, no workspace).
#include "common.cuh"
#include "logits.h"

namespace gemma {

constexpr int kLgThreads = 256;
constexpr int kLgUnroll = 4;                   // 16-byte vectors in flight per thread
constexpr int kLgMinChunk = 8192;              // logits per CTA at least
constexpr uint32_t kLgNoIndex = 0x7fffffffu;   // no non-NaN element seen
constexpr int kLgMaxRowCtas = 16;              // the largest cluster (non-portable above 8)

GEMMA_DEVINL uint32_t order_key(float f) {
    if (f != f) return 0u;         // NaN: below every number
    if (f == 0.f) f = 0.f;         // -0 equals +0
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
GEMMA_DEVINL unsigned long long pack_best(uint32_t key, uint32_t idx) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - idx);
}
GEMMA_DEVINL uint32_t unpack_index(unsigned long long w) {
    const uint32_t idx = 0xffffffffu - (uint32_t)(w & 0xffffffffull);
    return idx == kLgNoIndex ? 0u : idx;
}
GEMMA_DEVINL float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct LogitParams {
    const void* logits;
    void* capped;              // or nullptr
    int32_t* argmax;
    unsigned long long* part;  // [batch + n_cta] piece words
    long long total;           // batch * vocab
    int vocab, n_cta;
    float softcap, inv_cap;    // softcap 0: capped = x
};

// first flattened element of CTA c, and the CTA that owns element e (N elements, C CTAs)
GEMMA_DEVINL long long cta_begin(long long c, long long N, long long C) { return (c * N + C - 1) / C; }
GEMMA_DEVINL long long cta_of(long long e, long long N, long long C) { return e * C / N; }

// Per-vector operations on one 16-byte vector of logits: its maximum (NaN ignored unless all
// are NaN), element e, and the capped vector c * tanh(x / c). tanh: the hardware approximation
// for bf16 output (its relative error, below 2^-10.9, is a fraction of the bf16 rounding,
// 2^-8), the accurate library function for fp32 output.
template <typename T>
struct LgTraits;
template <>
struct LgTraits<__nv_bfloat16> {
    static constexpr int VEC = 8;
    GEMMA_DEVINL static float tanh1(float x) { return tanh_approx(x); }
    GEMMA_DEVINL static float vmax(const uint4& v) {
        uint32_t m;
        asm("{\n\t.reg .b32 t0, t1;\n\t"
            "max.bf16x2 t0, %1, %2;\n\tmax.bf16x2 t1, %3, %4;\n\tmax.bf16x2 %0, t0, t1;\n\t}"
            : "=r"(m) : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    GEMMA_DEVINL static float get(const uint4& v, int e) {
        const uint32_t w = (&v.x)[e >> 1];
        return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    GEMMA_DEVINL static uint4 capvec(const uint4& v, float c, float ic) {
        uint4 o;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t w = (&v.x)[k];
            const float y0 = c * tanh1(__uint_as_float(w << 16) * ic);
            const float y1 = c * tanh1(__uint_as_float(w & 0xffff0000u) * ic);
            (&o.x)[k] = pack_bf16(y0, y1);
        }
        return o;
    }
    GEMMA_DEVINL static float load1(const void* p, size_t i) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    }
    GEMMA_DEVINL static void store1(void* p, size_t i, float f) {
        reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(f);
    }
};
template <>
struct LgTraits<float> {
    static constexpr int VEC = 4;
    GEMMA_DEVINL static float tanh1(float x) { return tanhf(x); }
    GEMMA_DEVINL static float vmax(const uint4& v) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    GEMMA_DEVINL static float get(const uint4& v, int e) { return __uint_as_float((&v.x)[e]); }
    GEMMA_DEVINL static uint4 capvec(const uint4& v, float c, float ic) {
        uint4 o;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            (&o.x)[k] = __float_as_uint(c * tanh1(__uint_as_float((&v.x)[k]) * ic));
        return o;
    }
    GEMMA_DEVINL static float load1(const void* p, size_t i) {
        return reinterpret_cast<const float*>(p)[i];
    }
    GEMMA_DEVINL static void store1(void* p, size_t i, float f) {
        reinterpret_cast<float*>(p)[i] = f;
    }
};

// One thread's share of elements [i0, i1) of the row starting at flattened element `row`: the
// capped copy (CAPPED) and the thread's best packed (key, index) word.
template <typename T, bool CAPPED>
GEMMA_DEVINL unsigned long long scan_range(const LogitParams& p, long long row, int i0, int i1) {
    using Tr = LgTraits<T>;
    constexpr int VEC = Tr::VEC;
    auto cap = [&](float x) { return p.softcap > 0.f ? p.softcap * Tr::tanh1(x * p.inv_cap) : x; };
    // 16-byte aligned body [a0, a1) of [i0, i1); scalar head and tail around it
    const int mis = (int)((row + i0) % VEC);
    const int a0 = min(i1, i0 + (mis ? VEC - mis : 0));
    const int nvec = (i1 - a0) / VEC;
    const int a1 = a0 + nvec * VEC;
    uint32_t bk = 0u, bi = kLgNoIndex;
    auto see = [&](float x, int i) {
        const uint32_t k = order_key(x);
        if (k > bk) {  // elements arrive in increasing index order: ties keep the first
            bk = k;
            bi = (uint32_t)i;
        }
    };
    for (int i = i0 + (int)threadIdx.x; i < a0; i += blockDim.x) {
        const float x = Tr::load1(p.logits, row + i);
        see(x, i);
        if (CAPPED) Tr::store1(p.capped, row + i, cap(x));
    }
    const uint4* src =
        reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.logits) + row + a0);
    uint4* dst =
        CAPPED ? reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.capped) + row + a0) : nullptr;
    for (int v0 = (int)threadIdx.x; v0 < nvec; v0 += kLgUnroll * blockDim.x) {
        uint4 w[kLgUnroll];
#pragma unroll
        for (int u = 0; u < kLgUnroll; ++u) {
            const int v = v0 + u * blockDim.x;
            if (v < nvec) w[u] = __ldcs(src + v);
        }
#pragma unroll
        for (int u = 0; u < kLgUnroll; ++u) {
            const int v = v0 + u * blockDim.x;
            if (v >= nvec) break;
            // the vector's maximum first; only a new best is located inside the vector
            const float vm = Tr::vmax(w[u]);
            const uint32_t vk = order_key(vm);
            if (vk > bk) {
                int e = VEC - 1;  // first element equal to the maximum
#pragma unroll
                for (int k = VEC - 1; k >= 0; --k)
                    if (Tr::get(w[u], k) == vm) e = k;
                bk = vk;
                bi = (uint32_t)(a0 + v * VEC + e);
            }
            if (CAPPED)
                __stcs(dst + v, p.softcap > 0.f ? Tr::capvec(w[u], p.softcap, p.inv_cap) : w[u]);
        }
    }
    for (int i = a1 + (int)threadIdx.x; i < i1; i += blockDim.x) {
        const float x = Tr::load1(p.logits, row + i);
        see(x, i);
        if (CAPPED) Tr::store1(p.capped, row + i, cap(x));
    }
    return pack_best(bk, bi);
}

// The largest of the CTA's per-thread words, in warp 0 (all threads call it; s_best is free
// again when it returns)
GEMMA_DEVINL unsigned long long cta_max(unsigned long long best, unsigned long long* s_best) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < (int)(blockDim.x >> 5) ? s_best[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
    }
    __syncthreads();
    return best;
}

template <typename T, bool CAPPED>
__global__ void __launch_bounds__(kLgThreads) logit_split_kernel(const LogitParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    __shared__ unsigned long long s_best[kLgThreads / 32];
    const long long N = p.total, C = p.n_cta, c = blockIdx.x;
    const long long e_end = cta_begin(c + 1, N, C);
    for (long long e = cta_begin(c, N, C); e < e_end;) {  // one pass per row the range touches
        const int b = (int)(e / p.vocab);
        const long long row = (long long)b * p.vocab;
        const int i0 = (int)(e - row);
        const int i1 = (int)((e_end < row + p.vocab ? e_end : row + p.vocab) - row);
        const unsigned long long best = cta_max(scan_range<T, CAPPED>(p, row, i0, i1), s_best);
        if (threadIdx.x == 0) p.part[(long long)b + c] = best;
        e = row + i1;
    }
}

__global__ void __launch_bounds__(32) logit_finish_kernel(const LogitParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    const int b = blockIdx.x, lane = threadIdx.x;
    const long long N = p.total, C = p.n_cta;
    const long long first = (long long)b * p.vocab;
    const long long c_lo = cta_of(first, N, C), c_hi = cta_of(first + p.vocab - 1, N, C);
    unsigned long long best = 0ull;
    for (long long c = c_lo + lane; c <= c_hi; c += 32) {
        const unsigned long long w = p.part[(long long)b + c];
        best = w > best ? w : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) p.argmax[b] = (int32_t)unpack_index(best);
}

// The one-launch form: grid (k, batch), clusters of the k CTAs of a row (k <= 16); CTA x scans
// elements [ceil(x V / k), ceil((x + 1) V / k)) of row blockIdx.y and sends its word to slot x
// of the cluster's first CTA, which reduces the k words after a cluster barrier.
template <typename T, bool CAPPED>
__global__ void __launch_bounds__(kLgThreads) logit_row_kernel(const LogitParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel on the stream has completed
    __shared__ unsigned long long s_best[kLgThreads / 32];
    __shared__ unsigned long long s_piece[16];
    const int k = (int)gridDim.x, x = (int)blockIdx.x, b = (int)blockIdx.y;
    const long long row = (long long)b * p.vocab;
    const int i0 = (int)(((long long)x * p.vocab + k - 1) / k);
    const int i1 = (int)(((long long)(x + 1) * p.vocab + k - 1) / k);
    const unsigned long long best = cta_max(scan_range<T, CAPPED>(p, row, i0, i1), s_best);
    if (threadIdx.x == 0) {
        uint32_t dst;  // slot x of the first CTA's array (blockIdx.x is the rank in the cluster)
        asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(dst) : "r"(smem_u32(&s_piece[x])));
        asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(dst), "l"(best) : "memory");
    }
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
    if (x == 0 && threadIdx.x < 32) {
        unsigned long long w = (int)threadIdx.x < k ? s_piece[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, w, o);
            w = other > w ? other : w;
        }
        if (threadIdx.x == 0) p.argmax[b] = (int32_t)unpack_index(w);
    }
}

// resident CTAs per SM of the split kernel (the smallest over its instantiations), per device
static int logit_ctas_per_sm() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int m = 1 << 30, n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, logit_split_kernel<float, true>, kLgThreads, 0) == cudaSuccess) m = min(m, n);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, logit_split_kernel<float, false>, kLgThreads, 0) == cudaSuccess) m = min(m, n);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, logit_split_kernel<__nv_bfloat16, true>, kLgThreads, 0) == cudaSuccess) m = min(m, n);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, logit_split_kernel<__nv_bfloat16, false>, kLgThreads, 0) == cudaSuccess) m = min(m, n);
    if (m == (1 << 30) || m < 1) m = 1;
    if (dev >= 0 && dev < 64) cache[dev] = m;
    return m;
}

LogitPlan logit_plan(int batch, int vocab, int n_sm) {
    LogitPlan pl{1, 0, 0};
    if (batch < 1 || vocab < 1) return pl;
    const long long N = (long long)batch * vocab;
    long long c = (long long)n_sm * logit_ctas_per_sm();
    const long long by_size = (N + kLgMinChunk - 1) / kLgMinChunk;
    if (c > by_size) c = by_size;
    if (c < 1) c = 1;
    // rows of their own CTAs (a cluster of at most 16 per row) while that keeps at least half
    // the wave's CTAs busy
    long long k = c / batch;
    if (k < 1) k = 1;
    if (k > kLgMaxRowCtas) k = kLgMaxRowCtas;
    if (batch <= 65535 && 2 * k * batch >= c) {
        pl.n_cta = (int)(k * batch);
        pl.row_ctas = (int)k;
        return pl;
    }
    pl.n_cta = (int)c;
    pl.ws_bytes = (size_t)(batch + c) * sizeof(unsigned long long);
    return pl;
}

cudaError_t launch_logit_softcap_argmax(const void* logits, void* capped, int32_t* argmax,
                                        void* workspace, int batch, int vocab, int fp32,
                                        float softcap, const LogitPlan& pl, cudaStream_t st) {
    LogitParams p;
    p.logits = logits;
    p.capped = capped;
    p.argmax = argmax;
    p.part = static_cast<unsigned long long*>(workspace);
    p.total = (long long)batch * vocab;
    p.vocab = vocab;
    p.n_cta = pl.n_cta;
    p.softcap = softcap;
    p.inv_cap = softcap > 0.f ? 1.f / softcap : 0.f;
    cudaError_t e;
    if (pl.row_ctas > 0) {
        auto kernel = fp32 ? (capped ? logit_row_kernel<float, true> : logit_row_kernel<float, false>)
                           : (capped ? logit_row_kernel<__nv_bfloat16, true>
                                     : logit_row_kernel<__nv_bfloat16, false>);
        if (pl.row_ctas > 8) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)pl.row_ctas, (unsigned)batch);
        cfg.blockDim = dim3(kLgThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)pl.row_ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kernel, p);
    }
    const dim3 grid(pl.n_cta), block(kLgThreads);
    if (fp32)
        e = capped ? launch_pdl(logit_split_kernel<float, true>, grid, block, 0, st, p)
                   : launch_pdl(logit_split_kernel<float, false>, grid, block, 0, st, p);
    else
        e = capped ? launch_pdl(logit_split_kernel<__nv_bfloat16, true>, grid, block, 0, st, p)
                   : launch_pdl(logit_split_kernel<__nv_bfloat16, false>, grid, block, 0, st, p);
    if (e == cudaSuccess) e = launch_pdl(logit_finish_kernel, dim3(batch), dim3(32), 0, st, p);
    return e;
}

}  // namespace gemma
