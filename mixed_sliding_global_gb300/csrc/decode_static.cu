// decode_static.cu -- decode entry point for callers that cannot allocate device memory.
//
// gemma_attn_decode needs scratch for its split-over-keys partial results, and asks the caller
// for it. Some callers have no way to provide it: code that runs where cudaMalloc is not
// allowed or not wanted (inside a custom allocator or a memory-pool callback, a plugin host
// that owns every device allocation, a real-time path that must not hit the driver's
// allocator). gemma_attn_decode_static takes its scratch from a fixed array compiled into
// this library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds
// kStaticScratchBytes of it until the process exits. Host code cannot use the array's name
// as a device address: a call looks the address up with cudaGetSymbolAddress (with the
// device current) the first time it runs in a CUDA context and caches it with that context's
// unique id, so a device reset (which creates a new context) makes the next call look it up
// again; make the first call in each context before any stream capture. All calls share the
// one array and it keeps the previous call's contents; the decode kernels write every partial
// result before reading it, so nothing has to start at zero, but two calls whose kernels
// overlap on the GPU (different streams, or graphs replayed concurrently) race on the array
// and must be serialised by the caller.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/gemma_attn.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id;  // unique id of the context the address belongs to
    void* ptr;
};
Cached g_cache[kMaxDevices];
std::mutex g_cache_mutex;

// The current context's unique id, through the driver entry points the runtime hands out (the
// library does not link libcuda).
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            return false;
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context (looked up once per context).
int static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMMA_ERR_CUDA;
    unsigned long long id = 0;
    // false while no context is current yet (the lookup below makes the primary one current)
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    Cached& c = g_cache[dev];
    if (!have_id || !c.ptr || c.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return GEMMA_ERR_CUDA;
        if (!current_context_id(&id)) return GEMMA_ERR_CUDA;
        c.ptr = p;
        c.ctx_id = id;
    }
    *out = c.ptr;
    return GEMMA_OK;
}

}  // namespace

extern "C" int gemma_attn_decode_static(void* out, const void* q, const void* const* k_cache,
                                        const void* const* v_cache, const int32_t* owner_map,
                                        int n_layers, int layer, const int32_t* seq_lens,
                                        int max_seq_len, int batch, gemma_layer_kind kind,
                                        int window, int n_q, int n_kv, int head_dim, int k_eq_v,
                                        int kv_capacity, float scale, gemma_dtype dtype,
                                        uint32_t* device_error, void* stream) {
    const size_t need = gemma_attn_workspace_size(batch, kind, window, n_q, n_kv, head_dim,
                                                  max_seq_len, 1);
    if (need == (size_t)-1 || need > kStaticScratchBytes) {
        // No usable plan: gemma_attn_decode without a workspace runs every argument check in
        // its own order and returns the status it would return (GEMMA_ERR_WORKSPACE when the
        // arguments are valid but the plan needs more scratch than the built-in array), with
        // no launch.
        return gemma_attn_decode(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens,
                                 max_seq_len, batch, kind, window, n_q, n_kv, head_dim, k_eq_v,
                                 kv_capacity, scale, dtype, nullptr, 0, device_error, stream);
    }
    void* scratch = nullptr;
    if (need > 0) {
        const int st = static_scratch(&scratch);
        if (st != GEMMA_OK) return st;
    }
    return gemma_attn_decode(out, q, k_cache, v_cache, owner_map, n_layers, layer, seq_lens,
                             max_seq_len, batch, kind, window, n_q, n_kv, head_dim, k_eq_v,
                             kv_capacity, scale, dtype, scratch, need > 0 ? kStaticScratchBytes : 0,
                             device_error, stream);
}
