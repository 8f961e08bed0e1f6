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
// as a device address: the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; make that first call before
// any stream capture. All calls share the one array and it keeps the previous call's
// contents; the decode kernels write every partial result before reading it, so nothing has
// to start at zero, but two calls whose kernels overlap on the GPU (different streams, or
// graphs replayed concurrently) race on the array and must be serialised by the caller.
#include <atomic>

#include "../../include/gemma_attn.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
int static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMMA_ERR_CUDA;
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return GEMMA_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
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
    // same argument checks as gemma_attn_decode (it runs them again); the size check is here
    const size_t need = gemma_attn_workspace_size(batch, kind, window, n_q, n_kv, head_dim,
                                                  max_seq_len, 1);
    if (need == (size_t)-1) return GEMMA_ERR_INVALID_ARG;
    if (need > kStaticScratchBytes) return GEMMA_ERR_WORKSPACE;  // beyond the built-in scratch
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

