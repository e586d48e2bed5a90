// decode_static.cu -- flash-decoding without a caller-supplied workspace.
//
// attn_decode_splitkv needs a scratch buffer for the per-segment partial
// results, and it expects the caller to allocate it.  Some callers cannot do
// that: code that runs where every byte of device memory is owned by a host
// framework's allocator and raw cudaMalloc is not permitted, code whose
// memory budget is fully planned ahead of time, and latency-critical paths
// that must not call cudaMalloc/cudaFree because those calls can block or
// synchronise the device.  For them this file provides
// attn_decode_splitkv_static, which runs the same split-KV kernel and merge
// kernel on a fixed scratch area that lives in the library itself.
//
// The scratch area is a file-scope __device__ array of
// ATTN_DECODE_STATIC_SCRATCH_BYTES.  Every GPU on which the library is loaded
// holds it for the life of the process.  Host code cannot use the array's
// name as a device address, so the first call on each device asks the CUDA
// runtime for the address (cudaGetSymbolAddress, with that device current)
// and caches it.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once
// per device.  Returns nullptr if the runtime cannot provide it.
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" attn_status_t attn_decode_splitkv_static(const void* q, const void* k_cache,
                                                    const void* v_cache, void* o, float* lse,
                                                    int B, int Hq, int Hkv, int Nk, int d,
                                                    float scale, int num_splits,
                                                    attn_dtype_t dtype, void* stream) {
    // Resolve the segment count first so that the scratch need is known; the
    // full argument checks are those of attn_decode_splitkv, called below.
    int S = num_splits;
    if (S == 0 && B > 0 && Hq > 0 && Hkv > 0 && Nk > 0 && Hq % Hkv == 0 && (d == 64 || d == 128))
        S = attn_host::decode_auto_splits(B, Hq, Hkv, Nk, d);
    size_t need = 0;
    if (S > 1 && B > 0 && Hq > 0 && (d == 64 || d == 128))
        need = attn_host::decode_workspace_bytes(B, Hq, d, S);
    if (need > (size_t)ATTN_DECODE_STATIC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_for_current_device();
        if (scratch == nullptr) return ATTN_ERR_CUDA;
    }
    return attn_decode_splitkv(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale,
                               S > 0 ? S : num_splits, scratch, need, dtype, stream);
}
