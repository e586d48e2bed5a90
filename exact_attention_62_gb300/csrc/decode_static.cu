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
// and caches it together with the unique ID of the device's current context.
// A device reset or a primary-context teardown creates a new context, in
// which the module is loaded again and the array may sit elsewhere; the ID
// then differs and the address is looked up again.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_STATIC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_scratch_mutex;
void* g_scratch_addr[attn_host::kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[attn_host::kMaxDevices] = {0};

// Unique ID of the calling thread's current context (0 if it cannot be read).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_decode_scratch on the current device, looked up on the
// first call in each context (cudaGetSymbolAddress also initialises the
// device's primary context when no call has done so yet).  Returns nullptr if
// the runtime cannot provide it.
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= attn_host::kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long ctx = current_context_id();
    if (ctx != 0 && g_scratch_addr[dev] != nullptr && g_scratch_ctx[dev] == ctx) return g_scratch_addr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    // With no readable context ID (0) nothing is reused: the next call looks
    // the address up again.
    ctx = current_context_id();
    g_scratch_addr[dev] = ctx != 0 ? p : nullptr;
    g_scratch_ctx[dev] = ctx;
    return p;
}

}  // namespace

extern "C" attn_status_t attn_decode_splitkv_static(const void* q, const void* k_cache,
                                                    const void* v_cache, void* o, float* lse,
                                                    int B, int Hq, int Hkv, int Nk, int d,
                                                    float scale, int num_splits,
                                                    attn_dtype_t dtype, void* stream) {
    // The argument checks of attn_decode_splitkv come first, so that an
    // invalid call is reported as such whatever scratch it would need.
    int S = 0;
    bool empty = false;
    const attn_status_t st = attn_host::check_decode_args(q, k_cache, v_cache, o, lse, B, Hq, Hkv,
                                                          Nk, d, scale, num_splits, dtype, &S, &empty);
    if (st != ATTN_OK) return st;
    if (empty)
        return attn_decode_splitkv(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale, num_splits,
                                   nullptr, 0, dtype, stream);
    const size_t need = attn_host::decode_workspace_bytes(B, Hq, d, S);
    if (need > (size_t)ATTN_DECODE_STATIC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_for_current_device();
        if (scratch == nullptr) return ATTN_ERR_CUDA;
    }
    return attn_decode_splitkv(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale, S, scratch,
                               need, dtype, stream);
}
