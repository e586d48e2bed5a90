// api.cu -- the extern "C" entry points of libattn.so (declared and
// documented in include/attn.h, and the test-only ones in
// include/attn_test.h): argument checks, TMA tensor-map encoding and
// dispatch to the kernels.  Nothing here allocates device memory,
// synchronises a stream (except the two explicitly synchronous status
// readers) or keeps state between calls.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

bool bad_scale(float s) { return !std::isfinite(s) || !(s > 0.f); }

__global__ void fill_empty_kernel(void* o, float* lse, long long o_elems, long long n_lse,
                                  bool out_bf16) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < o_elems; i += stride) {
        if (out_bf16)
            static_cast<__nv_bfloat16*>(o)[i] = __float2bfloat16_rn(0.f);
        else
            static_cast<float*>(o)[i] = 0.f;
    }
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_lse; i += stride)
        lse[i] = -INFINITY;
}

}  // namespace

namespace attn_host {

bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows,
                     int elem_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t e = static_cast<cuuint64_t>(elem_bytes);
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * e, (cuuint64_t)H * d * e, (cuuint64_t)N * H * d * e};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elem_bytes), 1u, (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapDataType dt = elem_bytes == 2   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_vt_map(CUtensorMap* map, const void* base, int B, int H, int d, long long ld, int box_keys) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {(cuuint64_t)ld, (cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)ld, (cuuint64_t)d * ld, (cuuint64_t)H * d * ld};
    cuuint32_t box[4] = {(cuuint32_t)box_keys, (cuuint32_t)d, 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_page_heads_map(CUtensorMap* map, const void* pages, int num_pages, int page_size, int H, int d) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    // The pool is [pages][page_size][H][d]; the map lists its dimensions as
    // (d, key, head, page), so a box of a whole page lands in shared memory
    // head by head, each head's keys in consecutive 128-byte rows.
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)page_size, (cuuint64_t)H, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)H * d * 2, (cuuint64_t)d * 2, (cuuint64_t)page_size * H * d * 2};
    cuuint32_t box[4] = {64u, (cuuint32_t)page_size, (cuuint32_t)H, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pages), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
    static PerDevice<int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int n = 0;
    const bool ok = cache.get(dev, &n, [&](int* out) {
        return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && *out > 0;
    });
    return ok ? n : 0;
}

attn_status_t check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                                const void* o, const float* lse, int B, int Hq, int Hkv, int Nk,
                                int d, float scale, int num_splits, attn_dtype_t dtype, int* S,
                                bool* empty) {
    *S = 0;
    *empty = false;
    if (B < 0 || Hq < 0 || Hkv < 1 || Nk < 0 || d < 1 || num_splits < 0) return ATTN_ERR_INVALID;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0) {
        *empty = true;
        return ATTN_OK;
    }
    if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(q, 16) || misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    if (Nk == 0) {
        *empty = true;
        return ATTN_OK;
    }
    if (k_cache == nullptr || v_cache == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(k_cache, 16) || misaligned(v_cache, 16)) return ATTN_ERR_INVALID;
    if (num_splits > Nk) return ATTN_ERR_INVALID;
    int s = num_splits;
    if (s == 0) s = decode_auto_splits(B, Hq, Hkv, Nk, d);
    if (s < 1) return ATTN_ERR_CUDA;
    if (s > 65535) return ATTN_ERR_UNSUPPORTED;
    *S = s;
    return ATTN_OK;
}

attn_status_t launch_fill_empty(void* o, float* lse, long long rows_o, int d, long long n_lse,
                                bool out_bf16, cudaStream_t stream) {
    const long long o_elems = rows_o * d;
    const long long work = o_elems > n_lse ? o_elems : n_lse;
    long long blocks = (work + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    fill_empty_kernel<<<(unsigned)blocks, 256, 0, stream>>>(o, lse, o_elems, n_lse, out_bf16);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                       attn_dtype_t dtype, void* stream) {
    if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || Hkv < 1 || d < 1) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || Nq == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (Nk > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID;
    if (misaligned(q, 16) || misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    if (Nk > 0 && (misaligned(k, 16) || misaligned(v, 16))) return ATTN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf16 = dtype == ATTN_BF16;
    if (Nk == 0)
        return attn_host::launch_fill_empty(o, lse, (long long)B * Nq * Hq, d,
                                            (long long)B * Hq * Nq, bf16, st);
    if (bf16)
        return attn_host::launch_fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, st);
    return attn_host::launch_fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                     static_cast<const float*>(v), static_cast<float*>(o), lse, B,
                                     Hq, Hkv, Nq, Nk, d, causal, scale, st);
}

attn_status_t attn_fwd_test(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                            const attn_test_options_t* opt, void* stream) {
    if (opt == nullptr || opt->wait_limit_cycles < 0 || opt->o_extent_slack < 0 ||
        !(opt->rescale_threshold >= 0.f) || !(opt->rescale_threshold <= 8.f))
        return ATTN_ERR_INVALID;
    if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || Hkv < 1 || d < 1) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || Nq == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (Nk > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID;
    if (misaligned(q, 16) || misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    if (Nk > 0 && (misaligned(k, 16) || misaligned(v, 16))) return ATTN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Nk == 0)
        return attn_host::launch_fill_empty(o, lse, (long long)B * Nq * Hq, d,
                                            (long long)B * Hq * Nq, true, st);
    return attn_host::launch_fwd_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, st, opt);
}

double attn_decode_model_time(int units, int slots, int Nk, int d, int num_splits,
                              double cta_bytes_per_s, double hbm_bytes_per_s, double cta_fixed_s,
                              double merge_fixed_s) {
    if (units < 1 || slots < 1 || Nk < 1 || d < 1 || num_splits < 1 || !(cta_bytes_per_s > 0.0) ||
        !(hbm_bytes_per_s > 0.0) || !(cta_fixed_s >= 0.0) || !(merge_fixed_s >= 0.0))
        return -1.0;
    const attn_host::SplitModel m = {cta_bytes_per_s, hbm_bytes_per_s, cta_fixed_s, merge_fixed_s};
    return attn_host::split_model_time(units, slots, Nk, d, num_splits, m);
}

int attn_decode_model_best(int units, int slots, int Nk, int d, double cta_bytes_per_s,
                           double hbm_bytes_per_s, double cta_fixed_s, double merge_fixed_s,
                           int single_wave) {
    if (units < 1 || slots < 1 || Nk < 1 || d < 1 || !(cta_bytes_per_s > 0.0) ||
        !(hbm_bytes_per_s > 0.0) || !(cta_fixed_s >= 0.0) || !(merge_fixed_s >= 0.0))
        return -1;
    const attn_host::SplitModel m = {cta_bytes_per_s, hbm_bytes_per_s, cta_fixed_s, merge_fixed_s};
    return attn_host::split_model_best(units, slots, Nk, d, m, single_wave != 0);
}

int attn_decode_num_splits(int B, int Hq, int Hkv, int Nk, int d) {
    return attn_host::decode_auto_splits(B, Hq, Hkv, Nk, d);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nk, int d, int num_splits) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nk < 1 || (d != 64 && d != 128) ||
        num_splits < 0 || num_splits > Nk)
        return 0;
    int S = num_splits;
    if (S == 0) S = attn_host::decode_auto_splits(B, Hq, Hkv, Nk, d);
    if (S < 1) return 0;
    return attn_host::decode_workspace_bytes(B, Hq, d, S);
}

// Runs the split-KV decode after the workspace check (shared by
// attn_decode_splitkv and attn_decode_test).
static attn_status_t decode_checked(const void* q, const void* k_cache, const void* v_cache,
                                    void* o, float* lse, int B, int Hq, int Hkv, int Nk, int d,
                                    float scale, int num_splits, void* workspace,
                                    size_t workspace_bytes, attn_dtype_t dtype, void* stream,
                                    const attn_test_options_t* test) {
    int S = 0;
    bool empty = false;
    const attn_status_t st = attn_host::check_decode_args(q, k_cache, v_cache, o, lse, B, Hq, Hkv,
                                                          Nk, d, scale, num_splits, dtype, &S, &empty);
    if (st != ATTN_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (empty)
        return (B == 0 || Hq == 0) ? ATTN_OK
                                   : attn_host::launch_fill_empty(o, lse, (long long)B * Hq, d,
                                                                  (long long)B * Hq, true, cs);
    if (S > 1) {
        if (workspace == nullptr || misaligned(workspace, 16)) return ATTN_ERR_INVALID;
        if (workspace_bytes < attn_host::decode_workspace_bytes(B, Hq, d, S))
            return ATTN_ERR_INVALID;
    }
    return attn_host::launch_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale, S,
                                    workspace, cs, test);
}

attn_status_t attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o,
                                  float* lse, int B, int Hq, int Hkv, int Nk, int d, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  attn_dtype_t dtype, void* stream) {
    return decode_checked(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale, num_splits,
                          workspace, workspace_bytes, dtype, stream, nullptr);
}

attn_status_t attn_decode_test(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, int B, int Hq, int Hkv, int Nk, int d, float scale,
                               int num_splits, void* workspace, size_t workspace_bytes,
                               const attn_test_options_t* opt, void* stream) {
    if (opt == nullptr || opt->wait_limit_cycles < 0 || opt->o_extent_slack < 0) return ATTN_ERR_INVALID;
    return decode_checked(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nk, d, scale, num_splits,
                          workspace, workspace_bytes, ATTN_BF16, stream, opt);
}

static bool paged_page_size_ok(int page_size) {
    return page_size == 16 || page_size == 32 || (page_size > 0 && page_size % 64 == 0);
}

int attn_decode_paged_num_splits(int B, int Hq, int Hkv, int d, int page_size, int max_seq_len) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_seq_len < 1 || (d != 64 && d != 128) ||
        !paged_page_size_ok(page_size))
        return -1;
    return attn_host::decode_paged_auto_splits(B, Hq, Hkv, max_seq_len, d, page_size);
}

attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                int B, int Hq, int Hkv, int d, int num_pages, int page_size,
                                int max_pages_per_seq, int max_seq_len, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                attn_dtype_t dtype, void* stream) {
    if (B < 0 || Hq < 0 || Hkv < 1 || d < 1 || num_pages < 0 || page_size < 1 ||
        max_pages_per_seq < 0 || max_seq_len < 0 || num_splits < 0)
        return ATTN_ERR_INVALID;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if ((long long)max_pages_per_seq * page_size < max_seq_len) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (!paged_page_size_ok(page_size)) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(q, 16) || misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (max_seq_len == 0)
        return attn_host::launch_fill_empty(o, lse, (long long)B * Hq, d, (long long)B * Hq, true,
                                            st);
    if (num_pages < 1 || k_pages == nullptr || v_pages == nullptr || block_table == nullptr ||
        seq_lens == nullptr)
        return ATTN_ERR_INVALID;
    if (misaligned(k_pages, 16) || misaligned(v_pages, 16) || misaligned(block_table, 4) ||
        misaligned(seq_lens, 4))
        return ATTN_ERR_INVALID;
    if (num_splits > max_seq_len) return ATTN_ERR_INVALID;
    int S = num_splits;
    if (S == 0) S = attn_host::decode_paged_auto_splits(B, Hq, Hkv, max_seq_len, d, page_size);
    if (S < 1) return ATTN_ERR_CUDA;
    if (S > 65535 || !attn_host::paged_splits_fit(max_seq_len, page_size, S))
        return ATTN_ERR_UNSUPPORTED;
    if (S > 1) {
        if (workspace == nullptr || misaligned(workspace, 16)) return ATTN_ERR_INVALID;
        if (workspace_bytes < attn_host::decode_workspace_bytes(B, Hq, d, S))
            return ATTN_ERR_INVALID;
    }
    return attn_host::launch_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, B,
                                          Hq, Hkv, d, num_pages, page_size, max_pages_per_seq,
                                          max_seq_len, scale, S, workspace, st);
}

attn_status_t attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int N, int H,
                                int d, void* stream) {
    if (B < 0 || N < 0 || H < 0 || d < 2 || d % 2 != 0) return ATTN_ERR_INVALID;
    if (B == 0 || N == 0 || H == 0) return ATTN_OK;
    if (x == nullptr || codes == nullptr || scales == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(x, 16) || misaligned(codes, 16) || misaligned(scales, 4)) return ATTN_ERR_INVALID;
    return attn_host::launch_quantize_fp8(x, codes, scales, B, N, H, d, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                                        int B, int N, int H, int d, void* stream) {
    if (B < 0 || N < 0 || H < 0 || d < 1) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || N == 0 || H == 0) return ATTN_OK;
    if (x == nullptr || signs == nullptr || codes == nullptr || scales == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(x, 16) || misaligned(signs, 16) || misaligned(codes, 16) || misaligned(scales, 4))
        return ATTN_ERR_INVALID;
    return attn_host::launch_quantize_fp8_rotated(x, signs, codes, scales, B, N, H, d,
                                                  static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v, const float* q_scales,
                           const float* k_scales, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                           int Nk, int d, int causal, float scale, void* stream) {
    if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || Nq == 0) return ATTN_OK;
    if (o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Nk == 0)
        return attn_host::launch_fill_empty(o, lse, (long long)B * Nq * Hq, d, (long long)B * Hq * Nq,
                                            true, st);
    if (q8 == nullptr || k8 == nullptr || v == nullptr || q_scales == nullptr || k_scales == nullptr)
        return ATTN_ERR_INVALID;
    if (misaligned(q8, 16) || misaligned(k8, 16) || misaligned(v, 16) || misaligned(q_scales, 4) ||
        misaligned(k_scales, 4))
        return ATTN_ERR_INVALID;
    return attn_host::launch_fwd_fp8(q8, k8, v, q_scales, k_scales, o, lse, B, Hq, Hkv, Nq, Nk, d,
                                     causal, scale, st);
}

attn_status_t attn_quantize_fp8_v(const void* v, void* vt8, float* scales, int B, int N, int H, int d,
                                  void* stream) {
    if (B < 0 || N < 0 || H < 0 || d < 1) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || N == 0 || H == 0) return ATTN_OK;
    if (v == nullptr || vt8 == nullptr || scales == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(v, 16) || misaligned(vt8, 16) || misaligned(scales, 4)) return ATTN_ERR_INVALID;
    return attn_host::launch_quantize_fp8_v(v, vt8, scales, B, N, H, d, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_fp8_pv(const void* q8, const void* k8, const void* vt8, const float* q_scales,
                              const float* k_scales, const float* v_scales, void* o, float* lse, int B,
                              int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                              void* stream) {
    if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || Nq == 0) return ATTN_OK;
    if (o == nullptr || lse == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(o, 16) || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Nk == 0)
        return attn_host::launch_fill_empty(o, lse, (long long)B * Nq * Hq, d, (long long)B * Hq * Nq,
                                            true, st);
    if (q8 == nullptr || k8 == nullptr || vt8 == nullptr || q_scales == nullptr || k_scales == nullptr ||
        v_scales == nullptr)
        return ATTN_ERR_INVALID;
    if (misaligned(q8, 16) || misaligned(k8, 16) || misaligned(vt8, 16) || misaligned(q_scales, 4) ||
        misaligned(k_scales, 4) || misaligned(v_scales, 4))
        return ATTN_ERR_INVALID;
    return attn_host::launch_fwd_fp8_pv(q8, k8, vt8, q_scales, k_scales, v_scales, o, lse, B, Hq, Hkv, Nq,
                                        Nk, d, causal, scale, st);
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Nq) {
    if (B < 0 || Hq < 0 || Nq < 0) return 0;
    return attn_host::bwd_workspace_bytes(B, Hq, Nq);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                       int Nq, int Nk, int d, int causal, float scale, void* workspace,
                       size_t workspace_bytes, attn_dtype_t dtype, void* stream) {
    if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1) return ATTN_ERR_INVALID;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (bad_scale(scale)) return ATTN_ERR_INVALID;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;
    if (Nq == 0 || Nk == 0) return ATTN_ERR_UNSUPPORTED;  // empty sides: nothing to differentiate
    const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (ptr == nullptr || misaligned(ptr, 16)) return ATTN_ERR_INVALID;
    if (lse == nullptr || misaligned(lse, 4)) return ATTN_ERR_INVALID;
    if (workspace == nullptr || misaligned(workspace, 16) ||
        workspace_bytes < attn_host::bwd_workspace_bytes(B, Hq, Nq))
        return ATTN_ERR_INVALID;
    return attn_host::launch_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, causal,
                                 scale, workspace, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_merge_lse(const float* o_parts, const float* lse_parts, int num_parts,
                             long long rows, int d, void* o, float* lse, attn_dtype_t out_dtype,
                             void* stream) {
    if (num_parts < 1 || rows < 0 || d < 4 || d > 512 || d % 4 != 0) return ATTN_ERR_INVALID;
    if (out_dtype != ATTN_BF16 && out_dtype != ATTN_F32) return ATTN_ERR_INVALID;
    if (rows == 0) return ATTN_OK;
    if (o_parts == nullptr || lse_parts == nullptr || o == nullptr) return ATTN_ERR_INVALID;
    if (misaligned(o_parts, 16) || misaligned(lse_parts, 4) || misaligned(o, 16) ||
        (lse != nullptr && misaligned(lse, 4)))
        return ATTN_ERR_INVALID;
    return attn_host::launch_merge(o_parts, lse_parts, num_parts, rows, d, o, lse,
                                   out_dtype == ATTN_BF16, static_cast<cudaStream_t>(stream));
}

const char* attn_status_string(attn_status_t status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
        case ATTN_ERR_BOUNDS: return "in-kernel bounds check refused an access";
    }
    return "unknown status";
}

attn_status_t attn_check_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned a = 0, b = 0, c = 0, f = 0, e = 0;
    if (attn_host::fwd_tc_read_status(&a, true) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_host::decode_read_status(&b, true) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_host::bwd_read_status(&c, true) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_host::fwd_f32_read_status(&f, true) != cudaSuccess) return ATTN_ERR_CUDA;
    if (attn_host::fp8_read_status(&e, true) != cudaSuccess) return ATTN_ERR_CUDA;
    const unsigned all = a | b | c | f | e;
    if (all & attn_dev::kStatusBounds) return ATTN_ERR_BOUNDS;
    return all ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

attn_status_t attn_read_tile_counter(unsigned long long* count, int reset) {
    if (count == nullptr) return ATTN_ERR_INVALID;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    return attn_host::fwd_tc_read_tiles(count, reset != 0) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

const char* attn_version(void) { return "exact_attention_gb300 0.1 sm_103a"; }

}  // extern "C"
