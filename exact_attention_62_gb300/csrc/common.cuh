// common.cuh -- host-side declarations shared by the translation units of
// libattn.so (launchers, status words, tensor-map helper).  Not part of the
// public ABI; that is include/attn.h (and include/attn_test.h for tests).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "per_device.h"
#include "../../include/attn_test.h"

namespace attn_host {

// One-time launch set-up of a kernel, per device.  The dynamic shared-memory
// limit that cudaFuncSetAttribute sets belongs to the current device, and the
// register count is read for the device that will run the kernel, so a
// process that drives several GPUs (even from one thread) needs both for
// each device: a PerDevice cache (per_device.h), in which a failed set-up is
// not kept (the next call retries).
struct KernelSetup {
    cudaError_t err;
    int num_regs;
};

template <auto Kernel>
KernelSetup kernel_setup(int dyn_smem_bytes) {
    static PerDevice<int> regs;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return {cudaErrorInvalidDevice, 0};
    cudaError_t err = cudaSuccess;
    int n = 0;
    const bool ok = regs.get(dev, &n, [&](int* out) {
        if (dyn_smem_bytes > 0) {
            err = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem_bytes);
            if (err != cudaSuccess) return false;
        }
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, Kernel);
        if (err != cudaSuccess) return false;
        *out = fa.numRegs;
        return true;
    });
    if (!ok) return {err != cudaSuccess ? err : cudaErrorInvalidDevice, 0};
    return {cudaSuccess, n};
}

// Encodes a 4-D TMA tensor map over a row-major [B, N, H, d] tensor of
// `elem_bytes`-byte elements, with a box of (64 elements, 1 head, box_rows,
// 1 batch) and 128-byte swizzle.  Returns false if the driver rejects it.
bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d,
                     int box_rows, int elem_bytes);

// Row length (keys, padded) of the transposed e4m3 V, [B, H, d, ld]: a
// multiple of 16 so that every row starts on a 16-byte boundary.
inline long long fp8_v_ld(int N) { return ((long long)N + 15) / 16 * 16; }

// Encodes a 4-D TMA tensor map over the transposed e4m3 V [B, H, d, ld]
// (keys innermost), with a box of (box_keys keys, all d rows, 1 head, 1
// batch) and 128-byte swizzle: a K-major operand tile of d rows.
bool encode_vt_map(CUtensorMap* map, const void* base, int B, int H, int d, long long ld, int box_keys);
// Paged K or V pool [pages][page_size][H][d] (bf16) as whole-page boxes of
// all H heads: 64 columns x page_size keys x H heads, 128-byte swizzle, rows
// ordered head by head.
bool encode_page_heads_map(CUtensorMap* map, const void* pages, int num_pages, int page_size, int H, int d);

// Number of SMs of the current device (cached per device); 0 on failure.
int device_sm_count();

// The argument checks of attn_decode_splitkv (everything but the workspace),
// shared by the entry points that run the split-KV decode.  On success *S is
// the segment count to use (num_splits, or the automatic count for 0) and
// *empty is set when there is nothing to stream (B, Hq or Nk is 0).
attn_status_t check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                                const void* o, const float* lse, int B, int Hq, int Hkv, int Nk,
                                int d, float scale, int num_splits, attn_dtype_t dtype, int* S,
                                bool* empty);

// ---- bf16 tensor-core forward (fwd_tc.cu).  `test` is NULL on the
// production path; attn_fwd_test passes its options.  lse_ld is the number
// of floats between the LSE rows of consecutive heads (0: Nq, the layout of
// a whole call; a call over a block of rows of a longer sequence passes that
// sequence's length).
attn_status_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, cudaStream_t stream,
                            const attn_test_options_t* test = nullptr, long long lse_ld = 0);
cudaError_t fwd_tc_read_status(unsigned* out, bool clear);
cudaError_t fwd_f32_read_status(unsigned* out, bool clear);
cudaError_t fp8_read_status(unsigned* out, bool clear);
cudaError_t fwd_tc_read_tiles(unsigned long long* out, bool reset);

// ---- fp32 CUDA-core forward (fwd_f32.cu)
attn_status_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o,
                             float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                             int causal, float scale, cudaStream_t stream);

// ---- split-KV decode and LSE merge (decode.cu)
// The segment-count model (Lecture 11, sections 6.3-6.4), as pure host
// arithmetic: see decode.cu.
struct SplitModel {
    double cta_bw;       // bytes/s one CTA streams with its ring full
    double hbm;          // bytes/s the whole GPU streams
    double cta_fixed;    // start-up of one CTA wave, s
    double merge_fixed;  // the merge launch, s
};
double split_model_time(long long units, long long slots, int Nk, int d, int S, const SplitModel& m);
int split_model_best(long long units, long long slots, int Nk, int d, const SplitModel& m, bool single_wave);
int decode_auto_splits(int B, int Hq, int Hkv, int Nk, int d);
size_t decode_workspace_bytes(int B, int Hq, int d, int splits);
attn_status_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nk, int d, float scale, int splits,
                            void* workspace, cudaStream_t stream,
                            const attn_test_options_t* test = nullptr);
attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int parts,
                           long long rows, int d, void* o, float* lse, bool out_bf16,
                           cudaStream_t stream, long long o_slack = 0);
cudaError_t decode_read_status(unsigned* out, bool clear);
bool paged_splits_fit(int max_seq_len, int page_size, int splits);
int decode_paged_auto_splits(int B, int Hq, int Hkv, int max_seq_len, int d, int page_size);
attn_status_t launch_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                  const int* block_table, const int* seq_lens, void* o, float* lse,
                                  int B, int Hq, int Hkv, int d, int num_pages, int page_size,
                                  int max_pages, int max_seq_len, float scale, int splits,
                                  void* workspace, cudaStream_t stream);

// ---- FP8 block quantisation (fp8.cu) and FP8 forward (fwd_tc.cu)
attn_status_t launch_quantize_fp8(const void* x, void* codes, float* scales, int B, int N, int H, int d,
                                  cudaStream_t stream);
attn_status_t launch_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                                          int B, int N, int H, int d, cudaStream_t stream);
attn_status_t launch_fwd_fp8(const void* q8, const void* k8, const void* v, const float* q_scales,
                             const float* k_scales, void* o, float* lse, int B, int Hq, int Hkv,
                             int Nq, int Nk, int d, int causal, float scale, cudaStream_t stream);
attn_status_t launch_quantize_fp8_v(const void* v, void* vt8, float* scales, int B, int N, int H, int d,
                                    cudaStream_t stream);
attn_status_t launch_fwd_fp8_pv(const void* q8, const void* k8, const void* vt8, const float* q_scales,
                                const float* k_scales, const float* v_scales, void* o, float* lse, int B,
                                int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                                cudaStream_t stream);

// ---- backward pass (bwd_tc.cu)
size_t bwd_workspace_bytes(int B, int Hq, int Nq);
attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                         int Nq, int Nk, int d, int causal, float scale, void* workspace,
                         cudaStream_t stream);
cudaError_t bwd_read_status(unsigned* out, bool clear);

// ---- small utility kernels (api.cu)
attn_status_t launch_fill_empty(void* o, float* lse, long long rows_o, int d, long long n_lse,
                                bool out_bf16, cudaStream_t stream);

}  // namespace attn_host
