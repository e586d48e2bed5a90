// common.cuh -- host-side declarations shared by the translation units of
// libattn.so (launchers, status words, tensor-map helper).  Not part of the
// public ABI; the public ABI is include/attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn_host {

// Encodes a 4-D TMA tensor map over a row-major [B, N, H, d] tensor of
// `elem_bytes`-byte elements, with a box of (64 elements, 1 head, box_rows,
// 1 batch) and 128-byte swizzle.  Returns false if the driver rejects it.
bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d,
                     int box_rows, int elem_bytes);

// Number of SMs of the current device (cached per device); 0 on failure.
int device_sm_count();

// ---- bf16 tensor-core forward (fwd_tc.cu)
attn_status_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, cudaStream_t stream);
cudaError_t fwd_tc_read_status(unsigned* out, bool clear);
cudaError_t fwd_tc_read_tiles(unsigned long long* out, bool reset);

// ---- fp32 CUDA-core forward (fwd_f32.cu)
attn_status_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o,
                             float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                             int causal, float scale, cudaStream_t stream);

// ---- split-KV decode and LSE merge (decode.cu)
int decode_auto_splits(int B, int Hq, int Hkv, int Nk, int d);
size_t decode_workspace_bytes(int B, int Hq, int d, int splits);
attn_status_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nk, int d, float scale, int splits,
                            void* workspace, cudaStream_t stream);
attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int parts,
                           long long rows, int d, void* o, float* lse, bool out_bf16,
                           cudaStream_t stream);
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
