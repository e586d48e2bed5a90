// fp8.cu -- block quantisation of bf16 [B, N, H, d] tensors to e4m3 for the
// FP8 forward (the block quantisation of Lecture 11 - Kernel Optimization
// Techniques, section 4.5, FP8 item).
//
// One CTA per (row block of 128, head, batch): amax = max |x| over the
// block's 128 rows x d columns; scale = amax / 448 and inv = 448 / amax in
// fp32 (IEEE division; 1 and 1 for an all-zero block); each element becomes
// e4m3(x * inv), rounded to nearest even and saturated to +-448.  Every step
// is an IEEE-defined operation, so the codes are reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace {

constexpr int kBlockRows = 128;
constexpr int kQThreads = 256;
constexpr float kFp8Max = 448.0f;

__global__ void __launch_bounds__(kQThreads)
    quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                        float* __restrict__ scales, int N, int H, int d) {
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nb = gridDim.x;
    const int r0 = blk * kBlockRows;
    const int rows = min(kBlockRows, N - r0);
    const int pairs = rows * (d / 2);  // element pairs of the block
    auto pair_offset = [&](int e) -> long long {
        const int r = e / (d / 2), c = 2 * (e % (d / 2));
        return (((long long)b * N + r0 + r) * H + h) * d + c;
    };
    float amax = 0.f;
    for (int e = threadIdx.x; e < pairs; e += kQThreads) {
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + pair_offset(e)));
        amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
    __shared__ float red[kQThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const bool nz = amax > 0.f;
    const float inv = nz ? kFp8Max / amax : 1.f;
    if (threadIdx.x == 0) scales[((long long)b * H + h) * nb + blk] = nz ? amax / kFp8Max : 1.f;
    for (int e = threadIdx.x; e < pairs; e += kQThreads) {
        const long long o = pair_offset(e);
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + o));
        const float2 y = make_float2(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv));
        const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
        *reinterpret_cast<__nv_fp8x2_storage_t*>(codes + o) = q;
    }
}

}  // namespace

namespace attn_host {

attn_status_t launch_quantize_fp8(const void* x, void* codes, float* scales, int B, int N, int H, int d,
                                  cudaStream_t stream) {
    const int nb = (N + kBlockRows - 1) / kBlockRows;
    if (nb > 0x7fffffff || H > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;
    dim3 grid(nb, H, B);
    quantize_fp8_kernel<<<grid, kQThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                        static_cast<uint8_t*>(codes), scales, N, H, d);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn_host
