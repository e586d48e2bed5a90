// fp8.cu -- block quantisation of bf16 [B, N, H, d] tensors to e4m3 for the
// FP8 forward (the block quantisation of Lecture 11 - Kernel Optimization
// Techniques, section 4.5, FP8 item), optionally after a random orthogonal
// transform of each row (the same item's incoherent processing).
//
// One CTA per (row block of 128, head, batch): amax = max |x| over the
// block's 128 rows x d columns; scale = amax / 448 and inv = 448 / amax in
// fp32 (IEEE division; 1 and 1 for an all-zero block); each element becomes
// e4m3(x * inv), rounded to nearest even and saturated to +-448.  Every step
// is an IEEE-defined operation, so the codes are reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

// Status word of the quantisers: only the bounds-checked build sets it.
__device__ unsigned g_fp8_status = 0;

constexpr int kBlockRows = 128;
constexpr int kQThreads = 256;
constexpr float kFp8Max = 448.0f;

// Maximum of `v` over the CTA (every thread gets it).
__device__ __forceinline__ float block_max(float v) {
    __shared__ float red[kQThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) v = fmaxf(v, red[i]);
    return v;
}

// d = 64 or 128: the block is read once, with 16-byte loads (D / 8 threads
// per row), and held in registers while its amax is reduced; each thread
// then writes 8 codes per chunk.  Same arithmetic as the general kernel.
template <int D>
__global__ void __launch_bounds__(kQThreads)
    quantize_fp8_regs_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                             float* __restrict__ scales, int N, int H) {
    constexpr int kC = D / 8;                             // 16-byte chunks per row
    constexpr int kK = kBlockRows * kC / kQThreads;       // chunks per thread
    static_assert(kBlockRows * kC % kQThreads == 0, "chunk split");
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nb = gridDim.x;
    const int r0 = blk * kBlockRows;
    const int rows = min(kBlockRows, N - r0);
    uint4 v[kK];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int i = threadIdx.x + k * kQThreads;
        const int r = i / kC, c = i % kC;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8, (long long)gridDim.z * N * H * D,
                                  &g_fp8_status))
            v[k] = __ldg(reinterpret_cast<const uint4*>(x + (((long long)b * N + r0 + r) * H + h) * D) + c);
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e[t]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    amax = block_max(amax);
    const bool nz = amax > 0.f;
    const float inv = nz ? kFp8Max / amax : 1.f;
    if (threadIdx.x == 0 && in_bounds(((long long)b * H + h) * nb + blk, 1, (long long)gridDim.z * H * nb, &g_fp8_status))
        scales[((long long)b * H + h) * nb + blk] = nz ? amax / kFp8Max : 1.f;
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int i = threadIdx.x + k * kQThreads;
        const int r = i / kC, c = i % kC;
        if (r >= rows) continue;
        if (!in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8, (long long)gridDim.z * N * H * D,
                       &g_fp8_status))
            continue;
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
        uint32_t w[2];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e[t]);
            const float2 y = make_float2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
            const uint32_t q = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
            if (t & 1)
                w[t >> 1] |= q << 16;
            else
                w[t >> 1] = q;
        }
        *reinterpret_cast<uint2*>(codes + (((long long)b * N + r0 + r) * H + h) * D + 8 * c) =
            make_uint2(w[0], w[1]);
    }
}

// Rotated variant ("incoherent processing"), d = 64 or 128: each row is
// multiplied by diag(signs) and the d x d Sylvester Hadamard matrix before
// the block quantisation.  A thread holds 8 consecutive elements of a row
// (kC = D / 8 threads per row, consecutive lanes, so every load instruction
// reads whole rows), the butterflies with h = 1, 2, 4 stay in registers and
// h = 8 .. D/2 pair lane c with lane c ^ (h / 8) of the same row.  Every
// butterfly is one fp32 add and one fp32 subtract, (a, b) -> (a + b, a - b),
// taken stage by stage in increasing h, so the result is reproducible bit for
// bit.  The block scale is multiplied by c_norm = 1 / sqrt(d) at the end,
// which makes the transform orthogonal.  (Two threads per row, with only the
// last stage across lanes, was measured slower: its loads no longer read
// whole rows per instruction.)
template <int D>
__global__ void __launch_bounds__(kQThreads)
    quantize_fp8_rot_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ signs,
                            uint8_t* __restrict__ codes, float* __restrict__ scales, int N, int H,
                            float c_norm) {
    constexpr int kC = D / 8;                             // threads (16-byte chunks) per row
    constexpr int kK = kBlockRows * kC / kQThreads;       // chunks per thread
    static_assert(kBlockRows * kC % kQThreads == 0 && kQThreads % kC == 0 && 32 % kC == 0, "chunk split");
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nb = gridDim.x;
    const int r0 = blk * kBlockRows;
    const int rows = min(kBlockRows, N - r0);
    const int c = threadIdx.x % kC;  // the chunk of its rows this thread holds (the same for every k)
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(signs) + 2 * c);
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(signs) + 2 * c + 1);
    const float sg[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float y[kK][8];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int r = (threadIdx.x + k * kQThreads) / kC;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows && in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8, (long long)gridDim.z * N * H * D,
                                  &g_fp8_status))
            raw = __ldg(reinterpret_cast<const uint4*>(x + (((long long)b * N + r0 + r) * H + h) * D) + c);
        const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e2[t]);
            y[k][2 * t] = f.x * sg[2 * t];
            y[k][2 * t + 1] = f.y * sg[2 * t + 1];
        }
#pragma unroll
        for (int hh = 1; hh < 8; hh <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if ((e & hh) == 0) {
                    const float a = y[k][e], bb = y[k][e + hh];
                    y[k][e] = __fadd_rn(a, bb);
                    y[k][e + hh] = __fsub_rn(a, bb);
                }
            }
        }
#pragma unroll
        for (int m = 1; m < kC; m <<= 1) {
            const bool upper = (c & m) != 0;  // this lane holds the b of each pair
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, y[k][e], m);
                y[k][e] = upper ? __fsub_rn(o, y[k][e]) : __fadd_rn(y[k][e], o);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[k][e]));
    }
    amax = block_max(amax);
    const bool nz = amax > 0.f;
    const float inv = nz ? kFp8Max / amax : 1.f;
    if (threadIdx.x == 0 && in_bounds(((long long)b * H + h) * nb + blk, 1, (long long)gridDim.z * H * nb, &g_fp8_status))
        scales[((long long)b * H + h) * nb + blk] = __fmul_rn(nz ? amax / kFp8Max : 1.f, c_norm);
#pragma unroll
    for (int k = 0; k < kK; ++k) {
        const int r = (threadIdx.x + k * kQThreads) / kC;
        if (r >= rows) continue;
        if (!in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8, (long long)gridDim.z * N * H * D,
                       &g_fp8_status))
            continue;
        uint32_t w[2];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 q2 = make_float2(__fmul_rn(y[k][2 * t], inv), __fmul_rn(y[k][2 * t + 1], inv));
            const uint32_t q = __nv_cvt_float2_to_fp8x2(q2, __NV_SATFINITE, __NV_E4M3);
            if (t & 1)
                w[t >> 1] |= q << 16;
            else
                w[t >> 1] = q;
        }
        *reinterpret_cast<uint2*>(codes + (((long long)b * N + r0 + r) * H + h) * D + 8 * c) =
            make_uint2(w[0], w[1]);
    }
}

// ---- V for the e4m3 P V product.  One scale per (batch, head) over the
// whole sequence (a per-key-block scale would vary along the product's
// contraction); the codes are written transposed, [B, H, d, ld] with the
// keys innermost, so that V^T is a K-major operand tile like K.  Three
// passes: the head's amax, the codes, the scales.

// Pass 1: each CTA reduces the amax of 128 rows x D of one (batch, head)
// and folds it into amax_bits[b, h] with an integer atomicMax on the float's
// bits (both are non-negative, where the integer order is the float order).
// amax_bits starts at 0.
template <int D>
__global__ void __launch_bounds__(kQThreads)
    fp8_v_amax_kernel(const __nv_bfloat16* __restrict__ v, unsigned* __restrict__ amax_bits, int N, int H) {
    constexpr int kC = D / 8;  // 16-byte chunks per row
    const int r0 = blockIdx.x * kBlockRows, h = blockIdx.y, b = blockIdx.z;
    const int rows = min(kBlockRows, N - r0);
    float amax = 0.f;
    for (int i = threadIdx.x; i < rows * kC; i += kQThreads) {
        const int r = i / kC, c = i % kC;
        if (!in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8, (long long)gridDim.z * N * H * D,
                       &g_fp8_status))
            continue;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(v + (((long long)b * N + r0 + r) * H + h) * D) + c);
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e[t]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    amax = block_max(amax);
    if (threadIdx.x == 0 && in_bounds((long long)b * H + h, 1, (long long)gridDim.z * H, &g_fp8_status))
        atomicMax(amax_bits + (long long)b * H + h, __float_as_uint(amax));
}

// Pass 2: each CTA quantises 128 keys x D of one (batch, head) with
// inv = 448 / amax (1 for an all-zero head), the arithmetic of the block
// quantiser, and writes them transposed through shared memory.  Loads:
// consecutive threads take consecutive keys of one 8-column chunk, so the
// byte stores into the [D][128] tile hit consecutive bytes; stores: eight
// threads write one 128-byte row of codes.  Keys from N to ld get code 0.
template <int D>
__global__ void __launch_bounds__(kQThreads)
    fp8_v_quant_kernel(const __nv_bfloat16* __restrict__ v, const unsigned* __restrict__ amax_bits,
                       uint8_t* __restrict__ vt, int N, int H, long long ld) {
    constexpr int kC = D / 8;
    constexpr int kRow = kBlockRows + 16;  // tile row stride: 16-byte aligned, rows 4 banks apart
    __shared__ __align__(16) uint8_t tile[D * kRow];
    const int r0 = blockIdx.x * kBlockRows, h = blockIdx.y, b = blockIdx.z;
    const float amax = in_bounds((long long)b * H + h, 1, (long long)gridDim.z * H, &g_fp8_status)
                           ? __uint_as_float(amax_bits[(long long)b * H + h]) : 0.f;
    const bool nz = amax > 0.f;
    const float inv = nz ? kFp8Max / amax : 1.f;
    for (int i = threadIdx.x; i < kBlockRows * kC; i += kQThreads) {
        const int r = i % kBlockRows, c = i / kBlockRows;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + r < N && in_bounds((((long long)b * N + r0 + r) * H + h) * D + 8 * c, 8,
                                    (long long)gridDim.z * N * H * D, &g_fp8_status))
            raw = __ldg(reinterpret_cast<const uint4*>(v + (((long long)b * N + r0 + r) * H + h) * D) + c);
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e[t]);
            const float2 y = make_float2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
            const uint32_t q = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
            tile[(8 * c + 2 * t) * kRow + r] = (uint8_t)(q & 0xFFu);
            tile[(8 * c + 2 * t + 1) * kRow + r] = (uint8_t)(q >> 8);
        }
    }
    __syncthreads();
    const long long base = ((long long)b * H + h) * D * ld;
    for (int i = threadIdx.x; i < D * (kBlockRows / 16); i += kQThreads) {
        const int row = i / (kBlockRows / 16), ch = i % (kBlockRows / 16);
        const long long key = (long long)r0 + 16 * ch;
        if (key >= ld || !in_bounds(base + row * ld + key, 16, (long long)gridDim.z * H * D * ld, &g_fp8_status))
            continue;
        *reinterpret_cast<uint4*>(vt + base + row * ld + key) =
            *reinterpret_cast<const uint4*>(tile + row * kRow + 16 * ch);
    }
}

// Pass 3: scales[i] = amax / 448 (1 for an all-zero head), over the bits
// pass 1 left in the same words.
__global__ void fp8_v_scale_kernel(float* __restrict__ scales, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float amax = __uint_as_float(reinterpret_cast<const unsigned*>(scales)[i]);
    scales[i] = amax > 0.f ? amax / kFp8Max : 1.f;
}

// Any even d: pairs of elements, two passes over the block.
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
    const long long extent = (long long)gridDim.z * N * H * d;
    float amax = 0.f;
    for (int e = threadIdx.x; e < pairs; e += kQThreads) {
        if (!in_bounds(pair_offset(e), 2, extent, &g_fp8_status)) continue;
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + pair_offset(e)));
        amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
    amax = block_max(amax);
    const bool nz = amax > 0.f;
    const float inv = nz ? kFp8Max / amax : 1.f;
    if (threadIdx.x == 0 && in_bounds(((long long)b * H + h) * nb + blk, 1, (long long)gridDim.z * H * nb, &g_fp8_status))
        scales[((long long)b * H + h) * nb + blk] = nz ? amax / kFp8Max : 1.f;
    for (int e = threadIdx.x; e < pairs; e += kQThreads) {
        const long long o = pair_offset(e);
        if (!in_bounds(o, 2, extent, &g_fp8_status)) continue;
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
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    uint8_t* cb = static_cast<uint8_t*>(codes);
    if (d == 128)
        quantize_fp8_regs_kernel<128><<<grid, kQThreads, 0, stream>>>(xb, cb, scales, N, H);
    else if (d == 64)
        quantize_fp8_regs_kernel<64><<<grid, kQThreads, 0, stream>>>(xb, cb, scales, N, H);
    else
        quantize_fp8_kernel<<<grid, kQThreads, 0, stream>>>(xb, cb, scales, N, H, d);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_quantize_fp8_v(const void* v, void* vt8, float* scales, int B, int N, int H, int d,
                                    cudaStream_t stream) {
    const int nb = (N + kBlockRows - 1) / kBlockRows;
    if (H > 65535 || B > 65535 || (d != 64 && d != 128)) return ATTN_ERR_UNSUPPORTED;
    const int n = B * H;
    if (cudaMemsetAsync(scales, 0, (size_t)n * sizeof(float), stream) != cudaSuccess) return ATTN_ERR_CUDA;
    dim3 grid(nb, H, B);
    const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(v);
    unsigned* bits = reinterpret_cast<unsigned*>(scales);
    uint8_t* out = static_cast<uint8_t*>(vt8);
    const long long ld = fp8_v_ld(N);
    if (d == 128) {
        fp8_v_amax_kernel<128><<<grid, kQThreads, 0, stream>>>(vb, bits, N, H);
        fp8_v_quant_kernel<128><<<grid, kQThreads, 0, stream>>>(vb, bits, out, N, H, ld);
    } else {
        fp8_v_amax_kernel<64><<<grid, kQThreads, 0, stream>>>(vb, bits, N, H);
        fp8_v_quant_kernel<64><<<grid, kQThreads, 0, stream>>>(vb, bits, out, N, H, ld);
    }
    fp8_v_scale_kernel<<<(n + 255) / 256, 256, 0, stream>>>(scales, n);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                                          int B, int N, int H, int d, cudaStream_t stream) {
    const int nb = (N + kBlockRows - 1) / kBlockRows;
    if (H > 65535 || B > 65535 || (d != 64 && d != 128)) return ATTN_ERR_UNSUPPORTED;
    dim3 grid(nb, H, B);
    const float c_norm = (float)(1.0 / std::sqrt((double)d));
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    uint8_t* cb = static_cast<uint8_t*>(codes);
    if (d == 128)
        quantize_fp8_rot_kernel<128><<<grid, kQThreads, 0, stream>>>(xb, signs, cb, scales, N, H, c_norm);
    else
        quantize_fp8_rot_kernel<64><<<grid, kQThreads, 0, stream>>>(xb, signs, cb, scales, N, H, c_norm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

cudaError_t fp8_read_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_fp8_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fp8_status, &zero, sizeof(unsigned));
}

}  // namespace attn_host
