// fwd_f32.cu -- fp32 exact-attention forward on CUDA cores.
//
// Same computation as the bf16 tensor-core kernel (Lecture 11 - Kernel
// Optimization Techniques, sections 2, 3.1 and 3.3: online softmax over key
// tiles with deferred normalisation, causal tiles beyond the diagonal
// skipped per section 5.3), but every operand and every product stays in
// fp32 so that fp32 inputs meet fp32 accuracy; the tensor-core path would
// round P and the inputs to bf16/tf32.
//
// One CTA of 128 threads owns R query rows of one (batch, head): 32 rows,
// four threads to a row, or, when that leaves SMs idle (a single 256-row
// head: 8 CTAs), 8 rows with sixteen threads to a row.  Per 32-key tile each
// thread computes 32 R / 128 scores of its row, the row's max and sum are
// reduced across its threads with shuffles, P goes to shared memory, and each
// thread accumulates D R / 128 output columns.  K and V tiles are
// double-buffered in shared memory with cp.async, so the next tile's loads
// overlap this tile's arithmetic.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

// Status word of this kernel family: only the bounds-checked build sets it.
__device__ unsigned g_f32_status = 0;

__device__ __forceinline__ long long llmin(long long a, long long b) { return a < b ? a : b; }

// 16-byte global -> shared copy that completes asynchronously (cp.async,
// cached in L1), and its group commit and wait.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kKeys = 32;
constexpr int kThreadsF32 = 128;

struct F32Params {
    int B, Hq, Hkv, Nq, Nk, G, causal;
    float scale;
};

template <int D, int R>  // R: query rows per CTA (8 or 32)
struct F32Layout {
    static constexpr int kTpr = kThreadsF32 / R;  // threads per row
    static constexpr int kLd = D + 4;             // padded row stride (floats)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + R * kLd;          // two buffers
    static constexpr int kV = kK + 2 * kKeys * kLd;  // two buffers
    static constexpr int kP = kV + 2 * kKeys * kLd;
    static constexpr int kFloats = kP + R * (kKeys + 1);
    static constexpr int kBytes = kFloats * 4;
    static_assert(kKeys % kTpr == 0 && D / 4 % kTpr == 0, "whole keys and float4 chunks per thread");
    static_assert(kTpr <= 32 && 32 % kTpr == 0, "a row's threads in one warp");
};

template <int D, int R>
__global__ void __launch_bounds__(kThreadsF32, 1)
    fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                   const F32Params p) {
    using L = F32Layout<D, R>;
    constexpr int kRows = R;
    constexpr int kTpr = L::kTpr;
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    float* Qs = sm + L::kQ;
    float* Ps = sm + L::kP;
    constexpr int C4 = D / 4;        // float4 chunks per row
    constexpr int NCH = C4 / kTpr;   // float4 chunks of the output each thread owns
    constexpr int NS = kKeys / kTpr; // scores per thread and tile
    const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
    const int g = hq / p.G;
    const int tid = threadIdx.x;
    const int r = tid / kTpr, cg = tid % kTpr;
    const int row = qt * kRows + r;
    const long long kv_extent = (long long)p.B * p.Nk * p.Hkv * D;

    // K_jt and V_jt into buffer jt & 1: cp.async for keys inside the cache,
    // zeros past its end
    auto load_tile = [&](int jt) {
        float* Ks = sm + L::kK + (jt & 1) * kKeys * L::kLd;
        float* Vs = sm + L::kV + (jt & 1) * kKeys * L::kLd;
        for (int idx = tid; idx < kKeys * C4; idx += kThreadsF32) {
            const int rr = idx / C4, c4 = idx % C4;
            const int key = jt * kKeys + rr;
            const long long off = (((long long)b * p.Nk + key) * p.Hkv + g) * D + 4 * c4;
            if (key < p.Nk && in_bounds(off, 4, kv_extent, &g_f32_status)) {
                cp_async16(Ks + rr * L::kLd + 4 * c4, k + off);
                cp_async16(Vs + rr * L::kLd + 4 * c4, v + off);
            } else {
                *reinterpret_cast<float4*>(Ks + rr * L::kLd + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(Vs + rr * L::kLd + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        cp_async_commit();
    };

    for (int idx = tid; idx < kRows * C4; idx += kThreadsF32) {
        const int rr = idx / C4, c4 = idx % C4;
        const int qr = qt * kRows + rr;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qr < p.Nq) {
            const long long qoff = (((long long)b * p.Nq + qr) * p.Hq + hq) * D;
            if (in_bounds(qoff + 4 * c4, 4, (long long)p.B * p.Nq * p.Hq * D, &g_f32_status))
                val = __ldg(reinterpret_cast<const float4*>(q + qoff) + c4);
        }
        *reinterpret_cast<float4*>(Qs + rr * L::kLd + 4 * c4) = val;
    }
    int nkv;
    if (!p.causal) {
        nkv = (p.Nk + kKeys - 1) / kKeys;
    } else {
        const int last_row = min(qt * kRows + kRows - 1, p.Nq - 1);
        const long long last = llmin((long long)p.Nk - 1, (long long)last_row + (p.Nk - p.Nq));
        nkv = last < 0 ? 0 : (int)(last / kKeys) + 1;
    }
    const long long diag = (long long)row + (p.Nk - p.Nq);

    float m = -INFINITY, l = 0.f;
    float4 acc[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);

    if (nkv > 0) load_tile(0);
    for (int jt = 0; jt < nkv; ++jt) {
        // the next tile streams in while this one is used
        if (jt + 1 < nkv) {
            load_tile(jt + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // tile jt (and, at jt = 0, Q) visible to every thread
        const float* Ks = sm + L::kK + (jt & 1) * kKeys * L::kLd;
        const float* Vs = sm + L::kV + (jt & 1) * kKeys * L::kLd;

        float s[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) s[i] = 0.f;
#pragma unroll 4
        for (int c4 = 0; c4 < C4; ++c4) {
            const float4 qv = *reinterpret_cast<const float4*>(Qs + r * L::kLd + 4 * c4);
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                const float4 kv = *reinterpret_cast<const float4*>(Ks + (cg + kTpr * i) * L::kLd + 4 * c4);
                s[i] = fmaf(qv.x, kv.x, s[i]);
                s[i] = fmaf(qv.y, kv.y, s[i]);
                s[i] = fmaf(qv.z, kv.z, s[i]);
                s[i] = fmaf(qv.w, kv.w, s[i]);
            }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            const int key = jt * kKeys + cg + kTpr * i;
            const bool keep = key < p.Nk && (!p.causal || (long long)key <= diag);
            s[i] = keep ? s[i] * p.scale : -INFINITY;
            mx = fmaxf(mx, s[i]);
        }
#pragma unroll
        for (int off = 1; off < kTpr; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = expf(m - m_use);
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            const float pi = expf(s[i] - m_use);
            ps += pi;
            Ps[r * (kKeys + 1) + cg + kTpr * i] = pi;
        }
#pragma unroll
        for (int off = 1; off < kTpr; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = fmaf(l, alpha, ps);
        m = m_new;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            acc[i].x *= alpha;
            acc[i].y *= alpha;
            acc[i].z *= alpha;
            acc[i].w *= alpha;
        }
        __syncwarp();  // the threads of a row live in one warp
#pragma unroll 4
        for (int jj = 0; jj < kKeys; ++jj) {
            const float pj = Ps[r * (kKeys + 1) + jj];
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                const float4 vv = *reinterpret_cast<const float4*>(Vs + jj * L::kLd + 4 * (cg + kTpr * i));
                acc[i].x = fmaf(pj, vv.x, acc[i].x);
                acc[i].y = fmaf(pj, vv.y, acc[i].y);
                acc[i].z = fmaf(pj, vv.z, acc[i].z);
                acc[i].w = fmaf(pj, vv.w, acc[i].w);
            }
        }
        __syncthreads();  // buffer jt & 1 fully read before tile jt + 2 lands in it
    }

    if (row < p.Nq) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* orow = o + (((long long)b * p.Nq + row) * p.Hq + hq) * D;
        if (in_bounds(orow - o, D, (long long)p.B * p.Nq * p.Hq * D, &g_f32_status)) {
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                float4 w = acc[i];
                w.x *= inv;
                w.y *= inv;
                w.z *= inv;
                w.w *= inv;
                reinterpret_cast<float4*>(orow)[cg + kTpr * i] = w;
            }
        }
        if (cg == 0 &&
            in_bounds(((long long)b * p.Hq + hq) * p.Nq + row, 1, (long long)p.B * p.Hq * p.Nq, &g_f32_status))
            lse[((long long)b * p.Hq + hq) * p.Nq + row] = l > 0.f ? m + logf(l) : -INFINITY;
    }
}

template <int D, int R>
attn_status_t launch_rows(const float* q, const float* k, const float* v, float* o, float* lse,
                          const F32Params& prm, cudaStream_t stream) {
    using L = F32Layout<D, R>;
    if (attn_host::kernel_setup<fwd_f32_kernel<D, R>>(L::kBytes).err != cudaSuccess) return ATTN_ERR_CUDA;
    const long long qtiles = (prm.Nq + R - 1) / R;
    if (qtiles > 0x7fffffffLL || prm.Hq > 65535 || prm.B > 65535) return ATTN_ERR_UNSUPPORTED;
    dim3 grid((unsigned)qtiles, prm.Hq, prm.B);
    fwd_f32_kernel<D, R><<<grid, kThreadsF32, L::kBytes, stream>>>(q, k, v, o, lse, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// 32-row CTAs, unless they would leave SMs idle: then 8-row CTAs, four times
// as many (GB300, fp32: a 256-row head 32.0 -> 17.2 us; B4 H16 N4096 causal
// 16.5 TFLOP/s with 32 rows against 13.0 with 8, which re-read K and V
// four times as often).
template <int D>
attn_status_t launch_impl(const float* q, const float* k, const float* v, float* o, float* lse,
                          const F32Params& prm, cudaStream_t stream) {
    const long long ctas32 = (long long)(prm.Nq + 31) / 32 * prm.Hq * prm.B;
    const int sms = attn_host::device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    return ctas32 < sms ? launch_rows<D, 8>(q, k, v, o, lse, prm, stream)
                        : launch_rows<D, 32>(q, k, v, o, lse, prm, stream);
}

}  // namespace

namespace attn_host {

attn_status_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o,
                             float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                             int causal, float scale, cudaStream_t stream) {
    F32Params prm{B, Hq, Hkv, Nq, Nk, Hq / Hkv, causal, scale};
    if (d == 128) return launch_impl<128>(q, k, v, o, lse, prm, stream);
    if (d == 64) return launch_impl<64>(q, k, v, o, lse, prm, stream);
    return ATTN_ERR_UNSUPPORTED;
}

cudaError_t fwd_f32_read_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_f32_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_f32_status, &zero, sizeof(unsigned));
}

}  // namespace attn_host
