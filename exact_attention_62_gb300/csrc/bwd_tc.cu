// bwd_tc.cu -- bf16 exact-attention backward pass on sm_103a tensor cores.
//
// What it computes (Lecture 11 - Kernel Optimization Techniques, section
// 5.1): with S = scale Q K^T, P = softmax(S) and O = P V, given dO,
//     dV = P^T dO,   dP = dO V^T,   D_i = rowsum(dO_i * O_i),
//     dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q,
// where P is not stored but recomputed from the forward's per-row
// log-sum-exp L: P_ij = exp(S_ij - L_i) (one exp per score, no running max).
// A KV head's dK and dV sum over the query heads that share it.
//
// How (GB300 design):
//  * bwd_dot_kernel: D_i = rowsum(dO_i * O_i) into a workspace (the identity
//    section 5.1 uses so that D needs only one row of O and dO).
//  * bwd_dq_kernel: one CTA per 128-row query tile (query tile outer, like
//    the forward).  Per key tile j: S = Q K_j^T and dP = dO V_j^T
//    (tcgen05, operands in shared memory, accumulators in TMEM), then the
//    elementwise warpgroup (one row per thread) forms dS = P * (dP - D) as
//    bf16 over the first S columns, then dQ += dS K_j (A operand read from
//    TMEM).  dQ is written once, scaled, at the end -- no atomics.
//  * bwd_dkdv_kernel: one CTA per 128-key tile (key tile outer), looping over
//    the query heads of its KV group and their query tiles.  With keys as the
//    TMEM lanes: S^T = K Q_i^T and dP^T = V dO_i^T, then P^T and dS^T (bf16)
//    over the first columns of each, then dV += P^T dO_i and dK += dS^T Q_i
//    with both A operands read from TMEM.  The four accumulators fill the 512
//    TMEM columns.  Each thread (one key) needs L and D of all 128 query rows
//    of the tile: they are staged in shared memory, double-buffered.
//  * Both main kernels: warp 0 issues the TMA loads, warp 1 (convergent, one
//    elected lane) the MMAs, warps 4-7 do the elementwise work; rings of
//    K/V (dQ kernel) or Q/dO (dK/dV kernel) tiles stream through shared
//    memory.  Fully masked tiles (causality) are skipped.
//  * This pays 7 matrix products per (query tile, key tile) pair instead of
//    the 5 of a kernel that owns all three accumulators, in exchange for no
//    dQ atomics and one accumulator owner per output.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

__device__ unsigned g_bwd_status = 0;

constexpr int kT = 128;        // rows (queries or keys) per tile
constexpr int kThreads = 256;  // 8 warps: 0 producer, 1 MMA, 2-3 idle, 4-7 elementwise
constexpr int kPanel = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* do_;
    const float* lse;  // [B, Hq, Nq] natural log units of the scaled scores
    const float* dvec; // [B, Hq, Nq] D_i
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int B, Hq, Hkv, Nq, Nk, G, causal;
    float scale, scale_log2;
};

__device__ __forceinline__ long long llmin(long long a, long long b) { return a < b ? a : b; }

// Key tiles a query tile starting at row rs visits (as in the forward).
__device__ __forceinline__ int kv_tiles_for(int rs, const BwdParams& p) {
    if (rs >= p.Nq) return 0;
    if (!p.causal) return (p.Nk + kT - 1) / kT;
    const int re = min(rs + kT, p.Nq) - 1;
    const long long last = llmin((long long)p.Nk - 1, (long long)re + (p.Nk - p.Nq));
    return last < 0 ? 0 : (int)(last / kT) + 1;
}

// First query tile that has an allowed key in the key tile starting at c0.
__device__ __forceinline__ int first_q_tile(int c0, const BwdParams& p) {
    if (!p.causal) return 0;
    const long long r = (long long)c0 - (p.Nk - p.Nq);  // first row allowed to see key c0
    return r <= 0 ? 0 : (int)(r / kT);
}

// ------------------------------------------------------------------ D = rowsum(dO * O)
template <int D>
__global__ void __launch_bounds__(256)
    bwd_dot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                   float* __restrict__ dvec, int B, int Nq, int Hq) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, i, hq) row-major
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)B * Nq * Hq;
    if (row >= rows) return;
    float acc = 0.f;
    for (int c = lane * 4; c < D; c += 128) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + row * D + c);
        const uint2 b = *reinterpret_cast<const uint2*>(dout + row * D + c);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 fa = __bfloat1622float2(pa[e]);
            const float2 fb = __bfloat1622float2(pb[e]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        const int hq = (int)(row % Hq);
        const long long bi = row / Hq;
        const int i = (int)(bi % Nq);
        const int b = (int)(bi / Nq);
        dvec[((long long)b * Hq + hq) * Nq + i] = acc;
    }
}

// Shared layout of both main kernels: two resident tiles (X0, X1), a ring of
// STAGES stages of two streamed tiles each, barriers, misc.
template <int D, int STAGES>
struct BwdLay {
    static constexpr int kTile = kT * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kOffX0 = 0;
    static constexpr int kOffX1 = kTile;
    static constexpr int kOffRing = 2 * kTile;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kOffLD = kOffRing + STAGES * kStage;  // L and D, 2 buffers x 2 x 128 floats
    static constexpr int kOffBar = kOffLD + 2 * 2 * kT * 4;
    // barriers: X full, ring full[STAGES], ring empty[STAGES], S full, dS full, acc full
    static constexpr int kBarX = 0;
    static constexpr int kBarFull = 1;
    static constexpr int kBarEmpty = kBarFull + STAGES;
    static constexpr int kBarS = kBarEmpty + STAGES;
    static constexpr int kBarDS = kBarS + 1;
    static constexpr int kBarAcc = kBarDS + 1;
    static constexpr int kNumBars = kBarAcc + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int D>
constexpr int bwd_stages() { return D == 128 ? 2 : 4; }

// ------------------------------------------------------------------ dQ
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const BwdParams p) {
    constexpr int STAGES = bwd_stages<D>();
    using L = BwdLay<D, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc + 4);

    // tile: longest first (causal: the last query tiles see the most keys)
    const int n_qt = (p.Nq + kT - 1) / kT;
    const int bh = blockIdx.x % (p.B * p.Hq);
    const int qt = n_qt - 1 - (int)(blockIdx.x / (p.B * p.Hq));
    const int b = bh / p.Hq, hq = bh % p.Hq, g = hq / p.G;
    const int r0 = qt * kT;
    const int n = kv_tiles_for(r0, p);

    if (n == 0) {  // rows with no allowed key: dQ = 0
        for (int e = threadIdx.x; e < kT * (D / 8); e += kThreads) {
            const int rr = e / (D / 8), c = e % (D / 8);
            if (r0 + rr < p.Nq)
                reinterpret_cast<uint4*>(p.dq + (((long long)b * p.Nq + r0 + rr) * p.Hq + hq) * D)[c] =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), i == L::kBarDS ? 128u : 1u);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kOffMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t kS = 0, kDP = 128, kDQ = 256;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmDO);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(bar(L::kBarX), 2 * L::kTile);
            for (int pp = 0; pp < L::kPanels; ++pp) {
                tma_load_4d(sbase + L::kOffX0 + pp * kPanel, &tmQ, bar(L::kBarX), 64 * pp, hq, r0, b);
                tma_load_4d(sbase + L::kOffX1 + pp * kPanel, &tmDO, bar(L::kBarX), 64 * pp, hq, r0, b);
            }
            for (int j = 0; j < n; ++j) {
                const int st = j % STAGES;
                if (!mbar_wait(bar(L::kBarEmpty + st), ((j / STAGES) & 1) ^ 1, abort_flag, &g_bwd_status))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarFull + st), L::kStage);
                const uint32_t dst = sbase + L::kOffRing + st * L::kStage;
                for (int pp = 0; pp < L::kPanels; ++pp) {
                    tma_load_4d(dst + pp * kPanel, &tmK, bar(L::kBarFull + st), 64 * pp, g, j * kT, b);
                    tma_load_4d(dst + L::kTile + pp * kPanel, &tmV, bar(L::kBarFull + st), 64 * pp, g,
                                j * kT, b);
                }
            }
        }
    } else if (warp == 1) {
        constexpr uint32_t kIdSS = idesc_bf16_f32(kT, kT, false);  // S, dP: N = 128 keys
        constexpr uint32_t kIdDQ = idesc_bf16_f32(kT, D, true);    // dQ: N = D, B = K N-major
        constexpr uint32_t kHi = sdesc_sw128_hi(1024);
        constexpr uint32_t kKLbo = D == 128 ? kPanel : 1024;
        bool ok = mbar_wait_warp(bar(L::kBarX), 0, abort_flag, &g_bwd_status);
        tc_fence_after();
        const uint32_t q_lo = sdesc_sw128_lo(sbase + L::kOffX0, 16);
        const uint32_t do_lo = sdesc_sw128_lo(sbase + L::kOffX1, 16);
        for (int j = 0; j < n && ok; ++j) {
            const int st = j % STAGES;
            ok = mbar_wait_warp(bar(L::kBarFull + st), (j / STAGES) & 1, abort_flag, &g_bwd_status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kaddr = sbase + L::kOffRing + st * L::kStage;
            const uint32_t k_lo = sdesc_sw128_lo(kaddr, 16);
            const uint32_t v_lo = sdesc_sw128_lo(kaddr + L::kTile, 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kS, q_lo + off, kHi, k_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO V^T
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kDP, do_lo + off, kHi, v_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
            tc_commit_elect(bar(L::kBarS));
            ok = mbar_wait_warp(bar(L::kBarDS), j & 1, abort_flag, &g_bwd_status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kn_lo = sdesc_sw128_lo(kaddr, kKLbo);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk) {  // dQ += dS K  (dS bf16 in TMEM, 16 keys = 8 columns)
                const uint32_t k_off = (kk * 16 * 128) >> 4;
                mma_ts_elect(tmem + kDQ, tmem + kS + kk * 8, kn_lo + k_off, kHi, kIdDQ,
                             (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit_elect(bar(L::kBarEmpty + st));  // K_j and V_j fully read
            if (j == n - 1) tc_commit_elect(bar(L::kBarAcc));
        }
    } else if (warp >= 4) {
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int row = r0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        float lse2 = INFINITY, dval = 0.f;  // rows past Nq: P = 0
        if (row < p.Nq) {
            const float l = p.lse[((long long)b * p.Hq + hq) * p.Nq + row];
            lse2 = l == -INFINITY ? INFINITY : l * kLog2e;  // a row with no allowed key: P = 0
            dval = p.dvec[((long long)b * p.Hq + hq) * p.Nq + row];
        }
        const long long diag = (long long)row + (p.Nk - p.Nq);
        const long long diag_tile = (long long)r0 + (p.Nk - p.Nq);
        const float sl = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (!mbar_wait(bar(L::kBarS), j & 1, abort_flag, &g_bwd_status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int col0 = j * kT;
            const bool need_mask = (col0 + kT > p.Nk) ||
                                   (p.causal && (long long)(col0 + kT - 1) > diag_tile);
            // allowed keys of the row: tile columns [0, lim)
            int lim = kT;
            if (need_mask) {
                long long end = p.Nk;
                if (p.causal && diag + 1 < end) end = diag + 1;
                end -= col0;
                lim = end < 0 ? 0 : end > kT ? kT : (int)end;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t s[64], dp[64];
                tmem_ld64_sync(tmem + lane_base + kS + 64 * h, s);
                tmem_ld64_sync(tmem + lane_base + kDP + 64 * h, dp);
                if (need_mask) {
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc)
                        if (64 * h + cc >= lim) s[cc] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float pr[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int cc = 2 * c + e;
                        const float x = fmaf(__uint_as_float(s[cc]), sl, -lse2);
                        const float pv = ex2(x);
                        pr[e] = pv * (__uint_as_float(dp[cc]) - dval);
                    }
                    pk[c] = pack_bf16(pr[0], pr[1]);
                }
                tmem_st32(tmem + lane_base + kS + 32 * h, pk);  // dS (bf16) over S columns 0..63
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS));
        }
        if (ok && mbar_wait(bar(L::kBarAcc), 0, abort_flag, &g_bwd_status)) {
            tc_fence_after();
            uint32_t xo[64];
            __nv_bfloat16* out = p.dq + (((long long)b * p.Nq + row) * p.Hq + hq) * D;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tmem_ld64_sync(tmem + lane_base + kDQ + 64 * h, xo);
                if (row < p.Nq) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(xo[8 * c + 0]) * p.scale, __uint_as_float(xo[8 * c + 1]) * p.scale);
                        w.y = pack_bf16(__uint_as_float(xo[8 * c + 2]) * p.scale, __uint_as_float(xo[8 * c + 3]) * p.scale);
                        w.z = pack_bf16(__uint_as_float(xo[8 * c + 4]) * p.scale, __uint_as_float(xo[8 * c + 5]) * p.scale);
                        w.w = pack_bf16(__uint_as_float(xo[8 * c + 6]) * p.scale, __uint_as_float(xo[8 * c + 7]) * p.scale);
                        reinterpret_cast<uint4*>(out + 64 * h)[c] = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ dK, dV
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const BwdParams p) {
    constexpr int STAGES = bwd_stages<D>();
    using L = BwdLay<D, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc + 4);

    // key tile, longest first (causal: the first key tiles are seen by the most rows)
    const int n_kt = (p.Nk + kT - 1) / kT;
    const int bg = blockIdx.x % (p.B * p.Hkv);
    const int kt = (int)(blockIdx.x / (p.B * p.Hkv));
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int c0 = kt * kT;
    const int n_qt = (p.Nq + kT - 1) / kT;
    const int i0 = min(first_q_tile(c0, p), n_qt);
    const int per_head = n_qt - i0;
    const int n = per_head * p.G;  // (query head, query tile) iterations
    (void)n_kt;

    if (n == 0) {  // no query row sees these keys: dK = dV = 0
        for (int e = threadIdx.x; e < kT * (D / 8); e += kThreads) {
            const int rr = e / (D / 8), c = e % (D / 8);
            if (c0 + rr < p.Nk) {
                const long long off = (((long long)b * p.Nk + c0 + rr) * p.Hkv + g) * D;
                reinterpret_cast<uint4*>(p.dk + off)[c] = make_uint4(0u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(p.dv + off)[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), i == L::kBarDS ? 128u : 1u);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kOffMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t kS = 0, kDP = 128, kDV = 256, kDK = 384;
    auto it_head = [&](int it) { return g * p.G + it / per_head; };
    auto it_tile = [&](int it) { return i0 + it % per_head; };

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmDO);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(bar(L::kBarX), 2 * L::kTile);
            for (int pp = 0; pp < L::kPanels; ++pp) {
                tma_load_4d(sbase + L::kOffX0 + pp * kPanel, &tmK, bar(L::kBarX), 64 * pp, g, c0, b);
                tma_load_4d(sbase + L::kOffX1 + pp * kPanel, &tmV, bar(L::kBarX), 64 * pp, g, c0, b);
            }
            for (int it = 0; it < n; ++it) {
                const int st = it % STAGES;
                if (!mbar_wait(bar(L::kBarEmpty + st), ((it / STAGES) & 1) ^ 1, abort_flag, &g_bwd_status))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarFull + st), L::kStage);
                const uint32_t dst = sbase + L::kOffRing + st * L::kStage;
                const int hh = it_head(it), rq = it_tile(it) * kT;
                for (int pp = 0; pp < L::kPanels; ++pp) {
                    tma_load_4d(dst + pp * kPanel, &tmQ, bar(L::kBarFull + st), 64 * pp, hh, rq, b);
                    tma_load_4d(dst + L::kTile + pp * kPanel, &tmDO, bar(L::kBarFull + st), 64 * pp, hh, rq,
                                b);
                }
            }
        }
    } else if (warp == 1) {
        constexpr uint32_t kIdSS = idesc_bf16_f32(kT, kT, false);  // S^T, dP^T: M = keys, N = query rows
        constexpr uint32_t kIdAcc = idesc_bf16_f32(kT, D, true);   // dV, dK: N = D, B N-major
        constexpr uint32_t kHi = sdesc_sw128_hi(1024);
        constexpr uint32_t kNLbo = D == 128 ? kPanel : 1024;
        bool ok = mbar_wait_warp(bar(L::kBarX), 0, abort_flag, &g_bwd_status);
        tc_fence_after();
        const uint32_t k_lo = sdesc_sw128_lo(sbase + L::kOffX0, 16);
        const uint32_t v_lo = sdesc_sw128_lo(sbase + L::kOffX1, 16);
        for (int it = 0; it < n && ok; ++it) {
            const int st = it % STAGES;
            ok = mbar_wait_warp(bar(L::kBarFull + st), (it / STAGES) & 1, abort_flag, &g_bwd_status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t qaddr = sbase + L::kOffRing + st * L::kStage;
            const uint32_t q_lo = sdesc_sw128_lo(qaddr, 16);
            const uint32_t do_lo = sdesc_sw128_lo(qaddr + L::kTile, 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // S^T = K Q^T
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kS, k_lo + off, kHi, q_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V dO^T
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kDP, v_lo + off, kHi, do_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
            tc_commit_elect(bar(L::kBarS));
            ok = mbar_wait_warp(bar(L::kBarDS), it & 1, abort_flag, &g_bwd_status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t qn_lo = sdesc_sw128_lo(qaddr, kNLbo);
            const uint32_t don_lo = sdesc_sw128_lo(qaddr + L::kTile, kNLbo);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk) {  // 16 query rows = 8 bf16 columns of P^T / dS^T
                const uint32_t r_off = (kk * 16 * 128) >> 4;
                const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                mma_ts_elect(tmem + kDV, tmem + kS + kk * 8, don_lo + r_off, kHi, kIdAcc, acc);   // dV += P^T dO
                mma_ts_elect(tmem + kDK, tmem + kDP + kk * 8, qn_lo + r_off, kHi, kIdAcc, acc);   // dK += dS^T Q
            }
            tc_commit_elect(bar(L::kBarEmpty + st));  // Q_i and dO_i fully read
            if (it == n - 1) tc_commit_elect(bar(L::kBarAcc));
        }
    } else if (warp >= 4) {
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;  // the key this thread owns
        const int key = c0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const int tid = threadIdx.x - 128;  // 0..127 within the warpgroup
        float* ldbuf = reinterpret_cast<float*>(sgen + L::kOffLD);  // [2][2][128]: L*log2e, D
        const float sl = p.scale_log2;
        // L and D of query row `rq + tid` of head hh (rows past Nq: P = 0)
        auto fetch = [&](int it, float& l2, float& dv) {
            const int hh = it_head(it), row = it_tile(it) * kT + tid;
            l2 = INFINITY;
            dv = 0.f;
            if (row < p.Nq) {
                const long long o = ((long long)b * p.Hq + hh) * p.Nq + row;
                const float l = p.lse[o];
                l2 = l == -INFINITY ? INFINITY : l * kLog2e;
                dv = p.dvec[o];
            }
        };
        float nl2, ndv;
        fetch(0, nl2, ndv);
        bool ok = true;
        // Every thread of the warpgroup runs every iteration, also after a
        // bounded wait has given up (the abort flag then ends the remaining
        // waits at once): the named barrier below must never miss a thread.
        for (int it = 0; it < n; ++it) {
            const int buf = it & 1;
            ldbuf[(buf * 2 + 0) * kT + tid] = nl2;
            ldbuf[(buf * 2 + 1) * kT + tid] = ndv;
            named_bar_sync(1, 128);  // this iteration's L and D are visible to the warpgroup
            if (it + 1 < n) fetch(it + 1, nl2, ndv);  // in flight while this tile is processed
            const float* lrow = ldbuf + (buf * 2 + 0) * kT;
            const float* drow = ldbuf + (buf * 2 + 1) * kT;
            if (ok) ok = mbar_wait(bar(L::kBarS), it & 1, abort_flag, &g_bwd_status);
            if (!ok) continue;
            tc_fence_after();
            const int rq = it_tile(it) * kT;
            // causal: query row i may see this key iff key <= i + (Nk - Nq)
            const bool need_mask = key >= p.Nk || (p.causal && (long long)c0 + kT - 1 > (long long)rq + (p.Nk - p.Nq));
            // the query rows that may see this key: tile columns [lo, kT)
            int lo = 0;
            if (need_mask) {
                long long first = key >= p.Nk ? (long long)kT
                                              : (p.causal ? (long long)key - (p.Nk - p.Nq) - rq : 0ll);
                lo = first < 0 ? 0 : first > kT ? kT : (int)first;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t s[64], dp[64];
                tmem_ld64_sync(tmem + lane_base + kS + 64 * h, s);
                tmem_ld64_sync(tmem + lane_base + kDP + 64 * h, dp);
                if (need_mask) {
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc)
                        if (64 * h + cc < lo) s[cc] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[32], dk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float pv[2], dsv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int cc = 64 * h + 2 * c + e;  // query row rq + cc
                        const float x = fmaf(__uint_as_float(s[2 * c + e]), sl, -lrow[cc]);
                        pv[e] = ex2(x);
                        dsv[e] = pv[e] * (__uint_as_float(dp[2 * c + e]) - drow[cc]);
                    }
                    pk[c] = pack_bf16(pv[0], pv[1]);
                    dk[c] = pack_bf16(dsv[0], dsv[1]);
                }
                tmem_st32(tmem + lane_base + kS + 32 * h, pk);   // P^T over S^T columns 0..63
                tmem_st32(tmem + lane_base + kDP + 32 * h, dk);  // dS^T over dP^T columns 0..63
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS));
        }
        if (ok && mbar_wait(bar(L::kBarAcc), 0, abort_flag, &g_bwd_status)) {
            tc_fence_after();
            uint32_t xo[64];
            const long long off = (((long long)b * p.Nk + key) * p.Hkv + g) * D;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tmem_ld64_sync(tmem + lane_base + kDV + 64 * h, xo);
                if (key < p.Nk) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(xo[8 * c + 0]), __uint_as_float(xo[8 * c + 1]));
                        w.y = pack_bf16(__uint_as_float(xo[8 * c + 2]), __uint_as_float(xo[8 * c + 3]));
                        w.z = pack_bf16(__uint_as_float(xo[8 * c + 4]), __uint_as_float(xo[8 * c + 5]));
                        w.w = pack_bf16(__uint_as_float(xo[8 * c + 6]), __uint_as_float(xo[8 * c + 7]));
                        reinterpret_cast<uint4*>(p.dv + off + 64 * h)[c] = w;
                    }
                }
                tmem_ld64_sync(tmem + lane_base + kDK + 64 * h, xo);
                if (key < p.Nk) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(xo[8 * c + 0]) * p.scale, __uint_as_float(xo[8 * c + 1]) * p.scale);
                        w.y = pack_bf16(__uint_as_float(xo[8 * c + 2]) * p.scale, __uint_as_float(xo[8 * c + 3]) * p.scale);
                        w.z = pack_bf16(__uint_as_float(xo[8 * c + 4]) * p.scale, __uint_as_float(xo[8 * c + 5]) * p.scale);
                        w.w = pack_bf16(__uint_as_float(xo[8 * c + 6]) * p.scale, __uint_as_float(xo[8 * c + 7]) * p.scale);
                        reinterpret_cast<uint4*>(p.dk + off + 64 * h)[c] = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
attn_status_t launch_bwd_impl(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Nq, int Nk, int causal, float scale,
                              float* dvec, cudaStream_t stream) {
    using L = BwdLay<D, bwd_stages<D>()>;
    CUtensorMap mq, mdo, mk, mv;
    if (!attn_host::encode_bshd_map(&mq, q, B, Nq, Hq, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mdo, dout, B, Nq, Hq, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mk, k, B, Nk, Hkv, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mv, v, B, Nk, Hkv, D, kT, 2))
        return ATTN_ERR_CUDA;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            L::kSmem);
    });
    if (attr_err != cudaSuccess) return ATTN_ERR_CUDA;
    BwdParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.k = static_cast<const __nv_bfloat16*>(k);
    prm.do_ = static_cast<const __nv_bfloat16*>(dout);
    prm.lse = lse;
    prm.dvec = dvec;
    prm.dq = static_cast<__nv_bfloat16*>(dq);
    prm.dk = static_cast<__nv_bfloat16*>(dk);
    prm.dv = static_cast<__nv_bfloat16*>(dv);
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    prm.causal = causal;
    prm.scale = scale;
    prm.scale_log2 = scale * kLog2e;
    const long long rows = (long long)B * Nq * Hq;
    const long long dot_blocks = (rows + 7) / 8;
    const long long dq_blocks = (long long)B * Hq * ((Nq + kT - 1) / kT);
    const long long dkv_blocks = (long long)B * Hkv * ((Nk + kT - 1) / kT);
    if (dot_blocks > 0x7fffffffLL || dq_blocks > 0x7fffffffLL || dkv_blocks > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    bwd_dot_kernel<D><<<(unsigned)dot_blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                               prm.do_, dvec, B, Nq, Hq);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    bwd_dkdv_kernel<D><<<(unsigned)dkv_blocks, kThreads, L::kSmem, stream>>>(mq, mdo, mk, mv, prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    bwd_dq_kernel<D><<<(unsigned)dq_blocks, kThreads, L::kSmem, stream>>>(mq, mdo, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

size_t bwd_workspace_bytes(int B, int Hq, int Nq) {
    return ((size_t)B * Hq * Nq * 4 + 255) / 256 * 256;
}

attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                         int Nq, int Nk, int d, int causal, float scale, void* workspace,
                         cudaStream_t stream) {
    float* dvec = static_cast<float*>(workspace);
    if (d == 128)
        return launch_bwd_impl<128>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, causal, scale,
                                    dvec, stream);
    return launch_bwd_impl<64>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, causal, scale, dvec,
                               stream);
}

cudaError_t bwd_read_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned));
}

}  // namespace attn_host
