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
//    the forward).  Per key tile j: S_j = Q K_j^T and dP_j = dO V_j^T
//    (tcgen05, operands in shared memory, accumulators in TMEM); the
//    elementwise warps read both into registers and say so, which lets the
//    MMA warp issue S_{j+1} and dP_{j+1} while they form dS_j = P * (dP - D)
//    as bf16 into one of two spare 64-column TMEM buffers; then
//    dQ += dS_j K_j (A operand read from TMEM).  dQ is written once, scaled,
//    at the end -- no atomics.
//  * bwd_dkdv_kernel: one CTA per 128-key tile (key tile outer), looping over
//    the query heads of its KV group and their query tiles.  With keys as the
//    TMEM lanes: S^T = K Q_i^T and dP^T = V dO_i^T, then P^T and dS^T (bf16)
//    over the dP^T columns just read, then dV += P^T dO_i and dK += dS^T Q_i
//    with both A operands read from TMEM.  Once the elementwise warps hold
//    S^T in registers, the next tile's S^T may be issued (when its Q tile
//    is already loaded) while they work.  The four accumulators fill the 512
//    TMEM columns.  Each thread (one key) needs L and D of the query rows it
//    handles: they are staged in shared memory, double-buffered.
//  * Both main kernels: warp 0 issues the TMA loads, warp 1 (convergent, one
//    elected lane) the MMAs, and two elementwise warpgroups (warps 4-7 and
//    8-11) split each tile's 128 columns between them, so each thread of a
//    row (TMEM lane) handles 64 scores per tile.  Rings of K/V (dQ kernel) or
//    Q/dO (dK/dV kernel) tiles stream through shared memory.  Fully masked
//    tiles (causality) are skipped.
//  * This pays 7 matrix products per (query tile, key tile) pair instead of
//    the 5 of a kernel that owns all three accumulators, in exchange for no
//    dQ atomics and one accumulator owner per output.
//  * Launch order: rowsum, dK/dV, then dQ as a programmatic dependent of the
//    dK/dV grid (dQ reads nothing that grid writes), so the dQ CTAs start on
//    the SMs the dK/dV grid's last wave frees.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

__device__ unsigned g_bwd_status = 0;

constexpr int kT = 128;        // rows (queries or keys) per tile
// 12 warps: 0 producer, 1 MMA, 2-3 idle, 4-7 and 8-11 elementwise (one
// warpgroup per half of a tile's columns).
constexpr int kThreads = 384;
// Register split: compiled for kLaunchRegs per thread (the most 384 threads
// allow); warpgroup 0 gives registers back to the elementwise warpgroups.
constexpr int kLaunchRegs = 168;
constexpr int kRegsWG0 = 56;
constexpr int kRegsEW = 224;
static_assert(128 * kRegsWG0 + 256 * kRegsEW <= kThreads * kLaunchRegs, "register split");
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
// HBM-bound: each row is D bf16 of O and of dO.  A group of D/8 threads takes
// a row with 16-byte loads; every thread has kDotRows rows' loads in flight
// before it reduces any of them.
constexpr int kDotThreads = 256;
constexpr int kDotRows = 4;
template <int D>
__global__ void __launch_bounds__(kDotThreads)
    bwd_dot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                   float* __restrict__ dvec, int B, int Nq, int Hq) {
    constexpr int kTpr = D / 8;                       // threads per row
    constexpr int kRowsPerPass = kDotThreads / kTpr;  // rows a block covers per pass
    const long long rows = (long long)B * Nq * Hq;
    const int sub = threadIdx.x % kTpr;
    const long long base = (long long)blockIdx.x * kRowsPerPass * kDotRows + threadIdx.x / kTpr;
    uint4 a[kDotRows], c[kDotRows];
#pragma unroll
    for (int u = 0; u < kDotRows; ++u) {
        const long long row = base + (long long)u * kRowsPerPass;  // (b, i, hq) row-major
        a[u] = make_uint4(0u, 0u, 0u, 0u);
        c[u] = a[u];
        if (row < rows && in_bounds(row * D + 8 * sub, 8, rows * D, &g_bwd_status)) {
            a[u] = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
            c[u] = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + sub);
        }
    }
#pragma unroll
    for (int u = 0; u < kDotRows; ++u) {
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
        const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c[u]);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(pa[e]);
            const float2 fc = __bfloat1622float2(pc[e]);
            acc = fmaf(fa.x, fc.x, acc);
            acc = fmaf(fa.y, fc.y, acc);
        }
#pragma unroll
        for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long row = base + (long long)u * kRowsPerPass;
        if (sub == 0 && row < rows) {
            const int hq = (int)(row % Hq);
            const long long bi = row / Hq;
            const int i = (int)(bi % Nq);
            const int b = (int)(bi / Nq);
            if (in_bounds(((long long)b * Hq + hq) * Nq + i, 1, rows, &g_bwd_status))
                dvec[((long long)b * Hq + hq) * Nq + i] = acc;
        }
    }
}

// Shared layout of the dK/dV kernel: two resident tiles (X0 = K, X1 = V), a
// ring of STAGES stages of two streamed tiles each (Q_i, dO_i), the staged L
// and D rows, barriers, misc.
template <int D, int STAGES>
struct BwdLay {
    static constexpr int kTile = kT * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kOffX0 = 0;
    static constexpr int kOffX1 = kTile;
    static constexpr int kOffRing = 2 * kTile;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kOffLD = kOffRing + STAGES * kStage;  // L and D: 2 buffers x 2 warpgroups x 2 x 64 floats
    static constexpr int kOffBar = kOffLD + 2 * 2 * kT * 4;
    // barriers: X full, ring full[STAGES], ring empty[STAGES], S full, consumed, dS full, acc full
    static constexpr int kBarX = 0;
    static constexpr int kBarFull = 1;
    static constexpr int kBarEmpty = kBarFull + STAGES;
    static constexpr int kBarS = kBarEmpty + STAGES;
    static constexpr int kBarC = kBarS + 1;   // S^T, dP^T read into registers (256 threads)
    static constexpr int kBarDS = kBarC + 1;  // P^T, dS^T in TMEM (256 threads)
    static constexpr int kBarAcc = kBarDS + 1;
    static constexpr int kNumBars = kBarAcc + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int D>
constexpr int bwd_stages() { return D == 128 ? 2 : 4; }

// ------------------------------------------------------------------ dQ
// Shared layout of the dQ kernel: Q and dO resident, K and V in separate
// rings.  A V tile is released as soon as dP has read it; a K tile only after
// dQ += dS K has, and S of the next tile is issued while the current dS is
// still being formed, so the K ring is one stage deeper.
template <int D>
struct DqLay {
    static constexpr int kTile = kT * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kKSt = D == 128 ? 3 : 4;
    static constexpr int kVSt = D == 128 ? 2 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kTile;
    static constexpr int kOffK = 2 * kTile;
    static constexpr int kOffV = kOffK + kKSt * kTile;
    static constexpr int kOffBar = kOffV + kVSt * kTile;
    static constexpr int kBarX = 0;                      // Q and dO loaded
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kKSt;
    static constexpr int kBarVFull = kBarKEmpty + kKSt;
    static constexpr int kBarVEmpty = kBarVFull + kVSt;
    static constexpr int kBarS = kBarVEmpty + kVSt;      // S_j and dP_j in TMEM (commit)
    static constexpr int kBarC = kBarS + 1;              // S_j, dP_j read into registers (256 threads)
    static constexpr int kBarDS = kBarC + 1;             // dS_j in TMEM buffer j & 1 (256 threads; two barriers)
    static constexpr int kBarAcc = kBarDS + 2;
    static constexpr int kNumBars = kBarAcc + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
    __host__ __device__ static constexpr unsigned count(int i) {
        return (i == kBarC || i == kBarDS || i == kBarDS + 1) ? 2u * kT : 1u;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const BwdParams p) {
    using L = DqLay<D>;
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
            if (r0 + rr < p.Nq &&
                in_bounds((((long long)b * p.Nq + r0 + rr) * p.Hq + hq) * D + 8 * c, 8,
                          (long long)p.B * p.Nq * p.Hq * D, &g_bwd_status))
                reinterpret_cast<uint4*>(p.dq + (((long long)b * p.Nq + r0 + rr) * p.Hq + hq) * D)[c] =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), L::count(i));
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
    // TMEM columns: S, dP (128 fp32 each), the dQ accumulator (D), and two
    // 64-column buffers of bf16 dS (128 keys, two per column) from 384 on.
    constexpr uint32_t kS = 0, kDP = 128, kDQ = 256, kDSb = 384;

    if (warp < 4) {
        warpgroup_reg_dealloc<kRegsWG0>();
        if (warp == 0) {
            if (lane == 0) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmDO);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmV);
                mbar_arrive_expect_tx(bar(L::kBarX), 2 * L::kTile);
                for (int pp = 0; pp < L::kPanels; ++pp) {
                    tma_load_4d(sbase + L::kOffQ + pp * kPanel, &tmQ, bar(L::kBarX), 64 * pp, hq, r0, b);
                    tma_load_4d(sbase + L::kOffDO + pp * kPanel, &tmDO, bar(L::kBarX), 64 * pp, hq, r0, b);
                }
                for (int j = 0; j < n; ++j) {
                    const int ks = j % L::kKSt, vs = j % L::kVSt;
                    if (!mbar_wait(bar(L::kBarKEmpty + ks), ((j / L::kKSt) & 1) ^ 1, abort_flag, &g_bwd_status))
                        break;
                    mbar_arrive_expect_tx(bar(L::kBarKFull + ks), L::kTile);
                    for (int pp = 0; pp < L::kPanels; ++pp)
                        tma_load_4d(sbase + L::kOffK + ks * L::kTile + pp * kPanel, &tmK, bar(L::kBarKFull + ks),
                                    64 * pp, g, j * kT, b);
                    if (!mbar_wait(bar(L::kBarVEmpty + vs), ((j / L::kVSt) & 1) ^ 1, abort_flag, &g_bwd_status))
                        break;
                    mbar_arrive_expect_tx(bar(L::kBarVFull + vs), L::kTile);
                    for (int pp = 0; pp < L::kPanels; ++pp)
                        tma_load_4d(sbase + L::kOffV + vs * L::kTile + pp * kPanel, &tmV, bar(L::kBarVFull + vs),
                                    64 * pp, g, j * kT, b);
                }
            }
        } else if (warp == 1) {
            constexpr uint32_t kIdSS = idesc_bf16_f32(kT, kT, false);  // S, dP: N = 128 keys
            constexpr uint32_t kIdDQ = idesc_bf16_f32(kT, D, true);    // dQ: N = D, B = K N-major
            constexpr uint32_t kHi = sdesc_sw128_hi(1024);
            constexpr uint32_t kKLbo = D == 128 ? kPanel : 1024;
            bool ok = mbar_wait_warp(bar(L::kBarX), 0, abort_flag, &g_bwd_status);
            tc_fence_after();
            const uint32_t q_lo = sdesc_sw128_lo(sbase + L::kOffQ, 16);
            const uint32_t do_lo = sdesc_sw128_lo(sbase + L::kOffDO, 16);
            // S_j = Q K_j^T and dP_j = dO V_j^T into TMEM; V_j is free once dP_j is done
            auto issue_sdp = [&](int j) {
                const int ks = j % L::kKSt, vs = j % L::kVSt;
                if (ok) ok = mbar_wait_warp(bar(L::kBarKFull + ks), (j / L::kKSt) & 1, abort_flag, &g_bwd_status);
                if (ok) ok = mbar_wait_warp(bar(L::kBarVFull + vs), (j / L::kVSt) & 1, abort_flag, &g_bwd_status);
                if (!ok) return;
                tc_fence_after();
                const uint32_t k_lo = sdesc_sw128_lo(sbase + L::kOffK + ks * L::kTile, 16);
                const uint32_t v_lo = sdesc_sw128_lo(sbase + L::kOffV + vs * L::kTile, 16);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                    mma_ss_elect(tmem + kS, q_lo + off, kHi, k_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                    mma_ss_elect(tmem + kDP, do_lo + off, kHi, v_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
                }
                tc_commit_elect(bar(L::kBarS));
                tc_commit_elect(bar(L::kBarVEmpty + vs));
            };
            issue_sdp(0);
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n) {
                    // the elementwise warps hold S_j and dP_j: the next pair may overwrite them
                    ok = mbar_wait_warp(bar(L::kBarC), j & 1, abort_flag, &g_bwd_status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_sdp(j + 1);
                    if (!ok) break;
                }
                ok = mbar_wait_warp(bar(L::kBarDS + (j & 1)), (j >> 1) & 1, abort_flag, &g_bwd_status);
                if (!ok) break;
                tc_fence_after();
                const int ks = j % L::kKSt;
                const uint32_t kn_lo = sdesc_sw128_lo(sbase + L::kOffK + ks * L::kTile, kKLbo);
                const uint32_t ds = tmem + kDSb + 64u * (uint32_t)(j & 1);
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk) {  // dQ += dS K  (16 keys = 8 bf16 columns of dS)
                    const uint32_t k_off = (kk * 16 * 128) >> 4;
                    mma_ts_elect(tmem + kDQ, ds + kk * 8, kn_lo + k_off, kHi, kIdDQ, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit_elect(bar(L::kBarKEmpty + ks));  // K_j fully read
                if (j == n - 1) tc_commit_elect(bar(L::kBarAcc));
            }
        }
    } else {
        warpgroup_reg_alloc<kRegsEW>();
        // Two elementwise warpgroups share each row (TMEM lane): warpgroup w
        // takes keys 64w .. 64w + 63 of every key tile.
        const int w = (warp - 4) >> 2;
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int row = r0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        float lse2 = INFINITY, dval = 0.f;  // rows past Nq: P = 0
        if (row < p.Nq && in_bounds(((long long)b * p.Hq + hq) * p.Nq + row, 1,
                                    (long long)p.B * p.Hq * p.Nq, &g_bwd_status)) {
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
            uint32_t s[64], dp[64];
            tmem_ld64_sync(tmem + lane_base + kS + 64 * w, s);
            tmem_ld64_sync(tmem + lane_base + kDP + 64 * w, dp);
            tc_fence_before();
            mbar_arrive(bar(L::kBarC));
            const int col0 = j * kT;
            const bool need_mask = (col0 + kT > p.Nk) ||
                                   (p.causal && (long long)(col0 + kT - 1) > diag_tile);
            if (need_mask) {
                // allowed keys of the row: tile columns [0, lim)
                long long end = p.Nk;
                if (p.causal && diag + 1 < end) end = diag + 1;
                end -= col0;
                const int lim = end < 0 ? 0 : end > kT ? kT : (int)end;
#pragma unroll
                for (int cc = 0; cc < 64; ++cc)
                    if (64 * w + cc >= lim) s[cc] = __float_as_uint(-INFINITY);
            }
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float pr[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int cc = 2 * c + e;
                    const float pv = ex2(fmaf(__uint_as_float(s[cc]), sl, -lse2));
                    pr[e] = pv * (__uint_as_float(dp[cc]) - dval);
                }
                pk[c] = pack_bf16(pr[0], pr[1]);
            }
            tmem_st32(tmem + lane_base + kDSb + 64u * (uint32_t)(j & 1) + 32u * (uint32_t)w, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS + (j & 1)));
        }
        if (ok && mbar_wait(bar(L::kBarAcc), 0, abort_flag, &g_bwd_status)) {
            tc_fence_after();
            // warpgroup w writes dQ columns [w D/2, (w + 1) D/2)
            __nv_bfloat16* out = p.dq + (((long long)b * p.Nq + row) * p.Hq + hq) * D + w * (D / 2);
            const bool out_ok =
                row >= p.Nq || in_bounds(out - p.dq, D / 2, (long long)p.B * p.Nq * p.Hq * D, &g_bwd_status);
            uint32_t xo[32];
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tmem_ld32_sync(tmem + lane_base + kDQ + w * (D / 2) + 32 * h, xo);
                if (row < p.Nq && out_ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(xo[8 * c + 0]) * p.scale, __uint_as_float(xo[8 * c + 1]) * p.scale);
                        v.y = pack_bf16(__uint_as_float(xo[8 * c + 2]) * p.scale, __uint_as_float(xo[8 * c + 3]) * p.scale);
                        v.z = pack_bf16(__uint_as_float(xo[8 * c + 4]) * p.scale, __uint_as_float(xo[8 * c + 5]) * p.scale);
                        v.w = pack_bf16(__uint_as_float(xo[8 * c + 6]) * p.scale, __uint_as_float(xo[8 * c + 7]) * p.scale);
                        reinterpret_cast<uint4*>(out + 32 * h)[c] = v;
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
    // The dQ kernel, launched next as a programmatic dependent, reads nothing
    // this kernel writes: let its CTAs take the SMs this grid's last wave frees.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
                if (in_bounds(off + 8 * c, 8, (long long)p.B * p.Nk * p.Hkv * D, &g_bwd_status)) {
                    reinterpret_cast<uint4*>(p.dk + off)[c] = make_uint4(0u, 0u, 0u, 0u);
                    reinterpret_cast<uint4*>(p.dv + off)[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i)
            mbar_init(bar(i), (i == L::kBarDS || i == L::kBarC) ? 2u * kT : 1u);
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

    if (warp < 4) {
      warpgroup_reg_dealloc<kRegsWG0>();
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
        auto ring = [&](int it) { return sbase + L::kOffRing + (it % STAGES) * L::kStage; };
        auto wait_full = [&](int it) {
            if (ok) ok = mbar_wait_warp(bar(L::kBarFull + it % STAGES), (it / STAGES) & 1, abort_flag, &g_bwd_status);
            if (ok) tc_fence_after();
        };
        auto issue_s = [&](int it) {  // S^T = K Q_it^T
            const uint32_t q_lo = sdesc_sw128_lo(ring(it), 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kS, k_lo + off, kHi, q_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_dp = [&](int it) {  // dP^T = V dO_it^T
            const uint32_t do_lo = sdesc_sw128_lo(ring(it) + L::kTile, 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
                mma_ss_elect(tmem + kDP, v_lo + off, kHi, do_lo + off, kHi, kIdSS, kk > 0 ? 1u : 0u);
            }
        };
        wait_full(0);
        if (ok) {
            issue_s(0);
            issue_dp(0);
            tc_commit_elect(bar(L::kBarS));
        }
        for (int it = 0; it < n && ok; ++it) {
            bool s_next = false;  // S^T of the next tile already issued
            if (it + 1 < n) {
                // The elementwise warps hold S^T and dP^T and write P^T, dS^T over
                // dP^T only, so the S columns are free: if the next Q tile is
                // already loaded, its S^T goes to the tensor core now.
                ok = mbar_wait_warp(bar(L::kBarC), it & 1, abort_flag, &g_bwd_status);
                if (!ok) break;
                s_next = __all_sync(0xffffffffu,
                                    mbar_try_wait(bar(L::kBarFull + (it + 1) % STAGES), ((it + 1) / STAGES) & 1));
                if (s_next) {
                    tc_fence_after();
                    issue_s(it + 1);
                }
            }
            ok = mbar_wait_warp(bar(L::kBarDS), it & 1, abort_flag, &g_bwd_status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t qn_lo = sdesc_sw128_lo(ring(it), kNLbo);
            const uint32_t don_lo = sdesc_sw128_lo(ring(it) + L::kTile, kNLbo);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk) {  // 16 query rows = 8 bf16 columns of P^T / dS^T
                const uint32_t r_off = (kk * 16 * 128) >> 4;
                const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                // query rows 16kk..: warpgroup kk / 4 wrote P^T at dP^T column 64 (kk / 4) + 8 (kk % 4)
                // and dS^T 32 columns further
                const uint32_t pc = (kk >> 2) * 64 + (kk & 3) * 8;
                mma_ts_elect(tmem + kDV, tmem + kDP + pc, don_lo + r_off, kHi, kIdAcc, acc);       // dV += P^T dO
                mma_ts_elect(tmem + kDK, tmem + kDP + 32 + pc, qn_lo + r_off, kHi, kIdAcc, acc);  // dK += dS^T Q
            }
            tc_commit_elect(bar(L::kBarEmpty + it % STAGES));  // Q_i and dO_i fully read
            if (it + 1 < n) {
                if (!s_next) {
                    wait_full(it + 1);
                    if (!ok) break;
                    issue_s(it + 1);
                }
                issue_dp(it + 1);  // after dV, dK have read P^T, dS^T (in-order pipe)
                tc_commit_elect(bar(L::kBarS));
            }
            if (it == n - 1) tc_commit_elect(bar(L::kBarAcc));
        }
      }
    } else {
        warpgroup_reg_alloc<kRegsEW>();
        // Two elementwise warpgroups share each key (TMEM lane): warpgroup w
        // takes query rows 64w .. 64w + 63 of every query tile.
        const int w = (warp - 4) >> 2;
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int key = c0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const int tid = threadIdx.x - 128 * (1 + w);  // 0..127 within the warpgroup
        // [buffer][warpgroup][L*log2e | D][64 query rows]
        float* ldbuf = reinterpret_cast<float*>(sgen + L::kOffLD);
        const float sl = p.scale_log2;
        // thread tid stages L (tid < 64) or D (tid >= 64) of query row 64w + tid % 64
        // of head hh (rows past Nq: P = 0)
        auto fetch = [&](int it) {
            const int hh = it_head(it), row = it_tile(it) * kT + 64 * w + (tid & 63);
            float x = tid < 64 ? INFINITY : 0.f;
            if (row < p.Nq && in_bounds(((long long)b * p.Hq + hh) * p.Nq + row, 1,
                                        (long long)p.B * p.Hq * p.Nq, &g_bwd_status)) {
                const long long o = ((long long)b * p.Hq + hh) * p.Nq + row;
                if (tid < 64) {
                    const float l = p.lse[o];
                    x = l == -INFINITY ? INFINITY : l * kLog2e;
                } else {
                    x = p.dvec[o];
                }
            }
            return x;
        };
        float nx = fetch(0);
        bool ok = true;
        // Every thread of the warpgroup runs every iteration, also after a
        // bounded wait has given up (the abort flag then ends the remaining
        // waits at once): the named barrier below must never miss a thread.
        for (int it = 0; it < n; ++it) {
            const int buf = it & 1;
            float* lrow = ldbuf + ((buf * 2 + w) * 2 + 0) * 64;
            float* drow = ldbuf + ((buf * 2 + w) * 2 + 1) * 64;
            (tid < 64 ? lrow : drow)[tid & 63] = nx;
            named_bar_sync(1 + w, 128);  // this iteration's L and D are visible to the warpgroup
            if (it + 1 < n) nx = fetch(it + 1);  // in flight while this tile is processed
            if (ok) ok = mbar_wait(bar(L::kBarS), it & 1, abort_flag, &g_bwd_status);
            if (!ok) continue;
            tc_fence_after();
            const int rq = it_tile(it) * kT;
            // causal: query row i may see this key iff key <= i + (Nk - Nq)
            const bool need_mask = key >= p.Nk || (p.causal && (long long)c0 + kT - 1 > (long long)rq + (p.Nk - p.Nq));
            uint32_t s[64], dp[64];
            tmem_ld64_sync(tmem + lane_base + kS + 64 * w, s);
            tmem_ld64_sync(tmem + lane_base + kDP + 64 * w, dp);
            tc_fence_before();
            mbar_arrive(bar(L::kBarC));  // the S^T columns may be overwritten now
            if (need_mask) {
                // the query rows that may see this key: tile columns [lo, kT)
                const long long first = key >= p.Nk ? (long long)kT
                                                     : (p.causal ? (long long)key - (p.Nk - p.Nq) - rq : 0ll);
                const int lo = first < 0 ? 0 : first > kT ? kT : (int)first;
#pragma unroll
                for (int cc = 0; cc < 64; ++cc)
                    if (64 * w + cc < lo) s[cc] = __float_as_uint(-INFINITY);
            }
            uint32_t pk[32], dk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float pv[2], dsv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int cc = 2 * c + e;  // query row rq + 64w + cc
                    pv[e] = ex2(fmaf(__uint_as_float(s[cc]), sl, -lrow[cc]));
                    dsv[e] = pv[e] * (__uint_as_float(dp[cc]) - drow[cc]);
                }
                pk[c] = pack_bf16(pv[0], pv[1]);
                dk[c] = pack_bf16(dsv[0], dsv[1]);
            }
            // each warpgroup writes only dP^T columns it has read itself
            tmem_st32(tmem + lane_base + kDP + 64 * w, pk);       // P^T
            tmem_st32(tmem + lane_base + kDP + 64 * w + 32, dk);  // dS^T
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS));
        }
        if (ok && mbar_wait(bar(L::kBarAcc), 0, abort_flag, &g_bwd_status)) {
            tc_fence_after();
            // warpgroup w writes columns [w D/2, (w + 1) D/2) of dV and dK
            const long long off = (((long long)b * p.Nk + key) * p.Hkv + g) * D + w * (D / 2);
            const bool out_ok =
                key >= p.Nk || in_bounds(off, D / 2, (long long)p.B * p.Nk * p.Hkv * D, &g_bwd_status);
            uint32_t xo[32];
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tmem_ld32_sync(tmem + lane_base + kDV + w * (D / 2) + 32 * h, xo);
                if (key < p.Nk && out_ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(xo[8 * c + 0]), __uint_as_float(xo[8 * c + 1]));
                        v.y = pack_bf16(__uint_as_float(xo[8 * c + 2]), __uint_as_float(xo[8 * c + 3]));
                        v.z = pack_bf16(__uint_as_float(xo[8 * c + 4]), __uint_as_float(xo[8 * c + 5]));
                        v.w = pack_bf16(__uint_as_float(xo[8 * c + 6]), __uint_as_float(xo[8 * c + 7]));
                        reinterpret_cast<uint4*>(p.dv + off + 32 * h)[c] = v;
                    }
                }
                tmem_ld32_sync(tmem + lane_base + kDK + w * (D / 2) + 32 * h, xo);
                if (key < p.Nk && out_ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(xo[8 * c + 0]) * p.scale, __uint_as_float(xo[8 * c + 1]) * p.scale);
                        v.y = pack_bf16(__uint_as_float(xo[8 * c + 2]) * p.scale, __uint_as_float(xo[8 * c + 3]) * p.scale);
                        v.z = pack_bf16(__uint_as_float(xo[8 * c + 4]) * p.scale, __uint_as_float(xo[8 * c + 5]) * p.scale);
                        v.w = pack_bf16(__uint_as_float(xo[8 * c + 6]) * p.scale, __uint_as_float(xo[8 * c + 7]) * p.scale);
                        reinterpret_cast<uint4*>(p.dk + off + 32 * h)[c] = v;
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
    using LQ = DqLay<D>;
    CUtensorMap mq, mdo, mk, mv;
    if (!attn_host::encode_bshd_map(&mq, q, B, Nq, Hq, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mdo, dout, B, Nq, Hq, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mk, k, B, Nk, Hkv, D, kT, 2) ||
        !attn_host::encode_bshd_map(&mv, v, B, Nk, Hkv, D, kT, 2))
        return ATTN_ERR_CUDA;
    // The register split inside both kernels assumes exactly kLaunchRegs per
    // thread at launch; refuse to launch a build that differs.
    const attn_host::KernelSetup s_dq = attn_host::kernel_setup<bwd_dq_kernel<D>>(LQ::kSmem);
    if (s_dq.err != cudaSuccess) return ATTN_ERR_CUDA;
    const attn_host::KernelSetup s_dkdv = attn_host::kernel_setup<bwd_dkdv_kernel<D>>(L::kSmem);
    if (s_dkdv.err != cudaSuccess) return ATTN_ERR_CUDA;
    if (s_dq.num_regs != kLaunchRegs || s_dkdv.num_regs != kLaunchRegs) return ATTN_ERR_UNSUPPORTED;
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
    const long long dot_rows_per_block = (long long)(kDotThreads / (D / 8)) * kDotRows;
    const long long dot_blocks = (rows + dot_rows_per_block - 1) / dot_rows_per_block;
    const long long dq_blocks = (long long)B * Hq * ((Nq + kT - 1) / kT);
    const long long dkv_blocks = (long long)B * Hkv * ((Nk + kT - 1) / kT);
    if (dot_blocks > 0x7fffffffLL || dq_blocks > 0x7fffffffLL || dkv_blocks > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    bwd_dot_kernel<D><<<(unsigned)dot_blocks, kDotThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                               prm.do_, dvec, B, Nq, Hq);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    bwd_dkdv_kernel<D><<<(unsigned)dkv_blocks, kThreads, L::kSmem, stream>>>(mq, mdo, mk, mv, prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    // dQ depends only on the row sums of bwd_dot_kernel, complete before the
    // dK/dV grid started; as a programmatic dependent of that grid it fills
    // the SMs of its last wave instead of waiting for all of it.  Work queued
    // after this call still waits for both grids.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)dq_blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = LQ::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D>, mq, mdo, mk, mv, prm) == cudaSuccess ? ATTN_OK
                                                                                      : ATTN_ERR_CUDA;
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
