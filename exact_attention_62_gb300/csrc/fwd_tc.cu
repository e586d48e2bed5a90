// fwd_tc.cu -- bf16 exact-attention forward on sm_103a tensor cores.
//
// What it computes: for every query row, O = softmax(scale * q K^T) V over
// the allowed keys and LSE = log sum exp(scale * q K^T) ("algorithm 0" of
// Lecture 11 - Kernel Optimization Techniques, section 2), evaluated tile by
// tile with the online softmax (section 3.1) and deferred normalisation
// (section 3.3): per key tile, m_new = max(m, rowmax S), alpha = exp(m -
// m_new), P = exp(S - m_new), l = alpha l + rowsum P, acc = alpha acc + P V;
// O = acc / l at the end.  This is the loop of the "FlashAttention v1"
// concept pseudocode on the CUDA Kernel course index page, run in the
// query-block-outer order of FlashAttention-2 (Lecture 11, section 4.2).
//
// How (GB300 design; the pages' FA2/FA3 kernels are prior art, not copied):
//  * Persistent: one CTA per SM walks a static list of work units.  A unit
//    is two 128-row query tiles (256 rows) of one (batch, head).  Units are
//    ordered longest first for causal masks and dealt to the CTAs in snake
//    order (c, 2G-1-c, 2G+c, ...), which balances the decreasing unit costs.
//    Consecutive units walk the heads of one batch, so the query heads of a
//    GQA group (which read the same K/V) run side by side and share L2.
//  * Warp 0 (one thread) is the TMA producer: each unit's Q tiles (as soon
//    as the previous unit's last S has read the buffer), then K_j and V_j
//    into separate multi-stage rings that run on across units.
//  * Warp 1 issues every tcgen05.mma (the warp runs convergent, one elected
//    lane issues): S_t = Q_t K_j^T into TMEM and O_t += P_t V_j into TMEM,
//    and signals completion with tcgen05.commit.  Issue order  PV0(j), S0(j+1), PV1(j), S1(j+1)  lets the
//    softmax of one query tile run while the tensor core works on the other
//    (the ping-pong of the FA3 section of the course index, rebuilt around
//    single-thread async MMA and TMEM accumulators); the next unit's first
//    two S products follow the current unit's last PV with no gap.
//  * Warps 4-7 and 8-11 are the softmax warpgroups of query tiles 0 and 1.
//    Each thread owns one row (one TMEM lane): it loads its 128 scores,
//    masks them only on tiles that need it (ragged tail, causal diagonal),
//    applies the online update with exp2 (scale * log2 e folded in), writes
//    P as bf16 into TMEM over the consumed scores (or into shared memory in
//    the debugging variant), rescales its O row in TMEM when the reference
//    max moved, and at the end of a unit loads O, hands the TMEM columns back
//    to the MMA warp at once, and stores O = acc / l and LSE = m + ln l
//    straight to global memory.
//  * Key tiles that are fully masked by causality are never loaded or
//    computed (Lecture 11, section 5.3).
#include <cuda_fp8.h>

#include <cstdio>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

__device__ __forceinline__ long long llmin(long long a, long long b) { return a < b ? a : b; }

// 2^x for two values on the FMA and integer pipes instead of the MUFU unit
// (software exp2, which the FA4 section of Lecture 11 describes for Blackwell;
// this formulation and its polynomial are our own).  x is clamped to >= -125
// (masked scores are -inf; 2^-125 is invisible next to a row sum >= 1), split
// as x = j + f with j = round(x) by adding 1.5 * 2^23 (the sum's low mantissa
// bits then hold j, and f = x - j lies in [-1/2, 1/2]), 2^f comes from a cubic
// whose constant term is exactly 1 (so 2^0 = 1 exactly, as on the MUFU path),
// and j is added into the exponent field: the sum's bit pattern shifted left by
// 23 is exactly j << 23 because the constant's low nine bits are zero.  The
// cubic was fitted for minimax relative error on [-1/2, 1/2] (iteratively
// reweighted least squares): max relative error 1.0e-4 in fp32 arithmetic,
// against the 2^-9 of the bf16 rounding that P goes through next.
constexpr float kExp2C1 = 0.6932829022f;
constexpr float kExp2C2 = 0.2422109842f;
constexpr float kExp2C3 = 0.0550089292f;
__device__ __forceinline__ uint64_t exp2_poly_x2(float x0, float x1) {
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    const uint64_t x = f2_pack(fmaxf(x0, -125.0f), fmaxf(x1, -125.0f));
    const uint64_t t = f2_add(x, f2_pack(kRound, kRound));
    const uint64_t j = f2_add(t, f2_pack(-kRound, -kRound));
    const uint64_t f = f2_fma(j, f2_pack(-1.0f, -1.0f), x);
    uint64_t q = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
    q = f2_fma(q, f, f2_pack(kExp2C1, kExp2C1));
    q = f2_fma(q, f, f2_pack(1.0f, 1.0f));
    const uint32_t r0 = static_cast<uint32_t>(q) + (static_cast<uint32_t>(t) << 23);
    const uint32_t r1 = static_cast<uint32_t>(q >> 32) + (static_cast<uint32_t>(t >> 32) << 23);
    return (static_cast<uint64_t>(r1) << 32) | r0;
}

__device__ unsigned g_fwd_status = 0;
__device__ unsigned long long g_fwd_tiles = 0;

constexpr int kBM = 128;        // query rows per tile (one TMEM lane each)
constexpr int kBN = 128;        // keys per tile
constexpr int kQT = 2;          // query tiles per unit
// 12 warps: warpgroup 0 = producer (warp 0), MMA issuer (warp 1), two idle
// warps; warpgroups 1 and 2 = softmax of query tiles 0 and 1.
constexpr int kThreads = 384;
// Register split.  The kernel is compiled for kLaunchRegs per thread (the
// most 384 threads allow: each SM sub-partition holds three warps of 32 lanes
// and 16384 registers).  Warpgroup 0 then gives registers back and the two
// softmax warpgroups take them: 128 * kRegsWG0 + 256 * kRegsSoftmax must not
// exceed 384 * kLaunchRegs (63488 <= 64512; per sub-partition 112 + 2 * 192 <= 512).
constexpr int kLaunchRegs = 168;
constexpr int kRegsWG0 = 112;
constexpr int kRegsSoftmax = 192;
static_assert(128 * kRegsWG0 + 256 * kRegsSoftmax <= kThreads * kLaunchRegs, "register split");
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 128 B: one 64-column swizzled panel
// In the POLY variant of the kernel every kPolyEvery-th pair of probabilities
// is computed by exp2_poly_x2 (FMA and integer pipes) instead of the MUFU unit.
// Measured on GB300 it is slower at every fraction tried (1/8 .. all): with the
// MUFU unit's doubled exp2 rate the exp loop is bound by instruction issue, not
// by MUFU, so the default kernel keeps every exp2 on MUFU.
constexpr int kPolyEvery = 4;
constexpr float kLn2 = 0.69314718055994530942f;

struct FwdParams {
    float* lse;
    long long lse_ld;  // elements between the LSE rows of consecutive heads (Nq for a whole call)
    __nv_bfloat16* o;
    int B, Hq, Hkv, Nq, Nk, G;
    int causal;
    int num_pairs;
    int num_units;
    float scale_log2;
    float rescale_thr;  // log2 units; 0 = rescale whenever the max grows
    long long wait_limit;  // bound of every mbarrier wait, SM cycles
    int skip_load;         // tests only: ring position whose K/V block 0 never loads (-1: none)
    long long o_slack;     // bounds-checked build, tests only: O's extent taken as this much smaller
    // FP8 inputs only: e4m3 Q and K with one scale per (batch, head, 128-row block)
    const float* q_scales;  // [B, Hq, nqb]
    const float* k_scales;  // [B, Hkv, nkb]
    // FP8 V only: one scale per (batch, KV head)
    const float* v_scales;  // [B, Hkv]
    int nqb, nkb;
};

template <int D, bool P_TMEM, bool F8 = false, bool F8V = false>
struct Layout {
    // Q and K are bf16 or (F8) e4m3.  A swizzled panel is 128 rows of 128
    // bytes: 64 bf16 or 128 e4m3 elements per row.  V is bf16, [keys][D]
    // in D/64 panels, or (F8V) e4m3 and transposed, [D][128 keys]: one panel
    // of D rows, K-major like K.
    static constexpr int kQKElem = F8 ? 1 : 2;
    static constexpr int kQKPanels = D * kQKElem / 128;
    static constexpr int kPanels = D / 64;  // V panels (bf16 V: 64 columns each)
    static_assert(F8V || kPanels * 64 == D, "bf16 V in whole 64-column panels");
    static constexpr int kQBytes = kBM * D * kQKElem;
    static constexpr int kKBytes = kBN * D * kQKElem;
    static constexpr int kKVBytes = kBN * D * (F8V ? 1 : 2);  // one V tile
    static_assert(!F8V || (F8 && P_TMEM), "e4m3 V goes with e4m3 Q, K and P in tensor memory");
    static constexpr int kPBytes = P_TMEM ? 0 : kBM * kBN * 2;
    static constexpr int kKSt = F8 ? 3 : P_TMEM ? (D == 128 ? 2 : 3) : (D == 128 ? 1 : 2);
    static constexpr int kVSt = kKSt;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQT * kQBytes;
    static constexpr int kOffK = kOffP + kQT * kPBytes;
    static constexpr int kOffV = kOffK + kKSt * kKBytes;
    static constexpr int kOffBar = kOffV + kVSt * kKVBytes;
    static constexpr int kBarQFull = 0;
    static constexpr int kBarQEmpty = kBarQFull + kQT;
    static constexpr int kBarKFull = kBarQEmpty + kQT;
    static constexpr int kBarKEmpty = kBarKFull + kKSt;
    static constexpr int kBarVFull = kBarKEmpty + kKSt;
    static constexpr int kBarVEmpty = kBarVFull + kVSt;
    static constexpr int kBarSFull = kBarVEmpty + kVSt;
    static constexpr int kBarPFull = kBarSFull + kQT;
    static constexpr int kBarOFull = kBarPFull + kQT;
    static constexpr int kBarOEmpty = kBarOFull + kQT;
    static constexpr int kNumBars = kBarOEmpty + kQT;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    // TMEM columns: S_0, S_1 (128 fp32 each; P_t overwrites the first 64 of
    // S_t when it lives in TMEM), then O_0, O_1 (D fp32 each).
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return t ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    static constexpr uint32_t kTmemCols = 512;
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // 128 threads arrive per phase on these; one arrival (expect_tx or commit) on the rest
    __host__ __device__ static constexpr bool per_thread_bar(int i) {
        return (i >= kBarPFull && i < kBarPFull + kQT) || (i >= kBarOEmpty && i < kBarOEmpty + kQT);
    }
};

// One work unit: 256 query rows of one (batch, head) and the key-tile count
// of each of its two 128-row tiles.
struct Unit {
    int b, hq, g, row0;
    int n[kQT];
};

// Number of key tiles a 128-row query tile starting at row `rs` must visit.
__device__ __forceinline__ int kv_tiles_for(int rs, const FwdParams& p) {
    if (rs >= p.Nq) return 0;
    if (!p.causal) return (p.Nk + kBN - 1) / kBN;
    const int re = min(rs + kBM, p.Nq) - 1;
    const long long last = llmin((long long)p.Nk - 1, (long long)re + (p.Nk - p.Nq));
    return last < 0 ? 0 : (int)(last / kBN) + 1;
}

// The k-th unit of this CTA (snake order over a longest-first list), or -1.
__device__ __forceinline__ int unit_index(int k, const FwdParams& p) {
    const int G = gridDim.x, c = blockIdx.x;
    const long long u = (long long)k * G + ((k & 1) ? (G - 1 - c) : c);
    return u < p.num_units ? (int)u : -1;
}

__device__ __forceinline__ Unit unit_at(int u, const FwdParams& p) {
    const int BH = p.B * p.Hq;
    const int bh = u % BH;
    const int pr = u / BH;
    const int pair = p.causal ? (p.num_pairs - 1 - pr) : pr;
    Unit x;
    x.hq = bh % p.Hq;
    x.b = bh / p.Hq;
    x.g = x.hq / p.G;
    x.row0 = pair * (kQT * kBM);
#pragma unroll
    for (int t = 0; t < kQT; ++t) x.n[t] = kv_tiles_for(x.row0 + t * kBM, p);
    return x;
}

template <int D, bool P_TMEM, bool POLY, bool F8, bool F8V>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = Layout<D, P_TMEM, F8, F8V>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc + 4);

    // ---- set-up: barriers, TMEM
    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), L::per_thread_bar(i) ? 128u : 1u);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::kOffMisc, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp < 4) {
      warpgroup_reg_dealloc<kRegsWG0>();
      if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int kv = 0;                 // key tiles loaded so far (ring position)
            int q_loads[kQT] = {0, 0};  // Q_t loads so far
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int u = unit_index(k, p);
                if (u < 0) break;
                const Unit x = unit_at(u, p);
                for (int t = 0; t < kQT && ok; ++t) {
                    if (x.n[t] == 0) continue;
                    if (q_loads[t] > 0)  // the previous unit's last S_t has read Q_t
                        ok = mbar_wait(bar(L::kBarQEmpty + t), (q_loads[t] - 1) & 1, abort_flag,
                                       &g_fwd_status, p.wait_limit);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(L::kBarQFull + t), L::kQBytes);
                    for (int pp = 0; pp < L::kQKPanels; ++pp)
                        tma_load_4d(sbase + L::kOffQ + t * L::kQBytes + pp * kPanelBytes, &tmQ,
                                    bar(L::kBarQFull + t), (128 / L::kQKElem) * pp, x.hq,
                                    x.row0 + t * kBM, x.b);
                    ++q_loads[t];
                }
                const int n = max(x.n[0], x.n[1]);
                for (int j = 0; j < n && ok; ++j, ++kv) {
                    // Fault injection for tests: block 0 never loads ring position
                    // skip_load, so the waits for it run out (production: -1).
                    const bool skip = kv == p.skip_load && blockIdx.x == 0;
                    const int ks = kv % L::kKSt;
                    ok = mbar_wait(bar(L::kBarKEmpty + ks), ((kv / L::kKSt) & 1) ^ 1, abort_flag,
                                   &g_fwd_status, p.wait_limit);
                    if (!ok) break;
                    if (!skip) {
                        mbar_arrive_expect_tx(bar(L::kBarKFull + ks), L::kKBytes);
                        for (int pp = 0; pp < L::kQKPanels; ++pp)
                            tma_load_4d(sbase + L::kOffK + ks * L::kKBytes + pp * kPanelBytes, &tmK,
                                        bar(L::kBarKFull + ks), (128 / L::kQKElem) * pp, x.g, j * kBN, x.b);
                    }
                    const int vs = kv % L::kVSt;
                    ok = mbar_wait(bar(L::kBarVEmpty + vs), ((kv / L::kVSt) & 1) ^ 1, abort_flag,
                                   &g_fwd_status, p.wait_limit);
                    if (!ok) break;
                    if (!skip) {
                        mbar_arrive_expect_tx(bar(L::kBarVFull + vs), L::kKVBytes);
                        if constexpr (F8V)  // V^T [b][g][D rows][keys]: 128 keys x D rows
                            tma_load_4d(sbase + L::kOffV + vs * L::kKVBytes, &tmV, bar(L::kBarVFull + vs),
                                        j * kBN, 0, x.g, x.b);
                        else
                            for (int pp = 0; pp < L::kPanels; ++pp)
                                tma_load_4d(sbase + L::kOffV + vs * L::kKVBytes + pp * kPanelBytes, &tmV,
                                            bar(L::kBarVFull + vs), 64 * pp, x.g, j * kBN, x.b);
                    }
                }
            }
        }
      } else if (warp == 1) {
        // ================================================= MMA issuer
        // The whole warp runs the issue loop convergent, so addresses and
        // descriptors stay warp-uniform, and one elected lane issues every
        // tcgen05 instruction.  Each buffer's descriptor is built once; a
        // k-step only adds a compile-time offset (16-byte units) to its
        // start-address field.  Keeping the issue path this short matters: the
        // warp shares its SM sub-partition with two busy softmax warps.
        {
            constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t kIdS8 = idesc_e4m3_f32(kBM, kBN);
            constexpr uint32_t kIdPV = idesc_bf16_f32(kBM, D, true);
            constexpr uint32_t kIdPV8 = idesc_e4m3_f32(kBM, D);  // e4m3 P (TMEM) times e4m3 V^T
            constexpr uint32_t kHi = sdesc_sw128_hi(1024);  // every operand: 8-row groups 1024 B apart
            // V is [keys][D] with D contiguous: an N-major B operand.  Along N the
            // 64-column panels are kPanelBytes apart (LBO; one panel when D = 64);
            // along K every 8 keys are 1024 B apart (SBO).
            constexpr uint32_t kVLbo = D == 128 ? kPanelBytes : 1024;
            auto wait = [&](uint32_t b, uint32_t parity) {
                return mbar_wait_warp(b, parity, abort_flag, &g_fwd_status, p.wait_limit);
            };
            bool ok = true;
            int kv = 0;                     // ring position of the unit's first key tile
            int q_waits[kQT] = {0, 0};      // Q_t phases consumed
            int p_waits[kQT] = {0, 0};      // P_t phases consumed
            int units_t[kQT] = {0, 0};      // units in which tile t was active
            unsigned long long tiles = 0;
            for (int k = 0; ok; ++k) {
                const int u = unit_index(k, p);
                if (u < 0) break;
                const Unit x = unit_at(u, p);
                const int n = max(x.n[0], x.n[1]);
                for (int t = 0; t < kQT && ok; ++t) {
                    if (x.n[t] == 0) continue;
                    ok = wait(bar(L::kBarQFull + t), q_waits[t] & 1);
                    ++q_waits[t];
                }
                int k_ready = -1, v_ready = -1;
                auto wait_k = [&](int j) {
                    if (ok && j > k_ready) {
                        const int r = kv + j;
                        ok = wait(bar(L::kBarKFull + r % L::kKSt), (r / L::kKSt) & 1);
                        tc_fence_after();
                        k_ready = j;
                    }
                };
                auto wait_v = [&](int j) {
                    if (ok && j > v_ready) {
                        const int r = kv + j;
                        ok = wait(bar(L::kBarVFull + r % L::kVSt), (r / L::kVSt) & 1);
                        tc_fence_after();
                        v_ready = j;
                    }
                };
                // S_t = Q_t K_j^T  (M=128 rows, N=128 keys, K=D in steps of 16)
                auto issue_s = [&](int t, int j) {
                    wait_k(j);
                    if (!ok) return;
                    const uint32_t q_lo = sdesc_sw128_lo(sbase + L::kOffQ + t * L::kQBytes, 16);
                    const uint32_t k_lo =
                        sdesc_sw128_lo(sbase + L::kOffK + ((kv + j) % L::kKSt) * L::kKBytes, 16);
                    const uint32_t dS = tmem + L::tm_s(t);
                    // a k-step is 32 bytes of each row: 16 bf16 or 32 e4m3 elements
                    constexpr int kSteps = F8 ? D / 32 : D / 16;
#pragma unroll
                    for (int kk = 0; kk < kSteps; ++kk) {
                        const uint32_t off = ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
                        if constexpr (F8)
                            mma_ss_elect_f8(dS, q_lo + off, kHi, k_lo + off, kHi, kIdS8, kk > 0 ? 1u : 0u);
                        else
                            mma_ss_elect(dS, q_lo + off, kHi, k_lo + off, kHi, kIdS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_elect(bar(L::kBarSFull + t));
                    if (j == x.n[t] - 1) tc_commit_elect(bar(L::kBarQEmpty + t));  // Q_t fully read
                };
                // O_t += P_t V_j  (M=128 rows, N=D, K=128 keys in steps of 16)
                auto issue_pv = [&](int t, int j) {
                    wait_v(j);
                    if (!ok) return;
                    ok = wait(bar(L::kBarPFull + t), p_waits[t] & 1);
                    ++p_waits[t];
                    if (ok && j == 0 && units_t[t] > 0)  // previous unit's epilogue read O_t
                        ok = wait(bar(L::kBarOEmpty + t), (units_t[t] - 1) & 1);
                    if (!ok) return;
                    tc_fence_after();
                    const uint32_t dO = tmem + L::tm_o(t);
                    if constexpr (F8V) {
                        // V^T is K-major like K: a k-step is 32 keys, 32 bytes of each of
                        // its D rows; P packs four e4m3 keys per 32-bit column, 8 columns
                        const uint32_t v_lo =
                            sdesc_sw128_lo(sbase + L::kOffV + ((kv + j) % L::kVSt) * L::kKVBytes, 16);
#pragma unroll
                        for (int kk = 0; kk < kBN / 32; ++kk)
                            mma_ts_elect_f8(dO, tmem + L::tm_s(t) + kk * 8, v_lo + ((kk * 32) >> 4), kHi,
                                            kIdPV8, (j > 0 || kk > 0) ? 1u : 0u);
                        if (j == x.n[t] - 1) {
                            tc_commit_elect(bar(L::kBarOFull + t));
                            ++units_t[t];
                        }
                        return;
                    }
                    const uint32_t v_lo =
                        sdesc_sw128_lo(sbase + L::kOffV + ((kv + j) % L::kVSt) * L::kKVBytes, kVLbo);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint32_t v_off = (kk * 16 * 128) >> 4;  // 16 keys of 128 B rows
                        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (P_TMEM) {
                            // bf16 P packed two per 32-bit column: 16 keys = 8 columns
                            mma_ts_elect(dO, tmem + L::tm_s(t) + kk * 8, v_lo + v_off, kHi, kIdPV, acc);
                        } else {
                            const uint32_t p_lo = sdesc_sw128_lo(sbase + L::kOffP + t * L::kPBytes, 16);
                            const uint32_t off = ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
                            mma_ss_elect(dO, p_lo + off, kHi, v_lo + v_off, kHi, kIdPV, acc);
                        }
                    }
                    if (j == x.n[t] - 1) {
                        tc_commit_elect(bar(L::kBarOFull + t));
                        ++units_t[t];
                    }
                };
                if (x.n[0] > 0) issue_s(0, 0);
                if (x.n[1] > 0) issue_s(1, 0);
                if (n > 0 && ok) tc_commit_elect(bar(L::kBarKEmpty + kv % L::kKSt));
                for (int j = 0; j < n && ok; ++j) {
                    if (j < x.n[0]) issue_pv(0, j);
                    if (j + 1 < x.n[0]) issue_s(0, j + 1);
                    if (j < x.n[1]) issue_pv(1, j);
                    if (ok) tc_commit_elect(bar(L::kBarVEmpty + (kv + j) % L::kVSt));
                    if (j + 1 < x.n[1]) issue_s(1, j + 1);
                    if (j + 1 < n && ok) tc_commit_elect(bar(L::kBarKEmpty + (kv + j + 1) % L::kKSt));
                }
                kv += n;
                tiles += (unsigned long long)(x.n[0] + x.n[1]);
            }
            if (ok && tiles && lane == 0) atomicAdd(&g_fwd_tiles, tiles);
        }
      }
    } else {
        warpgroup_reg_alloc<kRegsSoftmax>();
        // ================================================= softmax warpgroups
        const int t = (warp - 4) >> 2;
        const int q4 = warp & 3;  // TMEM lane quarter this warp may access
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const uint32_t tS = tmem + lane_base + L::tm_s(t);
        const uint32_t tO = tmem + lane_base + L::tm_o(t);
        const float sl = p.scale_log2;
        int s_waits = 0, o_waits = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int u = unit_index(k, p);
            if (u < 0) break;
            const Unit x = unit_at(u, p);
            const int rs = x.row0 + t * kBM;
            const int row = rs + r;
            const int nt = x.n[t];
            __nv_bfloat16* orow = p.o + (((long long)x.b * p.Nq + row) * p.Hq + x.hq) * D;
            float* lse_out = p.lse + ((long long)x.b * p.Hq + x.hq) * p.lse_ld + row;
            // (bounds-checked build) the row's D outputs and its LSE, inside O and LSE
            auto o_row_ok = [&]() {
                return in_bounds(orow - p.o, D, (long long)p.B * p.Nq * p.Hq * D - p.o_slack, &g_fwd_status);
            };
            auto lse_ok = [&]() {
                return in_bounds(lse_out - p.lse, 1, ((long long)p.B * p.Hq - 1) * p.lse_ld + p.Nq,
                                 &g_fwd_status);
            };
            if (nt == 0) {
                // Tile beyond Nq, or rows with no allowed key at all.
                if (row < p.Nq) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    if (o_row_ok()) {
#pragma unroll
                        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                    }
                    if (lse_ok()) *lse_out = -INFINITY;
                }
                continue;
            }
            const long long diag = (long long)row + (p.Nk - p.Nq);  // last causal key of the row
            const long long diag_tile = (long long)rs + (p.Nk - p.Nq);
            // FP8: S from the e4m3 codes is rescaled by the tile's q-block and k-block scales
            float q_block_scale = 1.f;
            const float* k_block_scale = nullptr;
            if constexpr (F8) {
                q_block_scale = p.q_scales[((long long)x.b * p.Hq + x.hq) * p.nqb + rs / kBM];
                k_block_scale = p.k_scales + ((long long)x.b * p.Hkv + x.g) * p.nkb;
            }
            // FP8 V: P is formed as 2^kPExp P and O = acc * v_scale / l
            constexpr float kPExp = F8V ? 8.f : 0.f;
            float v_scale = 1.f;
            if constexpr (F8V) v_scale = p.v_scales[(long long)x.b * p.Hkv + x.g];
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < nt; ++j) {
                float slj = sl;
                if constexpr (F8) slj = sl * q_block_scale * k_block_scale[j];
                if (!mbar_wait(bar(L::kBarSFull + t), s_waits & 1, abort_flag, &g_fwd_status, p.wait_limit)) {
                    ok = false;
                    break;
                }
                ++s_waits;
                tc_fence_after();
                uint32_t s[kBN];
                tmem_ld128_sync(tS, s);
                const int col0 = j * kBN;
                const bool need_mask = (col0 + kBN > p.Nk) ||
                                       (p.causal && (long long)(col0 + kBN - 1) > diag_tile);
                if (need_mask) {
                    // The allowed keys of a row form a prefix of the tile: columns
                    // [0, lim) with lim = min(Nk, last causal key + 1) - col0, clamped
                    // to [0, kBN].  One compare against a constant per score.
                    long long end = p.Nk;
                    if (p.causal && diag + 1 < end) end = diag + 1;
                    end -= col0;
                    const int lim = end < 0 ? 0 : end > kBN ? kBN : (int)end;
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c >= lim) s[c] = __float_as_uint(-INFINITY);
                }
                // row max: 8 independent chains of three-input maxima
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    mx[i] = fmax3(__uint_as_float(s[i]), __uint_as_float(s[i + 8]),
                                  __uint_as_float(s[i + 16]));
#pragma unroll
                    for (int c = 24; c < 120; c += 16)
                        mx[i] = fmax3(mx[i], __uint_as_float(s[c + i]), __uint_as_float(s[c + 8 + i]));
                    mx[i] = fmaxf(mx[i], __uint_as_float(s[120 + i]));
                }
                const float m_tile = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                                 mx[6]), mx[7]) * slj;
                // The reference max moves only when the tile's max exceeds it by more
                // than rescale_thr (log2 units; 0 = whenever it grows).  acc and l always
                // share the reference, so O = acc / l and LSE = m + log l are exact for
                // any threshold; a stale reference only bounds P by 2^rescale_thr.
                float m_new = m, alpha = 1.f;
                if (m_tile > m + p.rescale_thr) {
                    m_new = m_tile;
                    alpha = ex2(m - m_new);  // 0 on the first non-empty tile
                }
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                // P = exp2(s * scale log2 e - m): the scale-subtract and the row sum run on
                // packed fp32 pairs, exp2 on the MUFU unit.
                // FP8 V: P is formed as 256 P (2^8 folded into the subtrahend), so
                // that its e4m3 codes keep three mantissa bits down to P = 2^-14; l
                // then sums 256 P and the epilogue takes the 8 back out of the LSE.
                const uint64_t sl2 = f2_pack(slj, slj);
                const float nm = F8V ? kPExp - m_use : -m_use;
                const uint64_t nm2 = f2_pack(nm, nm);
                uint64_t sum2[2] = {0ull, 0ull};
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) {
                    const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[2 * c]),
                                                      __uint_as_float(s[2 * c + 1])), sl2, nm2);
                    float p0, p1;
                    if (POLY && c % kPolyEvery == kPolyEvery - 1) {
                        const uint64_t y = exp2_poly_x2(f2_lo(x), f2_hi(x));
                        p0 = f2_lo(y);
                        p1 = f2_hi(y);
                    } else {
                        p0 = ex2(f2_lo(x));
                        p1 = ex2(f2_hi(x));
                    }
                    sum2[c & 1] = f2_add(sum2[c & 1], f2_pack(p0, p1));
                    if constexpr (F8V) {
                        // e4m3, round to nearest even, saturating: four keys per word
                        const uint32_t q2 = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE,
                                                                     __NV_E4M3);
                        if (c & 1)
                            pk[c >> 1] |= q2 << 16;
                        else
                            pk[c >> 1] = q2;
                        if (c == 31) tmem_st16(tS, pk);  // keys 0-63 out while computing the rest
                    } else {
                        pk[c] = pack_bf16(p0, p1);
                        if constexpr (P_TMEM) {
                            if (c == 31) tmem_st32(tS, pk);  // first half out while computing the rest
                        }
                    }
                }
                const uint64_t sum = f2_add(sum2[0], sum2[1]);
                // While a row has no finite score its "probabilities" are the
                // polynomial's clamped 2^-125, not 0: they must not count.  (acc
                // gets only such values; a later finite score rescales it by
                // alpha = 0, and with l = 0 the row's O is 0 and its LSE -inf.)
                const float tile_sum = m_new == -INFINITY ? 0.f : f2_lo(sum) + f2_hi(sum);
                l = fmaf(l, alpha, tile_sum);
                if constexpr (F8V) {
                    tmem_st16(tS + 16, pk + 16);
                } else if constexpr (P_TMEM) {
                    tmem_st32(tS + 32, pk + 32);
                } else {
                    const uint32_t pa = sbase + L::kOffP + t * L::kPBytes;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {  // 16 chunks of 8 keys
                        const int panel = c >> 3, cc = c & 7;
                        st_shared_v4(pa + panel * kPanelBytes + r * 128 + ((cc ^ (r & 7)) << 4),
                                     pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                    fence_proxy_async_smem();
                }
                // O_t holds the sum through key tile j-1 (its PV completed before S_t(j)
                // did); bring it to the new reference if some row of the warp moved.
                // One TMEM round trip, packed multiplies.
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    uint32_t xo[D];
                    if constexpr (D == 128)
                        tmem_ld128_sync(tO, xo);
                    else
                        tmem_ld64_sync(tO, xo);
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int i = 0; i < D / 2; ++i) {
                        const uint64_t y = f2_mul(f2_pack(__uint_as_float(xo[2 * i]),
                                                          __uint_as_float(xo[2 * i + 1])), a2);
                        xo[2 * i] = __float_as_uint(f2_lo(y));
                        xo[2 * i + 1] = __float_as_uint(f2_hi(y));
                    }
#pragma unroll
                    for (int c = 0; c < D; c += 32) tmem_st32(tO + c, xo + c);
                }
                tmem_st_wait();  // P and any rescaled O are in TMEM before the MMA is told
                tc_fence_before();
                mbar_arrive(bar(L::kBarPFull + t));
                m = m_new;
            }
            if (!ok) break;
            // ---- epilogue: O = acc / l, LSE = m + ln l
            if (!mbar_wait(bar(L::kBarOFull + t), o_waits & 1, abort_flag, &g_fwd_status, p.wait_limit)) {
                ok = false;
                break;
            }
            ++o_waits;
            tc_fence_after();
            uint32_t xo[D];
            tmem_ld64_sync(tO, xo);
            if constexpr (D == 128) tmem_ld64_sync(tO + 64, xo + 64);
            tc_fence_before();
            mbar_arrive(bar(L::kBarOEmpty + t));  // the next unit's PV may overwrite O_t now
            if (row < p.Nq && o_row_ok()) {
                const float inv = l > 0.f ? v_scale / l : 0.f;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(xo[8 * c + 0]) * inv, __uint_as_float(xo[8 * c + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(xo[8 * c + 2]) * inv, __uint_as_float(xo[8 * c + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(xo[8 * c + 4]) * inv, __uint_as_float(xo[8 * c + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(xo[8 * c + 6]) * inv, __uint_as_float(xo[8 * c + 7]) * inv);
                    reinterpret_cast<uint4*>(orow)[c] = w;
                }
            }
            if (row < p.Nq && lse_ok()) *lse_out = l > 0.f ? (m + lg2(l) - kPExp) * kLn2 : -INFINITY;
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool P_TMEM, bool POLY, bool F8 = false, bool F8V = false>
attn_status_t launch_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int Hq, int Hkv, int Nq, int Nk, float scale, int causal,
                          cudaStream_t stream, const attn_test_options_t* test, long long lse_ld,
                          const float* q_scales = nullptr, const float* k_scales = nullptr,
                          const float* v_scales = nullptr) {
    using L = Layout<D, P_TMEM, F8, F8V>;
    CUtensorMap mq, mk, mv;
    const bool v_ok = F8V ? attn_host::encode_vt_map(&mv, v, B, Hkv, D, attn_host::fp8_v_ld(Nk), kBN)
                          : attn_host::encode_bshd_map(&mv, v, B, Nk, Hkv, D, kBN, 2);
    if (!attn_host::encode_bshd_map(&mq, q, B, Nq, Hq, D, kBM, L::kQKElem) ||
        !attn_host::encode_bshd_map(&mk, k, B, Nk, Hkv, D, kBN, L::kQKElem) || !v_ok)
        return ATTN_ERR_CUDA;
    // The register split inside the kernel assumes exactly kLaunchRegs per
    // thread at launch; refuse to launch a build that differs (the split's
    // register increase would otherwise wait forever).
    const attn_host::KernelSetup ks =
        attn_host::kernel_setup<fwd_tc_kernel<D, P_TMEM, POLY, F8, F8V>>(L::kSmemBytes);
    if (ks.err != cudaSuccess) return ATTN_ERR_CUDA;
    if (ks.num_regs != kLaunchRegs) return ATTN_ERR_UNSUPPORTED;
    FwdParams prm;
    prm.lse = lse;
    prm.lse_ld = lse_ld > 0 ? lse_ld : Nq;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    prm.causal = causal;
    prm.num_pairs = (Nq + kQT * kBM - 1) / (kQT * kBM);
    const long long units = (long long)prm.num_pairs * B * Hq;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    prm.num_units = (int)units;
    prm.scale_log2 = scale * 1.4426950408889634f;
    // Production: rescale whenever the max grows (tau = 0) and the standard
    // wait bound.  tau = 0 keeps the dominant P entry of a near one-hot row at
    // exactly 1, so bf16 rounding of P adds no error there.
    prm.rescale_thr = test ? test->rescale_threshold : 0.0f;
    prm.wait_limit = (test && test->wait_limit_cycles > 0) ? test->wait_limit_cycles : kWaitLimitCycles;
    prm.skip_load = test ? test->skip_load : -1;
    prm.o_slack = test ? test->o_extent_slack : 0;
    prm.q_scales = q_scales;
    prm.k_scales = k_scales;
    prm.v_scales = v_scales;
    prm.nqb = (Nq + kBM - 1) / kBM;
    prm.nkb = (Nk + kBN - 1) / kBN;
    const int sms = attn_host::device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const int grid = (int)(units < sms ? units : sms);
    fwd_tc_kernel<D, P_TMEM, POLY, F8, F8V><<<grid, kThreads, L::kSmemBytes, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_host {

attn_status_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, cudaStream_t stream, const attn_test_options_t* test,
                            long long lse_ld) {
    // Production: P in tensor memory, every exponential on MUFU.  The other
    // variants are reached only through attn_fwd_test.
    const bool smem_p = test && test->p_in_smem;
    const bool poly = test && test->exp2_poly;
    if (d == 128)
        return smem_p ? launch_impl<128, false, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld)
               : poly ? launch_impl<128, true, true>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld)
                      : launch_impl<128, true, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld);
    if (d == 64)
        return smem_p ? launch_impl<64, false, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld)
               : poly ? launch_impl<64, true, true>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld)
                      : launch_impl<64, true, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, test, lse_ld);
    return ATTN_ERR_UNSUPPORTED;
}

attn_status_t launch_fwd_fp8(const void* q8, const void* k8, const void* v, const float* q_scales,
                             const float* k_scales, void* o, float* lse, int B, int Hq, int Hkv,
                             int Nq, int Nk, int d, int causal, float scale, cudaStream_t stream) {
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    return launch_impl<128, true, false, true>(q8, k8, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal,
                                               stream, nullptr, 0, q_scales, k_scales);
}

attn_status_t launch_fwd_fp8_pv(const void* q8, const void* k8, const void* vt8, const float* q_scales,
                                const float* k_scales, const float* v_scales, void* o, float* lse, int B,
                                int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                                cudaStream_t stream) {
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    return launch_impl<128, true, false, true, true>(q8, k8, vt8, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal,
                                                     stream, nullptr, 0, q_scales, k_scales, v_scales);
}

cudaError_t fwd_tc_read_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_fwd_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(unsigned));
}

cudaError_t fwd_tc_read_tiles(unsigned long long* out, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_fwd_tiles, sizeof(unsigned long long));
    if (e != cudaSuccess || !reset) return e;
    const unsigned long long zero = 0;
    return cudaMemcpyToSymbol(g_fwd_tiles, &zero, sizeof(unsigned long long));
}

}  // namespace attn_host
