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
//  * One CTA owns two 128-row query tiles of one (batch, head) -- 256 rows.
//    Consecutive CTAs walk the heads of one batch, so the query heads of a
//    GQA group (which read the same K/V) run side by side and share L2.
//    For causal masks the longest row blocks are scheduled first.
//  * Warp 0 (one thread) is the TMA producer: both Q tiles once, then K_j
//    and V_j into separate multi-stage rings (mbarrier full/empty pairs).
//  * Warp 1 (one thread) issues every tcgen05.mma: S_t = Q_t K_j^T into TMEM
//    and O_t += P_t V_j into TMEM, and signals completion with
//    tcgen05.commit.  Issue order  PV0(j), S0(j+1), PV1(j), S1(j+1)  lets the
//    softmax of one query tile run while the tensor core works on the other
//    (the ping-pong of the FA3 section of the course index, rebuilt around
//    single-thread async MMA and TMEM accumulators).
//  * Warps 2-5 and 6-9 are the softmax warpgroups of query tiles 0 and 1.
//    Each thread owns one row (one TMEM lane): it loads its 128 scores,
//    masks them only on tiles that need it (ragged tail, causal diagonal),
//    applies the online update with exp2 (scale * log2 e folded in), writes
//    P as bf16 (into TMEM over the consumed scores, or into shared memory),
//    rescales its O row in TMEM only when the running max grew by more than a
//    threshold (the conditional rescale of the FA4 section of the course
//    index; exact, see below), and at the end
//    writes O = acc / l through shared memory with a TMA store and LSE =
//    m + ln l.
//  * Key tiles that are fully masked by causality are never loaded or
//    computed (Lecture 11, section 5.3).
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

__device__ __forceinline__ long long llmin(long long a, long long b) { return a < b ? a : b; }

__device__ unsigned g_fwd_status = 0;
__device__ unsigned long long g_fwd_tiles = 0;

constexpr int kBM = 128;        // query rows per tile (one TMEM lane each)
constexpr int kBN = 128;        // keys per tile
constexpr int kQT = 2;          // query tiles per CTA
constexpr int kThreads = 320;   // 10 warps
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 128 B: one 64-column swizzled panel
constexpr float kLn2 = 0.69314718055994530942f;

struct FwdParams {
    float* lse;
    __nv_bfloat16* o;  // only for rows that have no allowed key
    int B, Hq, Hkv, Nq, Nk, G;
    int causal;
    int num_pairs;
    float scale_log2;
    float rescale_thr;  // log2 units; 0 = rescale whenever the max grows
};

template <int D, bool P_TMEM>
struct Layout {
    static constexpr int kPanels = D / 64;
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kKVBytes = kBN * D * 2;
    static constexpr int kPBytes = P_TMEM ? 0 : kBM * kBN * 2;
    static constexpr int kKSt = P_TMEM ? (D == 128 ? 2 : 3) : (D == 128 ? 1 : 2);
    static constexpr int kVSt = kKSt;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQT * kQBytes;
    static constexpr int kOffK = kOffP + kQT * kPBytes;
    static constexpr int kOffV = kOffK + kKSt * kKVBytes;
    static constexpr int kOffBar = kOffV + kVSt * kKVBytes;
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = kBarQFull + kQT;
    static constexpr int kBarKEmpty = kBarKFull + kKSt;
    static constexpr int kBarVFull = kBarKEmpty + kKSt;
    static constexpr int kBarVEmpty = kBarVFull + kVSt;
    static constexpr int kBarSFull = kBarVEmpty + kVSt;
    static constexpr int kBarPFull = kBarSFull + kQT;
    static constexpr int kBarOFull = kBarPFull + kQT;
    static constexpr int kBarStaged = kBarOFull + kQT;
    static constexpr int kNumBars = kBarStaged + kQT;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    // TMEM columns: S_0, S_1 (128 fp32 each; P_t overwrites the first 64 of
    // S_t when it lives in TMEM), then O_0, O_1 (D fp32 each).
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return t ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    static constexpr uint32_t kTmemCols = 512;
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Number of key tiles a 128-row query tile starting at row `rs` must visit.
__device__ __forceinline__ int kv_tiles_for(int rs, const FwdParams& p) {
    if (rs >= p.Nq) return 0;
    if (!p.causal) return (p.Nk + kBN - 1) / kBN;
    const int re = min(rs + kBM, p.Nq) - 1;
    const long long last = llmin((long long)p.Nk - 1, (long long)re + (p.Nk - p.Nq));
    return last < 0 ? 0 : (int)(last / kBN) + 1;
}

template <int D, bool P_TMEM>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
    using L = Layout<D, P_TMEM>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * (uint32_t)i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc + 4);

    // ---- work unit: (pair of query tiles, head, batch)
    const int BH = p.B * p.Hq;
    const int bh = blockIdx.x % BH;
    const int pr = blockIdx.x / BH;
    const int pair = p.causal ? (p.num_pairs - 1 - pr) : pr;
    const int hq = bh % p.Hq;
    const int b = bh / p.Hq;
    const int g = hq / p.G;
    const int row0 = pair * (kQT * kBM);
    int n_t[kQT];
#pragma unroll
    for (int t = 0; t < kQT; ++t) n_t[t] = kv_tiles_for(row0 + t * kBM, p);
    const int n = max(n_t[0], n_t[1]);

    // ---- set-up: barriers, TMEM
    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kNumBars; ++i) {
            const bool per_thread = (i >= L::kBarPFull && i < L::kBarPFull + kQT) ||
                                    (i >= L::kBarStaged && i < L::kBarStaged + kQT);
            mbar_init(bar(i), per_thread ? 128u : 1u);
        }
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

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmO);
            for (int t = 0; t < kQT; ++t) {
                if (n_t[t] == 0) continue;
                mbar_arrive_expect_tx(bar(L::kBarQFull + t), L::kQBytes);
                for (int pp = 0; pp < L::kPanels; ++pp)
                    tma_load_4d(sbase + L::kOffQ + t * L::kQBytes + pp * kPanelBytes, &tmQ,
                                bar(L::kBarQFull + t), 64 * pp, hq, row0 + t * kBM, b);
            }
            for (int j = 0; j < n; ++j) {
                const int ks = j % L::kKSt;
                if (!mbar_wait(bar(L::kBarKEmpty + ks), ((j / L::kKSt) & 1) ^ 1, abort_flag,
                               &g_fwd_status))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarKFull + ks), L::kKVBytes);
                for (int pp = 0; pp < L::kPanels; ++pp)
                    tma_load_4d(sbase + L::kOffK + ks * L::kKVBytes + pp * kPanelBytes, &tmK,
                                bar(L::kBarKFull + ks), 64 * pp, g, j * kBN, b);
                const int vs = j % L::kVSt;
                if (!mbar_wait(bar(L::kBarVEmpty + vs), ((j / L::kVSt) & 1) ^ 1, abort_flag,
                               &g_fwd_status))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarVFull + vs), L::kKVBytes);
                for (int pp = 0; pp < L::kPanels; ++pp)
                    tma_load_4d(sbase + L::kOffV + vs * L::kKVBytes + pp * kPanelBytes, &tmV,
                                bar(L::kBarVFull + vs), 64 * pp, g, j * kBN, b);
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t kIdPV = idesc_bf16_f32(kBM, D, true);
            bool ok = true;
            for (int t = 0; t < kQT; ++t)
                if (n_t[t] > 0 && ok)
                    ok = mbar_wait(bar(L::kBarQFull + t), 0, abort_flag, &g_fwd_status);
            int k_ready = -1, v_ready = -1;
            auto wait_k = [&](int j) {
                if (ok && j > k_ready) {
                    ok = mbar_wait(bar(L::kBarKFull + j % L::kKSt), (j / L::kKSt) & 1, abort_flag,
                                   &g_fwd_status);
                    tc_fence_after();
                    k_ready = j;
                }
            };
            auto wait_v = [&](int j) {
                if (ok && j > v_ready) {
                    ok = mbar_wait(bar(L::kBarVFull + j % L::kVSt), (j / L::kVSt) & 1, abort_flag,
                                   &g_fwd_status);
                    tc_fence_after();
                    v_ready = j;
                }
            };
            // S_t = Q_t K_j^T  (M=128 rows, N=128 keys, K=D in steps of 16)
            auto issue_s = [&](int t, int j) {
                wait_k(j);
                if (!ok) return;
                const uint32_t qa = sbase + L::kOffQ + t * L::kQBytes;
                const uint32_t ka = sbase + L::kOffK + (j % L::kKSt) * L::kKVBytes;
                const uint32_t dS = tmem + L::tm_s(t);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                    mma_ss(dS, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                           kIdS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(L::kBarSFull + t));
            };
            // O_t += P_t V_j  (M=128 rows, N=D, K=128 keys in steps of 16)
            auto issue_pv = [&](int t, int j) {
                wait_v(j);
                if (!ok) return;
                ok = mbar_wait(bar(L::kBarPFull + t), j & 1, abort_flag, &g_fwd_status);
                if (!ok) return;
                tc_fence_after();
                const uint32_t va = sbase + L::kOffV + (j % L::kVSt) * L::kKVBytes;
                const uint32_t dO = tmem + L::tm_o(t);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // V is [keys][D] with D contiguous: an N-major B operand.  Along N the
                    // 64-column panels are kPanelBytes apart (LBO); along K every 8 keys
                    // are 1024 B apart (SBO).
                    const uint64_t bd = sdesc_sw128(va + kk * 16 * 128, kPanelBytes, 1024);
                    const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (P_TMEM) {
                        // bf16 P packed two per 32-bit column: 16 keys = 8 columns
                        mma_ts(dO, tmem + L::tm_s(t) + kk * 8, bd, kIdPV, acc);
                    } else {
                        const uint32_t pa = sbase + L::kOffP + t * L::kPBytes;
                        const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                        mma_ss(dO, sdesc_sw128(pa + off, 16, 1024), bd, kIdPV, acc);
                    }
                }
                if (j == n_t[t] - 1) tc_commit(bar(L::kBarOFull + t));
            };
            if (n_t[0] > 0) issue_s(0, 0);
            if (n_t[1] > 0) issue_s(1, 0);
            if (n > 0 && ok) tc_commit(bar(L::kBarKEmpty + 0));
            for (int j = 0; j < n && ok; ++j) {
                if (j < n_t[0]) issue_pv(0, j);
                if (j + 1 < n_t[0]) issue_s(0, j + 1);
                if (j < n_t[1]) issue_pv(1, j);
                if (ok) tc_commit(bar(L::kBarVEmpty + j % L::kVSt));
                if (j + 1 < n_t[1]) issue_s(1, j + 1);
                if (j + 1 < n && ok) tc_commit(bar(L::kBarKEmpty + (j + 1) % L::kKSt));
            }
            if (ok) atomicAdd(&g_fwd_tiles, (unsigned long long)(n_t[0] + n_t[1]));
        }
    } else {
        // ================================================= softmax warpgroups
        const int t = (warp - 2) >> 2;
        const int q4 = warp & 3;  // TMEM lane quarter this warp may access
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const uint32_t tS = tmem + lane_base + L::tm_s(t);
        const uint32_t tO = tmem + lane_base + L::tm_o(t);
        const int rs = row0 + t * kBM;
        const int row = rs + r;
        const int nt = n_t[t];
        const long long diag = (long long)row + (p.Nk - p.Nq);  // last causal key of this row
        const long long diag_tile = (long long)rs + (p.Nk - p.Nq);
        const float sl = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            if (!mbar_wait(bar(L::kBarSFull + t), j & 1, abort_flag, &g_fwd_status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[kBN];
            tmem_ld64_sync(tS, s);
            tmem_ld64_sync(tS + 64, s + 64);
            const int col0 = j * kBN;
            const bool need_mask = (col0 + kBN > p.Nk) ||
                                   (p.causal && (long long)(col0 + kBN - 1) > diag_tile);
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const int col = col0 + c;
                    const bool keep = col < p.Nk && (!p.causal || (long long)col <= diag);
                    if (!keep) s[c] = __float_as_uint(-INFINITY);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                mx0 = fmaxf(mx0, __uint_as_float(s[c]));
                mx1 = fmaxf(mx1, __uint_as_float(s[c + 1]));
            }
            // Conditional rescale: the reference max moves only when the tile's max
            // exceeds it by more than rescale_thr (log2 units).  acc and l always share
            // the reference, so O = acc / l and LSE = m + log l stay exact; a stale
            // reference only bounds P by 2^rescale_thr.
            const float m_tile = fmaxf(mx0, mx1) * sl;
            float m_new = m, alpha = 1.f;
            if (m_tile > m + p.rescale_thr) {
                m_new = m_tile;
                alpha = ex2(m - m_new);  // 0 on the first non-empty tile
            }
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            float sum0 = 0.f, sum1 = 0.f;
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int c = 0; c < kBN / 2; ++c) {
                const float p0 = ex2(fmaf(__uint_as_float(s[2 * c]), sl, -m_use));
                const float p1 = ex2(fmaf(__uint_as_float(s[2 * c + 1]), sl, -m_use));
                sum0 += p0;
                sum1 += p1;
                pk[c] = pack_bf16(p0, p1);
            }
            l = fmaf(l, alpha, sum0 + sum1);
            if constexpr (P_TMEM) {
                tmem_st32(tS, pk);
                tmem_st32(tS + 32, pk + 32);
                tmem_st_wait();
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
            // Deferred normalisation: O_t still holds the sum through key tile j-1 (its PV
            // completed before S_t(j) did); rescale it only when some row's max grew.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t x[32];
                    tmem_ld32_sync(tO + c, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * alpha);
                    tmem_st32(tO + c, x);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull + t));
            m = m_new;
        }
        if (nt == 0) {
            // Tile beyond Nq, or rows with no allowed key at all.
            if (row < p.Nq) {
                __nv_bfloat16* orow = p.o + (((long long)b * p.Nq + row) * p.Hq + hq) * D;
                uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                p.lse[((long long)b * p.Hq + hq) * p.Nq + row] = -INFINITY;
            }
        } else if (ok && mbar_wait(bar(L::kBarOFull + t), 0, abort_flag, &g_fwd_status)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const uint32_t stage = sbase + L::kOffQ + t * L::kQBytes;  // Q_t is no longer read
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t x[32];
                tmem_ld32_sync(tO + c, x);
                uint32_t h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h[i] = pack_bf16(__uint_as_float(x[2 * i]) * inv,
                                     __uint_as_float(x[2 * i + 1]) * inv);
                const int panel = c >> 6;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int cc = ((c & 63) >> 3) + i;
                    st_shared_v4(stage + panel * kPanelBytes + r * 128 + ((cc ^ (r & 7)) << 4),
                                 h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(L::kBarStaged + t));
            if (r == 0 && mbar_wait(bar(L::kBarStaged + t), 0, abort_flag, &g_fwd_status)) {
                for (int pp = 0; pp < L::kPanels; ++pp)
                    tma_store_4d(&tmO, stage + pp * kPanelBytes, 64 * pp, hq, rs, b);
                tma_store_commit_and_wait_all();
            }
            if (row < p.Nq)
                p.lse[((long long)b * p.Hq + hq) * p.Nq + row] =
                    l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
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

// Threshold of the conditional rescale in log2 units.  8 keeps every P below
// 256 (exact in bf16's range, no fp32 overflow risk in l or acc).
// ATTN_FWD_RESCALE_THRESHOLD overrides it (0 = rescale on every max increase).
float rescale_threshold() {
    static const float v = [] {
        const char* e = std::getenv("ATTN_FWD_RESCALE_THRESHOLD");
        if (e == nullptr) return 8.0f;
        const float x = std::strtof(e, nullptr);
        return (x >= 0.f && x <= 16.f) ? x : 8.0f;
    }();
    return v;
}

template <int D, bool P_TMEM>
attn_status_t launch_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int Hq, int Hkv, int Nq, int Nk, float scale, int causal,
                          cudaStream_t stream) {
    using L = Layout<D, P_TMEM>;
    CUtensorMap mq, mk, mv, mo;
    if (!attn_host::encode_bshd_map(&mq, q, B, Nq, Hq, D, kBM, 2) ||
        !attn_host::encode_bshd_map(&mk, k, B, Nk, Hkv, D, kBN, 2) ||
        !attn_host::encode_bshd_map(&mv, v, B, Nk, Hkv, D, kBN, 2) ||
        !attn_host::encode_bshd_map(&mo, o, B, Nq, Hq, D, kBM, 2))
        return ATTN_ERR_CUDA;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(fwd_tc_kernel<D, P_TMEM>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        L::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return ATTN_ERR_CUDA;
    FwdParams prm;
    prm.lse = lse;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    prm.causal = causal;
    prm.num_pairs = (Nq + kQT * kBM - 1) / (kQT * kBM);
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.rescale_thr = rescale_threshold();
    const long long grid = (long long)prm.num_pairs * B * Hq;
    if (grid > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    fwd_tc_kernel<D, P_TMEM><<<(unsigned)grid, kThreads, L::kSmemBytes, stream>>>(mq, mk, mv, mo,
                                                                                  prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Debug switch: ATTN_FWD_P_SMEM=1 routes P through shared memory (SS MMA)
// instead of tensor memory (TS MMA).  Both compute the same thing.
bool p_in_smem() {
    static const bool v = [] {
        const char* e = std::getenv("ATTN_FWD_P_SMEM");
        return e != nullptr && e[0] == '1';
    }();
    return v;
}

}  // namespace

namespace attn_host {

attn_status_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, cudaStream_t stream) {
    const bool smem_p = p_in_smem();
    if (d == 128)
        return smem_p ? launch_impl<128, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream)
                      : launch_impl<128, true>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream);
    if (d == 64)
        return smem_p ? launch_impl<64, false>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream)
                      : launch_impl<64, true>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream);
    return ATTN_ERR_UNSUPPORTED;
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
