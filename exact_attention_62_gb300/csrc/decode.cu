// decode.cu -- flash-decoding on sm_103a: split-KV kernel + log-sum-exp merge.
//
// What it computes (Lecture 11 - Kernel Optimization Techniques, section 6.2):
// with one query per sequence, the key/value length is cut into S segments;
// for each (sequence, query head, segment) the segment's normalised output
// o_s and lse_s = log sum_{j in segment} exp(scale q.k_j) are formed
// (steps 1-2), and a second small kernel merges them:
// lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s (step 3).  This
// is the associative merge of section 3.2 written in lse form.
//
// How (GB300 design):
//  * Grid (segment, query-head group, sequence).  The G = Hq/Hkv query heads
//    that share one KV head are packed into the columns of one small matrix
//    product, so each K/V byte of the segment is read from HBM exactly once
//    for the whole group (section 6.2, GQA paragraph).
//  * Warp 0 streams the segment's K and V tiles (64 keys each) with TMA into
//    a multi-stage shared-memory ring (128-byte swizzle, mbarrier full/empty
//    pairs).  Two groups of four consumer warps take alternate tiles, and the
//    four warps of a group each take 16 keys of the tile.
//  * The consumer work per tile is two tiny matrix products done with warp
//    MMA (m16n8k16, bf16 in, fp32 accumulate): S^T = K Q^T with the keys as
//    the 16 rows and up to 8 query heads as the columns, then
//    O^T += V^T P^T.  The transposed P operand is formed in registers with
//    movmatrix.  The online-softmax state (m, l) lives per query column in
//    registers; the running max is kept in base-2 units (scale log2 e
//    folded in).  The kernel is HBM-bound; the tensor-core products just keep
//    the instruction count far below the memory time.
//  * At the end the eight warps' states are merged through shared memory
//    (the same (m, l, acc) merge).  With a single segment the kernel writes
//    O (bf16) and LSE directly and no merge kernel runs; otherwise the merge
//    kernel is launched as a programmatic dependent (one pass over the
//    partials for up to 16 segments per thread, two passes beyond).
//  * Paged caches with pages of 16 keys and 2, 4 or 8 KV heads take a second kernel,
//    decode_heads_kernel, in which one CTA reads whole pages for all KV
//    heads (its own comment below says why).
#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

using namespace attn_dev;

namespace {

__device__ unsigned g_dec_status = 0;

constexpr int kTileKeys = 64;
// Consumer warps come in groups of four; group i takes the tiles t with
// t % kGroups == i, so kGroups tiles are consumed at once.
constexpr int kGroups = 2;
constexpr int kConsumerWarps = 4 * kGroups;
constexpr int kDecThreads = 32 * (1 + kConsumerWarps);
constexpr float kLn2 = 0.69314718055994530942f;

struct DecParams {
    const __nv_bfloat16* q;  // [B, 1, Hq, D]
    __nv_bfloat16* o;        // [B, 1, Hq, D]  (single segment)
    float* lse;              // [B, Hq]        (single segment)
    float* o_parts;          // [S, B*Hq, D]   (several segments)
    float* lse_parts;        // [S, B*Hq]
    int B, Hq, Hkv, Nk, G, splits, seg_len;  // Nk: cache length (paged: the maximum)
    float scale_log2;
    long long wait_limit;    // bound of every mbarrier wait, SM cycles
    int skip_load;           // tests only: tile of block (0, 0, 0) that is never loaded (-1: none)
    long long o_slack;       // bounds-checked build, tests only: O's extent taken as this much smaller
    // paged cache only
    const int* table;        // [B, max_pages] page of each block of page_size keys
    const int* seq_lens;     // [B]
    int page_size, max_pages;
};

// Paged cache: block-table entries one CTA may need (its segment's pages),
// staged in shared memory by the producer warp.  The host keeps segments
// short enough for this.
constexpr int kTableCap = 4096;

template <int D, int STAGES, bool PAGED = false>
struct DecLayout {
    static constexpr int kPanelBytes = kTileKeys * 128;  // 64 keys x 64 columns x 2 B
    static constexpr int kTileBytes = kTileKeys * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;   // K tile then V tile
    static constexpr int kOffBar = STAGES * kStageBytes;
    static constexpr int kNumBars = 2 * STAGES;          // full[STAGES], empty[STAGES]
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffTable = kOffMisc + 16;
    static constexpr int kSmemBytes = kOffTable + (PAGED ? kTableCap * 4 : 0) + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // Cross-warp merge scratch [warp][8 query columns][D + 2], reusing the
    // stage buffers once every tile has been consumed.
    static constexpr int kRedStride = D + 2;
    static_assert(kConsumerWarps * 8 * kRedStride * 4 <= STAGES * kStageBytes, "merge scratch");
    // Tiles t and t + STAGES share a stage.  Only if they belong to the same
    // consumer group does program order keep that group at most one phase
    // ahead of the stage's barriers; otherwise a parity wait can be satisfied
    // by the phase before the awaited one.
    static_assert(STAGES % kGroups == 0, "each ring stage must belong to one consumer group");
};

template <int D>
constexpr int dec_stages() { return D == 128 ? 6 : 8; }

__device__ __forceinline__ uint32_t ld_b32(const __nv_bfloat16* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

template <int D, int GC, bool PAGED>
__global__ void __launch_bounds__(kDecThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecParams p) {
    constexpr int STAGES = dec_stages<D>();
    using L = DecLayout<D, STAGES, PAGED>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int st) -> uint32_t { return sbase + L::kOffBar + 8u * st; };
    auto empty_bar = [&](int st) -> uint32_t { return sbase + L::kOffBar + 8u * (STAGES + st); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc);

    const int seg = blockIdx.x;
    const int hq0 = blockIdx.y * GC;
    const int b = blockIdx.z;
    const int g = hq0 / p.G;
    // Keys of this sequence: all Nk, or (paged) its own length, clamped to
    // [0, Nk] where Nk is the caller's maximum.
    int len = p.Nk;
    if constexpr (PAGED) {
        len = 0;
        if (in_bounds(b, 1, p.B, &g_dec_status)) len = min(max(p.seq_lens[b], 0), p.Nk);
    }
    // (bounds-checked build) extents of the outputs and of the partials
    const long long o_extent = (long long)p.B * p.Hq * D - p.o_slack;
    const long long parts_rows = (long long)p.splits * p.B * p.Hq;
    const int j0 = seg * p.seg_len;
    const int j1 = min(j0 + p.seg_len, len);
    const int ntiles = j1 > j0 ? (j1 - j0 + kTileKeys - 1) / kTileKeys : 0;
    const long long R = (long long)p.B * p.Hq;

    if (ntiles == 0) {  // empty segment: o_s = 0, lse_s = -inf
        for (int e = threadIdx.x; e < GC * D; e += blockDim.x) {
            const long long row = (long long)b * p.Hq + hq0 + e / D;
            if (p.splits == 1) {  // a sequence with no keys at all
                if (in_bounds(row * D + (e % D), 1, o_extent, &g_dec_status))
                    p.o[row * D + (e % D)] = __float2bfloat16_rn(0.f);
                if (e % D == 0 && in_bounds(row, 1, (long long)p.B * p.Hq, &g_dec_status)) p.lse[row] = -INFINITY;
            } else {
                const long long po = ((long long)seg * R + row) * D + (e % D);
                if (in_bounds(po, 1, parts_rows * D, &g_dec_status)) p.o_parts[po] = 0.f;
                if (e % D == 0 && in_bounds((long long)seg * R + row, 1, parts_rows, &g_dec_status))
                    p.lse_parts[(long long)seg * R + row] = -INFINITY;
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), 4);  // the four warps of the group that read it
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================================================= TMA producer
        // Paged cache: the tensor maps view the page pools as [pages,
        // page_size, Hkv, D]; a tile's keys come from the pages the block
        // table names.  Pages of 64 or more keys hold whole tiles (segments
        // start at multiples of 64); smaller pages are loaded as 64/page_size
        // boxes, skipping those past the sequence.
        int first_page = 0;
        const int* tab = nullptr;
        if constexpr (PAGED) {
            int* st_tab = reinterpret_cast<int*>(sgen + L::kOffTable);
            first_page = j0 / p.page_size;
            const int n_pages = (j1 - 1) / p.page_size - first_page + 1;
            const long long t0 = (long long)b * p.max_pages + first_page;
            for (int e = lane; e < n_pages; e += 32)
                st_tab[e] = in_bounds(t0 + e, 1, (long long)p.B * p.max_pages, &g_dec_status) ? p.table[t0 + e] : 0;
            __syncwarp();
            tab = st_tab;
        }
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        if (PAGED && p.page_size < kTileKeys) {
            // Small pages: 64 / page_size boxes per panel and tile.  The whole
            // warp runs the loop; lane 0 posts the stage's byte count and lane
            // r issues the boxes of the tile's r-th page.
            const int ps = p.page_size;
            for (int t = 0; t < ntiles; ++t) {
                const int st = t % STAGES;
                if (!mbar_wait_warp(empty_bar(st), ((t / STAGES) & 1) ^ 1, abort_flag, &g_dec_status,
                                    p.wait_limit))
                    break;
                const uint32_t kdst = sbase + st * L::kStageBytes;
                const int key0 = j0 + t * kTileKeys;
                const int nsub = min(kTileKeys / ps, (j1 - key0 + ps - 1) / ps);
                if (lane == 0) mbar_arrive_expect_tx(full_bar(st), (uint32_t)(nsub * ps * D * 2 * 2));
                __syncwarp();
                if (lane < nsub) {
                    const int page = tab[(key0 + lane * ps) / ps - first_page];
                    const uint32_t off = (uint32_t)(lane * ps * 128);
#pragma unroll
                    for (int pp = 0; pp < D / 64; ++pp) {
                        tma_load_4d(kdst + pp * L::kPanelBytes + off, &tmK, full_bar(st), 64 * pp, g, 0,
                                    page);
                        tma_load_4d(kdst + L::kTileBytes + pp * L::kPanelBytes + off, &tmV, full_bar(st),
                                    64 * pp, g, 0, page);
                    }
                }
            }
        } else if (lane == 0) {
            // Fault injection for tests: block (0, 0, 0) never loads tile
            // skip_load, so the waits for it run out (production: -1).
            const int skip = (blockIdx.x | blockIdx.y | blockIdx.z) == 0 ? p.skip_load : -1;
            for (int t = 0; t < ntiles; ++t) {
                const int st = t % STAGES;
                if (!mbar_wait(empty_bar(st), ((t / STAGES) & 1) ^ 1, abort_flag, &g_dec_status,
                               p.wait_limit))
                    break;
                if (t == skip) continue;
                const uint32_t kdst = sbase + st * L::kStageBytes;
                const int key0 = j0 + t * kTileKeys;
                if (PAGED) {  // pages of 64 or more keys: one box per panel
                    const int ps = p.page_size;
                    mbar_arrive_expect_tx(full_bar(st), L::kStageBytes);
                    const int page = tab[key0 / ps - first_page];
                    const int row = key0 % ps;
#pragma unroll
                    for (int pp = 0; pp < D / 64; ++pp) {
                        tma_load_4d(kdst + pp * L::kPanelBytes, &tmK, full_bar(st), 64 * pp, g, row, page);
                        tma_load_4d(kdst + L::kTileBytes + pp * L::kPanelBytes, &tmV, full_bar(st),
                                    64 * pp, g, row, page);
                    }
                } else {
                    mbar_arrive_expect_tx(full_bar(st), L::kStageBytes);
#pragma unroll
                    for (int pp = 0; pp < D / 64; ++pp) {
                        tma_load_4d(kdst + pp * L::kPanelBytes, &tmK, full_bar(st), 64 * pp, g, key0, b);
                        tma_load_4d(kdst + L::kTileBytes + pp * L::kPanelBytes, &tmV, full_bar(st),
                                    64 * pp, g, key0, b);
                    }
                }
            }
        }
        return;  // the producer takes no part in the consumers' named barriers
    }

    // ===================================================== consumers
    const int cw = warp - 1;
    const int grp = cw >> 2;  // which tiles: t % kGroups == grp
    const int kw = cw & 3;    // which 16 keys of those tiles
    const int g8 = lane >> 2;  // fragment row group
    const int t4 = lane & 3;   // fragment column pair
    const int mi = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
    const int rr = lane & 7;   // ldmatrix: which row of it

    // Q^T as the B operand of S^T = K Q^T: column n = query head hq0 + n.
    uint32_t qb[D / 16][2];
    {
        const long long qoff = ((long long)b * p.Hq + hq0 + (g8 < GC ? g8 : 0)) * D;
        const bool qv = g8 < GC && in_bounds(qoff, D, (long long)p.B * p.Hq * D, &g_dec_status);
        const __nv_bfloat16* qrow = p.q + qoff;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[kk][0] = qv ? ld_b32(qrow + kk * 16 + 2 * t4) : 0u;
            qb[kk][1] = qv ? ld_b32(qrow + kk * 16 + 8 + 2 * t4) : 0u;
        }
    }
    float acc[D / 16][4];
#pragma unroll
    for (int mb = 0; mb < D / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
    // online-softmax state of this lane's two query columns (2 t4, 2 t4 + 1)
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const float sl = p.scale_log2;
    const int kkey = 16 * kw + rr + 8 * (mi & 1);  // K row this lane addresses
    const int vkey = 16 * kw + rr + 8 * (mi >> 1); // V row this lane addresses

    for (int t = grp; t < ntiles; t += kGroups) {
        const int st = t % STAGES;
        if (!mbar_wait(full_bar(st), (t / STAGES) & 1, abort_flag, &g_dec_status, p.wait_limit)) break;
        const uint32_t kb = sbase + st * L::kStageBytes;
        const uint32_t vb = kb + L::kTileBytes;
        // Paged cache: V rows past the sequence hold whatever the pool has
        // there (or stale stage data); P is 0 for them but 0 * NaN is not,
        // so the warp zeroes its own such rows (K needs nothing: masked
        // scores are replaced, not multiplied).
        bool zeroed = false;
        if constexpr (PAGED) {
            const int kbase = j0 + t * kTileKeys + 16 * kw;
            if (kbase + 16 > j1) {
                for (int e = lane; e < 16 * (D / 8); e += 32) {
                    const int rrow = e / (D / 8), ch = e % (D / 8);
                    if (kbase + rrow >= j1)
                        st_shared_v4(vb + (ch >> 3) * L::kPanelBytes + (16 * kw + rrow) * 128 + ((ch & 7) << 4),
                                     0u, 0u, 0u, 0u);
                }
                __syncwarp();
                zeroed = true;
            }
        }

        // S^T (16 keys x 8 query columns) = K (16 x D) Q^T (D x 8); even and odd
        // k-steps accumulate separately to halve the dependent MMA chain.
        float ce[4] = {0.f, 0.f, 0.f, 0.f}, co[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int ch = 2 * kk + (mi >> 1);
            const uint32_t addr =
                kb + (ch >> 3) * L::kPanelBytes + kkey * 128 + (((ch & 7) ^ (kkey & 7)) << 4);
            uint32_t a[4];
            ldsm_x4(addr, a);
            if (kk & 1)
                mma_16816(co, a, qb[kk][0], qb[kk][1]);
            else
                mma_16816(ce, a, qb[kk][0], qb[kk][1]);
        }
        const float c[4] = {ce[0] + co[0], ce[1] + co[1], ce[2] + co[2], ce[3] + co[3]};
        // keys of this lane: rows g8 and g8 + 8 of the warp's 16
        const int key = j0 + t * kTileKeys + 16 * kw + g8;
        const bool in0 = key < j1, in1 = key + 8 < j1;
        const float x0 = in0 ? c[0] * sl : -INFINITY;  // (key,   col 2t4)
        const float x1 = in0 ? c[1] * sl : -INFINITY;  // (key,   col 2t4+1)
        const float x2 = in1 ? c[2] * sl : -INFINITY;  // (key+8, col 2t4)
        const float x3 = in1 ? c[3] * sl : -INFINITY;  // (key+8, col 2t4+1)
        float mxa = fmaxf(x0, x2), mxb = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
        }
        const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
        const float mua = mna == -INFINITY ? 0.f : mna;
        const float mub = mnb == -INFINITY ? 0.f : mnb;
        const float aa = ex2(m_a - mua), ab = ex2(m_b - mub);
        const float p0 = ex2(x0 - mua), p2 = ex2(x2 - mua);
        const float p1 = ex2(x1 - mub), p3 = ex2(x3 - mub);
        l_a = fmaf(l_a, aa, p0 + p2);
        l_b = fmaf(l_b, ab, p1 + p3);
        m_a = mna;
        m_b = mnb;
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) {
            acc[mb][0] *= aa;
            acc[mb][1] *= ab;
            acc[mb][2] *= aa;
            acc[mb][3] *= ab;
        }
        // P^T as the B operand (keys x query columns)
        const uint32_t b01 = movmatrix_trans(pack_bf16(p0, p1));
        const uint32_t b23 = movmatrix_trans(pack_bf16(p2, p3));
        // O^T (D x 8) += V^T (D x 16 keys) P^T (16 keys x 8)
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) {
            const int ch = 2 * mb + (mi & 1);
            const uint32_t addr =
                vb + (ch >> 3) * L::kPanelBytes + vkey * 128 + (((ch & 7) ^ (vkey & 7)) << 4);
            uint32_t a[4];
            ldsm_x4_trans(addr, a);
            mma_16816(acc[mb], a, b01, b23);
        }
        // order the zeroing stores before the stage's next TMA write
        if (zeroed) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
    }

    // The merge kernel (launched as a programmatic dependent) may start now;
    // it waits for this grid's completion before reading any partial.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // per-warp partial sums of l over the warp's keys
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    // every tile has been consumed: the stage buffers are free for the merge
    named_bar_sync(1, 32 * kConsumerWarps);
    float* red = reinterpret_cast<float*>(sgen);
    {
        float* ra = red + (cw * 8 + 2 * t4) * L::kRedStride;
        float* rb = ra + L::kRedStride;
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) {
            ra[mb * 16 + g8] = acc[mb][0];
            rb[mb * 16 + g8] = acc[mb][1];
            ra[mb * 16 + g8 + 8] = acc[mb][2];
            rb[mb * 16 + g8 + 8] = acc[mb][3];
        }
        if (g8 == 0) {
            ra[D] = m_a;
            ra[D + 1] = l_a;
            rb[D] = m_b;
            rb[D + 1] = l_b;
        }
    }
    named_bar_sync(1, 32 * kConsumerWarps);
    for (int e = threadIdx.x - 32; e < GC * D; e += 32 * kConsumerWarps) {
        const int qc = e / D, dd = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red[(w * 8 + qc) * L::kRedStride + D]);
        float lsum = 0.f, ov = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float* rw = red + (w * 8 + qc) * L::kRedStride;
                if (rw[D] != -INFINITY) {
                    const float cwt = ex2(rw[D] - M);
                    lsum = fmaf(cwt, rw[D + 1], lsum);
                    ov = fmaf(cwt, rw[dd], ov);
                }
            }
        }
        const long long row = (long long)b * p.Hq + hq0 + qc;
        const float outv = lsum > 0.f ? ov / lsum : 0.f;
        const float lsev = lsum > 0.f ? (M + lg2(lsum)) * kLn2 : -INFINITY;
        if (p.splits == 1) {
            if (in_bounds(row * D + dd, 1, o_extent, &g_dec_status)) p.o[row * D + dd] = __float2bfloat16_rn(outv);
            if (dd == 0 && in_bounds(row, 1, (long long)p.B * p.Hq, &g_dec_status)) p.lse[row] = lsev;
        } else {
            const long long po = ((long long)seg * R + row) * D + dd;
            if (in_bounds(po, 1, parts_rows * D, &g_dec_status)) p.o_parts[po] = outv;
            if (dd == 0 && in_bounds((long long)seg * R + row, 1, parts_rows, &g_dec_status))
                p.lse_parts[(long long)seg * R + row] = lsev;
        }
    }
}

// ------------------------------------------------------------- pages of 16 keys
// A paged cache with pages of 16 keys holds, in each page, the rows of all KV
// heads side by side (16 keys x Hkv heads x D).  decode_split_kernel, one CTA
// per KV head, reads such a page as 16 rows of D bf16 spread Hkv * D * 2
// bytes apart: one small TMA box per page, head and panel.  A read-only probe
// of that pattern on GB300 (64K keys, pages in random order) streamed 3960
// GB/s with 96 CTAs, against 6320 GB/s when each CTA loaded whole pages of
// all 8 heads.  So for Hkv = 2, 4 or 8 this kernel takes a segment of pages
// for all KV heads in one CTA.  A page arrives as one box per K/V panel
// (16 keys x Hkv heads x 64 columns), and a stage holds 8 / Hkv pages; each
// of the eight consumer warps takes one (KV head, page) pair of the stage
// and works on that head's 16 keys with the same two warp-MMA products as
// decode_split_kernel (S^T = K Q^T with the G <= 8 query heads of the KV
// head as columns, then O^T += V^T P^T).  The tensor maps list the pool's
// dimensions as (d, key, head, page), so a head's 16 keys are consecutive
// 128-byte rows of the page and the 128-byte swizzle keeps every ldmatrix
// conflict-free.  At the end the warps of one head (8 / Hkv of them) merge
// their online-softmax states through shared memory, and one warp per head
// writes the head's partial (or, with one segment, its O and LSE).
constexpr int kHeadsWarps = 8;  // consumer warps: one (KV head, page slot) pair each
constexpr int kHeadsThreads = 32 * (1 + kHeadsWarps);
constexpr int kSmallPage = 16;  // keys per page on this path
// CTAs (segments x sequences) the automatic segment count aims at: about
// 27/32 of the SMs.  On GB300 (152 SMs) 128 CTAs measured best at every batch
// tried with pages of 16 keys (B = 1 x 16K and 64K keys, 4 x 16K, 8 x 8K,
// 16 x 8K): one wave, and at B = 1 still few enough partials per row for the
// one-pass merge.
inline int heads_target_ctas(int sms) { return sms * 27 / 32; }

template <int D, int NH>  // NH = Hkv: 8, 4 or 2
struct HeadsLayout {
    static constexpr int kSlots = kHeadsWarps / NH;                // pages per stage
    static constexpr int kPanels = D / 64;
    static constexpr int kPanelBytes = kSmallPage * NH * 128;      // a page's panel: 16 keys x NH heads x 128 B
    static constexpr int kPageBytes = 2 * kPanels * kPanelBytes;   // K panels, then V panels
    static constexpr int kStageBytes = kSlots * kPageBytes;        // 32 KB per 64 columns of d
    static constexpr int kStages = D == 128 ? 3 : 6;               // 192 KB in flight
    static constexpr int kOffBar = kStages * kStageBytes;          // full[kStages], empty[kStages]
    static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    // the heads' cross-warp merge: [warp][lane][acc (D/16 x 4), m_a, m_b, l_a, l_b]
    // floats, over the stage buffers once every page has been consumed
    static constexpr int kRedFloats = D / 16 * 4 + 4;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kPanelBytes % 1024 == 0, "swizzle atoms start on 1024-byte boundaries");
    static_assert(kHeadsWarps % NH == 0, "whole page slots");
    static_assert(kHeadsWarps * 32 * kRedFloats * 4 <= kStages * kStageBytes, "merge scratch");
};

template <int D, int NH>
__global__ void __launch_bounds__(kHeadsThreads)
    decode_heads_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecParams p) {
    using L = HeadsLayout<D, NH>;
    constexpr int STAGES = L::kStages;
    constexpr int SLOTS = L::kSlots;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int st) -> uint32_t { return sbase + L::kOffBar + 8u * st; };
    auto empty_bar = [&](int st) -> uint32_t { return sbase + L::kOffBar + 8u * (STAGES + st); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kOffMisc);

    const int seg = blockIdx.x;
    const int b = blockIdx.z;
    int len = 0;  // this sequence's keys, clamped to [0, Nk] (Nk: the caller's maximum)
    if (in_bounds(b, 1, p.B, &g_dec_status)) len = min(max(p.seq_lens[b], 0), p.Nk);
    const long long R = (long long)p.B * p.Hq;
    const long long o_extent = R * D - p.o_slack;
    const long long parts_rows = (long long)p.splits * R;
    const int j0 = seg * p.seg_len;  // seg_len is a multiple of the page size
    const int j1 = min(j0 + p.seg_len, len);
    const int npages = j1 > j0 ? (j1 - j0 + kSmallPage - 1) / kSmallPage : 0;
    const int nstages = (npages + SLOTS - 1) / SLOTS;  // SLOTS pages per stage, the last maybe fewer

    if (npages == 0) {  // empty segment: o_s = 0, lse_s = -inf for every query head
        for (int e = threadIdx.x; e < p.Hq * D; e += blockDim.x) {
            const long long row = (long long)b * p.Hq + e / D;
            if (p.splits == 1) {  // a sequence with no keys at all
                if (in_bounds(row * D + (e % D), 1, o_extent, &g_dec_status))
                    p.o[row * D + (e % D)] = __float2bfloat16_rn(0.f);
                if (e % D == 0 && in_bounds(row, 1, R, &g_dec_status)) p.lse[row] = -INFINITY;
            } else {
                const long long po = ((long long)seg * R + row) * D + (e % D);
                if (in_bounds(po, 1, parts_rows * D, &g_dec_status)) p.o_parts[po] = 0.f;
                if (e % D == 0 && in_bounds((long long)seg * R + row, 1, parts_rows, &g_dec_status))
                    p.lse_parts[(long long)seg * R + row] = -INFINITY;
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), kHeadsWarps);  // every consumer warp releases every stage
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================================================= TMA producer
        // The whole warp runs the loop: the lanes fetch the block-table
        // entries of 32 pages at a time (SLOTS divides 32, so a stage's
        // pages never straddle two fetches), lane 0 issues the loads.
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        const long long tab0 = (long long)b * p.max_pages + j0 / kSmallPage;
        int page_of_lane = 0;
        for (int t = 0; t < nstages; ++t) {
            const int pg = t * SLOTS;  // first page of the stage
            if ((pg & 31) == 0) {
                const int i = pg + lane;
                page_of_lane = (i < npages && in_bounds(tab0 + i, 1, (long long)p.B * p.max_pages, &g_dec_status))
                                   ? p.table[tab0 + i]
                                   : 0;
            }
            const int st = t % STAGES;
            if (!mbar_wait_warp(empty_bar(st), ((t / STAGES) & 1) ^ 1, abort_flag, &g_dec_status, p.wait_limit))
                break;
            const int np = min(SLOTS, npages - pg);  // pages in this stage
            if (lane == 0) mbar_arrive_expect_tx(full_bar(st), (uint32_t)(np * L::kPageBytes));
#pragma unroll
            for (int sl = 0; sl < SLOTS; ++sl) {
                const int page = __shfl_sync(0xffffffffu, page_of_lane, (pg + sl) & 31);
                if (lane == 0 && sl < np) {
                    const uint32_t dst = sbase + st * L::kStageBytes + sl * L::kPageBytes;
#pragma unroll
                    for (int pp = 0; pp < L::kPanels; ++pp) {
                        tma_load_4d(dst + pp * L::kPanelBytes, &tmK, full_bar(st), 64 * pp, 0, 0, page);
                        tma_load_4d(dst + (L::kPanels + pp) * L::kPanelBytes, &tmV, full_bar(st), 64 * pp, 0, 0,
                                    page);
                    }
                }
            }
            __syncwarp();
        }
        return;  // the producer takes no part in the consumers' work
    }

    // ===================================================== consumers
    const int cw = warp - 1;
    const int h = cw % NH;      // KV head of this warp
    const int slot = cw / NH;   // which page of each stage it takes
    const int G = p.G;          // the head's query heads, 1..8: the MMA columns
    const int hq0 = h * G;
    const int g8 = lane >> 2;   // fragment row group
    const int t4 = lane & 3;    // fragment column pair
    const int mi = lane >> 3;   // ldmatrix: which 8x8 matrix this lane addresses
    const int rr = lane & 7;    // ldmatrix: which row of it

    // Q^T of the head's query heads as the B operand of S^T = K Q^T
    uint32_t qb[D / 16][2];
    {
        const long long qoff = ((long long)b * p.Hq + hq0 + (g8 < G ? g8 : 0)) * D;
        const bool qv = g8 < G && in_bounds(qoff, D, R * D, &g_dec_status);
        const __nv_bfloat16* qrow = p.q + qoff;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[kk][0] = qv ? ld_b32(qrow + kk * 16 + 2 * t4) : 0u;
            qb[kk][1] = qv ? ld_b32(qrow + kk * 16 + 8 + 2 * t4) : 0u;
        }
    }
    float acc[D / 16][4];
#pragma unroll
    for (int mb = 0; mb < D / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;  // columns 2 t4 and 2 t4 + 1
    const float sl = p.scale_log2;
    const int krow = h * kSmallPage + rr + 8 * (mi & 1);   // K row (of the page) this lane addresses
    const int vrow = h * kSmallPage + rr + 8 * (mi >> 1);  // V row this lane addresses

    for (int t = 0; t < nstages; ++t) {
        const int st = t % STAGES;
        if (!mbar_wait(full_bar(st), (t / STAGES) & 1, abort_flag, &g_dec_status, p.wait_limit)) break;
        const int pi = t * SLOTS + slot;  // this warp's page of the stage (the last stage may lack it)
        if (pi < npages) {
            const uint32_t kb = sbase + st * L::kStageBytes + slot * L::kPageBytes;
            const uint32_t vb = kb + L::kPanels * L::kPanelBytes;
            const int key0 = j0 + pi * kSmallPage;
            // Keys of the last page past the sequence: their pool slots hold
            // whatever is there (P is 0 for them, but 0 * NaN is not), so the
            // warp zeroes its head's V rows there (K needs nothing: masked
            // scores are replaced, not multiplied).
            const bool zeroed = key0 + kSmallPage > j1;
            if (zeroed) {
                for (int e = lane; e < kSmallPage * (D / 8); e += 32) {
                    const int r = e / (D / 8), ch = e % (D / 8);
                    const int row = h * kSmallPage + r;
                    if (key0 + r >= j1)
                        st_shared_v4(vb + (ch >> 3) * L::kPanelBytes + row * 128 + (((ch & 7) ^ (row & 7)) << 4),
                                     0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }

            // S^T (16 keys x 8 query columns) = K (16 x D) Q^T (D x 8); even and
            // odd k-steps accumulate separately to halve the dependent MMA chain.
            float ce[4] = {0.f, 0.f, 0.f, 0.f}, co[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int ch = 2 * kk + (mi >> 1);
                const uint32_t addr = kb + (ch >> 3) * L::kPanelBytes + krow * 128 + (((ch & 7) ^ (krow & 7)) << 4);
                uint32_t a[4];
                ldsm_x4(addr, a);
                if (kk & 1)
                    mma_16816(co, a, qb[kk][0], qb[kk][1]);
                else
                    mma_16816(ce, a, qb[kk][0], qb[kk][1]);
            }
            const float c[4] = {ce[0] + co[0], ce[1] + co[1], ce[2] + co[2], ce[3] + co[3]};
            const int key = key0 + g8;  // keys of this lane: rows g8 and g8 + 8 of the page
            const bool in0 = key < j1, in1 = key + 8 < j1;
            const float x0 = in0 ? c[0] * sl : -INFINITY;  // (key,   col 2t4)
            const float x1 = in0 ? c[1] * sl : -INFINITY;  // (key,   col 2t4+1)
            const float x2 = in1 ? c[2] * sl : -INFINITY;  // (key+8, col 2t4)
            const float x3 = in1 ? c[3] * sl : -INFINITY;  // (key+8, col 2t4+1)
            float mxa = fmaxf(x0, x2), mxb = fmaxf(x1, x3);
    #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
            }
            const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
            const float mua = mna == -INFINITY ? 0.f : mna;
            const float mub = mnb == -INFINITY ? 0.f : mnb;
            const float aa = ex2(m_a - mua), ab = ex2(m_b - mub);
            const float p0 = ex2(x0 - mua), p2 = ex2(x2 - mua);
            const float p1 = ex2(x1 - mub), p3 = ex2(x3 - mub);
            l_a = fmaf(l_a, aa, p0 + p2);
            l_b = fmaf(l_b, ab, p1 + p3);
            m_a = mna;
            m_b = mnb;
    #pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) {
                acc[mb][0] *= aa;
                acc[mb][1] *= ab;
                acc[mb][2] *= aa;
                acc[mb][3] *= ab;
            }
            // P^T as the B operand (keys x query columns), then
            // O^T (D x 8) += V^T (D x 16 keys) P^T (16 keys x 8)
            const uint32_t b01 = movmatrix_trans(pack_bf16(p0, p1));
            const uint32_t b23 = movmatrix_trans(pack_bf16(p2, p3));
    #pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) {
                const int ch = 2 * mb + (mi & 1);
                const uint32_t addr = vb + (ch >> 3) * L::kPanelBytes + vrow * 128 + (((ch & 7) ^ (vrow & 7)) << 4);
                uint32_t a[4];
                ldsm_x4_trans(addr, a);
                mma_16816(acc[mb], a, b01, b23);
            }
            if (zeroed) fence_proxy_async_smem();  // the zeroing stores before the stage's next TMA write
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
    }

    // The merge kernel (launched as a programmatic dependent) may start now;
    // it waits for this grid's completion before reading any partial.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // l over the warp's 16 key rows; m is already the same in those lanes
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    if constexpr (SLOTS > 1) {
        // The SLOTS warps of a head merge their (m, l, acc) through shared
        // memory (every page has been consumed, so the stage buffers are
        // free); the slot-0 warp of each head takes the others' states
        // lane by lane, fragment position by fragment position.
        named_bar_sync(1, 32 * kHeadsWarps);
        float* red = reinterpret_cast<float*>(sgen);
        {
            float* mine = red + ((size_t)cw * 32 + lane) * L::kRedFloats;
#pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) {
#pragma unroll
                for (int i = 0; i < 4; ++i) mine[mb * 4 + i] = acc[mb][i];
            }
            mine[D / 16 * 4 + 0] = m_a;
            mine[D / 16 * 4 + 1] = m_b;
            mine[D / 16 * 4 + 2] = l_a;
            mine[D / 16 * 4 + 3] = l_b;
        }
        named_bar_sync(1, 32 * kHeadsWarps);
        if (slot != 0) return;
#pragma unroll
        for (int sl = 1; sl < SLOTS; ++sl) {
            const float* o = red + ((size_t)(h + sl * NH) * 32 + lane) * L::kRedFloats;
            const float om_a = o[D / 16 * 4 + 0], om_b = o[D / 16 * 4 + 1];
            const float ol_a = o[D / 16 * 4 + 2], ol_b = o[D / 16 * 4 + 3];
            const float Ma = fmaxf(m_a, om_a), Mb = fmaxf(m_b, om_b);
            // a warp that saw no key has m = -inf and weight 0
            const float wa = m_a == -INFINITY ? 0.f : ex2(m_a - Ma);
            const float xa = om_a == -INFINITY ? 0.f : ex2(om_a - Ma);
            const float wb = m_b == -INFINITY ? 0.f : ex2(m_b - Mb);
            const float xb = om_b == -INFINITY ? 0.f : ex2(om_b - Mb);
            l_a = fmaf(l_a, wa, ol_a * xa);
            l_b = fmaf(l_b, wb, ol_b * xb);
#pragma unroll
            for (int mb = 0; mb < D / 16; ++mb) {
                acc[mb][0] = fmaf(acc[mb][0], wa, o[mb * 4 + 0] * xa);
                acc[mb][1] = fmaf(acc[mb][1], wb, o[mb * 4 + 1] * xb);
                acc[mb][2] = fmaf(acc[mb][2], wa, o[mb * 4 + 2] * xa);
                acc[mb][3] = fmaf(acc[mb][3], wb, o[mb * 4 + 3] * xb);
            }
            m_a = Ma;
            m_b = Mb;
        }
    }
    // This head's result for query columns 2 t4 and 2 t4 + 1: O = acc / l
    // (acc[mb][c] holds d = 16 mb + g8, acc[mb][2 + c] d + 8), LSE = m + ln l.
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int qc = 2 * t4 + c;
        if (qc >= G) continue;
        const float l = c ? l_b : l_a, m = c ? m_b : m_a;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lsev = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
        const long long row = (long long)b * p.Hq + hq0 + qc;
#pragma unroll
        for (int mb = 0; mb < D / 16; ++mb) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int dd = mb * 16 + g8 + 8 * h;
                const float v = acc[mb][2 * h + c] * inv;
                if (p.splits == 1) {
                    if (in_bounds(row * D + dd, 1, o_extent, &g_dec_status)) p.o[row * D + dd] = __float2bfloat16_rn(v);
                } else {
                    const long long po = ((long long)seg * R + row) * D + dd;
                    if (in_bounds(po, 1, parts_rows * D, &g_dec_status)) p.o_parts[po] = v;
                }
            }
        }
        if (g8 == 0) {
            if (p.splits == 1) {
                if (in_bounds(row, 1, R, &g_dec_status)) p.lse[row] = lsev;
            } else if (in_bounds((long long)seg * R + row, 1, parts_rows, &g_dec_status)) {
                p.lse_parts[(long long)seg * R + row] = lsev;
            }
        }
    }
}

// lse = M + log sum_s exp(lse_s - M), o = sum_s exp(lse_s - lse) o_s, one CTA
// per row.  The merge sits between two HBM-bound launches and moves a few
// hundred KB, so its cost is round trips, not bytes: every load of a pass is
// independent.  Pass 1 reads all P lse_s at once (one per thread) and reduces
// max and sum across the CTA; pass 2 spreads (segment, 4-column group) pairs
// over the threads, so the P x d/4 partial loads are issued together, and the
// per-segment sums are reduced through shared memory.
constexpr int kMergeThreads = 256;
constexpr int kMergeChunk = 1024;  // segment weights staged in shared memory per pass

__device__ __forceinline__ float block_reduce(float x, bool is_max, float* red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, off);
        x = is_max ? fmaxf(x, y) : x + y;
    }
    __syncthreads();  // red may still be read from a previous reduction
    if (lane == 0) red[w] = x;
    __syncthreads();
    x = red[0];
#pragma unroll
    for (int i = 1; i < kMergeThreads / 32; ++i) x = is_max ? fmaxf(x, red[i]) : x + red[i];
    return x;
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads)
    merge_lse_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int P,
                     long long rows, int d, void* __restrict__ o, float* __restrict__ lse, long long o_slack) {
    __shared__ float red[kMergeThreads / 32];
    __shared__ float wts[kMergeChunk];
    __shared__ float4 part[kMergeThreads];
    // Launched as a programmatic dependent of the split kernel: wait until that
    // grid has completed and its partials are visible (a no-op otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long row = blockIdx.x;
    const int tid = threadIdx.x;
    // (bounds-checked build) a partial's LSE, or -inf if it lies outside lse_parts
    auto lse_part = [&](int s) {
        const long long off = (long long)s * rows + row;
        return in_bounds(off, 1, (long long)P * rows, &g_dec_status) ? lse_parts[off] : -INFINITY;
    };
    float M = -INFINITY;
    for (int s = tid; s < P; s += kMergeThreads) M = fmaxf(M, lse_part(s));
    M = block_reduce(M, true, red);
    float Lr = -INFINITY;
    if (M != -INFINITY) {  // uniform across the CTA
        float sum = 0.f;
        for (int s = tid; s < P; s += kMergeThreads) sum += expf(lse_part(s) - M);
        Lr = M + logf(block_reduce(sum, false, red));
    }
    const int C = d >> 2;               // 4-column groups, 1..128
    const int SL = kMergeThreads / C;   // segment lanes, >= 2
    const int c4 = tid % C, sl = tid / C;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Lr != -INFINITY) {
        for (int s0 = 0; s0 < P; s0 += kMergeChunk) {
            const int n = min(kMergeChunk, P - s0);
            __syncthreads();  // wts of the previous chunk fully consumed
            for (int i = tid; i < n; i += kMergeThreads) {
                const float ls = lse_part(s0 + i);
                wts[i] = ls == -INFINITY ? 0.f : expf(ls - Lr);
            }
            __syncthreads();
            if (sl < SL) {
#pragma unroll 4
                for (int i = sl; i < n; i += SL) {
                    const float w = wts[i];
                    const long long off = ((long long)(s0 + i) * rows + row) * d + 4 * c4;
                    if (!in_bounds(off, 4, (long long)P * rows * d, &g_dec_status)) continue;
                    const float4 x = *reinterpret_cast<const float4*>(o_parts + off);
                    a.x = fmaf(w, x.x, a.x);
                    a.y = fmaf(w, x.y, a.y);
                    a.z = fmaf(w, x.z, a.z);
                    a.w = fmaf(w, x.w, a.w);
                }
            }
        }
    }
    part[tid] = a;
    __syncthreads();
    if (tid < C && in_bounds(row * d + 4 * tid, 4, rows * d - o_slack, &g_dec_status)) {
        for (int j = 1; j < SL; ++j) {
            const float4 x = part[j * C + tid];
            a.x += x.x;
            a.y += x.y;
            a.z += x.z;
            a.w += x.w;
        }
        if constexpr (OUT_BF16) {
            uint2 h;
            h.x = pack_bf16(a.x, a.y);
            h.y = pack_bf16(a.z, a.w);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + row * d + 4 * tid) = h;
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(o) + row * d + 4 * tid) = a;
        }
    }
    if (tid == 0 && lse != nullptr && in_bounds(row, 1, rows, &g_dec_status)) lse[row] = Lr;
}

// The same merge in one pass for few segments (at most NSEG per thread:
// kShortSeg, or kShortSegWide for up to 152 segments at d = 128): every thread issues the loads of its segments' LSE and partial
// outputs at once, so the merge costs one round trip to L2 instead of two;
// o = sum_s e^{lse_s - M} o_s / sum_s e^{lse_s - M} and lse = M + ln of that
// sum (M = max_s lse_s), the same value as merge_lse_kernel up to rounding.
constexpr int kShortSeg = 4;   // segments per thread of the one-pass merge (P <= 32 at d = 128)
constexpr int kShortSegWide = 19;  // the same for P <= 152 at d = 128 (many-segment paged decodes)

template <bool OUT_BF16, int NSEG>
__global__ void __launch_bounds__(kMergeThreads)
    merge_lse_short_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int P,
                           long long rows, int d, void* __restrict__ o, float* __restrict__ lse,
                           long long o_slack) {
    __shared__ float red[kMergeThreads / 32];
    __shared__ float4 part[kMergeThreads];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long row = blockIdx.x;
    const int tid = threadIdx.x;
    const int C = d >> 2;              // 4-column groups, 1..128
    const int SL = kMergeThreads / C;  // segment lanes, >= 2
    const int c4 = tid % C, sl = tid / C;
    float ls[NSEG];
    float4 x[NSEG];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < NSEG; ++r) {
        const int s = sl + r * SL;
        const long long lo = (long long)s * rows + row, oo = lo * d + 4 * c4;
        const bool ok = sl < SL && s < P && in_bounds(lo, 1, (long long)P * rows, &g_dec_status) &&
                        in_bounds(oo, 4, (long long)P * rows * d, &g_dec_status);
        ls[r] = ok ? lse_parts[lo] : -INFINITY;
        x[r] = ok ? *reinterpret_cast<const float4*>(o_parts + oo) : make_float4(0.f, 0.f, 0.f, 0.f);
        M = fmaxf(M, ls[r]);
    }
    M = block_reduce(M, true, red);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    if (M != -INFINITY) {  // uniform across the CTA
#pragma unroll
        for (int r = 0; r < NSEG; ++r) {
            if (ls[r] == -INFINITY) continue;
            const float w = expf(ls[r] - M);
            a.x = fmaf(w, x[r].x, a.x);
            a.y = fmaf(w, x[r].y, a.y);
            a.z = fmaf(w, x[r].z, a.z);
            a.w = fmaf(w, x[r].w, a.w);
            if (c4 == 0) lsum += w;  // each segment counted once
        }
    }
    part[tid] = a;
    lsum = block_reduce(lsum, false, red);  // its barriers also publish part[]
    if (tid < C && in_bounds(row * d + 4 * tid, 4, rows * d - o_slack, &g_dec_status)) {
        for (int j = 1; j < SL; ++j) {
            const float4 y = part[j * C + tid];
            a.x += y.x;
            a.y += y.y;
            a.z += y.z;
            a.w += y.w;
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        a.x *= inv;
        a.y *= inv;
        a.z *= inv;
        a.w *= inv;
        if constexpr (OUT_BF16) {
            uint2 h;
            h.x = pack_bf16(a.x, a.y);
            h.y = pack_bf16(a.z, a.w);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + row * d + 4 * tid) = h;
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(o) + row * d + 4 * tid) = a;
        }
    }
    if (tid == 0 && lse != nullptr && in_bounds(row, 1, rows, &g_dec_status))
        lse[row] = lsum > 0.f ? M + logf(lsum) : -INFINITY;
}

// decode_heads_kernel serves pages of 16 keys with 2, 4 or 8 KV heads of at
// most 8 query heads each; every other paged cache takes decode_split_kernel.
bool heads_path(int Hq, int Hkv, int page_size, int d) {
    return page_size == kSmallPage && (Hkv == 8 || Hkv == 4 || Hkv == 2) && Hq % Hkv == 0 &&
           Hq / Hkv <= 8 && (d == 64 || d == 128);
}

template <int D, int NH>
attn_status_t launch_heads_nh(const CUtensorMap& mk, const CUtensorMap& mv, const DecParams& prm,
                              cudaStream_t stream) {
    using L = HeadsLayout<D, NH>;
    if (attn_host::kernel_setup<decode_heads_kernel<D, NH>>(L::kSmemBytes).err != cudaSuccess)
        return ATTN_ERR_CUDA;
    dim3 grid(prm.splits, 1, prm.B);
    decode_heads_kernel<D, NH><<<grid, kHeadsThreads, L::kSmemBytes, stream>>>(mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
attn_status_t launch_heads(const CUtensorMap& mk, const CUtensorMap& mv, const DecParams& prm,
                           cudaStream_t stream) {
    return prm.Hkv == 8   ? launch_heads_nh<D, 8>(mk, mv, prm, stream)
           : prm.Hkv == 4 ? launch_heads_nh<D, 4>(mk, mv, prm, stream)
                          : launch_heads_nh<D, 2>(mk, mv, prm, stream);
}

int group_cols(int G) {
    if (G % 8 == 0) return 8;
    if (G % 4 == 0) return 4;
    if (G % 2 == 0) return 2;
    return 1;
}

template <int D, int GC, bool PAGED>
attn_status_t launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const DecParams& prm,
                           cudaStream_t stream) {
    using L = DecLayout<D, dec_stages<D>(), PAGED>;
    if (attn_host::kernel_setup<decode_split_kernel<D, GC, PAGED>>(L::kSmemBytes).err != cudaSuccess)
        return ATTN_ERR_CUDA;
    dim3 grid(prm.splits, prm.Hq / GC, prm.B);
    decode_split_kernel<D, GC, PAGED><<<grid, kDecThreads, L::kSmemBytes, stream>>>(mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <bool PAGED>
attn_status_t launch_split_any(int d, const CUtensorMap& mk, const CUtensorMap& mv,
                               const DecParams& prm, cudaStream_t stream) {
    const int GC = group_cols(prm.G);
    if (d == 128)
        return GC == 8   ? launch_split<128, 8, PAGED>(mk, mv, prm, stream)
               : GC == 4 ? launch_split<128, 4, PAGED>(mk, mv, prm, stream)
               : GC == 2 ? launch_split<128, 2, PAGED>(mk, mv, prm, stream)
                         : launch_split<128, 1, PAGED>(mk, mv, prm, stream);
    return GC == 8   ? launch_split<64, 8, PAGED>(mk, mv, prm, stream)
           : GC == 4 ? launch_split<64, 4, PAGED>(mk, mv, prm, stream)
           : GC == 2 ? launch_split<64, 2, PAGED>(mk, mv, prm, stream)
                     : launch_split<64, 1, PAGED>(mk, mv, prm, stream);
}

// Resident split-kernel CTAs per SM on the current device (cached per device).
template <int D>
int ctas_per_sm() {
    static attn_host::PerDevice<int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int n = 1;
    const bool ok = cache.get(dev, &n, [&](int* out) {
        using L = DecLayout<D, dec_stages<D>()>;
        int k = 0;
        if (attn_host::kernel_setup<decode_split_kernel<D, 4, false>>(L::kSmemBytes).err != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, decode_split_kernel<D, 4, false>,
                                                          kDecThreads, L::kSmemBytes) != cudaSuccess)
            return false;
        *out = std::max(1, k);
        return true;
    });
    return ok ? n : 1;
}

}  // namespace

namespace attn_host {

// Segment count from a CTA-by-wave time model (Lecture 11, sections 6.3-6.4,
// whose exercise 9 works the same model on an A100: 32 segments of 64 CTAs in
// one wave beat 64 segments of 128 CTAs in two): split_model_time and
// split_model_best below.
// Contiguous cache: fitted on GB300 to the measured best segment counts of
// B = 1 x 2K-64K, B = 4 x 4K and 16K, B = 8 x 8K, B = 16 x 8K and B = 32 x 2K
// keys (Hq = 32, Hkv = 8, d = 128), timed with L2 holding only clean lines;
// a CTA streams ~80-110 GB/s while few compete and the grid as a whole
// ~7-7.7 TB/s once the ring is full, so one long sequence wants ~12 segments
// and batches of several sequences few or none.
constexpr SplitModel kDenseSplitModel = {8.0e10, 7.5e12, 0.5e-6, 4.0e-6};

// Modelled time (seconds) of S segments when every segment has `units` CTAs
// and `slots` CTAs fit on the GPU at once: waves of CTAs, each streaming its
// segment's K/V rows at min(cta_bw, hbm / concurrent CTAs) after a fixed
// start-up, then (S > 1) the merge launch and its partial traffic.
double split_model_time(long long units, long long slots, int Nk, int d, int S, const SplitModel& m) {
    const long long ctas = units * S;
    const long long waves = (ctas + slots - 1) / slots;
    const double conc = (double)std::min(ctas, slots);
    const double bw = std::min(m.cta_bw, m.hbm / conc);
    const double row_bytes = 2.0 * d * 2.0;  // one key's K and V for one head
    const int seg = (Nk + S - 1) / S;
    return (double)waves * (seg * row_bytes / bw + m.cta_fixed) +
           (S > 1 ? m.merge_fixed + 2.0 * units * 8 * S * (d + 1) * 4.0 / m.hbm : 0.0);
}

// The segment count with the smallest modelled time (ties, within 0.5%, go
// to fewer segments).  With single_wave the count is capped so that all CTAs
// run in one wave and segments are whole 64-key tiles.
int split_model_best(long long units, long long slots, int Nk, int d, const SplitModel& m, bool single_wave) {
    int best = 1;
    double best_t = 1e30;
    int max_s = std::min(Nk, 1024);
    if (single_wave) {
        // (paged) segments are whole 64-key tiles: more than Nk / 64 of them would be empty
        max_s = std::min(max_s, (Nk + kTileKeys - 1) / kTileKeys);
        max_s = (int)std::max(1LL, std::min((long long)max_s, slots / units));
    }
    for (int S = 1; S <= max_s; ++S) {
        const double t = split_model_time(units, slots, Nk, d, S, m);
        if (t < best_t * 0.995) {
            best_t = t;
            best = S;
        }
    }
    return best;
}

static int auto_splits_model(int B, int Hq, int Hkv, int Nk, int d, const SplitModel& m, bool single_wave) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nk < 1 || (d != 64 && d != 128)) return -1;
    const int sms = device_sm_count();
    if (sms <= 0) return -1;
    const int per_sm = d == 128 ? ctas_per_sm<128>() : ctas_per_sm<64>();
    const long long slots = (long long)sms * per_sm;
    const long long units = (long long)B * (Hq / group_cols(Hq / Hkv));
    return split_model_best(units, slots, Nk, d, m, single_wave);
}

int decode_auto_splits(int B, int Hq, int Hkv, int Nk, int d) {
    return auto_splits_model(B, Hq, Hkv, Nk, d, kDenseSplitModel, false);
}

size_t decode_workspace_bytes(int B, int Hq, int d, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = (size_t)B * Hq;
    const size_t o_bytes = (size_t)splits * rows * d * 4;
    const size_t o_round = (o_bytes + 255) / 256 * 256;
    return o_round + (size_t)splits * rows * 4;
}

attn_status_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                            int Hq, int Hkv, int Nk, int d, float scale, int splits,
                            void* workspace, cudaStream_t stream, const attn_test_options_t* test) {
    CUtensorMap mk, mv;
    if (!encode_bshd_map(&mk, k, B, Nk, Hkv, d, kTileKeys, 2) ||
        !encode_bshd_map(&mv, v, B, Nk, Hkv, d, kTileKeys, 2))
        return ATTN_ERR_CUDA;
    DecParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    prm.splits = splits;
    prm.seg_len = (Nk + splits - 1) / splits;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.wait_limit = (test && test->wait_limit_cycles > 0) ? test->wait_limit_cycles : kWaitLimitCycles;
    prm.skip_load = test ? test->skip_load : -1;
    prm.o_slack = test ? test->o_extent_slack : 0;
    const size_t rows = (size_t)B * Hq;
    if (splits > 1) {
        const size_t o_bytes = (size_t)splits * rows * d * 4;
        prm.o_parts = static_cast<float*>(workspace);
        prm.lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                 (o_bytes + 255) / 256 * 256);
    } else {
        prm.o_parts = nullptr;
        prm.lse_parts = nullptr;
    }
    prm.table = nullptr;
    prm.seq_lens = nullptr;
    prm.page_size = 0;
    prm.max_pages = 0;
    const attn_status_t st = launch_split_any<false>(d, mk, mv, prm, stream);
    if (st != ATTN_OK || splits == 1) return st;
    return launch_merge(prm.o_parts, prm.lse_parts, splits, (long long)rows, d, o, lse, true, stream,
                        prm.o_slack);
}

// Segment length of the paged kernel: whole 64-key tiles, so that a tile never
// straddles a page of 64 or more keys.
static int paged_seg_len(int max_seq_len, int splits) {
    const int seg = (max_seq_len + splits - 1) / splits;
    return (seg + kTileKeys - 1) / kTileKeys * kTileKeys;
}

bool paged_splits_fit(int max_seq_len, int page_size, int splits) {
    // pages one segment can touch: its keys / page_size, plus one partial page at each end
    const long long seg = paged_seg_len(max_seq_len, splits);
    return seg / page_size + 2 <= kTableCap;
}

int decode_paged_auto_splits(int B, int Hq, int Hkv, int max_seq_len, int d, int page_size) {
    int S;
    if (heads_path(Hq, Hkv, page_size, d)) {
        // One CTA per (segment, sequence) for all KV heads, one CTA per SM,
        // each segment whole 64-key tiles.
        const int sms = device_sm_count();
        if (sms <= 0) return -1;
        const int max_s = std::max(1, (max_seq_len + kTileKeys - 1) / kTileKeys);
        S = std::max(1, std::min(max_s, heads_target_ctas(sms) / std::max(1, B)));
    } else {
        // Pages of 64 or more keys stream like the contiguous cache.  Smaller
        // pages split every tile into 64 / page_size boxes at random places,
        // and one CTA sustains less (rates fitted to 64K and 16K keys, d =
        // 128: ~33 GB/s with 16-key pages, ~52 with 32-key pages), so more
        // CTAs are needed to keep HBM busy; but a second wave of such CTAs
        // costs more than it gains (B = 16 x 8K keys: one segment per
        // sequence beats eight), so they are kept to one wave.
        const bool small = page_size < 64;
        const double cta_bw = !small ? 6.0e10 : page_size >= 32 ? 5.2e10 : 3.3e10;
        S = auto_splits_model(B, Hq, Hkv, max_seq_len, d, SplitModel{cta_bw, 6.5e12, 1.5e-6, 3.0e-6}, small);
        if (S < 1) return S;
    }
    // every count attn_decode_paged accepts keeps one segment's pages within
    // the block-table staging area
    while (!paged_splits_fit(max_seq_len, page_size, S) && S < max_seq_len) ++S;
    return S;
}

attn_status_t launch_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                  const int* block_table, const int* seq_lens, void* o, float* lse,
                                  int B, int Hq, int Hkv, int d, int num_pages, int page_size,
                                  int max_pages, int max_seq_len, float scale, int splits,
                                  void* workspace, cudaStream_t stream) {
    const bool heads = heads_path(Hq, Hkv, page_size, d);
    const int box = page_size < kTileKeys ? page_size : kTileKeys;
    CUtensorMap mk, mv;
    if (heads ? (!encode_page_heads_map(&mk, k_pages, num_pages, page_size, Hkv, d) ||
                 !encode_page_heads_map(&mv, v_pages, num_pages, page_size, Hkv, d))
              : (!encode_bshd_map(&mk, k_pages, num_pages, page_size, Hkv, d, box, 2) ||
                 !encode_bshd_map(&mv, v_pages, num_pages, page_size, Hkv, d, box, 2)))
        return ATTN_ERR_CUDA;
    DecParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nk = max_seq_len;
    prm.G = Hq / Hkv;
    prm.splits = splits;
    prm.seg_len = paged_seg_len(max_seq_len, splits);
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.wait_limit = kWaitLimitCycles;
    prm.skip_load = -1;
    prm.o_slack = 0;
    prm.table = block_table;
    prm.seq_lens = seq_lens;
    prm.page_size = page_size;
    prm.max_pages = max_pages;
    const size_t rows = (size_t)B * Hq;
    if (splits > 1) {
        const size_t o_bytes = (size_t)splits * rows * d * 4;
        prm.o_parts = static_cast<float*>(workspace);
        prm.lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                 (o_bytes + 255) / 256 * 256);
    } else {
        prm.o_parts = nullptr;
        prm.lse_parts = nullptr;
    }
    const attn_status_t st = heads ? (d == 128 ? launch_heads<128>(mk, mv, prm, stream)
                                               : launch_heads<64>(mk, mv, prm, stream))
                                   : launch_split_any<true>(d, mk, mv, prm, stream);
    if (st != ATTN_OK || splits == 1) return st;
    return launch_merge(prm.o_parts, prm.lse_parts, splits, (long long)rows, d, o, lse, true, stream);
}

attn_status_t launch_merge(const float* o_parts, const float* lse_parts, int parts,
                           long long rows, int d, void* o, float* lse, bool out_bf16,
                           cudaStream_t stream, long long o_slack) {
    if (rows == 0) return ATTN_OK;
    if (rows > 0x7fffffffLL || d < 4 || d > 4 * kMergeThreads / 2 || d % 4 != 0)
        return ATTN_ERR_UNSUPPORTED;
    const long long blocks = rows;
    // Programmatic dependent launch: the merge grid is scheduled while the
    // previous kernel on the stream drains, instead of after a full launch gap.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int seg_lanes = kMergeThreads / (d / 4);
    cudaError_t e;
    if (parts <= kShortSeg * seg_lanes)
        e = out_bf16 ? cudaLaunchKernelEx(&cfg, merge_lse_short_kernel<true, kShortSeg>, o_parts, lse_parts, parts,
                                          rows, d, o, lse, o_slack)
                     : cudaLaunchKernelEx(&cfg, merge_lse_short_kernel<false, kShortSeg>, o_parts, lse_parts, parts,
                                          rows, d, o, lse, o_slack);
    else if (parts <= kShortSegWide * seg_lanes)
        e = out_bf16 ? cudaLaunchKernelEx(&cfg, merge_lse_short_kernel<true, kShortSegWide>, o_parts, lse_parts,
                                          parts, rows, d, o, lse, o_slack)
                     : cudaLaunchKernelEx(&cfg, merge_lse_short_kernel<false, kShortSegWide>, o_parts, lse_parts,
                                          parts, rows, d, o, lse, o_slack);
    else
        e = out_bf16 ? cudaLaunchKernelEx(&cfg, merge_lse_kernel<true>, o_parts, lse_parts, parts, rows, d, o, lse, o_slack)
                     : cudaLaunchKernelEx(&cfg, merge_lse_kernel<false>, o_parts, lse_parts, parts, rows, d, o, lse, o_slack);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

cudaError_t decode_read_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_dec_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_dec_status, &zero, sizeof(unsigned));
}

}  // namespace attn_host
