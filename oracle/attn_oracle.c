/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of exact attention and of the
 * flash-decoding merge.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library; the product path (the CUDA
 * library) never calls it, links it or shares code with it.
 *
 * Sources (page titles; sections as printed on the pages):
 *   [L11]  "Lecture 11 - Kernel Optimization Techniques: FlashAttention,
 *          flash-decoding and megakernel" (CS349E notes).
 *   [IDX]  "CUDA Kernel course index - FlashAttention v1->v4 diagrams".
 *
 * Conventions shared with the CUDA path only through the public header's
 * documented meaning (no code is shared):
 *   q, o : [B, Nq, Hq, d] row-major;  k, v : [B, Nk, Hkv, d] row-major.
 *   lse  : [B, Hq, Nq].
 *   GQA  : query head hq reads key/value head hq / (Hq / Hkv).
 *   causal: query row i may attend key j iff j <= i + (Nk - Nq)
 *          (bottom-right alignment; with Nq == Nk this is j <= i).
 *   A row with no allowed key has O = 0 and LSE = -inf.
 *
 * Inputs arrive as float32 arrays.  Every bf16 and every fp32 value is
 * exactly representable in float32, so the oracle sees the same numbers as
 * the GPU; all arithmetic below is in double.
 *
 * Parity pins: every exported function is pinned by tests that do not
 * re-derive it (worked example of [L11] exercise 1, causal block fraction of
 * [L11] section 5.3, closed forms, invariants, brute force on tiny inputs).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Last key index row i may attend (inclusive), or -1 if none. */
static long last_allowed_key(long i, long Nq, long Nk, int causal) {
    long last = Nk - 1;
    if (causal) {
        long lim = i + (Nk - Nq);
        if (lim < last) last = lim;
    }
    return last < 0 ? -1 : last;
}

static const float* qrow(const float* q, long b, long i, long h, long Nq, long Hq, long d) {
    return q + ((b * Nq + i) * Hq + h) * d;
}
static const float* kvrow(const float* k, long b, long j, long g, long Nk, long Hkv, long d) {
    return k + ((b * Nk + j) * Hkv + g) * d;
}

/*
 * One output row of standard attention, "algorithm 0" ([L11] section 2):
 *   S = Q K^T * scale   (one row, materialised in s[]),
 *   P = softmax(S)      (safe softmax: subtract the row max, [L11] 3.4),
 *   O = P V,            and LSE = m + ln(l) ([L11] 5.1, the statistic the
 *                       forward pass stores for the backward pass).
 */
static void attn_row(const float* q, const float* k, const float* v,
                     long B, long Hq, long Hkv, long Nq, long Nk, long d,
                     int causal, double scale, long b, long hq, long i,
                     double* s, double* o_row, double* lse_out) {
    (void)B;
    long G = Hq / Hkv;
    long g = hq / G;
    long last = last_allowed_key(i, Nq, Nk, causal);
    for (long t = 0; t < d; ++t) o_row[t] = 0.0;
    if (last < 0) {
        *lse_out = -INFINITY;
        return;
    }
    const float* qi = qrow(q, b, i, hq, Nq, Hq, d);
    /* S row */
    for (long j = 0; j <= last; ++j) {
        const float* kj = kvrow(k, b, j, g, Nk, Hkv, d);
        double acc = 0.0;
        for (long t = 0; t < d; ++t) acc += (double)qi[t] * (double)kj[t];
        s[j] = acc * scale;
    }
    /* P row = softmax(S row) */
    double m = -INFINITY;
    for (long j = 0; j <= last; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (long j = 0; j <= last; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (long j = 0; j <= last; ++j) s[j] /= l;
    /* O row = P row V */
    for (long j = 0; j <= last; ++j) {
        const float* vj = kvrow(v, b, j, g, Nk, Hkv, d);
        double pj = s[j];
        for (long t = 0; t < d; ++t) o_row[t] += pj * (double)vj[t];
    }
    *lse_out = m + log(l);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int bad_shape(long B, long Hq, long Hkv, long Nq, long Nk, long d) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

/* Full forward: every (b, hq, i) row.  o: [B,Nq,Hq,d]; lse: [B,Hq,Nq]. */
int oracle_attn_fwd(const float* q, const float* k, const float* v,
                    long B, long Hq, long Hkv, long Nq, long Nk, long d,
                    int causal, double scale, double* o, double* lse) {
    if (bad_shape(B, Hq, Hkv, Nq, Nk, d)) return 1;
    long rows = B * Hq * Nq;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            long i = r % Nq;
            long hq = (r / Nq) % Hq;
            long b = r / (Nq * Hq);
            double* o_row = o + ((b * Nq + i) * Hq + hq) * d;
            attn_row(q, k, v, B, Hq, Hkv, Nq, Nk, d, causal, scale, b, hq, i,
                     s, o_row, lse + (b * Hq + hq) * Nq + i);
        }
        free(s);
    }
    return 0;
}

/* Selected rows only: sel holds nsel triples (b, hq, i); o_sel [nsel, d]. */
int oracle_attn_rows(const float* q, const float* k, const float* v,
                     long B, long Hq, long Hkv, long Nq, long Nk, long d,
                     int causal, double scale, long nsel, const long* sel,
                     double* o_sel, double* lse_sel) {
    if (bad_shape(B, Hq, Hkv, Nq, Nk, d)) return 1;
    for (long r = 0; r < nsel; ++r) {
        long b = sel[3 * r], hq = sel[3 * r + 1], i = sel[3 * r + 2];
        if (b < 0 || b >= B || hq < 0 || hq >= Hq || i < 0 || i >= Nq) return 2;
    }
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < nsel; ++r) {
            attn_row(q, k, v, B, Hq, Hkv, Nq, Nk, d, causal, scale,
                     sel[3 * r], sel[3 * r + 1], sel[3 * r + 2], s,
                     o_sel + r * d, lse_sel + r);
        }
        free(s);
    }
    return 0;
}

/*
 * Tiled forward with the online softmax, in the order of the "FlashAttention
 * v1" concept pseudocode of [IDX] (one query block at a time, key/value blocks
 * streamed), with deferred normalisation ([L11] 3.3: scale the accumulator by
 * alpha per block, divide by l once at the end).  Per block j and row:
 *   m_new = max(m, rowmax(S_ij));  alpha = exp(m - m_new);
 *   P = exp(S_ij - m_new);  l = alpha*l + rowsum(P);  acc = alpha*acc + P V_j.
 * Blocks whose every entry is causally masked are skipped ([L11] 5.3); the
 * number of (query block, key block) pairs actually computed is returned in
 * *blocks_computed so the skip rule can be checked against the fractions the
 * notes report.
 */
int oracle_attn_fwd_tiled(const float* q, const float* k, const float* v,
                          long B, long Hq, long Hkv, long Nq, long Nk, long d,
                          int causal, double scale, long Br, long Bc,
                          double* o, double* lse, long* blocks_computed) {
    if (bad_shape(B, Hq, Hkv, Nq, Nk, d) || Br < 1 || Bc < 1) return 1;
    long G = Hq / Hkv;
    long Tr = (Nq + Br - 1) / Br, Tc = (Nk + Bc - 1) / Bc;
    long total_blocks = 0;
#pragma omp parallel reduction(+ : total_blocks)
    {
        double* m = (double*)malloc(sizeof(double) * (size_t)Br);
        double* l = (double*)malloc(sizeof(double) * (size_t)Br);
        double* acc = (double*)malloc(sizeof(double) * (size_t)(Br * d));
        double* S = (double*)malloc(sizeof(double) * (size_t)(Br * Bc));
#pragma omp for schedule(dynamic, 1)
        for (long w = 0; w < B * Hq * Tr; ++w) {
            long ti = w % Tr, hq = (w / Tr) % Hq, b = w / (Tr * Hq);
            long g = hq / G;
            long i0 = ti * Br, i1 = i0 + Br < Nq ? i0 + Br : Nq;
            for (long r = 0; r < i1 - i0; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (long t = 0; t < d; ++t) acc[r * d + t] = 0.0;
            }
            for (long tj = 0; tj < Tc; ++tj) {
                long j0 = tj * Bc, j1 = j0 + Bc < Nk ? j0 + Bc : Nk;
                /* skip a block only if it is masked for every row */
                if (causal && j0 > last_allowed_key(i1 - 1, Nq, Nk, causal)) continue;
                total_blocks += 1;
                for (long r = 0; r < i1 - i0; ++r) {
                    long i = i0 + r;
                    long last = last_allowed_key(i, Nq, Nk, causal);
                    const float* qi = qrow(q, b, i, hq, Nq, Hq, d);
                    double* Sr = S + r * Bc;
                    double rowmax = -INFINITY;
                    for (long j = j0; j < j1; ++j) {
                        if (j > last) { Sr[j - j0] = -INFINITY; continue; }
                        const float* kj = kvrow(k, b, j, g, Nk, Hkv, d);
                        double a = 0.0;
                        for (long t = 0; t < d; ++t) a += (double)qi[t] * (double)kj[t];
                        Sr[j - j0] = a * scale;
                        if (Sr[j - j0] > rowmax) rowmax = Sr[j - j0];
                    }
                    double m_new = m[r] > rowmax ? m[r] : rowmax;
                    if (m_new == -INFINITY) continue; /* nothing allowed yet */
                    double alpha = exp(m[r] - m_new);
                    double rowsum = 0.0;
                    for (long t = 0; t < d; ++t) acc[r * d + t] *= alpha;
                    for (long j = j0; j < j1; ++j) {
                        double p = exp(Sr[j - j0] - m_new);
                        rowsum += p;
                        if (p == 0.0) continue;
                        const float* vj = kvrow(v, b, j, g, Nk, Hkv, d);
                        for (long t = 0; t < d; ++t) acc[r * d + t] += p * (double)vj[t];
                    }
                    l[r] = alpha * l[r] + rowsum;
                    m[r] = m_new;
                }
            }
            for (long r = 0; r < i1 - i0; ++r) {
                long i = i0 + r;
                double* o_row = o + ((b * Nq + i) * Hq + hq) * d;
                if (l[r] > 0.0) {
                    for (long t = 0; t < d; ++t) o_row[t] = acc[r * d + t] / l[r];
                    lse[(b * Hq + hq) * Nq + i] = m[r] + log(l[r]);
                } else {
                    for (long t = 0; t < d; ++t) o_row[t] = 0.0;
                    lse[(b * Hq + hq) * Nq + i] = -INFINITY;
                }
            }
        }
        free(m); free(l); free(acc); free(S);
    }
    if (blocks_computed) *blocks_computed = total_blocks;
    return 0;
}

/*
 * Online softmax over one score row x[0..n), consumed in blocks of `block`
 * entries ([L11] 3.1; [L11] exercise 1 is the worked example).  After block
 * b the running max and sum are stored in m_trace[b], l_trace[b], and the
 * factor alpha = exp(m_old - m_new) applied to the old sum in alpha_trace[b]
 * (alpha of the first block is 0 by the convention exp(-inf)).
 */
void oracle_online_trace(const double* x, long n, long block,
                         double* m_trace, double* l_trace, double* alpha_trace) {
    double m = -INFINITY, l = 0.0;
    long nb = 0;
    for (long j0 = 0; j0 < n; j0 += block, ++nb) {
        long j1 = j0 + block < n ? j0 + block : n;
        double bm = -INFINITY;
        for (long j = j0; j < j1; ++j)
            if (x[j] > bm) bm = x[j];
        double m_new = m > bm ? m : bm;
        double alpha = exp(m - m_new);
        double s = 0.0;
        for (long j = j0; j < j1; ++j) s += exp(x[j] - m_new);
        l = alpha * l + s;
        m = m_new;
        m_trace[nb] = m;
        l_trace[nb] = l;
        alpha_trace[nb] = alpha;
    }
}

/*
 * Partial state of one key segment [j0, j1) for one query row ([L11] 3.2):
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  acc = sum_j exp(s_j - m) v_j
 * (acc unnormalised).  An empty or fully masked segment gives m = -inf,
 * l = 0, acc = 0.
 */
void oracle_segment_state(const float* q, const float* k, const float* v,
                          long B, long Hq, long Hkv, long Nq, long Nk, long d,
                          int causal, double scale, long b, long hq, long i,
                          long j0, long j1, double* m_out, double* l_out,
                          double* acc_out) {
    (void)B;
    long G = Hq / Hkv, g = hq / G;
    long last = last_allowed_key(i, Nq, Nk, causal);
    if (j1 > last + 1) j1 = last + 1;
    for (long t = 0; t < d; ++t) acc_out[t] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (j1 <= j0) return;
    const float* qi = qrow(q, b, i, hq, Nq, Hq, d);
    double* s = (double*)malloc(sizeof(double) * (size_t)(j1 - j0));
    double m = -INFINITY;
    for (long j = j0; j < j1; ++j) {
        const float* kj = kvrow(k, b, j, g, Nk, Hkv, d);
        double a = 0.0;
        for (long t = 0; t < d; ++t) a += (double)qi[t] * (double)kj[t];
        s[j - j0] = a * scale;
        if (s[j - j0] > m) m = s[j - j0];
    }
    double l = 0.0;
    for (long j = j0; j < j1; ++j) {
        double p = exp(s[j - j0] - m);
        l += p;
        const float* vj = kvrow(v, b, j, g, Nk, Hkv, d);
        for (long t = 0; t < d; ++t) acc_out[t] += p * (double)vj[t];
    }
    free(s);
    *m_out = m;
    *l_out = l;
}

/*
 * Merge of two partial states (m_a, l_a, acc_a) and (m_b, l_b, acc_b) of the
 * same row ([L11] 3.2; the printed formula is lost, this is the reading that
 * the running update of [L11] 3.1 implies):
 *   m = max(m_a, m_b);  l = exp(m_a - m) l_a + exp(m_b - m) l_b;
 *   acc = exp(m_a - m) acc_a + exp(m_b - m) acc_b.
 * A state with m = -inf is empty and contributes nothing.  Output may alias
 * either input.
 */
void oracle_state_merge(double m_a, double l_a, const double* acc_a,
                        double m_b, double l_b, const double* acc_b, long d,
                        double* m_out, double* l_out, double* acc_out) {
    double m = m_a > m_b ? m_a : m_b;
    if (m == -INFINITY) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        for (long t = 0; t < d; ++t) acc_out[t] = 0.0;
        return;
    }
    double ca = m_a == -INFINITY ? 0.0 : exp(m_a - m);
    double cb = m_b == -INFINITY ? 0.0 : exp(m_b - m);
    for (long t = 0; t < d; ++t) acc_out[t] = ca * acc_a[t] + cb * acc_b[t];
    *l_out = ca * l_a + cb * l_b;
    *m_out = m;
}

/*
 * Flash-decoding merge in log-sum-exp form ([L11] 6.2, step 3):
 *   lse = log sum_s exp(lse_s);  o = sum_s exp(lse_s - lse) o_s,
 * with every o_s already normalised within its segment.  The sum is taken
 * after subtracting max_s lse_s so that no term overflows.  Parts with
 * lse_s = -inf (empty segments) contribute nothing; if all are empty the row
 * gets o = 0, lse = -inf.
 * o_parts: [nparts, rows, d]; lse_parts: [nparts, rows]; o: [rows, d].
 */
void oracle_merge_lse(long nparts, long rows, long d, const double* o_parts,
                      const double* lse_parts, double* o, double* lse) {
    for (long r = 0; r < rows; ++r) {
        double mx = -INFINITY;
        for (long s = 0; s < nparts; ++s)
            if (lse_parts[s * rows + r] > mx) mx = lse_parts[s * rows + r];
        double* orow = o + r * d;
        for (long t = 0; t < d; ++t) orow[t] = 0.0;
        if (mx == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (long s = 0; s < nparts; ++s) {
            double ls = lse_parts[s * rows + r];
            if (ls != -INFINITY) sum += exp(ls - mx);
        }
        double L = mx + log(sum);
        for (long s = 0; s < nparts; ++s) {
            double ls = lse_parts[s * rows + r];
            if (ls == -INFINITY) continue;
            double w = exp(ls - L);
            const double* os = o_parts + (s * rows + r) * d;
            for (long t = 0; t < d; ++t) orow[t] += w * os[t];
        }
        lse[r] = L;
    }
}

/*
 * Flash-decoding split step ([L11] 6.2, steps 1-2) for Nq = 1: the key range
 * [0, Nk) of every (b, kv head) is cut into nsplit segments of length
 * L = ceil(Nk / nsplit), segment s covering [s L, min((s+1) L, Nk)).  For each
 * query row (b, hq) and segment the normalised partial output o_s and
 * lse_s = log sum_{j in segment} exp(s_j) are written:
 *   o_parts [nsplit, B*Hq, d], lse_parts [nsplit, B*Hq]  (row = b*Hq + hq).
 * q: [B, 1, Hq, d]; k, v: [B, Nk, Hkv, d].
 */
int oracle_decode_split(const float* q, const float* k, const float* v,
                        long B, long Hq, long Hkv, long Nk, long d,
                        double scale, long nsplit, double* o_parts,
                        double* lse_parts) {
    if (bad_shape(B, Hq, Hkv, 1, Nk, d) || nsplit < 1) return 1;
    long L = (Nk + nsplit - 1) / nsplit;
    long rows = B * Hq;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (long s = 0; s < nsplit; ++s) {
        for (long r = 0; r < rows; ++r) {
            long b = r / Hq, hq = r % Hq;
            long j0 = s * L, j1 = j0 + L < Nk ? j0 + L : Nk;
            double m, l;
            double* os = o_parts + (s * rows + r) * d;
            oracle_segment_state(q, k, v, B, Hq, Hkv, 1, Nk, d, 0, scale, b, hq,
                                 0, j0, j1, &m, &l, os);
            if (l > 0.0) {
                for (long t = 0; t < d; ++t) os[t] /= l;
                lse_parts[s * rows + r] = m + log(l);
            } else {
                lse_parts[s * rows + r] = -INFINITY;
            }
        }
    }
    return 0;
}
