/*
 * attn.h -- C ABI of libattn.so: fused exact attention forward and
 * split-KV flash-decoding for NVIDIA GB300 (sm_103a).
 *
 * Sources (page titles, sections as printed on the pages):
 *   [L11] "Lecture 11 - Kernel Optimization Techniques: FlashAttention,
 *         flash-decoding and megakernel" (CS349E notes).
 *   [IDX] "CUDA Kernel course index - FlashAttention v1->v4 diagrams".
 *
 * General conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.
 *     The caller owns every buffer, including decode workspaces.  The
 *     library allocates and frees nothing, never synchronises the stream
 *     and keeps no per-call state; calls are asynchronous on `stream`
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - Layouts are row-major and contiguous ("BSHD"):
 *       q, o   [B, Nq, Hq, d]      k, v   [B, Nk, Hkv, d]
 *       lse    [B, Hq, Nq]  float32 (natural log of the scaled scores)
 *   - GQA: query head hq reads key/value head hq / (Hq / Hkv).
 *   - Causal masking is bottom-right aligned: query row i may attend key j
 *     iff j <= i + (Nk - Nq).  A row with no allowed key gets O = 0 and
 *     LSE = -inf.
 *   - Arguments are checked before anything is launched; a rejected call
 *     launches nothing and writes nothing.  Errors inside a kernel (a bounded
 *     wait that ran out) are recorded in a device status word that
 *     attn_check_device_status() reads and clears.
 *   - Pointers to q/k/v/o and to workspaces must be 16-byte aligned (TMA
 *     and 128-bit accesses); lse must be 4-byte aligned.
 */
#ifndef EXACT_ATTENTION_GB300_ATTN_H
#define EXACT_ATTENTION_GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,      /* bad pointer, size, alignment or scale     */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (d, dtype, G)   */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed         */
    ATTN_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out        */
    ATTN_ERR_BOUNDS = 5        /* debug build only: an in-kernel index check
                                  refused an access outside its buffer      */
} attn_status_t;

typedef enum {
    ATTN_BF16 = 0,  /* q/k/v/o bfloat16, fp32 accumulation, P rounded to bf16 */
    ATTN_F32 = 1    /* q/k/v/o float32, fp32 arithmetic throughout            */
} attn_dtype_t;

/*
 * attn_fwd -- exact attention forward with per-row log-sum-exp.
 *
 * Computes, for every (b, hq, i),
 *     O[b,i,hq,:] = softmax_j( scale * q[b,i,hq,:] . k[b,j,g,:] ) v[b,j,g,:]
 *     lse[b,hq,i] = log sum_j exp( scale * q[b,i,hq,:] . k[b,j,g,:] )
 * over the allowed keys j (g = hq / (Hq/Hkv); causal rule above).  This is
 * standard attention ("algorithm 0", [L11] section 2) evaluated tile by tile
 * with the online softmax and deferred normalisation ([L11] 3.1, 3.3; the
 * "FlashAttention v1" pseudocode of [IDX]); L = m + log l is the statistic of
 * [L11] 5.1.  The result is exact up to floating-point rounding ([L11] 4.1,
 * theorem 1).
 *
 *   q, k, v  inputs (dtype elements, layouts above); read only.
 *   o        output [B, Nq, Hq, d] (dtype elements); fully overwritten.
 *   lse      output [B, Hq, Nq] float32; fully overwritten.
 *   B, Hq, Hkv, Nq, Nk   sizes; B, Hq, Nq may be 0 (nothing to do, ATTN_OK);
 *            Hkv >= 1, Hq % Hkv == 0, Nk >= 0 (Nk == 0: every row empty).
 *   d        head dimension: 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 *   causal   0 or 1.
 *   scale    multiplies q.k; finite and > 0 (commonly 1/sqrt(d)).
 *   dtype    ATTN_BF16: tcgen05 tensor-core kernel (TMA, TMEM accumulators).
 *            ATTN_F32: fp32 CUDA-core kernel (for fp32 accuracy).
 * Returns ATTN_OK once the work is enqueued on `stream`.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int Nq, int Nk,
                       int d, int causal, float scale, attn_dtype_t dtype,
                       void* stream);

/*
 * attn_fwd_host -- attn_fwd with the inputs and outputs in host memory; the
 * transfers overlap the computation.  The pages define no such call; it is
 * the library's end-to-end entry point.
 *   q_h, k_h, v_h, o_h, lse_h  host buffers with the layouts of attn_fwd
 *            (page-locked memory lets the copies run asynchronously; any
 *            host memory is accepted).
 *   q_d, k_d, v_d, o_d, lse_d  device buffers of the same full sizes,
 *            caller-owned, aligned as for attn_fwd.
 *   chunks   the number of chunks n, 1..16; 0 = min(B, 4) for a batch and
 *            16 for one sequence.  With B > 1 (or fp32 inputs, or a causal
 *            Nq > Nk) chunk c holds sequences [B c / n, B (c + 1) / n),
 *            n <= B.  With one bf16 sequence chunk c holds the query rows
 *            [256 floor(U c / n), 256 floor(U (c + 1) / n)) (U = ceil(Nq /
 *            256), n <= U; the last chunk ends at Nq) together with the keys
 *            those rows may see that no earlier chunk sent: all Nk keys go
 *            with the first chunk without a mask, keys up to the chunk's last
 *            row + (Nk - Nq) with the causal mask.
 *   stream   the compute stream; h2d_stream and d2h_stream carry the two
 *            copy directions (NULL: the compute stream, i.e. no overlap).
 * Chunk c is copied host -> device on h2d_stream, computed once it has
 * arrived, and copied back on d2h_stream once computed and once every chunk
 * has been copied in (the two directions share the host link), so chunk
 * c + 1 moves in while chunk c computes.  Even chunks compute on `stream`, odd chunks on
 * a second compute stream of the library's, so that one chunk's forward can
 * start on the SMs the previous one's last wave leaves idle.  The other
 * streams first wait for the work already queued on `stream`, and `stream`
 * finally waits for the last read back: once `stream` has completed, o_h and
 * lse_h hold the results, equal bit for bit to one attn_fwd call over the
 * whole batch.  Errors as attn_fwd, checked before anything is queued (a
 * CUDA failure later returns ATTN_ERR_CUDA with part of the work queued).
 * The library keeps a few CUDA events and one non-blocking stream per host
 * thread and device for this call (devices 0..63; a higher device number
 * returns ATTN_ERR_UNSUPPORTED).
 */
attn_status_t attn_fwd_host(const void* q_h, const void* k_h, const void* v_h,
                            void* o_h, float* lse_h, void* q_d, void* k_d,
                            void* v_d, void* o_d, float* lse_d, int B, int Hq,
                            int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, attn_dtype_t dtype, int chunks,
                            void* stream, void* h2d_stream, void* d2h_stream);

/*
 * attn_decode_num_splits -- the number of key segments attn_decode_splitkv
 * uses when called with num_splits = 0.  It follows the CTA-by-wave model of
 * [L11] 6.3-6.4: too few segments leave SMs idle, too many add waves and
 * merge overhead, so the count is picked from B, the head counts, Nk and the
 * SM count of the current device.  Returns >= 1, or -1 on invalid sizes or if
 * the device cannot be queried.
 */
int attn_decode_num_splits(int B, int Hq, int Hkv, int Nk, int d);

/*
 * attn_decode_workspace_bytes -- bytes of device workspace that
 * attn_decode_splitkv needs for these sizes (num_splits = 0 resolves through
 * attn_decode_num_splits).  Returns 0 on invalid sizes.
 *
 * Workspace layout after a call with S segments (S > 1), R = B*Hq rows,
 * row r = b*Hq + hq, all float32:
 *     o_parts   [S, R, d]  at byte offset 0: segment outputs, each already
 *                          normalised within its segment ([L11] 6.2 step 2);
 *     lse_parts [S, R]     at byte offset round_up(S*R*d*4, 256).
 * An empty segment holds o = 0, lse = -inf.  With S == 1 the workspace is
 * not touched and may be NULL.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nk, int d,
                                   int num_splits);

/*
 * attn_decode_splitkv -- flash-decoding ([L11] 6.2): one query per sequence.
 *
 *   q        [B, 1, Hq, d]      query of the current step.
 *   k_cache, v_cache  [B, Nk, Hkv, d]  dense KV cache, Nk >= 0 valid rows
 *            (Nk = 0: o = 0 and lse = -inf, nothing is read).
 *   o        [B, 1, Hq, d] output (dtype elements).
 *   lse      [B, Hq] float32 output.
 *   num_splits  0 = automatic (attn_decode_num_splits), else 1..Nk.
 *            Segment s covers keys [s*L, min((s+1)*L, Nk)), L = ceil(Nk/S).
 *   workspace, workspace_bytes  scratch of at least
 *            attn_decode_workspace_bytes(...) bytes, 16-byte aligned; its
 *            contents on return are the partials documented above.
 *   dtype    ATTN_BF16 only (ATTN_F32 returns ATTN_ERR_UNSUPPORTED).
 * Head dimension d is 64 or 128; any G = Hq/Hkv is accepted (query heads of
 * one group are packed into the rows of one tile, [L11] 6.2 GQA paragraph).
 *
 * Step 1-2: the split kernel, one CTA per (segment, group of up to 8 query
 * heads of one KV head, sequence), streams its K/V segment once and writes
 * (o_s, lse_s).  Step 3: attn_merge_lse on the same stream.  With S == 1 the
 * split kernel writes O and LSE directly and no merge runs.
 */
attn_status_t attn_decode_splitkv(const void* q, const void* k_cache,
                                  const void* v_cache, void* o, float* lse,
                                  int B, int Hq, int Hkv, int Nk, int d,
                                  float scale, int num_splits,
                                  void* workspace, size_t workspace_bytes,
                                  attn_dtype_t dtype, void* stream);

/*
 * attn_decode_splitkv_static -- attn_decode_splitkv for callers that cannot
 * allocate device memory.  The pages have no counterpart; this is a library
 * convenience.
 *
 * Some callers cannot provide the decode workspace: code whose device memory
 * is owned by a host framework's allocator (raw cudaMalloc not allowed), code
 * whose memory budget is planned ahead of time, and latency-critical paths
 * that must not call cudaMalloc/cudaFree (those calls can block or
 * synchronise the device).  This entry point takes the same arguments as
 * attn_decode_splitkv minus the workspace and computes the same result with
 * the same kernels, using a scratch area built into the library: a
 * file-scope device array of ATTN_DECODE_STATIC_SCRATCH_BYTES that every GPU
 * on which the library is loaded keeps until the process exits.
 *
 *   - It allocates and frees nothing.
 *   - Its first call on a device looks up the scratch area's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with
 *     the ID of the device's current context; make that first call before
 *     any stream capture.  After a device reset (a new context, in which the
 *     array may sit elsewhere) the next call looks the address up again, so
 *     that call too belongs before any capture.
 *   - Sizes whose partials need more than ATTN_DECODE_STATIC_SCRATCH_BYTES
 *     (see attn_decode_workspace_bytes) return ATTN_ERR_UNSUPPORTED and
 *     launch nothing; use attn_decode_splitkv with a larger workspace instead.
 *   - All calls share the one scratch area, which keeps the last call's
 *     partials (nothing in it needs to start at zero: every partial is written
 *     before it is read).  Calls whose kernels overlap on the GPU (different
 *     streams, or concurrent host threads) race on it; calls ordered on one
 *     stream do not.
 * Other arguments, results and errors: as attn_decode_splitkv.
 */
#define ATTN_DECODE_STATIC_SCRATCH_BYTES (8u << 20)
attn_status_t attn_decode_splitkv_static(const void* q, const void* k_cache,
                                         const void* v_cache, void* o, float* lse,
                                         int B, int Hq, int Hkv, int Nk, int d,
                                         float scale, int num_splits,
                                         attn_dtype_t dtype, void* stream);

/*
 * attn_decode_paged -- flash-decoding over a paged KV cache.  [L11] 9 names
 * paged KV caches as what decode kernels built on the flash-decoding split
 * of [L11] 6.2 read; the pages fix no layout, and this one is the plainest:
 *
 *   q          [B, 1, Hq, d]  query of the current step.
 *   k_pages, v_pages  [num_pages, page_size, Hkv, d]  page pools (bf16).
 *   block_table [B, max_pages_per_seq] int32, device memory: the keys of
 *              sequence b are positions 0 .. seq_lens[b]-1 of its pages
 *              block_table[b, 0], block_table[b, 1], ... in that order.
 *              Entries past a sequence's last page are never read; an entry
 *              outside [0, num_pages) reads zeros.
 *   seq_lens   [B] int32, device memory; values are clamped to
 *              [0, max_seq_len].  A sequence of length 0 gets o = 0,
 *              lse = -inf.
 *   o          [B, 1, Hq, d] output (bf16).   lse [B, Hq] float32 output.
 *   page_size  16, 32, or a multiple of 64.
 *   max_seq_len  upper bound of seq_lens (host-known; it sets the segment
 *              length and the workspace); max_seq_len <=
 *              max_pages_per_seq * page_size.
 *   num_splits 0 = automatic (attn_decode_paged_num_splits), else
 *              1..max_seq_len.  Segment s covers positions [s*L, (s+1)*L)
 *              with L = ceil(max_seq_len / S) rounded up to a multiple of
 *              64; the pages one segment touches must fit a 4096-entry
 *              table (else ATTN_ERR_UNSUPPORTED).
 *   workspace  as attn_decode_splitkv, sized by
 *              attn_decode_workspace_bytes(B, Hq, Hkv, max_seq_len, d, S).
 * Slots of a page past a sequence's length may hold anything (NaN
 * included); they do not affect the result.  The caller owns all buffers;
 * nothing is allocated.  Errors: as attn_decode_splitkv, plus
 * ATTN_ERR_UNSUPPORTED for other page sizes.
 */
attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seq_lens, void* o,
                                float* lse, int B, int Hq, int Hkv, int d, int num_pages,
                                int page_size, int max_pages_per_seq, int max_seq_len,
                                float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, attn_dtype_t dtype, void* stream);

/*
 * attn_decode_paged_num_splits -- the segment count attn_decode_paged uses
 * with num_splits = 0.  With pages of 16 keys and Hkv = 2, 4 or 8 (at most 8
 * query heads per KV head) one CTA takes every KV head of a segment, and the count
 * aims at 27/32 of the SMs in CTAs (segments x sequences: 128 on GB300), at
 * most one segment per 64 keys of max_seq_len.  Otherwise it is the
 * CTA-by-wave time model of attn_decode_num_splits with per-CTA rates that
 * depend on the page size (one wave of CTAs for pages under 64 keys),
 * raised until one segment's pages fit the block-table staging area.
 * Returns -1 on invalid sizes.
 */
int attn_decode_paged_num_splits(int B, int Hq, int Hkv, int d, int page_size,
                                 int max_seq_len);

/*
 * attn_quantize_fp8 -- block quantisation to e4m3 ([L11] 4.5, FP8 item):
 *   x      [B, N, H, d] bf16 input (d even).
 *   codes  [B, N, H, d] uint8 output: e4m3 codes.
 *   scales [B, H, ceil(N/128)] float32 output.
 * Per (batch, head, block of 128 rows): amax = max |x|, scale = amax / 448
 * and inv = 448 / amax in float32 (1 and 1 for an all-zero block); each code
 * is e4m3(x * inv) rounded to nearest even and saturated to +-448, so that
 * x ~= code_value * scale.  All steps are IEEE-defined: the result is
 * reproducible bit for bit.
 */
attn_status_t attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int N, int H,
                                int d, void* stream);

/*
 * attn_quantize_fp8_rotated -- attn_quantize_fp8 after a random orthogonal
 * transform of every row ("incoherent processing", [L11] 4.5, FP8 item, and
 * the FP8 path of the FA3 section of the course index: multiplying by a
 * random orthogonal matrix spreads outlier features over all d columns
 * before quantisation).  The transform is R = diag(signs) H / sqrt(d), with H
 * the d x d Sylvester Hadamard matrix (H H^T = d I), so R R^T = I and
 * (q R)(k R)^T = q k^T: Q and K rotated with the same signs give the same
 * scores, and attn_fwd_fp8 takes the codes and scales unchanged.
 *   x      [B, N, H, d] bf16 input; d is 64 or 128.
 *   signs  [d] float32 on the device, 16-byte aligned, each +1 or -1 (the
 *          random draw; the caller supplies it and uses the same signs for
 *          Q and K).
 *   codes  [B, N, H, d] uint8 output;  scales [B, H, ceil(N/128)] float32.
 * Arithmetic, all fp32 and reproducible bit for bit: y = signs * x, then
 * the fast Walsh-Hadamard butterflies (a, b) -> (a + b, a - b) on index
 * pairs (i, i + h) for h = 1, 2, 4, ..., d/2 in that order (y becomes y H);
 * then the block quantisation of attn_quantize_fp8 on y; each block's scale
 * is finally multiplied by c = float(1 / sqrt(d)) (rounded from double), so
 * that code_value * scale ~= (x R).
 */
attn_status_t attn_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                                        int B, int N, int H, int d, void* stream);

/*
 * attn_fwd_fp8 -- attn_fwd with Q and K block-quantised to e4m3 (as produced
 * by attn_quantize_fp8): S = scale * (q_code * q_scale) (k_code * k_scale)^T
 * is formed on the tensor cores from the e4m3 codes (fp32 accumulation) and
 * the block scales; softmax, P and P V are as in attn_fwd with bf16 V.
 *   q8 [B, Nq, Hq, d], k8 [B, Nk, Hkv, d] uint8 e4m3 codes;
 *   q_scales [B, Hq, ceil(Nq/128)], k_scales [B, Hkv, ceil(Nk/128)] float32;
 *   v [B, Nk, Hkv, d] bf16;  o [B, Nq, Hq, d] bf16;  lse [B, Hq, Nq] float32.
 * d = 128 only.  Relative to the exact attention of the unquantised inputs,
 * the error of row i is bounded by the largest change delta_i that
 * quantisation makes to one of its scaled scores: |dLSE_i| <= delta_i and
 * |dO_i| <= (exp(2 delta_i) - 1) max_j |v_j - O_i| (plus the bf16 error of
 * attn_fwd).  P V stays in bf16.
 */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v, const float* q_scales,
                           const float* k_scales, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                           int Nk, int d, int causal, float scale, void* stream);

/*
 * attn_quantize_fp8_v -- e4m3 quantisation of V for attn_fwd_fp8_pv ([L11]
 * 4.5, FP8 item: FA3's FP8 path quantises both products' operands).  One
 * block per (batch, head): the whole sequence shares one scale, because a
 * scale that changed along the keys would change along the P V product's
 * contraction.  The codes are written transposed, keys innermost, so that
 * V^T is read as a K-major operand like K.
 *   v      [B, N, H, d] bf16 input; d is 64 or 128.
 *   vt8    [B, H, d, ld] uint8 output, ld = round_up(N, 16) (each row of
 *          keys starts on a 16-byte boundary): vt8[b, h, c, n] is the code of
 *          v[b, n, h, c]; the ld - N padding keys hold 0.
 *   scales [B, H] float32 output.
 * amax = max |v| over the head's N x d values; scale = amax / 448 and
 * inv = 448 / amax in float32 (1 and 1 for an all-zero head); each code is
 * e4m3(v * inv), rounded to nearest even and saturated: attn_quantize_fp8's
 * arithmetic with blocks of N rows, reproducible bit for bit.  `scales` is
 * also the working buffer of the amax pass (cleared with cudaMemsetAsync on
 * `stream` first).  Errors: ATTN_ERR_INVALID for negative sizes, NULL or
 * misaligned pointers (v, vt8: 16 bytes; scales: 4); ATTN_ERR_UNSUPPORTED for
 * other d or B, H above 65535.
 */
attn_status_t attn_quantize_fp8_v(const void* v, void* vt8, float* scales, int B, int N, int H, int d,
                                  void* stream);

/*
 * attn_fwd_fp8_pv -- attn_fwd_fp8 with P V in e4m3 as well: V quantised by
 * attn_quantize_fp8_v, P formed per key tile as 256 P (the factor 2^8
 * folded into the exponent, so P keeps e4m3's three mantissa bits down to
 * P = 2^-14), rounded to e4m3 (nearest even) and multiplied with the V codes
 * on the tensor cores (fp32 accumulation).  The row sum l is taken over the
 * unrounded fp32 P, so LSE is as in attn_fwd_fp8; O = acc * v_scale / l.
 *   q8, k8, q_scales, k_scales, o, lse: as attn_fwd_fp8;
 *   vt8 [B, Hkv, d, round_up(Nk, 16)] uint8, v_scales [B, Hkv] float32:
 *          attn_quantize_fp8_v's output for V [B, Nk, Hkv, d].
 * d = 128 only.  Against the attention of the dequantised inputs (q8, k8 and
 * vt8 times their scales) the error of row i, column c is bounded by the
 * rounding of P: |dO_ic| <= 2^-4 sum_j w_ij |v_jc| + 2^-18 sum_j |v_jc| (w
 * the softmax weights; 2^-4 is half an e4m3 step relative, 2^-18 the largest
 * error of a P below e4m3's normal range) plus attn_fwd's bf16 error.
 * Errors: as attn_fwd_fp8, and ATTN_ERR_INVALID for a NULL or misaligned
 * vt8 (16 bytes) or v_scales (4 bytes).
 */
attn_status_t attn_fwd_fp8_pv(const void* q8, const void* k8, const void* vt8, const float* q_scales,
                              const float* k_scales, const float* v_scales, void* o, float* lse, int B,
                              int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                              void* stream);

/*
 * attn_bwd -- backward pass of attn_fwd ([L11] 5.1): given dO, the gradients
 *     dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i * O_i),
 *     dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
 * with P recomputed from the forward's LSE, P_ij = exp(S_ij - LSE_i), and a
 * KV head's dK, dV summed over the query heads that share it.
 *
 *   q, o, dout  [B, Nq, Hq, d] bf16 (o: the forward's output);
 *   k, v        [B, Nk, Hkv, d] bf16;
 *   lse         [B, Hq, Nq] float32 (the forward's LSE);
 *   dq          [B, Nq, Hq, d] bf16 output;  dk, dv [B, Nk, Hkv, d] bf16 output.
 *   causal, scale: as in the forward call that produced o and lse.
 *   workspace   at least attn_bwd_workspace_bytes(B, Hq, Nq) bytes, 16-byte
 *               aligned (holds D); d is 64 or 128; dtype ATTN_BF16 only.
 * Every gradient is written exactly once (no atomics, no zero-fill needed);
 * rows and keys that no allowed (row, key) pair touches get 0.  Three kernels
 * run on `stream`: D, then dK/dV (key tile outer), then dQ (query tile outer).
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Nq);
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                       float scale, void* workspace, size_t workspace_bytes,
                       attn_dtype_t dtype, void* stream);

/*
 * attn_merge_lse -- exact merge of partial attention results in log-sum-exp
 * form ([L11] 6.2 step 3; the associative merge of [L11] 3.2):
 *     lse[r] = log sum_p exp(lse_parts[p, r])
 *     o[r,:] = sum_p exp(lse_parts[p, r] - lse[r]) * o_parts[p, r, :]
 * computed after subtracting max_p lse_parts[p, r].  Parts with lse = -inf
 * are empty and ignored; a row whose parts are all empty gets o = 0,
 * lse = -inf.
 *
 *   o_parts   [num_parts, rows, d] float32, each normalised within its part.
 *   lse_parts [num_parts, rows] float32.
 *   o         [rows, d] output in out_dtype (ATTN_BF16 or ATTN_F32).
 *   lse       [rows] float32 output (may be NULL if not wanted).
 *   num_parts >= 1, rows >= 0, d a multiple of 4 in [4, 512].
 */
attn_status_t attn_merge_lse(const float* o_parts, const float* lse_parts,
                             int num_parts, long long rows, int d, void* o,
                             float* lse, attn_dtype_t out_dtype, void* stream);

/* Static English text for a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * attn_check_device_status -- reads and clears the device status words of
 * every kernel family in the library (synchronises the device first).
 * Returns ATTN_ERR_BOUNDS if an in-kernel index check refused an access since
 * the last call (only the bounds-checked debug build, libattn_bounds.so, built
 * with ATTN_BOUNDS_CHECK, makes these checks: on every global load and store
 * that is not a TMA copy, in every kernel family; a refused access is
 * skipped, nothing traps), else
 * ATTN_ERR_TIMEOUT if any bounded wait ran out, ATTN_ERR_CUDA if the device
 * could not be read, else ATTN_OK.
 */
attn_status_t attn_check_device_status(void);

/*
 * attn_read_tile_counter -- number of (query tile, key tile) pairs the bf16
 * forward kernel has computed since the last reset (synchronises the device;
 * reset != 0 clears it after reading).  Tiles are 128 x 128.  A causal call
 * with Nq = Nk = N computes T(T+1)/2 of the T^2 pairs, T = N/128, i.e. the
 * fraction 1/2 + 1/(2T) of [L11] 5.3 (0.516 at N = 4096).
 */
attn_status_t attn_read_tile_counter(unsigned long long* count, int reset);

/* Library version string, e.g. "exact_attention_gb300 0.1 sm_103a". */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_GB300_ATTN_H */
