/*
 * attn_test.h -- entry points of libattn.so for tests and measurements
 * only.  A production caller uses include/attn.h; nothing here is needed to
 * compute attention.
 *
 * attn_fwd_test and attn_decode_test run the same kernels as attn_fwd and
 * attn_decode_splitkv with settings the production entry points keep fixed:
 *   - variants of the forward used to check that alternative formulations
 *     give the same answer and to measure what they cost (P staged in
 *     shared memory, part of the exponentials on the FMA pipe, a
 *     conditional-rescale threshold);
 *   - the bound of every device-side wait, and a fault injection that makes
 *     one wait run out on purpose, so that tests can check the error path
 *     that keeps a lost signal from hanging a GPU.
 * attn_decode_model_time / _best expose the decode's segment-count model as
 * host arithmetic, so that it can be checked without a GPU.
 *
 * The injection stops one TMA load from being issued: the producer of
 * block 0 posts no byte count and issues no copy for that ring position.
 * The wait for it then ends when the bound runs out; the kernel sets its
 * abort flag, every role of that block drains to the block's teardown (TMEM
 * freed, no copy or MMA in flight), the status word records the timeout and
 * the launch completes normally.  attn_check_device_status() then returns
 * ATTN_ERR_TIMEOUT and clears the word; the outputs of such a call are
 * unspecified, and later calls are unaffected.
 */
#ifndef EXACT_ATTENTION_GB300_ATTN_TEST_H
#define EXACT_ATTENTION_GB300_ATTN_TEST_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    /* forward only: 1 = P goes through shared memory and the
     * shared-memory form of the P V product (the default keeps P in
     * tensor memory) */
    int p_in_smem;
    /* forward only: 1 = every fourth pair of exponentials is computed by a
     * polynomial on the FMA pipe instead of the MUFU unit (software exp2 of
     * the FA4 section of the course index) */
    int exp2_poly;
    /* forward only: conditional-rescale threshold in log2 units, 0..8 (the
     * production value is 0: the reference max moves whenever it grows) */
    float rescale_threshold;
    /* bound of every device-side wait in SM clock cycles; 0 = the
     * production bound (2^32 cycles, about 2 s) */
    long long wait_limit_cycles;
    /* -1 = none.  Otherwise the TMA producer of block 0 skips this load:
     * forward, the K and V tiles at this position of the block's key ring
     * (0 = the first key tile it loads); decode, this tile of the block's
     * segment (0 = its first 64 keys). */
    int skip_load;
    /* Only the bounds-checked debug build (libattn_bounds.so) reads this:
     * the kernels take O's extent as this many elements less than B*Nq*Hq*d
     * (decode: B*Hq*d, for the split kernel's and the merge's stores), so
     * that the index check refuses the stores of the last rows, skips them
     * and reports ATTN_ERR_BOUNDS (a test of the check itself; the buffer is
     * whole, so nothing is ever written outside it).  0 = the true extent;
     * negative = ATTN_ERR_INVALID.  Production builds ignore it. */
    long long o_extent_slack;
} attn_test_options_t;

/*
 * attn_fwd_test -- attn_fwd (ATTN_BF16 only) with the options above.  Same
 * arguments, layouts and errors as attn_fwd, plus ATTN_ERR_INVALID for a
 * NULL `opt`, a threshold outside [0, 8], a negative wait bound or a
 * negative extent slack.
 */
attn_status_t attn_fwd_test(const void* q, const void* k, const void* v, void* o,
                            float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                            int causal, float scale, const attn_test_options_t* opt,
                            void* stream);

/*
 * attn_decode_test -- attn_decode_splitkv with the wait bound and the load
 * injection of `opt` (the forward-only fields are ignored).  Same
 * arguments and errors as attn_decode_splitkv, plus ATTN_ERR_INVALID for a
 * NULL `opt`, a negative wait bound or a negative extent slack.
 */
attn_status_t attn_decode_test(const void* q, const void* k_cache, const void* v_cache,
                               void* o, float* lse, int B, int Hq, int Hkv, int Nk, int d,
                               float scale, int num_splits, void* workspace,
                               size_t workspace_bytes, const attn_test_options_t* opt,
                               void* stream);

/*
 * attn_decode_model_time / attn_decode_model_best -- the segment-count model
 * behind attn_decode_num_splits (the CTA-by-wave model of [L11] 6.3-6.4) as
 * plain host arithmetic, with the machine described by the arguments instead
 * of the current device; no CUDA call is made.
 *   units      CTAs per segment (sequences x query-head groups)
 *   slots      CTAs resident on the GPU at once (SMs x CTAs per SM)
 *   Nk, d      keys and head dimension (bf16 K and V: 4 d bytes per key)
 *   cta_bytes_per_s, hbm_bytes_per_s  one CTA's and the GPU's stream rate
 *   cta_fixed_s, merge_fixed_s        start-up of a wave; the merge launch
 * Time of S segments: ceil(units S / slots) waves, each streaming a segment
 * of ceil(Nk / S) keys at min(cta rate, hbm / min(units S, slots)) plus the
 * start-up, plus (S > 1) the merge launch and its partial traffic.  _best
 * returns the S in 1..min(Nk, 1024) of least time (ties within 0.5% to fewer
 * segments; single_wave caps S so that all CTAs fit in one wave), or -1 on
 * invalid arguments; _time returns -1 on invalid arguments.
 */
double attn_decode_model_time(int units, int slots, int Nk, int d, int num_splits,
                              double cta_bytes_per_s, double hbm_bytes_per_s,
                              double cta_fixed_s, double merge_fixed_s);
int attn_decode_model_best(int units, int slots, int Nk, int d, double cta_bytes_per_s,
                           double hbm_bytes_per_s, double cta_fixed_s, double merge_fixed_s,
                           int single_wave);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_GB300_ATTN_TEST_H */
