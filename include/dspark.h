/*
 * dspark.h -- C ABI of libdspark: the data-parallel hot path of DSpark-style
 * speculative decoding on one GB300 (sm_103a) GPU.
 *
 * One decoding round for a batch of B requests with block length G over a
 * vocabulary of V tokens is three calls:
 *
 *   dspark_draft_sample     draft G tokens per request with the
 *                           semi-autoregressive Markov head;
 *   dspark_schedule_prefix  calibrate per-position confidences and choose how
 *                           many draft tokens of each request to verify
 *                           (dspark_schedule_policy: other policies);
 *   dspark_verify           lossless rejection-sampling verification against
 *                           the target logits, with residual resampling or a
 *                           bonus token.
 *
 * Conventions shared by every entry point
 *  - Every array argument is a DEVICE pointer owned by the caller, row-major
 *    and contiguous (the last index is contiguous).  The library never
 *    allocates or frees memory.  Pointers to logits, E_in and W_out must be
 *    16-byte aligned; V must be a multiple of 8.
 *  - "dtype" arrays hold bf16 (DSPARK_BF16) or fp32 (DSPARK_F32) values; all
 *    arithmetic is fp32 on the device (the scheduler accumulates tau and
 *    Theta in float-float, an unevaluated sum of two floats of about 44
 *    significant bits, and returns Theta as a double).
 *  - Logits must be finite.  Mask a token with a large negative finite value
 *    (-3e4, say): its probability is then 0 in fp32 and it is never drawn.
 *    An IEEE -inf base logit is not supported on the bf16 path, whose base
 *    add on the tensor cores multiplies every base logit of a tile by 0 or 1.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls only enqueue work: they do not synchronise.
 *  - `workspace` is caller-owned device scratch memory of at least
 *    dspark_workspace_bytes(...) bytes, 256-byte aligned.  One workspace must
 *    not be shared by two calls that may run concurrently.
 *  - Host-side argument errors return DSPARK_ERR_INVALID_ARG before any launch
 *    and leave the outputs untouched.  CUDA launch errors return
 *    DSPARK_ERR_CUDA.  The message of the last failure on the calling thread
 *    is available from dspark_last_error().
 *  - Device-resident inputs (token ids, temperatures, verify lengths) are
 *    checked by the kernels: a request with an out-of-range value gets -1 in
 *    its output tokens and sets a bit in the workspace's flag word, which
 *    dspark_read_device_flags() returns.  Kernels never read out of bounds.
 *  - Randomness: Philox4x32-10 (Salmon et al., SC'11) with key =
 *    (seed mod 2^32, seed >> 32) and counter = (v >> 2, j, request_id,
 *    stream), output word v & 3; u = ((w >> 9) + 0.5) * 2^-23.  Streams:
 *    0 draft Gumbel noise, 1 acceptance uniform, 2 residual Gumbel noise,
 *    3 bonus Gumbel noise; each token v of a Gumbel-max draw takes its own
 *    word.  A call is reproducible from (seed, request ids).
 *  - Precision: the arithmetic is fp32 on fp32 or bf16 data.  The kernels
 *    screen tokens in fp32 and form the Gumbel keys of the few tokens that
 *    can still win in float-float arithmetic (about 44 significant bits), and
 *    the merges of row partials (log-sum-exp, log q, log p) and the acceptance
 *    test work in float-float as well, so a draw or an
 *    acceptance differs from an exact evaluation only on a tie far below fp32
 *    rounding (about 1e-7 of decisions or fewer, in the test suite none in
 *    2.5 million).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dspark_status {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1,   /* bad size, pointer, alignment or workspace */
    DSPARK_ERR_UNSUPPORTED = 2,   /* valid request the library does not handle */
    DSPARK_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    DSPARK_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up */
} dspark_status;

typedef enum dspark_dtype {
    DSPARK_BF16 = 0,
    DSPARK_F32 = 1
} dspark_dtype;

/* which workspace: argument of dspark_workspace_bytes */
enum {
    DSPARK_WS_DRAFT = 0,
    DSPARK_WS_SCHEDULE = 1,
    DSPARK_WS_VERIFY = 2,
    DSPARK_WS_DRAFT_RNN = 3
};

/* bits of the device flag word */
enum {
    DSPARK_FLAG_BAD_TOKEN = 1u,        /* an anchor or draft token outside [0, V) */
    DSPARK_FLAG_BAD_TEMPERATURE = 2u,  /* a temperature that is negative, NaN or inf */
    DSPARK_FLAG_BAD_VERIFY_LEN = 4u,   /* a verify length outside [0, G] */
    DSPARK_FLAG_BAD_POS_TEMP = 8u,     /* a calibration temperature <= 0 or NaN */
    DSPARK_FLAG_TIMEOUT = 16u,         /* a bounded device-side wait gave up */
    DSPARK_FLAG_BAD_TARGET_ROW = 32u   /* a packed target row outside the array */
};

/* Library version, major * 10000 + minor * 100 + patch. */
DSPARK_API int dspark_version(void);

/* Message of the last failed call on the calling thread ("" if none). */
DSPARK_API const char *dspark_last_error(void);

/* Bytes of workspace needed by one call of the given kind (DSPARK_WS_*), for
 * B requests, block length G, vocabulary V, Markov rank r.  Returns 0 for
 * invalid sizes. */
DSPARK_API size_t dspark_workspace_bytes(int which, int B, int G, int V, int r);

/*
 * Draft sampling with the semi-autoregressive Markov head.
 *
 * Defined by "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
 * "Un po' di autoregressione basta", equation for p_k: the draft distribution
 * of position j is softmax(U_j + B_j) where the bias B_j = E_in[x_{j-1}] W_out
 * is the rank-r Markov head (B = W1 W2, with W1 = E_in and W2 = W_out^T)
 * driven by the previous token (the
 * anchor x_0 for the first position), and tokens are drawn left to right so
 * each keeps an explicit softmax probability.
 *
 * For each request b and j = 0 .. G-1, with prev = anchor[b] (j = 0) or
 * draft_tokens[b][j-1]:
 *   z[v]  = base_logits[b][j][v] + sum_k e_in[prev][k] * w_out[v][k]   (fp32)
 *   T > 0: s = z / T, lse = log sum exp s, x_j drawn from softmax(s) by
 *          per-token Gumbel-max: x_j = argmax_v s[v] - ln(-ln u_v) with
 *          u_v = u(seed, request_id[b], j, v, stream 0), the lowest id on an
 *          exact tie; logq = s[x_j] - lse
 *   T = 0: x_j = argmax_v z[v] (lowest id on ties), lse = max z, logq = 0
 *
 * base_logits [B][G][V] dtype   e_in [V][r] dtype   w_out [V][r] dtype (row v
 * scores token v, the layout of a language-model output head)
 * anchor [B] int32              temperature [B] fp32 (>= 0)
 * request_id [B] uint32 or NULL (then request b uses id b)
 * outputs: draft_tokens [B][G] int32, draft_lse [B][G] fp32,
 *          draft_logq [B][G] fp32, draft_logits [B][G][V] fp32 z or NULL.
 * Limits: 1 <= B, 1 <= G <= 64, 8 <= V <= 2^20 with V % 8 == 0 (the token id
 *         shares a 64-bit key word with the key; larger V returns
 *         DSPARK_ERR_UNSUPPORTED),
 *         16 <= r <= 256 with r % 16 == 0 (bf16) or 4 <= r <= 256 with
 *         r % 4 == 0 (fp32).  bf16 runs the bias on the tcgen05 tensor cores;
 *         fp32 runs it with CUDA-core FMAs (no TF32 rounding).
 */
DSPARK_API dspark_status dspark_draft_sample(
    const void *base_logits, const void *e_in, const void *w_out,
    const int32_t *anchor, const float *temperature, const uint32_t *request_id,
    int B, int G, int V, int r, dspark_dtype dtype, uint64_t seed,
    int32_t *draft_tokens, float *draft_lse, float *draft_logq, float *draft_logits,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Draft sampling with the recurrent (RNN) head.
 *
 * "DSpark, la bozza che sa quando fermarsi" (paithon.it), section "Un po' di
 * autoregressione basta", names a recurrent head beside the Markov head: the
 * bias of position j comes from a state carried along the block instead of
 * from x_{j-1} alone.  The pages give no cell; this one is an Elman cell
 * driven by the previous token's embedding, its state kept in bf16:
 *   h_{-1} = 0,  h_j[n] = bf16(tanh(e_in[prev][n] + sum_k w_h[n][k] h_{j-1}[k]))
 *   z[v] = base_logits[b][j][v] + sum_k h_j[k] * w_out[v][k]          (fp32)
 * with prev = anchor[b] (j = 0) or draft_tokens[b][j-1]; everything after z
 * (temperature, Gumbel-max draw, lse, logq, greedy rows, streams) is exactly
 * as in dspark_draft_sample.
 *
 * Arguments as in dspark_draft_sample, plus w_h [r][r] bf16 (row n holds the
 * weights of state unit n) and h_states: [B][G][r] bf16 output of the states
 * h_j, or NULL.  The state sum is compensated, and tanh is taken in fp32 and
 * redone in fp64 when the result lies near a bf16 rounding boundary, so h_j
 * is the exactly rounded value except within ~1e-13 of such a boundary.
 * dtype must be DSPARK_BF16 (else DSPARK_ERR_UNSUPPORTED).  The workspace is
 * DSPARK_WS_DRAFT_RNN.  Verify such a block with dspark_verify
 * given the draft_logits this call stored (the draft distribution of the
 * rejected position is then read, not recomputed).
 */
DSPARK_API dspark_status dspark_draft_sample_rnn(
    const void *base_logits, const void *e_in, const void *w_h, const void *w_out,
    const int32_t *anchor, const float *temperature, const uint32_t *request_id,
    int B, int G, int V, int r, dspark_dtype dtype, uint64_t seed,
    int32_t *draft_tokens, float *draft_lse, float *draft_logq, float *draft_logits,
    void *h_states, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Confidence calibration and the load-aware prefix scheduler.
 *
 * Defined by "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
 * "Verificare meglio, non di piu'": c = per-position temperature-scaled
 * confidence, a_{b,j} = prod_{i<=j} c_{b,i}, Theta = tau * SPS(B); candidates
 * of all requests are admitted in decreasing a while Theta grows, stopping at
 * the first one that does not raise it.
 *
 *   c[b][j]   = 1 / (1 + exp(-conf_logits[b][j] / pos_temp[j]))
 *   a[b][j]   = prod_{i <= j} c[b][i]
 *   start:    L_b = L_min, tau = sum_b (1 + sum_{j < L_b} a[b][j]),
 *             n = sum_b (L_b + 1) batch tokens
 *   candidates (b, j), L_min <= j < L_max, in order (a desc, j asc, b asc):
 *             admit (L_b = j + 1) while (tau + a) * sps[n + 1] > tau * sps[n]
 *
 * conf_logits [B][G] fp32, pos_temp [G] fp32 (> 0), sps [sps_len] fp32 with
 * sps[n] = engine steps per second at n batch tokens, sps_len >=
 * B * (L_max + 1) + 1.  Outputs: conf, cum_conf [B][G] fp32, verify_len [B]
 * int32, theta_out [1] fp64 (final Theta) or NULL.
 * Limits: 0 <= L_min <= L_max <= G <= 64, B * G <= 16384.
 * c and a are computed in fp32; tau and Theta are accumulated in float-float
 * (about 44 significant bits).
 */
DSPARK_API dspark_status dspark_schedule_prefix(
    const float *conf_logits, const float *pos_temp, const float *sps, int sps_len,
    int B, int G, int L_min, int L_max,
    float *conf, float *cum_conf, int32_t *verify_len, double *theta_out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Verify lengths under another policy; the early stop above is policy 0.
 *
 * Defined by "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
 * "Che cosa resta da verificare" (the deployed scheduler takes confidences
 * from two rounds earlier and drops the early stop) and section "Verificare
 * meglio, non di piu'" (a fixed confidence threshold as the comparator):
 *
 *   DSPARK_SCHED_EARLY_STOP (0)  as dspark_schedule_prefix;
 *   DSPARK_SCHED_BEST_PREFIX (1) the same candidate order, admitting the first
 *        n whose Theta(n) = tau_n * sps[n_0 + n] is largest over n = 0 .. all
 *        candidates (no early stop; for a fixed n the top-a set is the best
 *        one, so this is the optimum over every vector of lengths);
 *   DSPARK_SCHED_THRESHOLD_CUM (2)  L_b grows from L_min while
 *        a[b][L_b] > threshold (L_b < L_max);
 *   DSPARK_SCHED_THRESHOLD_CONF (3) the same on c[b][L_b] (a leading run).
 *
 * For the lagged production mode pass the confidence logits of round t - 2
 * with policy 1 (the library keeps no history).  Arguments, outputs and
 * limits as dspark_schedule_prefix; theta_out is Theta of the chosen lengths
 * for every policy.  `threshold` is used by policies 2 and 3 only and must be
 * finite.  An unknown policy returns DSPARK_ERR_INVALID_ARG.
 */
typedef enum {
    DSPARK_SCHED_EARLY_STOP = 0,
    DSPARK_SCHED_BEST_PREFIX = 1,
    DSPARK_SCHED_THRESHOLD_CUM = 2,
    DSPARK_SCHED_THRESHOLD_CONF = 3
} dspark_sched_policy;

DSPARK_API dspark_status dspark_schedule_policy(
    const float *conf_logits, const float *pos_temp, const float *sps, int sps_len,
    int B, int G, int L_min, int L_max, int policy, float threshold,
    float *conf, float *cum_conf, int32_t *verify_len, double *theta_out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Lossless rejection-sampling verification of one block per request.
 *
 * Defined by "Les mathematiques derriere l'acceleration : comment le decodage
 * speculatif masque la latence sans modifier les sorties" (seventnews.com),
 * section "La garantie de l'echantillonnage par rejet" (accept x with
 * probability min(1, p(x)/q(x)), stop at the first rejection and resample that
 * token from the residual distribution), and "DeepSeek发布DSpark"
 * (learnblockchain.cn), section "DSpark 是什么？" (a bonus token is appended
 * when the whole block is accepted).
 *
 * For request b with L = verify_len[b] (G if verify_len is NULL) and T > 0:
 *   row j < L of target_logits is the target's logits for draft position j;
 *   p_j = softmax(target[b][j] / T), q_j = the draft distribution (from the
 *   draft's logq and lse);
 *   accept x_j while u(seed, id, j, 0, stream 1) < min(1, p_j(x_j)/q_j(x_j));
 *   at the first rejection d: y is drawn from normalise(max(0, p_d - q_d)) by
 *   per-token Gumbel-max on stream 2, y = argmax over {v: p_v > q_v} of
 *   ln(p_v - q_v) - ln(-ln u(seed, id, d, v, stream 2)) (from p_d itself if no
 *   entry has p > q) (the draft logits of row d are recomputed from
 *   base_logits, e_in and w_out, or read from draft_logits when it is not
 *   NULL);
 *   if all L are accepted: y is drawn from softmax(target[b][L] / T) by
 *   per-token Gumbel-max on stream 3.
 * T = 0: accept while x_j == argmax target[b][j]; y = that argmax at the first
 * mismatch, else argmax target[b][L].
 *
 * target_logits [B][G+1][V] dtype; base_logits, e_in, w_out as for
 * dspark_draft_sample (may be NULL when draft_logits is given);
 * draft_logits [B][G][V] fp32 or NULL; anchor [B]; draft_tokens, draft_lse,
 * draft_logq [B][G] from dspark_draft_sample; verify_len [B] or NULL;
 * temperature [B]; request_id [B] or NULL.
 * Outputs: accept_len [B] int32; out_tokens [B][G+1] int32 = accepted draft
 * tokens then the resampled or bonus token, padded with -1; num_out [B] =
 * accept_len + 1; target_lse [B][G+1] fp32 or NULL (lse of rows j < L at
 * T > 0, max of the row at T = 0; NaN where not computed); logp_sel [B][G]
 * fp32 or NULL (log p_j(x_j) of the tested rows, NaN elsewhere).  There is
 * no q output: log q_j(x_j) is the caller's draft_logq input, which the
 * acceptance test uses as given.
 */
DSPARK_API dspark_status dspark_verify(
    const void *target_logits, const void *base_logits, const void *e_in, const void *w_out,
    const float *draft_logits,
    const int32_t *anchor, const int32_t *draft_tokens, const float *draft_lse,
    const float *draft_logq, const int32_t *verify_len,
    const float *temperature, const uint32_t *request_id,
    int B, int G, int V, int r, dspark_dtype dtype, uint64_t seed,
    int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
    float *target_lse, float *logp_sel,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * dspark_verify on a packed target: only the rows verification reads.
 *
 * The scheduler of "DSpark, la bozza che sa quando fermarsi" (paithon.it),
 * section "Verificare meglio, non di piu'", sizes the target's batch by the
 * verify lengths: request b needs target rows 0 .. L_b (L_b = verify_len[b]),
 * sum_b (L_b + 1) rows in all, not B (G + 1).  Here request b's row j is row
 * target_row0[b] + j of target_logits [n_target_rows][V]; rows 0 .. L_b must
 * lie inside the array (else the request's outputs are marked as for a bad
 * token and DSPARK_FLAG_BAD_TARGET_ROW is raised).  target_row0 [B] int64 is a
 * device array.  Everything else, the results included, is dspark_verify's.
 */
DSPARK_API dspark_status dspark_verify_packed(
    const void *target_logits, const int64_t *target_row0, int64_t n_target_rows,
    const void *base_logits, const void *e_in, const void *w_out,
    const float *draft_logits, const int32_t *anchor, const int32_t *draft_tokens,
    const float *draft_lse, const float *draft_logq, const int32_t *verify_len,
    const float *temperature, const uint32_t *request_id, int B, int G, int V, int r,
    dspark_dtype dtype, uint64_t seed, int32_t *accept_len, int32_t *out_tokens,
    int32_t *num_out, float *target_lse, float *logp_sel, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * Gather the target rows verification reads into the packed layout.
 *
 * For each request b with L_b = verify_len[b] (G if verify_len is NULL),
 * copies rows 0 .. L_b of target_logits [B][G+1][V] (dtype) to
 * target_packed, requests in order: target_row0[b] = sum_{b' < b} (L_b' + 1),
 * and n_rows[0] = sum_b (L_b + 1) when n_rows is not NULL.  A request with an
 * invalid length contributes no row (dspark_verify_packed flags it).
 * target_logits may be device memory or pinned host memory mapped into the
 * device's address space; then only these rows cross the host link.
 * target_packed needs room for B (G+1) rows; verify_len, target_row0
 * ([B] int64) and n_rows ([1] int64) are device arrays.  Nothing is read back
 * to the host: pass n_target_rows = B (G+1) (the buffer's size) to
 * dspark_verify_packed.
 */
DSPARK_API dspark_status dspark_pack_target(
    const void *target_logits, const int32_t *verify_len, int B, int G, int V, dspark_dtype dtype,
    void *target_packed, int64_t *target_row0, int64_t *n_rows, void *stream);

/*
 * dspark_verify without a workspace argument, for callers that cannot
 * allocate device memory.  The paper has no counterpart: this is a deployment
 * convenience of this library.
 *
 * Who needs it: runtimes that plan all device memory ahead of time and hand
 * it out only to tensors, plugins that run inside another framework where
 * cudaMalloc is not allowed, and foreign-function callers without an
 * allocator.  Arguments and results are those of dspark_verify; the caller
 * still owns every input and output buffer.
 *
 * Scratch: a fixed DSPARK_NOALLOC_SCRATCH_BYTES array in the library's device
 * image, held by every GPU that loads the library until the process exits.
 * Its device address is looked up on the first call on each device (with that
 * device current) and kept for the life of the process, so a cudaDeviceReset
 * invalidates it: make that first call before any stream capture begins, and
 * do not use this entry point after a device reset.
 * Every call shares the array and finds the previous call's contents in it
 * (the flag word is cleared on each call); calls whose GPU work overlaps
 * (other streams, unordered host threads) race on it and must be avoided.
 * Sizes whose verify scratch exceeds the array return DSPARK_ERR_UNSUPPORTED
 * with a message in dspark_last_error().  No call allocates or frees memory.
 * The device flag word of the array (invalid inputs, a timeout, a packed row
 * outside its array) is read with dspark_read_noalloc_flags().
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

DSPARK_API dspark_status dspark_verify_noalloc(
    const void *target_logits, const void *base_logits, const void *e_in, const void *w_out,
    const float *draft_logits,
    const int32_t *anchor, const int32_t *draft_tokens, const float *draft_lse,
    const float *draft_logq, const int32_t *verify_len,
    const float *temperature, const uint32_t *request_id,
    int B, int G, int V, int r, dspark_dtype dtype, uint64_t seed,
    int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
    float *target_lse, float *logp_sel, void *stream);

/* Copy the device flag word of dspark_verify_noalloc's fixed array to *flags
 * (waits for `stream`; the word of the last call, subject to the same race
 * between overlapping calls).  Returns DSPARK_OK, DSPARK_ERR_INVALID_ARG for a
 * NULL flags pointer, or DSPARK_ERR_CUDA. */
DSPARK_API dspark_status dspark_read_noalloc_flags(void *stream, uint32_t *flags);

/*
 * Self-test of the bounded device-side waits (the library's failure
 * detection): one block waits, with the helpers every kernel uses and a limit
 * of limit_us microseconds (1 .. 10^6), on an mbarrier phase that nothing
 * completes and on a device counter that nothing increments.  *result (host)
 * receives bit 0 if the mbarrier wait gave up and bit 1 if the counter wait
 * did: 3 when both report their timeout.  Synchronises the stream.  The
 * context stays usable afterwards.
 */
DSPARK_API dspark_status dspark_selftest_bounded_wait(unsigned int limit_us, uint32_t *result, void *stream);

/*
 * The device's rate for the draw's random words: a grid of 2048 threads per
 * SM draws Philox4x32-10 blocks with the same code as the draft kernel's
 * per-token words (four consecutive counters per step, the parts fixed by
 * request and position precomputed), iters x 4 blocks per thread, and
 * *blocks_per_second receives the measured rate (CUDA events on `stream`;
 * synchronises it).  This is the ALU roof of the per-token Gumbel-max draw,
 * which needs one block per four tokens.  workspace: device scratch of at
 * least 256 bytes per SM (the words are folded into it so that none is
 * optimised away), 256-byte aligned; 1 <= iters <= 2^20.
 */
DSPARK_API dspark_status dspark_selftest_philox_rate(void *workspace, size_t workspace_bytes, int iters,
                                                     double *blocks_per_second, void *stream);

/* Copy the device flag word of a workspace to *flags (waits for `stream`).
 * Returns DSPARK_OK or DSPARK_ERR_CUDA. */
DSPARK_API dspark_status dspark_read_device_flags(const void *workspace, void *stream, uint32_t *flags);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
