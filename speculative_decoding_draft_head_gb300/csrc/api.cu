// extern "C" entry points of libdspark: argument checks, workspace planning
// and the launch sequence of each step.  Nothing here computes on the host.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"

namespace dspark {
namespace {

thread_local char g_last_error[512] = "";

#define fail set_last_error

dspark_status cuda_fail(cudaError_t e, const char *where) {
    return fail(DSPARK_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dspark_status check_common(int B, int G, int V, int r, dspark_dtype dt) {
    if (B < 1) return fail(DSPARK_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
    if (G < 1 || G > kMaxG) return fail(DSPARK_ERR_INVALID_ARG, "G must be in [1, %d] (got %d)", kMaxG, G);
    if (V < 8 || V % 8 != 0) return fail(DSPARK_ERR_INVALID_ARG, "V must be a positive multiple of 8 (got %d)", V);
    if (V > kMaxV) return fail(DSPARK_ERR_UNSUPPORTED, "V must be at most %d (got %d)", kMaxV, V);
    if (dt != DSPARK_BF16 && dt != DSPARK_F32) return fail(DSPARK_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    if (r < 1 || r > 256) return fail(DSPARK_ERR_INVALID_ARG, "r must be in [1, 256] (got %d)", r);
    if (dt == DSPARK_BF16 && r % 16 != 0) return fail(DSPARK_ERR_INVALID_ARG, "bf16 needs r %% 16 == 0 (got %d)", r);
    if (dt == DSPARK_F32 && r % 4 != 0) return fail(DSPARK_ERR_INVALID_ARG, "fp32 needs r %% 4 == 0 (got %d)", r);
    if ((long)B * G * (long)V > (1L << 40)) return fail(DSPARK_ERR_INVALID_ARG, "B*G*V too large");
    return DSPARK_OK;
}

dspark_status check_ws(void *ws, size_t have, size_t need) {
    if (!ws) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(DSPARK_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (have < need) return fail(DSPARK_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", have, need);
    return DSPARK_OK;
}


}  // namespace

// Host-side checks of dspark_verify's sizes, pointers and alignment (before
// any workspace check), shared with dspark_verify_noalloc.
dspark_status verify_check_args(const void *target_logits, const void *base_logits, const void *e_in,
                                const void *w_out, const float *draft_logits, const int32_t *anchor,
                                const int32_t *draft_tokens, const float *draft_lse, const float *draft_logq,
                                const float *temperature, int B, int G, int V, int r, dspark_dtype dtype,
                                const int32_t *accept_len, const int32_t *out_tokens, const int32_t *num_out) {
    dspark_status st = check_common(B, G, V, r, dtype);
    if (st != DSPARK_OK) return st;
    if (!target_logits || !anchor || !draft_tokens || !draft_lse || !draft_logq || !temperature ||
        !accept_len || !out_tokens || !num_out)
        return fail(DSPARK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!draft_logits && (!base_logits || !e_in || !w_out))
        return fail(DSPARK_ERR_INVALID_ARG, "need draft_logits or (base_logits, e_in, w_out)");
    if (!aligned(target_logits, 16) || (base_logits && !aligned(base_logits, 16)) ||
        (e_in && !aligned(e_in, 16)) || (w_out && !aligned(w_out, 16)) ||
        (draft_logits && !aligned(draft_logits, 16)))
        return fail(DSPARK_ERR_INVALID_ARG, "logits and weights must be 16-byte aligned");
    return DSPARK_OK;
}

namespace {

dspark_status verify_impl(const void *target_logits, const int64_t *target_row0, int64_t n_target_rows,
                          const void *base_logits, const void *e_in,
                            const void *w_out, const float *draft_logits, const int32_t *anchor,
                            const int32_t *draft_tokens, const float *draft_lse, const float *draft_logq,
                            const int32_t *verify_len, const float *temperature,
                            const uint32_t *request_id, int B, int G, int V, int r, dspark_dtype dtype,
                            uint64_t seed, int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
                            float *target_lse, float *logp_sel, void *workspace, size_t workspace_bytes,
                            void *stream) {
    dspark_status st = verify_check_args(target_logits, base_logits, e_in, w_out, draft_logits, anchor, draft_tokens,
                                         draft_lse, draft_logq, temperature, B, G, V, r, dtype, accept_len,
                                         out_tokens, num_out);
    if (st != DSPARK_OK) return st;
    const VerifyPlan plan = plan_verify(B, G, V, r, dtype);
    if ((st = check_ws(workspace, workspace_bytes, plan.ws_bytes)) != DSPARK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // (the first launch clears the flag words)
    VerifyArgs a{target_logits, target_row0, n_target_rows, base_logits, e_in, w_out, draft_logits, anchor, draft_tokens, draft_lse,
                 draft_logq, verify_len, temperature, request_id, B, G, V, r, dtype, seed, accept_len,
                 out_tokens, num_out, target_lse, logp_sel, static_cast<unsigned char *>(workspace)};
    const cudaError_t e = launch_verify(a, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
    return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

namespace dspark {
dspark_status set_last_error(dspark_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}
}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_version(void) { return 100; }

const char *dspark_last_error(void) { return g_last_error; }

size_t dspark_workspace_bytes(int which, int B, int G, int V, int r) {
    if (B < 1 || G < 1 || G > kMaxG || V < 8 || V % 8 != 0 || r < 1 || r > 256) return 0;
    switch (which) {
        case DSPARK_WS_DRAFT: {
            const size_t a = plan_draft(B, G, V, r, DSPARK_BF16).ws_bytes;
            const size_t b = plan_draft(B, G, V, r, DSPARK_F32).ws_bytes;
            return a > b ? a : b;
        }
        case DSPARK_WS_DRAFT_RNN: return plan_draft_rnn(B, G, V, r).ws_bytes;
        case DSPARK_WS_SCHEDULE: return kFlagBytes;
        case DSPARK_WS_VERIFY: {
            const size_t a = plan_verify(B, G, V, r, DSPARK_BF16).ws_bytes;
            const size_t b = plan_verify(B, G, V, r, DSPARK_F32).ws_bytes;
            return a > b ? a : b;
        }
        default: return 0;
    }
}

dspark_status dspark_draft_sample(const void *base_logits, const void *e_in, const void *w_out,
                                  const int32_t *anchor, const float *temperature,
                                  const uint32_t *request_id, int B, int G, int V, int r,
                                  dspark_dtype dtype, uint64_t seed, int32_t *draft_tokens,
                                  float *draft_lse, float *draft_logq, float *draft_logits,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    dspark_status st = check_common(B, G, V, r, dtype);
    if (st != DSPARK_OK) return st;
    if (!base_logits || !e_in || !w_out || !anchor || !temperature || !draft_tokens || !draft_lse || !draft_logq)
        return fail(DSPARK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned(base_logits, 16) || !aligned(e_in, 16) || !aligned(w_out, 16) ||
        (draft_logits && !aligned(draft_logits, 16)))
        return fail(DSPARK_ERR_INVALID_ARG, "logits and weights must be 16-byte aligned");
    const DraftPlan plan = plan_draft(B, G, V, r, dtype);
    if ((st = check_ws(workspace, workspace_bytes, plan.ws_bytes)) != DSPARK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the flag words, and on the tensor path the row-wide best words and the
    // barrier counters after them, in one clear
    cudaError_t e = cudaMemsetAsync(workspace, 0, plan.clear_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the flag words, best words and barrier counters");
    DraftArgs a{base_logits, e_in, w_out, anchor, temperature, request_id, B, G, V, r, dtype, seed,
                draft_tokens, draft_lse, draft_logq, draft_logits, static_cast<unsigned char *>(workspace)};
    if (plan.tensor_path) {
        // the tokens feed the next position through the best words; the
        // partials of every position are merged once at the end
        e = launch_draft_tensor(a, plan, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft sample launch");
        e = launch_draft_finalize(a, plan, 0, G, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft finalize launch");
        return DSPARK_OK;
    }
    if (simt_writes_rows(plan)) {  // one segment per row: every position in one launch
        e = launch_draft_simt(a, plan, 0, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft sample launch");
        return DSPARK_OK;
    }
    for (int j = 0; j < G; ++j) {
        e = launch_draft_simt(a, plan, j, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft sample launch");
        e = launch_draft_finalize(a, plan, j, 1, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft finalize launch");
    }
    return DSPARK_OK;
}

dspark_status dspark_draft_sample_rnn(const void *base_logits, const void *e_in, const void *w_h,
                                      const void *w_out, const int32_t *anchor, const float *temperature,
                                      const uint32_t *request_id, int B, int G, int V, int r,
                                      dspark_dtype dtype, uint64_t seed, int32_t *draft_tokens,
                                      float *draft_lse, float *draft_logq, float *draft_logits,
                                      void *h_states, void *workspace, size_t workspace_bytes, void *stream) {
    dspark_status st = check_common(B, G, V, r, dtype);
    if (st != DSPARK_OK) return st;
    if (dtype != DSPARK_BF16) return fail(DSPARK_ERR_UNSUPPORTED, "the recurrent head runs on bf16 weights only");
    if (!base_logits || !e_in || !w_h || !w_out || !anchor || !temperature || !draft_tokens || !draft_lse ||
        !draft_logq)
        return fail(DSPARK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned(base_logits, 16) || !aligned(e_in, 16) || !aligned(w_h, 16) || !aligned(w_out, 16) ||
        (draft_logits && !aligned(draft_logits, 16)) || (h_states && !aligned(h_states, 2)))
        return fail(DSPARK_ERR_INVALID_ARG, "logits and weights must be 16-byte aligned");
    const RnnPlan plan = plan_draft_rnn(B, G, V, r);
    if ((st = check_ws(workspace, workspace_bytes, plan.ws_bytes)) != DSPARK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // the flag words, the row-wide best words and the barrier counters in one clear
    cudaError_t e = cudaMemsetAsync(workspace, 0, plan.draft.clear_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the flag words and best words");
    DraftArgs a{base_logits, e_in, w_out, anchor, temperature, request_id, B, G, V, r, dtype, seed,
                draft_tokens, draft_lse, draft_logq, draft_logits, ws};
    __nv_bfloat16 *h_ws = reinterpret_cast<__nv_bfloat16 *>(ws + plan.h_offset);
    RnnStateArgs ra{static_cast<const __nv_bfloat16 *>(e_in), static_cast<const __nv_bfloat16 *>(w_h), anchor,
                    reinterpret_cast<const unsigned long long *>(ws + plan.draft.best_offset), h_ws,
                    static_cast<__nv_bfloat16 *>(h_states), B, G, V, r};
    // position j: the state from x_{j-1} and h_{j-1}, then the draw with h_j
    // as the tensor-core A operand; the partials are merged once at the end
    for (int j = 0; j < G; ++j) {
        e = launch_rnn_state(ra, j, s);
        if (e != cudaSuccess) return cuda_fail(e, "recurrent state launch");
        e = launch_draft_tensor_rows(a, plan.draft, j, h_ws + (size_t)j * B * r, s);
        if (e != cudaSuccess) return cuda_fail(e, "draft sample launch");
    }
    e = launch_draft_finalize(a, plan.draft, 0, G, s);
    if (e != cudaSuccess) return cuda_fail(e, "draft finalize launch");
    return DSPARK_OK;
}

dspark_status dspark_schedule_prefix(const float *conf_logits, const float *pos_temp, const float *sps,
                                     int sps_len, int B, int G, int L_min, int L_max, float *conf,
                                     float *cum_conf, int32_t *verify_len, double *theta_out,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    return dspark_schedule_policy(conf_logits, pos_temp, sps, sps_len, B, G, L_min, L_max,
                                  DSPARK_SCHED_EARLY_STOP, 0.f, conf, cum_conf, verify_len, theta_out, workspace,
                                  workspace_bytes, stream);
}

dspark_status dspark_schedule_policy(const float *conf_logits, const float *pos_temp, const float *sps,
                                     int sps_len, int B, int G, int L_min, int L_max, int policy, float threshold,
                                     float *conf, float *cum_conf, int32_t *verify_len, double *theta_out,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    if (policy < DSPARK_SCHED_EARLY_STOP || policy > DSPARK_SCHED_THRESHOLD_CONF)
        return fail(DSPARK_ERR_INVALID_ARG, "unknown scheduling policy %d", policy);
    if (policy >= DSPARK_SCHED_THRESHOLD_CUM && !std::isfinite(threshold))
        return fail(DSPARK_ERR_INVALID_ARG, "threshold must be finite");
    if (B < 1 || G < 1 || G > kMaxG) return fail(DSPARK_ERR_INVALID_ARG, "bad B=%d or G=%d", B, G);
    if (L_min < 0 || L_min > L_max || L_max > G)
        return fail(DSPARK_ERR_INVALID_ARG, "need 0 <= L_min <= L_max <= G (got %d, %d, %d)", L_min, L_max, G);
    if ((long)B * G > kScheduleMaxCells) return fail(DSPARK_ERR_UNSUPPORTED, "B*G > %d", kScheduleMaxCells);
    if ((long)sps_len < (long)B * (L_max + 1) + 1)
        return fail(DSPARK_ERR_INVALID_ARG, "sps_len must be >= B*(L_max+1)+1 = %ld", (long)B * (L_max + 1) + 1);
    if (!conf_logits || !pos_temp || !sps || !conf || !cum_conf || !verify_len)
        return fail(DSPARK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (schedule_smem_bytes(B, G, L_min, L_max) > (size_t)kScheduleMaxSmem)
        return fail(DSPARK_ERR_UNSUPPORTED, "too many scheduler candidates");
    dspark_status st = check_ws(workspace, workspace_bytes, kFlagBytes);
    if (st != DSPARK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // (the kernel clears the flag words itself)
    ScheduleArgs a{conf_logits, pos_temp, sps, sps_len, B, G, L_min, L_max, conf, cum_conf, verify_len,
                   theta_out, static_cast<unsigned char *>(workspace), policy, threshold};
    const cudaError_t e = launch_schedule(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "schedule launch");
    return DSPARK_OK;
}

dspark_status dspark_verify(const void *target_logits, const void *base_logits, const void *e_in,
                            const void *w_out, const float *draft_logits, const int32_t *anchor,
                            const int32_t *draft_tokens, const float *draft_lse, const float *draft_logq,
                            const int32_t *verify_len, const float *temperature,
                            const uint32_t *request_id, int B, int G, int V, int r, dspark_dtype dtype,
                            uint64_t seed, int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
                            float *target_lse, float *logp_sel, void *workspace, size_t workspace_bytes,
                            void *stream) {
    return verify_impl(target_logits, nullptr, 0, base_logits, e_in, w_out, draft_logits, anchor, draft_tokens,
                       draft_lse, draft_logq, verify_len, temperature, request_id, B, G, V, r, dtype, seed,
                       accept_len, out_tokens, num_out, target_lse, logp_sel, workspace, workspace_bytes, stream);
}

dspark_status dspark_verify_packed(const void *target_logits, const int64_t *target_row0, int64_t n_target_rows,
                                   const void *base_logits, const void *e_in, const void *w_out,
                                   const float *draft_logits, const int32_t *anchor, const int32_t *draft_tokens,
                                   const float *draft_lse, const float *draft_logq, const int32_t *verify_len,
                                   const float *temperature, const uint32_t *request_id, int B, int G, int V, int r,
                                   dspark_dtype dtype, uint64_t seed, int32_t *accept_len, int32_t *out_tokens,
                                   int32_t *num_out, float *target_lse, float *logp_sel, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    if (!target_row0) return fail(DSPARK_ERR_INVALID_ARG, "target_row0 is NULL");
    if (n_target_rows < 1) return fail(DSPARK_ERR_INVALID_ARG, "n_target_rows must be >= 1");
    if (n_target_rows > (1LL << 40) / (V > 0 ? V : 1))
        return fail(DSPARK_ERR_INVALID_ARG, "n_target_rows * V too large");
    return verify_impl(target_logits, target_row0, n_target_rows, base_logits, e_in, w_out, draft_logits, anchor,
                       draft_tokens, draft_lse, draft_logq, verify_len, temperature, request_id, B, G, V, r, dtype,
                       seed, accept_len, out_tokens, num_out, target_lse, logp_sel, workspace, workspace_bytes,
                       stream);
}

dspark_status dspark_pack_target(const void *target_logits, const int32_t *verify_len, int B, int G, int V,
                                 dspark_dtype dtype, void *target_packed, int64_t *target_row0, int64_t *n_rows,
                                 void *stream) {
    if (B < 1 || G < 1 || G > kMaxG) return fail(DSPARK_ERR_INVALID_ARG, "bad B=%d or G=%d", B, G);
    if (V < 8 || V % 8 != 0) return fail(DSPARK_ERR_INVALID_ARG, "V must be a positive multiple of 8 (got %d)", V);
    if (dtype != DSPARK_BF16 && dtype != DSPARK_F32) return fail(DSPARK_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if ((long)B * (G + 1) * (long)V > (1L << 40)) return fail(DSPARK_ERR_INVALID_ARG, "B*(G+1)*V too large");
    if (!target_logits || !target_packed || !target_row0)
        return fail(DSPARK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned(target_logits, 16) || !aligned(target_packed, 16) || !aligned(target_row0, 8) ||
        (n_rows && !aligned(n_rows, 8)))
        return fail(DSPARK_ERR_INVALID_ARG, "target arrays must be 16-byte aligned");
    cudaError_t e = launch_pack_target(target_logits, verify_len, B, G, V, dtype == DSPARK_BF16 ? 2 : 4,
                                       target_packed, target_row0, n_rows, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    return DSPARK_OK;
}

dspark_status dspark_selftest_bounded_wait(unsigned int limit_us, uint32_t *result, void *stream) {
    if (!result) return fail(DSPARK_ERR_INVALID_ARG, "result is NULL");
    if (limit_us < 1 || limit_us > 1000000) return fail(DSPARK_ERR_INVALID_ARG, "limit_us must be in [1, 1e6]");
    cudaError_t e = run_bounded_wait_probe(limit_us, result, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test");
    return DSPARK_OK;
}

dspark_status dspark_selftest_philox_rate(void *workspace, size_t workspace_bytes, int iters, double *blocks_per_second,
                                         void *stream) {
    if (!blocks_per_second) return fail(DSPARK_ERR_INVALID_ARG, "blocks_per_second is NULL");
    if (iters < 1 || iters > (1 << 20)) return fail(DSPARK_ERR_INVALID_ARG, "iters must be in [1, 2^20]");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    dspark_status st = check_ws(workspace, workspace_bytes, philox_probe_sink_bytes(sms));
    if (st != DSPARK_OK) return st;
    e = run_philox_probe(workspace, sms, iters, blocks_per_second, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "Philox rate probe");
    return DSPARK_OK;
}

dspark_status dspark_read_device_flags(const void *workspace, void *stream, uint32_t *flags) {
    if (!workspace || !flags) return fail(DSPARK_ERR_INVALID_ARG, "NULL workspace or flags");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the flag word");
    return DSPARK_OK;
}

}  // extern "C"
