// Host-side declarations shared by the entry points and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr int kNumSMs = 152;            // GB300: 2 dies x 76 SMs
constexpr size_t kFlagBytes = 256;      // flag word region at the head of every workspace
constexpr int kMaxG = 64;
constexpr int kMaxV = 1 << 20;         // token ids fit the 20-bit field of the key words

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A set-up call made once per device, such as raising a kernel's dynamic
// shared-memory limit (a property of the function on each device).
struct PerDeviceOnce {
    std::mutex mu;
    bool done[64] = {};
    cudaError_t result[64] = {};
    template <typename Fn>
    cudaError_t run(Fn &&fn) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            result[dev] = fn();
            done[dev] = true;
        }
        return result[dev];
    }
};

// Record the message returned by dspark_last_error() and return `st`.
dspark_status set_last_error(dspark_status st, const char *fmt, ...);

// dspark_verify's host-side checks of sizes, pointers and alignment.
dspark_status verify_check_args(const void *target_logits, const void *base_logits, const void *e_in,
                                const void *w_out, const float *draft_logits, const int32_t *anchor,
                                const int32_t *draft_tokens, const float *draft_lse, const float *draft_logq,
                                const float *temperature, int B, int G, int V, int r, dspark_dtype dtype,
                                const int32_t *accept_len, const int32_t *out_tokens, const int32_t *num_out);

// ------------------------------------------------------------- selftest ----
cudaError_t run_bounded_wait_probe(unsigned int limit_us, uint32_t *result, cudaStream_t s);
size_t philox_probe_sink_bytes(int sms);
cudaError_t run_philox_probe(void *sink, int sms, int iters, double *blocks_per_s, cudaStream_t s);

// ----------------------------------------------------------------- pack ----
cudaError_t launch_pack_target(const void *src, const int32_t *verify_len, int B, int G, int V, size_t elem_bytes,
                               void *dst, int64_t *row0, int64_t *n_rows, cudaStream_t s);

// ---------------------------------------------------------------- draft ----
struct DraftPlan {
    bool tensor_path;      // tcgen05 Markov-head kernel (bf16) vs SIMT kernel
    int rows_per_block;    // SIMT: requests per block
    int row_blocks;        // SIMT: ceil(B / rows_per_block); tensor path: M tiles
    int nsplit;            // vocabulary segments per row (partials per row)
    int chunk;             // vocabulary entries per segment (SIMT; a multiple of 16)
    size_t partial_offset; // byte offset of the per-(row, segment) partials ([G][B][nsplit] on the tensor path)
    size_t best_offset;    // [G][B] 64-bit row-wide best (key, token) words (tensor path), right after the flags
    size_t bar_offset;     // [row_blocks] barrier counters between positions (tensor path), after the words
    size_t clear_bytes;    // bytes from offset 0 zeroed per call: flag words (+ best words + counters)
    size_t ws_bytes;
};
DraftPlan plan_draft(int B, int G, int V, int r, dspark_dtype dt);
// the recurrent head's workspace: a bf16 draft plan plus the [G][B][r] states
// at h_offset
struct RnnPlan {
    DraftPlan draft;
    size_t h_offset;
    size_t ws_bytes;
};
RnnPlan plan_draft_rnn(int B, int G, int V, int r);

struct DraftArgs {
    const void *base;
    const void *e_in;
    const void *w_out;
    const int32_t *anchor;
    const float *temperature;
    const uint32_t *request_id;
    int B, G, V, r;
    dspark_dtype dt;
    uint64_t seed;
    int32_t *tokens;
    float *lse;
    float *logq;
    float *z_out;
    unsigned char *ws;
};
cudaError_t launch_draft_simt(const DraftArgs &a, const DraftPlan &p, int j, cudaStream_t s);
// whether the SIMT launch writes its tokens, lse and log q itself (one
// vocabulary segment per row: no finalize launch, and one launch from position
// j to the last)
bool simt_writes_rows(const DraftPlan &p);
// merges the partials of positions j .. j + npos - 1 into tokens, lse and log q
cudaError_t launch_draft_finalize(const DraftArgs &a, const DraftPlan &p, int j, int npos, cudaStream_t s);
// every block position (one cooperative launch, else one launch per position)
cudaError_t launch_draft_tensor(const DraftArgs &a, const DraftPlan &p, cudaStream_t s);
// recurrent head: h_j = bf16(tanh(E_in[x_{j-1}] + W_h h_{j-1})) into h_ws + j B r
struct RnnStateArgs {
    const __nv_bfloat16 *e_in;        // [V][r]
    const __nv_bfloat16 *w_h;         // [r][r], row n = weights of state unit n
    const int32_t *anchor;            // [B]
    const unsigned long long *best;   // [G][B] row-wide best words of the draft launches
    __nv_bfloat16 *h_ws;              // [G][B][r] states
    __nv_bfloat16 *h_out;             // optional [B][G][r] copy of the states
    int B, G, V, r;
};
int rnn_rows_per_block(int B);
cudaError_t launch_rnn_state(const RnnStateArgs &a, int j, cudaStream_t s);
// block position j alone, with the A operand of request b read from a_rows + b r
// (bf16) instead of E_in[x_{j-1}]
cudaError_t launch_draft_tensor_rows(const DraftArgs &a, const DraftPlan &p, int j, const void *a_rows,
                                     cudaStream_t s);

// tensor-core kernel geometry (bf16): 128-request row blocks x vocabulary segments
int tc_row_blocks(int B);
int tc_row_replication(int B);
int tc_segments(int B, int V);
size_t tc_residual_state_bytes();

// final draw of verification on the tensor cores: residual rows (rejected at
// position d, draft logits rebuilt with the Markov bias) and bonus rows
// (fully accepted, Gumbel-max over target row L)
struct FinalArgs {
    const void *target;
    const int64_t *target_row0;
    int64_t n_target_rows;
    const void *base;
    const void *e_in;
    const void *w_out;
    const int32_t *anchor;
    const int32_t *tokens;
    const float *temperature;
    const uint32_t *request_id;
    const int32_t *final_code; // [B]: -1, (1 << 16) | d residual, (2 << 16) | L bonus
    const float2 *lse_t_row;   // [B] target lse of the rejected row, natural log as float-float (hi, lo)
    const float *draft_lse;    // [B][G] natural log
    int B, G, V, r, nseg;
    int pass;                  // traversal direction of the vocabulary segments (odd: backwards)
    uint64_t seed;
    void *rpart;               // [B][nseg] final-draw partials
    uint32_t *res_best;        // [B] row-wide best residual key (ordered encoding), zeroed by the decide pass
    uint32_t *flags;
};
cudaError_t launch_final_tensor(const FinalArgs &a, cudaStream_t s);

// --------------------------------------------------------------- verify ----
struct VerifyPlan {
    bool tensor_residual;   // residual rows rebuilt on the tensor cores (bf16)
    int row_split;          // segments per target row in the row pass
    int row_chunk;
    int res_split;          // segments per residual row, SIMT kernel
    int res_chunk;          // entries per segment, SIMT kernel
    int res_split_tc;       // segments per residual row, tensor-core kernel (0 = unused)
    size_t row_part_offset; // [B][G+1][row_split] RowState
    size_t res_row_offset;  // [B] int32: rejected position or -1
    size_t lse_t_offset;    // [B] float2: target lse of the rejected row (natural log, hi + lo)
    size_t res_part_offset; // [B][res_split] ResidualState
    size_t res_best_offset; // [B] uint32 row-wide best residual key of the tensor-core final draw
    size_t ws_bytes;
};
VerifyPlan plan_verify(int B, int G, int V, int r, dspark_dtype dt);

struct VerifyArgs {
    const void *target;
    const int64_t *target_row0;  // packed target: request b's row 0 (nullptr: dense [B][G+1][V])
    int64_t n_target_rows;
    const void *base;
    const void *e_in;
    const void *w_out;
    const float *z_in;
    const int32_t *anchor;
    const int32_t *draft_tokens;
    const float *draft_lse;
    const float *draft_logq;
    const int32_t *verify_len;
    const float *temperature;
    const uint32_t *request_id;
    int B, G, V, r;
    dspark_dtype dt;
    uint64_t seed;
    int32_t *accept_len;
    int32_t *out_tokens;
    int32_t *num_out;
    float *target_lse;
    float *logp_sel;
    unsigned char *ws;
};
cudaError_t launch_verify(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s);

// ------------------------------------------------------------- schedule ----
struct ScheduleArgs {
    const float *conf_logits;
    const float *pos_temp;
    const float *sps;
    int sps_len;
    int B, G, L_min, L_max;
    float *conf;
    float *cum_conf;
    int32_t *verify_len;
    double *theta_out;
    unsigned char *ws;
    int policy;        // dspark_sched_policy
    float threshold;   // policies 2 and 3
};
constexpr int kScheduleMaxCells = 16384;  // B * G
constexpr int kScheduleMaxSmem = 200 * 1024;  // dynamic shared memory of the scheduler's block, at most
size_t schedule_smem_bytes(int B, int G, int L_min, int L_max);
cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s);

// Launch `kernel` as a programmatic dependent of the stream's previous kernel:
// its blocks may be scheduled while that kernel drains, and every kernel
// launched this way starts with griddepcontrol.wait (griddep_wait), which
// returns once the previous kernel has completed and its writes are visible.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dspark
