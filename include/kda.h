/*
 * libkda — Kimi Delta Attention (KDA) recurrent decode for GB300 (sm_103a).
 *
 * One decode step of the KDA recurrence per (row, head) "unit".  The state
 * S of a unit is a 128 x 128 matrix stored as S[k][v]: row = key channel,
 * column = value channel, value channel contiguous.  With q, k L2-normalised
 * (eps 1e-6), g the per-key-channel log decay and beta the delta-rule rate:
 *
 *     S_d = diag(exp(g)) S
 *     u   = beta * (v - S_d^T k)
 *     S'  = S_d + k u^T                  (written back in place)
 *     o   = scale * S'^T q               (scale = 1/sqrt(128) by default)
 *
 * Sources, cited by page title and section:
 *   [P1] "flashinfer.kda_decode" (module overview): the Kimi-Linear T=1 gate
 *        -exp(A_log) * softplus(g + dt_bias), beta sigmoid and QK
 *        normalisation in-kernel; Q, K, V may be views into one padded
 *        projection row and raw G / beta may have independent row strides;
 *        packed cu_seqlens form with ragged lengths and null slots
 *        ("Frozen / speculative-verify mode").
 *   [P2] "flashinfer.kda_decode.fused_kda_decode" (Parameters): the fused
 *        conv + KDA + gated RMSNorm contract.
 *   [P3] "feat(cake_kda): add serving-native packed decode backend" ("Exact
 *        contract"): the packed Kimi K3 T=1 contract.
 *   [P4] "feat(kda): add fused speculative decode kernel - #4809": the
 *        packed fused operation (description) that updates conv and
 *        recurrent caches from accepted-token metadata; the review of the
 *        T=1 row mapping (token rows past the last sequence are padding
 *        that write zero and touch no slot); the bf16-state follow-up
 *        (float32 recurrence across tokens, one rounding per checkpoint).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor data pointers are DEVICE memory owned by the caller.  The
 *   library allocates nothing, never synchronises the host, and never reads
 *   device memory on the host, so every call can be captured in a CUDA graph.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *   stream) of the calling thread's current device, which must be a
 *   compute-capability 10.3 (GB300) device.  An unsupported device returns
 *   KDA_ERR_UNSUPPORTED; there is no fallback path.
 * - Every call launches exactly one kernel.  Any contract breach (dtype,
 *   rank, shape, stride, alignment, aliasing) is detected on the host and
 *   returned as a status WITHOUT launching anything; kda_last_error_message()
 *   then describes it.  A launch failure returns KDA_ERR_CUDA.
 * - state_indices: contiguous int32, one entry per decode row (per sequence
 *   and checkpoint column for kda_packed_fused_decode).  A row whose
 *   index is <= 0 or >= num_slots is a null row: its output is zero and no
 *   cache slot is read or written (slot 0 is the reserved null slot).  Live
 *   indices must be unique; that is a caller contract the library does not
 *   check (it would need a device read).
 * - State pool [num_slots, H, 128, 128], float32 or bfloat16: each slot's
 *   [H, 128, 128] block is contiguous, the slot stride is any value >=
 *   H*128*128 that keeps 16-byte alignment.  The recurrence runs in float32;
 *   a bfloat16 state is rounded once (round-to-nearest-even) on write-back.
 * - Outputs are bfloat16 and contiguous, rounded to nearest even.
 * - Strides are in elements.  Activation vectors need unit stride on the
 *   channel axis and 16-byte (float32) or 8-byte (bfloat16) aligned rows.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* bad dtype / rank / shape / stride / alignment / null pointer */
  KDA_ERR_UNSUPPORTED = 2, /* valid request this build does not serve (device, head count) */
  KDA_ERR_ALIAS = 3,       /* a written tensor overlaps another argument */
  KDA_ERR_CUDA = 4         /* a CUDA runtime call or the launch failed */
} kda_status;

typedef enum kda_dtype { KDA_F32 = 0, KDA_BF16 = 1, KDA_I32 = 2 } kda_dtype;

/* A strided view of device memory.  shape/stride entries past ndim are ignored. */
typedef struct kda_tensor {
  void* data;        /* device address of element [0, ..., 0] */
  int32_t dtype;     /* kda_dtype */
  int32_t ndim;      /* 1..4 */
  int64_t shape[4];
  int64_t stride[4]; /* in elements */
} kda_tensor;

/*
 * kda_recurrent_decode — T=1 recurrent decode with split q, k, v.
 * [P1] Kimi-Linear T=1 equal-head schedules; [P2] "lower_bound" for the
 * bounded gate.
 *
 *   q, k, v     [B, H, 128] or [B, 1, H, 128], float32 or bfloat16 (one dtype
 *               for all three); any positive row and head strides.
 *   raw_gate    same shape as q, float32 or bfloat16 (pre-gate values).
 *   raw_beta    [B, H] or [B, 1, H], float32 or bfloat16 (logits).
 *   A_log       [H] float32, contiguous.
 *   dt_bias     [H*128] or [H, 128] float32, contiguous.
 *   state_indices [B] int32, contiguous.
 *   state       [num_slots, H, 128, 128] float32 or bfloat16, updated in place.
 *   out         [B, H, 128] or [B, 1, H, 128] bfloat16, contiguous (written).
 *   has_lower_bound = 0: g = -exp(A_log[h]) * softplus(raw_gate + dt_bias).
 *   has_lower_bound = 1: g = lower_bound * sigmoid(exp(A_log[h]) * (raw_gate + dt_bias)),
 *               lower_bound < 0.
 *   scale       output scale (> 0), normally 1/sqrt(128).
 */
kda_status kda_recurrent_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                const kda_tensor* raw_gate, const kda_tensor* raw_beta,
                                const kda_tensor* A_log, const kda_tensor* dt_bias,
                                const kda_tensor* state_indices, const kda_tensor* state,
                                const kda_tensor* out, int32_t has_lower_bound,
                                float lower_bound, float scale, void* stream);

/*
 * kda_packed_decode — serving-native packed Kimi K3 T=1 decode ([P3] "Exact
 * contract"): H = 12, K = V = 128, bfloat16 data and bfloat16 state, fixed
 * scale 1/sqrt(128), L2 eps 1e-6 and lower_bound -5.
 *
 *   mixed_qkv   [B, 4608] bfloat16: q | k | v, each 12 x 128 head-major;
 *               channel stride 1, any row stride.
 *   raw_gate    [B, 1536] bfloat16, channel stride 1, any row stride.
 *   raw_beta    [B, 12] bfloat16.
 *   A_log       [12] float32;  dt_bias [1536] float32.
 *   state_indices [B] int32 (-1 = inactive graph-padding row).
 *   state       [num_slots, 12, 128, 128] bfloat16, updated in place.
 *   out         [B, 1, 12, 128] or [B, 12, 128] bfloat16, contiguous.
 */
kda_status kda_packed_decode(const kda_tensor* mixed_qkv, const kda_tensor* raw_gate,
                             const kda_tensor* raw_beta, const kda_tensor* A_log,
                             const kda_tensor* dt_bias, const kda_tensor* state_indices,
                             const kda_tensor* state, const kda_tensor* out, void* stream);

/*
 * kda_fused_decode — width-4 depthwise causal conv + SiLU, one KDA step and
 * gated RMSNorm ([P2] "fused_kda_decode", Parameters).  conv_state and state
 * are updated in place; null rows touch neither.
 *
 *   x           [rows, 3*H*128] bfloat16 packed q|k|v projection, channel stride 1.
 *   conv_weight [3, 4, H*128] float32 contiguous (section q/k/v, tap, channel).
 *   conv_state  [num_slots, 3*H*128, 3] bfloat16 with strides
 *               [slot_stride, 1, 3*H*128]: cached raw samples, oldest first.
 *   raw_gate    [1, rows, H, 128] or [rows, H, 128] bfloat16.
 *   raw_beta    [1, rows, H] or [rows, H] bfloat16.
 *   A_log [H], dt_bias [H*128] float32;  state_indices [rows] int32.
 *   state       [num_slots, H, 128, 128] float32 or bfloat16 (same num_slots
 *               as conv_state).
 *   output_gate [rows, H, 128] or [1, rows, H, 128] bfloat16 (gate logits).
 *   norm_weight [128] float32.
 *   has_lower_bound / lower_bound: gate form as in kda_recurrent_decode
 *               (the pages' default is the bounded gate with -5).
 *   norm_eps    RMSNorm epsilon (>= 0, default 1e-5).
 *   out         [1, rows, H, 128] or [rows, H, 128] bfloat16 contiguous:
 *               RMSNorm(o) * norm_weight * sigmoid(output_gate).
 */
kda_status kda_fused_decode(const kda_tensor* x, const kda_tensor* conv_weight,
                            const kda_tensor* conv_state, const kda_tensor* raw_gate,
                            const kda_tensor* raw_beta, const kda_tensor* A_log,
                            const kda_tensor* dt_bias, const kda_tensor* state_indices,
                            const kda_tensor* state, const kda_tensor* output_gate,
                            const kda_tensor* norm_weight, int32_t has_lower_bound,
                            float lower_bound, float norm_eps, const kda_tensor* out,
                            void* stream);

/*
 * kda_spec_decode — packed speculative decode, T >= 1 tokens per row with
 * ragged cu_seqlens ([P1] Cake T=1..6 family with precomputed gates and
 * "Frozen / speculative-verify mode"'s packed cu_seqlens form; [P4] padding).
 *
 *   q, k, v     [R, H, 128] float32 or bfloat16 token rows (one dtype).
 *   g           [R, H, 128] float32 precomputed log decay (<= 0).
 *   beta        [R, H] float32 or bfloat16: logits if beta_is_logit, else rates.
 *   cu_seqlens  [N+1] int32 contiguous, read on the device: row n owns token
 *               rows cu[n] .. cu[n+1]-1, processed in order with the state
 *               kept in float32 on chip; its final state goes to its slot.
 *               Token rows outside [cu[0], cu[N]) are padding: zero output.
 *               Rows are clamped to [0, R); empty rows do nothing.
 *   t_max       host hint: longest row expected (>= 1); used for scheduling
 *               only, longer rows are still processed correctly.
 *   state_indices [N] int32;  state [num_slots, H, 128, 128] float32/bfloat16.
 *   out         [R, H, 128] bfloat16 contiguous.
 *   scale       output scale (> 0).
 */
kda_status kda_spec_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                           const kda_tensor* g, const kda_tensor* beta, int32_t beta_is_logit,
                           const kda_tensor* cu_seqlens, int32_t t_max,
                           const kda_tensor* state_indices, const kda_tensor* state,
                           const kda_tensor* out, float scale, void* stream);

/*
 * kda_spec_verify_decode — speculative-verify mode ([P1] "Frozen /
 * speculative-verify mode"): the kda_spec_decode outputs for up to 16 tokens
 * per row computed from a read-only committed state pool; the state is never
 * written.  Arguments as kda_spec_decode (state is read only, t_max <= 16),
 * plus two optional slot-indexed out-params for a later commit of the
 * accepted tokens (either may be NULL):
 *   correction_cache [num_slots, H, T_cap, 128] float32 contiguous: for the
 *                token at position t < T_cap of a live row, its delta-rule
 *                correction u_t = beta (v - S_d^T k_hat);
 *   kg_cache     [num_slots, H, T_cap, 256] float32 contiguous: that token's
 *                raw key (128) followed by its log decay g (128).
 * T_cap (1..16) is the caches' third extent (equal when both are given).  The
 * state after accepting the first a tokens of a row is, token by token,
 * S <- diag(exp(g)) S + normalise(k) u^T.  Null and empty rows write no cache
 * entry; tokens at positions >= T_cap are decoded but not cached.
 */
kda_status kda_spec_verify_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                  const kda_tensor* g, const kda_tensor* beta, int32_t beta_is_logit,
                                  const kda_tensor* cu_seqlens, int32_t t_max,
                                  const kda_tensor* state_indices, const kda_tensor* state,
                                  const kda_tensor* out, const kda_tensor* correction_cache,
                                  const kda_tensor* kg_cache, float scale, void* stream);

/*
 * kda_packed_fused_decode — packed fused speculative decode with per-token
 * checkpoints ([P4] description, the review thread on the T=1 row mapping,
 * and its bf16-state follow-up): the kda_fused_decode step (conv + SiLU, KDA,
 * gated RMSNorm) run over the T >= 1 token rows of each of N packed
 * sequences, one sequence after another's rows in x.
 *
 *   x, conv_weight, conv_state, raw_gate, raw_beta, A_log, dt_bias,
 *   output_gate, norm_weight, has_lower_bound, lower_bound, norm_eps, out:
 *               as kda_fused_decode, with R token rows in place of rows.
 *   state_indices [N, C] int32, column stride 1: checkpoint slots of each
 *               sequence (C >= 1).
 *   query_start_loc [N+1] int32 contiguous, read on the device: sequence n
 *               owns token rows qsl[n] .. qsl[n+1]-1 (clamped to [0, R)).
 *   num_accepted_tokens [N] int32, read on the device: a_n.
 *   state       [num_slots, H, 128, 128] float32 or bfloat16.
 * Sequence n starts from the conv and recurrent caches of slot
 * state_indices[n, a_n - 1] and, after its j-th token (j < C), writes both
 * caches to slot state_indices[n, j]; a slot outside [1, num_slots) there is
 * skipped.  The recurrence stays in float32 across the tokens; a bfloat16
 * checkpoint is rounded once when stored.  A sequence whose start slot is
 * null, or whose a_n is outside 1..C, writes zero output rows and no cache;
 * empty sequences do nothing; token rows outside [qsl[0], qsl[N]) are
 * padding with zero output.  Checkpoint slots must be distinct across the
 * call (the start slot may be one of the sequence's own).  The rows of x,
 * raw_gate and output_gate are copied to shared memory in 16-byte pieces:
 * their base addresses and outer strides must be multiples of 16 bytes
 * (KDA_ERR_UNSUPPORTED otherwise).
 */
kda_status kda_packed_fused_decode(const kda_tensor* x, const kda_tensor* conv_weight,
                                   const kda_tensor* conv_state, const kda_tensor* raw_gate,
                                   const kda_tensor* raw_beta, const kda_tensor* A_log,
                                   const kda_tensor* dt_bias, const kda_tensor* state_indices,
                                   const kda_tensor* query_start_loc,
                                   const kda_tensor* num_accepted_tokens, const kda_tensor* state,
                                   const kda_tensor* output_gate, const kda_tensor* norm_weight,
                                   int32_t has_lower_bound, float lower_bound, float norm_eps,
                                   const kda_tensor* out, void* stream);

/* ---- host-only queries (no CUDA calls) ---------------------------------- */

/* Operation ids for kda_plan_split. */
typedef enum kda_op {
  KDA_OP_RECURRENT = 0,
  KDA_OP_PACKED = 1,
  KDA_OP_FUSED = 2,
  KDA_OP_SPEC = 3,
  KDA_OP_PACKED_FUSED = 4
} kda_op;

/*
 * Value-column split the dispatcher picks for `units` = rows * heads on a
 * device with `sm_count` SMs (state_dtype: KDA_F32 / KDA_BF16; t_max: tokens
 * per row, 1 for T=1).  Each CTA then owns 128/split value columns of one
 * unit.  Returns the split (1, 2, 4, 8 or 16), or 0 on invalid arguments.
 * Honors kda_set_split_override.  For KDA_OP_PACKED_FUSED (units =
 * sequences * heads) the split is the size of the thread-block cluster that
 * shares a unit (1, 2, 4 or 8; a forced 16 runs as 8); for KDA_OP_FUSED it
 * is the cluster size of the split schedule: 1 unless forced (2 or 4; a
 * forced 8 or 16 runs as 4).
 */
int32_t kda_plan_split(int32_t op, int64_t units, int32_t state_dtype, int32_t t_max,
                       int32_t sm_count);

/*
 * Force the split of every later call in this process (0 restores the
 * measured policy).  For sweeps and tests.  Returns KDA_ERR_INVALID_ARG for
 * a split this build has no kernel for.  A forced split selects the split
 * schedule for the T=1 entry points unless a schedule is forced too.
 */
kda_status kda_set_split_override(int32_t split);

/*
 * Kernel schedules of the T=1 entry points (kda_recurrent_decode,
 * kda_packed_decode, kda_fused_decode).  SPLIT: one CTA per (row, head,
 * value split; the fused entry point's splits form a thread-block cluster
 * that shares the RMSNorm), the state block streamed through registers;
 * best for latency-bound batches.
 * STREAM: one persistent CTA per SM, a loader warp moving whole state
 * blocks (TMA, swizzled) and the unit's activation vectors into
 * shared-memory stages with bulk asynchronous copies while consumer warps
 * update earlier ones; needs every activation head vector (and, fused, the
 * conv-cache slots and conv_weight) 16-byte aligned, otherwise the call uses SPLIT, or
 * returns KDA_ERR_UNSUPPORTED if STREAM is forced.
 * MMA (kda_spec_decode and kda_spec_verify_decode with a bfloat16 state
 * pool): the chunked form of the token loop on the tensor cores ([P1]
 * "Frozen / speculative-verify mode" names the WY-parallel tensor-core form
 * of these rows): per chunk of up to 8 tokens, S^T [P k | P q] and the
 * rank-T update run as tcgen05 MMAs with float32 accumulators in tensor
 * memory, every operand as three bf16 pieces (within 2^-24 of its float32
 * value); one persistent CTA per SM.  The dispatcher picks it for a bfloat16
 * state pool with t_max >= 14 (unless a split or the SPLIT/STREAM schedule is
 * forced); forcing MMA with a float32 state returns KDA_ERR_UNSUPPORTED.
 * The speculative entry points otherwise use SPLIT (one CTA per row, head
 * and value slab, the state in registers).
 */
typedef enum kda_schedule {
  KDA_SCHED_AUTO = 0,
  KDA_SCHED_SPLIT = 1,
  KDA_SCHED_STREAM = 2,
  KDA_SCHED_MMA = 3
} kda_schedule;

/* Schedule the dispatcher picks (same arguments as kda_plan_split); 0 on invalid arguments. */
int32_t kda_plan_schedule(int32_t op, int64_t units, int32_t state_dtype, int32_t t_max,
                          int32_t sm_count);

/* Force the schedule of later calls (KDA_SCHED_AUTO restores the policy):
 * SPLIT / STREAM apply to the T=1 entry points, SPLIT / MMA to the
 * speculative ones; a schedule an entry point does not have is ignored
 * there. */
kda_status kda_set_schedule_override(int32_t schedule);

/*
 * Device error word of the streaming kernels on the current device: bit 0 =
 * a wait for a filled stage timed out (2 s), bit 1 = a wait for a free stage
 * timed out, bit 2 = the kda_selftest_wait_timeout wait gave up (expected),
 * bit 3 = a wait of the tensor-core (MMA) speculative kernel timed out.  A
 * kernel that times out records the bit and returns early, its results for
 * the affected units are undefined.  Synchronises the device;
 * clears the word when `clear` is non-zero.
 */
kda_status kda_device_error(uint32_t* flags, int32_t clear);

/*
 * Diagnostic of the bounded waits: launches one warp on `stream` that waits
 * on a barrier nothing completes.  The wait gives up after 2 s and sets bit
 * 2 (value 4) of the device error word, so the timeout path can be checked
 * without faulting or hanging the GPU; the context stays usable.
 */
kda_status kda_selftest_wait_timeout(void* stream);

const char* kda_status_string(kda_status s);
/* Detail of the last non-OK status returned on the calling thread. */
const char* kda_last_error_message(void);
/* Library version string. */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
