/*
 * longstraw.h -- C ABI of the GB300 branch-replay library.
 *
 * The library implements the per-GPU hot path of LongStraw-style branch replay for GRPO
 * (LongStraw review, dimensionstp.github.io "LongStraw": section 1-1 problem definition and
 * the L_policy equation; section 2-1 the five-step transaction; section 3-2 (1) no-grad
 * prompt capture, (3) restore without mutating the prompt state, (4) serial suffix replay;
 * section 4-3 (5) the architecture-adapter interface).  One call sequence per GRPO group:
 *
 *   ls_prefix_prepare          register the resident prompt K/V, zero the fp32 accumulators
 *   for each response i (serially, on one stream):
 *     ls_replay_fwd            suffix attention over [prompt; response_i], causal suffix
 *     ls_grpo_loss             clipped-surrogate loss contribution + dlogits
 *     ls_replay_bwd            dQ, suffix dK/dV; prompt dK/dV added into the accumulators
 *   ls_prefix_grad_finalize    one finalization of the group-summed prompt gradient
 *
 * Around that sequence: ls_token_logp (+ ls_replay_fwd) scores responses without
 * gradients (old/reference policy); ls_block_replay_fwd/bwd replay one long response block
 * by block (section 3-2 (4)); ls_replay_fwd_packed/bwd_packed replay a whole group in one
 * launch per kernel; ls_replay_*_prompt_only with ls_attn_merge and ls_sum_bf16 split the
 * prompt into context-parallel shards (section 3-2 (2)); a handle may be kept across groups
 * (prefix reuse, section 4-2) with ls_prefix_grad_finalize(..., reset_acc = 1) between them.
 *
 * Conventions shared by every entry point
 *  - Pointers named "device" must point to device memory of the current CUDA device,
 *    allocated and owned by the caller.  The library allocates no device memory and never
 *    frees caller memory; it keeps only host-side metadata in the prefix handle.
 *  - Tensors are dense row-major.  "THD" means [tokens, heads, head_dim], contiguous.
 *    bf16 is IEEE bfloat16 stored in 2 bytes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *    work is enqueued on it; calls return before the GPU finishes.
 *  - Argument errors are detected on the host and returned before anything is enqueued.
 *    Launch failures return LS_ERR_CUDA; ls_last_error() gives the CUDA message.
 *    Kernels never trap: a device-side check that fails (a bounded wait that gave up, an
 *    index outside its buffer) sets a device status word that ls_get_device_status()
 *    reads back.
 *  - Prompt-gradient accumulation is atomic-free: every ls_replay_bwd on one handle must
 *    be ordered on one stream (or otherwise serialised by the caller).  The handle is not
 *    thread-safe.
 */
#ifndef LONGSTRAW_H
#define LONGSTRAW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LS_OK = 0,
  LS_ERR_INVALID_ARGUMENT = 1, /* null pointer, non-positive size, bad enum value        */
  LS_ERR_UNSUPPORTED = 2,      /* shape outside the supported set (see ls_prefix_desc)  */
  LS_ERR_NOT_PREPARED = 3,     /* handle is NULL, destroyed or not from ls_prefix_prepare */
  LS_ERR_MISALIGNED = 4,       /* a device pointer is not 16-byte aligned               */
  LS_ERR_CUDA = 5,             /* a CUDA runtime/driver call or a launch failed         */
  LS_ERR_TIMEOUT = 6,          /* a kernel's bounded wait gave up (device status)       */
  LS_ERR_DEVICE_STATUS = 7,    /* a kernel recorded another device-side check failure   */
  LS_ERR_WORKSPACE = 8,        /* workspace pointer NULL or smaller than required       */
  LS_ERR_WRONG_DEVICE = 9      /* current device or stream device differs from handle's */
} ls_status;

/* Opaque prefix handle: host metadata and TMA descriptors of the resident prompt K/V. */
typedef struct ls_prefix_s* ls_prefix_t;

/*
 * Description of the resident prompt state of ONE attention layer (the captured
 * "continuation state" of the review's section 3-2 (1): the prompt's keys and values).
 *   P              prompt length, 1 <= P < 2^31.
 *   Hq, Hkv        query and key/value heads; Hq % Hkv == 0 and g = Hq/Hkv <= 16.  Query
 *                  head h reads kv head h / g (contiguous groups).
 *   D              head dimension, 64 or 128.
 *   softmax_scale  scale s applied to q.k; 0 selects 1/sqrt(D).
 *   k_prefix, v_prefix  device, bf16 THD [P, Hkv, D], 16-byte aligned.  Borrowed: they
 *                  must stay valid and unmodified until ls_prefix_destroy; the library
 *                  only reads them (the review's rule that a replay must not mutate the
 *                  shared prompt state, section 3-2 (3)).
 *   dk_acc, dv_acc device, fp32 [P, Hkv, D], 16-byte aligned.  Borrowed; zeroed by
 *                  ls_prefix_prepare, then each ls_replay_bwd adds that response's
 *                  d loss / d (prompt K, V) into them.
 */
typedef struct {
  int64_t P;
  int32_t Hq;
  int32_t Hkv;
  int32_t D;
  float softmax_scale;
  const void* k_prefix;
  const void* v_prefix;
  float* dk_acc;
  float* dv_acc;
} ls_prefix_desc;

/*
 * ls_prefix_prepare -- prompt capture hand-off (review section 2-1 step 1; section 3-2 (1)).
 * Validates `desc`, encodes the TMA descriptors of the prompt K/V once, and enqueues the
 * zeroing of dk_acc/dv_acc on `stream`.  On success *out receives a new handle bound to
 * the current device.  On error *out is left unchanged and nothing is enqueued.
 */
ls_status ls_prefix_prepare(const ls_prefix_desc* desc, ls_prefix_t* out, void* stream);

/* Release the handle's host metadata.  Does not touch device memory. NULL is a no-op. */
ls_status ls_prefix_destroy(ls_prefix_t h);

/*
 * ls_replay_fwd -- forward replay of one response against the resident prompt
 * (review section 2-1 step 4, "serial policy replay"; section 3-2 (4)).
 * For suffix row t (0 <= t < R) and query head h, with kv = h / g:
 *     keys visible to (t, h):  all P prompt keys, then suffix keys 0..t (causal)
 *     O[t,h,:]  = sum_j softmax_j(s * q[t,h,:] . k_j) v_j
 *     lse[t,h]  = log sum_j exp(s * q[t,h,:] . k_j)        (natural log)
 *   q       device bf16 THD [R, Hq, D]
 *   k_suffix, v_suffix  device bf16 THD [R, Hkv, D]
 *   o       device bf16 THD [R, Hq, D]   (written)
 *   lse     device fp32 [R, Hq]          (written; ls_replay_bwd needs it)
 *   R >= 1.  All pointers 16-byte aligned.
 */
ls_status ls_replay_fwd(ls_prefix_t h, int64_t R, const void* q, const void* k_suffix,
                        const void* v_suffix, void* o, float* lse, void* stream);

/* Bytes of device workspace ls_replay_bwd needs for a response of R tokens. */
size_t ls_replay_bwd_workspace_bytes(ls_prefix_t h, int64_t R);

/*
 * ls_replay_bwd -- backward replay of one response (review section 2-1 step 4: "the
 * suffix graph is released after its backward and only gradients are accumulated";
 * section 2-2, the gradient decomposition at the prompt boundary z_P).
 * With P = softmax(s Q K^T) recomputed from `lse`, dP = dO V^T, Delta = rowsum(dO * O),
 * dS = P * (dP - Delta):
 *     dq       = s dS K                    device bf16 THD [R, Hq, D]   (written)
 *     dk_suffix= s dS^T Q  (suffix keys)   device bf16 THD [R, Hkv, D]  (written)
 *     dv_suffix= P^T dO    (suffix keys)   device bf16 THD [R, Hkv, D]  (written)
 *     dk_acc  += s dS^T Q  (prompt keys)   fp32, the handle's accumulator
 *     dv_acc  += P^T dO    (prompt keys)   fp32, the handle's accumulator
 * kv-head gradients sum over the g query heads of the group.  Inputs q, k_suffix,
 * v_suffix, o (bf16 THD) and lse (fp32 [R, Hq]) are the ones given to / produced by
 * ls_replay_fwd for this response; d_out is bf16 THD [R, Hq, D].
 * The prompt accumulators are read-modified-written by exactly one CTA per tile, in
 * stream order with other calls on the handle: no atomics, bitwise deterministic.
 * workspace: device, >= ls_replay_bwd_workspace_bytes(h, R) bytes, 16-byte aligned.
 */
ls_status ls_replay_bwd(ls_prefix_t h, int64_t R, const void* q, const void* k_suffix,
                        const void* v_suffix, const void* o, const float* lse,
                        const void* d_out, void* dq, void* dk_suffix, void* dv_suffix,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packed replay of several responses in one launch per kernel: the shared-prefix tree
 * [prompt; y_1; ...; y_G] in which every y_b attends to the prompt and, causally, to itself
 * only (the prompt as state shared by the group: LongStraw review, section 2; a shared-prefix
 * tree of trajectories: QwenGyre news article, devotd.net, trajectory-processor paragraph).
 * Response b owns packed rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of q, k_suffix, v_suffix,
 * o, lse, d_out, dq, dk_suffix, dv_suffix (THD layouts as for one response, with the packed
 * row count cu_seqlens[G] in place of R).  cu_seqlens is a HOST array of G+1 int64 values,
 * cu_seqlens[0] = 0, strictly increasing (every response has at least one token);
 * 1 <= G <= 64 (LS_ERR_UNSUPPORTED above).  The results are those of G ls_replay_fwd /
 * ls_replay_bwd calls on the responses one by one; in the backward every prompt 128-key
 * tile accumulates the contributions of all G responses on chip and is added into the
 * fp32 accumulators once.  Activation memory grows with G (the serial calls keep it at
 * one response).
 */
ls_status ls_replay_fwd_packed(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens,
                               const void* q, const void* k_suffix, const void* v_suffix,
                               void* o, float* lse, void* stream);
size_t ls_replay_bwd_packed_workspace_bytes(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens);
ls_status ls_replay_bwd_packed(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens,
                               const void* q, const void* k_suffix, const void* v_suffix,
                               const void* o, const float* lse, const void* d_out, void* dq,
                               void* dk_suffix, void* dv_suffix, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Blockwise suffix replay (review section 3-2 (4), "Blockwise suffix replay": a response is
 * replayed block by block instead of as one graph, which bounds the response's activation
 * peak; attention state has to carry across block boundaries exactly).
 *
 * Layout: the handle's K/V buffers hold [prompt; response] -- the prompt keys in rows
 * 0 .. P0-1 and the response's keys and values in rows P0 .. P0+R_total-1, written by the
 * caller before the block that produces them is replayed; the handle is prepared with
 * P = P0 + R_total (or more).  A block of R rows that starts at response token t0 calls with
 * prefix_len = P0 + t0: its queries see the prefix rows 0 .. prefix_len-1 (prompt and
 * earlier blocks) and, causally, the block's own rows prefix_len .. prefix_len+R-1.
 *
 * ls_block_replay_fwd -- O and lse of the block, exactly as ls_replay_fwd would give them
 * for these rows with prompt = rows 0 .. prefix_len-1 and suffix = the block's own rows.
 *   q device bf16 THD [R, Hq, D]; o device bf16 THD [R, Hq, D] (written);
 *   lse device fp32 [R, Hq] (written).  1 <= prefix_len, prefix_len + R <= P.
 *
 * ls_block_replay_bwd -- the block's dq (bf16 THD [R, Hq, D], written) and the key/value
 * gradients of every row it sees: rows 0 .. prefix_len+R-1 of dk_acc/dv_acc get
 * += s dS^T Q and += P^T dO.  After the last block the response rows of the accumulators
 * hold the complete gradient of the response's keys and values (every later block has
 * added its part), and the prompt rows the prompt's part; read them out with
 * ls_prefix_grad_finalize_rows.  Inputs as ls_replay_bwd; workspace as
 * ls_replay_bwd_workspace_bytes(h, R).  Accumulation is atomic-free and deterministic, as
 * for the prompt in ls_replay_bwd.
 */
ls_status ls_block_replay_fwd(ls_prefix_t h, int64_t prefix_len, int64_t R, const void* q,
                              void* o, float* lse, void* stream);
ls_status ls_block_replay_bwd(ls_prefix_t h, int64_t prefix_len, int64_t R, const void* q,
                              const void* o, const float* lse, const void* d_out, void* dq,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace ls_grpo_loss needs for R token rows. */
size_t ls_grpo_loss_workspace_bytes(int64_t R);

/*
 * ls_grpo_loss -- fused GRPO clipped-surrogate loss of one response (review section 1-1,
 * equation L_policy).  Per token row t of logits x [R, V] with sampled id y_t:
 *     lse   = log sum_v exp(x_v);  logp = x_y - lse;  rho = exp(logp - logp_old[t])
 *     surr  = min(rho A, clip(rho, 1-eps, 1+eps) A)
 *     *loss_accum += -(1/(G R)) sum_t surr          (fp64 device scalar, accumulated)
 *     clip_mask[t] = 1 iff (A > 0 and rho > 1+eps) or (A < 0 and rho < 1-eps)
 *     dlogits[t,v] = g_t (1[v = y_t] - exp(x_v - lse)),  g_t = -A rho [not clipped]/(G R)
 *     logp_out[t]  = logp
 *   logits   device bf16 [R, V];  ids device int32 [R], 0 <= id < V (an id outside that
 *            range sets the device status and its row's outputs are zero)
 *   logp_old device fp32 [R];  advantage A and eps (0 <= eps < 1) host scalars; G >= 1
 *   loss_accum device double (accumulated, not cleared); dlogits device bf16 [R, V]
 *   clip_mask device uint8 [R]; logp_out device fp32 [R] (may be NULL)
 *   workspace device, >= ls_grpo_loss_workspace_bytes(R) bytes, 16-byte aligned.
 * Precision: the row sums of exp are compensated fp32 sums; lse, logp and the loss terms
 * are fp64; the clip decision and g use rho evaluated in fp32 from the fp64 log-ratio
 * (relative error ~2e-7, so the mask equals an exact evaluation except for rho within
 * ~1e-6 of 1 +- eps).  The loss reduction is a fixed-order tree (deterministic).
 * Failure: if a bounded wait inside the kernel gives up (ls_get_device_status then returns
 * LS_ERR_TIMEOUT), every row not finished before it gets a NaN loss term (so *loss_accum
 * becomes NaN), a zero dlogits row, clip_mask 0 and a NaN logp_out; the call itself still
 * returns LS_OK, since the failure happens after it returned.
 */
ls_status ls_grpo_loss(int64_t R, int64_t V, int32_t G, const void* logits, const int32_t* ids,
                       const float* logp_old, double advantage, double eps, double* loss_accum,
                       void* dlogits, uint8_t* clip_mask, float* logp_out, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * ls_token_logp -- token log-probabilities without gradients, for the old- and
 * reference-policy scoring of the responses from the preserved prompt state (review
 * section 2-1 step 2; section 4-2 step 4 of the GLM recipe):
 *     logp_out[t] = x[t, y_t] - log sum_v exp(x[t, v])     (natural log)
 *   logits device bf16 [R, V]; ids device int32 [R] (an id outside [0, V) sets the device
 *   status and gives 0); logp_out device fp32 [R] (written).  One read of the logits; the
 *   row log-sum-exp is combined in fp64 as in ls_grpo_loss (so the values are identical to
 *   ls_grpo_loss's logp_out).  The attention part of scoring is ls_replay_fwd.  Rows left
 *   unfinished by a bounded wait that gave up (LS_ERR_TIMEOUT) get a NaN log-prob.
 */
ls_status ls_token_logp(int64_t R, int64_t V, const void* logits, const int32_t* ids,
                        float* logp_out, void* stream);

/*
 * ls_grpo_loss_noalloc -- ls_grpo_loss for callers that cannot allocate device memory.
 * (The reviewed pages have no counterpart: this is a deployment variant of the loss.)
 * Same arguments, semantics and outputs as ls_grpo_loss, without the workspace: the
 * per-row loss terms live in a fixed scratch array compiled into the library
 * (ls_grpo_loss_noalloc_max_rows() rows of fp64, 512 KB, held by every GPU that loads the
 * library until the process exits).  It is meant for callers that must not call
 * cudaMalloc, e.g. code inside a fixed memory plan or an allocator-free host runtime that
 * only passes pointers to buffers it already owns; it makes no cudaMalloc, cudaFree or other
 * allocating call.
 *   R > ls_grpo_loss_noalloc_max_rows() returns LS_ERR_UNSUPPORTED (message in
 *   ls_last_error()) before anything is enqueued.
 *   The first call on a device looks up the scratch array's device address (once, with
 *   that device current); make that first call before any stream capture.
 *   All calls on a device share the scratch: calls whose kernels may overlap on the GPU
 *   (unordered streams or threads) race; calls ordered on one stream are safe.  Every
 *   scratch entry a call reads was written earlier in the same call (a row left unfinished
 *   by a bounded wait that gave up writes NaN, as in ls_grpo_loss), so no clearing is
 *   needed between calls.  The stream must belong to the current device
 *   (LS_ERR_WRONG_DEVICE otherwise), as for ls_grpo_loss.
 */
ls_status ls_grpo_loss_noalloc(int64_t R, int64_t V, int32_t G, const void* logits,
                               const int32_t* ids, const float* logp_old, double advantage,
                               double eps, double* loss_accum, void* dlogits,
                               uint8_t* clip_mask, float* logp_out, void* stream);

/* Largest R that ls_grpo_loss_noalloc accepts (its fixed scratch capacity in rows). */
int64_t ls_grpo_loss_noalloc_max_rows(void);

/*
 * Context-parallel prompt sharding (LongStraw review, section 3-2 (2) "Physical page
 * ownership": each rank owns a slice of the prompt's K/V pages; local attention results are
 * combined by a cross-rank log-sum-exp and output merge).  Every shard is its own handle
 * over its prompt rows; exactly one shard (the suffix owner) also sees the response's causal
 * suffix and uses ls_replay_fwd/ls_replay_bwd, the others use the prompt-only calls below.
 * Forward: every shard produces a partial (o_r, lse_r) for all R query rows, and
 * ls_attn_merge combines them.  Backward: every shard runs with the MERGED o and lse (so its
 * softmax probabilities are the global ones), adds the exact gradient of its own keys into
 * its accumulators and returns its part of dq; ls_sum_bf16 adds the parts.  On several
 * GPUs the merge inputs arrive by an all-gather and the dq parts leave by a reduce(-scatter);
 * on one GPU the shards are separate handles and the calls below are the whole exchange.
 *
 * ls_replay_fwd_prompt_only / ls_replay_bwd_prompt_only: as ls_replay_fwd / ls_replay_bwd
 * with the handle's prompt keys only (no suffix keys; no suffix gradients).  q, o, d_out,
 * dq bf16 THD [R, Hq, D]; lse fp32 [R, Hq]; workspace as ls_replay_bwd_workspace_bytes.
 *
 * ls_attn_merge: lse[i] = log sum_r exp(lse_parts[r][i]);
 *                o[i, :] = sum_r exp(lse_parts[r][i] - lse[i]) o_parts[r][i, :]
 *   over the R * Hq rows; o_parts / lse_parts are HOST arrays of n device pointers (bf16
 *   [R, Hq, D] / fp32 [R, Hq]); 1 <= n <= 16, D a multiple of 8 (else LS_ERR_UNSUPPORTED).
 *   Weights and sums in fp32.
 *
 * ls_sum_bf16: out[i] = bf16(sum_r float(parts[r][i])), 0 <= i < count; parts a HOST array
 *   of n device pointers (bf16); 1 <= n <= 16, count a multiple of 8.
 *
 * ls_bf16_to_f32 / ls_f32_to_bf16: the element conversions around the cross-rank fp32 sum
 *   of the dq parts (each rank widens its bf16 part exactly, the collective sums in fp32,
 *   the sum is rounded back to bf16 to nearest, ties to even).  count values (a multiple of
 *   8, else LS_ERR_UNSUPPORTED); in and out device, 16-byte aligned, not overlapping.
 */
ls_status ls_replay_fwd_prompt_only(ls_prefix_t h, int64_t R, const void* q, void* o, float* lse,
                                    void* stream);
ls_status ls_replay_bwd_prompt_only(ls_prefix_t h, int64_t R, const void* q, const void* o,
                                    const float* lse, const void* d_out, void* dq,
                                    void* workspace, size_t workspace_bytes, void* stream);
ls_status ls_attn_merge(int32_t n, int64_t R, int32_t Hq, int32_t D, const void* const* o_parts,
                        const float* const* lse_parts, void* o, float* lse, void* stream);
ls_status ls_sum_bf16(int32_t n, int64_t count, const void* const* parts, void* out, void* stream);
ls_status ls_bf16_to_f32(int64_t count, const void* in, float* out, void* stream);
ls_status ls_f32_to_bf16(int64_t count, const float* in, void* out, void* stream);

/*
 * ls_prefix_grad_finalize -- the group's one finalization (review section 2-1 step 5;
 * section 3-2 (7)).  out = scale * acc for the prompt dK and dV accumulators.
 *   dk_out, dv_out  device [P, Hkv, D], bf16 (out_is_fp32 = 0) or fp32 (out_is_fp32 = 1);
 *                   both NULL scales the accumulators in place (fp32).
 *   reset_acc       non-zero: zero the accumulators after reading them (not allowed with
 *                   in-place output).
 * On one GPU no collective is involved.
 */
ls_status ls_prefix_grad_finalize(ls_prefix_t h, float scale, void* dk_out, void* dv_out,
                                  int out_is_fp32, int reset_acc, void* stream);

/*
 * ls_prefix_grad_finalize_rows -- ls_prefix_grad_finalize over accumulator rows
 * row0 .. row0+nrows-1 only (0 <= row0, row0 + nrows <= P); dk_out, dv_out [nrows, Hkv, D].
 * Used to take a response's key/value gradients out of the response rows after blockwise
 * replay (with reset_acc so the rows can hold the next response) and the prompt rows at
 * the end of the group.
 */
ls_status ls_prefix_grad_finalize_rows(ls_prefix_t h, int64_t row0, int64_t nrows, float scale,
                                       void* dk_out, void* dv_out, int out_is_fp32,
                                       int reset_acc, void* stream);

/*
 * Read (and clear) the device status word of the current device: synchronises `stream`,
 * returns LS_OK, LS_ERR_TIMEOUT or LS_ERR_DEVICE_STATUS.  *bits (may be NULL) receives
 * the raw word (1 = a bounded wait gave up, 2 = an index was outside its buffer).
 */
ls_status ls_get_device_status(void* stream, uint32_t* bits);

/*
 * Kernel timing (tracing aid).  While enabled, the library brackets every kernel launch it
 * makes with a pair of CUDA events recorded on the launch's own stream.  ls_timing_read
 * synchronises those events and returns, per kernel id, the summed device time (ms) and
 * the number of launches since the previous read, then forgets them.  Host-side state
 * only; thread-compatible, not thread-safe.  Disabled by default (zero overhead).
 */
typedef enum {
  LS_KERNEL_ZERO = 0,          /* accumulator zeroing (prepare)                   */
  LS_KERNEL_REPLAY_FWD = 1,    /* forward replay                                  */
  LS_KERNEL_BWD_PREP = 2,      /* Delta and row statistics                        */
  LS_KERNEL_BWD_DKDV = 3,      /* dK/dV and prompt accumulation                   */
  LS_KERNEL_BWD_DQ = 4,        /* dQ                                              */
  LS_KERNEL_GRPO_LOSS = 5,     /* loss row pass + fixed-order reduction           */
  LS_KERNEL_FINALIZE = 6,      /* prompt-gradient finalization                    */
  LS_KERNEL_TOKEN_LOGP = 7,    /* scoring: token log-prob only                    */
  LS_KERNEL_MERGE = 8,         /* context-parallel partial-attention merge        */
  LS_KERNEL_SUM = 9,           /* context-parallel dQ part sum                    */
  LS_KERNEL_CAST = 10,         /* context-parallel bf16 <-> fp32 conversions      */
  LS_KERNEL_COUNT = 11
} ls_kernel_id;

ls_status ls_timing_enable(int enable);
/* total_ms and launches have room for n >= LS_KERNEL_COUNT entries (host arrays). */
ls_status ls_timing_read(double* total_ms, int64_t* launches, int n);

/*
 * Failure-detection self test: enqueues one kernel whose bounded mbarrier wait can never
 * complete; after limit_ns (0 < limit_ns <= 10 s) it records the same "bounded wait gave
 * up" bit the replay kernels record, and exits without faulting.  A following
 * ls_get_device_status() returns LS_ERR_TIMEOUT (and clears the word); the context stays
 * usable.
 */
ls_status ls_debug_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * Launch-failure injection (test aid for the error paths; no GPU fault is involved).
 * ls_debug_fail_launch(after) arms a countdown of the library's launch attempts: the next
 * `after` attempts launch normally and the one after them is not made -- the entry point
 * making it returns LS_ERR_CUDA with "launch failure injected" in ls_last_error(), exactly
 * as for a real launch error, and the countdown disarms.  after < 0 disarms it.  A call that
 * launches several kernels (ls_replay_bwd: prep, dK/dV, dQ; the two halves of the zeroing and
 * of the finalization) counts each as one attempt, so a failure can be placed between them.
 * Calls rejected by their argument checks make no attempt and do not consume the countdown.
 * ls_debug_fail_launch_pending() returns the countdown (-1 when disarmed).  Process-wide.
 */
ls_status ls_debug_fail_launch(int64_t after);
int64_t ls_debug_fail_launch_pending(void);

const char* ls_status_string(ls_status s);

/* Message of the last CUDA failure seen by this thread ("" if none). */
const char* ls_last_error(void);

/* Library version string, e.g. "0.1.0". */
const char* ls_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LONGSTRAW_H */
