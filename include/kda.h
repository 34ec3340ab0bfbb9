/*
 * kda.h -- C ABI of libkda, Kimi Delta Attention (KDA) on NVIDIA GB300 (sm_103a).
 *
 * KDA is the per-channel gated delta rule.  For one head with key width dk and
 * value width dv, state S (dk x dv, fp32) and tokens t = 1, 2, ...:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * The pages define the step in words: "Kimi K3 Architecture Teardown",
 * section "Hybrid Attention for 1M Tokens", Visual 5 -- decay every key
 * channel of the state, erase a beta-scaled share of what it holds under the
 * current key, write the new key-value pair scaled by the same beta;
 * "Kimi K3 Architecture: KDA, MoE, and Attention", section "Memory as a
 * First-Class Problem" -- alpha is a per-channel decay, one beta erases and
 * writes, and the output queries the UPDATED state.  A checkpointed state can
 * resume prefill (prefix-cache hit): "Kimi K3 Architecture Teardown", section
 * "Scale: Total vs Active Parameters and Serving Economics", and "Kimi K3
 * architecture: KDA, MLA and MoE", section "Serving K3 means managing two
 * cache lifecycles".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers to row-major, contiguous memory
 *   owned by the caller.  The library allocates no memory and keeps no state
 *   between calls, except one device status word used to report a timed-out
 *   wait inside a kernel, and, in bounds-checked diagnostic builds, an index
 *   that left its buffer (see kda_device_status).
 * - Layouts (T = shape->total_tokens, N = shape->num_seqs):
 *     q, k       [T, H, dk]   dtype
 *     v, out     [T, H, dv]   dtype
 *     log_alpha  [T, H, dk]   fp32, log of the decay alpha in (0, 1], so <= 0;
 *                             -inf (alpha = 0) is allowed
 *     beta       [T, H]       dtype, the write strength (no clamp is applied)
 *     states     [N, H, dk, dv] fp32
 *   A dense batch [B, T', H, d] is the same memory with N = B, T = B*T' and
 *   cu_seqlens = NULL.
 * - q and k are expected to be L2-normalised by the caller; the library does
 *   not normalise them.  There is no query scale: o_t = S_t^T q_t exactly.
 * - Supported: dtype KDA_BF16 or KDA_F32; dk, dv in {64, 128}.
 * - Pointers q, k, v, out, log_alpha and the state pointers must be 16-byte
 *   aligned (else KDA_ERR_UNSUPPORTED); beta must be aligned to its element.
 * - Every call is asynchronous on `stream`: it validates its arguments on the
 *   host, enqueues kernels and returns.  On any error nothing is enqueued.
 * - Arithmetic: fp32 accumulation and an fp32 state throughout.  With bf16
 *   inputs and dk = dv = 128 prefill runs the chunkwise tensor-core kernel
 *   (bf16 operands, fp32 accumulators); other shapes run an fp32 recurrent
 *   kernel.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad cu_seqlens  */
    KDA_ERR_UNSUPPORTED = 2,  /* dtype / head size / alignment not supported  */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed          */
    KDA_ERR_TIMEOUT = 4,      /* a bounded in-kernel wait gave up (see below)  */
    KDA_ERR_BOUNDS = 5        /* bounds-checked builds only: an index left its buffer */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

typedef struct {
    int32_t num_seqs;       /* N: sequences (prefill) or rows (decode), >= 0  */
    int64_t total_tokens;   /* T: packed token count, >= 0                     */
    int32_t H;              /* heads, >= 1                                    */
    int32_t dk;             /* key / query width per head                     */
    int32_t dv;             /* value width per head                           */
    kda_dtype dtype;        /* dtype of q, k, v, beta and out                 */
} kda_shape;

/*
 * kda_prefill -- run the recurrence over N packed sequences.
 *
 * cu_seqlens: DEVICE int32 [N+1], cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[N] = T; tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 form
 *   sequence n.  NULL means N equal sequences of T/N tokens (T % N must be
 *   0).  The device copy cannot be checked on the host without a sync; the
 *   kernels clamp every offset into [0, T] and treat a reversed range as an
 *   empty sequence, so a bad table never causes an out-of-bounds access.
 *   kda_check_cu_seqlens validates a host copy.
 * initial_state: [N, H, dk, dv] fp32 state each sequence starts from, or NULL
 *   for zeros (a prefix-cache hit passes the checkpointed state here).
 * final_state: [N, H, dk, dv] fp32 state after each sequence's last token,
 *   or NULL (not written).  It may alias initial_state.
 * out: [T, H, dv] in dtype, o_t for every token.
 * Errors: KDA_ERR_INVALID_ARG for a NULL shape, q, k, v, log_alpha, beta or
 *   out (when T > 0), negative sizes, N = 0 with T > 0, or T % N != 0 without
 *   cu_seqlens; KDA_ERR_UNSUPPORTED for an unsupported dtype, head size or
 *   alignment; KDA_ERR_CUDA if a launch fails.
 */
kda_status kda_prefill(const kda_shape* shape, const void* q, const void* k,
                       const void* v, const float* log_alpha, const void* beta,
                       const float* initial_state, const int32_t* cu_seqlens,
                       void* out, float* final_state, kda_stream_t stream);

/*
 * kda_prefill_checkpointed -- kda_prefill that also saves the state at chosen
 * points of each sequence, for the prefix-cache checkpoints that "Kimi K3
 * architecture: KDA, MLA and MoE" (section "Serving K3 means managing two
 * cache lifecycles") describes: KDA states kept only at reusable prefix
 * boundaries, from which a later request resumes prefill.
 *
 * All other arguments and layouts are those of kda_prefill.
 * ckpt_cu:     DEVICE int32 [N+1]; checkpoints ckpt_cu[n] .. ckpt_cu[n+1]-1
 *              belong to sequence n (ckpt_cu[0] = 0, non-decreasing).
 * ckpt_pos:    DEVICE int32 [ckpt_cu[N]]; for each checkpoint, the number of
 *              tokens of its sequence after which the state is saved: strictly
 *              increasing within a sequence, each a multiple of 64 or equal to
 *              the sequence length.  A position that breaks these rules is not
 *              written (kda_check_checkpoints validates a host copy).
 * ckpt_states: [ckpt_cu[N], H, dk, dv] fp32, caller-owned; checkpoint c of a
 *              sequence and head h lands at ckpt_states[c, h].
 * The saved state equals the final state of a kda_prefill over the same
 * prefix.  Errors: those of kda_prefill, plus KDA_ERR_INVALID_ARG for a NULL
 * checkpoint pointer and KDA_ERR_UNSUPPORTED for a misaligned one (ckpt_states
 * 16 bytes, the tables 4 bytes).
 */
kda_status kda_prefill_checkpointed(const kda_shape* shape, const void* q, const void* k,
                                    const void* v, const float* log_alpha, const void* beta,
                                    const float* initial_state, const int32_t* cu_seqlens,
                                    void* out, float* final_state, const int32_t* ckpt_cu,
                                    const int32_t* ckpt_pos, float* ckpt_states,
                                    kda_stream_t stream);

/*
 * kda_prefill_gated -- kda_prefill whose stored output is the KDA layer's
 * gated output instead of o: "Kimi K3 architecture: KDA, MLA and MoE"
 * (section "Scale: Total vs Active Parameters and Serving Economics",
 * Visual 1, the KDA inset) passes the KDA output through a norm and multiplies
 * it by a sigmoid gate.  Per token t and head h:
 *
 *   out[t, h, j] = o[t, h, j] / sqrt(mean_j' o[t, h, j']^2 + norm_eps)
 *                  * norm_weight[j] * sigmoid(gate[t, h, j])
 *
 * (an RMSNorm over the dv value channels with one weight per channel shared by
 * the heads -- the figure says only "a norm"; this is the reading).
 * gate:        [T, H, dv] in dtype, the gate logits, 16-byte aligned.
 * norm_weight: [dv] fp32.   norm_eps: finite and > 0 (an all-zero output row, which
 *              beta = 0 from a zero state produces, is then mapped to zero, not 0/0).
 * All other arguments are those of kda_prefill; final_state is unchanged by the
 * gate.  The gate is applied by a second, memory-bound pass over out on the same
 * stream (one read of o and of the gate, one write).
 * Errors: those of kda_prefill, plus KDA_ERR_INVALID_ARG for a NULL gate or
 *   weight or a bad eps and KDA_ERR_UNSUPPORTED for a misaligned gate.
 */
kda_status kda_prefill_gated(const kda_shape* shape, const void* q, const void* k,
                             const void* v, const float* log_alpha, const void* beta,
                             const float* initial_state, const int32_t* cu_seqlens,
                             const void* gate, const float* norm_weight, float norm_eps,
                             void* out, float* final_state, kda_stream_t stream);

/*
 * kda_prefill_split -- kda_prefill for inputs with few (sequence, head) pairs and
 * long sequences (the 1M-token contexts of "Kimi K3 Architecture Teardown", section
 * "Hybrid Attention for 1M Tokens").  kda_prefill runs each (sequence, head) on one
 * SM, so one sequence with 32 heads keeps 32 SMs busy whatever its length.  Here the
 * work that does not depend on the state entering a chunk (the decayed factors, the
 * Gram products, the UT solve and the WY factors W' and U) first runs for every chunk
 * of every head at once, leaving one record per chunk in `workspace`; a second kernel
 * per (sequence, head) then carries the state through the records in order.  A single
 * sequence of at least 16384 tokens (with at most 64 heads) runs in segments of 8192
 * tokens: the chunk records of segment s + 1 are built, on an internal second stream and
 * on the SMs the state chains leave free, while the chains of segment s run on `stream`;
 * the chains carry the fp32 state from segment to segment, so the results are those of
 * one pass.  The call's work on the second stream is ordered after `stream`'s earlier
 * work and before its later work; calls from several host threads serialise on it.
 *
 * All arguments but the workspace are those of kda_prefill, with the same results
 * (the same arithmetic in a different order of kernels; within the tolerances of the
 * tensor-core path).  workspace: DEVICE memory of at least
 * kda_prefill_split_workspace_size bytes, 256-byte aligned, owned by the caller,
 * overwritten by the call and free again once the call's work on `stream` is done;
 * two calls in flight at once need two workspaces.  For shapes the split kernels do
 * not take (anything but bf16 with dk = dv = 128) the call runs kda_prefill's kernels
 * and leaves the workspace untouched.
 * Errors: those of kda_prefill, plus KDA_ERR_INVALID_ARG for a NULL or too small
 * workspace and KDA_ERR_UNSUPPORTED for a misaligned one.
 */
kda_status kda_prefill_split(const kda_shape* shape, const void* q, const void* k, const void* v,
                             const float* log_alpha, const void* beta, const float* initial_state,
                             const int32_t* cu_seqlens, void* out, float* final_state, void* workspace,
                             size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_prefill_split_workspace_size -- bytes of workspace kda_prefill_split needs for
 * `shape`: H * (ceil(T / 64) + N) chunk records of 96 KB plus a 4-byte mode word each
 * (about 1.5 KB per token and head); for a single sequence run in segments (see
 * kda_prefill_split) the records of two segments, H * 129 each, plus two fp32 states per
 * head, whatever the length.  Depends on the shape only, not on the sequence lengths.
 * Writes *bytes; KDA_ERR_INVALID_ARG for a NULL pointer, otherwise the shape errors of
 * kda_prefill.  No CUDA call.
 */
kda_status kda_prefill_split_workspace_size(const kda_shape* shape, size_t* bytes);

/*
 * kda_prefill_split_static -- kda_prefill_split for callers that cannot allocate device
 * memory: the same two kernels and results, with the workspace in a fixed array that the
 * library itself owns (KDA_PREFILL_SPLIT_STATIC_BYTES, 64 MiB) instead of caller memory.
 * The pages have no counterpart of this entry point; it exists for code that runs where a
 * cudaMalloc is not allowed or not possible (inside another framework's memory pool, under
 * a fixed memory budget, without an allocator handle).  It allocates nothing.
 *
 * Arguments, layouts and results are those of kda_prefill_split without the workspace.
 * Limits: bf16 with dk = dv = 128 only, and the shape's workspace
 * (kda_prefill_split_workspace_size: 96 KB per chunk record, H * (ceil(T/64) + N) records)
 * must fit the array, about 680 records (e.g. 32 heads and up to 1,280 tokens in one
 * sequence); otherwise KDA_ERR_UNSUPPORTED and nothing is enqueued.
 * Every GPU that loads the library holds the array until the process exits.  All calls on
 * a device share it and it keeps the last call's contents; nothing in it needs to start at
 * zero.  Calls whose work overlaps on the GPU (two streams, or two host threads) race on
 * the array: order them on one stream or synchronise between them.  The first call on a
 * device looks up the array's device address with that device current (no allocation),
 * so make that first call before any stream capture.
 * Errors: those of kda_prefill_split (other than the workspace ones), KDA_ERR_UNSUPPORTED
 * for a shape beyond the limits above, KDA_ERR_CUDA if the address lookup or a launch fails.
 */
#define KDA_PREFILL_SPLIT_STATIC_BYTES (64u << 20)
kda_status kda_prefill_split_static(const kda_shape* shape, const void* q, const void* k, const void* v,
                                    const float* log_alpha, const void* beta, const float* initial_state,
                                    const int32_t* cu_seqlens, void* out, float* final_state,
                                    kda_stream_t stream);

/*
 * kda_check_checkpoints -- validate HOST copies of a cu_seqlens table and of a
 * checkpoint table against the rules of kda_prefill_checkpointed.  Returns
 * KDA_OK or KDA_ERR_INVALID_ARG.  No CUDA call.
 */
kda_status kda_check_checkpoints(const int32_t* host_cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, const int32_t* host_ckpt_cu,
                                 const int32_t* host_ckpt_pos);

/*
 * kda_decode_step -- a decode step of T tokens (1 <= T <= 16) for each of N
 * independent sequences, each starting from the state in state_inout.
 *
 * shape->num_seqs = N and shape->total_tokens = N * T.  q, k, log_alpha are
 * [N*T, H, dk], v and out [N*T, H, dv], beta [N*T, H]; rows n*T .. n*T+T-1 are
 * the tokens of sequence n in order (T = 1 is the ordinary one-token step).
 * state_inout [N, H, dk, dv] fp32 is read once and overwritten in place with
 * the state after the sequence's last token; out receives o_t = S_t^T q_t for
 * every token.  The state crosses HBM once in each direction whatever T is.
 * Errors: as kda_prefill; in addition KDA_ERR_INVALID_ARG if state_inout is
 * NULL or total_tokens is not a positive multiple of num_seqs (num_seqs = 0
 * with total_tokens = 0 is a no-op), KDA_ERR_UNSUPPORTED if T > 16 (use
 * kda_prefill with initial_state for longer runs).
 */
kda_status kda_decode_step(const kda_shape* shape, const void* q, const void* k,
                           const void* v, const float* log_alpha,
                           const void* beta, float* state_inout, void* out,
                           kda_stream_t stream);

/*
 * kda_frontend -- the steps of a KDA layer between its projections and the
 * recurrence, as "Kimi K3 architecture: KDA, MLA and MoE" (section "Scale:
 * Total vs Active Parameters and Serving Economics", Visual 1, the KDA inset)
 * draws them: q and k pass a short convolution, SiLU and an L2 norm; v a short
 * convolution and SiLU; the decay and beta a sigmoid.  Per sequence, token and
 * head (W = conv_width):
 *
 *   y[t, c]   = sum_{i<W} conv[h, c, i] * x_raw[t-(W-1)+i, h, c]   (0 before the
 *               sequence start: the convolution never reads another sequence)
 *   q         = SiLU(y_q) / sqrt(|SiLU(y_q)|^2 + eps)    (norm over dk)
 *   k         = SiLU(y_k) / sqrt(|SiLU(y_k)|^2 + eps)
 *   v         = SiLU(y_v)
 *   log_alpha = logsigmoid(a_raw),  beta = sigmoid(b_raw)
 *
 * The convolution width, its causal and depthwise form and eps are readings:
 * the figure names the steps only.  The projections are the caller's GEMMs.
 * shape:     as kda_prefill; q_raw, k_raw, v_raw, b_raw and the outputs q, k, v,
 *            beta are in shape->dtype; a_raw and log_alpha are fp32.
 * q_raw, k_raw, a_raw [T, H, dk]; v_raw [T, H, dv]; b_raw [T, H].
 * conv_q, conv_k [H, dk, W], conv_v [H, dv, W]: fp32 taps, tap W-1 on the current
 *            token; 1 <= W <= 4.
 * eps:       added to the sum of squares of the L2 norm, finite and > 0 (so an
 *            all-zero row normalises to zero instead of 0/0).
 * q, k, v, log_alpha, beta: written in kda_prefill's input layout; they must not
 *            overlap the raw inputs.
 * cu_seqlens: as kda_prefill (NULL: N equal sequences).
 * Errors: those of kda_prefill for the shape and the pointers, plus
 *   KDA_ERR_UNSUPPORTED for W outside 1..4 and KDA_ERR_INVALID_ARG for a bad eps
 *   or a NULL conv pointer.
 */
kda_status kda_frontend(const kda_shape* shape, int32_t conv_width, float eps,
                        const void* q_raw, const void* k_raw, const void* v_raw,
                        const float* a_raw, const void* b_raw, const float* conv_q,
                        const float* conv_k, const float* conv_v,
                        const int32_t* cu_seqlens, void* q, void* k, void* v,
                        float* log_alpha, void* beta, kda_stream_t stream);

/*
 * kda_prefill_frontend -- kda_frontend and kda_prefill in one pass: the prefill reads the
 * raw projections and runs the front end of Visual 1 ("Kimi K3 architecture: KDA, MLA
 * and MoE", section "Scale: Total vs Active Parameters and Serving Economics", the KDA
 * inset: short convolution, SiLU and L2 norm for q and k, convolution and SiLU for v,
 * sigmoid gates) on each chunk's tiles as they arrive, before the recurrence.  The
 * processed q, k, v, log_alpha and beta never go to memory.
 *
 * Arguments: the raw inputs, taps, conv_width and eps of kda_frontend (same layouts and
 * readings), and initial_state, cu_seqlens, out, final_state of kda_prefill.  out and
 * final_state are those kda_prefill gives on kda_frontend's outputs, within the bf16
 * tolerance (the front end's values are rounded to bf16 at the same points).
 * Supported: bf16 with dk = dv = 128 (otherwise KDA_ERR_UNSUPPORTED; run kda_frontend
 * and kda_prefill instead).
 * Errors: the shape and pointer errors of kda_prefill, and those of kda_frontend for
 * conv_width, eps and the taps.
 */
kda_status kda_prefill_frontend(const kda_shape* shape, int32_t conv_width, float eps, const void* q_raw,
                                const void* k_raw, const void* v_raw, const float* a_raw, const void* b_raw,
                                const float* conv_q, const float* conv_k, const float* conv_v,
                                const float* initial_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, kda_stream_t stream);

/*
 * kda_decode_step_gated -- kda_decode_step whose stored output is the gated
 * output of kda_prefill_gated (gate [N*T, H, dv] in dtype, norm_weight [dv]
 * fp32, norm_eps finite and > 0), fused into the step's output store.  The state update
 * is that of kda_decode_step.  Errors: those of kda_decode_step and of the gate
 * arguments of kda_prefill_gated.
 */
kda_status kda_decode_step_gated(const kda_shape* shape, const void* q, const void* k,
                                 const void* v, const float* log_alpha, const void* beta,
                                 const void* gate, const float* norm_weight, float norm_eps,
                                 float* state_inout, void* out, kda_stream_t stream);

/*
 * kda_check_cu_seqlens -- validate a HOST copy of a cu_seqlens table:
 * cu[0] == 0, non-decreasing, cu[num_seqs] == total_tokens.  Returns KDA_OK
 * or KDA_ERR_INVALID_ARG.  No CUDA call.
 */
kda_status kda_check_cu_seqlens(const int32_t* host_cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens);

/*
 * kda_selftest_timeout -- diagnostic for the timeout path.  Enqueues on
 * `stream` one single-thread kernel that waits, with the same bounded wait as
 * every kernel of the library, on a barrier that nothing completes; after
 * `limit_ns` nanoseconds (1e3 .. 1e9) the wait gives up and the kernel sets the
 * timeout bit of the status word, so the next kda_device_status returns
 * KDA_ERR_TIMEOUT.  No GPU fault, trap or hang is involved.  Returns KDA_OK
 * (enqueued), KDA_ERR_INVALID_ARG for a limit out of range (nothing enqueued)
 * or KDA_ERR_CUDA if the launch fails.
 */
kda_status kda_selftest_timeout(uint64_t limit_ns, kda_stream_t stream);

/*
 * kda_device_status -- synchronise `stream`, then read the device status word
 * and clear the bits that were read (an atomic clear on `stream`, so a bit set
 * meanwhile by a kernel on another stream survives for the next call).  The
 * word is one per device, shared by every stream and every call of the
 * library: a bit reports an event since it was last read, whichever stream's
 * kernel caused it.  Returns KDA_ERR_TIMEOUT if a kernel's bounded wait gave up
 * since the last call (that kernel's outputs are then undefined), KDA_ERR_BOUNDS
 * if, in a library built with -DKDA_CHECK_BOUNDS (a diagnostic build), a kernel
 * skipped a global-memory access whose index left its buffer, KDA_OK otherwise,
 * or KDA_ERR_CUDA if the synchronisation fails.  Setting the
 * environment variable KDA_DEBUG_SYNC=1 makes kda_prefill and kda_decode_step
 * call this themselves before returning.
 */
kda_status kda_device_status(kda_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* kda_status_string(kda_status status);

/* Library version string, e.g. "kda-gb300 0.1.0 sm_103a". */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
