/*
 * kda.h -- C ABI of the Kimi Delta Attention (KDA) library for one GB300
 * (sm_103a).
 *
 * The operation (per sequence n and head h, tokens t in order), from
 * "Kimi K3 Open Weights: What Is Actually New In Its 2.8 Trillion Parameter
 * Architecture", section 1 "Kimi Delta Attention is a real new kernel family":
 *
 *     g_t     = -5 * sigmoid(e^{A_h} * z_t)           (gate equation; per channel)
 *     alpha_t = e^{g_t}                                in [e^-5, 1]
 *     S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t     = S_t^T q_t                              (recurrence equation)
 *
 * with q_t, k_t L2-normalised inside the call ("Q/K normalization" in the
 * section's prefill bullet) when KDA_FLAG_L2NORM_QK is set:
 *     x_hat = x / sqrt(sum x^2 + 1e-6),   q_hat additionally times `scale`.
 * S is d_k x d_v per (sequence, head), kept in fp32.  Prefill processes tokens
 * "parallel within chunks, recurrent between"; decode advances one token with
 * the state persistent in device memory (same section, runtime split).
 *
 * Conventions shared by every call
 *   - Memory: every tensor pointer is a DEVICE pointer owned by the caller
 *     (the library allocates nothing).  Layouts are token-major and dense:
 *     x[token][head][channel].  States are [n][H][d_k][d_v] row-major fp32.
 *   - Alignment: q, k, v, z, o, states: 16-byte aligned; beta: element
 *     aligned; A, cu_seqlens, slots: 4-byte aligned.
 *   - Sizes: d_k, d_v in {32, 64, 128}; other values -> KDA_ERR_UNSUPPORTED.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  A call validates its arguments on
 *     the host, launches, and returns; host-detectable errors return a
 *     negative status and launch nothing.  A CUDA launch failure returns
 *     KDA_ERR_CUDA.  No exception or abort crosses this boundary.
 *   - Calls are re-entrant.  The library's only mutable global state is
 *     lazily resolved driver entry points and, for kda_prefill_noalloc, its
 *     fixed device array and the per-device cache of that array's address
 *     (see there).
 *   - A device cu_seqlens array is trusted only as far as the token range:
 *     kernels clamp every entry to [0, total_T] and end each sequence no
 *     earlier than it starts, so a malformed array (without the host mirror
 *     that would have caught it) gives meaningless results but never reads
 *     or writes outside the caller's buffers.
 *   - Input buffers must not alias output buffers unless stated.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad cu_seqlens mirror   */
    KDA_ERR_UNSUPPORTED = -2,  /* head dim or dtype outside the supported set      */
    KDA_ERR_ALIGNMENT = -3,    /* a pointer violates the alignment rule above       */
    KDA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required        */
    KDA_ERR_CUDA = -5,         /* a CUDA runtime/driver call failed                 */
    KDA_ERR_TIMEOUT = -6       /* a kernel gave up a bounded wait (see kda_workspace_status) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

enum {
    KDA_FLAG_L2NORM_QK = 1,    /* L2-normalise q and k inside the call (default on)  */
    KDA_FLAG_RECURRENT = 2,    /* kda_prefill only: run the fused recurrent kernel
                                  (fp32 arithmetic, one token at a time) even where
                                  the chunked tensor-core kernel applies */
    KDA_FLAG_SOFTPLUS_GATE = 4, /* Kimi Linear's unbounded gate g = -softplus(e^A z),
                                   alpha = e^g = sigmoid(-e^A z), in place of
                                   g = -5 sigmoid(e^A z) (section 1 names it as the
                                   decay K3 replaced).  Its decay has no lower bound,
                                   so the 16-token reciprocal tiles of the chunked
                                   kernels do not apply: prefill runs the fused
                                   recurrent kernel (fp32), decode is unchanged. */
    KDA_FLAG_CONV_SILU = 8,     /* kda_short_conv, kda_decode_step_conv: SiLU,
                                   y * sigmoid(y), after each short convolution */
    KDA_FLAG_SHORT_PEER_WAITS = 16 /* kda_prefill, test aid: the split kernel's
                                   waits on other CTAs give up after one poll,
                                   so that its bounded-wait exit runs; the call
                                   then reports KDA_ERR_TIMEOUT through
                                   kda_workspace_status and its outputs are
                                   invalid.  No effect on other kernels. */
};
#define KDA_DEFAULT_FLAGS KDA_FLAG_L2NORM_QK

/*
 * Bytes of device workspace that let kda_prefill pick its fastest kernel for
 * these sizes on the current device.  Always > 0 and a multiple of 256.
 *
 * Any workspace of at least 256 + 4 * N * H bytes (rounded up to 256) is
 * accepted.  With bf16 and d_k = d_v = 128 (up to 1024 sequences and 256
 * heads), a larger workspace -- the size returned here, a ring of 16 slots of
 * 66,048 bytes (about 1.06 MB) per consumer CTA, at most a quarter of the SMs
 * (about 40 MB on 152 SMs; 24 slots on up to a third of the SMs, about 80 MB,
 * where that halves the batches of units) whatever the sequence lengths --
 * selects the split kernel, which spreads each (sequence, head) pair's chunks over all SMs and
 * passes every chunk's operand tiles through the ring; a smaller one selects
 * the single-pass kernel.  The split kernel needs one CTA on every SM at once
 * and is launched cooperatively, which guarantees that; where the device
 * cannot take it (another context holds SMs, a partitioned GPU) the call runs
 * the single-pass kernel instead, with the same results.  The workspace is
 * scratch: its content on entry does not matter and it may be reused by the
 * next call on the same stream.
 */
KDA_API size_t kda_prefill_workspace_bytes(int32_t N, int32_t total_T, int32_t H,
                                   int32_t d_k, int32_t d_v, kda_dtype dt);

/*
 * kda_prefill -- chunked prefill over N packed sequences.
 *
 *  q, k, z        [total_T, H, d_k]  dt
 *  v              [total_T, H, d_v]  dt
 *  beta           [total_T, H]       dt, values in [0, 1]
 *  A              [H]                fp32, log-scale of the gate (e^A multiplies z)
 *  initial_state  [N, H, d_k, d_v]   fp32, or NULL for zeros
 *  cu_seqlens     [N + 1] int32 DEVICE array of sequence starts (0 = first,
 *                 total_T = last), or NULL for N equal sequences of total_T / N
 *                 (total_T % N must be 0).
 *  cu_seqlens_host  optional HOST mirror of cu_seqlens.  When given it is
 *                 validated (starts at 0, non-decreasing, ends at total_T)
 *                 and used to schedule long sequences first.
 *  scale          multiplies q_hat (1.0 = none)
 *  flags          KDA_FLAG_L2NORM_QK, KDA_FLAG_RECURRENT, KDA_FLAG_SOFTPLUS_GATE,
 *                 KDA_FLAG_SHORT_PEER_WAITS (or 0)
 *  o              [total_T, H, d_v]  dt, output (o_t for every token)
 *  final_state    [N, H, d_k, d_v] fp32, or NULL.  May alias initial_state
 *                 (in-place update is allowed).
 *  workspace      device scratch, 256-byte aligned; see kda_prefill_workspace_bytes()
 *
 * A zero-length sequence returns final_state = initial_state (or zeros).
 * bf16 with d_k = d_v = 128 runs a tcgen05/TMEM chunked kernel (single-pass,
 * or split when the workspace allows it; both give bit-identical results);
 * every other size/dtype runs the fused recurrent kernel (fp32 arithmetic).
 */
KDA_API int kda_prefill(const void* q, const void* k, const void* v, const void* z,
                const void* beta, const float* A, const float* initial_state,
                const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                kda_dtype dt, float scale, uint32_t flags,
                void* o, float* final_state,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_prefill_checkpointed -- kda_prefill that also saves the state at
 * chunk-aligned token boundaries: for sequence n and every m >= 1 with
 * m * ckpt_interval <= its length, the state after its first
 * m * ckpt_interval tokens.  This is what prefix reuse needs: a later request
 * that shares those first tokens can start its prefill or decode from that
 * state ("Kimi K3 Open Weights: What Is Actually New In Its 2.8 Trillion
 * Parameter Architecture", section "Why 104B active still understates the
 * systems problem": reuse is valid only where the prefix and the KDA state
 * checkpoint agree at the same token boundary).
 *
 *  ckpt_interval   tokens between checkpoints, a positive multiple of 64
 *  ckpt_pool       [ckpt_pool_size, H, d_k, d_v] fp32 state pool (the layout
 *                  kda_decode_step and kda_state_io use), 16-byte aligned,
 *                  not overlapping any other output
 *  ckpt_slots      device [n_checkpoints] int32: the pool row of each
 *                  checkpoint, or NULL for row = checkpoint index.  The
 *                  checkpoints of sequence n follow those of sequences
 *                  0 .. n-1 (see kda_checkpoint_count); checkpoint m of
 *                  sequence n has index (checkpoints before n) + m - 1.  Rows
 *                  outside [0, ckpt_pool_size) are skipped.  Checkpoints are
 *                  written (and ckpt_slots read) only below the count the host
 *                  can vouch for: kda_checkpoint_count of cu_seqlens_host, or
 *                  of the equal split without cu_seqlens, or -- with a device
 *                  cu_seqlens and no host mirror -- floor(total_T /
 *                  ckpt_interval), the largest count a valid array can give.
 *  ckpt_pool_size  rows in the pool (>= 1)
 * Every other argument and result is that of kda_prefill; ckpt_interval == 0
 * (with a NULL pool) is exactly kda_prefill.  Errors: KDA_ERR_INVALID_ARG for
 * an interval that is negative or not a multiple of 64, or a missing pool;
 * KDA_ERR_ALIGNMENT for a misaligned pool or slot array.
 */
KDA_API int kda_prefill_checkpointed(const void* q, const void* k, const void* v,
                const void* z, const void* beta, const float* A,
                const float* initial_state, const int32_t* cu_seqlens,
                const int32_t* cu_seqlens_host, int32_t N, int32_t total_T, int32_t H,
                int32_t d_k, int32_t d_v, kda_dtype dt, float scale, uint32_t flags,
                void* o, float* final_state, int32_t ckpt_interval, float* ckpt_pool,
                const int32_t* ckpt_slots, int32_t ckpt_pool_size,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_checkpoint_count -- how many checkpoints kda_prefill_checkpointed writes
 * (before slot mapping): the sum over sequences of floor(length /
 * ckpt_interval).  cu_seqlens_host: HOST array [N + 1] of sequence starts, or
 * NULL for N equal sequences of total_T / N.  Negative on invalid arguments.
 */
KDA_API int64_t kda_checkpoint_count(const int32_t* cu_seqlens_host, int32_t N,
                                     int32_t total_T, int32_t ckpt_interval);

/*
 * kda_workspace_status -- wait for `stream`, then read the status word a
 * kda_prefill launch left in `workspace`.  Returns KDA_OK, KDA_ERR_TIMEOUT
 * (a bounded wait inside the kernel ran out; its outputs are invalid) or
 * KDA_ERR_CUDA.  Synchronising; meant for tests and diagnostics.
 */
KDA_API int kda_workspace_status(const void* workspace, void* stream);

/*
 * kda_decode_step -- one token for each of B sequences, state updated in
 * place in a pool (section 1: "one recurrent-state update per layer and
 * token, with ... recurrent state kept persistent").
 *
 *  q, k, z        [B, H, d_k]  dt;   v [B, H, d_v] dt;   beta [B, H] dt
 *  A              [H] fp32
 *  state          [pool_size, H, d_k, d_v] fp32, read and written in place
 *  slots          [B] int32 device array: row b uses state[slots[b]]; NULL
 *                 means slots[b] = b (then pool_size >= B is required).
 *                 Slots must be distinct; a slot outside [0, pool_size)
 *                 leaves that state untouched and writes NaN to its o row.
 *  o              [B, H, d_v] dt
 */
KDA_API int kda_decode_step(const void* q, const void* k, const void* v, const void* z,
                    const void* beta, const float* A, float* state,
                    const int32_t* slots, int32_t pool_size,
                    int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                    kda_dtype dt, float scale, uint32_t flags,
                    void* o, void* stream);

/*
 * kda_short_conv -- the short convolutions of q, k and v that precede the KDA
 * step in prefill (section 1, prefill bullet: "short convolutions"; decode
 * bullet: the convolution state kept persistent; section "Why 104B active
 * still understates the systems problem": a fixed-size short-convolution
 * state per request and layer).  The pages give no formula; the library reads
 * it as a causal depthwise convolution along time of width W on every
 * channel,
 *     y_t[c] = sum_{j < W} w[c][j] * x_{t-W+1+j}[c],
 * then y * sigmoid(y) when KDA_FLAG_CONV_SILU is set.  Inputs before a
 * sequence's first token are rows of its conv state (zeros without one).
 * Feed q_out, k_out, v_out to kda_prefill; hand conv_state_out to
 * kda_decode_step_conv.
 *
 *  q, k            [total_T, H, d_k] dt;  v [total_T, H, d_v] dt
 *  conv_w          [H, 2 d_k + d_v, W] fp32: per head the taps of the q
 *                  channels, then k, then v; tap W-1 weights the current token
 *  conv_state_in   [N, H, W-1, 2 d_k + d_v] dt, or NULL for zeros: row r is
 *                  the input W-1-r tokens before the sequence's first one
 *  conv_state_out  same shape, or NULL: the last W-1 inputs of each sequence
 *                  (taken from conv_state_in where a sequence is shorter)
 *  cu_seqlens      as kda_prefill (device [N + 1], or NULL for equal lengths)
 *  W               1 .. 4;  flags: 0 or KDA_FLAG_CONV_SILU
 *  q_out, k_out, v_out   the convolved tensors, layouts of q, k, v, rounded
 *                  to dt (round to nearest even); the taps and sums in fp32,
 *                  the SiLU on the approximate exp2 and reciprocal (relative
 *                  error near 1e-7 before that rounding)
 * Buffers are device memory owned by the caller, 16-byte aligned (conv_w
 * too).  Errors (nothing is launched): KDA_ERR_INVALID_ARG for a missing
 * buffer, W outside 1 .. 4, an unknown flag, bad cu_seqlens_host, an output
 * overlapping an input or another output, or conv_state_out overlapping
 * conv_state_in; KDA_ERR_UNSUPPORTED / KDA_ERR_ALIGNMENT as kda_prefill.
 */
KDA_API int kda_short_conv(const void* q, const void* k, const void* v, const float* conv_w,
                           const void* conv_state_in, void* conv_state_out,
                           const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                           int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                           int32_t W, kda_dtype dt, uint32_t flags,
                           void* q_out, void* k_out, void* v_out, void* stream);

/*
 * kda_prefill_conv -- kda_short_conv followed by kda_prefill on its outputs,
 * in one call: the same o, final state and conv_state_out, bit for bit.
 *
 * With bf16, d_k = d_v = 128 and K3's gate, where the split kernel runs with
 * all (sequence, head) pairs in one batch (at most one pair per four SMs: 38
 * on 152 SMs), the convolutions are fused into it: its producers
 * convolve each chunk's q and k in shared memory before the Q/K
 * normalisation and its v into the chunk's operand tiles, with the same
 * arithmetic and rounding to bf16 as kda_short_conv, and the consumers write
 * each sequence's final conv state; the convolved tensors never go to HBM.
 * Otherwise (more pairs, whose producers have no slack for the extra work;
 * other dtypes or sizes; the softplus gate; KDA_FLAG_RECURRENT; a device
 * that cannot take the split kernel's cooperative launch) the call runs
 * kda_short_conv into the workspace and then kda_prefill.
 *
 *  q, k, v, z, beta, A, initial_state, cu_seqlens, cu_seqlens_host, N,
 *  total_T, H, d_k, d_v, dt, scale, o, final_state: as kda_prefill (q, k, v
 *                  the convolutions' inputs)
 *  flags           kda_prefill's flags, plus KDA_FLAG_CONV_SILU
 *  conv_w, conv_state_in, conv_state_out, W: as kda_short_conv
 *  workspace       kda_prefill_conv_workspace_bytes(...) bytes, 256-byte
 *                  aligned; it begins with the prefill's workspace, so
 *                  kda_workspace_status on it reports the split kernel's
 *                  bounded waits
 * Errors: as kda_prefill and kda_short_conv.
 */
KDA_API int kda_prefill_conv(const void* q, const void* k, const void* v, const void* z,
                             const void* beta, const float* A, const float* initial_state,
                             const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                             int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                             kda_dtype dt, float scale, uint32_t flags,
                             const float* conv_w, const void* conv_state_in,
                             void* conv_state_out, int32_t W, void* o, float* final_state,
                             void* workspace, size_t workspace_bytes, void* stream);

/* kda_prefill_conv_workspace_bytes -- the workspace kda_prefill_conv needs:
 * the prefill's (with the larger slots of the fused kernel, which also carry
 * the convolved v of each chunk) and room for the convolved q, k, v of the
 * two-pass path (0 for invalid sizes). */
KDA_API size_t kda_prefill_conv_workspace_bytes(int32_t N, int32_t total_T, int32_t H,
                                                int32_t d_k, int32_t d_v, kda_dtype dt);

/*
 * kda_decode_step_conv -- kda_decode_step preceded by the token's short
 * convolutions of q, k and v (as kda_short_conv, width W) with the conv
 * state kept persistent beside the recurrent state (section 1, decode
 * bullet).  Two launches on `stream`: a memory-bound pass convolves the
 * token of every row into `workspace` (rounded to dt, as kda_short_conv's
 * outputs) and shifts each row's conv state by the token in place; the
 * decode step then runs on the convolved q, k, v.
 *
 *  conv_w       [H, 2 d_k + d_v, W] fp32, as kda_short_conv (16-byte aligned)
 *  conv_state   [pool_size, H, W-1, 2 d_k + d_v] dt; row slots[b] (or b) is
 *               read and rewritten in place; may be NULL when W == 1
 *  W            1 .. 4
 *  flags        KDA_FLAG_L2NORM_QK, KDA_FLAG_SOFTPLUS_GATE, KDA_FLAG_CONV_SILU
 *  workspace    device scratch of kda_decode_conv_workspace_bytes(B, H, d_k,
 *               d_v, dt) bytes, 16-byte aligned, overlapping none of the
 *               other buffers; its contents need no initialisation
 * Every other argument is that of kda_decode_step; a slot outside
 * [0, pool_size) leaves both of its states untouched and writes NaN to its
 * o row.  Errors as kda_decode_step, plus KDA_ERR_WORKSPACE for a missing or
 * short workspace and KDA_ERR_UNSUPPORTED for B > 65535.
 */
KDA_API int kda_decode_step_conv(const void* q, const void* k, const void* v, const void* z,
                                 const void* beta, const float* A, float* state,
                                 const int32_t* slots, int32_t pool_size,
                                 const float* conv_w, void* conv_state, int32_t W,
                                 int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dt, float scale, uint32_t flags,
                                 void* o, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* kda_decode_conv_workspace_bytes -- the scratch kda_decode_step_conv needs:
 * the convolved q, k, v of one token per row (0 for negative sizes). */
KDA_API size_t kda_decode_conv_workspace_bytes(int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                                               kda_dtype dt);

/*
 * kda_backward -- gradients of the KDA recurrence for training: given
 * dL/do for every token and dL/dS_T (optional), the gradients of L with
 * respect to q, k, v, z, beta, A and the initial state, through the
 * delta-rule step, the gate (K3's or, with KDA_FLAG_SOFTPLUS_GATE, Kimi
 * Linear's) and the Q/K normalisation (section 1 of the K3 architecture
 * page gives the forward step; the backward is its reverse mode).
 *
 * Two forms, both launched by this call on `stream`:
 *  - chunked, on the tensor cores: bf16 inputs, d_k = d_v = 128, K3's gate,
 *    and sequence lengths the host can vouch for (cu_seqlens_host given, or
 *    no cu_seqlens), when the split prefill can run.  That prefill keeps a
 *    record of every 64-token chunk (its operand tiles and start state); a
 *    reverse chain then carries dL/dS through the chunks of each (sequence,
 *    head), last to first, and one CTA per (chunk, head) forms every
 *    gradient of its tokens (the chunk's adjoint products on the tensor
 *    core, the decay chains in fp32 on the CUDA cores).  bf16 operands, fp32
 *    accumulation: the bf16 accuracy of the forward.
 *  - recurrent, fp32 arithmetic, d_v / 32 CTAs per (sequence, head), for
 *    every other case: the states at every 64-token chunk start come from the
 *    checkpointed forward prefill; the chunks are walked last to first, each
 *    recomputed forward in fp32 into a scratch and its tokens walked in
 *    reverse; a second kernel adds the per-CTA column sums and applies the
 *    gate and normalisation derivatives.
 * Both are deterministic (no atomics in any sum).
 *
 *  q, k, v, z, beta, A, initial_state, cu_seqlens, cu_seqlens_host, N,
 *  total_T, H, d_k, d_v, dt, scale: as kda_prefill (the forward's inputs)
 *  flags       KDA_FLAG_L2NORM_QK, KDA_FLAG_SOFTPLUS_GATE (as the forward)
 *  dO          [total_T, H, d_v] dt: dL/do
 *  dS_final    [N, H, d_k, d_v] fp32 or NULL (zero): dL/dS_T
 *  dq, dk, dz  [total_T, H, d_k] fp32;  dv [total_T, H, d_v] fp32;
 *  dbeta       [total_T, H] fp32;  dA [H] fp32;  dS0 [N, H, d_k, d_v] fp32
 *              (written, not accumulated; dS0 is written also when
 *              initial_state is NULL)
 *  workspace   kda_backward_workspace_bytes(N, total_T, H, d_k, d_v, dt) bytes,
 *              256-byte aligned, no initialisation needed; it begins with the
 *              forward prefill's workspace, so kda_workspace_status on it
 *              reports that prefill's bounded waits
 * Errors: as kda_prefill (KDA_ERR_WORKSPACE for a short workspace), and
 * KDA_ERR_INVALID_ARG for a missing gradient buffer.
 */
KDA_API int kda_backward(const void* q, const void* k, const void* v, const void* z,
                         const void* beta, const float* A, const float* initial_state,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                         kda_dtype dt, float scale, uint32_t flags,
                         const void* dO, const float* dS_final,
                         float* dq, float* dk, float* dv, float* dz, float* dbeta, float* dA,
                         float* dS0, void* workspace, size_t workspace_bytes, void* stream);

/* kda_backward_workspace_bytes -- the workspace kda_backward needs, for
 * either form: the forward prefill's workspace and outputs, the chunk-start
 * states, then the larger of the recurrent form's scratch (64 states per
 * (sequence, head) and the column partials) and the chunked form's chunk
 * records (132 KB per chunk and head, at most total_T / 64 + N chunks) and
 * dL/dS tiles (32 KB each), and the per-token dA shares (0 for invalid
 * sizes). */
KDA_API size_t kda_backward_workspace_bytes(int32_t N, int32_t total_T, int32_t H, int32_t d_k,
                                            int32_t d_v, kda_dtype dt);

/*
 * kda_state_io -- moves fp32 states of shape [H, d_k, d_v] each (the
 * persistent KDA state that prefill hands to decode).
 *
 *  KDA_STATE_ZERO     dst[i] = 0 for i < n, or dst[slots[i]] = 0 when slots
 *                     is given (then dst is a pool of pool_size states).
 *  KDA_STATE_COPY     dst[0..n) = src[0..n); any direction (host or device
 *                     pointers, cudaMemcpyDefault).  slots must be NULL.
 *  KDA_STATE_GATHER   dst[i] = src[slots[i]]   (pool -> batch), i < n
 *  KDA_STATE_SCATTER  dst[slots[i]] = src[i]   (batch -> pool), i < n
 * A slot outside [0, pool_size) skips its state, except in GATHER, which
 * fills dst[i] with NaN for it (as kda_decode_step writes NaN to the o row of
 * such a slot), so that a bad slot cannot hand a stale state to decode
 * unnoticed.  For GATHER/SCATTER/ZERO the pointers are device pointers.
 */
typedef enum {
    KDA_STATE_ZERO = 0,
    KDA_STATE_COPY = 1,
    KDA_STATE_GATHER = 2,
    KDA_STATE_SCATTER = 3
} kda_state_op;

KDA_API int kda_state_io(kda_state_op op, float* dst, const float* src,
                 const int32_t* slots, int32_t n, int32_t pool_size,
                 int32_t H, int32_t d_k, int32_t d_v, void* stream);

/*
 * kda_prefill_noalloc -- kda_prefill without a caller-provided workspace.
 *
 * The pages have no counterpart to this call.  It exists for callers that
 * are not allowed to allocate device memory themselves -- for example a
 * plugin inside a host framework that owns all device memory and passes the
 * plugin only its inputs and outputs, or a latency-critical loop that must
 * not call into the CUDA allocator after start-up.  It allocates nothing:
 * the workspace kda_prefill needs comes from a fixed array of
 * 256 + 16384 * 4 bytes in the library's own device memory, held by every
 * GPU that loads the library until the process exits.
 *
 * Arguments, layouts and results are those of kda_prefill, which it calls
 * with the array as its workspace (so bf16 d=128 runs the single-pass
 * kernel).  More than 16384 (sequence, head) pairs return KDA_ERR_WORKSPACE
 * without launching.  The first call in a device's CUDA context looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and caches it with the context's unique id, so make that first call -- and
 * the first call after a cudaDeviceReset -- before any stream capture.
 * Every call shares the one array: calls that overlap on the GPU (other
 * streams, other threads) race on it.  The status word in the array is
 * cleared by each call; read it with kda_prefill_noalloc_status.
 */
KDA_API int kda_prefill_noalloc(const void* q, const void* k, const void* v, const void* z,
                                const void* beta, const float* A, const float* initial_state,
                                const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                                kda_dtype dt, float scale, uint32_t flags,
                                void* o, float* final_state, void* stream);

/*
 * kda_prefill_noalloc_status -- wait for `stream`, then read the status word
 * the last kda_prefill_noalloc call on the current device left in the fixed
 * array: KDA_OK, KDA_ERR_TIMEOUT (a bounded wait inside the kernel ran out;
 * that call's outputs are invalid) or KDA_ERR_CUDA.  The counterpart of
 * kda_workspace_status for callers that never see a workspace pointer.
 * Synchronising; allocates nothing.  No counterpart on the pages.
 */
KDA_API int kda_prefill_noalloc_status(void* stream);

/* Human-readable name of a kda_status value (static storage). */
KDA_API const char* kda_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
