/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention operator.
 *
 * The operator is the per-head gated delta-rule recurrence
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,            alpha_t = exp(g_t)  (one factor per key channel)
 *
 * from "Understanding Kimi K3's Attention" (state-update and readout
 * equations, symbol table) and "Kimi K3.1 and the Road From Softmax Attention
 * to Kimi Delta Attention" (section "5. Kimi Delta Attention").  The readout
 * uses the state after the token's own write ("Kimi K3 course, lesson 2";
 * "Inside Kimi K3", section "Sequence mixing": the intra-chunk causal matrix
 * includes the diagonal).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensors are row-major and contiguous, in DEVICE memory, owned by
 *    the caller.  The library allocates no device memory, with two
 *    exceptions: the KDA_PREFILL_TC_SPLIT prefill variant (its ring of chunk
 *    operands, about 0.28 MB per (sequence, head) it runs at once, at most
 *    27 MB) and the KDA_PREFILL_TC_2PASS variant (8 KB per chunk and head)
 *    take stream-ordered scratch from a memory pool of the library's own, and
 *    return it on the same stream when the call's work is done.
 *  - q, k  [T_tot, H, d_k];  v, out [T_tot, H, d_v];  g [T_tot, H, d_k] fp32
 *    (log-decay); beta [T_tot, H] fp32; states [N, H, d_k, d_v] fp32 with row
 *    i = key channel i (the decay scales rows: "Hybrid Attention", section
 *    "Forgetting can be selective, too").
 *  - No scaling, normalisation or gating is applied: q and k arrive already
 *    L2-normalised, the 1/sqrt(d) readout scale and the output gate belong to
 *    the caller ("Understanding Kimi K3's Attention", symbol table and output
 *    equation).
 *  - Preconditions that are documented but not checked on the device (they
 *    would need a read of device memory): g in [-5, 0] (the log-decay bound
 *    g_t = g_min Sigmoid(e^A z_t), g_min = -5) and beta in [0, 1].  Inputs
 *    outside them give finite but unspecified results; they never fault.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  KDA_OK means "enqueued".  Arguments are validated on
 *    the host before anything is launched; an error return launches nothing.
 *  - Supported head sizes: d_k == d_v, either 64 or 128.  Anything else
 *    returns KDA_ERR_UNSUPPORTED.
 */
#ifndef KDA_H
#define KDA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, bad dtype */
    KDA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (head size, dtype combo) */
    KDA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
    KDA_ERR_TIMEOUT = 4           /* a bounded device-side wait gave up */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/* Prefill kernel selection: a diagnostic and test selector, not a tuning
 * knob.  KDA_PREFILL_DEFAULT (what callers should pass) picks TC where it
 * supports the call, else FP32.  TC_SPLIT and TC_2PASS run only when named
 * (both are slower than TC on the 96-head layer).  The tensor-core kernels
 * take d_k = d_v = 128, bf16 q/k/v, and q, k, v, g (or z) and out 16-byte
 * aligned; TC_SPLIT also needs a device that supports cooperative launches.
 * TC_2PASS takes 8 KB of stream-ordered scratch per chunk and head (about
 * 0.2 GB for a 96-head, 8192-token layer) from a pool of the library's own.
 * Naming a variant that does not support the call returns
 * KDA_ERR_UNSUPPORTED. */
typedef enum {
    KDA_PREFILL_DEFAULT = 0,
    KDA_PREFILL_FP32 = 1,     /* CUDA-core fp32 chunked kernel (any supported shape) */
    KDA_PREFILL_TC = 2,       /* tcgen05 kernel, one CTA per (sequence, head) (d = 128) */
    KDA_PREFILL_TC_SPLIT = 3, /* tcgen05 kernel with the state recurrence and the intra-chunk
                                 work on different SMs, one cooperative launch (d = 128) */
    KDA_PREFILL_TC_2PASS = 4  /* tcgen05, two launches: the intra-chunk products of every
                                 chunk on every SM, then the state recurrence (d = 128) */
} kda_prefill_variant;

typedef void *kda_stream_t; /* a cudaStream_t */

typedef struct {
    int32_t num_seqs;     /* N >= 0 */
    int32_t total_tokens; /* T_tot >= 0 (decode: must equal num_seqs) */
    int32_t num_heads;    /* H >= 1 */
    int32_t d_k;          /* key/query head size */
    int32_t d_v;          /* value head size */
    int32_t in_dtype;     /* kda_dtype of q, k, v */
    int32_t out_dtype;    /* kda_dtype of out */
    int32_t variant;      /* kda_prefill_variant (ignored by decode) */
} kda_dims;

/*
 * kda_prefill -- chunk-parallel prefill over a packed variable-length batch.
 *
 * Evaluates the recurrence for every sequence n and head h over tokens
 * [cu_seqlens[n], cu_seqlens[n+1]), starting from init_state[n,h] (zeros if
 * init_state is NULL), writes o_t for every token into `out` and, if
 * final_state is non-NULL, the state after the last token of each sequence.
 * Tokens inside a chunk are evaluated together and the state is carried
 * from chunk to chunk ("Inside Kimi K3", section "Sequence mixing";
 * "Hybrid Attention", section "But isn't a recurrent update sequential?");
 * the result equals the token-by-token recurrence up to rounding, for any
 * sequence length (no divisibility requirement).
 *
 *   q, k, v     device, in_dtype, layouts above.
 *   g, beta     device, fp32.
 *   init_state  device fp32 [N, H, d_k, d_v] or NULL.
 *   cu_seqlens  device int32 [N+1] or NULL.  If NULL, T_tot must be a
 *               multiple of N and sequence n covers [n T, (n+1) T) with
 *               T = T_tot / N.  Otherwise cu[0] = 0, non-decreasing,
 *               cu[N] = T_tot; entries outside [0, T_tot] are clamped on the
 *               device and a decreasing pair is read as an empty sequence, so
 *               a malformed array can never cause an out-of-bounds access.
 *               An empty sequence copies init_state (or zeros) to final_state.
 *   out         device, out_dtype [T_tot, H, d_v].
 *   final_state device fp32 [N, H, d_k, d_v] or NULL.  May alias init_state
 *               exactly (each slice is read before it is written).
 *
 * No output (out, final_state, and the checkpoints of the calls below) may
 * share a byte with an input or with another output, except final_state ==
 * init_state: the kernels read later chunks' inputs while they write earlier
 * outputs.  KDA_ERR_INVALID_ARGUMENT if one does.
 *
 * Accumulation is fp32; a bf16 `out` is the round-to-nearest-even of the
 * value an fp32 `out` would hold.
 */
kda_status kda_prefill(const kda_dims *dims, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const float *init_state,
                       const int32_t *cu_seqlens, void *out, float *final_state,
                       kda_stream_t stream);

/*
 * kda_prefill_noalloc -- kda_prefill that allocates nothing.
 *
 * The pages have no counterpart of this call: it is an interface addition for
 * callers that may not allocate device memory during a call -- hosts whose own
 * caching allocator owns all of the GPU's memory from start-up (an allocation
 * outside it can fail or fragment it) and latency-bound services that keep
 * allocation off their serving path.
 *
 * Same arguments, layouts, semantics and errors as kda_prefill; dims->variant
 * is ignored.  It always runs the KDA_PREFILL_TC_SPLIT kernel, with that
 * kernel's scratch (ring of chunk operands, hand-off words, step table) in a
 * fixed array of the library (about 5 MB, which every device that loads the
 * library keeps until the process exits) instead of pool memory.  That array
 * limits a call to at most 16 chains of at most 4096 (sequence, head) pairs
 * each and at most 65536 sequences; a batch beyond that, or one the split
 * kernel does not take (d_k = d_v != 128, fp32 inputs, q/k/v/g/out not
 * 16-byte aligned, a device without cooperative launches), returns
 * KDA_ERR_UNSUPPORTED and launches nothing.
 *
 * The first call on a device looks up the device address of the array
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture on the device.  Every call shares the one array
 * and clears the parts that must start at zero itself; calls that overlap on
 * the GPU (on different streams or from different host threads) race on it
 * and must be serialised by the caller.
 */
kda_status kda_prefill_noalloc(const kda_dims *dims, const void *q, const void *k, const void *v,
                               const float *g, const float *beta, const float *init_state,
                               const int32_t *cu_seqlens, void *out, float *final_state,
                               kda_stream_t stream);

/* Chunk length of the prefill kernels; checkpoint intervals are multiples of it. */
#define KDA_CHUNK 32

/*
 * kda_prefill_checkpointed -- kda_prefill that also writes state checkpoints.
 *
 * Prefix reuse restores the recurrent state at a token boundary from sparse
 * state checkpoints ("Inside Kimi K3", section "Sequence mixing: fixed-state
 * KDA alongside global MLA").  Besides everything kda_prefill does, this call
 * writes the state of every sequence after each `interval` tokens:
 * checkpoint j (j = 1 .. floor(len_n / interval)) of sequence n is the state
 * after its first j * interval tokens, i.e. the final_state a prefill over
 * that prefix alone would return.
 *
 *   checkpoints device fp32 [capacity, H, d_k, d_v], 4-byte aligned.  Sequence n
 *               uses rows base_n .. base_n + floor(len_n / interval) - 1 with
 *               base_n = sum over m < n of floor(len_m / interval).  Rows at
 *               or beyond `capacity` are not written; checkpoints may be NULL
 *               only with capacity 0 (then this is kda_prefill).
 *   interval    tokens between checkpoints: a positive multiple of KDA_CHUNK.
 *   capacity    number of rows the caller allocated (>= 0).
 *
 * Every other argument, and every other error, is as in kda_prefill;
 * KDA_ERR_INVALID_ARGUMENT if interval is not a positive multiple of
 * KDA_CHUNK, capacity < 0, or checkpoints is NULL or misaligned while
 * capacity > 0.  The checkpoint stores add 4 d_k d_v bytes per checkpoint
 * and head to the prefill's traffic.
 */
kda_status kda_prefill_checkpointed(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, float *checkpoints,
                                    int64_t interval, int64_t capacity, kda_stream_t stream);

/*
 * kda_prefill_gated -- kda_prefill with the gate prologue fused into the load
 * stage: the call takes the decay logits and the write-strength logits and
 * forms, per token t, head h and key channel c,
 *
 *   g[t,h,c] = g_min Sigmoid(e^{A_h} z[t,h,c]),  g_min = -5,
 *   beta[t,h] = Sigmoid(beta_logit[t,h])
 *
 * ("Understanding Kimi K3's Attention": the log-decay bound equation, and the
 * symbol table for z_t, A_h and beta_t), then evaluates the same recurrence
 * as kda_prefill.  g never goes through memory; z costs 2 bytes per channel
 * in bf16 where g costs 4.
 *
 *   z           device, in_dtype, [T_tot, H, d_k]: the decay logits (an input:
 *               must not overlap `out`).
 *   a_log       device fp32 [H]: the per-head log-scales A_h.
 *   beta_logit  device fp32 [T_tot, H].
 *
 * Every other argument, and every other error, is as in kda_prefill;
 * KDA_ERR_INVALID_ARGUMENT if there are tokens and z or a_log is NULL.
 */
kda_status kda_prefill_gated(const kda_dims *dims, const void *q, const void *k, const void *v,
                             const void *z, const float *a_log, const float *beta_logit,
                             const float *init_state, const int32_t *cu_seqlens, void *out,
                             float *final_state, kda_stream_t stream);

/*
 * kda_prefill_output_gated -- kda_prefill followed by the layer's output gate,
 * fused into the store of the output where the kernel allows:
 *
 *   y[t,h,j] = Sigmoid(gate_logit[t,h,j]) * o~[t,h,j] / sqrt(ms + eps) * w[j],
 *   ms = (1/d_v) sum_j o~[t,h,j]^2
 *
 * with o~ the ungated readout that kda_prefill would write.  The pages give
 * the layer output as W_o [Sigmoid(W_g x_t) . RMSNorm(o~_t)] ("Inside Kimi
 * K3", section "Sequence mixing: fixed-state KDA alongside global MLA"); this
 * call forms the bracket.  The pages do not define the norm further; here it
 * is the root-mean-square over one head's d_v channels with eps inside the
 * root and an optional per-channel weight.  The projections W_g, W_o stay
 * with the caller.
 *
 *   gate_logit  device, in_dtype, [T_tot, H, d_v]: W_g x_t per head (an input:
 *               must not overlap `out`).
 *   norm_weight device fp32 [d_v], 4-byte aligned, or NULL (weight 1).
 *   eps         finite, > 0.
 *
 * The tensor-core kernel applies the gate before its store when out is bf16
 * and gate_logit is 16-byte aligned; otherwise the prefill writes o~ and a
 * second kernel gates `out` in place (with a bf16 `out`, o~ is then rounded
 * to bf16 once before the norm).  Every other argument, and every other
 * error, is as in kda_prefill; KDA_ERR_INVALID_ARGUMENT if there are tokens
 * and gate_logit is NULL or equals out, or eps is not a positive finite
 * number, or norm_weight is misaligned.
 */
kda_status kda_prefill_output_gated(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const void *gate_logit, const float *norm_weight, float eps,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, kda_stream_t stream);

/*
 * kda_output_gate -- the output gate alone, in place: for every row (token t,
 * head h) of `out`,
 *
 *   out[t,h,j] <- Sigmoid(gate_logit[t,h,j]) * out[t,h,j] / sqrt(ms + eps) * w[j],
 *   ms = (1/d_v) sum_j out[t,h,j]^2,
 *
 * the same gate as kda_prefill_output_gated, for outputs that another call
 * wrote: kda_prefill_gated's, or kda_decode's (dims->total_tokens rows).
 *
 *   out          device, out_dtype, [T_tot, H, d_v], read and overwritten.
 *   gate_logit   device, in_dtype, [T_tot, H, d_v]; must not overlap out.
 *   norm_weight  device fp32 [d_v], 4-byte aligned, or NULL (weight 1).
 *   eps          finite, > 0.
 *
 * dims->num_seqs and dims->variant are not used; d_k must equal d_v as
 * everywhere.  KDA_ERR_INVALID_ARGUMENT for a bad dims, a NULL or misaligned
 * pointer while there are rows, out overlapping gate_logit or norm_weight,
 * or a bad eps.
 */
kda_status kda_output_gate(const kda_dims *dims, void *out, const void *gate_logit,
                           const float *norm_weight, float eps, kda_stream_t stream);

/*
 * kda_qkv_prologue -- q, k and v from their projections: for every stream
 * (q, k, v), token t, head h and channel j,
 *
 *   c[t,h,j] = sum_{i=0..3} w[s,h,j,3-i] * x_s[t-i,h,j]
 *   y        = c * Sigmoid(c)                                  (Swish)
 *   q, k     = y / sqrt(sum_j y[t,h,j]^2 + eps)                 v = y
 *
 * The pages define q, k = L2Norm(Swish(ShortConv(W x))) and v =
 * Swish(ShortConv(W_v x)) ("Understanding Kimi K3's Attention", symbol
 * table), with a convolution of width 4 ("Inside Kimi K3", section "Sequence
 * mixing: fixed-state KDA alongside global MLA") that is causal ("Hybrid
 * Attention", section "KDA: don't write the same information twice").
 * Here it is a per-channel convolution over the tokens of one sequence, with
 * no bias, and L2Norm is taken over one head's d channels with eps inside
 * the root.  The projections W x stay with the caller.
 *
 *   dims        num_seqs N, total_tokens T, num_heads H, d_k = d_v = d (64 or
 *               128); in_dtype is the type of x_*, out_dtype that of q, k, v;
 *               variant is not used.
 *   x_q, x_k, x_v  device, in_dtype, [T, H, d]: the projections.
 *   conv_weight device fp32 [3, H, d, 4], 16-byte aligned: streams q, k, v;
 *               tap 3 multiplies the current token, tap 3-i the token i places
 *               earlier.
 *   conv_state_in  device fp32 [N, 3, 3, H, d] or NULL (zeros): for each
 *               sequence and stream, the three inputs before its first token,
 *               entry 0 the oldest.  Aligned to d/32 floats.
 *   cu_seqlens  device int32 [N+1] as in kda_prefill, or NULL (N equal
 *               sequences).  The convolution restarts at every sequence start.
 *               With N = 0 the call does nothing and returns KDA_OK.
 *   q, k, v     device, out_dtype, [T, H, d]: written.
 *   conv_state_out device fp32 [N, 3, 3, H, d] or NULL: the last three inputs
 *               of each sequence, entry 0 the oldest (taken from
 *               conv_state_in, or 0, where a sequence is shorter than three).
 *               This is the conv_state_in of the next segment: a decode step
 *               is a call with one token per sequence.
 *   eps         finite, > 0.
 *
 * x_* and q, k, v must be aligned to d/32 elements.  No output may overlap an
 * input or another output (the two conv states included); alternate two state
 * buffers between calls.  KDA_ERR_INVALID_ARGUMENT for a bad dims, a bad eps,
 * a NULL or misaligned pointer that is needed, or an overlap;
 * KDA_ERR_UNSUPPORTED for d other than 64 or 128, or sizes beyond one grid.
 */
kda_status kda_qkv_prologue(const kda_dims *dims, const void *x_q, const void *x_k,
                            const void *x_v, const float *conv_weight,
                            const float *conv_state_in, const int32_t *cu_seqlens, void *q,
                            void *k, void *v, float *conv_state_out, float eps,
                            kda_stream_t stream);

/*
 * kda_prefill_scalar_decay -- the same chunked prefill for the two special
 * cases of the recurrence the pages build KDA from ("Kimi K3.1 and the Road
 * From Softmax Attention to Kimi Delta Attention", sections "3. The delta
 * rule" and "4. Gating"):
 *
 *   Gated DeltaNet: S_t = (I - beta_t k_t k_t^T) alpha_t S_{t-1} + beta_t k_t v_t^T
 *                   with one decay alpha_t = exp(g_head[t,h]) per head and step;
 *   delta rule:     g_head == NULL, alpha_t = 1.
 *
 * A scalar decay is the channel-wise decay with one value repeated over the
 * key channels, so the result equals kda_prefill with g[t,h,c] = g_head[t,h]
 * (the kernels form the same running sums from it, and the same output).
 * The per-channel decay tensor is not read: 4 bytes per (token, head)
 * replace 4 d_k.
 *
 *   g_head  device fp32 [T_tot, H], 4-byte aligned, values in [-5, 0]; or
 *           NULL (no decay).
 *
 * Every other argument, and every other error, is as in kda_prefill.
 */
kda_status kda_prefill_scalar_decay(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g_head, const float *beta,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, kda_stream_t stream);

/*
 * kda_backward -- gradients of kda_prefill.  Given the upstream gradients
 * d_out = dL/d out and d_final_state = dL/d final_state (NULL => 0), writes
 * dL/dq, dL/dk, dL/dv, dL/dg, dL/dbeta and dL/d init_state for the same packed
 * batch.  The pages train the chunked computation and check its gradients
 * against the recurrent version ("Hybrid Attention", section "But isn't a
 * recurrent update sequential?"); this call computes them chunk by chunk,
 * walking each sequence's chunks in reverse and carrying the adjoint of the
 * state, from the forward's state at the start of every chunk.
 *
 *   chunk_states   device fp32 [chunk_capacity, H, d_k, d_v]: the checkpoints
 *                  kda_prefill_checkpointed writes with interval = KDA_CHUNK
 *                  for the same inputs (row layout as there).  It may be NULL
 *                  only if T_tot <= KDA_CHUNK (then no sequence has a second
 *                  chunk).  Rows at or past chunk_capacity are never read.  With
 *                  cu_seqlens NULL a capacity below the rows the batch needs
 *                  returns KDA_ERR_INVALID_ARGUMENT; with cu_seqlens (lengths
 *                  known only on the device) a needed row past the capacity is
 *                  recorded in the device status word, which
 *                  kda_get_last_device_error then reports as
 *                  KDA_ERR_INVALID_ARGUMENT (those gradients are not valid).
 *   d_out          device, in_dtype, [T_tot, H, d_v].
 *   d_final_state  device fp32 [N, H, d_k, d_v] or NULL.
 *   dq, dk, dv     device, out_dtype: [T_tot, H, d_k], [T_tot, H, d_k], [T_tot, H, d_v].
 *   dg             device fp32 [T_tot, H, d_k];  dbeta  device fp32 [T_tot, H].
 *   d_init_state   device fp32 [N, H, d_k, d_v] or NULL (not written).
 *
 * No gradient may share a byte with an input or with another gradient.
 * Arithmetic: with bf16 inputs at d_k = d_v = 128 (16-byte aligned q, k, v, g
 * and d_out) the products run on the tensor cores with tf32 operands and fp32
 * accumulation; otherwise (fp32 inputs, d = 64) everything is fp32 on the CUDA
 * cores.
 * Every other argument (q, k, v, g, beta, init_state, cu_seqlens, dims) and
 * every other error is as in kda_prefill; KDA_ERR_INVALID_ARGUMENT also if
 * chunk_capacity < 0, chunk_states is NULL or misaligned where it is needed,
 * or a gradient overlaps an input or another gradient.
 */
kda_status kda_backward(const kda_dims *dims, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const float *init_state,
                        const int32_t *cu_seqlens, const float *chunk_states,
                        int64_t chunk_capacity, const void *d_out, const float *d_final_state,
                        void *dq, void *dk, void *dv, float *dg, float *dbeta,
                        float *d_init_state, kda_stream_t stream);

/*
 * kda_decode -- one single-token update of N independent fixed-size states.
 *
 * For each sequence n and head h: M = Diag(exp g) S, u = beta (v - M^T k),
 * S <- M + k u^T (in place), o = S^T q -- the delta form of the recurrence
 * ("Understanding Kimi K3's Attention", rewritten update; "Hybrid
 * Attention", recurrent implementation).  Each fp32 state is read once and
 * written once.
 *
 *   dims        total_tokens must equal num_seqs (one token per sequence).
 *   q, k, v     device, in_dtype, [N, H, d]; g device fp32 [N, H, d_k];
 *               beta device fp32 [N, H].
 *   state_inout device fp32 [N, H, d_k, d_v], updated in place.
 *   out         device, out_dtype [N, H, d_v].
 *
 * Neither out nor the state may share a byte with an input or with each
 * other (KDA_ERR_INVALID_ARGUMENT).
 */
kda_status kda_decode(const kda_dims *dims, const void *q, const void *k, const void *v,
                      const float *g, const float *beta, float *state_inout, void *out,
                      kda_stream_t stream);

/*
 * kda_get_last_device_error -- report, then clear, the device-side status.
 *
 * The tensor-core prefill kernels wait on their own asynchronous copies,
 * tensor-core operations and (the split kernel) on each other's CTAs with
 * bounded waits; a wait that gives up makes the kernel stop early (outputs of
 * the affected sequences are then incomplete) and records a status word on
 * the device instead of trapping.  kda_backward records a device-side
 * argument check there too (a needed chunk-state row past chunk_capacity).
 * This call synchronises `stream` and, since the previous call, returns
 * KDA_ERR_INVALID_ARGUMENT if the backward's check failed, else
 * KDA_ERR_TIMEOUT if any wait gave up, else KDA_OK; then it resets the
 * words.  KDA_ERR_CUDA if the synchronisation itself fails.
 */
kda_status kda_get_last_device_error(kda_stream_t stream);

/*
 * kda_selftest_timeout -- diagnostic of the bounded-wait path (not part of
 * the method).  Enqueues a one-warp kernel on `stream` that waits, with the
 * same bounded wait the prefill kernel uses, on a barrier nothing arrives on;
 * the wait gives up after a few milliseconds and records the device status
 * word, so that the next kda_get_last_device_error() returns KDA_ERR_TIMEOUT.
 * Nothing traps or hangs and the CUDA context stays usable.
 */
kda_status kda_selftest_timeout(kda_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *kda_status_string(kda_status status);

/* Text of the most recent CUDA error seen by this thread's calls into the
 * library ("" if none).  Static storage per thread; valid until the next call. */
const char *kda_last_cuda_error(void);

/* Library version as 10000*major + 100*minor + patch. */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
