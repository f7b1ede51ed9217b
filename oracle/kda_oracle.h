/*
 * kda_oracle.h -- fp64 CPU oracle of the KDA recurrence.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the CUDA product path.
 *
 * All arrays are fp64 (bf16 or fp32 inputs are widened exactly by the
 * caller); layouts as in kda_oracle.c.  Returns 0 on success, -1 on a bad
 * argument or an input outside the gates' domain (g in [-5, 0], beta in
 * [0, 1]).  num_threads <= 0 uses every online CPU.
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

int kda_oracle_num_cpus(void);

/* Token-by-token recurrence over a packed batch.  init_state may be NULL
 * (zeros); cu_seqlens may be NULL (num_seqs equal-length sequences);
 * final_state may be NULL (not written). */
int kda_oracle_prefill(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                       int32_t d_k, int32_t d_v, const double *q, const double *k,
                       const double *v, const double *g, const double *beta,
                       const double *init_state, const int32_t *cu_seqlens,
                       double *out, double *final_state, int32_t num_threads);

/* Gated DeltaNet (one decay per head and step: alpha_t = exp(g_head[t,h]),
 * g_head [total_tokens, num_heads]) and, with g_head NULL, the delta rule
 * (alpha_t = 1).  Other arguments as kda_oracle_prefill. */
int kda_oracle_prefill_scalar_decay(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    int32_t d_k, int32_t d_v, const double *q, const double *k,
                                    const double *v, const double *g_head, const double *beta,
                                    const double *init_state, const int32_t *cu_seqlens,
                                    double *out, double *final_state, int32_t num_threads);

/* Gradients of kda_oracle_prefill's outputs and final states, reverse mode:
 * given d_out [T, H, d_v] and d_final_state [N, H, d_k, d_v] (NULL => 0),
 * writes dq, dk, dg [T, H, d_k], dv [T, H, d_v], dbeta [T, H] and
 * d_init_state [N, H, d_k, d_v].  Other arguments as kda_oracle_prefill. */
int kda_oracle_backward(int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t d_k,
                        int32_t d_v, const double *q, const double *k, const double *v,
                        const double *g, const double *beta, const double *init_state,
                        const int32_t *cu_seqlens, const double *d_out,
                        const double *d_final_state, double *dq, double *dk, double *dv,
                        double *dg, double *dbeta, double *d_init_state, int32_t num_threads);

/* One decode step: one token per sequence, state updated in place. */
int kda_oracle_decode(int32_t num_seqs, int32_t num_heads, int32_t d_k, int32_t d_v,
                      const double *q, const double *k, const double *v,
                      const double *g, const double *beta, double *state_inout,
                      double *out, int32_t num_threads);

/* Gate prologue: for every token t, head h and key channel c,
 * g[t,h,c] = g_min Sigmoid(e^{a_log[h]} z[t,h,c]) with g_min = -5, and
 * beta[t,h] = Sigmoid(beta_logit[t,h]).  Returns 0. */
int kda_oracle_gate(int32_t total_tokens, int32_t num_heads, int32_t d_k, const double *z,
                    const double *a_log, const double *beta_logit, double *g, double *beta);

/* Output gate: y[t,h,j] = Sigmoid(gate_logit[t,h,j]) * o[t,h,j] /
 * sqrt(mean_j o[t,h,:]^2 + eps) * norm_weight[j] (norm_weight NULL => 1),
 * over [total_tokens, num_heads, d_v] arrays.  eps > 0.  Returns -1 on a bad
 * argument, else 0. */
int kda_oracle_output_gate(int32_t total_tokens, int32_t num_heads, int32_t d_v,
                           const double *o, const double *gate_logit,
                           const double *norm_weight, double eps, double *y);

/* q, k, v prologue: per channel, the causal width-4 convolution over the
 * tokens of each sequence (the three inputs before a sequence's start come
 * from conv_state_in, or are 0 if it is NULL), then Swish(c) = c Sigmoid(c),
 * then for q and k (streams 0, 1; v is stream 2) division by sqrt(sum over
 * the head's d channels of the square + eps).  x, y [3][T][H][d]; conv_weight
 * [3][H][d][4] (tap 3 on the current token); conv states [N][3][3][H][d]
 * (entry 0 the oldest); conv_state_out may be NULL.  cu_seqlens [N+1] is
 * required.  Returns -1 on a bad argument, else 0. */
int kda_oracle_qkv_prologue(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                            int32_t d, const int32_t *cu_seqlens, const double *x,
                            const double *conv_weight, const double *conv_state_in, double eps,
                            double *y, double *conv_state_out);

#ifdef __cplusplus
}
#endif
#endif
