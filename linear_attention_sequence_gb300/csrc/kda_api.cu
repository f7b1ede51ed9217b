// kda_api.cu -- the C ABI front end: argument validation, kernel selection,
// launch and error mapping.  Declarations and semantics: include/kda.h.

#include <initializer_list>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "kda_common.cuh"

namespace {

thread_local char g_last_cuda_error[256] = "";

kda_status cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", where,
             cudaGetErrorName(e), cudaGetErrorString(e));
    return KDA_ERR_CUDA;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Do the byte ranges [a, a + na) and [b, b + nb) share a byte?
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const char *x = (const char *)a, *y = (const char *)b;
    return x < y + nb && y < x + na;
}

// A buffer a call touches: its address and size in bytes (a NULL buffer is empty).
struct Span {
    const void *p;
    size_t n;
};

// Does a written buffer share a byte with a read buffer or with another
// written buffer?  The kernels read inputs (some by TMA, chunks ahead) while
// they write outputs, so any such overlap would be a race.
bool conflict(std::initializer_list<Span> writes, std::initializer_list<Span> reads) {
    for (const Span *w = writes.begin(); w != writes.end(); ++w) {
        for (const Span &r : reads)
            if (overlaps(w->p, w->n, r.p, r.n)) return true;
        for (const Span *w2 = w + 1; w2 != writes.end(); ++w2)
            if (overlaps(w->p, w->n, w2->p, w2->n)) return true;
    }
    return false;
}

size_t esize(int32_t dtype) { return dtype == KDA_DTYPE_BF16 ? 2 : 4; }

bool valid_dtype(int32_t d) { return d == KDA_DTYPE_F32 || d == KDA_DTYPE_BF16; }

// Shared checks of the dims struct.  Fills P on success.
kda_status check_dims(const kda_dims *d, kda::Problem &P) {
    if (!d) return KDA_ERR_INVALID_ARGUMENT;
    if (d->num_seqs < 0 || d->total_tokens < 0 || d->num_heads < 1 || d->d_k < 1 || d->d_v < 1)
        return KDA_ERR_INVALID_ARGUMENT;
    if (!valid_dtype(d->in_dtype) || !valid_dtype(d->out_dtype)) return KDA_ERR_INVALID_ARGUMENT;
    if (d->variant < KDA_PREFILL_DEFAULT || d->variant > KDA_PREFILL_TC_2PASS) return KDA_ERR_INVALID_ARGUMENT;
    if (d->d_k != d->d_v || (d->d_k != 64 && d->d_k != 128)) return KDA_ERR_UNSUPPORTED;
    // element counts must fit the kernels' 64-bit index arithmetic comfortably
    const int64_t elems = (int64_t)d->total_tokens * d->num_heads * d->d_k;
    const int64_t states = (int64_t)d->num_seqs * d->num_heads * d->d_k * d->d_v;
    if (elems > ((int64_t)1 << 50) || states > ((int64_t)1 << 50)) return KDA_ERR_INVALID_ARGUMENT;
    P.N = d->num_seqs;
    P.T = d->total_tokens;
    P.H = d->num_heads;
    P.dk = d->d_k;
    P.dv = d->d_v;
    P.in_dtype = d->in_dtype;
    P.out_dtype = d->out_dtype;
    P.variant = d->variant;
    P.seq_len = 0;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

const char *kda_last_cuda_error(void) { return g_last_cuda_error; }

int32_t kda_version(void) { return 100; /* 0.1.0 */ }

kda_status kda_selftest_timeout(kda_stream_t stream) {
    cudaError_t e = kda_launch_selftest_timeout((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kda_selftest_timeout");
    return KDA_OK;
}

kda_status kda_get_last_device_error(kda_stream_t stream) {
    unsigned status = 0;
    cudaError_t e = kda_read_device_status((cudaStream_t)stream, &status);
    if (e != cudaSuccess) return cuda_fail(e, "kda_get_last_device_error");
    if (status & kda::kBwdMissingState) return KDA_ERR_INVALID_ARGUMENT;
    return status ? KDA_ERR_TIMEOUT : KDA_OK;
}

namespace {

// The optional parts of a prefill call (all off by default).
struct Extras {
    float *ckpt = nullptr;            // state checkpoints
    int64_t ckpt_interval = 0, ckpt_capacity = 0;
    const void *z = nullptr;          // gate prologue: decay logits instead of g
    const float *a_log = nullptr;
    const void *ogate = nullptr;      // output gate
    const float *onorm_w = nullptr;
    float oeps = 0.f;
    bool scalar_decay = false;        // one log-decay per (token, head) instead of g
    const float *g_head = nullptr;    // (nullptr: no decay, the delta rule)
    bool noalloc = false;             // the split kernel on the library's fixed scratch array
};

kda_status prefill_common(const kda_dims *dims, const void *q, const void *k, const void *v,
                          const float *g, const float *beta, const float *init_state,
                          const int32_t *cu_seqlens, void *out, float *final_state,
                          const Extras &x, kda_stream_t stream, const char *where) {
    const void *z = x.z;
    const float *a_log = x.a_log;
    kda::Problem P;
    kda_status st = check_dims(dims, P);
    if (st != KDA_OK) return st;
    // with the gate prologue, z (decay logits) takes the place of g; with a
    // scalar decay there is no per-channel decay tensor at all
    const void *g_in = a_log ? z : (const void *)g;
    if (P.T > 0 && (!q || !k || !v || (!g_in && !x.scalar_decay) || !beta || !out))
        return KDA_ERR_INVALID_ARGUMENT;
    if (P.T > 0 && a_log && (z == (const void *)out)) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens) {
        if (P.N == 0 ? P.T != 0 : P.T % P.N != 0) return KDA_ERR_INVALID_ARGUMENT;
        P.seq_len = P.N ? P.T / P.N : 0;
    }
    {
        // outputs against inputs; final_state may be init_state itself (each
        // slice is read before it is written), but not overlap it otherwise
        const size_t tk = (size_t)P.T * P.H * P.dk, tv = (size_t)P.T * P.H * P.dv;
        const size_t sb = (size_t)P.N * P.H * P.dk * P.dv * sizeof(float);
        const size_t gb = x.scalar_decay ? (size_t)P.T * P.H * 4 : a_log ? tk * esize(P.in_dtype) : tk * 4;
        const void *gp = x.scalar_decay ? (const void *)x.g_head : g_in;
        const float *init_read = final_state == init_state ? nullptr : init_state;
        if (conflict({{out, tv * esize(P.out_dtype)}, {final_state, sb},
                      {x.ckpt_capacity > 0 ? x.ckpt : nullptr,
                       (size_t)x.ckpt_capacity * P.H * P.dk * P.dv * sizeof(float)}},
                     {{q, tk * esize(P.in_dtype)}, {k, tk * esize(P.in_dtype)},
                      {v, tv * esize(P.in_dtype)}, {gp, gb}, {beta, (size_t)P.T * P.H * 4},
                      {a_log, (size_t)P.H * 4}, {init_read, sb},
                      {cu_seqlens, cu_seqlens ? (size_t)(P.N + 1) * 4 : 0},
                      {x.ogate, x.ogate ? tv * esize(P.in_dtype) : 0},
                      {x.onorm_w, x.onorm_w ? (size_t)P.dv * 4 : 0}}))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    P.z = a_log ? z : nullptr;
    P.a_log = a_log;
    P.scalar_decay = x.scalar_decay;
    P.g_head = x.scalar_decay ? x.g_head : nullptr;
    P.ckpt = x.ckpt_capacity > 0 ? x.ckpt : nullptr;
    P.ckpt_interval = x.ckpt_interval;
    P.ckpt_capacity = x.ckpt_capacity;
    if (P.T > 0 && x.ogate) {
        P.ogate = x.ogate;
        P.onorm_w = x.onorm_w;
        P.oeps = x.oeps;
    }
    const bool tc_ok = kda_prefill_tc_supported(P, q, k, v, (const float *)g_in, out);
    const bool split_ok = x.noalloc ? kda_prefill_noalloc_fits(P, q, k, v, (const float *)g_in, out)
                                    : tc_ok && kda_prefill_chain_supported(P, q, k, v, (const float *)g_in, out);
    if (P.variant == KDA_PREFILL_TC && !tc_ok) return KDA_ERR_UNSUPPORTED;
    if (P.variant == KDA_PREFILL_TC_SPLIT && !split_ok) return KDA_ERR_UNSUPPORTED;
    const bool twopass_ok = tc_ok && kda_prefill_2pass_supported(P);
    if (P.variant == KDA_PREFILL_TC_2PASS && !twopass_ok) return KDA_ERR_UNSUPPORTED;
    if (P.N == 0) return KDA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    // the default takes the one-CTA-per-head tensor-core kernel where it supports the
    // call, else the CUDA-core kernel; the split kernel runs only when it is named
    const bool use_split = P.variant == KDA_PREFILL_TC_SPLIT;
    const bool use_2pass = P.variant == KDA_PREFILL_TC_2PASS;
    const bool use_tc = P.variant == KDA_PREFILL_TC || (P.variant == KDA_PREFILL_DEFAULT && tc_ok);
    // The split kernel gates a bf16 output in its epilogue, off the state chain's
    // critical path.  Every other case gates `out` in place after the prefill:
    // on the one-CTA-per-head kernel the fused epilogue sat on the chain warps and
    // made the call slower than the two calls.
    P.ogate_fused = P.ogate && !P.a_log && P.out_dtype == KDA_DTYPE_BF16 && (use_split || use_2pass);
    cudaError_t e = x.noalloc ? kda_launch_prefill_noalloc(P, q, k, v, g, beta, init_state, cu_seqlens,
                                                           out, final_state, s)
                    : use_2pass ? kda_launch_prefill_2pass(P, q, k, v, g, beta, init_state, cu_seqlens, out,
                                                           final_state, s)
                    : use_split ? kda_launch_prefill_chain(P, q, k, v, g, beta, init_state, cu_seqlens, out,
                                                         final_state, s)
                    : use_tc  ? kda_launch_prefill_tc(P, q, k, v, g, beta, init_state, cu_seqlens,
                                                      out, final_state, s)
                              : kda_launch_prefill_fp32(P, q, k, v, g, beta, init_state,
                                                        cu_seqlens, out, final_state, s);
    if (e == cudaSuccess && P.ogate && !P.ogate_fused) e = kda_launch_output_gate(P, out, s);
    if (e != cudaSuccess) return cuda_fail(e, where);
    return KDA_OK;
}

}  // namespace

kda_status kda_prefill(const kda_dims *dims, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const float *init_state,
                       const int32_t *cu_seqlens, void *out, float *final_state,
                       kda_stream_t stream) {
    return prefill_common(dims, q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                          Extras(), stream, "kda_prefill");
}

kda_status kda_prefill_noalloc(const kda_dims *dims, const void *q, const void *k, const void *v,
                               const float *g, const float *beta, const float *init_state,
                               const int32_t *cu_seqlens, void *out, float *final_state,
                               kda_stream_t stream) {
    if (!dims) return KDA_ERR_INVALID_ARGUMENT;
    kda_dims d = *dims;
    d.variant = KDA_PREFILL_TC_SPLIT;   // the one kernel this entry point runs
    Extras x;
    x.noalloc = true;
    return prefill_common(&d, q, k, v, g, beta, init_state, cu_seqlens, out, final_state, x, stream,
                          "kda_prefill_noalloc");
}

kda_status kda_prefill_checkpointed(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, float *checkpoints,
                                    int64_t interval, int64_t capacity, kda_stream_t stream) {
    if (interval <= 0 || interval % KDA_CHUNK != 0 || capacity < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (capacity > 0 && (!checkpoints || ((uintptr_t)checkpoints & 3u)))
        return KDA_ERR_INVALID_ARGUMENT;
    Extras x;
    x.ckpt = checkpoints;
    x.ckpt_interval = interval;
    x.ckpt_capacity = capacity;
    return prefill_common(dims, q, k, v, g, beta, init_state, cu_seqlens, out, final_state, x,
                          stream, "kda_prefill_checkpointed");
}

kda_status kda_prefill_gated(const kda_dims *dims, const void *q, const void *k, const void *v,
                             const void *z, const float *a_log, const float *beta_logit,
                             const float *init_state, const int32_t *cu_seqlens, void *out,
                             float *final_state, kda_stream_t stream) {
    if (!dims) return KDA_ERR_INVALID_ARGUMENT;
    if (dims->total_tokens > 0 && (!z || !a_log)) return KDA_ERR_INVALID_ARGUMENT;
    // with no tokens nothing is read: the call only copies the initial states
    const bool any = dims->total_tokens > 0;
    Extras x;
    x.z = any ? z : nullptr;
    x.a_log = any ? a_log : nullptr;
    return prefill_common(dims, q, k, v, nullptr, beta_logit, init_state, cu_seqlens, out,
                          final_state, x, stream, "kda_prefill_gated");
}

kda_status kda_prefill_output_gated(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const void *gate_logit, const float *norm_weight, float eps,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, kda_stream_t stream) {
    if (!dims) return KDA_ERR_INVALID_ARGUMENT;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARGUMENT;
    if (norm_weight && ((uintptr_t)norm_weight & 3u)) return KDA_ERR_INVALID_ARGUMENT;
    if (dims->total_tokens > 0 && (!gate_logit || gate_logit == (const void *)out))
        return KDA_ERR_INVALID_ARGUMENT;
    if (gate_logit && ((uintptr_t)gate_logit & (dims->in_dtype == KDA_DTYPE_BF16 ? 1u : 3u)))
        return KDA_ERR_INVALID_ARGUMENT;
    Extras x;
    x.ogate = gate_logit;
    x.onorm_w = norm_weight;
    x.oeps = eps;
    return prefill_common(dims, q, k, v, g, beta, init_state, cu_seqlens, out, final_state, x,
                          stream, "kda_prefill_output_gated");
}

kda_status kda_output_gate(const kda_dims *dims, void *out, const void *gate_logit,
                           const float *norm_weight, float eps, kda_stream_t stream) {
    kda::Problem P;
    kda_status st = check_dims(dims, P);
    if (st != KDA_OK) return st;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARGUMENT;
    if (norm_weight && ((uintptr_t)norm_weight & 3u)) return KDA_ERR_INVALID_ARGUMENT;
    if (P.T == 0) return KDA_OK;
    if (!out || !gate_logit) return KDA_ERR_INVALID_ARGUMENT;
    {
        const size_t tv = (size_t)P.T * P.H * P.dv;
        if (conflict({{out, tv * esize(P.out_dtype)}},
                     {{gate_logit, tv * esize(P.in_dtype)},
                      {norm_weight, norm_weight ? (size_t)P.dv * 4 : 0}}))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    const uintptr_t ga = P.in_dtype == KDA_DTYPE_BF16 ? 1u : 3u, oa = P.out_dtype == KDA_DTYPE_BF16 ? 1u : 3u;
    if (((uintptr_t)gate_logit & ga) || ((uintptr_t)out & oa)) return KDA_ERR_INVALID_ARGUMENT;
    P.ogate = gate_logit;
    P.onorm_w = norm_weight;
    P.oeps = eps;
    cudaError_t e = kda_launch_output_gate(P, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kda_output_gate");
    return KDA_OK;
}

kda_status kda_prefill_scalar_decay(const kda_dims *dims, const void *q, const void *k,
                                    const void *v, const float *g_head, const float *beta,
                                    const float *init_state, const int32_t *cu_seqlens,
                                    void *out, float *final_state, kda_stream_t stream) {
    if (g_head && ((uintptr_t)g_head & 3u)) return KDA_ERR_INVALID_ARGUMENT;
    Extras x;
    x.scalar_decay = true;
    x.g_head = g_head;
    return prefill_common(dims, q, k, v, nullptr, beta, init_state, cu_seqlens, out, final_state,
                          x, stream, "kda_prefill_scalar_decay");
}

kda_status kda_backward(const kda_dims *dims, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const float *init_state,
                        const int32_t *cu_seqlens, const float *chunk_states,
                        int64_t chunk_capacity, const void *d_out, const float *d_final_state,
                        void *dq, void *dk, void *dv, float *dg, float *dbeta,
                        float *d_init_state, kda_stream_t stream) {
    kda::Problem P;
    kda_status st = check_dims(dims, P);
    if (st != KDA_OK) return st;
    if (chunk_capacity < 0 || (chunk_capacity > 0 && !chunk_states)) return KDA_ERR_INVALID_ARGUMENT;
    if (chunk_states && ((uintptr_t)chunk_states & 3u)) return KDA_ERR_INVALID_ARGUMENT;
    if (P.T > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta))
        return KDA_ERR_INVALID_ARGUMENT;
    // a sequence longer than one chunk needs the forward's state at its chunk starts
    if (P.T > KDA_CHUNK && !chunk_states) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens) {
        if (P.N == 0 ? P.T != 0 : P.T % P.N != 0) return KDA_ERR_INVALID_ARGUMENT;
        P.seq_len = P.N ? P.T / P.N : 0;
        // equal lengths: the chunk-state rows needed are known here.  Sequence n's
        // rows start at n * floor(T / C) and it reads ceil(T / C) - 1 of them.
        const int64_t per = P.seq_len / KDA_CHUNK, nch = (P.seq_len + KDA_CHUNK - 1) / KDA_CHUNK;
        if (P.N > 0 && nch > 1 && chunk_capacity < (int64_t)(P.N - 1) * per + nch - 1)
            return KDA_ERR_INVALID_ARGUMENT;
    }
    {
        // the gradients must not overwrite what the kernel still reads, nor each other
        const size_t tk = (size_t)P.T * P.H * P.dk, tv = (size_t)P.T * P.H * P.dv;
        const size_t sb = (size_t)P.N * P.H * P.dk * P.dv * sizeof(float);
        const size_t ei = esize(P.in_dtype), eo = esize(P.out_dtype);
        if (conflict({{dq, tk * eo}, {dk, tk * eo}, {dv, tv * eo}, {dg, tk * 4},
                      {dbeta, (size_t)P.T * P.H * 4}, {d_init_state, sb}},
                     {{q, tk * ei}, {k, tk * ei}, {v, tv * ei}, {g, tk * 4},
                      {beta, (size_t)P.T * P.H * 4}, {d_out, tv * ei}, {init_state, sb},
                      {d_final_state, sb},
                      {chunk_states, (size_t)chunk_capacity * P.H * P.dk * P.dv * sizeof(float)},
                      {cu_seqlens, cu_seqlens ? (size_t)(P.N + 1) * 4 : 0}}))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if (P.N == 0) return KDA_OK;
    cudaError_t e = kda_launch_backward(P, q, k, v, g, beta, init_state, cu_seqlens, chunk_states,
                                        chunk_capacity, d_out, d_final_state, dq, dk, dv, dg,
                                        dbeta, d_init_state, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kda_backward");
    return KDA_OK;
}

kda_status kda_qkv_prologue(const kda_dims *dims, const void *x_q, const void *x_k,
                            const void *x_v, const float *conv_weight,
                            const float *conv_state_in, const int32_t *cu_seqlens, void *q,
                            void *k, void *v, float *conv_state_out, float eps,
                            kda_stream_t stream) {
    kda::Problem P;
    kda_status st = check_dims(dims, P);
    if (st != KDA_OK) return st;
    if (!(eps > 0.f) || !(eps < INFINITY)) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens) {
        if (P.N == 0 ? P.T != 0 : P.T % P.N != 0) return KDA_ERR_INVALID_ARGUMENT;
        P.seq_len = P.N ? P.T / P.N : 0;
    }
    // no sequence: no token belongs to one and no state is carried (as in kda_prefill)
    if (P.N == 0) return KDA_OK;
    if (P.T > 0 && (!conv_weight || !x_q || !x_k || !x_v || !q || !k || !v))
        return KDA_ERR_INVALID_ARGUMENT;
    // vector accesses: a lane moves d/32 consecutive elements of a row
    const int per = P.dk / 32;
    const uintptr_t in_al = (uintptr_t)per * (P.in_dtype == KDA_DTYPE_BF16 ? 2 : 4) - 1;
    const uintptr_t out_al = (uintptr_t)per * (P.out_dtype == KDA_DTYPE_BF16 ? 2 : 4) - 1;
    const uintptr_t st_al = (uintptr_t)per * 4 - 1;
    for (const void *p : {x_q, x_k, x_v})
        if ((uintptr_t)p & in_al) return KDA_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)q, (const void *)k, (const void *)v})
        if ((uintptr_t)p & out_al) return KDA_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)conv_weight & 15u) || ((uintptr_t)conv_state_in & st_al) ||
        ((uintptr_t)conv_state_out & 3u))
        return KDA_ERR_INVALID_ARGUMENT;
    // no output may overlap an input (neighbouring tiles read each other's rows)
    const size_t row_elems = (size_t)P.T * P.H * P.dk;
    const size_t in_b = row_elems * (P.in_dtype == KDA_DTYPE_BF16 ? 2 : 4);
    const size_t out_b = row_elems * (P.out_dtype == KDA_DTYPE_BF16 ? 2 : 4);
    const size_t w_b = (size_t)3 * P.H * P.dk * 4 * sizeof(float);
    const size_t st_b = (size_t)P.N * 9 * P.H * P.dk * sizeof(float);
    const void *ins[] = {x_q, x_k, x_v, conv_weight, conv_state_in};
    const size_t in_sz[] = {in_b, in_b, in_b, w_b, conv_state_in ? st_b : 0};
    const void *outs[] = {q, k, v, conv_state_out};
    const size_t out_sz[] = {out_b, out_b, out_b, conv_state_out ? st_b : 0};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 5; ++i)
            if (overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return KDA_ERR_INVALID_ARGUMENT;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlaps(outs[o], out_sz[o], outs[o2], out_sz[o2])) return KDA_ERR_INVALID_ARGUMENT;
    }
    // grid sizes (16 tokens x one (stream, head) per warp, 4 warps a block)
    const int64_t blocks = ((int64_t)P.T + 15) / 16 * 3 * P.H / 4 + 1;
    const int64_t st_blocks = ((int64_t)P.N * 9 * P.H * P.dk + 255) / 256;
    if (blocks > INT32_MAX || st_blocks > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    cudaError_t e = kda_launch_qkv_prologue(P, x_q, x_k, x_v, conv_weight, conv_state_in,
                                            cu_seqlens, q, k, v, conv_state_out, eps,
                                            (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kda_qkv_prologue");
    return KDA_OK;
}

kda_status kda_decode(const kda_dims *dims, const void *q, const void *k, const void *v,
                      const float *g, const float *beta, float *state_inout, void *out,
                      kda_stream_t stream) {
    kda::Problem P;
    kda_status st = check_dims(dims, P);
    if (st != KDA_OK) return st;
    if (P.T != P.N) return KDA_ERR_INVALID_ARGUMENT;
    if (P.N == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state_inout || !out) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(state_inout)) return KDA_ERR_INVALID_ARGUMENT;  // 16-byte vector access
    {
        // the state is updated in place; out and the state must not overlap an input or each other
        const size_t nk = (size_t)P.N * P.H * P.dk, nv = (size_t)P.N * P.H * P.dv;
        const size_t ei = esize(P.in_dtype);
        if (conflict({{out, nv * esize(P.out_dtype)}, {state_inout, nk * P.dv * sizeof(float)}},
                     {{q, nk * ei}, {k, nk * ei}, {v, nv * ei}, {g, nk * 4},
                      {beta, (size_t)P.N * P.H * 4}}))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    cudaError_t e = kda_launch_decode(P, q, k, v, g, beta, state_inout, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kda_decode");
    return KDA_OK;
}

}  // extern "C"
