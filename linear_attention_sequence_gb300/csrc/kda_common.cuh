// kda_common.cuh -- small helpers shared by the KDA kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Element loads/stores for the two supported activation dtypes.
__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Sequence bounds for sequence n.  Entries of cu_seqlens are clamped into
// [0, total] and a decreasing pair is read as an empty sequence, so a
// malformed array never leads to an out-of-range access.
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int n, int64_t total,
                                           int64_t seq_len, int64_t &a, int64_t &b) {
    if (cu) {
        int64_t x = cu[n], y = cu[n + 1];
        x = x < 0 ? 0 : (x > total ? total : x);
        y = y < 0 ? 0 : (y > total ? total : y);
        a = x;
        b = y < x ? x : y;
    } else {
        a = (int64_t)n * seq_len;
        b = a + seq_len;
    }
}

// Bit of the device status word set by a device-side argument check (the
// backward's missing chunk-state rows); the other bits are bounded waits that
// gave up.
constexpr unsigned kBwdMissingState = 0x1000u;

// Host-side launch parameters after validation.
struct Problem {
    int32_t N, T, H, dk, dv;
    int32_t in_dtype, out_dtype, variant;
    int64_t seq_len;  // used when cu_seqlens == NULL
    // gate prologue (kda_prefill_gated): with a_log != nullptr the kernels
    // read the decay logits z (in_dtype) instead of g, and beta logits
    const void *z = nullptr;
    const float *a_log = nullptr;
    // state checkpoints (kda_prefill_checkpointed); ckpt == nullptr: none
    float *ckpt = nullptr;
    int64_t ckpt_interval = 0;  // tokens between checkpoints, a multiple of the chunk length
    int64_t ckpt_capacity = 0;  // rows of [capacity, H, d_k, d_v] that may be written
    // output gate (kda_prefill_output_gated): y = Sigmoid(gate) RMSNorm(o~) w
    const void *ogate = nullptr;     // gate logits, in_dtype [T, H, d_v]; nullptr: none
    const float *onorm_w = nullptr;  // [d_v] or nullptr (weight 1)
    float oeps = 0.f;
    bool ogate_fused = false;        // applied by the tensor-core kernel before its store
    // scalar decay (kda_prefill_scalar_decay): one log-decay per (token, head)
    // replaces g; g_head == nullptr means no decay (the delta rule)
    bool scalar_decay = false;
    const float *g_head = nullptr;   // fp32 [T, H]
};

// Gate prologue ("Understanding Kimi K3's Attention", log-decay bound and
// symbol table): g = g_min Sigmoid(e^{A_h} z) per key channel, beta =
// Sigmoid(logit).  `scale` is e^{A_h}.  The fast reciprocal of +inf is +0, so
// a very negative argument (e^{-x} = inf) gives exactly 0, the limit.
constexpr float kGMin = -5.f;
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float gate_g(float z, float scale) { return kGMin * sigmoid_f(scale * z); }

// Longest-first order of the sequences of a packed batch: the sequence that the
// CTAs of scheduling slot `slot` process.  Slots are launched in order, so the
// longest sequences start first and the shortest fill in at the end.  Each
// thread of the block ranks one sequence (by descending length, ties by index)
// and the one ranked `slot` answers through `*answer` (shared memory).  A batch
// of equal lengths (cu == nullptr) or of more sequences than threads keeps the
// given order.  Every thread of the block must call it.
__device__ __forceinline__ int longest_first(const int32_t *cu, int N, int64_t total,
                                             int64_t seq_len, int slot, int *answer) {
    if (!cu || N > (int)blockDim.x) return slot;
    const int m = threadIdx.x;
    if (m < N) {
        int64_t a, b;
        seq_bounds(cu, m, total, seq_len, a, b);
        const int64_t len = b - a;
        int rank = 0;
        for (int m2 = 0; m2 < N; ++m2) {
            int64_t a2, b2;
            seq_bounds(cu, m2, total, seq_len, a2, b2);
            const int64_t len2 = b2 - a2;
            rank += (len2 > len || (len2 == len && m2 < m)) ? 1 : 0;
        }
        if (rank == slot) *answer = m;
    }
    __syncthreads();
    return *answer;
}

// Row of the first checkpoint of sequence n: the checkpoints of the earlier
// sequences come first, floor(length / interval) of them each.
__device__ __forceinline__ int64_t ckpt_first_row(const int32_t *cu, int n, int64_t total,
                                                  int64_t seq_len, int64_t interval) {
    if (!cu) return (int64_t)n * (seq_len / interval);
    int64_t row = 0;
    for (int m = 0; m < n; ++m) {
        int64_t a, b;
        seq_bounds(cu, m, total, seq_len, a, b);
        row += (b - a) / interval;
    }
    return row;
}

}  // namespace kda

// Host: the TMA view of a [T, H, 128] tensor that the tensor-core prefill uses:
// (element within a 128-byte segment, token, segment index along the H*128 row),
// box = one head's segments for 32 tokens, 128-byte swizzle.  False if the
// driver entry point is missing or the encoding fails.
bool kda_make_tile_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                       int64_t T, int H);

// Host: the TMA view of an fp32 array of 128 x 128 states as rows of 128
// floats, box 128 rows x 32 floats, 128-byte swizzle.
bool kda_make_state_map(CUtensorMap *m, const float *base, int64_t rows);

// Launchers (return cudaError_t of the launch).
cudaError_t kda_launch_decode(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float *state, void *out,
                              cudaStream_t stream);
bool kda_prefill_tc_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const void *out);
cudaError_t kda_launch_prefill_tc(const kda::Problem &P, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta,
                                  const float *init_state, const int32_t *cu, void *out,
                                  float *final_state, cudaStream_t stream);
cudaError_t kda_launch_output_gate(const kda::Problem &P, void *out, cudaStream_t stream);
cudaError_t kda_launch_backward(const kda::Problem &P, const void *q, const void *k,
                                const void *v, const float *g, const float *beta,
                                const float *init_state, const int32_t *cu,
                                const float *chunk_states, int64_t chunk_capacity,
                                const void *d_out, const float *d_final, void *dq, void *dk,
                                void *dv, float *dg, float *dbeta, float *d_init,
                                cudaStream_t stream);
cudaError_t kda_launch_qkv_prologue(const kda::Problem &P, const void *xq, const void *xk,
                                    const void *xv, const float *w, const float *cin,
                                    const int32_t *cu, void *q, void *k, void *v, float *cout,
                                    float eps, cudaStream_t stream);
cudaError_t kda_read_device_status(cudaStream_t stream, unsigned *status);
cudaError_t kda_tc_read_status(unsigned *status);
bool kda_tma_available();
cudaError_t kda_launch_selftest_timeout(cudaStream_t stream);
bool kda_prefill_chain_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                                 const float *g, const void *out);
cudaError_t kda_launch_prefill_chain(const kda::Problem &P, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const float *init_state, const int32_t *cu, void *out,
                                     float *final_state, cudaStream_t stream);
cudaError_t kda_chain_read_status(unsigned *status);
cudaError_t kda_bwd_read_status(unsigned *status);
bool kda_backward_tc_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                               const float *g, const void *d_out);
cudaError_t kda_launch_backward_tc(const kda::Problem &P, const void *q, const void *k,
                                   const void *v, const float *g, const float *beta,
                                   const float *init_state, const int32_t *cu,
                                   const float *chunk_states, int64_t chunk_capacity,
                                   const void *d_out, const float *d_final, void *dq, void *dk,
                                   void *dv, float *dg, float *dbeta, float *d_init,
                                   cudaStream_t stream);
cudaError_t kda_bwdtc_read_status(unsigned *status);
bool kda_prefill_noalloc_fits(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const void *out);
cudaError_t kda_launch_prefill_noalloc(const kda::Problem &P, const void *q, const void *k,
                                       const void *v, const float *g, const float *beta,
                                       const float *init_state, const int32_t *cu, void *out,
                                       float *final_state, cudaStream_t stream);
bool kda_prefill_2pass_supported(const kda::Problem &P);
cudaError_t kda_launch_prefill_2pass(const kda::Problem &P, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const float *init_state, const int32_t *cu, void *out,
                                     float *final_state, cudaStream_t stream);
cudaError_t kda_2pass_read_status(unsigned *status);
cudaError_t kda_launch_prefill_fp32(const kda::Problem &P, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *init_state, const int32_t *cu, void *out,
                                    float *final_state, cudaStream_t stream);
