// kda_prefill_fp32.cu -- chunked KDA prefill on the CUDA cores, fp32 throughout.
//
// This is the accuracy path (fp32 inputs are checked at 1e-4 of rms) and the
// kernel for shapes the tensor-core path does not take.  It evaluates the
// chunk form of the recurrence: tokens of a chunk are processed together and
// the state is carried from chunk to chunk ("Inside Kimi K3", section
// "Sequence mixing"; "Hybrid Attention", section "But isn't a recurrent update
// sequential?").  Within a chunk of C tokens (positions r = 0..C-1), with
// Gamma_r = sum_{i<=r} g_i per key channel and S0 the state entering it,
// unrolling the token recurrence gives (exactly, up to rounding):
//
//   u_r = beta_r (v_r - S0^T (e^{Gamma_r} . k_r)) - sum_{i<r} Akk[r,i] u_i
//   o_r = S0^T (e^{Gamma_r} . q_r) + sum_{i<=r} Aqk[r,i] u_i
//   S_C = Diag(e^{Gamma_{C-1}}) S0 + sum_i (e^{Gamma_{C-1} - Gamma_i} . k_i) u_i^T
//
//   Akk[r,i] = beta_r sum_c k_rc k_ic e^{Gamma_rc - Gamma_ic}   (i <  r)
//   Aqk[r,i] =        sum_c q_rc k_ic e^{Gamma_rc - Gamma_ic}   (i <= r: the
//                                           diagonal is included, each token
//                                           reads the state after its write)
//
// The u_r form is a forward substitution with the unit lower-triangular
// (I + Akk), the "triangular solve" of the chunkwise form.  The Gram matrices
// are products of factors taken against the chunk midpoint Gamma_15:
// k_r e^{Gamma_r - Gamma_15} and q_r e^{Gamma_r - Gamma_15} against
// k_i e^{Gamma_15 - Gamma_i}.  With g >= -5 and C = 32 every such factor is
// within e^{+-80} ("Understanding Kimi K3's Attention", log-decay bound), inside
// the fp32 range; the other decay factors are exponentials of non-positive
// numbers.  Rows past the end of a sequence are loaded as zeros (k = q =
// v = 0, g = 0, beta = 0): they neither decay nor write the state, and their
// outputs are not stored, so sequence lengths need not divide C.
//
// Grid: one CTA per (d_v block of BV columns, head, sequence).  Columns of the
// state evolve independently given k, g and beta, so d_v splits without
// communication; the Gram matrices are recomputed per block.

#include "kda_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int BV = 32;  // state columns per CTA (one per lane)

template <int DK, int C>
struct Smem {
    // rows of DK + 4 floats: 16-byte aligned, and rows four banks apart
    float G[C][DK + 4];    // Gamma, then e^{Gamma} . k
    float K[C][DK + 4];    // k, then k e^{Gamma - Gamma_15}, then e^{Gamma_last - Gamma} . k
    float Q[C][DK + 4];    // q, then q e^{Gamma - Gamma_15}, then e^{Gamma} . q
    float B1[C][DK + 4];   // k e^{Gamma_15 - Gamma}: the Gram's right factor
    float e15[DK], eC15[DK];   // e^{Gamma_15}, e^{Gamma_last - Gamma_15}
    float S[DK][BV];   // state slice (fp32)
    float U[C][BV];    // v, then v', then u
    float Akk[C][C + 1];
    float Aqk[C][C + 1];
    float beta[C];
    float glast[DK];   // Gamma of the last row
    int seq_of_slot;   // the sequence this CTA runs (longest first)
};

template <int DK, int C, typename IN_T, typename OUT_T>
__global__ void __launch_bounds__(kThreads)
kda_prefill_fp32_kernel(const IN_T *__restrict__ q, const IN_T *__restrict__ k,
                        const IN_T *__restrict__ v, const float *__restrict__ g,
                        const float *__restrict__ beta, const float *init_state,
                        const int32_t *__restrict__ cu, OUT_T *__restrict__ out,
                        float *final_state, int H, int DV, int64_t total,
                        int64_t seq_len, float *__restrict__ ckpt, int64_t ckpt_every,
                        int64_t ckpt_cap, const IN_T *__restrict__ z,
                        const float *__restrict__ a_log, int sdecay,
                        const float *__restrict__ g_head) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<DK, C> &sm = *reinterpret_cast<Smem<DK, C> *>(smem_raw);

    const int vb = blockIdx.x, h = blockIdx.y;
    const int n = kda::longest_first(cu, (int)gridDim.z, total, seq_len, blockIdx.z,
                                     &sm.seq_of_slot);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int j0 = vb * BV;

    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);

    const int64_t state_off = ((int64_t)n * H + h) * DK * (int64_t)DV;
    for (int idx = t; idx < DK * BV; idx += kThreads) {
        const int c = idx / BV, j = idx % BV;
        sm.S[c][j] = init_state ? init_state[state_off + (int64_t)c * DV + j0 + j] : 0.f;
    }

    const int64_t rowK = (int64_t)H * DK, rowV = (int64_t)H * DV;
    // gate prologue: z (decay logits) and beta logits instead of g and beta
    const float gscale = z ? __expf(a_log[h]) : 0.f;
    // state checkpoints: after every ckpt_every chunks that end inside the sequence
    const int64_t ck_row0 = ckpt ? kda::ckpt_first_row(cu, n, total, seq_len, ckpt_every * C) : 0;
    int64_t chunk = 0;
    for (int64_t t0 = a; t0 < b; t0 += C, ++chunk) {
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        __syncthreads();  // previous chunk done with every buffer
        // ---- load the chunk (rows >= L are zeros): every load of a thread is
        // issued before its first store, so their latencies overlap ----
        {
            constexpr int PER = C * DK / kThreads, PERV = C * BV / kThreads;
            float gv[PER], kv[PER], qv[PER], vv[PERV];
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int idx = t + m * kThreads, r = idx / DK, c = idx % DK;
                gv[m] = kv[m] = qv[m] = 0.f;
                if (r < L) {
                    const int64_t off = (t0 + r) * rowK + (int64_t)h * DK + c;
                    // the decay: from its logits, one per (token, head), or per channel
                    gv[m] = z        ? kda::gate_g(kda::ld_elem(z + off), gscale)
                            : sdecay ? (g_head ? g_head[(t0 + r) * H + h] : 0.f)
                                     : g[off];
                    kv[m] = kda::ld_elem(k + off);
                    qv[m] = kda::ld_elem(q + off);
                }
            }
#pragma unroll
            for (int m = 0; m < PERV; ++m) {
                const int idx = t + m * kThreads, r = idx / BV, j = idx % BV;
                vv[m] = r < L ? kda::ld_elem(v + (t0 + r) * rowV + (int64_t)h * DV + j0 + j) : 0.f;
            }
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int idx = t + m * kThreads, r = idx / DK, c = idx % DK;
                sm.G[r][c] = gv[m];
                sm.K[r][c] = kv[m];
                sm.Q[r][c] = qv[m];
            }
#pragma unroll
            for (int m = 0; m < PERV; ++m) {
                const int idx = t + m * kThreads, r = idx / BV, j = idx % BV;
                sm.U[r][j] = vv[m];
            }
        }
        if (t < C) {
            const float bt = t < L ? beta[(t0 + t) * H + h] : 0.f;
            sm.beta[t] = t < L ? (z ? kda::sigmoid_f(bt) : bt) : 0.f;
        }
        __syncthreads();

        // ---- Gamma: running sum of g over the chunk, per key channel ----
        if (t < DK) {
            float run = 0.f;
            for (int r = 0; r < C; ++r) {
                run += sm.G[r][t];
                sm.G[r][t] = run;
            }
            sm.glast[t] = run;
        }
        __syncthreads();

        // ---- the Gram factors around the midpoint Gamma_15 ----
        for (int idx = t; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, c = idx % DK;
            const float d1 = sm.G[r][c] - sm.G[15][c];
            const float e = __expf(d1), kv = sm.K[r][c];
            sm.K[r][c] = kv * e;                // k e^{Gamma - Gamma_15}
            sm.Q[r][c] *= e;                    // q e^{Gamma - Gamma_15}
            sm.B1[r][c] = kv * __expf(-d1);     // k e^{Gamma_15 - Gamma}
        }
        if (t < DK) {
            sm.e15[t] = __expf(sm.G[15][t]);
            sm.eC15[t] = __expf(sm.glast[t] - sm.G[15][t]);
        }
        __syncthreads();

        // ---- Gram matrices Akk = diag(beta) tril_s(K1 B1^T) on threads 0-127 and
        // Aqk = tril(Q1 B1^T) on 128-255: lane i takes column i, each thread 8 rows
        // (rows of B1 are four banks apart, so the column reads do not conflict) ----
        {
            const bool qhalf = t >= kThreads / 2;   // warp-uniform
            const int th = t & (kThreads / 2 - 1);
            const int i = th & 31, r8 = (th >> 5) * 8;
            const float(*Am)[DK + 4] = qhalf ? sm.Q : sm.K;
            float acc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = 0.f;
            for (int c = 0; c < DK; c += 4) {
                const float4 y = *reinterpret_cast<const float4 *>(&sm.B1[i][c]);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 x = *reinterpret_cast<const float4 *>(&Am[r8 + u][c]);
                    acc[u] += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r8 + u;
                if (qhalf) sm.Aqk[r][i] = i <= r ? acc[u] : 0.f;
                else sm.Akk[r][i] = i < r ? sm.beta[r] * acc[u] : 0.f;
            }
        }
        __syncthreads();

        // ---- decay-weighted operands for the state terms (from the factored copies
        // and the per-channel factors) ----
        for (int idx = t; idx < C * DK; idx += kThreads) {
            const int r = idx / DK, c = idx % DK;
            const float k1 = sm.K[r][c];
            sm.G[r][c] = k1 * sm.e15[c];               // e^{Gamma} . k
            sm.Q[r][c] *= sm.e15[c];                   // e^{Gamma} . q
            sm.K[r][c] = sm.B1[r][c] * sm.eC15[c];     // e^{Gamma_last - Gamma} . k
        }
        __syncthreads();

        // ---- v' = v - (e^Gamma . K) S0 and the inter-chunk readout (e^Gamma . Q) S0 ----
        constexpr int RPW = C / kWarps;  // rows per warp
        float o_acc[RPW];
        {
            float vs[RPW];
#pragma unroll
            for (int x = 0; x < RPW; ++x) { vs[x] = 0.f; o_acc[x] = 0.f; }
            for (int c = 0; c < DK; ++c) {
                const float s = sm.S[c][lane];
#pragma unroll
                for (int x = 0; x < RPW; ++x) {
                    const int r = warp * RPW + x;
                    vs[x] += sm.G[r][c] * s;
                    o_acc[x] += sm.Q[r][c] * s;
                }
            }
#pragma unroll
            for (int x = 0; x < RPW; ++x) sm.U[warp * RPW + x][lane] -= vs[x];
        }
        __syncthreads();

        // ---- forward substitution: u_r = beta_r v'_r - sum_{i<r} Akk[r,i] u_i, the
        // column of lane j held in registers ----
        if (warp == 0) {
            float u[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = sm.beta[r] * sm.U[r][lane];
#pragma unroll
                for (int i = 0; i < r; ++i) acc -= sm.Akk[r][i] * u[i];
                u[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < C; ++r) sm.U[r][lane] = u[r];
        }
        __syncthreads();

        // ---- intra-chunk readout and output store ----
#pragma unroll
        for (int x = 0; x < RPW; ++x) {
            const int r = warp * RPW + x;
            float acc = o_acc[x];
            for (int i = 0; i <= r; ++i) acc += sm.Aqk[r][i] * sm.U[i][lane];
            if (r < L) kda::st_elem(out + (t0 + r) * rowV + (int64_t)h * DV + j0 + lane, acc);
        }

        // ---- state carry: S = Diag(e^{Gamma_last}) S0 + Kbar^T U ----
        constexpr int CPW = DK / kWarps;  // state rows per warp
#pragma unroll
        for (int x = 0; x < CPW; ++x) {
            const int c = warp * CPW + x;
            float acc = __expf(sm.glast[c]) * sm.S[c][lane];
            for (int r = 0; r < C; ++r) acc += sm.K[r][c] * sm.U[r][lane];
            sm.S[c][lane] = acc;
        }
        if (ckpt && (chunk + 1) % ckpt_every == 0 && t0 + C <= b) {
            const int64_t row = ck_row0 + (chunk + 1) / ckpt_every - 1;
            if (row < ckpt_cap) {
                __syncthreads();
                const int64_t off = (row * H + h) * DK * (int64_t)DV;
                for (int idx = t; idx < DK * BV; idx += kThreads) {
                    const int c = idx / BV, j = idx % BV;
                    ckpt[off + (int64_t)c * DV + j0 + j] = sm.S[c][j];
                }
            }
        }
    }
    __syncthreads();
    if (final_state) {
        for (int idx = t; idx < DK * BV; idx += kThreads) {
            const int c = idx / BV, j = idx % BV;
            final_state[state_off + (int64_t)c * DV + j0 + j] = sm.S[c][j];
        }
    }
}

template <int DK, int C, typename IN_T, typename OUT_T>
cudaError_t launch(const kda::Problem &P, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *init_state,
                   const int32_t *cu, void *out, float *final_state, cudaStream_t stream) {
    if (P.N == 0) return cudaSuccess;
    auto kern = kda_prefill_fp32_kernel<DK, C, IN_T, OUT_T>;
    const size_t smem = sizeof(Smem<DK, C>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P.dv / BV, P.H, P.N);
    kern<<<grid, kThreads, smem, stream>>>((const IN_T *)q, (const IN_T *)k, (const IN_T *)v, g,
                                           beta, init_state, cu, (OUT_T *)out, final_state, P.H,
                                           P.dv, (int64_t)P.T, P.seq_len, P.ckpt,
                                           P.ckpt ? P.ckpt_interval / C : 1, P.ckpt_capacity,
                                           P.a_log ? (const IN_T *)P.z : nullptr, P.a_log,
                                           P.scalar_decay ? 1 : 0, P.g_head);
    return cudaGetLastError();
}

template <int DK>
cudaError_t dispatch_dtypes(const kda::Problem &P, const void *q, const void *k, const void *v,
                            const float *g, const float *beta, const float *init,
                            const int32_t *cu, void *out, float *fin, cudaStream_t s) {
    constexpr int C = 32;
    const bool in_bf = P.in_dtype == KDA_DTYPE_BF16, out_bf = P.out_dtype == KDA_DTYPE_BF16;
    if (in_bf && out_bf)
        return launch<DK, C, __nv_bfloat16, __nv_bfloat16>(P, q, k, v, g, beta, init, cu, out, fin, s);
    if (in_bf) return launch<DK, C, __nv_bfloat16, float>(P, q, k, v, g, beta, init, cu, out, fin, s);
    if (out_bf) return launch<DK, C, float, __nv_bfloat16>(P, q, k, v, g, beta, init, cu, out, fin, s);
    return launch<DK, C, float, float>(P, q, k, v, g, beta, init, cu, out, fin, s);
}

}  // namespace

cudaError_t kda_launch_prefill_fp32(const kda::Problem &P, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *init_state, const int32_t *cu, void *out,
                                    float *final_state, cudaStream_t stream) {
    if (P.dk == 128)
        return dispatch_dtypes<128>(P, q, k, v, g, beta, init_state, cu, out, final_state, stream);
    return dispatch_dtypes<64>(P, q, k, v, g, beta, init_state, cu, out, final_state, stream);
}
