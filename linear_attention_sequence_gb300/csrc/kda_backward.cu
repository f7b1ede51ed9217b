// kda_backward.cu -- gradients of the chunked KDA prefill (CUDA cores, fp32).
//
// "Hybrid Attention", section "But isn't a recurrent update sequential?": the
// chunkwise computation is trained by comparing its outputs and gradients with
// the recurrent version.  This kernel computes the gradients chunk by chunk,
// walking the chunks of a sequence in reverse and carrying the adjoint dS of
// the state between them, from the forward's state at the start of every chunk
// (the checkpoints that kda_prefill_checkpointed writes at an interval of one
// chunk).
//
// Per chunk (C = 32 tokens; Gamma the running sum of g inside the chunk,
// gamma = e^Gamma, gC its last row; products taken pairwise as
// e^{Gamma_r - Gamma_i} <= 1, so nothing overflows):
//
//   forward again:  G[r,i] = sum_c k_rc k_ic e^{Gamma_rc - Gamma_ic} (i < r),
//                   P[r,i] = sum_c q_rc k_ic e^{...} (i <= r), T = (I + diag(beta) G)^{-1},
//                   Kt = K.gamma, Qt = Q.gamma, Kb = K.(gC / gamma),
//                   Y = V - Kt S0, B = diag(beta) Y, U = T B
//   backward:       dU = Kb dS + P^T dO,   dP = tril(dO U^T),   dB = T^T dU,
//                   dT = dU B^T,   dA = -T^T dT T^T (strict lower),
//                   dbeta = rowsum(dB . Y) + rowsum(dA . G),   dY = diag(beta) dB = dV,
//                   dQt = dO S0^T,   dKt = -dY S0^T,   dKb = U dS^T,
//                   dS0 = diag(gC) dS + Qt^T dO - Kt^T dY   (the adjoint for the chunk before),
//   then the pairwise terms of dG = diag(beta) dA and dP into dq, dk and dGamma, the
//   element-wise terms of Qt, Kt, Kb, and dg = the reverse running sum of dGamma.
//
// One CTA of 512 threads per (sequence, head).  The adjoint dS (d x d) stays in
// shared memory for the whole sequence; the value axis is processed in blocks of
// 32 columns, each block's contributions to the cross-column sums (dP, dT,
// dbeta, dQt, dKt, dKb) accumulated over the blocks.  fp32 throughout.

#include "kda_common.cuh"

namespace {

constexpr int C = 32;          // tokens per chunk (the checkpoint interval)
constexpr int BV = 32;         // value columns per block
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

template <int D>
struct BwdSmem {
    float dS[D][D + 1];        // adjoint of the state at the end of the current chunk
    float S0[D][BV + 1];       // the chunk's start state, one column block
    float Q[C][D], K[C][D];    // q, k of the chunk (rows past its end are 0)
    float Gam[C][D];           // Gamma
    float Qt[C][D], Kt[C][D], Kb[C][D];   // q.gamma, k.gamma, k.gamma_last/gamma
    float V[C][BV + 1], dO[C][BV + 1], Y[C][BV + 1], U[C][BV + 1], dU[C][BV + 1];
    float G[C][C + 1], P[C][C + 1], T[C][C + 1], dP[C][C + 1], dT[C][C + 1];
    float beta[C], dbeta[C];
    float gC[D], gsum[D];      // gamma_last; sum_j dS . S0 by row (the gamma_last term)
};

template <typename IN_T, typename OUT_T, int D>
__global__ void __launch_bounds__(kThreads, 1)
kda_backward_kernel(const IN_T *__restrict__ q, const IN_T *__restrict__ k,
                    const IN_T *__restrict__ v, const float *__restrict__ g,
                    const float *__restrict__ beta, const float *__restrict__ init_state,
                    const int32_t *__restrict__ cu, const float *__restrict__ chunk_states,
                    int64_t chunk_capacity, const IN_T *__restrict__ d_out, const float *__restrict__ d_final,
                    OUT_T *__restrict__ dq, OUT_T *__restrict__ dk, OUT_T *__restrict__ dv,
                    float *__restrict__ dg, float *__restrict__ dbeta,
                    float *__restrict__ d_init, int H, int64_t total, int64_t seq_len) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<D> &sm = *reinterpret_cast<BwdSmem<D> *>(smem_raw);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);
    const int nchunks = (int)((b - a + C - 1) / C);
    const int64_t rowK = (int64_t)H * D;
    const int64_t sdd = (int64_t)D * D;
    // checkpoint row of chunk 1 of this sequence: the rows of earlier sequences first
    const int64_t ck0 = kda::ckpt_first_row(cu, n, total, seq_len, C);

    // ownership of the C x D accumulators: channel c, rows r0 + RSTEP m
    constexpr int RSTEP = kThreads / D;        // 4 (D = 128) or 8 (D = 64)
    constexpr int RPT = C / RSTEP;             // rows per thread: 8 or 4
    const int oc = t % D, or0 = t / D;

    for (int idx = t; idx < D * D; idx += kThreads) {
        const int r = idx / D, c = idx % D;
        sm.dS[r][c] = d_final ? d_final[((int64_t)n * H + h) * sdd + idx] : 0.f;
    }

    for (int ch = nchunks - 1; ch >= 0; --ch) {
        const int64_t t0 = a + (int64_t)ch * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        // the state at the start of the chunk: the initial state, or checkpoint row
        // ck0 + ch - 1 (rows past the caller's capacity are never read)
        const int64_t crow = ck0 + ch - 1;
        const float *S0g = ch == 0 ? (init_state ? init_state + ((int64_t)n * H + h) * sdd : nullptr)
                           : (chunk_states && crow < chunk_capacity)
                               ? chunk_states + (crow * H + h) * sdd
                               : nullptr;
        __syncthreads();   // the previous chunk is done with every buffer

        // ---- load q, k, g (rows past the end are 0) and beta ----
        for (int idx = t; idx < C * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < L) {
                const int64_t off = (t0 + r) * rowK + (int64_t)h * D + c;
                qv = kda::ld_elem(q + off);
                kv = kda::ld_elem(k + off);
                gv = g[off];
            }
            sm.Q[r][c] = qv;
            sm.K[r][c] = kv;
            sm.Gam[r][c] = gv;
        }
        if (t < C) {
            sm.beta[t] = t < L ? beta[(t0 + t) * H + h] : 0.f;
            sm.dbeta[t] = 0.f;
        }
        __syncthreads();
        // ---- Gamma (running sum per channel), gamma_last ----
        if (t < D) {
            float run = 0.f;
            for (int r = 0; r < C; ++r) {
                run += sm.Gam[r][t];
                sm.Gam[r][t] = run;
            }
            sm.gC[t] = __expf(run);
            sm.gsum[t] = 0.f;
        }
        __syncthreads();
        // ---- decay-weighted copies ----
        for (int idx = t; idx < C * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            const float gam = sm.Gam[r][c];
            const float e = __expf(gam), eb = __expf(sm.Gam[C - 1][c] - gam);
            sm.Qt[r][c] = sm.Q[r][c] * e;
            sm.Kt[r][c] = sm.K[r][c] * e;
            sm.Kb[r][c] = sm.K[r][c] * eb;
        }
        // ---- G (strict) and P (inclusive): one warp per (r, i) pair ----
        for (int p = warp; p < C * C; p += kWarps) {
            const int r = p / C, i = p % C;
            float gg = 0.f, pp = 0.f;
            if (i <= r) {
                for (int c = lane; c < D; c += 32) {
                    const float e = __expf(sm.Gam[r][c] - sm.Gam[i][c]);
                    const float ke = sm.K[i][c] * e;
                    gg += sm.K[r][c] * ke;
                    pp += sm.Q[r][c] * ke;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    gg += __shfl_xor_sync(0xffffffffu, gg, o);
                    pp += __shfl_xor_sync(0xffffffffu, pp, o);
                }
            }
            if (lane == 0) {
                sm.G[r][i] = i < r ? gg : 0.f;
                sm.P[r][i] = pp;   // 0 above the diagonal
                sm.dP[r][i] = 0.f;
                sm.dT[r][i] = 0.f;
            }
        }
        __syncthreads();
        // ---- T = (I + diag(beta) G)^{-1}: lane j solves column j (warp 0) ----
        if (warp == 0) {
            float x[C];
#pragma unroll
            for (int i = 0; i < C; ++i) x[i] = i == lane ? 1.f : 0.f;
#pragma unroll
            for (int i = 1; i < C; ++i) {
                float acc = x[i];
                const float bi = sm.beta[i];
#pragma unroll
                for (int m = 0; m < i; ++m) acc -= bi * sm.G[i][m] * x[m];
                x[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < C; ++i) sm.T[i][lane] = x[i];
        }
        float aQt[RPT], aKt[RPT], aKb[RPT];   // dQt, dKt, dKb of (or0 + RSTEP m, oc)
#pragma unroll
        for (int m = 0; m < RPT; ++m) aQt[m] = aKt[m] = aKb[m] = 0.f;

        for (int j0 = 0; j0 < D; j0 += BV) {
            __syncthreads();   // T is ready; the previous block is done with V, dO, Y, U, dU, S0
            // ---- this block of S0, V and dO ----
            for (int idx = t; idx < D * BV; idx += kThreads) {
                const int c = idx / BV, j = idx % BV;
                sm.S0[c][j] = S0g ? S0g[(int64_t)c * D + j0 + j] : 0.f;
            }
            for (int idx = t; idx < C * BV; idx += kThreads) {
                const int r = idx / BV, j = idx % BV;
                const int64_t off = (t0 + r) * rowK + (int64_t)h * D + j0 + j;
                sm.V[r][j] = r < L ? kda::ld_elem(v + off) : 0.f;
                sm.dO[r][j] = r < L ? kda::ld_elem(d_out + off) : 0.f;
            }
            __syncthreads();
            // ---- Y = V - Kt S0 and dU = Kb dS + P^T dO (thread: column lane, rows warp, warp + 16) ----
#pragma unroll
            for (int rr = 0; rr < C; rr += kWarps) {
                const int r = rr + warp, j = lane;
                float y = sm.V[r][j], du = 0.f;
                for (int c = 0; c < D; ++c) {
                    y -= sm.Kt[r][c] * sm.S0[c][j];
                    du += sm.Kb[r][c] * sm.dS[c][j0 + j];
                }
                for (int r2 = r; r2 < C; ++r2) du += sm.P[r2][r] * sm.dO[r2][j];
                sm.Y[r][j] = y;
                sm.dU[r][j] = du;
            }
            __syncthreads();
            // ---- U = T diag(beta) Y; dB = T^T dU (in place of dU after the reads below) ----
            float dbv[C / kWarps];
#pragma unroll
            for (int x = 0; x < C / kWarps; ++x) {
                const int r = x * kWarps + warp, j = lane;
                float u = 0.f, db = 0.f;
                for (int i = 0; i <= r; ++i) u += sm.T[r][i] * sm.beta[i] * sm.Y[i][j];
                for (int r2 = r; r2 < C; ++r2) db += sm.T[r2][r] * sm.dU[r2][j];
                sm.U[r][j] = u;
                dbv[x] = db;
            }
            __syncthreads();
            // ---- dP += tril(dO U^T), dT += dU (diag(beta) Y)^T (strict), dbeta += rowsum(dB . Y) ----
#pragma unroll
            for (int x = 0; x < C / kWarps; ++x) {
                const int r = x * kWarps + warp, i = lane;
                float sp = 0.f, st = 0.f;
                for (int j = 0; j < BV; ++j) {
                    sp += sm.dO[r][j] * sm.U[i][j];
                    st += sm.dU[r][j] * sm.Y[i][j];
                }
                if (i <= r) sm.dP[r][i] += sp;
                if (i < r) sm.dT[r][i] += st * sm.beta[i];
                float yb = dbv[x] * sm.Y[r][lane];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) yb += __shfl_xor_sync(0xffffffffu, yb, o);
                if (lane == 0) sm.dbeta[r] += yb;
            }
            __syncthreads();
            // ---- dY = diag(beta) dB (the value gradient), kept in dU ----
#pragma unroll
            for (int x = 0; x < C / kWarps; ++x) {
                const int r = x * kWarps + warp, j = lane;
                const float dy = sm.beta[r] * dbv[x];
                sm.dU[r][j] = dy;
                if (r < L) kda::st_elem(dv + (t0 + r) * rowK + (int64_t)h * D + j0 + j, dy);
            }
            __syncthreads();
            // ---- dQt += dO S0^T, dKt -= dY S0^T, dKb += U dS^T (old dS), gamma_last term ----
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int r = or0 + RSTEP * m, c = oc;
                float sq = 0.f, sk = 0.f, sb = 0.f;
                for (int j = 0; j < BV; ++j) {
                    const float s0 = sm.S0[c][j];
                    sq += sm.dO[r][j] * s0;
                    sk += sm.dU[r][j] * s0;
                    sb += sm.U[r][j] * sm.dS[c][j0 + j];
                }
                aQt[m] += sq;
                aKt[m] -= sk;
                aKb[m] += sb;
            }
            if (t < D) {
                float s = 0.f;
                for (int j = 0; j < BV; ++j) s += sm.dS[t][j0 + j] * sm.S0[t][j];
                sm.gsum[t] += s;
            }
            __syncthreads();
            // ---- dS <- diag(gC) dS + Qt^T dO - Kt^T dY on this block's columns ----
            for (int idx = t; idx < D * BV; idx += kThreads) {
                const int c = idx / BV, j = idx % BV;
                float s = sm.gC[c] * sm.dS[c][j0 + j];
                for (int r = 0; r < C; ++r) s += sm.Qt[r][c] * sm.dO[r][j] - sm.Kt[r][c] * sm.dU[r][j];
                sm.dS[c][j0 + j] = s;
            }
        }
        __syncthreads();
        // ---- dA = -T^T tril_s(dT) T^T (strict lower): M1 = tril_s(dT) T^T into dU's space ----
        float (*M1)[BV + 1] = sm.Y;   // C x C scratch (BV == C)
#pragma unroll
        for (int x = 0; x < C / kWarps; ++x) {
            const int r = x * kWarps + warp, i = lane;
            float s = 0.f;
            for (int bb = 0; bb < r && bb <= i; ++bb) s += sm.dT[r][bb] * sm.T[i][bb];
            M1[r][i] = s;
        }
        __syncthreads();
        // dA[r][i] for i < r, then dG = beta_r dA (into G's space) and dbeta += rowsum(dA . G)
#pragma unroll
        for (int x = 0; x < C / kWarps; ++x) {
            const int r = x * kWarps + warp, i = lane;
            float s = 0.f;
            for (int a2 = r; a2 < C; ++a2) s -= sm.T[a2][r] * M1[a2][i];
            const float da = i < r ? s : 0.f;
            float gb = da * sm.G[r][i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gb += __shfl_xor_sync(0xffffffffu, gb, o);
            __syncwarp();
            sm.G[r][i] = sm.beta[r] * da;   // dG (this thread read G[r][i] above)
            if (lane == 0) sm.dbeta[r] += gb;
        }
        __syncthreads();
        // ---- pairwise terms, element-wise terms and dGamma for the owned (r, c) ----
        float dgam[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int x = or0 + RSTEP * m, c = oc;
            const float gx = sm.Gam[x][c], kx = sm.K[x][c], qx = sm.Q[x][c];
            float dqx = 0.f, dkx = 0.f, dgx = 0.f;
            // x as the later token r: pairs (x, i), i <= x
            for (int i = 0; i <= x; ++i) {
                const float e = __expf(gx - sm.Gam[i][c]);
                const float ki = sm.K[i][c] * e;
                const float dgp = sm.G[x][i], dpp = sm.dP[x][i];
                dqx += dpp * ki;
                dkx += dgp * ki;
                dgx += (dgp * kx + dpp * qx) * ki;
            }
            // x as the earlier token i: pairs (r, x), r >= x
            for (int r = x; r < C; ++r) {
                const float e = __expf(sm.Gam[r][c] - gx);
                const float dgp = sm.G[r][x], dpp = sm.dP[r][x];
                const float w = (dgp * sm.K[r][c] + dpp * sm.Q[r][c]) * e;
                dkx += w;
                dgx -= w * kx;
            }
            const float gam = __expf(gx), kb = sm.Kb[x][c];
            dqx += aQt[m] * gam;
            dkx += aKt[m] * gam + aKb[m] * __expf(sm.Gam[C - 1][c] - gx);
            dgx += aQt[m] * sm.Qt[x][c] + aKt[m] * sm.Kt[x][c] - aKb[m] * kb;
            if (x < L) {
                const int64_t off = (t0 + x) * rowK + (int64_t)h * D + c;
                kda::st_elem(dq + off, dqx);
                kda::st_elem(dk + off, dkx);
            }
            dgam[m] = dgx;
        }
        // the gamma_last terms: column sums of dKb . Kb, and gC sum_j dS . S0
        __syncthreads();   // every read of Kt / Qt above is done: reuse Kt for dGamma
#pragma unroll
        for (int m = 0; m < RPT; ++m) sm.Kt[or0 + RSTEP * m][oc] = dgam[m];
        // (column sums of dKb . Kb over rows: the owned rows' part, reduced below)
        float kbk = 0.f;
#pragma unroll
        for (int m = 0; m < RPT; ++m) kbk += aKb[m] * sm.Kb[or0 + RSTEP * m][oc];
        sm.Qt[or0][oc] = kbk;   // Qt is free: one partial per (row group, channel)
        __syncthreads();
        // ---- dg = reverse running sum of dGamma over the chunk (thread per channel) ----
        if (t < D) {
            float last = sm.gC[t] * sm.gsum[t];
            for (int r0 = 0; r0 < RSTEP; ++r0) last += sm.Qt[r0][t];
            float run = 0.f;
            for (int r = C - 1; r >= 0; --r) {
                run += sm.Kt[r][t] + (r == C - 1 ? last : 0.f);
                if (r < L) dg[(t0 + r) * rowK + (int64_t)h * D + t] = run;
            }
        }
        if (t < C && t < L) dbeta[(t0 + t) * H + h] = sm.dbeta[t];
    }
    __syncthreads();
    if (d_init)
        for (int idx = t; idx < D * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            d_init[((int64_t)n * H + h) * sdd + idx] = sm.dS[r][c];
        }
}

template <typename IN_T, typename OUT_T, int D>
cudaError_t launch(const kda::Problem &P, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *init_state, const int32_t *cu,
                   const float *chunk_states, int64_t cap, const void *d_out,
                   const float *d_final, void *dq, void *dk, void *dv, float *dg, float *dbeta,
                   float *d_init, cudaStream_t stream) {
    auto kern = kda_backward_kernel<IN_T, OUT_T, D>;
    const size_t smem = sizeof(BwdSmem<D>);
    static_assert(sizeof(BwdSmem<128>) <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((int64_t)P.N * P.H);
    kern<<<blocks, kThreads, smem, stream>>>(
        (const IN_T *)q, (const IN_T *)k, (const IN_T *)v, g, beta, init_state, cu, chunk_states,
        cap, (const IN_T *)d_out, d_final, (OUT_T *)dq, (OUT_T *)dk, (OUT_T *)dv, dg, dbeta, d_init,
        P.H, (int64_t)P.T, P.seq_len);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch(const kda::Problem &P, const void *q, const void *k, const void *v,
                     const float *g, const float *beta, const float *init, const int32_t *cu,
                     const float *cs, int64_t cap, const void *d_out, const float *d_final,
                     void *dq, void *dk, void *dv, float *dg, float *dbeta, float *d_init,
                     cudaStream_t s) {
    const bool in_bf = P.in_dtype == KDA_DTYPE_BF16, out_bf = P.out_dtype == KDA_DTYPE_BF16;
    if (in_bf && out_bf)
        return launch<__nv_bfloat16, __nv_bfloat16, D>(P, q, k, v, g, beta, init, cu, cs, cap, d_out,
                                                       d_final, dq, dk, dv, dg, dbeta, d_init, s);
    if (in_bf)
        return launch<__nv_bfloat16, float, D>(P, q, k, v, g, beta, init, cu, cs, cap, d_out, d_final,
                                               dq, dk, dv, dg, dbeta, d_init, s);
    if (out_bf)
        return launch<float, __nv_bfloat16, D>(P, q, k, v, g, beta, init, cu, cs, cap, d_out, d_final,
                                               dq, dk, dv, dg, dbeta, d_init, s);
    return launch<float, float, D>(P, q, k, v, g, beta, init, cu, cs, cap, d_out, d_final, dq, dk, dv,
                                   dg, dbeta, d_init, s);
}

}  // namespace

cudaError_t kda_launch_backward(const kda::Problem &P, const void *q, const void *k,
                                const void *v, const float *g, const float *beta,
                                const float *init_state, const int32_t *cu,
                                const float *chunk_states, int64_t chunk_capacity,
                                const void *d_out, const float *d_final, void *dq, void *dk,
                                void *dv, float *dg, float *dbeta, float *d_init,
                                cudaStream_t stream) {
    if (P.N == 0) return cudaSuccess;
    if (P.dk == 128)
        return dispatch<128>(P, q, k, v, g, beta, init_state, cu, chunk_states, chunk_capacity, d_out, d_final, dq,
                             dk, dv, dg, dbeta, d_init, stream);
    return dispatch<64>(P, q, k, v, g, beta, init_state, cu, chunk_states, chunk_capacity, d_out, d_final, dq, dk,
                        dv, dg, dbeta, d_init, stream);
}
