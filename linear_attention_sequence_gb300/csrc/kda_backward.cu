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
    // rows of 36 floats (16-byte aligned: read four columns at a time); Y keeps 33
    // (read down its columns)
    float V[C][BV + 4], dO[C][BV + 4], U[C][BV + 4], dU[C][BV + 4];
    float Y[C][BV + 1];
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
        // ---- G (strict) and P (inclusive) over the lower triangle: each warp takes
        // four (r, i) pairs at a time, lanes over channels, so that the four
        // reductions overlap; the upper triangle is zero ----
        for (int idx = t; idx < C * C; idx += kThreads) {
            const int r = idx / C, i = idx % C;
            if (i > r) sm.G[r][i] = sm.P[r][i] = sm.dP[r][i] = sm.dT[r][i] = 0.f;
        }
        constexpr int NPAIR = C * (C + 1) / 2;
        for (int p0 = 4 * warp; p0 < NPAIR; p0 += 4 * kWarps) {
            int rr[4], ii[4];
            float gg[4], pp[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = p0 + u < NPAIR ? p0 + u : NPAIR - 1;
                int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
                while (r * (r + 1) / 2 > p) --r;
                while ((r + 1) * (r + 2) / 2 <= p) ++r;
                rr[u] = r;
                ii[u] = p - r * (r + 1) / 2;
                gg[u] = pp[u] = 0.f;
            }
            for (int c = lane; c < D; c += 32) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float e = __expf(sm.Gam[rr[u]][c] - sm.Gam[ii[u]][c]);
                    const float ke = sm.K[ii[u]][c] * e;
                    gg[u] += sm.K[rr[u]][c] * ke;
                    pp[u] += sm.Q[rr[u]][c] * ke;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    gg[u] += __shfl_xor_sync(0xffffffffu, gg[u], o);
                    pp[u] += __shfl_xor_sync(0xffffffffu, pp[u], o);
                }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (lane == u && p0 + u < NPAIR) {
                    const int r = rr[u], i = ii[u];
                    sm.G[r][i] = i < r ? gg[u] : 0.f;
                    sm.P[r][i] = pp[u];
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
            // ---- Y = V - Kt S0 (threads 0-255) and dU = Kb dS + P^T dO (threads 256-511),
            // each thread a tile of 2 rows x 2 columns ----
            {
                const bool du_half = t >= kThreads / 2;   // warp-uniform
                const int th = t & (kThreads / 2 - 1);
                const int jp = (th & 15) * 2, r2 = (th >> 4) * 2;
                const float(*A)[D] = du_half ? sm.Kb : sm.Kt;
                float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
                for (int c = 0; c < D; c += 4) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(&A[r2][c]);
                    const float4 x1 = *reinterpret_cast<const float4 *>(&A[r2 + 1][c]);
                    float b0[4], b1[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        b0[q2] = du_half ? sm.dS[c + q2][j0 + jp] : sm.S0[c + q2][jp];
                        b1[q2] = du_half ? sm.dS[c + q2][j0 + jp + 1] : sm.S0[c + q2][jp + 1];
                    }
                    a00 += x0.x * b0[0] + x0.y * b0[1] + x0.z * b0[2] + x0.w * b0[3];
                    a01 += x0.x * b1[0] + x0.y * b1[1] + x0.z * b1[2] + x0.w * b1[3];
                    a10 += x1.x * b0[0] + x1.y * b0[1] + x1.z * b0[2] + x1.w * b0[3];
                    a11 += x1.x * b1[0] + x1.y * b1[1] + x1.z * b1[2] + x1.w * b1[3];
                }
                if (!du_half) {
                    sm.Y[r2][jp] = sm.V[r2][jp] - a00;
                    sm.Y[r2][jp + 1] = sm.V[r2][jp + 1] - a01;
                    sm.Y[r2 + 1][jp] = sm.V[r2 + 1][jp] - a10;
                    sm.Y[r2 + 1][jp + 1] = sm.V[r2 + 1][jp + 1] - a11;
                } else {
                    for (int rp = r2; rp < C; ++rp) {   // P^T dO (P[rp][r] is 0 for rp < r)
                        const float p0v = sm.P[rp][r2], p1v = sm.P[rp][r2 + 1];
                        const float o0 = sm.dO[rp][jp], o1 = sm.dO[rp][jp + 1];
                        a00 += p0v * o0;
                        a01 += p0v * o1;
                        a10 += p1v * o0;
                        a11 += p1v * o1;
                    }
                    sm.dU[r2][jp] = a00;
                    sm.dU[r2][jp + 1] = a01;
                    sm.dU[r2 + 1][jp] = a10;
                    sm.dU[r2 + 1][jp + 1] = a11;
                }
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
                for (int j = 0; j < BV; j += 4) {
                    const float4 o4 = *reinterpret_cast<const float4 *>(&sm.dO[r][j]);
                    const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[i][j]);
                    const float4 d4 = *reinterpret_cast<const float4 *>(&sm.dU[r][j]);
                    sp += o4.x * u4.x + o4.y * u4.y + o4.z * u4.z + o4.w * u4.w;
                    st += d4.x * sm.Y[i][j] + d4.y * sm.Y[i][j + 1] + d4.z * sm.Y[i][j + 2] +
                          d4.w * sm.Y[i][j + 3];
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
            for (int j = 0; j < BV; j += 4) {
                float s0v[4], dsv[4];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                    s0v[q2] = sm.S0[oc][j + q2];
                    dsv[q2] = sm.dS[oc][j0 + j + q2];
                }
#pragma unroll
                for (int m = 0; m < RPT; ++m) {
                    const int r = or0 + RSTEP * m;
                    const float4 o4 = *reinterpret_cast<const float4 *>(&sm.dO[r][j]);
                    const float4 y4 = *reinterpret_cast<const float4 *>(&sm.dU[r][j]);
                    const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[r][j]);
                    aQt[m] += o4.x * s0v[0] + o4.y * s0v[1] + o4.z * s0v[2] + o4.w * s0v[3];
                    aKt[m] -= y4.x * s0v[0] + y4.y * s0v[1] + y4.z * s0v[2] + y4.w * s0v[3];
                    aKb[m] += u4.x * dsv[0] + u4.y * dsv[1] + u4.z * dsv[2] + u4.w * dsv[3];
                }
            }
            if (t < D) {
                float s = 0.f;
                for (int j = 0; j < BV; ++j) s += sm.dS[t][j0 + j] * sm.S0[t][j];
                sm.gsum[t] += s;
            }
            __syncthreads();
            // ---- dS <- diag(gC) dS + Qt^T dO - Kt^T dY on this block's columns,
            // each thread a tile of 4 channels x 2 columns (D / 4 x 16 threads:
            // all 512 for D = 128, warps 0-7 for D = 64) ----
            if (t < (D / 4) * 16) {
                const int jp = (t & 15) * 2, c4 = (t >> 4) * 4;
                float acc[4][2];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    acc[m][0] = sm.gC[c4 + m] * sm.dS[c4 + m][j0 + jp];
                    acc[m][1] = sm.gC[c4 + m] * sm.dS[c4 + m][j0 + jp + 1];
                }
                for (int r = 0; r < C; ++r) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&sm.Qt[r][c4]);
                    const float4 kv = *reinterpret_cast<const float4 *>(&sm.Kt[r][c4]);
                    const float o0 = sm.dO[r][jp], o1 = sm.dO[r][jp + 1];
                    const float y0 = sm.dU[r][jp], y1 = sm.dU[r][jp + 1];
                    const float qa[4] = {qv.x, qv.y, qv.z, qv.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        acc[m][0] += qa[m] * o0 - ka[m] * y0;
                        acc[m][1] += qa[m] * o1 - ka[m] * y1;
                    }
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    sm.dS[c4 + m][j0 + jp] = acc[m][0];
                    sm.dS[c4 + m][j0 + jp + 1] = acc[m][1];
                }
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
