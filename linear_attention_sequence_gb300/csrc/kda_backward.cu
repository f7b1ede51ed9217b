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
// gamma = e^Gamma, gC its last row):
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
// Every decay factor is taken against the chunk midpoint Gamma_15 ("Understanding
// Kimi K3's Attention", log-decay bound: |Gamma_r - Gamma_15| <= 16 x 5 = 80 inside a
// 32-token chunk, so each factor stays in the fp32 range): with Q1 = q e^{Gamma -
// Gamma_15}, A1 = k e^{Gamma - Gamma_15} and B1 = k e^{Gamma_15 - Gamma}, G = A1 B1^T and
// P = Q1 B1^T are plain products, the pairwise gradient terms are R1 = dP B1,
// R2 = dG B1, R3 = dG^T A1 + dP^T Q1, and Qt, Kt, Kb differ from Q1, A1, B1 by the
// per-channel factors e^{Gamma_15} and e^{Gamma_C - Gamma_15}, folded into the operands
// and results.
//
// One CTA of 512 threads per (sequence, head).  The adjoint dS (d x d) stays in
// shared memory for the whole sequence; the value axis is processed in blocks of
// 32 columns, each block's contributions to the cross-column sums (dP, dT,
// dbeta, dQt, dKt, dKb) accumulated over the blocks.  fp32 throughout.

#include "kda_common.cuh"

// Device-side argument check of the backward: set when a chunk-state row the
// gradients need lies past chunk_capacity (only checkable on the device when the
// sequence lengths come from cu_seqlens).
__device__ unsigned int g_kda_bwd_status;

namespace {

constexpr int C = 32;          // tokens per chunk (the checkpoint interval)
constexpr int BV = 32;         // value columns per block
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

template <int D>
struct BwdSmem {
    float dS[D][D + 4];        // adjoint of the state at the end of the current chunk
    float S0[D][BV + 4];       // e^{Gamma_15} . S0 (the chunk's start state), one column block
    float Gam[C][D + 4];       // Gamma
    // decay factored around the chunk midpoint (|Gamma - Gamma_15| <= 80: no factor
    // leaves the fp32 range): q e^{Gamma - Gamma_15}, k e^{Gamma - Gamma_15}, k e^{Gamma_15 - Gamma}
    float Q1[C][D + 4], A1[C][D + 4], B1[C][D + 4];
    // rows of 36 floats (16-byte aligned: read four columns at a time); Y keeps 33
    // (read down its columns)
    float V[C][BV + 4], dO[C][BV + 4], U[C][BV + 4], dU[C][BV + 4];
    float Y[C][BV + 1];
    float G[C][C + 4], P[C][C + 4], dP[C][C + 4];   // G holds dG after the column blocks
    float T[C][C + 1], dT[C][C + 1];
    float beta[C], dbeta[C];
    float e15[D], fC[D], gC[D], gsum[D];   // e^{Gamma_15}, e^{Gamma_C - Gamma_15}, e^{Gamma_C}, sum dS . S0
};

template <typename IN_T, typename OUT_T, int D>
__global__ void __launch_bounds__(kThreads, 1)
kda_backward_kernel(const IN_T *__restrict__ q, const IN_T *__restrict__ k,
                    const IN_T *__restrict__ v, const float *__restrict__ g,
                    const float *__restrict__ beta, const float *__restrict__ init_state,
                    const int32_t *__restrict__ cu, const float *__restrict__ chunk_states,
                    int64_t chunk_capacity, const IN_T *__restrict__ d_out,
                    const float *__restrict__ d_final, OUT_T *__restrict__ dq,
                    OUT_T *__restrict__ dk, OUT_T *__restrict__ dv, float *__restrict__ dg,
                    float *__restrict__ dbeta, float *__restrict__ d_init, int H, int64_t total,
                    int64_t seq_len) {
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
    // 2 x 2 tiles of a C x C or C x BV product, one half of the block per product
    const bool hi_half = t >= kThreads / 2;    // warp-uniform
    const int th = t & (kThreads / 2 - 1);
    const int tcol = (th & 15) * 2, trow = (th >> 4) * 2;

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
        // a needed row the caller did not provide: the gradients are wrong, and
        // kda_get_last_device_error reports KDA_ERR_INVALID_ARGUMENT
        if (ch > 0 && S0g == nullptr && t == 0) atomicOr(&g_kda_bwd_status, kda::kBwdMissingState);
        __syncthreads();   // the previous chunk is done with every buffer

        // ---- load q (into Q1), k (into A1), g (into Gam); rows past the end are 0 ----
        for (int idx = t; idx < C * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < L) {
                const int64_t off = (t0 + r) * rowK + (int64_t)h * D + c;
                qv = kda::ld_elem(q + off);
                kv = kda::ld_elem(k + off);
                gv = g[off];
            }
            sm.Q1[r][c] = qv;
            sm.A1[r][c] = kv;
            sm.Gam[r][c] = gv;
        }
        if (t < C) {
            sm.beta[t] = t < L ? beta[(t0 + t) * H + h] : 0.f;
            sm.dbeta[t] = 0.f;
        }
        __syncthreads();
        // ---- Gamma (running sum per channel) and the per-channel factors ----
        if (t < D) {
            float run = 0.f, g15 = 0.f;
            for (int r = 0; r < C; ++r) {
                run += sm.Gam[r][t];
                sm.Gam[r][t] = run;
                if (r == 15) g15 = run;
            }
            sm.e15[t] = __expf(g15);
            sm.fC[t] = __expf(run - g15);
            sm.gC[t] = __expf(run);
            sm.gsum[t] = 0.f;
        }
        __syncthreads();
        // ---- decay-factored copies ----
        for (int idx = t; idx < C * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            const float d1 = sm.Gam[r][c] - sm.Gam[15][c];
            const float kv = sm.A1[r][c];
            sm.Q1[r][c] *= __expf(d1);
            sm.A1[r][c] = kv * __expf(d1);
            sm.B1[r][c] = kv * __expf(-d1);
        }
        __syncthreads();
        // ---- G = A1 B1^T (strict) on one half, P = Q1 B1^T (inclusive) on the other ----
        {
            const float(*Am)[D + 4] = hi_half ? sm.Q1 : sm.A1;
            float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
            for (int c = 0; c < D; c += 4) {
                const float4 x0 = *reinterpret_cast<const float4 *>(&Am[trow][c]);
                const float4 x1 = *reinterpret_cast<const float4 *>(&Am[trow + 1][c]);
                const float4 y0 = *reinterpret_cast<const float4 *>(&sm.B1[tcol][c]);
                const float4 y1 = *reinterpret_cast<const float4 *>(&sm.B1[tcol + 1][c]);
                a00 += x0.x * y0.x + x0.y * y0.y + x0.z * y0.z + x0.w * y0.w;
                a01 += x0.x * y1.x + x0.y * y1.y + x0.z * y1.z + x0.w * y1.w;
                a10 += x1.x * y0.x + x1.y * y0.y + x1.z * y0.z + x1.w * y0.w;
                a11 += x1.x * y1.x + x1.y * y1.y + x1.z * y1.z + x1.w * y1.w;
            }
            const float av[2][2] = {{a00, a01}, {a10, a11}};
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    const int r = trow + u, i = tcol + w2;
                    if (hi_half) sm.P[r][i] = i <= r ? av[u][w2] : 0.f;
                    else sm.G[r][i] = i < r ? av[u][w2] : 0.f;
                }
        }
        for (int idx = t; idx < C * C; idx += kThreads) {
            const int r = idx / C, i = idx % C;
            sm.dP[r][i] = 0.f;
            sm.dT[r][i] = 0.f;
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
        // e^{Gamma_15}-scaled accumulators: aQ = e15 . dQt, aK = e15 . dKt, aB = dKb
        float aQ[RPT], aK[RPT], aB[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) aQ[m] = aK[m] = aB[m] = 0.f;

        for (int j0 = 0; j0 < D; j0 += BV) {
            __syncthreads();   // T is ready; the previous block is done with its buffers
            // ---- this block of e15 . S0, V and dO ----
            for (int idx = t; idx < D * BV; idx += kThreads) {
                const int c = idx / BV, j = idx % BV;
                sm.S0[c][j] = S0g ? sm.e15[c] * S0g[(int64_t)c * D + j0 + j] : 0.f;
            }
            for (int idx = t; idx < C * BV; idx += kThreads) {
                const int r = idx / BV, j = idx % BV;
                const int64_t off = (t0 + r) * rowK + (int64_t)h * D + j0 + j;
                sm.V[r][j] = r < L ? kda::ld_elem(v + off) : 0.f;
                sm.dO[r][j] = r < L ? kda::ld_elem(d_out + off) : 0.f;
            }
            __syncthreads();
            // ---- Y = V - A1 (e15 . S0) on one half, dU = B1 (fC . dS) + P^T dO on the other ----
            {
                const float(*Am)[D + 4] = hi_half ? sm.B1 : sm.A1;
                float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
                for (int c = 0; c < D; c += 4) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(&Am[trow][c]);
                    const float4 x1 = *reinterpret_cast<const float4 *>(&Am[trow + 1][c]);
                    float b0[4], b1[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {   // two adjacent columns per 8-byte load
                        if (hi_half) {
                            const float f = sm.fC[c + q2];
                            const float2 d2 = *reinterpret_cast<const float2 *>(&sm.dS[c + q2][j0 + tcol]);
                            b0[q2] = f * d2.x;
                            b1[q2] = f * d2.y;
                        } else {
                            const float2 s2 = *reinterpret_cast<const float2 *>(&sm.S0[c + q2][tcol]);
                            b0[q2] = s2.x;
                            b1[q2] = s2.y;
                        }
                    }
                    a00 += x0.x * b0[0] + x0.y * b0[1] + x0.z * b0[2] + x0.w * b0[3];
                    a01 += x0.x * b1[0] + x0.y * b1[1] + x0.z * b1[2] + x0.w * b1[3];
                    a10 += x1.x * b0[0] + x1.y * b0[1] + x1.z * b0[2] + x1.w * b0[3];
                    a11 += x1.x * b1[0] + x1.y * b1[1] + x1.z * b1[2] + x1.w * b1[3];
                }
                if (!hi_half) {
                    sm.Y[trow][tcol] = sm.V[trow][tcol] - a00;
                    sm.Y[trow][tcol + 1] = sm.V[trow][tcol + 1] - a01;
                    sm.Y[trow + 1][tcol] = sm.V[trow + 1][tcol] - a10;
                    sm.Y[trow + 1][tcol + 1] = sm.V[trow + 1][tcol + 1] - a11;
                } else {
                    for (int rp = trow; rp < C; ++rp) {   // P^T dO (P[rp][r] is 0 for rp < r)
                        const float p0v = sm.P[rp][trow], p1v = sm.P[rp][trow + 1];
                        const float o0 = sm.dO[rp][tcol], o1 = sm.dO[rp][tcol + 1];
                        a00 += p0v * o0;
                        a01 += p0v * o1;
                        a10 += p1v * o0;
                        a11 += p1v * o1;
                    }
                    sm.dU[trow][tcol] = a00;
                    sm.dU[trow][tcol + 1] = a01;
                    sm.dU[trow + 1][tcol] = a10;
                    sm.dU[trow + 1][tcol + 1] = a11;
                }
            }
            __syncthreads();
            // ---- U = T diag(beta) Y; dB = T^T dU (kept in registers) ----
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
            // ---- aQ += dO (e15 S0)^T, aK -= dY (e15 S0)^T, aB += U dS^T (dS before the
            // update below); the gamma_last term sum_j dS . (e15 S0) ----
            for (int j = 0; j < BV; j += 4) {
                const float4 s4 = *reinterpret_cast<const float4 *>(&sm.S0[oc][j]);
                const float4 d4 = *reinterpret_cast<const float4 *>(&sm.dS[oc][j0 + j]);
#pragma unroll
                for (int m = 0; m < RPT; ++m) {
                    const int r = or0 + RSTEP * m;
                    const float4 o4 = *reinterpret_cast<const float4 *>(&sm.dO[r][j]);
                    const float4 y4 = *reinterpret_cast<const float4 *>(&sm.dU[r][j]);
                    const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[r][j]);
                    aQ[m] += o4.x * s4.x + o4.y * s4.y + o4.z * s4.z + o4.w * s4.w;
                    aK[m] -= y4.x * s4.x + y4.y * s4.y + y4.z * s4.z + y4.w * s4.w;
                    aB[m] += u4.x * d4.x + u4.y * d4.y + u4.z * d4.z + u4.w * d4.w;
                }
            }
            if (t < D) {
                float s = 0.f;
                for (int j = 0; j < BV; j += 4) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(&sm.S0[t][j]);
                    const float4 d4 = *reinterpret_cast<const float4 *>(&sm.dS[t][j0 + j]);
                    s += s4.x * d4.x + s4.y * d4.y + s4.z * d4.z + s4.w * d4.w;
                }
                sm.gsum[t] += s;
            }
            __syncthreads();
            // ---- dS <- diag(gC) dS + diag(e15) (Q1^T dO - A1^T dY) on this block's columns,
            // each thread a tile of 4 channels x 2 columns (D / 4 x 16 threads:
            // all 512 for D = 128, warps 0-7 for D = 64) ----
            if (t < (D / 4) * 16) {
                const int jp = (t & 15) * 2, c4 = (t >> 4) * 4;
                float acc[4][2];
#pragma unroll
                for (int m = 0; m < 4; ++m) acc[m][0] = acc[m][1] = 0.f;
                for (int r = 0; r < C; ++r) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&sm.Q1[r][c4]);
                    const float4 kv = *reinterpret_cast<const float4 *>(&sm.A1[r][c4]);
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
                    const int c = c4 + m;
                    sm.dS[c][j0 + jp] = sm.gC[c] * sm.dS[c][j0 + jp] + sm.e15[c] * acc[m][0];
                    sm.dS[c][j0 + jp + 1] = sm.gC[c] * sm.dS[c][j0 + jp + 1] + sm.e15[c] * acc[m][1];
                }
            }
        }
        __syncthreads();
        // ---- dA = -T^T tril_s(dT) T^T (strict lower): M1 = tril_s(dT) T^T into Y's space ----
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
            sm.G[r][i] = sm.beta[r] * da;   // dG (this thread read G[r][i] above)
            if (lane == 0) sm.dbeta[r] += gb;
        }
        __syncthreads();
        // ---- pairwise terms R1 = dP B1, R2 = dG B1, R3 = dG^T A1 + dP^T Q1, then the
        // gradients of the owned (x, c):
        //   dq = e^{Gamma - Gamma_15} (aQ + R1)
        //   dk = e^{Gamma - Gamma_15} (aK + R2) + e^{Gamma_C - Gamma} aB + e^{Gamma_15 - Gamma} R3
        //   dGamma = Q1 (aQ + R1) + A1 (aK + R2) - B1 (fC aB + R3) ----
        float R1[RPT], R2[RPT], R3[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) R1[m] = R2[m] = R3[m] = 0.f;
        for (int i = 0; i < C; i += 4) {
            float bq[4], aq[4], qq[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                bq[q2] = sm.B1[i + q2][oc];
                aq[q2] = sm.A1[i + q2][oc];
                qq[q2] = sm.Q1[i + q2][oc];
            }
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int x = or0 + RSTEP * m;
                const float4 p4 = *reinterpret_cast<const float4 *>(&sm.dP[x][i]);
                const float4 g4 = *reinterpret_cast<const float4 *>(&sm.G[x][i]);
                R1[m] += p4.x * bq[0] + p4.y * bq[1] + p4.z * bq[2] + p4.w * bq[3];
                R2[m] += g4.x * bq[0] + g4.y * bq[1] + g4.z * bq[2] + g4.w * bq[3];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2)
                    R3[m] += sm.G[i + q2][x] * aq[q2] + sm.dP[i + q2][x] * qq[q2];
            }
        }
        float dgam[RPT];
        float kbk = 0.f;   // this thread's part of sum_i fC aB_i B1_i (the gamma_last term)
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int x = or0 + RSTEP * m, c = oc;
            const float gx = sm.Gam[x][c], g15 = sm.Gam[15][c];
            const float ex = __expf(gx - g15), ix = __expf(g15 - gx);
            const float sq = aQ[m] + R1[m], sk = aK[m] + R2[m];
            const float fb = sm.fC[c] * aB[m];
            if (x < L) {
                const int64_t off = (t0 + x) * rowK + (int64_t)h * D + c;
                kda::st_elem(dq + off, ex * sq);
                kda::st_elem(dk + off, ex * sk + __expf(sm.Gam[C - 1][c] - gx) * aB[m] + ix * R3[m]);
            }
            const float b1 = sm.B1[x][c];
            dgam[m] = sm.Q1[x][c] * sq + sm.A1[x][c] * sk - b1 * (fb + R3[m]);
            kbk += fb * b1;
        }
        __syncthreads();   // every read of Q1 / A1 above is done: reuse them
#pragma unroll
        for (int m = 0; m < RPT; ++m) sm.A1[or0 + RSTEP * m][oc] = dgam[m];
        sm.Q1[or0][oc] = kbk;   // one partial per (row group, channel)
        __syncthreads();
        // ---- dg = reverse running sum of dGamma over the chunk (thread per channel) ----
        if (t < D) {
            float last = sm.fC[t] * sm.gsum[t];
            for (int r0 = 0; r0 < RSTEP; ++r0) last += sm.Q1[r0][t];
            float run = 0.f;
            for (int r = C - 1; r >= 0; --r) {
                run += sm.A1[r][t] + (r == C - 1 ? last : 0.f);
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
    // bf16 inputs at d = 128: the tensor-core kernel (kda_backward_tc.cu)
    if (kda_backward_tc_supported(P, q, k, v, g, d_out))
        return kda_launch_backward_tc(P, q, k, v, g, beta, init_state, cu, chunk_states, chunk_capacity,
                                      d_out, d_final, dq, dk, dv, dg, dbeta, d_init, stream);
    if (P.dk == 128)
        return dispatch<128>(P, q, k, v, g, beta, init_state, cu, chunk_states, chunk_capacity, d_out, d_final, dq,
                             dk, dv, dg, dbeta, d_init, stream);
    return dispatch<64>(P, q, k, v, g, beta, init_state, cu, chunk_states, chunk_capacity, d_out, d_final, dq, dk,
                        dv, dg, dbeta, d_init, stream);
}

// Read and clear the backward's status word (ORed into *status).
cudaError_t kda_bwd_read_status(unsigned *status) {
    unsigned st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&st, g_kda_bwd_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_kda_bwd_status, &zero, sizeof(unsigned));
    *status |= st;
    return e;
}
