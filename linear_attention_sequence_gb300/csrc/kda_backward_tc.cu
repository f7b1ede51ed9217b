// kda_backward_tc.cu -- gradients of the chunked KDA prefill on the tensor
// cores (sm_103a, tcgen05), bf16 inputs, d_k = d_v = 128.
//
// "Hybrid Attention", section "But isn't a recurrent update sequential?": the
// chunkwise computation is trained by comparing its outputs and gradients with
// the recurrent version.  The algebra is the one of the CUDA-core backward
// (kda_backward.cu): per chunk (C = 32 tokens, walked in reverse, Gamma the
// running sum of g inside the chunk, S0 the chunk's start state from the
// forward's checkpoints, dS the adjoint of its end state),
//
//   forward again:  G = A1 B1^T (strict), P = Q1 B1^T (inclusive),
//                   T = (I + diag(beta) G)^{-1},  Y = V - Kt S0,  U = T diag(beta) Y
//   backward:       dU = Kb dS + P^T dO,  dB = T^T dU,  dY = diag(beta) dB (= dV),
//                   dP = tril(dO U^T),  dT = dU (beta Y)^T (strict),
//                   dA = -T^T dT T^T,  dG = diag(beta) dA,
//                   dbeta = rowsum(dB . Y) + rowsum(dA . G),
//                   aQ = dO (e15 S0)^T,  aK = -dY (e15 S0)^T,  aB = U dS^T,
//                   R1 = dP B1,  R2 = dG B1,  R3 = dG^T A1 + dP^T Q1,
//                   dS0 = diag(gamma_C) dS + diag(e15) (Q1^T dO - A1^T dY),
//
// with the decay factored around the chunk midpoint (|Gamma_r - Gamma_15| <= 80
// by the log-decay bound of "Understanding Kimi K3's Attention"): Q1 = q
// e^{Gamma - Gamma_15}, A1 = k e^{Gamma - Gamma_15}, B1 = k e^{Gamma_15 - Gamma},
// Kt = k e^{Gamma}, Kb = k e^{Gamma_C - Gamma}, e15 = e^{Gamma_15}.
//
// One CTA of 512 threads per (sequence, head).  The adjoint stays in tensor
// memory as dS^T (lane = value j, column = key channel c).  Every product with
// a 128-long side is one tcgen05.mma kind::tf32 group with M = 128 (values or
// key channels) and fp32 accumulation; its operands are written by the threads
// as K-major SW128 tf32 blocks in shared memory, or read from tensor memory.
// The 32 x 32 pieces (G, P, the solve, dP, dT, dA) run on the CUDA cores.  The
// phases of a chunk run one after another, separated by block barriers.

#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"
#include "kda_chunk_ops.cuh"

__device__ unsigned int g_kda_bwdtc_status;   // bounded waits that gave up; missing state rows

namespace {

using namespace sm100;
using namespace kda_chunk;

constexpr int C = 32;
constexpr int D = 128;
constexpr int kThreads = 512;
constexpr uint32_t kPollLimit = 1u << 23;

// Shared memory (byte offsets from a 1024-aligned base).
//   TILE   TMA tiles of the chunk: q, k, v, dO (bf16, 8 KB each), g (fp32, 16 KB;
//          Gamma in place).  After the preparation the q and k tiles hold the
//          operands T diag(beta), T^T, P^T (4 KB each), later U (16 KB).
//   STG    64 KB staging of 128-row operands: S0^T (rows j), then the fp32
//          copies of U, dU and Y, then S0 (rows c), then dS (rows c).
//   OPA    Kt rows (16 KB) and Kb rows (16 KB); later [dO ; -dY] (32 KB), then
//          [dP ; dG] (8 KB) and the B operand of R3 (8 KB).
//   OPQA   [Q1^T | A1^T] (rows c, K = 64, 32 KB).   OPB1T  B1^T (rows c, 16 KB).
constexpr uint32_t T_Q = 0, T_K = 8192, T_V = 16384, T_DO = 24576, T_G = 32768;
constexpr uint32_t O_TB = 0, O_TT = 4096, O_PT = 8192, O_U = 0;
constexpr uint32_t STG = 49152;
constexpr uint32_t OPA = STG + 65536;          // 114688
constexpr uint32_t O_KT = OPA, O_KB = OPA + 16384, O_OY = OPA, O_PG = OPA, O_R3B = OPA + 8192;
constexpr uint32_t OPQA = OPA + 32768;         // 147456
constexpr uint32_t OPB1T = OPQA + 32768;       // 180224
constexpr uint32_t SMALL = OPB1T + 16384;      // 196608
constexpr int LDS32 = C + 1;                   // row length of the 32 x 32 fp32 arrays

struct Small {
    float G[C][LDS32], P[C][LDS32], T[C][LDS32], dP[C][LDS32], dT[C][LDS32];
    float beta[C], dbeta[C], red[4][C];
    float e15[D], fC[D], gC[D], gsum[D];
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kSmem = SMALL + sizeof(Small) + 1024;
static_assert(kSmem <= 232448, "shared memory budget");
// fp32 staging of U, dU and Y inside STG (rows of 132 floats)
constexpr int LU = D + 4;
static_assert(3 * C * LU * 4 <= 65536, "U, dU, Y staging fits");

// Tensor-memory columns (lanes = value j for dS^T, X, Y, U, dU, dB, dO^T, dS_new;
// lanes = key channel c for aQ|aK, aB, R1|R2, R3).
constexpr uint32_t TM_DS = 0, TM_DN = 128, TM_X = 256, TM_Y = 288, TM_U = 320, TM_DU = 352,
                   TM_DB = 384, TM_DOT = 416, TM_R3 = 480;
constexpr uint32_t TM_AQK = 256, TM_AB = 320, TM_R12 = 352;

__device__ __forceinline__ uint32_t off_bf16(int r, int c) {   // TMA tile (SW128), bf16
    return (uint32_t)((c >> 6) * 4096 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ uint32_t off_f32(int r, int c) {    // TMA tile (SW128), fp32
    return (uint32_t)((c >> 5) * 4096 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + ((c & 3) << 2));
}
__device__ __forceinline__ float lds_bf16(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
// One K-major SW128 tf32 element store (row `row` of an operand with `rows` rows).
__device__ __forceinline__ void st_op(unsigned char *base, int rows, int row, int k, float x) {
    *reinterpret_cast<float *>(base + sw_off(rows, row, k)) = to_tf32(x);
}

// One MMA group: D[m][n] (+)= sum_k A[m][k] B[n][k], A and B K-major SW128 in
// shared memory (SS) with K-blocks of `akb` and `bkb` bytes; `ksteps` steps of 8.
__device__ __forceinline__ void mma_ss_group(uint32_t d, const unsigned char *a, uint32_t akb,
                                             const unsigned char *b, uint32_t bkb, int ksteps, int n,
                                             bool acc) {
    const uint64_t da = sdesc_sw128(smem_u32(a)), db = sdesc_sw128(smem_u32(b));
    for (int kk = 0; kk < ksteps; ++kk)
        mma_tf32_ss(d, da + (uint64_t)(((kk >> 2) * akb + (kk & 3) * 32) >> 4),
                    db + (uint64_t)(((kk >> 2) * bkb + (kk & 3) * 32) >> 4), idesc_tf32(128, n),
                    (acc || kk > 0) ? 1u : 0u);
}
// The same with A in tensor memory (8 columns per K step).
__device__ __forceinline__ void mma_ts_group(uint32_t d, uint32_t a, const unsigned char *b,
                                             uint32_t bkb, int ksteps, int n, bool acc) {
    const uint64_t db = sdesc_sw128(smem_u32(b));
    for (int kk = 0; kk < ksteps; ++kk)
        mma_tf32_ts(d, a + 8 * kk, db + (uint64_t)(((kk >> 2) * bkb + (kk & 3) * 32) >> 4),
                    idesc_tf32(128, n), (acc || kk > 0) ? 1u : 0u);
}

template <typename OUT_T>
__global__ void __launch_bounds__(kThreads, 1)
kda_backward_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_g, const float *__restrict__ beta,
                       const float *init_state, const int32_t *__restrict__ cu,
                       const float *__restrict__ chunk_states, int64_t chunk_capacity,
                       const float *__restrict__ d_final, OUT_T *__restrict__ dq,
                       OUT_T *__restrict__ dk, OUT_T *__restrict__ dv, float *__restrict__ dg,
                       float *__restrict__ dbeta, float *d_init, int H, int64_t total,
                       int64_t seq_len) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Small &sm = *reinterpret_cast<Small *>(base + SMALL);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int jl = 32 * q4 + lane;           // the TMEM lane (value or key channel) of this thread
    const int slice = warp >> 2;             // which quarter of the columns (0..3)
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);
    const int nchunks = (int)((b - a + C - 1) / C);
    const int64_t rowK = (int64_t)H * D;
    const int64_t sdd = (int64_t)D * D;
    const int64_t soff = ((int64_t)n * H + h) * sdd;
    const int64_t ck0 = kda::ckpt_first_row(cu, n, total, seq_len, C);

    if (t == 0) {
        mbar_init(&sm.tma_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
        sm.abort = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm.tmem_base;
    const uint32_t tl = tb + lane_off;
    uint32_t tma_par = 0, mma_par = 0;

    // MMA groups are issued and awaited by thread 0; the barrier releases the rest.
    auto mma_wait = [&]() {
        if (t == 0) {
            mma_commit(&sm.mma_bar);
            if (!mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit)) {
                sm.abort = 1;
                atomicOr(&g_kda_bwdtc_status, 0x400u);
            }
        }
        mma_par ^= 1u;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    // dS^T <- d_final^T (lane j holds column j of dS)
    if (slice == 0) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = d_final ? d_final[soff + (int64_t)(c0 + i) * D + jl] : 0.f;
            tmem_st32(tl + TM_DS + c0, x);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    for (int ch = nchunks - 1; ch >= 0; --ch) {
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;
        const int64_t t0 = a + (int64_t)ch * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        const int64_t crow = ck0 + ch - 1;
        const float *S0g = ch == 0 ? (init_state ? init_state + soff : nullptr)
                           : (chunk_states && crow < chunk_capacity) ? chunk_states + (crow * H + h) * sdd
                                                                     : nullptr;
        if (ch > 0 && S0g == nullptr && t == 0) atomicOr(&g_kda_bwdtc_status, kda::kBwdMissingState);

        // ---- phase 0: the chunk's tiles by TMA; beta ----
        if (t == 0) {
            mbar_arrive_expect_tx(&sm.tma_bar, 4 * 8192 + 16384);
            tma_load_3d(base + T_Q, &tm_q, &sm.tma_bar, 0, (int)t0, 2 * h);
            tma_load_3d(base + T_K, &tm_k, &sm.tma_bar, 0, (int)t0, 2 * h);
            tma_load_3d(base + T_V, &tm_v, &sm.tma_bar, 0, (int)t0, 2 * h);
            tma_load_3d(base + T_DO, &tm_do, &sm.tma_bar, 0, (int)t0, 2 * h);
            tma_load_3d(base + T_G, &tm_g, &sm.tma_bar, 0, (int)t0, 4 * h);
        }
        if (t < C) {
            sm.beta[t] = t < L ? beta[(t0 + t) * H + h] : 0.f;
            sm.dbeta[t] = 0.f;
        }
        if (t == 0 && !mbar_wait_bounded(&sm.tma_bar, tma_par, kPollLimit)) {
            sm.abort = 1;
            atomicOr(&g_kda_bwdtc_status, 0x800u);
        }
        tma_par ^= 1u;
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 1: threads 0-127 (channel c): Gamma and the decay-weighted
        // operands; threads 128-383: S0^T into STG (rows j, K = c) ----
        if (t < D) {
            const int c = t;
            float gam[C];
#pragma unroll
            for (int r = 0; r < C; ++r)
                gam[r] = r < L ? *reinterpret_cast<const float *>(base + T_G + off_f32(r, c)) : 0.f;
#pragma unroll
            for (int r = 1; r < C; ++r) gam[r] += gam[r - 1];
#pragma unroll
            for (int r = 0; r < C; ++r) *reinterpret_cast<float *>(base + T_G + off_f32(r, c)) = gam[r];
            const float g15 = gam[15], gl = gam[C - 1];
            sm.e15[c] = __expf(g15);
            sm.fC[c] = __expf(gl - g15);
            sm.gC[c] = __expf(gl);
            sm.gsum[c] = 0.f;
            float q1[4], a1[4], b1[4];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float qv = 0.f, kv = 0.f;
                if (r < L) {
                    qv = lds_bf16(base + T_Q + off_bf16(r, c));
                    kv = lds_bf16(base + T_K + off_bf16(r, c));
                }
                const float x = gam[r] - g15;
                const float e1 = __expf(x), inv = __expf(-x);
                st_op(base + O_KT, 32, r, c, kv * __expf(gam[r]));    // Kt = k e^{Gamma}
                st_op(base + O_KB, 32, r, c, kv * __expf(gl - gam[r]));   // Kb = k e^{Gamma_C - Gamma}
                q1[r & 3] = to_tf32(qv * e1);
                a1[r & 3] = to_tf32(kv * e1);
                b1[r & 3] = to_tf32(kv * inv);
                if ((r & 3) == 3) {
                    const uint32_t pos = (uint32_t)((((r >> 2) ^ (c & 7)) & 7) << 4);
                    *reinterpret_cast<float4 *>(base + OPQA + c * 128 + pos) = make_float4(q1[0], q1[1], q1[2], q1[3]);
                    *reinterpret_cast<float4 *>(base + OPQA + 16384 + c * 128 + pos) =
                        make_float4(a1[0], a1[1], a1[2], a1[3]);
                    *reinterpret_cast<float4 *>(base + OPB1T + c * 128 + pos) = make_float4(b1[0], b1[1], b1[2], b1[3]);
                }
            }
        } else if (t < D + 256) {
            const int u = t - D, j = u & 127, half = u >> 7;   // channels [64 half, 64 half + 64)
            float x[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) x[i] = S0g ? S0g[(int64_t)(64 * half + i) * D + j] : 0.f;
#pragma unroll
            for (int i = 0; i < 64; ++i) st_op(base + STG, 128, j, 64 * half + i, x[i]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- phase 2: G = A1 B1^T (strict) and P = Q1 B1^T (inclusive) from the
        // transposed operand blocks (threads: product, 2 x 2 tile) ----
        {
            const int prod = t >> 8, th = t & 255;
            const int r0 = (th >> 4) * 2, i0 = (th & 15) * 2;
            const unsigned char *Am = base + OPQA + (prod == 0 ? 16384 : 0);   // A1^T or Q1^T
            float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll 4
            for (int c = 0; c < D; ++c) {
                const float2 x = *reinterpret_cast<const float2 *>(Am + sw_off(128, c, r0));
                const float2 y = *reinterpret_cast<const float2 *>(base + OPB1T + sw_off(128, c, i0));
                a00 += x.x * y.x;
                a01 += x.x * y.y;
                a10 += x.y * y.x;
                a11 += x.y * y.y;
            }
            const float av[2][2] = {{a00, a01}, {a10, a11}};
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2)
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    const int r = r0 + u2, i = i0 + w2;
                    if (prod == 0) sm.G[r][i] = i < r ? av[u2][w2] : 0.f;
                    else sm.P[r][i] = i <= r ? av[u2][w2] : 0.f;
                }
        }
        __syncthreads();
        // T = (I + diag(beta) G)^{-1}: lane j solves column j (warp 0); warps 4-7:
        // dO^T into tensor memory (lane j, column r)
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
        } else if (warp >= 4 && warp < 8) {
            float x[32];
#pragma unroll
            for (int r = 0; r < C; ++r) x[r] = r < L ? lds_bf16(base + T_DO + off_bf16(r, jl)) : 0.f;
            tmem_st32(tl + TM_DOT, x);
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // T diag(beta), T^T and P^T as 32-row operands (in the q tile)
        for (int idx = t; idx < C * C; idx += kThreads) {
            const int r = idx >> 5, i = idx & 31;
            st_op(base + O_TB, 32, r, i, sm.T[r][i] * sm.beta[i]);
            st_op(base + O_TT, 32, r, i, sm.T[i][r]);
            st_op(base + O_PT, 32, r, i, sm.P[i][r]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- phase 3: X = S0^T Kt^T (Y = V - X), dU^T = dS^T Kb^T + dO^T P ----
        if (t == 0) {
            tc_fence_after();
            mma_ss_group(tb + TM_X, base + STG, 16384, base + O_KT, 4096, 16, 32, false);
            mma_ts_group(tb + TM_DU, tb + TM_DS, base + O_KB, 4096, 16, 32, false);
            mma_ts_group(tb + TM_DU, tb + TM_DOT, base + O_PT, 4096, 4, 32, true);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 4: Y^T = V^T - X into tensor memory; U^T = Y^T (T diag beta)^T,
        // dB^T = dU^T T ----
        if (warp < 4) {
            float x[32];
            tmem_ld32(tl + TM_X, x);
#pragma unroll
            for (int r = 0; r < C; ++r) x[r] = r < L ? lds_bf16(base + T_V + off_bf16(r, jl)) - x[r] : 0.f;
            tmem_st32(tl + TM_Y, x);
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        if (t == 0) {
            tc_fence_after();
            mma_ts_group(tb + TM_U, tb + TM_Y, base + O_TB, 4096, 4, 32, false);
            mma_ts_group(tb + TM_DB, tb + TM_DU, base + O_TT, 4096, 4, 32, false);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 5 (warps 0-3, lane j): dV = dY = diag(beta) dB; the dB . Y row
        // sums; -dY^T into tensor memory; U, dU, Y (fp32, STG) and the operands
        // [dO ; -dY] (rows, K = j) and U (rows, K = j) ----
        if (warp < 4) {
            float y[32], x[32];
            tmem_ld32(tl + TM_DB, x);
            tmem_ld32(tl + TM_Y, y);
            float *sY = reinterpret_cast<float *>(base + STG) + 2 * C * LU;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float dy = sm.beta[r] * x[r];
                if (r < L) kda::st_elem(dv + (t0 + r) * rowK + (int64_t)h * D + jl, dy);
                sY[r * LU + jl] = y[r];
                st_op(base + O_OY, 64, 32 + r, jl, -dy);
                x[r] *= y[r];          // dB . Y
                y[r] = -dy;
            }
            tmem_st32(tl + TM_DOT + 32, y);
            // row sums of dB . Y over j: reduce-scatter in the warp, then the four warps
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
                const bool up = (lane & sh) != 0;
#pragma unroll
                for (int i = 0; i < sh; ++i) {
                    const float send = up ? x[i] : x[i + sh];
                    const float keep = up ? x[i + sh] : x[i];
                    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
                }
            }
            sm.red[q4][lane] = x[0];
            tmem_wait_st();
        } else if (warp < 8) {
            float x[32];
            tmem_ld32(tl + TM_U, x);
            float *sU = reinterpret_cast<float *>(base + STG);
#pragma unroll
            for (int r = 0; r < C; ++r) {
                sU[r * LU + jl] = x[r];
                st_op(base + O_U, 32, r, jl, x[r]);
            }
        } else if (warp < 12) {
            float x[32];
            tmem_ld32(tl + TM_DU, x);
            float *sDU = reinterpret_cast<float *>(base + STG) + C * LU;
#pragma unroll
            for (int r = 0; r < C; ++r) sDU[r * LU + jl] = x[r];
        } else {
#pragma unroll
            for (int r = 0; r < C; ++r)
                st_op(base + O_OY, 64, r, jl, r < L ? lds_bf16(base + T_DO + off_bf16(r, jl)) : 0.f);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // dP = tril(dO U^T) and dT = dU (beta Y)^T (strict), 2 x 2 tiles over j
        {
            const int prod = t >> 8, th = t & 255;
            const int r0 = (th >> 4) * 2, i0 = (th & 15) * 2;
            const float *sU = reinterpret_cast<const float *>(base + STG);
            const float *sDU = sU + C * LU, *sY = sU + 2 * C * LU;
            float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
            if (prod == 0) {
#pragma unroll 4
                for (int j = 0; j < D; ++j) {
                    const float x0 = lds_bf16(base + T_DO + off_bf16(r0, j));
                    const float x1 = lds_bf16(base + T_DO + off_bf16(r0 + 1, j));
                    const float y0 = sU[i0 * LU + j], y1 = sU[(i0 + 1) * LU + j];
                    a00 += x0 * y0;
                    a01 += x0 * y1;
                    a10 += x1 * y0;
                    a11 += x1 * y1;
                }
            } else {
#pragma unroll 4
                for (int j = 0; j < D; ++j) {
                    const float x0 = sDU[r0 * LU + j], x1 = sDU[(r0 + 1) * LU + j];
                    const float y0 = sY[i0 * LU + j], y1 = sY[(i0 + 1) * LU + j];
                    a00 += x0 * y0;
                    a01 += x0 * y1;
                    a10 += x1 * y0;
                    a11 += x1 * y1;
                }
            }
            const float av[2][2] = {{a00, a01}, {a10, a11}};
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2)
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    const int r = r0 + u2, i = i0 + w2;
                    // rows past the chunk's end hold dO = 0 (U rows are 0 there too)
                    if (prod == 0) sm.dP[r][i] = (i <= r && r < L) ? av[u2][w2] : 0.f;
                    else sm.dT[r][i] = i < r ? av[u2][w2] * sm.beta[i] : 0.f;
                }
        }
        if (t < C) sm.dbeta[t] += sm.red[0][t] + sm.red[1][t] + sm.red[2][t] + sm.red[3][t];
        __syncthreads();
        // S0 (rows c, K = j) into STG: four threads per row, 32 channels of j each
        {
            const int c = t >> 2, j0 = (t & 3) * 32;
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (S0g) v4 = *reinterpret_cast<const float4 *>(S0g + (int64_t)c * D + j0 + i);
                x[i] = v4.x;
                x[i + 1] = v4.y;
                x[i + 2] = v4.z;
                x[i + 3] = v4.w;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(base + STG + sw_off(128, c, j0 + i)) =
                    make_float4(to_tf32(x[i]), to_tf32(x[i + 1]), to_tf32(x[i + 2]), to_tf32(x[i + 3]));
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- phase 6: [aQ^T | aK^T] / e15 = S0 [dO ; -dY]^T ----
        if (t == 0) {
            tc_fence_after();
            mma_ss_group(tb + TM_AQK, base + STG, 16384, base + O_OY, 8192, 16, 64, false);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;
        // dS (rows c, K = j) into STG from dS^T in tensor memory: lane j, its
        // quarter `slice` of the key channels
        {
            float x[32];
            tmem_ld32(tl + TM_DS + 32 * slice, x);
#pragma unroll
            for (int i = 0; i < 32; ++i) st_op(base + STG, 128, 32 * slice + i, jl, x[i]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // aB^T = dS U^T; the dS_0 increment (Q1^T dO - A1^T dY)^T = [dO^T | -dY^T] [Q1^T | A1^T]^T
        if (t == 0) {
            tc_fence_after();
            mma_ss_group(tb + TM_AB, base + STG, 16384, base + O_U, 4096, 16, 32, false);
            mma_ts_group(tb + TM_DN, tb + TM_DOT, base + OPQA, 16384, 8, 128, false);
        }
        // meanwhile: gsum[c] = sum_j dS[c][j] S0[c][j] (four threads per channel)
        {
            const int c = t >> 2, j0 = (t & 3) * 32;
            float s = 0.f;
            if (S0g) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(base + STG + sw_off(128, c, j0 + i));
                    const float4 s4 = *reinterpret_cast<const float4 *>(S0g + (int64_t)c * D + j0 + i);
                    s += d4.x * s4.x + d4.y * s4.y + d4.z * s4.z + d4.w * s4.w;
                }
            }
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((t & 3) == 0) sm.gsum[c] = s;
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 7: dS^T <- dS^T Diag(gamma_C) + (increment)^T Diag(e15) (lane j,
        // its quarter of the channels); dA, dG and the dA . G row sums ----
        {
            float x[32], y[32];
            tmem_ld32(tl + TM_DS + 32 * slice, x);
            tmem_ld32(tl + TM_DN + 32 * slice, y);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 32 * slice + i;
                x[i] = sm.gC[c] * x[i] + sm.e15[c] * y[i];
            }
            tmem_st32(tl + TM_DS + 32 * slice, x);
            tmem_wait_st();
        }
        {
            // M1 = tril_s(dT) T^T into dP's neighbour (the G array keeps G until dG)
            float(*M1)[LDS32] = reinterpret_cast<float(*)[LDS32]>(base + STG);   // STG is free again
            for (int idx = t; idx < C * C; idx += kThreads) {
                const int r = idx >> 5, i = idx & 31;
                float s = 0.f;
                for (int bb = 0; bb < r && bb <= i; ++bb) s += sm.dT[r][bb] * sm.T[i][bb];
                M1[r][i] = s;
            }
            __syncthreads();
            for (int idx = t; idx < C * C; idx += kThreads) {   // a warp = one row r
                const int r = idx >> 5, i = idx & 31;
                float s = 0.f;
                for (int a2 = r; a2 < C; ++a2) s -= sm.T[a2][r] * M1[a2][i];
                const float da = i < r ? s : 0.f;
                float gb = da * sm.G[r][i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) gb += __shfl_xor_sync(0xffffffffu, gb, o);
                sm.G[r][i] = sm.beta[r] * da;   // dG
                if (i == 0) sm.dbeta[r] += gb;
            }
        }
        __syncthreads();
        // [dP ; dG] (rows, K = i) and the B operand of R3 (rows x, K = [i | i']:
        // dP[i][x], dG[i][x]) into OPA
        for (int idx = t; idx < C * C; idx += kThreads) {
            const int r = idx >> 5, i = idx & 31;
            st_op(base + O_PG, 64, r, i, sm.dP[r][i]);
            st_op(base + O_PG, 64, 32 + r, i, sm.G[r][i]);
            st_op(base + O_R3B, 32, r, i, sm.dP[i][r]);
            st_op(base + O_R3B, 32, r, 32 + i, sm.G[i][r]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (t == 0) {
            tc_fence_after();
            mma_ss_group(tb + TM_R12, base + OPB1T, 16384, base + O_PG, 8192, 4, 64, false);
            mma_ss_group(tb + TM_R3, base + OPQA, 16384, base + O_R3B, 4096, 8, 32, false);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 8 (warps 0-3, lane = key channel c): dq, dk, dGamma, dg ----
        if (warp < 4) {
            const int c = jl;
            const float e15 = sm.e15[c], fC = sm.fC[c];
            const float gl = *reinterpret_cast<const float *>(base + T_G + off_f32(C - 1, c));
            const float g15 = *reinterpret_cast<const float *>(base + T_G + off_f32(15, c));
            float dgam[C];
            float kbk = 0.f;
#pragma unroll
            for (int x8 = 0; x8 < C; x8 += 8) {
                float aq[8], ak[8], ab[8], r1[8], r2[8], r3[8];
                tmem_ld8(tl + TM_AQK + x8, aq);
                tmem_ld8(tl + TM_AQK + 32 + x8, ak);
                tmem_ld8(tl + TM_AB + x8, ab);
                tmem_ld8(tl + TM_R12 + x8, r1);
                tmem_ld8(tl + TM_R12 + 32 + x8, r2);
                tmem_ld8(tl + TM_R3 + x8, r3);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int x = x8 + u;
                    const float gx = *reinterpret_cast<const float *>(base + T_G + off_f32(x, c));
                    const float ex = __expf(gx - g15), ix = __expf(g15 - gx);
                    const float sq = e15 * aq[u] + r1[u], sk = e15 * ak[u] + r2[u];
                    const float fb = fC * ab[u];
                    if (x < L) {
                        const int64_t off = (t0 + x) * rowK + (int64_t)h * D + c;
                        kda::st_elem(dq + off, ex * sq);
                        kda::st_elem(dk + off, ex * sk + __expf(gl - gx) * ab[u] + ix * r3[u]);
                    }
                    const float q1 = *reinterpret_cast<const float *>(base + OPQA + sw_off(128, c, x));
                    const float a1 = *reinterpret_cast<const float *>(base + OPQA + 16384 + sw_off(128, c, x));
                    const float b1 = *reinterpret_cast<const float *>(base + OPB1T + sw_off(128, c, x));
                    dgam[x] = q1 * sq + a1 * sk - b1 * (fb + r3[u]);
                    kbk += fb * b1;
                }
            }
            float run = 0.f;
            const float last = fC * e15 * sm.gsum[c] + kbk;
#pragma unroll
            for (int r = C - 1; r >= 0; --r) {
                run += dgam[r] + (r == C - 1 ? last : 0.f);
                if (r < L) dg[(t0 + r) * rowK + (int64_t)h * D + c] = run;
            }
        }
        if (t < C && t < L) dbeta[(t0 + t) * H + h] = sm.dbeta[t];
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // the initial state's gradient: dS (lane j holds column j)
    if (d_init && !*reinterpret_cast<volatile int *>(&sm.abort) && slice == 0) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            float x[32];
            tmem_ld32(tl + TM_DS + c0, x);
#pragma unroll
            for (int i = 0; i < 32; ++i) d_init[soff + (int64_t)(c0 + i) * D + jl] = x[i];
        }
    }
    if (t == 0) {   // every MMA issued has completed (after a stop too)
        tc_fence_after();
        mma_commit(&sm.mma_bar);
        mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

bool kda_backward_tc_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                               const float *g, const void *d_out) {
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    return P.dk == 128 && P.dv == 128 && P.in_dtype == KDA_DTYPE_BF16 && P.T > 0 &&
           P.T <= 0x7fffffff - C && al16(q) && al16(k) && al16(v) && al16(g) && al16(d_out);
}

cudaError_t kda_launch_backward_tc(const kda::Problem &P, const void *q, const void *k,
                                   const void *v, const float *g, const float *beta,
                                   const float *init_state, const int32_t *cu,
                                   const float *chunk_states, int64_t chunk_capacity,
                                   const void *d_out, const float *d_final, void *dq, void *dk,
                                   void *dv, float *dg, float *dbeta, float *d_init,
                                   cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mdo, mg;
    if (!kda_make_tile_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mdo, d_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.T, P.H))
        return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((int64_t)P.N * P.H);
    if (P.out_dtype == KDA_DTYPE_BF16) {
        auto kern = kda_backward_tc_kernel<__nv_bfloat16>;
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem); });
        if (attr != cudaSuccess) return attr;
        kern<<<blocks, kThreads, kSmem, stream>>>(mq, mk, mv, mdo, mg, beta, init_state, cu, chunk_states,
                                                  chunk_capacity, d_final, (__nv_bfloat16 *)dq,
                                                  (__nv_bfloat16 *)dk, (__nv_bfloat16 *)dv, dg, dbeta,
                                                  d_init, P.H, (int64_t)P.T, P.seq_len);
    } else {
        auto kern = kda_backward_tc_kernel<float>;
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem); });
        if (attr != cudaSuccess) return attr;
        kern<<<blocks, kThreads, kSmem, stream>>>(mq, mk, mv, mdo, mg, beta, init_state, cu, chunk_states,
                                                  chunk_capacity, d_final, (float *)dq, (float *)dk,
                                                  (float *)dv, dg, dbeta, d_init, P.H, (int64_t)P.T,
                                                  P.seq_len);
    }
    return cudaGetLastError();
}

cudaError_t kda_bwdtc_read_status(unsigned *status) {
    unsigned st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&st, g_kda_bwdtc_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_kda_bwdtc_status, &zero, sizeof(unsigned));
    *status |= st;
    return e;
}
