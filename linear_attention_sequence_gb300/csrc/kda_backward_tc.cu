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
// a 128-long side is a tcgen05.mma kind::tf32 group with M = 128 (values or
// key channels) and fp32 accumulation; its operands are written by the threads
// as K-major SW128 tf32 blocks in shared memory, or read from tensor memory.
// The pairs [G ; P] and dP, dT are M = 64 products whose 32-row operands are
// read with 32 further rows of shared memory past them (the rows of the result
// that those give are not read).  The solve, dA = -T^T dT T^T and the pairwise
// 32 x 32 terms run on the CUDA cores.  The phases of a chunk run one after
// another, separated by block barriers; within a phase the MMA groups for
// different accumulators are issued by elected lanes of up to three warps (the
// Gram and X also as two K halves summed when read), the solve runs on its own
// warp beside the state copy and X, and the next chunk's tiles and state are
// fetched by TMA during the last phases of the current one.  The kernel's code
// size matters: instruction fetch is a visible share of its stalls, so loops
// off the critical path are kept rolled.

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
constexpr int kIssuers = 3;   // warps that issue MMA groups (one elected lane each)
constexpr int kS0Issuer = 32; // issues the state loads (the tiles come from thread 0)

// Shared memory (byte offsets from a 1024-aligned base).
//   TILE   TMA tiles of the chunk: q, k, dO (bf16, 8 KB each), g (fp32, 16 KB) and v
//          (bf16, at 40 KB).  Once the preparation holds q, k, dO and g in registers,
//          the Gram A operand [A1 ; Q1] (rows, K = c) goes over them; then T diag(beta)
//          and T^T (4 KB each, at 32 KB); later U, dU and beta Y (16 KB each).  Once
//          the aB product has read U, the next chunk's tiles are loaded here.
//   STG    64 KB: S0 by TMA (rows c, K = j), loaded a chunk ahead; it is copied
//          transposed into TMEM and is the A operand of [aQ | aK]; then dS (rows c).
//   OPA    B1 rows and Kb rows (16 KB each); then P^T (4 KB); later [dO ; -dY]
//          (32 KB), then [dP ; dG] (8 KB), the B operand of R3 (8 KB), the dA
//          scratch (4.2 KB) and the dv rows; then the dq, dk and dg rows.
//   OPQA   [Q1^T | A1^T] (rows c, K = 64, 32 KB).   OPB1T  B1^T (rows c, 16 KB).
constexpr uint32_t T_Q = 0, T_K = 8192, T_DO = 16384, T_G = 24576, T_V = 40960;
constexpr uint32_t O_AQ = 0;                   // [A1 ; Q1]: 4 K-blocks of 64 rows
constexpr uint32_t O_TB = 32768, O_TT = 36864;
// the dP / dT operands U, dU and beta Y (rows, K = j; 16 KB each) in the tile area (an
// M = 64 product reads 32 further rows past dU: the beta Y rows, whose products it drops)
constexpr uint32_t O_U = 0, O_DU = 16384, O_BY = 32768;
constexpr uint32_t STG = 49152;
constexpr uint32_t OPA = STG + 65536;          // 114688
constexpr uint32_t O_B1 = OPA, O_KB = OPA + 16384, O_PT = OPA, O_OY = OPA, O_PG = OPA,
                   O_R3B = OPA + 8192, O_M1 = OPA + 16384;
// bf16 gradient rows staged for 16-byte stores: dv [32][128] (phase 7, beside the dA
// scratch), then dq, dk [32][128] and dg [32][128] fp32 (the epilogue)
constexpr uint32_t O_SV = OPA + 24576, O_SQ = OPA, O_SK = OPA + 8192, O_SG = OPA + 16384;
constexpr uint32_t OPQA = OPA + 32768;         // 147456
constexpr uint32_t OPB1T = OPQA + 32768;       // 180224
constexpr uint32_t SMALL = OPB1T + 16384;      // 196608
constexpr int LDS32 = C + 1;                   // row length of the 32 x 32 fp32 arrays

struct Small {
    float G[C][LDS32], P[C][LDS32], T[C][LDS32], dP[C][LDS32], dT[C][LDS32];
    float beta[C], dbeta[C], red[4][C];
    float e15[D], fC[D], gC[D], gsum[D];
    float red2[4][D];
    float akkT[C][C];          // solve scratch
    float tsc[3][16][20];
    uint64_t tma_bar, s0_bar, mma_bar;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kSmem = SMALL + sizeof(Small) + 1024;
static_assert(kSmem <= 232448, "shared memory budget");

// Tensor-memory columns (lanes = value j for dS^T, X, Y, U, dU, dB, dO^T, the dS0
// increment; lanes = key channel c for aQ|aK, aB, R1|R2, R3, e^{Gamma - Gamma_15}).
// The M = 64 products [G ; P] (in TM_G, before dB) and dP, dT (in TM_X, TM_Y after
// X and Y are read) put their rows 0-15 on lanes 0-15, 16-31 on lanes 32-47 and so
// on.  TM_DN holds e15 S0^T, then aQ|aK; the dS0 increment takes 256-383 once dP,
// dT, U and dU are read, and R1|R2, R3 take 256-351 after it.
constexpr uint32_t TM_DS = 0, TM_DN = 128, TM_X = 256, TM_Y = 288, TM_U = 320, TM_DU = 352,
                   TM_DB = 384, TM_DOT = 416, TM_EX = 480;
constexpr uint32_t TM_G = TM_DB, TM_AQK = TM_DN, TM_INC = 256, TM_AB = 384, TM_R12 = 256, TM_R3 = 320;

__device__ __forceinline__ uint32_t off_bf16(int r, int c) {   // TMA tile (SW128), bf16
    return (uint32_t)((c >> 6) * 4096 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ float lds_bf16(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
// One K-major SW128 tf32 element store (row `row` of an operand with `rows` rows).
__device__ __forceinline__ void st_op(unsigned char *base, int rows, int row, int k, float x) {
    *reinterpret_cast<float *>(base + sw_off(rows, row, k)) = to_tf32(x);
}

// Byte offsets of column k in row r of a K-major SW128 operand with `rows` rows
// (without the r * 128), for the eight values of r % 8; and the same for
// column c of the bf16 and fp32 TMA tiles.
__device__ __forceinline__ void op_offsets(int rows, int k, uint32_t (&o)[8]) {
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8)
        o[k8] = (uint32_t)((k >> 5) * rows * 128 + ((((k & 31) >> 2) ^ k8) << 4) + ((k & 3) << 2));
}
__device__ __forceinline__ void bf16_offsets(int c, uint32_t (&o)[8]) {
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) o[k8] = (uint32_t)((c >> 6) * 4096 + ((((c & 63) >> 3) ^ k8) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ void f32_offsets(int c, uint32_t (&o)[8]) {
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) o[k8] = (uint32_t)((c >> 5) * 4096 + ((((c & 31) >> 2) ^ k8) << 4) + ((c & 3) << 2));
}

// One MMA group, called by a whole warp (one elected lane issues): D[m][n] (+)=
// sum_k A[m][k] B[n][k], A and B K-major SW128 in shared memory (SS) with K-blocks
// of `akb` and `bkb` bytes; `ksteps` steps of 8.
__device__ __forceinline__ void mma_ss_group(uint32_t d, const unsigned char *a, uint32_t akb,
                                             const unsigned char *b, uint32_t bkb, int ksteps, int n,
                                             bool acc, int m = 128) {
    const uint64_t da = sdesc_sw128(smem_u32(a)), db = sdesc_sw128(smem_u32(b));
    for (int kk = 0; kk < ksteps; ++kk)
        mma_tf32_ss_el(d, da + (uint64_t)(((kk >> 2) * akb + (kk & 3) * 32) >> 4),
                    db + (uint64_t)(((kk >> 2) * bkb + (kk & 3) * 32) >> 4), idesc_tf32(m, n),
                    (acc || kk > 0) ? 1u : 0u);
}
// The same with A in tensor memory (8 columns per K step).
__device__ __forceinline__ void mma_ts_group(uint32_t d, uint32_t a, const unsigned char *b,
                                             uint32_t bkb, int ksteps, int n, bool acc) {
    const uint64_t db = sdesc_sw128(smem_u32(b));
    for (int kk = 0; kk < ksteps; ++kk)
        mma_tf32_ts_el(d, a + 8 * kk, db + (uint64_t)(((kk >> 2) * bkb + (kk & 3) * 32) >> 4),
                    idesc_tf32(128, n), (acc || kk > 0) ? 1u : 0u);
}

template <typename OUT_T>
__global__ void __launch_bounds__(kThreads, 1)
kda_backward_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_cs,
                       const __grid_constant__ CUtensorMap tm_init, int has_cs, int has_init, int vec_out,
                       const float *__restrict__ beta,
                       const float *init_state, const int32_t *__restrict__ cu,
                       const float *__restrict__ chunk_states, int64_t chunk_capacity,
                       const float *__restrict__ d_final, OUT_T *__restrict__ dq,
                       OUT_T *__restrict__ dk, OUT_T *__restrict__ dv, float *__restrict__ dg,
                       float *__restrict__ dbeta, float *d_init, int H, int64_t total,
                       int64_t seq_len) {
    // bf16 gradients with 16-byte aligned rows go out through shared memory as
    // 16-byte stores (a thread holds one channel of many tokens)
    const bool vstore = sizeof(OUT_T) == 2 && vec_out;
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
        mbar_init(&sm.s0_bar, 1);
        mbar_init(&sm.mma_bar, kIssuers);
        fence_mbar_init();
        sm.abort = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_g);
        if (has_cs) prefetch_tmap(&tm_cs);
        if (has_init) prefetch_tmap(&tm_init);
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
    uint32_t tma_par = 0, s0_par = 0, mma_par = 0;

    // The tiles of the chunk at token tx (q, k, v, dO bf16; g fp32) by TMA on tma_bar.
    // A chunk's tiles are issued while the chunk after it is finished (thread 0 keeps
    // the parity of the group in flight so that a stop can still wait for it).
    auto load_tiles = [&](int64_t tx) {
        mbar_arrive_expect_tx(&sm.tma_bar, 4 * 8192 + 16384);
        tma_load_3d(base + T_Q, &tm_q, &sm.tma_bar, 0, (int)tx, 2 * h);
        tma_load_3d(base + T_K, &tm_k, &sm.tma_bar, 0, (int)tx, 2 * h);
        tma_load_3d(base + T_V, &tm_v, &sm.tma_bar, 0, (int)tx, 2 * h);
        tma_load_3d(base + T_DO, &tm_do, &sm.tma_bar, 0, (int)tx, 2 * h);
        tma_load_3d(base + T_G, &tm_g, &sm.tma_bar, 0, (int)tx, 4 * h);
    };
    bool tiles_pending = false;
    uint32_t pend_par = 0;
    // The start state S0 of chunk cx (rows c, K = j) into STG, also a chunk ahead: four
    // 128-row boxes of 32 columns by TMA from the initial state (chunk 0) or the
    // checkpoint row, or zeros where there is none.  Called by every thread.
    auto s0_present = [&](int cx) -> bool {
        return cx == 0 ? init_state != nullptr : (chunk_states != nullptr && ck0 + cx - 1 < chunk_capacity);
    };
    bool s0_pending = false;   // thread kS0Issuer: a state load that no chunk has awaited yet
    auto fetch_s0 = [&](int cx) {
        if (s0_present(cx)) {
            if (t == kS0Issuer) {
                const CUtensorMap *map = cx == 0 ? &tm_init : &tm_cs;
                const int row = (int)((cx == 0 ? (int64_t)n * H + h : (ck0 + cx - 1) * H + h) * D);
                mbar_arrive_expect_tx(&sm.s0_bar, 65536);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) tma_load_2d(base + STG + kb * 16384, map, &sm.s0_bar, 32 * kb, row);
                s0_pending = true;
            }
        } else {
            for (int i = t; i < 65536 / 16; i += kThreads)
                reinterpret_cast<float4 *>(base + STG)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float bnext = 0.f;   // beta of the next chunk (threads 0..C-1)
    if (nchunks > 0) {   // the last chunk comes first
        const int64_t tx = a + (int64_t)(nchunks - 1) * C;
        if (t == 0) {
            load_tiles(tx);
            tiles_pending = true;
        }
        fetch_s0(nchunks - 1);
        if (t < C && tx + t < b) bnext = beta[(tx + t) * H + h];
    }

    // An MMA group is split over warps 0 .. kIssuers-1 (products for different
    // accumulators issue in parallel), each ending its share with a commit to mma_bar
    // (kIssuers arrivals a phase); thread 0 waits, the barrier releases the rest.
    auto mma_wait = [&]() {
        if (t == 0 && !mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit)) {
            sm.abort = 1;
            atomicOr(&g_kda_bwdtc_status, 0x400u);
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

        // ---- phase 0: the chunk's tiles (issued a chunk ahead) have landed; beta ----
        if (t < C) {
            sm.beta[t] = bnext;
            sm.dbeta[t] = 0.f;
        }
        if (t == 0) {
            if (mbar_wait_bounded(&sm.tma_bar, tma_par, kPollLimit)) {
                tiles_pending = false;
            } else {
                sm.abort = 1;
                atomicOr(&g_kda_bwdtc_status, 0x800u);
            }
        }
        tma_par ^= 1u;
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 1 (all 16 warps; thread = key channel c = its TMEM lane, tokens
        // 8 slice .. 8 slice + 7): Gamma, the decay-weighted operands, dO^T and
        // e^{Gamma - Gamma_15} into tensor memory ----
        {
            const int c = jl, r0 = 8 * slice;
            uint32_t ob[8], of[8], ok[8], og[8];
            bf16_offsets(c, ob);
            f32_offsets(c, of);
            op_offsets(32, c, ok);
            op_offsets(64, c, og);
            float gam[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u;
                gam[u] = r < L ? *reinterpret_cast<const float *>(base + T_G + r * 128 + of[u]) : 0.f;
            }
#pragma unroll
            for (int u = 1; u < 8; ++u) gam[u] += gam[u - 1];
            sm.red2[slice][c] = gam[7];
            uint32_t dov[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u;
                dov[u] = __float_as_uint(r < L ? lds_bf16(base + T_DO + r * 128 + ob[u]) : 0.f);
            }
            tmem_st8(tl + TM_DOT + r0, dov);
            float qv[8], kv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u;
                qv[u] = r < L ? lds_bf16(base + T_Q + r * 128 + ob[u]) : 0.f;
                kv[u] = r < L ? lds_bf16(base + T_K + r * 128 + ob[u]) : 0.f;
            }
            // every q, k, dO and g value is in registers: [A1 ; Q1] may go over the tiles
            __syncthreads();
            const float p0 = sm.red2[0][c], p1 = sm.red2[1][c], p2 = sm.red2[2][c], p3 = sm.red2[3][c];
            const float g15 = p0 + p1, gl = g15 + p2 + p3;
            // Gamma_r - Gamma_15 for this thread's tokens: the sums of the earlier slices
            const float base_x = (slice == 0 ? 0.f : slice == 1 ? p0 : slice == 2 ? g15 : g15 + p2) - g15;
            const float e15 = __expf(g15), fC = __expf(gl - g15);
            if (slice == 0) {
                sm.e15[c] = e15;
                sm.fC[c] = fC;
                sm.gC[c] = __expf(gl);
            }
            float q1[8], a1[8], b1[8];
            uint32_t exv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u;
                const float x = base_x + gam[u];             // in [-80, 80] by the log-decay bound
                const float e1 = __expf(x), inv = __expf(-x);
                const float ka = kv[u] * e1, kbv = kv[u] * inv;
                exv[u] = __float_as_uint(e1);
                q1[u] = to_tf32(qv[u] * e1);
                a1[u] = to_tf32(ka);
                b1[u] = to_tf32(kbv);
                // Kb = k e^{Gamma_C - Gamma} as rows (K = c); Kt = k e^{Gamma} = A1 e15
                // enters as A1 with e15 folded into S0^T
                *reinterpret_cast<float *>(base + O_KB + r * 128 + ok[u]) = to_tf32(kbv * fC);
                // the Gram operands: [A1 ; Q1] and B1 as rows (K = c)
                *reinterpret_cast<float *>(base + O_AQ + r * 128 + og[u]) = a1[u];
                *reinterpret_cast<float *>(base + O_AQ + (32 + r) * 128 + og[u]) = q1[u];
                *reinterpret_cast<float *>(base + O_B1 + r * 128 + ok[u]) = b1[u];
            }
            tmem_st8(tl + TM_EX + r0, exv);
            // [Q1^T | A1^T] and B1^T as rows c (K = token), four tokens per 16-byte store
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t pos = (uint32_t)(((((r0 >> 2) + h2) ^ (c & 7)) & 7) << 4);
                const int u = 4 * h2;
                *reinterpret_cast<float4 *>(base + OPQA + c * 128 + pos) = make_float4(q1[u], q1[u + 1], q1[u + 2], q1[u + 3]);
                *reinterpret_cast<float4 *>(base + OPQA + 16384 + c * 128 + pos) =
                    make_float4(a1[u], a1[u + 1], a1[u + 2], a1[u + 3]);
                *reinterpret_cast<float4 *>(base + OPB1T + c * 128 + pos) = make_float4(b1[u], b1[u + 1], b1[u + 2], b1[u + 3]);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- phase 2: [G ; P] = [A1 ; Q1] B1^T (M = 64: rows r of G on lanes 0-15 and
        // 32-47, of P on lanes 64-79 and 96-111), its K halves on warps 0 and 2 (into
        // TM_G and TM_X, summed when read), dU^T = dS^T Kb^T on warp 1.
        // Meanwhile warps 4-11 copy e15 S0^T into tensor memory (lane j, columns c of
        // this warp's half) once the state has landed, with the partial sums
        // gsum[c] = sum_j dS[c][j] S0[c][j].  Warps 0-3 then read G and P, hand G to
        // the solve (warp 12) and store P^T as an operand; thread 0 issues X =
        // (e15 S0^T) A1^T and dU^T += dO^T P, and warps 0-3 form Y^T = V^T - X. ----
        if (warp < kIssuers) {
            tc_fence_after();
            if (warp == 0) mma_ss_group(tb + TM_G, base + O_AQ, 8192, base + O_B1, 4096, 8, 32, false, 64);
            else if (warp == 2)
                mma_ss_group(tb + TM_X, base + O_AQ + 2 * 8192, 8192, base + O_B1 + 2 * 4096, 4096, 8, 32, false, 64);
            mma_commit_el(&sm.mma_bar);   // this phase of mma_bar waits for the Gram alone
            if (warp == 1) mma_ts_group(tb + TM_DU, tb + TM_DS, base + O_KB, 4096, 16, 32, false);
        }
        if (warp < 4) {
            if (t == 0 && !mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit)) {
                sm.abort = 1;
                atomicOr(&g_kda_bwdtc_status, 0x400u);
            }
            named_sync(3, 128);
            tc_fence_after();
            // the collective load runs on every lane of the warp; lanes 0-15 hold rows
            float x[32], x2[32];
            tmem_ld32(tl + TM_G, x);
            tmem_ld32(tl + TM_X, x2);
#pragma unroll
            for (int i = 0; i < C; ++i) x[i] += x2[i];
            if (lane < 16) {
                const int row = 16 * warp + lane;   // 0..63: G rows 0-31, then P rows 0-31
                const int r = row & 31;
#pragma unroll
                for (int i = 0; i < C; ++i) {
                    if (row < 32) sm.G[r][i] = i < r ? x[i] : 0.f;
                    else sm.P[r][i] = i <= r ? x[i] : 0.f;
                }
            }
            named_arrive(4, 160);   // G is ready for the solve
            named_sync(3, 128);
            for (int idx = t; idx < C * C; idx += 128) {
                const int r = idx >> 5, i = idx & 31;
                st_op(base + O_PT, 32, r, i, sm.P[i][r]);
            }
            fence_proxy_async_smem();
        } else if (warp < 12) {
            bool ok = true;
            if (S0g && lane == 0) ok = mbar_wait_bounded(&sm.s0_bar, s0_par, kPollLimit);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok && lane == 0) {
                sm.abort = 1;
                atomicOr(&g_kda_bwdtc_status, 0x800u);
            }
            const int half = (warp - 4) >> 2;
            // one 32-column block per iteration (the loop is kept rolled: code size)
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c0 = 64 * half + 32 * h2;
                float x[32], y[32], d[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = *reinterpret_cast<const float *>(base + STG + sw_off(128, c0 + i, jl));
                    y[i] = x[i];
                    x[i] *= sm.e15[c0 + i];
                }
                tmem_st32(tl + TM_DN + c0, x);
                tmem_ld32(tl + TM_DS + c0, d);
#pragma unroll
                for (int i = 0; i < 32; ++i) y[i] *= d[i];
                // sum over this warp's 32 lanes j: reduce-scatter, lane i ends with column c0 + i
#pragma unroll
                for (int sh = 16; sh >= 1; sh >>= 1) {
                    const bool up = (lane & sh) != 0;
#pragma unroll
                    for (int i = 0; i < sh; ++i) {
                        const float send = up ? y[i] : y[i + sh];
                        const float keep = up ? y[i + sh] : y[i];
                        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
                    }
                }
                sm.red2[q4][c0 + lane] = y[0];
            }
            tmem_wait_st();
        } else if (warp == 12) {   // blocked solve (scratch in the small arrays)
            named_sync(4, 160);
            float d[32];
#pragma unroll
            for (int i = 0; i < C; ++i) d[i] = sm.G[lane][i];
            solve_t(d, sm.beta[lane], lane, &sm.T[0][0], LDS32, sm.akkT, sm.tsc);
        }
        mma_par ^= 1u;
        if (warp < 12) {
            tc_fence_before();
            named_sync(2, 384);
            if (warp < kIssuers) {
                tc_fence_after();
                // X in two K halves (warps 0 and 2, into TM_X and TM_Y, summed when read)
                if (warp == 0) mma_ts_group(tb + TM_X, tb + TM_DN, base + O_AQ, 8192, 8, 32, false);
                else if (warp == 1) mma_ts_group(tb + TM_DU, tb + TM_DOT, base + O_PT, 4096, 4, 32, true);
                else mma_ts_group(tb + TM_Y, tb + TM_DN + 64, base + O_AQ + 2 * 8192, 8192, 8, 32, false);
                mma_commit_el(&sm.mma_bar);
            }
            if (t == 0 && !mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit)) {
                sm.abort = 1;
                atomicOr(&g_kda_bwdtc_status, 0x400u);
            }
            if (warp < 4) {   // Y^T = V^T - X into tensor memory
                named_sync(3, 128);
                tc_fence_after();
                float x[32], x2[32];
                tmem_ld32(tl + TM_X, x);
                tmem_ld32(tl + TM_Y, x2);
#pragma unroll
                for (int r = 0; r < C; ++r) x[r] = r < L ? lds_bf16(base + T_V + off_bf16(r, jl)) - (x[r] + x2[r]) : 0.f;
                tmem_st32(tl + TM_Y, x);
                tmem_wait_st();
            }
        }
        mma_par ^= 1u;
        if (S0g) s0_par ^= 1u;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (t == kS0Issuer && S0g) s0_pending = false;
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;
        if (t < D) sm.gsum[t] = sm.red2[0][t] + sm.red2[1][t] + sm.red2[2][t] + sm.red2[3][t];
        // T diag(beta) and T^T as 32-row operands
        for (int idx = t; idx < C * C; idx += kThreads) {
            const int r = idx >> 5, i = idx & 31;
            st_op(base + O_TB, 32, r, i, sm.T[r][i] * sm.beta[i]);
            st_op(base + O_TT, 32, r, i, sm.T[i][r]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- phases 3-4: U^T = Y^T (T diag beta)^T, dB^T = dU^T T ----
        if (warp < kIssuers) {
            tc_fence_after();
            if (warp == 0) mma_ts_group(tb + TM_U, tb + TM_Y, base + O_TB, 4096, 4, 32, false);
            else if (warp == 1) mma_ts_group(tb + TM_DB, tb + TM_DU, base + O_TT, 4096, 4, 32, false);
            mma_commit_el(&sm.mma_bar);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 5 (lane j): -dY^T = -diag(beta) dB^T into tensor memory and the
        // dB . Y row sums (warps 0-3); the operands U (warps 4-7), dU and beta Y (warps 8-11) and
        // [dO ; -dY] (warps 12-15) as rows ----
        if (warp < 4) {
            float y[32], x[32];
            tmem_ld32(tl + TM_DB, x);
            tmem_ld32(tl + TM_Y, y);
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float dy = sm.beta[r] * x[r];
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
            uint32_t o[8];
            op_offsets(32, jl, o);
            tmem_ld32(tl + TM_U, x);
#pragma unroll
            for (int r = 0; r < C; ++r)
                *reinterpret_cast<float *>(base + O_U + r * 128 + o[r & 7]) = to_tf32(x[r]);
        } else if (warp < 12) {
            float x[32];
            uint32_t o[8];
            op_offsets(32, jl, o);
            tmem_ld32(tl + TM_DU, x);
#pragma unroll
            for (int r = 0; r < C; ++r)
                *reinterpret_cast<float *>(base + O_DU + r * 128 + o[r & 7]) = to_tf32(x[r]);
            tmem_ld32(tl + TM_Y, x);
#pragma unroll
            for (int r = 0; r < C; ++r)
                *reinterpret_cast<float *>(base + O_BY + r * 128 + o[r & 7]) = to_tf32(sm.beta[r] * x[r]);
        } else {
            float x[32], y[32];
            uint32_t o[8];
            op_offsets(64, jl, o);
            tmem_ld32(tl + TM_DOT, y);   // dO^T (zero past the chunk's end)
            tmem_ld32(tl + TM_DB, x);
#pragma unroll
            for (int r = 0; r < C; ++r) {
                *reinterpret_cast<float *>(base + O_OY + r * 128 + o[r & 7]) = to_tf32(y[r]);
                *reinterpret_cast<float *>(base + O_OY + (32 + r) * 128 + o[r & 7]) = to_tf32(-sm.beta[r] * x[r]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // dP = dO U^T and dT = dU (beta Y)^T as M = 64 products (rows r on lanes 0-15
        // and 32-47; the second reads 32 rows past dU, whose products it drops), and
        // [aQ^T | aK^T] / e15 = S0 [dO ; -dY]^T with S0 still in STG
        if (warp < kIssuers) {
            tc_fence_after();
            if (warp == 0) mma_ss_group(tb + TM_X, base + O_OY, 8192, base + O_U, 4096, 16, 32, false, 64);
            else if (warp == 1) mma_ss_group(tb + TM_Y, base + O_DU, 4096, base + O_BY, 4096, 16, 32, false, 64);
            else mma_ss_group(tb + TM_AQK, base + STG, 16384, base + O_OY, 8192, 16, 64, false);
            mma_commit_el(&sm.mma_bar);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;
        if (warp < 2) {
            float x[32], y[32];
            tmem_ld32(tl + TM_X, x);
            tmem_ld32(tl + TM_Y, y);
            if (lane < 16) {
                const int r = 16 * warp + lane;
#pragma unroll
                for (int i = 0; i < C; ++i) {
                    // rows past the chunk's end hold other tokens' dO: their dP is 0
                    sm.dP[r][i] = (i <= r && r < L) ? x[i] : 0.f;
                    sm.dT[r][i] = i < r ? y[i] : 0.f;
                }
            }
        }
        if (t < C) sm.dbeta[t] += sm.red[0][t] + sm.red[1][t] + sm.red[2][t] + sm.red[3][t];
        // ---- phase 6: dS (rows c, K = j) into STG from dS^T in tensor memory (lane
        // j, its quarter `slice` of the key channels) ----
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
        if (warp < kIssuers) {
            tc_fence_after();
            if (warp == 0) mma_ss_group(tb + TM_AB, base + STG, 16384, base + O_U, 4096, 16, 32, false);
            else if (warp == 1) mma_ts_group(tb + TM_INC, tb + TM_DOT, base + OPQA, 16384, 8, 128, false);
            mma_commit_el(&sm.mma_bar);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // The tile area's last reader (the aB product) and STG's (the same product) are
        // complete: the next chunk's tiles, state and beta are fetched during the rest
        // of this one.
        if (ch > 0) {
            if (t == 0) {
                load_tiles(t0 - C);
                tiles_pending = true;
                pend_par = tma_par;
            }
            fetch_s0(ch - 1);
            if (t < C) bnext = beta[(t0 - C + t) * H + h];   // chunk ch - 1 is a whole chunk
        }

        // ---- phase 7: dS^T <- dS^T Diag(gamma_C) + (increment)^T Diag(e15) and the
        // stores of dV = dY (from -dY^T, still in TM_DOT) on warps 0-7 (lane j, half of
        // the channels and of the tokens each), while warps 8-15 form dA, dG and the
        // dA . G row sums ----
        if (warp < 8) {
            const int hh = warp >> 2;
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {   // 8-column blocks, rolled (code size)
                const int c0 = 64 * hh + 8 * q;
                float x[8], y[8];
                tmem_ld8(tl + TM_DS + c0, x);
                tmem_ld8(tl + TM_INC + c0, y);
                uint32_t z[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) z[i] = __float_as_uint(sm.gC[c0 + i] * x[i] + sm.e15[c0 + i] * y[i]);
                tmem_st8(tl + TM_DS + c0, z);
            }
            float y[16];
            tmem_ld16(tl + TM_DOT + 32 + 16 * hh, y);
            if (vstore) {
                __nv_bfloat16 *sv = reinterpret_cast<__nv_bfloat16 *>(base + O_SV);   // [C][D]
#pragma unroll
                for (int u = 0; u < 16; ++u) sv[(16 * hh + u) * D + jl] = __float2bfloat16_rn(-y[u]);
                named_sync(5, 256);
#pragma unroll
                for (int i = 0; i < 2; ++i) {   // 512 chunks of 8 channels
                    const int q = t + 256 * i, r = q >> 4, c8 = (q & 15) * 8;
                    if (r < L)
                        *reinterpret_cast<uint4 *>(dv + (t0 + r) * rowK + (int64_t)h * D + c8) =
                            *reinterpret_cast<const uint4 *>(sv + r * D + c8);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = 16 * hh + u;
                    if (r < L) kda::st_elem(dv + (t0 + r) * rowK + (int64_t)h * D + jl, -y[u]);
                }
            }
            tmem_wait_st();
        } else {
            // dA = -T^T tril_s(dT) T^T as two 32 x 32 products (T lower triangular and dT
            // strictly lower, so full-length sums need no bounds): M1 = dT T^T, then
            // dA = -T^T M1; thread = rows r0, r0+1 x columns i0, i0+1
            const int tp = t - 256;
            const int r0 = (tp >> 4) * 2, i0 = (tp & 15) * 2;
            float(*M1)[LDS32] = reinterpret_cast<float(*)[LDS32]>(base + O_M1);
            float m00 = 0.f, m01 = 0.f, m10 = 0.f, m11 = 0.f;
#pragma unroll 8
            for (int bb = 0; bb < C; ++bb) {
                const float d0 = sm.dT[r0][bb], d1 = sm.dT[r0 + 1][bb];
                const float t0v = sm.T[i0][bb], t1v = sm.T[i0 + 1][bb];
                m00 += d0 * t0v;
                m01 += d0 * t1v;
                m10 += d1 * t0v;
                m11 += d1 * t1v;
            }
            M1[r0][i0] = m00;
            M1[r0][i0 + 1] = m01;
            M1[r0 + 1][i0] = m10;
            M1[r0 + 1][i0 + 1] = m11;
            named_sync(1, 256);
            float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll 8
            for (int a2 = 0; a2 < C; ++a2) {
                const float t0v = sm.T[a2][r0], t1v = sm.T[a2][r0 + 1];
                const float x0 = M1[a2][i0], x1 = M1[a2][i0 + 1];
                a00 -= t0v * x0;
                a01 -= t0v * x1;
                a10 -= t1v * x0;
                a11 -= t1v * x1;
            }
            const float dav[2][2] = {{a00, a01}, {a10, a11}};
            float gb0 = 0.f, gb1 = 0.f;
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2)
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    const int r = r0 + u2, i = i0 + w2;
                    const float da = i < r ? dav[u2][w2] : 0.f;
                    const float gbv = da * sm.G[r][i];
                    if (u2 == 0) gb0 += gbv;
                    else gb1 += gbv;
                    sm.G[r][i] = sm.beta[r] * da;   // dG
                }
            // the dA . G row sums over the 16 threads of a row pair (adjacent lanes)
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                gb0 += __shfl_xor_sync(0xffffffffu, gb0, o);
                gb1 += __shfl_xor_sync(0xffffffffu, gb1, o);
            }
            if ((tp & 15) == 0) {
                sm.dbeta[r0] += gb0;
                sm.dbeta[r0 + 1] += gb1;
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
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
        if (warp < kIssuers) {
            tc_fence_after();
            if (warp == 0) mma_ss_group(tb + TM_R12, base + OPB1T, 16384, base + O_PG, 8192, 4, 64, false);
            else if (warp == 1) mma_ss_group(tb + TM_R3, base + OPQA, 16384, base + O_R3B, 4096, 8, 32, false);
            mma_commit_el(&sm.mma_bar);
        }
        mma_wait();
        if (*reinterpret_cast<volatile int *>(&sm.abort)) break;

        // ---- phase 8 (lane = key channel c, tokens 8 slice .. 8 slice + 7): dq, dk,
        // dGamma, and dg as its reverse running sum (within the thread's tokens, then
        // across the four slices through shared memory) ----
        {
            const int c = jl, x0 = 8 * slice;
            const float e15 = sm.e15[c], fC = sm.fC[c];
            float aq[8], ak[8], ab[8], r1[8], r2[8], r3[8], ex[8];
            tmem_ld8(tl + TM_AQK + x0, aq);
            tmem_ld8(tl + TM_AQK + 32 + x0, ak);
            tmem_ld8(tl + TM_AB + x0, ab);
            tmem_ld8(tl + TM_R12 + x0, r1);
            tmem_ld8(tl + TM_R12 + 32 + x0, r2);
            tmem_ld8(tl + TM_R3 + x0, r3);
            tmem_ld8(tl + TM_EX + x0, ex);
            float q1[8], a1[8], b1[8];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t pos = (uint32_t)(((((x0 >> 2) + h2) ^ (c & 7)) & 7) << 4);
                const float4 vq = *reinterpret_cast<const float4 *>(base + OPQA + c * 128 + pos);
                const float4 va = *reinterpret_cast<const float4 *>(base + OPQA + 16384 + c * 128 + pos);
                const float4 vb = *reinterpret_cast<const float4 *>(base + OPB1T + c * 128 + pos);
                q1[4 * h2] = vq.x; q1[4 * h2 + 1] = vq.y; q1[4 * h2 + 2] = vq.z; q1[4 * h2 + 3] = vq.w;
                a1[4 * h2] = va.x; a1[4 * h2 + 1] = va.y; a1[4 * h2 + 2] = va.z; a1[4 * h2 + 3] = va.w;
                b1[4 * h2] = vb.x; b1[4 * h2 + 1] = vb.y; b1[4 * h2 + 2] = vb.z; b1[4 * h2 + 3] = vb.w;
            }
            float dgam[8], kbk = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int x = x0 + u;
                const float ix = __fdividef(1.f, ex[u]);       // e^{Gamma_15 - Gamma_x}
                const float sq = e15 * aq[u] + r1[u], sk = e15 * ak[u] + r2[u];
                const float fb = fC * ab[u];
                const float dqv = ex[u] * sq;
                // e^{Gamma_C - Gamma_x} aB + e^{Gamma_15 - Gamma_x} R3 = e^{Gamma_15 - Gamma_x} (fC aB + R3)
                const float dkv = ex[u] * sk + ix * (fb + r3[u]);
                if (vstore) {
                    reinterpret_cast<__nv_bfloat16 *>(base + O_SQ)[x * D + c] = __float2bfloat16_rn(dqv);
                    reinterpret_cast<__nv_bfloat16 *>(base + O_SK)[x * D + c] = __float2bfloat16_rn(dkv);
                } else if (x < L) {
                    const int64_t off = (t0 + x) * rowK + (int64_t)h * D + c;
                    kda::st_elem(dq + off, dqv);
                    kda::st_elem(dk + off, dkv);
                }
                dgam[u] = q1[u] * sq + a1[u] * sk - b1[u] * (fb + r3[u]);
                kbk += fb * b1[u];
            }
#pragma unroll
            for (int u = 6; u >= 0; --u) dgam[u] += dgam[u + 1];
            // [4][D] each, in the dP array (staged as an operand by now)
            float *part_sum = &sm.dP[0][0], *part_kbk = &sm.dP[0][0] + 4 * D;
            part_sum[slice * D + c] = dgam[0];
            part_kbk[slice * D + c] = kbk;
            __syncthreads();
            float later = sm.fC[c] * sm.e15[c] * sm.gsum[c];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                later += part_kbk[s2 * D + c];
                if (s2 > slice) later += part_sum[s2 * D + c];
            }
            if (vstore) {
                float *sg = reinterpret_cast<float *>(base + O_SG);   // [C][D]
#pragma unroll
                for (int u = 0; u < 8; ++u) sg[(x0 + u) * D + c] = dgam[u] + later;
                __syncthreads();
                // dq, dk: 512 chunks of 8 bf16 each; dg: 1024 chunks of 4 fp32
                {
                    const int r = t >> 4, c8 = (t & 15) * 8;
                    if (r < L) {
                        const int64_t off = (t0 + r) * rowK + (int64_t)h * D + c8;
                        *reinterpret_cast<uint4 *>(dq + off) =
                            *reinterpret_cast<const uint4 *>(base + O_SQ + (r * D + c8) * 2);
                        *reinterpret_cast<uint4 *>(dk + off) =
                            *reinterpret_cast<const uint4 *>(base + O_SK + (r * D + c8) * 2);
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int q = t + kThreads * i, r = q >> 5, c4 = (q & 31) * 4;
                    if (r < L)
                        *reinterpret_cast<float4 *>(dg + (t0 + r) * rowK + (int64_t)h * D + c4) =
                            *reinterpret_cast<const float4 *>(sg + r * D + c4);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (x0 + u < L) dg[(t0 + x0 + u) * rowK + (int64_t)h * D + c] = dgam[u] + later;
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
    // every MMA and tile copy issued has completed (after a stop too)
    if (warp < kIssuers) {
        tc_fence_after();
        mma_commit_el(&sm.mma_bar);
    }
    if (t == 0) {
        mbar_wait_bounded(&sm.mma_bar, mma_par, kPollLimit);
        if (tiles_pending) mbar_wait_bounded(&sm.tma_bar, pend_par, kPollLimit);
    }
    if (t == kS0Issuer && s0_pending) mbar_wait_bounded(&sm.s0_bar, s0_par, kPollLimit);
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
    CUtensorMap mcs = {}, minit = {};
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    const int vec_out = P.out_dtype == KDA_DTYPE_BF16 && al16(dq) && al16(dk) && al16(dv) && al16(dg);
    const int has_cs = chunk_states && chunk_capacity > 0;
    const int has_init = init_state != nullptr;
    if (has_cs && !kda_make_state_map(&mcs, chunk_states, chunk_capacity * P.H * (int64_t)D))
        return cudaErrorInvalidValue;
    if (has_init && !kda_make_state_map(&minit, init_state, (int64_t)P.N * P.H * D))
        return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((int64_t)P.N * P.H);
    if (P.out_dtype == KDA_DTYPE_BF16) {
        auto kern = kda_backward_tc_kernel<__nv_bfloat16>;
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem); });
        if (attr != cudaSuccess) return attr;
        kern<<<blocks, kThreads, kSmem, stream>>>(mq, mk, mv, mdo, mg, mcs, minit, has_cs, has_init, vec_out,
                                                  beta, init_state, cu, chunk_states, chunk_capacity, d_final,
                                                  (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk,
                                                  (__nv_bfloat16 *)dv, dg, dbeta, d_init, P.H,
                                                  (int64_t)P.T, P.seq_len);
    } else {
        auto kern = kda_backward_tc_kernel<float>;
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem); });
        if (attr != cudaSuccess) return attr;
        kern<<<blocks, kThreads, kSmem, stream>>>(mq, mk, mv, mdo, mg, mcs, minit, has_cs, has_init, 0,
                                                  beta, init_state, cu, chunk_states, chunk_capacity, d_final,
                                                  (float *)dq, (float *)dk, (float *)dv, dg, dbeta, d_init,
                                                  P.H, (int64_t)P.T, P.seq_len);
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
