// kda_prefill_tc.cu -- chunked KDA prefill on the sm_103a tensor cores (tcgen05).
//
// Same chunk form as the fp32 kernel ("Inside Kimi K3", section "Sequence
// mixing": tokens of a chunk in parallel, inclusive diagonal, state carried
// between chunks; "Hybrid Attention", section "But isn't a recurrent update
// sequential?": a triangular solve resolves the in-chunk dependencies):
//
//   T   = (I + Akk)^{-1},  W = T diag(beta)(gamma . K),  U' = T diag(beta) V
//   U   = U' - W S0
//   O   = (gamma . Q) S0 + Aqk U
//   S_C = Diag(gamma_last) S0 + Kbar^T U,   Kbar_r = e^{Gamma_last - Gamma_r} . k_r
//
// with Gamma the running sum of g inside the chunk and gamma = e^Gamma.
//
// One CTA owns one (sequence, head) for the whole sequence; chunks of C = 32
// tokens.  Every product is a tcgen05.mma of kind::tf32 with an fp32
// accumulator in tensor memory; the state S^T (lanes = value index, columns =
// key channel) lives in TMEM for the whole sequence, is the A operand of the
// readout GEMM straight from TMEM and accumulates its own update in place.
//
// Warp specialisation.  Warps 0-7 prepare chunk n (decay prefix, decay-
// weighted operands, Gram MMA, triangular solve, W and U' MMAs) while warps
// 8-15 run the state chain of chunk n-1 (readout MMA, U = U' - W S and the
// state decay, intra-chunk readout and state-carry MMAs, output store).  The
// two groups hand buffers to each other through mbarriers; every wait is
// bounded.
// tf32 (not bf16) operands: on these inputs the intermediate u_t and the
// intra-chunk terms are several times larger than o_t, and bf16 operand
// rounding alone costs more than the 2e-2 error budget; tf32 keeps it near
// 5e-3.  Inputs of the next chunk are fetched by TMA while the current one
// is processed.
//
// Decay factoring.  Products e^{Gamma_r - Gamma_i} (i <= r) are split into
// two bounded factors around a reference inside the chunk.  The chunk is two
// 16-token sub-tiles; with the log-decay bounded below by g_min = -5 the
// cumulative decay over one sub-tile stays above e^{-80} ("Understanding Kimi
// K3's Attention", log-decay bound; "Kimi K3.1 and the Road ...", section 5),
// so e^{Gamma_r - Gamma_s} and its inverse stay inside fp32 range when r and s
// are in the same sub-tile.  Rows use the start of their own sub-tile as the
// reference; columns come in two variants (reference = start of sub-tile 0 or
// of sub-tile 1), so the Gram matrices are one 128 x 48 x 128 MMA:
//   rows  0..31 : k_r e^{Gamma_r - ref(r)}     rows 32..63: q_r e^{Gamma_r - ref(r)}
//   cols  0..15 : k_i e^{0 - Gamma_i}          (i in sub-tile 0, reference 0)
//   cols 16..47 : k_i e^{Gamma_15 - Gamma_i}   (i = 0..31,   reference Gamma_15)
// (the A operand is 128 rows; rows 64..127 alias the next buffer and their
// results are ignored).

#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"

__device__ unsigned int g_kda_device_status;  // nonzero after a bounded wait gave up

namespace {

using namespace sm100;

constexpr int C = 32;        // tokens per chunk
constexpr int D = 128;       // d_k = d_v
constexpr int kPrep = 256;   // threads of the chunk-preparation warps (warps 0-7)
constexpr int kChain = 256;  // threads of the state-chain warps (warps 8-15)
constexpr int kThreads = kPrep + kChain;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPollLimit = 1u << 23;  // about half a second of polling per wait

// named barriers (0 is __syncthreads)
constexpr uint32_t BAR_PREP = 1, BAR_CHAIN = 2, BAR_WG0 = 3;

// tensor-memory columns
constexpr uint32_t TM_S = 0;     // S^T (lanes = value index, columns = key channel), fp32 state
constexpr uint32_t TM_X = 128;   // two buffers of 64: [(W S)^T | (gamma Q S)^T -> O^T]
constexpr uint32_t TM_U = 256;   // two buffers of 32: U'^T, then U^T
constexpr uint32_t TM_W = 320;   // W^T (lanes = key channel)
constexpr uint32_t TM_G = 352;   // Gram, 48 columns
constexpr uint32_t TM_BGK = 400; // (beta gamma k)^T: lanes = key channel, columns = token
constexpr uint32_t TM_BV = 432;  // (beta v)^T: lanes = value index, columns = token

constexpr uint32_t kStageBytes = C * D * (2 + 2 + 2 + 4);

struct Stage {
    __nv_bfloat16 q[C * D];
    __nv_bfloat16 k[C * D];
    __nv_bfloat16 v[C * D];
    float g[C * D];  // g, then Gamma in place
};

struct alignas(1024) TcSmem {
    Stage in[2];               // TMA destinations, dense row-major [C][D], double-buffered
    float gramA[4 * 64 * 32];  // Gram A operand (tf32, SW128): rows 0-31 k~, 32-63 q~;
                               // also fp32 scratch of the triangular solve
    float gramB[4 * 48 * 32];  // Gram B operand; its first 8 KB are read as rows 64-127 of gramA
    float bX[4 * 64 * 32];     // readout B operand [W ; gamma q] (single buffer)
    float kbT[2][D * 32];      // Kbar^T (state-carry B operand), per chunk parity
    float aqk[2][32 * 32];     // Aqk (intra-chunk readout B operand), per chunk parity
    float tmat[32 * 32];       // T = (I + Akk)^{-1} (B operand of the W / U' MMAs)
    float akk[32][33];
    float beta[C];
    float gref[D], e01[D], glast[D];
    float gamC[2][D];          // e^{Gamma_last}, per chunk parity (state decay of the chain)
    uint64_t bar_tma[2], bar_gram, bar_wu, bar_bxfull, bar_bxempty, bar_x, bar_s;
    uint64_t bar_akempty[2], bar_xfree[2];
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void st_op(float *blk, int row, int k, float x) {
    *reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(blk) + sw128_off32(row, k)) =
        to_tf32(x);
}
// 16-byte store of the four consecutive-k elements k4*4 .. k4*4+3 of `row`.
__device__ __forceinline__ void st_op4(float *blk, int row, int k4, float a, float b, float c,
                                       float d) {
    const uint32_t addr = smem_u32(blk) + (uint32_t)(row * 128 + (((k4 ^ row) & 7) << 4));
    st_shared_v4(addr, to_tf32(a), to_tf32(b), to_tf32(c), to_tf32(d));
}

__device__ __forceinline__ void issue_stage_loads(Stage &st, uint64_t *bar, const CUtensorMap *mq,
                                                  const CUtensorMap *mk, const CUtensorMap *mv,
                                                  const CUtensorMap *mg, int h, int64_t t0) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    const int x = h * D, y = (int)t0;
    tma_load_2d(st.q, mq, bar, x, y);
    tma_load_2d(st.k, mk, bar, x, y);
    tma_load_2d(st.v, mv, bar, x, y);
    tma_load_2d(st.g, mg, bar, x, y);
}

// Bounded wait; on timeout raise the CTA abort flag and the device status.
__device__ __forceinline__ bool wait_phase(TcSmem &sm, uint64_t *bar, uint32_t parity,
                                           unsigned code) {
    if (!mbar_wait_bounded(bar, parity, kPollLimit)) {
        *reinterpret_cast<volatile int *>(&sm.abort) = 1;
        atomicOr(&g_kda_device_status, code);
        return false;
    }
    return true;
}
__device__ __forceinline__ bool aborted(TcSmem &sm) {
    return *reinterpret_cast<volatile int *>(&sm.abort) != 0;
}

// ---------------------------------------------------------------------------
// Preparation warps (0-7): everything of chunk n that does not depend on the
// state -- decay prefix, decay-weighted operands, Gram matrices, the
// triangular solve, W and U' -- done while the chain warps run chunk n-1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prep_loop(TcSmem &sm, const CUtensorMap *mq, const CUtensorMap *mk,
                                          const CUtensorMap *mv, const CUtensorMap *mg,
                                          const float *__restrict__ beta, int H, int h, int64_t a,
                                          int64_t b, int nchunks, uint32_t tb) {
    const int p = threadIdx.x;            // 0..255
    const int warp = p >> 5, lane = p & 31;
    const bool wg0 = p < 128;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t tma_par[2] = {0, 0}, ake_par[2] = {0, 0};
    uint32_t gram_par = 0, wu_par = 0, bxe_par = 0;
    // in-flight bookkeeping for the abort path (valid in the thread that gave up)
    bool pend_tma[2] = {false, false}, pend_gram = false, pend_wu = false;
    uint32_t pend_tma_par[2] = {0, 0};

    if (p == 0) {
        for (int s = 0; s < 2 && s < nchunks; ++s)
            issue_stage_loads(sm.in[s], &sm.bar_tma[s], mq, mk, mv, mg, h, a + (int64_t)s * C);
    }
    __syncwarp();
    for (int s = 0; s < 2; ++s) pend_tma[s] = s < nchunks;

    for (int n = 0; n < nchunks; ++n) {
        const int st = n & 1;
        const int64_t t0 = a + (int64_t)n * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        Stage &in = sm.in[st];

        // chunk n-2 (same parity) must be finished by the chain before its
        // aqk / kbT / gamC / U buffers are overwritten
        if (n >= 2) {
            wait_phase(sm, &sm.bar_akempty[st], ake_par[st], 32u);
            ake_par[st] ^= 1u;
        }
        if (wait_phase(sm, &sm.bar_tma[st], tma_par[st], 1u)) pend_tma[st] = false;
        tma_par[st] ^= 1u;
        if (named_sync_or(BAR_PREP, kPrep, aborted(sm))) break;

        // ---- a1: Gamma (running sum of g per key channel), beta ----
        if (wg0) {
            const int c = p;
            float run = 0.f, g15 = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                run += r < L ? in.g[r * D + c] : 0.f;
                in.g[r * D + c] = run;
                if (r == 15) g15 = run;
            }
            sm.gref[c] = g15;
            sm.e01[c] = __expf(g15);
            sm.glast[c] = run;
            sm.gamC[st][c] = __expf(run);
        } else if (p < 128 + C) {
            const int r = p - 128;
            sm.beta[r] = r < L ? beta[(t0 + r) * H + h] : 0.f;
        }
        named_sync(BAR_PREP, kPrep);

        // ---- a2: Gram operands, 4 tokens x 4 channels per thread ----
        // (warp w: tokens 4w..4w+3; lane: channels 4*lane..4*lane+3)
        {
            const int cb = lane, c0 = 4 * cb, kb = cb >> 3, k4 = cb & 7;
            const float4 gref4 = *reinterpret_cast<const float4 *>(&sm.gref[c0]);
            const float4 e014 = *reinterpret_cast<const float4 *>(&sm.e01[c0]);
            float *gA = sm.gramA + kb * 64 * 32;
            float *gB = sm.gramB + kb * 48 * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * warp + i;
                const bool live = r < L, sub1 = r >= 16;
                const float4 G = *reinterpret_cast<const float4 *>(&in.g[r * D + c0]);
                const uint2 kraw = *reinterpret_cast<const uint2 *>(&in.k[r * D + c0]);
                const uint2 qraw = *reinterpret_cast<const uint2 *>(&in.q[r * D + c0]);
                const __nv_bfloat162 k01 = *reinterpret_cast<const __nv_bfloat162 *>(&kraw.x);
                const __nv_bfloat162 k23 = *reinterpret_cast<const __nv_bfloat162 *>(&kraw.y);
                const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw.x);
                const __nv_bfloat162 q23 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw.y);
                float kv[4] = {__low2float(k01), __high2float(k01), __low2float(k23), __high2float(k23)};
                float qv[4] = {__low2float(q01), __high2float(q01), __low2float(q23), __high2float(q23)};
                const float gv[4] = {G.x, G.y, G.z, G.w};
                const float rf[4] = {gref4.x, gref4.y, gref4.z, gref4.w};
                const float ef[4] = {e014.x, e014.y, e014.z, e014.w};
                float ka[4], qa[4], kinv[4], kinv1[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!live) { kv[j] = 0.f; qv[j] = 0.f; }
                    const float e1 = __expf(gv[j] - (sub1 ? rf[j] : 0.f));  // [e^-80, 1]
                    const float inv = __frcp_rn(e1);                         // [1, e^80]
                    ka[j] = kv[j] * e1;
                    qa[j] = qv[j] * e1;
                    kinv[j] = kv[j] * inv;
                    kinv1[j] = kinv[j] * ef[j];
                }
                st_op4(gA, r, k4, ka[0], ka[1], ka[2], ka[3]);
                st_op4(gA, 32 + r, k4, qa[0], qa[1], qa[2], qa[3]);
                if (!sub1) {
                    st_op4(gB, r, k4, kinv[0], kinv[1], kinv[2], kinv[3]);
                    st_op4(gB, 16 + r, k4, kinv1[0], kinv1[1], kinv1[2], kinv1[3]);
                } else {
                    st_op4(gB, 16 + r, k4, kinv[0], kinv[1], kinv[2], kinv[3]);
                }
            }
        }
        fence_proxy_async_smem();
        named_sync(BAR_PREP, kPrep);
        if (p == 0) {
            tc_fence_after();
            const uint32_t aA = smem_u32(sm.gramA), aB = smem_u32(sm.gramB);
#pragma unroll 1
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t da = sdesc_sw128(aA + (kk >> 2) * (64 * 128) + (kk & 3) * 32);
                const uint64_t db = sdesc_sw128(aB + (kk >> 2) * (48 * 128) + (kk & 3) * 32);
                mma_tf32_ss(tb + TM_G, da, db, idesc_tf32(128, 48), kk > 0);
            }
            mma_commit(&sm.bar_gram);
        }
        __syncwarp();   // reconverge warp 0 before its warp-collective tcgen05 operations
        pend_gram = true;

        if (wg0) {
            // ---- (beta gamma k)^T into TMEM: thread = key channel, 32 tokens ----
            const int c = p;
            float v0[16], v1[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float kv = r < L ? __bfloat162float(in.k[r * D + c]) : 0.f;
                v0[r] = to_tf32(sm.beta[r] * __expf(in.g[r * D + c]) * kv);
                const int r1 = 16 + r;
                const float kv1 = r1 < L ? __bfloat162float(in.k[r1 * D + c]) : 0.f;
                v1[r] = to_tf32(sm.beta[r1] * __expf(in.g[r1 * D + c]) * kv1);
            }
            tmem_st16(tb + lane_off + TM_BGK, v0);
            tmem_st16(tb + lane_off + TM_BGK + 16, v1);
            tmem_wait_st();
            tc_fence_before();

            // ---- Gram -> Akk (strict, beta rows) and Aqk (inclusive) ----
            if (wait_phase(sm, &sm.bar_gram, gram_par, 2u)) pend_gram = false;
            gram_par ^= 1u;
            tc_fence_after();
            if (warp < 2) {
                float d0[16], d1[16], d2[16];
                tmem_ld16x2(tb + lane_off + TM_G, tb + lane_off + TM_G + 16, d0, d1);
                tmem_ld16(tb + lane_off + TM_G + 32, d2);
                const int r = lane;
                if (warp == 0) {
                    const float br = sm.beta[r];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float val = r < 16 ? (i < 16 ? d0[i] : 0.f) : (i < 16 ? d1[i] : d2[i - 16]);
                        sm.akk[r][i] = i < r ? br * val : 0.f;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float val = r < 16 ? (i < 16 ? d0[i] : 0.f) : (i < 16 ? d1[i] : d2[i - 16]);
                        st_op(sm.aqk[st], r, i, i <= r ? val : 0.f);
                    }
                }
            }
            tc_fence_before();
            named_sync(BAR_WG0, 128);

            // ---- T = (I + Akk)^{-1}, blocked 2 x 2 over 16-token sub-tiles ----
            float(*Tm)[33] = reinterpret_cast<float(*)[33]>(sm.gramA);           // fp32 T
            float(*Y)[17] = reinterpret_cast<float(*)[17]>(sm.gramA + 32 * 33);   // A10 T00
            if (warp == 0) {
                // diagonal blocks: lanes 0-15 -> columns of T00, lanes 16-31 -> columns of T11
                const int base = lane < 16 ? 0 : 16, col = lane & 15;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = r == col ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 15; ++m) {
                    const float xm = x[m];
#pragma unroll
                    for (int r = m + 1; r < 16; ++r) x[r] -= sm.akk[base + r][base + m] * xm;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    Tm[base + r][base + col] = x[r];
                    Tm[base + r][16 - base + col] = 0.f;   // upper off-diagonal block / placeholder
                }
            }
            named_sync(BAR_WG0, 128);
            {   // Y = A10 T00   (A10 = Akk[16..31][0..15]); 256 entries, 2 per thread
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int idx = p + 128 * e, i = idx >> 4, j = idx & 15;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc += sm.akk[16 + i][m] * Tm[m][j];
                    Y[i][j] = acc;
                }
            }
            named_sync(BAR_WG0, 128);
            {   // T10 = -T11 Y
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int idx = p + 128 * e, i = idx >> 4, j = idx & 15;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc += Tm[16 + i][16 + m] * Y[m][j];
                    Tm[16 + i][j] = -acc;
                }
            }
            named_sync(BAR_WG0, 128);
            {   // T into its tf32 operand: thread -> row p / 4, 8 consecutive columns
                const int r = p >> 2, c0 = (p & 3) * 8;
                st_op4(sm.tmat, r, c0 >> 2, Tm[r][c0], Tm[r][c0 + 1], Tm[r][c0 + 2], Tm[r][c0 + 3]);
                st_op4(sm.tmat, r, (c0 >> 2) + 1, Tm[r][c0 + 4], Tm[r][c0 + 5], Tm[r][c0 + 6],
                       Tm[r][c0 + 7]);
            }
            fence_proxy_async_smem();
        } else {
            // ---- (beta v)^T into TMEM and Kbar^T into smem: thread = channel ----
            const int c = p - 128;
            float v0[16], v1[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                v0[r] = to_tf32(r < L ? sm.beta[r] * __bfloat162float(in.v[r * D + c]) : 0.f);
                const int r1 = 16 + r;
                v1[r] = to_tf32(r1 < L ? sm.beta[r1] * __bfloat162float(in.v[r1 * D + c]) : 0.f);
            }
            tmem_st16(tb + lane_off + TM_BV, v0);
            tmem_st16(tb + lane_off + TM_BV + 16, v1);
            const float gl = sm.glast[c];
            float *kb = sm.kbT[st];
#pragma unroll
            for (int r4 = 0; r4 < 8; ++r4) {
                float kbar[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * r4 + j;
                    const float kv = r < L ? __bfloat162float(in.k[r * D + c]) : 0.f;
                    kbar[j] = kv * __expf(gl - in.g[r * D + c]);   // e^{Gamma_last - Gamma_r} <= 1
                }
                st_op4(kb, c, r4, kbar[0], kbar[1], kbar[2], kbar[3]);
            }
            tmem_wait_st();
            tc_fence_before();
            // gamma q rows of the readout operand: bX is single-buffered, so wait
            // for the readout MMA of chunk n-1 to have consumed it
            if (n >= 1) {
                wait_phase(sm, &sm.bar_bxempty, bxe_par, 4u);
                bxe_par ^= 1u;
            }
            const int q_ = c, cb = q_ & 31, c0 = 4 * cb, kb4 = cb >> 3, k4 = cb & 7;
            float *blk = sm.bX + kb4 * 64 * 32;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 8 * (q_ >> 5) + i;
                const bool live = r < L;
                const float4 G = *reinterpret_cast<const float4 *>(&in.g[r * D + c0]);
                const uint2 qraw = *reinterpret_cast<const uint2 *>(&in.q[r * D + c0]);
                const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw.x);
                const __nv_bfloat162 q23 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw.y);
                const float s = live ? 1.f : 0.f;
                st_op4(blk, 32 + r, k4, s * __low2float(q01) * __expf(G.x),
                       s * __high2float(q01) * __expf(G.y), s * __low2float(q23) * __expf(G.z),
                       s * __high2float(q23) * __expf(G.w));
            }
            fence_proxy_async_smem();
        }
        named_sync(BAR_PREP, kPrep);

        // ---- W^T = (beta gamma K)^T T^T ; U'^T = (beta V)^T T^T (A operands in TMEM) ----
        if (p == 0) {
            tc_fence_after();
            const uint32_t aT = smem_u32(sm.tmat);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_W, tb + TM_BGK + kk * 8, sdesc_sw128(aT + kk * 32),
                            idesc_tf32(128, 32), kk > 0);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_U + 32 * st, tb + TM_BV + kk * 8, sdesc_sw128(aT + kk * 32),
                            idesc_tf32(128, 32), kk > 0);
            mma_commit(&sm.bar_wu);
        }
        __syncwarp();
        pend_wu = true;
        if (wg0) {
            if (wait_phase(sm, &sm.bar_wu, wu_par, 8u)) pend_wu = false;
            wu_par ^= 1u;
            tc_fence_after();
            if (n >= 1) {   // bX single-buffered (see above)
                wait_phase(sm, &sm.bar_bxempty, bxe_par, 4u);
                bxe_par ^= 1u;
            }
            // W rows (token r, key channel c) of the readout operand
            float w0[16], w1[16];
            tmem_ld16x2(tb + lane_off + TM_W, tb + lane_off + TM_W + 16, w0, w1);
            const int c = p;
            float *blk = sm.bX + (c >> 5) * 64 * 32;
#pragma unroll
            for (int r = 0; r < 16; ++r) st_op(blk, r, c & 31, w0[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r) st_op(blk, 16 + r, c & 31, w1[r]);
            fence_proxy_async_smem();
            tc_fence_before();
        }
        const bool stop = named_sync_or(BAR_PREP, kPrep, aborted(sm));
        if (p == 0 && !stop) {
            mbar_arrive(&sm.bar_bxfull);   // chunk n ready for the chain
            if (n + 2 < nchunks) {
                issue_stage_loads(sm.in[st], &sm.bar_tma[st], mq, mk, mv, mg, h, t0 + 2 * C);
                pend_tma_par[st] = tma_par[st];
            }
        }
        __syncwarp();
        if (n + 2 < nchunks) pend_tma[st] = true;
        if (stop) break;
    }
    if (aborted(sm)) {   // drain what this thread saw in flight
        for (int s = 0; s < 2; ++s)
            if (pend_tma[s] && p == 0) mbar_wait_bounded(&sm.bar_tma[s], pend_tma_par[s], kPollLimit);
        if (pend_gram) mbar_wait_bounded(&sm.bar_gram, gram_par, kPollLimit);
        if (pend_wu) mbar_wait_bounded(&sm.bar_wu, wu_par, kPollLimit);
    }
}

// ---------------------------------------------------------------------------
// Chain warps (8-15): the state-dependent part of chunk n.
// ---------------------------------------------------------------------------
template <typename OUT_T>
__device__ __forceinline__ void chain_loop(TcSmem &sm, OUT_T *__restrict__ out, int H, int h,
                                           int64_t a, int64_t b, int nchunks, uint32_t tb) {
    const int ct = threadIdx.x - kPrep;   // 0..255
    const int warp = threadIdx.x >> 5;    // 8..15
    const bool wg2 = ct < 128;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int j = ct & 127;               // value index = TMEM lane
    const bool issuer = ct == 0;
    uint32_t bxf_par = 0, x_par = 0, s_par = 0, xfree_par[2] = {0, 0};
    bool pend_x = false, pend_s = false;

    for (int n = 0; n < nchunks; ++n) {
        const int st = n & 1;
        const int64_t t0 = a + (int64_t)n * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        const uint32_t tx = TM_X + 64 * st, tu = TM_U + 32 * st;

        if (issuer) {
            bool ok = wait_phase(sm, &sm.bar_bxfull, bxf_par, 64u);
            bxf_par ^= 1u;
            if (ok && n >= 2) {
                ok = wait_phase(sm, &sm.bar_xfree[st], xfree_par[st], 128u);
                xfree_par[st] ^= 1u;
            }
            if (ok) {
                tc_fence_after();
                // X^T = S^T [W ; gamma Q]^T, A operand = the state in TMEM
                const uint32_t aX = smem_u32(sm.bX);
#pragma unroll 1
                for (int kk = 0; kk < 16; ++kk)
                    mma_tf32_ts(tb + tx, tb + TM_S + kk * 8,
                                sdesc_sw128(aX + (kk >> 2) * (64 * 128) + (kk & 3) * 32),
                                idesc_tf32(128, 64), kk > 0);
                mma_commit(&sm.bar_x);
                mma_commit(&sm.bar_bxempty);
            }
        }
        __syncwarp();
        pend_x = true;
        if (wait_phase(sm, &sm.bar_x, x_par, 16u)) pend_x = false;
        x_par ^= 1u;
        tc_fence_after();
        if (named_sync_or(BAR_CHAIN, kChain, aborted(sm))) break;

        // U^T = U'^T - (W S)^T ; S^T <- S^T Diag(e^{Gamma_last})
        if (wg2) {
            float u0[16], u1[16], x0[16], x1[16];
            tmem_ld16x2(tb + lane_off + tu, tb + lane_off + tu + 16, u0, u1);
            tmem_ld16x2(tb + lane_off + tx, tb + lane_off + tx + 16, x0, x1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                u0[i] = to_tf32(u0[i] - x0[i]);
                u1[i] = to_tf32(u1[i] - x1[i]);
            }
            tmem_st16(tb + lane_off + tu, u0);
            tmem_st16(tb + lane_off + tu + 16, u1);
        }
        {
            const int cbase = wg2 ? 0 : 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float s0[16], s1[16];
                const uint32_t col = TM_S + cbase + c0;
                tmem_ld16x2(tb + lane_off + col, tb + lane_off + col + 16, s0, s1);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    s0[i] *= sm.gamC[st][cbase + c0 + i];
                    s1[i] *= sm.gamC[st][cbase + c0 + 16 + i];
                }
                tmem_st16(tb + lane_off + col, s0);
                tmem_st16(tb + lane_off + col + 16, s1);
            }
        }
        tmem_wait_st();
        tc_fence_before();
        named_sync(BAR_CHAIN, kChain);

        // O^T += U^T Aqk^T (into the gamma-Q-S half of X) ; S^T += U^T Kbar
        if (issuer) {
            tc_fence_after();
            const uint32_t aQ = smem_u32(sm.aqk[st]), aK = smem_u32(sm.kbT[st]);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + tx + 32, tb + tu + kk * 8, sdesc_sw128(aQ + kk * 32),
                            idesc_tf32(128, 32), 1u);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_S, tb + tu + kk * 8, sdesc_sw128(aK + kk * 32),
                            idesc_tf32(128, 128), 1u);
            mma_commit(&sm.bar_s);
            mma_commit(&sm.bar_akempty[st]);
        }
        __syncwarp();
        pend_s = true;
        if (wait_phase(sm, &sm.bar_s, s_par, 16u)) pend_s = false;
        s_par ^= 1u;
        tc_fence_after();

        // ---- output rows of chunk n (warpgroup 3), then release X[st] ----
        if (!wg2) {
            float o0[16], o1[16];
            tmem_ld16x2(tb + lane_off + tx + 32, tb + lane_off + tx + 48, o0, o1);
            OUT_T *dst = out + (t0 * H + h) * (int64_t)D + j;
            const int64_t row = (int64_t)H * D;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < L) kda::st_elem(dst + r * row, o0[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (16 + r < L) kda::st_elem(dst + (16 + r) * row, o1[r]);
            tc_fence_before();
            mbar_arrive(&sm.bar_xfree[st]);
        }
    }
    if (aborted(sm)) {
        if (pend_x) mbar_wait_bounded(&sm.bar_x, x_par, kPollLimit);
        if (pend_s) mbar_wait_bounded(&sm.bar_s, s_par, kPollLimit);
    }
}

template <typename OUT_T>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g, const float *__restrict__ beta,
                      const float *__restrict__ init_state, const int32_t *__restrict__ cu,
                      OUT_T *__restrict__ out, float *__restrict__ final_state, int H,
                      int64_t total, int64_t seq_len) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TcSmem &sm = *reinterpret_cast<TcSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int t = threadIdx.x, warp = t >> 5;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);
    const int nchunks = (int)((b - a + C - 1) / C);

    if (t == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.bar_tma[s], 1);
            mbar_init(&sm.bar_akempty[s], 1);
            mbar_init(&sm.bar_xfree[s], 128);
        }
        mbar_init(&sm.bar_gram, 1);
        mbar_init(&sm.bar_wu, 1);
        mbar_init(&sm.bar_bxfull, 1);
        mbar_init(&sm.bar_bxempty, 1);
        mbar_init(&sm.bar_x, 1);
        mbar_init(&sm.bar_s, 1);
        fence_mbar_init();
        sm.abort = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm.tmem_base;
    const int64_t state_off = ((int64_t)n * H + h) * D * D;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool state_wg = t >= kPrep && t < kPrep + 128;   // warpgroup 2: lanes = value index

    // initial state into TMEM: thread j holds column j of S (row j of S^T)
    if (state_wg) {
        const int j = t - kPrep;
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = init_state ? init_state[state_off + (int64_t)(c0 + i) * D + j] : 0.f;
            tmem_st16(tb + lane_off + TM_S + c0, v);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (t < kPrep)
        prep_loop(sm, &tm_q, &tm_k, &tm_v, &tm_g, beta, H, h, a, b, nchunks, tb);
    else
        chain_loop<OUT_T>(sm, out, H, h, a, b, nchunks, tb);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!aborted(sm) && final_state && state_wg) {
        const int j = t - kPrep;
        for (int c0 = 0; c0 < D; c0 += 16) {
            float s[16];
            tmem_ld16(tb + lane_off + TM_S + c0, s);
#pragma unroll
            for (int i = 0; i < 16; ++i) final_state[state_off + (int64_t)(c0 + i) * D + j] = s[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kTmemCols);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view [T rows, H*D columns] of a [T, H, D] tensor, box = C rows x D columns.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int64_t T,
              int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * D * esize};
    const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)C};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename OUT_T>
cudaError_t launch(const kda::Problem &P, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *init_state, const int32_t *cu,
                   void *out, float *final_state, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mg;
    if (!make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !make_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.T, P.H))
        return cudaErrorInvalidValue;
    auto kern = kda_prefill_tc_kernel<OUT_T>;
    const size_t smem = sizeof(TcSmem) + 1024;
    static_assert(sizeof(TcSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((int64_t)P.N * P.H);
    kern<<<blocks, kThreads, smem, stream>>>(mq, mk, mv, mg, beta, init_state, cu, (OUT_T *)out,
                                             final_state, P.H, (int64_t)P.T, P.seq_len);
    return cudaGetLastError();
}

}  // namespace

bool kda_prefill_tc_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g) {
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    return P.dk == 128 && P.dv == 128 && P.in_dtype == KDA_DTYPE_BF16 && P.T > 0 &&
           P.T <= 0x7fffffff - C && al16(q) && al16(k) && al16(v) && al16(g) && encode_fn() != nullptr;
}

cudaError_t kda_launch_prefill_tc(const kda::Problem &P, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta,
                                  const float *init_state, const int32_t *cu, void *out,
                                  float *final_state, cudaStream_t stream) {
    if (P.N == 0) return cudaSuccess;
    if (P.out_dtype == KDA_DTYPE_BF16)
        return launch<__nv_bfloat16>(P, q, k, v, g, beta, init_state, cu, out, final_state, stream);
    return launch<float>(P, q, k, v, g, beta, init_state, cu, out, final_state, stream);
}

cudaError_t kda_read_device_status(cudaStream_t stream, unsigned *status) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(status, g_kda_device_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_kda_device_status, &zero, sizeof(unsigned));
}
