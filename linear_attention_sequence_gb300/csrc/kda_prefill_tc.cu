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
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPollLimit = 1u << 23;  // about half a second of polling

// tensor-memory columns
constexpr uint32_t TM_S = 0;    // S^T, 128 columns (fp32 state)
constexpr uint32_t TM_X = 128;  // [ (W S)^T | (gamma Q S)^T -> O^T ], 64 columns
constexpr uint32_t TM_U = 192;  // U'^T, then U^T, 32 columns
constexpr uint32_t TM_W = 224;  // W^T (lanes = key channel), 32 columns
constexpr uint32_t TM_G = 256;  // Gram, 48 columns

constexpr uint32_t kChunkBytes = C * D * (2 + 2 + 2 + 4);

struct alignas(1024) TcSmem {
    // inputs of one chunk, TMA destinations, dense row-major [C][D]
    __nv_bfloat16 q[C * D];
    __nv_bfloat16 k[C * D];
    __nv_bfloat16 v[C * D];
    float g[C * D];           // g, then Gamma in place
    // MMA operands, tf32, K-major SW128 (see sm100_ptx.cuh)
    float gramA[4 * 64 * 32];  // 4 K-blocks x 64 rows; must be followed by >= 8 KB of smem
    float gramB[4 * 48 * 32];  // 4 K-blocks x 48 rows
    float bgkT[D * 32];        // (beta gamma k)^T: row = key channel, k = token
    float bvT[D * 32];         // (beta v)^T: row = value index, k = token
    float tmat[32 * 32];       // T: row = token r, k = token i
    float aqk[32 * 32];        // Aqk: row = token r, k = token i
    float bX[4 * 64 * 32];     // [W ; gamma q]: row = token, k = key channel
    float kbT[D * 32];         // Kbar^T: row = key channel, k = token
    // fp32 scratch
    float akk[32][33];
    float beta[C];
    float gref[D], e01[D], e1l[D], gamC[D];
    uint64_t bar_tma, bar_mma;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void st_op(float *blk, int row, int k, float x) {
    *reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(blk) + sw128_off32(row, k)) =
        to_tf32(x);
}

__device__ __forceinline__ void issue_chunk_loads(TcSmem &sm, const CUtensorMap *mq,
                                                  const CUtensorMap *mk, const CUtensorMap *mv,
                                                  const CUtensorMap *mg, int h, int64_t t0) {
    mbar_arrive_expect_tx(&sm.bar_tma, kChunkBytes);
    const int x = h * D, y = (int)t0;
    tma_load_2d(sm.q, mq, &sm.bar_tma, x, y);
    tma_load_2d(sm.k, mk, &sm.bar_tma, x, y);
    tma_load_2d(sm.v, mv, &sm.bar_tma, x, y);
    tma_load_2d(sm.g, mg, &sm.bar_tma, x, y);
}

// Bounded wait by every thread; on timeout raise the CTA-wide abort flag and
// the device status word.  Callers follow it with a barrier and test sm.abort.
__device__ __forceinline__ bool wait_phase(TcSmem &sm, uint64_t *bar, uint32_t parity,
                                           unsigned code) {
    if (!mbar_wait_bounded(bar, parity, kPollLimit)) {
        sm.abort = 1;
        atomicOr(&g_kda_device_status, code);
        return false;
    }
    return true;
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

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const bool wg0 = warp < 4;
    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);
    const int nchunks = (int)((b - a + C - 1) / C);

    if (t == 0) {
        mbar_init(&sm.bar_tma, 1);
        mbar_init(&sm.bar_mma, 1);
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
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int64_t state_off = ((int64_t)n * H + h) * D * D;

    // S^T into TMEM: thread j of warpgroup 0 holds column j of S (row j of S^T)
    if (wg0) {
        const int j = t;
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = init_state ? init_state[state_off + (int64_t)(c0 + i) * D + j] : 0.f;
            tmem_st16(tb + lane_off + TM_S + c0, v);
        }
        tmem_wait_st();
    }
    // Per-thread bookkeeping of what is in flight, for the abort path: a
    // pending copy or MMA stays pending in the thread whose wait gave up, with
    // the parity it was waiting for.
    uint32_t tma_phase = 0, mma_phase = 0, tma_pend_par = 0, mma_pend_par = 0;
    bool tma_pending = false, mma_pending = false;
    if (t == 0 && nchunks > 0) issue_chunk_loads(sm, &tm_q, &tm_k, &tm_v, &tm_g, h, a);
    tma_pending = nchunks > 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    for (int ci = 0; ci < nchunks; ++ci) {
        const int64_t t0 = a + (int64_t)ci * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);

        if (wait_phase(sm, &sm.bar_tma, tma_phase, 1u)) tma_pending = false;
        tma_phase ^= 1u;
        __syncthreads();
        if (sm.abort) break;

        // ---- a1: Gamma = running sum of g (rows past the sequence end count as 0) ----
        if (t < D) {
            float run = 0.f, g15 = 0.f;
            for (int r = 0; r < C; ++r) {
                run += r < L ? sm.g[r * D + t] : 0.f;
                sm.g[r * D + t] = run;
                if (r == 15) g15 = run;
            }
            sm.gref[t] = g15;
            sm.e01[t] = __expf(g15);
            sm.e1l[t] = __expf(run - g15);
            sm.gamC[t] = __expf(run);
        }
        if (t < C) sm.beta[t] = t < L ? beta[(t0 + t) * H + h] : 0.f;
        __syncthreads();

        // ---- a2: decay-weighted operands ----
        {
            const int c = t & (D - 1);
            const int kb = c >> 5, kc = c & 31;
            const float gref = sm.gref[c], e01 = sm.e01[c], e1l = sm.e1l[c];
            for (int r = t >> 7; r < C; r += kThreads / D) {
                const bool live = r < L;
                const int sub = r >> 4;
                const float G = sm.g[r * D + c];
                const float e1 = __expf(G - (sub ? gref : 0.f));    // in [e^-80, 1]
                const float inv = 1.0f / e1;                         // in [1, e^80]
                const float kv = live ? __bfloat162float(sm.k[r * D + c]) : 0.f;
                const float qv = live ? __bfloat162float(sm.q[r * D + c]) : 0.f;
                const float vv = live ? __bfloat162float(sm.v[r * D + c]) : 0.f;
                const float bt = sm.beta[r];
                float *gA = sm.gramA + kb * 64 * 32;
                float *gB = sm.gramB + kb * 48 * 32;
                st_op(gA, r, kc, kv * e1);
                st_op(gA, 32 + r, kc, qv * e1);
                const float kinv = kv * inv;
                if (sub == 0) {
                    st_op(gB, r, kc, kinv);
                    st_op(gB, 16 + r, kc, kinv * e01);
                } else {
                    st_op(gB, 16 + r, kc, kinv);
                }
                const float gam = sub ? e1 * e01 : e1;               // e^{Gamma_r}
                st_op(sm.bX + kb * 64 * 32, 32 + r, kc, gam * qv);
                st_op(sm.bgkT, c, r, bt * gam * kv);
                st_op(sm.bvT, c, r, bt * vv);
                const float kbar = (sub ? e1l : e1l * e01) * inv;    // e^{Gamma_last - Gamma_r}
                st_op(sm.kbT, c, r, kbar * kv);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // the input buffers are consumed: fetch the next chunk now
        if (ci + 1 < nchunks) {
            if (t == 0) issue_chunk_loads(sm, &tm_q, &tm_k, &tm_v, &tm_g, h, t0 + C);
            tma_pending = true;
            tma_pend_par = tma_phase;
        }

        // ---- a3: Gram matrices, one 128 x 48 x 128 MMA ----
        if (t == 0) {
            tc_fence_after();
            const uint32_t aA = smem_u32(sm.gramA), aB = smem_u32(sm.gramB);
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t da = sdesc_sw128(aA + (kk >> 2) * (64 * 128) + (kk & 3) * 32);
                const uint64_t db = sdesc_sw128(aB + (kk >> 2) * (48 * 128) + (kk & 3) * 32);
                mma_tf32_ss(tb + TM_G, da, db, idesc_tf32(128, 48), kk > 0);
            }
            mma_commit(&sm.bar_mma);
        }
        mma_pending = true;
        mma_pend_par = mma_phase;
        if (wait_phase(sm, &sm.bar_mma, mma_phase, 2u)) mma_pending = false;
        mma_phase ^= 1u;
        tc_fence_after();
        __syncthreads();
        if (sm.abort) break;

        // ---- a4: Akk (strict, beta rows) and Aqk (inclusive) from the Gram ----
        if (warp < 2) {
            float d0[16], d1[16], d2[16];
            tmem_ld16x2(tb + lane_off + TM_G + 0, tb + lane_off + TM_G + 16, d0, d1);
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
                    st_op(sm.aqk, r, i, i <= r ? val : 0.f);
                }
            }
        }
        __syncthreads();
        // T = (I + Akk)^{-1}: lane i of warp 0 solves column i (right-looking)
        if (warp == 0) {
            float x[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = r == lane ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 31; ++m) {
                const float xm = x[m];
#pragma unroll
                for (int r = m + 1; r < 32; ++r) x[r] -= sm.akk[r][m] * xm;
            }
#pragma unroll
            for (int r = 0; r < 32; ++r) st_op(sm.tmat, r, lane, x[r]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- W^T = (beta gamma K)^T T^T and U'^T = (beta V)^T T^T ----
        if (t == 0) {
            tc_fence_after();
            const uint32_t aW = smem_u32(sm.bgkT), aV = smem_u32(sm.bvT), aT = smem_u32(sm.tmat);
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ss(tb + TM_W, sdesc_sw128(aW + kk * 32), sdesc_sw128(aT + kk * 32),
                            idesc_tf32(128, 32), kk > 0);
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ss(tb + TM_U, sdesc_sw128(aV + kk * 32), sdesc_sw128(aT + kk * 32),
                            idesc_tf32(128, 32), kk > 0);
            mma_commit(&sm.bar_mma);
        }
        mma_pending = true;
        mma_pend_par = mma_phase;
        if (wait_phase(sm, &sm.bar_mma, mma_phase, 4u)) mma_pending = false;
        mma_phase ^= 1u;
        tc_fence_after();
        __syncthreads();
        if (sm.abort) break;

        // W (row = token, k = key channel) into the readout operand
        if (wg0) {
            float w0[16], w1[16];
            tmem_ld16x2(tb + lane_off + TM_W + 0, tb + lane_off + TM_W + 16, w0, w1);
            const int c = t;
            float *blk = sm.bX + (c >> 5) * 64 * 32;
#pragma unroll
            for (int r = 0; r < 16; ++r) st_op(blk, r, c & 31, w0[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r) st_op(blk, 16 + r, c & 31, w1[r]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- a5: X^T = S^T [W ; gamma Q]^T, A operand = the state in TMEM ----
        if (t == 0) {
            tc_fence_after();
            const uint32_t aX = smem_u32(sm.bX);
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32_ts(tb + TM_X, tb + TM_S + kk * 8,
                            sdesc_sw128(aX + (kk >> 2) * (64 * 128) + (kk & 3) * 32),
                            idesc_tf32(128, 64), kk > 0);
            mma_commit(&sm.bar_mma);
        }
        mma_pending = true;
        mma_pend_par = mma_phase;
        if (wait_phase(sm, &sm.bar_mma, mma_phase, 8u)) mma_pending = false;
        mma_phase ^= 1u;
        tc_fence_after();
        __syncthreads();
        if (sm.abort) break;

        // U^T = U'^T - (W S)^T (warpgroup 0); S^T <- S^T Diag(gamma_last) (warpgroup 1)
        if (wg0) {
            float u0[16], u1[16], x0[16], x1[16];
            tmem_ld16x2(tb + lane_off + TM_U + 0, tb + lane_off + TM_U + 16, u0, u1);
            tmem_ld16x2(tb + lane_off + TM_X + 0, tb + lane_off + TM_X + 16, x0, x1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                u0[i] = to_tf32(u0[i] - x0[i]);
                u1[i] = to_tf32(u1[i] - x1[i]);
            }
            tmem_st16(tb + lane_off + TM_U + 0, u0);
            tmem_st16(tb + lane_off + TM_U + 16, u1);
            tmem_wait_st();
        } else {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
                float s[16];
                tmem_ld16(tb + lane_off + TM_S + c0, s);
#pragma unroll
                for (int i = 0; i < 16; ++i) s[i] *= sm.gamC[c0 + i];
                tmem_st16(tb + lane_off + TM_S + c0, s);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();

        // ---- a5/a6: O^T += U^T Aqk^T ; S^T += U^T Kbar ----
        if (t == 0) {
            tc_fence_after();
            const uint32_t aQ = smem_u32(sm.aqk), aK = smem_u32(sm.kbT);
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_X + 32, tb + TM_U + kk * 8, sdesc_sw128(aQ + kk * 32),
                            idesc_tf32(128, 32), 1u);
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_S, tb + TM_U + kk * 8, sdesc_sw128(aK + kk * 32),
                            idesc_tf32(128, 128), 1u);
            mma_commit(&sm.bar_mma);
        }
        mma_pending = true;
        mma_pend_par = mma_phase;
        if (wait_phase(sm, &sm.bar_mma, mma_phase, 16u)) mma_pending = false;
        mma_phase ^= 1u;
        tc_fence_after();
        __syncthreads();
        if (sm.abort) break;

        // ---- a7: output rows of this chunk ----
        if (wg0) {
            float o0[16], o1[16];
            tmem_ld16x2(tb + lane_off + TM_X + 32, tb + lane_off + TM_X + 48, o0, o1);
            const int j = t;
            OUT_T *dst = out + (t0 * H + h) * (int64_t)D + j;
            const int64_t row = (int64_t)H * D;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < L) kda::st_elem(dst + r * row, o0[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (16 + r < L) kda::st_elem(dst + (16 + r) * row, o1[r]);
        }
        tc_fence_before();
    }

    __syncthreads();
    if (!sm.abort) {
        if (final_state && wg0) {
            const int j = t;
            for (int c0 = 0; c0 < D; c0 += 16) {
                float s[16];
                tmem_ld16(tb + lane_off + TM_S + c0, s);
#pragma unroll
                for (int i = 0; i < 16; ++i) final_state[state_off + (int64_t)(c0 + i) * D + j] = s[i];
            }
        }
    } else {
        // drain what is still in flight before the shared and tensor memory go away
        if (tma_pending) mbar_wait_bounded(&sm.bar_tma, tma_pend_par, kPollLimit);
        if (mma_pending) mbar_wait_bounded(&sm.bar_mma, mma_pend_par, kPollLimit);
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
