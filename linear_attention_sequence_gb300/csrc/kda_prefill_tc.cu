// kda_prefill_tc.cu -- chunked KDA prefill on the sm_103a tensor cores (tcgen05).
//
// Same chunk form as the fp32 kernel ("Inside Kimi K3", section "Sequence
// mixing": tokens of a chunk in parallel, inclusive diagonal, state carried
// between chunks; "Hybrid Attention", section "But isn't a recurrent update
// sequential?": a triangular solve resolves the in-chunk dependencies):
//
//   T   = (I + Akk)^{-1}
//   U   = T diag(beta) V - T diag(beta) (gamma . K) S0        (= U' - ...)
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
// Warp specialisation.  Warps 0-7 prepare chunk n: decay prefix,
// decay-weighted operands, the Gram MMA.  Warps 8-11 run the rest of a chunk.
// Warps 10 and 11 issue the readout MMA X = S^T [gamma Q; gamma K]^T as soon as
// the chunk's operand is in place (it needs no solve) and then decay their half
// of the state; meanwhile warps 8 and 9 extract the intra-chunk matrices from
// the Gram and solve the triangular system.  Then, on all four: U' = T diag(beta)
// V and the U MMA that subtracts (gamma K S) T diag(beta) with the X accumulator
// itself as A operand (one accumulator, one issuing thread), the rest of the
// state decay, one MMA group for the intra-chunk readout and the state carry
// together, and the output store (a TMA store of a staged tile for a full
// chunk).  The two groups hand buffers to each other through mbarriers; every
// wait is bounded.  The thread
// that issues a tcgen05.mma or a TMA load is held for roughly the time the
// unit needs to accept it, so each issue is given to a warp that has nothing
// else to do at that point.  A tcgen05.mma costs a roughly fixed time per
// instruction on these shapes, so the formulation minimises the instruction
// count: 16 for the Gram and 16 for the readout (K = d_k = 128), 4 each for
// U', U and the readout + state-carry group.  The loop bodies are long, and
// instruction fetch is a visible share of the stalls: a few loops are kept
// rolled or only partly unrolled where that costs no latency on the chunk's
// path (the state decay, the Gram A copy, the MMA issue loops).
// tf32 (not bf16) operands: on these inputs the intermediate u_t and the
// intra-chunk terms are several times larger than o_t, and bf16 operand
// rounding alone costs more than the 2e-2 error budget; tf32 keeps it near
// 5e-3.  Inputs of the next chunk are fetched by TMA while the current one
// is processed.
//
// Decay factoring.  Products e^{Gamma_r - Gamma_i} (i <= r) are split into
// two bounded factors around the reference Gamma_15 (the running sum after
// the 16th token of the chunk).  With the log-decay bounded below by
// g_min = -5, |Gamma_r - Gamma_15| <= 16 * 5 = 80 for every token r of a
// 32-token chunk ("Understanding Kimi K3's Attention", log-decay bound;
// "Kimi K3.1 and the Road ...", section 5), so e^{Gamma_r - Gamma_15} and its
// inverse stay inside the fp32 (and tf32) normal range.  The Gram matrices
// are then one 128 x 32 x 128 MMA group:
//   A rows  0..31 : k_r e^{Gamma_r - Gamma_15}     rows 32..63: q_r e^{Gamma_r - Gamma_15}
//   B rows  0..31 : k_i e^{Gamma_15 - Gamma_i}
// (the A operand sits in TMEM lanes 0-63; lanes 64-127 are not used and their
// results are ignored).

#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"

__device__ unsigned int g_kda_device_status;  // nonzero after a bounded wait gave up

namespace {

using namespace sm100;

constexpr int C = 32;        // tokens per chunk
constexpr int D = 128;       // d_k = d_v
constexpr int kPrep = 256;   // chunk-preparation threads (warps 0-7)
constexpr int kChain = 128;  // state-chain threads (warps 8-11; thread j <-> TMEM lane j)
constexpr int kThreads = kPrep + kChain;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPollLimit = 1u << 23;  // about half a second of polling per wait

// Named barriers.  A phase of an mbarrier is awaited by one thread, and a named
// barrier releases the threads that depend on it: hundreds of threads polling
// mbarriers slow every other mbarrier and tensor-core operation of the SM.
constexpr uint32_t BAR_PREP = 1, BAR_CHAIN = 2, BAR_E1 = 3, BAR_A1 = 5, BAR_XG = 6;
constexpr int kGramIssuer = 96;   // warp 3: issues the Gram MMA once its operands are in place
constexpr int kTmaIssuer = 224;   // warp 7: issues the first two stage loads
constexpr int kBetaRing = 4;      // beta of chunk n sits in slot n % 4 (the prep runs <= 2 chunks ahead)

// tensor-memory columns
constexpr uint32_t TM_S = 0;     // 128: S^T (lanes = value index, columns = key channel)
constexpr uint32_t TM_X = 128;   // 64: [(gamma Q S)^T, then O^T | (gamma K S)^T]
constexpr uint32_t TM_U = 192;   // 2 x 32: U'^T, then U^T, per chunk parity
constexpr uint32_t TM_BV = 256;  // 32: V^T of even chunks, A operand of the U' MMA
constexpr uint32_t TM_BV1 = 352; // 32: V^T of odd chunks
constexpr uint32_t TM_G = 288;   // 2 x 32: Gram, per chunk parity
constexpr uint32_t TM_GA = 384;  // 128: Gram A operand, lanes 0-31 k~, 32-63 q~

constexpr uint32_t kTileBf16 = C * D * 2;
constexpr uint32_t kTileF32 = C * D * 4;
constexpr uint32_t kStageBytes = 3 * kTileBf16 + kTileF32;
constexpr uint32_t kStageBytesGated = 4 * kTileBf16;   // z (bf16 decay logits) in place of g

// Input tiles arrive by TMA with the 128-byte swizzle: a bf16 tile is two
// 4 KB halves (32 rows x 64 elements), an fp32 tile four 4 KB quarters (32
// rows x 32 elements); the 16-byte chunk ch of row r sits at chunk position
// ch ^ (r % 8).  Rows of a warp then fall in distinct banks whether a warp
// walks along a row, down a column, or over 4-element blocks.
__device__ __forceinline__ uint32_t off_bf16(int r, int c) {
    return (uint32_t)((c >> 6) * 4096 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ uint32_t off_f32(int r, int c) {
    return (uint32_t)((c >> 5) * 4096 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + ((c & 3) << 2));
}

// A stage holds the TMA-loaded inputs of one chunk and then, once they are
// consumed, that chunk's readout B operand [gamma q ; gamma k] (32 KB, SW128
// K-major, over the q, k, v tiles and the first quarter of g) until the
// readout MMA has read it.
struct Stage {
    unsigned char q[kTileBf16];
    unsigned char k[kTileBf16];
    unsigned char v[kTileBf16];
    unsigned char g[kTileF32];  // g, then Gamma in place
};
static_assert(4 * 64 * 32 * 4 <= sizeof(Stage), "readout operand fits in a stage");

struct alignas(1024) TcSmem {
    Stage in[2];                // TMA destinations, double-buffered
    unsigned char ostage[2][kTileF32];   // output rows of a full chunk, stored by TMA (SW128)
    float gramA[4 * 64 * 32];   // staging of the Gram A operand [k~ ; q~] (tf32), copied to TMEM
    float gramB[4 * 32 * 32];   // Gram B operand k e^{Gamma_15 - Gamma}
    float kbaq[2][160 * 32];    // [Kbar^T ; Aqk]: B operand of the state-carry + readout MMA
    float tmat[2][32 * 32];     // T diag(beta): B operand of the U' MMA and, negated, of the U MMA
    float akkT[32][32];         // solve scratch: (beta-scaled strict lower Akk)^T
    float tsc[3][16][20];       // solve scratch: T11 by rows, T22^T, A21 T11 (rows padded)
    float betaS[kBetaRing][C];
    float ghS[kBetaRing][C];    // one log-decay per token (scalar-decay variants), like beta
    float gamC[2][D];           // e^{Gamma_last}: state decay over the chunk
    float gref[D], e01[D], e1l[D];
    uint64_t bar_tma[2], bar_gram[2], bar_bxfull[2], bar_gops[2], bar_akempty[2];
    uint64_t bar_x, bar_u, bar_s, bar_fin[3];
    uint32_t tma_issued[2];     // stage loads issued / awaited (for the drain after a stop)
    uint32_t tma_awaited[2];
    uint32_t tmem_base;
    int abort;
    int seq_of_slot;            // the sequence this CTA runs (longest first)
};

// Stores into K-major SW128 operand blocks (plain C++ stores, so the
// compiler can schedule around them; fence.proxy.async orders them before the
// MMAs that read them).
__device__ __forceinline__ void st_op(float *blk, int row, int k, float x) {
    *reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(blk) + sw128_off32(row, k)) =
        to_tf32(x);
}
// 16-byte store of the elements 4*k4 .. 4*k4+3 of `row`.
__device__ __forceinline__ void st_op4(float *blk, int row, int k4, float a, float b, float c,
                                       float d) {
    *reinterpret_cast<float4 *>(reinterpret_cast<unsigned char *>(blk) + row * 128 +
                                (((k4 ^ row) & 7) << 4)) =
        make_float4(to_tf32(a), to_tf32(b), to_tf32(c), to_tf32(d));
}
__device__ __forceinline__ float4 ld_f32x4(const void *tile, int r, int c) {
    return *reinterpret_cast<const float4 *>(reinterpret_cast<const unsigned char *>(tile) +
                                             off_f32(r, c));
}
__device__ __forceinline__ void ld_bf16x4(const unsigned char *tile, int r, int c, float (&x)[4]) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(tile + off_bf16(r, c));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    x[0] = __low2float(a);
    x[1] = __high2float(a);
    x[2] = __low2float(b);
    x[3] = __high2float(b);
}
__device__ __forceinline__ float ld_bf16(const unsigned char *tile, int r, int c) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + off_bf16(r, c)));
}

// How the decay arrives: 0 = the fp32 log-decay g by TMA; 1 = the bf16 decay
// logits z by TMA (gate prologue; `mg` maps z, two segments per head like q,
// and the box lands in the first half of the g tile); 2 = one log-decay per
// (token, head), fetched with beta (no tile).
constexpr int kDecayTile = 0, kDecayLogits = 1, kDecayScalar = 2;
__device__ __forceinline__ void issue_stage_loads(Stage &st, uint64_t *bar, const CUtensorMap *mq,
                                                  const CUtensorMap *mk, const CUtensorMap *mv,
                                                  const CUtensorMap *mg, int h, int64_t t0,
                                                  int gmode) {
    // one box per tensor: {128-byte segment, C tokens, the head's segments}
    mbar_arrive_expect_tx(bar, gmode == kDecayScalar   ? 3 * kTileBf16
                               : gmode == kDecayLogits ? kStageBytesGated
                                                       : kStageBytes);
    const int y = (int)t0;
    tma_load_3d(st.q, mq, bar, 0, y, 2 * h);
    tma_load_3d(st.k, mk, bar, 0, y, 2 * h);
    tma_load_3d(st.v, mv, bar, 0, y, 2 * h);
    if (gmode != kDecayScalar) tma_load_3d(st.g, mg, bar, 0, y, (gmode == kDecayLogits ? 2 : 4) * h);
}

// Bounded wait for a phase.  The first poll is inline; the polling loop (and
// the error path) is a single out-of-line copy, which keeps the loop bodies of
// the kernel small enough for the instruction caches.
__device__ __noinline__ bool wait_phase_slow(TcSmem &sm, uint64_t *bar, uint32_t parity,
                                             unsigned code) {
    if (!mbar_wait_bounded(bar, parity, kPollLimit)) {
        *reinterpret_cast<volatile int *>(&sm.abort) = 1;
        atomicOr(&g_kda_device_status, code);
        return false;
    }
    return true;
}
__device__ __forceinline__ bool wait_phase(TcSmem &sm, uint64_t *bar, uint32_t parity,
                                           unsigned code) {
    return mbar_try_wait(bar, parity) || wait_phase_slow(sm, bar, parity, code);
}
__device__ __forceinline__ bool aborted(TcSmem &sm) {
    return *reinterpret_cast<volatile int *>(&sm.abort) != 0;
}

// ---------------------------------------------------------------------------
// Preparation warps (0-7): the decay prefix and decay-weighted operands of
// chunk n and its Gram MMA, done while the chain warps run chunk n-1.
// ---------------------------------------------------------------------------
template <bool GATED, bool SDECAY>
__device__ __forceinline__ void prep_loop(TcSmem &sm, const CUtensorMap *mq, const CUtensorMap *mk,
                                          const CUtensorMap *mv, const CUtensorMap *mg,
                                          const float *__restrict__ beta,
                                          const float *__restrict__ g_head, int H, int h, int64_t a,
                                          int64_t b, int nchunks, uint32_t tb, float gscale) {
    constexpr bool gated = GATED;
    constexpr int gmode = GATED ? kDecayLogits : SDECAY ? kDecayScalar : kDecayTile;
    const int P = threadIdx.x;  // 0..255
    const int warp = P >> 5, lane = P & 31, qd = warp & 3, wg = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    uint32_t tma_par[2] = {0, 0}, ake_par[2] = {0, 0}, gram_par[2] = {0, 0};
    const bool beta_thread = P >= 128 && P < 128 + C;

    // beta of chunk 0 (asynchronous 4-byte copies; rows past the end are 0), and
    // with a scalar decay the log-decay of each token (0 without one: the delta rule)
    if (beta_thread) {
        const int r = P - 128;
        const bool in_seq = nchunks > 0 && a + r < b;
        if (in_seq) cp_async4(&sm.betaS[0][r], beta + (a + r) * H + h);
        else sm.betaS[0][r] = 0.f;
        if (SDECAY) {
            if (in_seq && g_head) cp_async4(&sm.ghS[0][r], g_head + (a + r) * H + h);
            else sm.ghS[0][r] = 0.f;
        }
        cp_async_commit();
    }
    if (P == kTmaIssuer)
        for (int s = 0; s < 2 && s < nchunks; ++s) {
            issue_stage_loads(sm.in[s], &sm.bar_tma[s], mq, mk, mv, mg, h, a + (int64_t)s * C, gmode);
            sm.tma_issued[s] = 1;
        }
    __syncwarp();

    for (int n = 0; n < nchunks; ++n) {
        const int st = n & 1;
        const int64_t t0 = a + (int64_t)n * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        Stage &in = sm.in[st];

        // The chain must be done with chunk n-2 (same parity) before its
        // buffers (kbaq, gamC, Gram TMEM) are overwritten, and the inputs of
        // chunk n must have landed.  One thread waits; the barrier below
        // releases the others (and orders their reads after the TMA writes).
        if (P == 0) {
            if (n >= 2) wait_phase(sm, &sm.bar_akempty[st], ake_par[st], 32u);
            if (wait_phase(sm, &sm.bar_tma[st], tma_par[st], 1u)) sm.tma_awaited[st] += 1;
        }
        if (n >= 2) ake_par[st] ^= 1u;
        tma_par[st] ^= 1u;
        if (beta_thread) {
            cp_async_wait_all();   // beta of chunk n has landed
            const int r = P - 128;
            if (gated && r < L) {   // beta = Sigmoid(logit) inside the sequence; zeros stay zeros
                float *bn = &sm.betaS[n % kBetaRing][r];
                *bn = kda::sigmoid_f(*bn);
            }
            const int64_t tn = t0 + C + r;
            const bool in_seq = n + 1 < nchunks && tn < b;
            float *dst = &sm.betaS[(n + 1) % kBetaRing][r];
            if (in_seq) cp_async4(dst, beta + tn * H + h);
            else *dst = 0.f;
            if (SDECAY) {
                float *gdst = &sm.ghS[(n + 1) % kBetaRing][r];
                if (in_seq && g_head) cp_async4(gdst, g_head + tn * H + h);
                else *gdst = 0.f;
            }
            cp_async_commit();
        }
        if (named_sync_or(BAR_PREP, kPrep, aborted(sm))) break;

        // ---- a1 (gate prologue): g = g_min Sigmoid(e^{A_h} z) from the bf16 logits,
        // on all eight warps: rows 0-15 on warps 0-3, rows 16-31 on warps 4-7, which
        // hand theirs over through the upper half of the g slot (the bf16 logits
        // fill only the lower half).  The barrier also orders every read of z
        // before Gamma (fp32) overwrites the slot. ----
        float zg[C / 2];
        if (gated) {
            const int c = P & (D - 1), hf = P / D;
#pragma unroll
            for (int r = 0; r < C / 2; ++r)
                zg[r] = kda::gate_g(ld_bf16(in.g, (C / 2) * hf + r, c), gscale);
            float *handoff = reinterpret_cast<float *>(in.g + kTileBf16);   // [C / 2][D]
            if (hf) {
#pragma unroll
                for (int r = 0; r < C / 2; ++r) handoff[r * D + c] = zg[r];
            }
            named_sync(BAR_PREP, kPrep);
        }

        // ---- a1: Gamma = running sum of g per key channel (all loads first) ----
        if (P < D) {
            const int c = P;
            float *g = reinterpret_cast<float *>(in.g);
            float gv[C];
            if (gated) {
                const float *handoff = reinterpret_cast<const float *>(in.g + kTileBf16);
#pragma unroll
                for (int r = 0; r < C / 2; ++r) {
                    gv[r] = zg[r];
                    gv[C / 2 + r] = handoff[r * D + c];
                }
                named_sync(BAR_A1, D);   // every hand-off value is read before Gamma overwrites it
            } else if (SDECAY) {
                // one log-decay per token, the same for every key channel
                const float *gh = sm.ghS[n % kBetaRing];
#pragma unroll
                for (int r = 0; r < C; ++r) gv[r] = gh[r];
            } else {
#pragma unroll
                for (int r = 0; r < C; ++r) gv[r] = g[off_f32(r, c) >> 2];
            }
            float run = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                run += r < L ? gv[r] : 0.f;
                gv[r] = run;
            }
#pragma unroll
            for (int r = 0; r < C; ++r) g[off_f32(r, c) >> 2] = gv[r];
            const float g15 = gv[15], gl = gv[C - 1];
            sm.gref[c] = g15;
            sm.e01[c] = __expf(g15);
            sm.e1l[c] = __expf(gl - g15);
            sm.gamC[st][c] = __expf(gl);
        }
        // the Gram MMA of chunk n-1 must be done with its operands (gramB in
        // shared memory, the A operand in TMEM) before they are rewritten
        if (P == 0 && n >= 1) wait_phase(sm, &sm.bar_gram[st ^ 1], gram_par[st ^ 1], 2u);
        if (n >= 1) gram_par[st ^ 1] ^= 1u;
        named_sync(BAR_PREP, kPrep);

        // ---- a2: one pass over (token, 4-channel) blocks: Gram operands, Kbar^T, and
        // the readout operand values (stored once the previous readout is done).
        // Thread P handles tokens (P % 8) + 8 it, channels 4 (P / 8) .. +3. ----
        float gq[4][4], gk[4][4];
        {
            const int cb = P >> 3, c = 4 * cb, kb = cb >> 3, k4 = cb & 7;
            float4 G[4];
            float kx[4][4], qx[4][4];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = (P & 7) + 8 * it;
                G[it] = ld_f32x4(in.g, r, c);
                ld_bf16x4(in.k, r, c, kx[it]);
                ld_bf16x4(in.q, r, c, qx[it]);
            }
            const float4 gr4 = *reinterpret_cast<const float4 *>(&sm.gref[c]);
            const float4 e4 = *reinterpret_cast<const float4 *>(&sm.e01[c]);
            const float4 l4 = *reinterpret_cast<const float4 *>(&sm.e1l[c]);
            const float gref[4] = {gr4.x, gr4.y, gr4.z, gr4.w};
            const float e01[4] = {e4.x, e4.y, e4.z, e4.w};
            const float e1l[4] = {l4.x, l4.y, l4.z, l4.w};
            float *gA = sm.gramA + kb * 64 * 32;
            float *gB = sm.gramB + kb * 32 * 32;
            float *kbq = sm.kbaq[st];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = (P & 7) + 8 * it;
                const float sc = r < L ? 1.f : 0.f;
                const float gv[4] = {G[it].x, G[it].y, G[it].z, G[it].w};
                float ka[4], qa[4], kv[4], kbar[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float e1 = __expf(gv[m] - gref[m]);      // e^{Gamma_r - Gamma_15}, [e^-80, e^75]
                    const float inv = __fdividef(1.f, e1);
                    const float kk = sc * kx[it][m], qq = sc * qx[it][m];
                    ka[m] = kk * e1;
                    qa[m] = qq * e1;
                    kv[m] = kk * inv;                               // k e^{Gamma_15 - Gamma_r}
                    gq[it][m] = qa[m] * e01[m];                     // q e^{Gamma_r}
                    gk[it][m] = ka[m] * e01[m];                     // k e^{Gamma_r}
                    kbar[m] = kv[m] * e1l[m];                       // k e^{Gamma_last - Gamma_r}
                }
                st_op4(gA, r, k4, ka[0], ka[1], ka[2], ka[3]);
                st_op4(gA, 32 + r, k4, qa[0], qa[1], qa[2], qa[3]);
                st_op4(gB, r, k4, kv[0], kv[1], kv[2], kv[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m) st_op(kbq, c + m, r, kbar[m]);
            }
        }
        fence_proxy_async_smem();
        named_sync(BAR_PREP, kPrep);

        // ---- a3: Gram A operand staging -> TMEM (warps 0, 1); V^T -> TMEM (warps 4-7) ----
        if (warp < 2) {
            tc_fence_after();   // after the Gram MMA of chunk n-1 (awaited above)
            const int r = lane, row = 32 * warp + r;     // warp 0: k~ rows, warp 1: q~ rows
#pragma unroll 2
            for (int c0 = 0; c0 < D; c0 += 16) {
                const float *blk = sm.gramA + (c0 >> 5) * 64 * 32;
                float vals[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k4 = ((c0 & 31) >> 2) + j;
                    const float4 x = *reinterpret_cast<const float4 *>(
                        reinterpret_cast<const unsigned char *>(blk) + row * 128 + (((k4 ^ row) & 7) << 4));
                    vals[4 * j + 0] = x.x;
                    vals[4 * j + 1] = x.y;
                    vals[4 * j + 2] = x.z;
                    vals[4 * j + 3] = x.w;
                }
                tmem_st16(tb + lane_off + TM_GA + c0, vals);
            }
            tmem_wait_st();
            tc_fence_before();
        } else if (wg == 1) {
            // V^T (thread = value index) into the buffer of this parity; the U' MMA
            // of chunk n-2 that read it is complete (akempty of chunk n-2, awaited above)
            tc_fence_after();
            const int j = P - 128;
            const uint32_t tbv = st ? TM_BV1 : TM_BV;
            float v0[16], v1[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                v0[r] = r < L ? ld_bf16(in.v, r, j) : 0.f;
                v1[r] = 16 + r < L ? ld_bf16(in.v, 16 + r, j) : 0.f;
            }
            tmem_st16(tb + lane_off + tbv, v0);
            tmem_st16(tb + lane_off + tbv + 16, v1);
            tmem_wait_st();
            tc_fence_before();
        }
        named_sync(BAR_PREP, kPrep);   // the inputs of chunk n are consumed
        // Beta and the Gram operands of chunk n are in place: the chain may start
        // its extraction once the Gram MMA, issued here, completes.  The issue
        // holds warp 3 for about a microsecond; its share of the stores below
        // waits meanwhile, and the readout MMA that needs them has slack.
        if (P == 0) mbar_arrive(&sm.bar_gops[st]);
        if (P == kGramIssuer) {
            tc_fence_after();
            const uint64_t dB = sdesc_sw128(smem_u32(sm.gramB));
#pragma unroll 8
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32_ts(tb + TM_G + 32 * st, tb + TM_GA + kk * 8,
                            dB + (uint64_t)(((kk >> 2) * (32 * 128) + (kk & 3) * 32) >> 4),
                            idesc_tf32(128, 32), kk > 0);
            mma_commit(&sm.bar_gram[st]);
        }
        __syncwarp();

        // ---- readout operand [gamma q ; gamma k] into the chunk's own stage ----
        {
            const int cb = P >> 3, k4 = cb & 7;
            float *blk = reinterpret_cast<float *>(&in) + (cb >> 3) * 64 * 32;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = (P & 7) + 8 * it;
                st_op4(blk, r, k4, gq[it][0], gq[it][1], gq[it][2], gq[it][3]);
                st_op4(blk, 32 + r, k4, gk[it][0], gk[it][1], gk[it][2], gk[it][3]);
            }
        }
        // End of chunk n: after the barrier thread 0 hands the chunk to the chain.
        fence_proxy_async_smem();
        named_sync(BAR_PREP, kPrep);
        if (P == 0) mbar_arrive(&sm.bar_bxfull[st]);   // chunk n is ready for the chain
        // (a stop is agreed on by the vote at the top of the next chunk)
    }
    if (beta_thread) cp_async_wait_all();
    if (P == kGramIssuer) {      // every Gram MMA issued here has completed
        mma_commit(&sm.bar_fin[0]);
        mbar_wait_bounded(&sm.bar_fin[0], 0, kPollLimit);
    }
}

// Element (r, c) of an output tile in the TMA box layout (SW128 segments of 128 bytes).
template <typename OUT_T>
__device__ __forceinline__ void st_stage(unsigned char *tile, int r, int c, float x) {
    if constexpr (sizeof(OUT_T) == 2)
        *reinterpret_cast<__nv_bfloat16 *>(tile + off_bf16(r, c)) = __float2bfloat16_rn(x);
    else
        *reinterpret_cast<float *>(tile + off_f32(r, c)) = x;
}

// S^T <- S^T Diag(e^{Gamma_last}) on the 32 lanes of the calling warp (`tl` =
// TMEM base + the warp's lane offset).
__device__ __forceinline__ void scale_state(TcSmem &sm, uint32_t tl, int st) {
    // rolled (each load waits for its data anyway): less code for the instruction caches
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
        float s0[16], s1[16];
        tmem_ld16x2(tl + TM_S + c0, tl + TM_S + c0 + 16, s0, s1);
        const float4 *gc = reinterpret_cast<const float4 *>(&sm.gamC[st][c0]);
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const float4 a4 = gc[i4], b4 = gc[4 + i4];
            s0[4 * i4] *= a4.x; s0[4 * i4 + 1] *= a4.y; s0[4 * i4 + 2] *= a4.z; s0[4 * i4 + 3] *= a4.w;
            s1[4 * i4] *= b4.x; s1[4 * i4 + 1] *= b4.y; s1[4 * i4 + 2] *= b4.z; s1[4 * i4 + 3] *= b4.w;
        }
        tmem_st16(tl + TM_S + c0, s0);
        tmem_st16(tl + TM_S + c0 + 16, s1);
    }
    tmem_wait_st();
    tc_fence_before();
}

// ---------------------------------------------------------------------------
// Chain warps (8-11): everything of chunk n from its Gram on.  Thread j owns
// TMEM lane j = value index j; warps 8 and 9 read the Gram rows (lanes 0-63).
// ---------------------------------------------------------------------------
template <typename OUT_T>
__device__ __forceinline__ void chain_loop(TcSmem &sm, const CUtensorMap *mq, const CUtensorMap *mk,
                                           const CUtensorMap *mv, const CUtensorMap *mg,
                                           const CUtensorMap *mo, OUT_T *__restrict__ out, int H,
                                           int h, int64_t a, int64_t b, int nchunks, uint32_t tb,
                                           float *__restrict__ ckpt, int64_t ckpt_every,
                                           int64_t ckpt_cap, int64_t ck_row0, int gmode) {
    const int j = threadIdx.x - kPrep;   // 0..127
    const int warp = threadIdx.x >> 5, cw = j >> 5, lane = j & 31;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool issuer = j == 0, xissuer = j == 96, ostorer = j == 32;
    uint32_t bxf_par[2] = {0, 0}, gops_par[2] = {0, 0}, gram_par[2] = {0, 0}, x_par = 0, u_par = 0, s_par = 0;

    for (int n = 0; n < nchunks; ++n) {
        const int st = n & 1;
        const int64_t t0 = a + (int64_t)n * C;
        const int L = (int)((b - t0) < C ? (b - t0) : C);
        const uint32_t tu = TM_U + 32 * st;
        const float *betaN = sm.betaS[n % kBetaRing];

        // Two hand-overs from the preparation warps: the Gram of chunk n (with its
        // beta) for the extraction and solve, and the whole chunk (gamma_last,
        // readout operand, Kbar^T, V^T) for the readout MMA and what follows.
        if (cw >= 2) {
            // ---- a5: X^T = S^T [gamma Q ; gamma K]^T (warps 10, 11).  It needs only
            // the state and the readout operand, so it runs while warps 8, 9
            // extract and solve; then S^T <- S^T Diag(e^{Gamma_last}) on lanes 64-127. ----
            if (xissuer) {
                if (wait_phase(sm, &sm.bar_bxfull[st], bxf_par[st], 64u)) {
                    tc_fence_after();
                    const uint64_t dX = sdesc_sw128(smem_u32(&sm.in[st]));   // the chunk's stage
                    // partly unrolled: the loop's code stays small for the
                    // instruction caches while the issues still run back to back
#pragma unroll 4
                    for (int kk = 0; kk < 16; ++kk)
                        mma_tf32_ts(tb + TM_X, tb + TM_S + kk * 8,
                                    dX + (uint64_t)(((kk >> 2) * (64 * 128) + (kk & 3) * 32) >> 4),
                                    idesc_tf32(128, 64), kk > 0);
                    mma_commit(&sm.bar_x);
                    if (wait_phase(sm, &sm.bar_x, x_par, 16u) && n + 2 < nchunks) {
                        // the stage is free again: refill it with chunk n+2
                        issue_stage_loads(sm.in[st], &sm.bar_tma[st], mq, mk, mv, mg, h, t0 + 2 * C,
                                          gmode);
                        sm.tma_issued[st] += 1;
                    }
                }
            }
            __syncwarp();
            named_sync(BAR_XG, 64);
            tc_fence_after();
            scale_state(sm, tb + lane_off, st);
        } else {
            // ---- a4: Akk (strict, beta rows) and Aqk (inclusive) from the Gram (warps 8, 9) ----
            if (issuer) {
                wait_phase(sm, &sm.bar_gops[st], gops_par[st], 64u);
                wait_phase(sm, &sm.bar_gram[st], gram_par[st], 2u);
            }
            named_sync(BAR_E1, 64);
            tc_fence_after();
            float d0[16], d1[16];
            tmem_ld16x2(tb + lane_off + TM_G + 32 * st, tb + lane_off + TM_G + 32 * st + 16, d0, d1);
            tc_fence_before();
            const int r = lane;
            if (cw == 0) {
                // Akk^T[m][r] = beta_r Gram[r][m] for m < r (row m of Akk^T is contiguous)
                const float br = betaN[r];
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    sm.akkT[m][r] = m < r ? br * (m < 16 ? d0[m] : d1[m - 16]) : 0.f;
                __syncwarp();
                // T = (I + Akk)^{-1} by 16 x 16 blocks.  The diagonal blocks
                // T11 = (I + A11)^{-1} (lanes 0-15) and T22 = (I + A22)^{-1} (lanes 16-31)
                // by forward substitution, one column per lane; then
                // T21 = -T22 (A21 T11), each lane 8 rows of one column.
                const int hb = lane >> 4, jj = lane & 15, b0 = 16 * hb;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = i == jj ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 15; ++m) {
                    const float xm = x[m];
                    const float4 *row = reinterpret_cast<const float4 *>(&sm.akkT[b0 + m][b0]);
#pragma unroll
                    for (int q4 = (m + 1) >> 2; q4 < 4; ++q4) {
                        const float4 a4 = row[q4];
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q4 + e > m) x[4 * q4 + e] -= av[e] * xm;
                    }
                }
                // T11 by rows (tsc[0][k][j] = T11[k][j]), T22 by columns (tsc[1][j][i] = T22[i][j])
                if (hb == 0) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) sm.tsc[0][k][jj] = x[k];
                } else {
#pragma unroll
                    for (int i4 = 0; i4 < 4; ++i4)
                        *reinterpret_cast<float4 *>(&sm.tsc[1][jj][4 * i4]) =
                            make_float4(x[4 * i4], x[4 * i4 + 1], x[4 * i4 + 2], x[4 * i4 + 3]);
                }
                __syncwarp();
                // M = A21 T11, rows 8 hb .. 8 hb + 7 of column jj (A21[i][k] = akkT[k][16 + i])
                float mm[8];
#pragma unroll
                for (int r8 = 0; r8 < 8; ++r8) mm[r8] = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float t = sm.tsc[0][k][jj];
                    const float4 a0 = *reinterpret_cast<const float4 *>(&sm.akkT[k][16 + 8 * hb]);
                    const float4 a1 = *reinterpret_cast<const float4 *>(&sm.akkT[k][20 + 8 * hb]);
                    mm[0] += a0.x * t; mm[1] += a0.y * t; mm[2] += a0.z * t; mm[3] += a0.w * t;
                    mm[4] += a1.x * t; mm[5] += a1.y * t; mm[6] += a1.z * t; mm[7] += a1.w * t;
                }
#pragma unroll
                for (int r8 = 0; r8 < 8; ++r8) sm.tsc[2][8 * hb + r8][jj] = mm[r8];
                __syncwarp();
                // T21 = -T22 M, the same rows and column
                float t21[8];
#pragma unroll
                for (int r8 = 0; r8 < 8; ++r8) t21[r8] = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float mk = sm.tsc[2][k][jj];
                    const float4 c0 = *reinterpret_cast<const float4 *>(&sm.tsc[1][k][8 * hb]);
                    const float4 c1 = *reinterpret_cast<const float4 *>(&sm.tsc[1][k][8 * hb + 4]);
                    t21[0] -= c0.x * mk; t21[1] -= c0.y * mk; t21[2] -= c0.z * mk; t21[3] -= c0.w * mk;
                    t21[4] -= c1.x * mk; t21[5] -= c1.y * mk; t21[6] -= c1.z * mk; t21[7] -= c1.w * mk;
                }
                // T diag(beta) as a tf32 operand (row i, column c): the diagonal block of
                // this half, then 8 rows of T21.  The block T12 = 0 is written once at the start.
                const float bd = betaN[b0 + jj], bl = betaN[jj];
#pragma unroll
                for (int i = 0; i < 16; ++i) st_op(sm.tmat[st], b0 + i, b0 + jj, x[i] * bd);
#pragma unroll
                for (int r8 = 0; r8 < 8; ++r8) st_op(sm.tmat[st], 16 + 8 * hb + r8, jj, t21[r8] * bl);
                fence_proxy_async_smem();
            } else {
                float av[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) av[i] = i <= r ? (i < 16 ? d0[i] : d1[i - 16]) : 0.f;
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4)
                    st_op4(sm.kbaq[st], 128 + r, i4, av[4 * i4], av[4 * i4 + 1], av[4 * i4 + 2], av[4 * i4 + 3]);
                fence_proxy_async_smem();
            }
        }
        bxf_par[st] ^= 1u;
        gops_par[st] ^= 1u;
        gram_par[st] ^= 1u;
        x_par ^= 1u;
        if (named_sync_or(BAR_CHAIN, kChain, aborted(sm))) break;

        // ---- a4 (state side): U'^T = V^T (T diag(beta))^T into TMEM U[st], then
        // U^T = U'^T - (gamma K S)^T (T diag(beta))^T accumulated onto it (same
        // accumulator and issuing thread, so the second group follows the first) ----
        if (issuer) {
            tc_fence_after();
            const uint64_t dT = sdesc_sw128(smem_u32(sm.tmat[st]));
            const uint32_t tbv = st ? TM_BV1 : TM_BV;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + tu, tb + tbv + kk * 8, dT + (uint64_t)((kk * 32) >> 4),
                            idesc_tf32(128, 32), kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + tu, tb + TM_X + 32 + kk * 8, dT + (uint64_t)((kk * 32) >> 4),
                            idesc_tf32_negb(128, 32), 1u);
            mma_commit(&sm.bar_u);
        }
        __syncwarp();
        // S^T <- S^T Diag(e^{Gamma_last}) on lanes 0-63, overlapping the U MMAs
        // (the readout MMA that read S is complete: warps 10, 11 awaited it)
        if (cw < 2) {
            tc_fence_after();
            scale_state(sm, tb + lane_off, st);
        }
        if (issuer) wait_phase(sm, &sm.bar_u, u_par, 16u);
        u_par ^= 1u;
        named_sync(BAR_CHAIN, kChain);

        // ---- a5/a6: [S^T | O^T] += U^T [Kbar^T ; Aqk]^T, one N = 160 MMA group ----
        if (issuer) {
            tc_fence_after();
            const uint64_t dK = sdesc_sw128(smem_u32(sm.kbaq[st]));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + TM_S, tb + tu + kk * 8, dK + (uint64_t)((kk * 32) >> 4),
                            idesc_tf32(128, 160), 1u);
            mma_commit(&sm.bar_s);
            mma_commit(&sm.bar_akempty[st]);
            wait_phase(sm, &sm.bar_s, s_par, 16u);
        }
        // the output staging buffer of this parity was last stored for chunk n-2
        if (ostorer) bulk_wait_group_read<1>();
        __syncwarp();
        s_par ^= 1u;
        named_sync(BAR_CHAIN, kChain);
        tc_fence_after();

        // ---- a7: output rows (read from TMEM by every thread before the next
        // chunk's readout MMA overwrites them) ----
        float o0[16], o1[16];
        tmem_ld16x2(tb + lane_off + TM_X, tb + lane_off + TM_X + 16, o0, o1);
        tc_fence_before();
        if (L == C) {
            // a full chunk: rows into the staging tile, one TMA store
            unsigned char *stg = sm.ostage[st];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                st_stage<OUT_T>(stg, r, j, o0[r]);
                st_stage<OUT_T>(stg, 16 + r, j, o1[r]);
            }
            fence_proxy_async_smem();
        }
        named_sync(BAR_CHAIN, kChain);
        if (L == C) {
            if (ostorer) {
                tma_store_3d(mo, sm.ostage[st], 0, (int)t0, (int)(sizeof(OUT_T) * D / 128) * h);
                bulk_commit_group();
            }
        } else {
            // the last chunk of a sequence: the rows past its end belong to the next one
            OUT_T *dst = out + (t0 * H + h) * (int64_t)D + j;
            const int64_t row = (int64_t)H * D;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < L) kda::st_elem(dst + r * row, o0[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (16 + r < L) kda::st_elem(dst + (16 + r) * row, o1[r]);
        }

        // ---- state checkpoint after every ckpt_every chunks that end inside the
        // sequence: S (after this chunk's carry) from TMEM, thread j writes column j ----
        if (ckpt && (n + 1) % ckpt_every == 0 && L == C) {
            const int64_t ck = ck_row0 + (n + 1) / ckpt_every - 1;
            if (ck < ckpt_cap) {
                float *dstS = ckpt + (ck * H + h) * (int64_t)D * D + j;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float sv[16];
                    tmem_ld16(tb + lane_off + TM_S + c0, sv);
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) dstS[(int64_t)(c0 + i) * D] = sv[i];
                }
                tc_fence_before();
            }
        }
    }
    if (ostorer) bulk_wait_group_all();   // every output store has been performed
    if (issuer || xissuer) {   // every MMA issued here has completed
        uint64_t *fin = &sm.bar_fin[issuer ? 1 : 2];
        mma_commit(fin);
        mbar_wait_bounded(fin, 0, kPollLimit);
    }
}

// init_state and final_state may be the same array (each CTA reads its slice
// before it writes it), so neither is declared __restrict__.
template <typename OUT_T, bool GATED, bool SDECAY>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g,
                      const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ beta,
                      const float *init_state, const int32_t *__restrict__ cu,
                      OUT_T *__restrict__ out, float *final_state, int H,
                      int64_t total, int64_t seq_len, float *__restrict__ ckpt,
                      int64_t ckpt_every, int64_t ckpt_cap, const float *__restrict__ a_log,
                      const float *__restrict__ g_head) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // Round up to 1024 bytes by pointer arithmetic on the shared array itself
    // (an integer round trip would lose the shared address space and turn
    // every access through `sm` into a generic one).
    TcSmem &sm = *reinterpret_cast<TcSmem *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));

    const int t = threadIdx.x, warp = t >> 5;
    const int h = blockIdx.x % H;
    const int n = kda::longest_first(cu, (int)(gridDim.x / H), total, seq_len, blockIdx.x / H,
                                     &sm.seq_of_slot);
    int64_t a, b;
    kda::seq_bounds(cu, n, total, seq_len, a, b);
    const int nchunks = (int)((b - a + C - 1) / C);

    if (t == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.bar_tma[s], 1);
            mbar_init(&sm.bar_akempty[s], 1);
            mbar_init(&sm.bar_gops[s], 1);
            mbar_init(&sm.bar_gram[s], 1);
            mbar_init(&sm.bar_bxfull[s], 1);
            mbar_init(&sm.bar_fin[s], 1);
        }
        mbar_init(&sm.bar_fin[2], 1);
        mbar_init(&sm.bar_x, 1);
        mbar_init(&sm.bar_u, 1);
        mbar_init(&sm.bar_s, 1);
        fence_mbar_init();
        sm.abort = 0;
        sm.tma_issued[0] = sm.tma_issued[1] = 0;
        sm.tma_awaited[0] = sm.tma_awaited[1] = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_o);
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
    const bool chain = t >= kPrep;

    // initial state into TMEM: chain thread j holds column j of S (row j of S^T)
    if (chain) {
        const int j = t - kPrep;
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = init_state ? init_state[state_off + (int64_t)(c0 + i) * D + j] : 0.f;
            tmem_st16(tb + lane_off + TM_S + c0, v);
        }
        tmem_wait_st();
        // the block T12 of T diag(beta) (rows 0-15, columns 16-31) is zero for every chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = j + 128 * q;
            st_op(sm.tmat[e >> 8], (e >> 4) & 15, 16 + (e & 15), 0.f);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (!chain)
        prep_loop<GATED, SDECAY>(sm, &tm_q, &tm_k, &tm_v, &tm_g, beta, g_head, H, h, a, b, nchunks,
                                 tb, GATED ? __expf(a_log[h]) : 0.f);
    else
        chain_loop<OUT_T>(sm, &tm_q, &tm_k, &tm_v, &tm_g, &tm_o, out, H, h, a, b, nchunks, tb,
                          ckpt, ckpt_every, ckpt_cap,
                          ckpt ? kda::ckpt_first_row(cu, n, total, seq_len, ckpt_every * C) : 0,
                          GATED ? kDecayLogits : SDECAY ? kDecayScalar : kDecayTile);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t == 0)   // after a stop, wait for stage loads still in flight
        for (int s = 0; s < 2; ++s)
            if (sm.tma_issued[s] > sm.tma_awaited[s])
                mbar_wait_bounded(&sm.bar_tma[s], (sm.tma_issued[s] - 1) & 1u, kPollLimit);
    if (!aborted(sm) && final_state && chain) {
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

template <typename OUT_T>
cudaError_t launch(const kda::Problem &P, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *init_state, const int32_t *cu,
                   void *out, float *final_state, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mg, mo;
    if (!kda_make_tile_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !(P.a_log          ? kda_make_tile_map(&mg, P.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H)
          : P.scalar_decay ? kda_make_tile_map(&mg, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H)   // unused
                           : kda_make_tile_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.T, P.H)) ||
        !(sizeof(OUT_T) == 2 ? kda_make_tile_map(&mo, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H)
                             : kda_make_tile_map(&mo, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.T, P.H)))
        return cudaErrorInvalidValue;
    auto kern = P.a_log          ? kda_prefill_tc_kernel<OUT_T, true, false>
                : P.scalar_decay ? kda_prefill_tc_kernel<OUT_T, false, true>
                                 : kda_prefill_tc_kernel<OUT_T, false, false>;
    const size_t smem = sizeof(TcSmem) + 1024;
    static_assert(sizeof(TcSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((int64_t)P.N * P.H);
    kern<<<blocks, kThreads, smem, stream>>>(mq, mk, mv, mg, mo, beta, init_state, cu,
                                             (OUT_T *)out, final_state, P.H, (int64_t)P.T,
                                             P.seq_len, P.ckpt, P.ckpt ? P.ckpt_interval / C : 1,
                                             P.ckpt_capacity, P.a_log, P.g_head);
    return cudaGetLastError();
}

}  // namespace

bool kda_prefill_tc_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const void *out) {
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    return P.dk == 128 && P.dv == 128 && P.in_dtype == KDA_DTYPE_BF16 && P.T > 0 &&
           P.T <= 0x7fffffff - C && al16(q) && al16(k) && al16(v) && (P.scalar_decay || al16(g)) && al16(out) &&
           kda_tma_available();
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

// Diagnostic of the bounded-wait path: one warp waits on an mbarrier that
// nothing arrives on; the wait gives up after `polls` polls (a few
// milliseconds) and records the status word exactly as the prefill kernel
// does when one of its waits gives up.  Nothing traps or hangs.
__global__ void kda_selftest_timeout_kernel(uint32_t polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (!sm100::mbar_wait_bounded(&bar, 0, polls) && threadIdx.x == 0)
        atomicOr(&g_kda_device_status, 0x100u);
}

cudaError_t kda_launch_selftest_timeout(cudaStream_t stream) {
    kda_selftest_timeout_kernel<<<1, 32, 0, stream>>>(1u << 16);
    return cudaGetLastError();
}

// Read and clear this kernel's status word (ORed into *status).
cudaError_t kda_tc_read_status(unsigned *status) {
    unsigned st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&st, g_kda_device_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_kda_device_status, &zero, sizeof(unsigned));
    *status |= st;
    return e;
}
