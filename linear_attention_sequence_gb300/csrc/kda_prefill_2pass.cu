// kda_prefill_2pass.cu -- chunked KDA prefill in two passes (sm_103a, tcgen05).
//
// The chunk form ("Inside Kimi K3", section "Sequence mixing": the tokens of a
// chunk in parallel, inclusive diagonal, the state carried between chunks;
// "Hybrid Attention", section "But isn't a recurrent update sequential?": a
// triangular solve resolves the dependencies inside a chunk), with Gamma the
// running sum of g inside a chunk of C = 32 tokens and gamma = e^Gamma:
//
//   T   = (I + Akk)^{-1},   Tb = T diag(beta)
//   U   = Tb (V - (gamma K) S0)
//   O   = (gamma Q) S0 + Aqk U
//   S_C = Diag(gamma_last) S0 + Kbar^T U,   Kbar_r = e^{Gamma_last - Gamma_r} k_r
//
// Pass 1 (kda_intra_kernel, one CTA per SM): everything that needs neither the
// state nor V -- the Gram matrices, the triangular solve -- for every chunk of
// every (sequence, head) at once, two chunks per unit of eight warps.  Per chunk
// it leaves 8 KB in a scratch array: Aqk (masked, inclusive diagonal) and Tb,
// each a K-major SW128 tf32 block of 32 rows, ready to be copied into shared
// memory as MMA operands.
//
// Pass 2 (kda_chain2_kernel, one CTA per (sequence, head) at a time): the state
// recurrence.  The CTA loads the chunk's q, k, v and g by TMA, forms its own
// decay prefix and decay-weighted operands, keeps S^T in tensor memory and runs
// three MMA groups a chunk:
//
//   X group  [X_Q | Y] = S^T [gamma Q ; -gamma K]^T  onto [0 | V^T]   (N = 64, K = 128)
//   U group  U^T = Y Tb^T                                              (N = 32, K = 32)
//   carry    [S'^T | O^T] = [S^T Diag(gamma_last) | X_Q] + U^T [Kbar^T ; Aqk]^T
//                                                                      (N = 160, K = 32)
//
// The state decay S^T Diag(gamma_last) is made element-wise into a second
// state buffer while the X and U groups run, so it is off the chain.
//
// Decay factoring in pass 1: products e^{Gamma_r - Gamma_i} (i <= r) are split
// around Gamma_15; with g >= g_min = -5, |Gamma_r - Gamma_15| <= 80 inside a
// 32-token chunk ("Understanding Kimi K3's Attention", log-decay bound), so both
// factors stay in the fp32/tf32 normal range.  Pass 2 needs only e^{Gamma_r}
// and e^{Gamma_last - Gamma_r}, both in (0, 1].
//
// Precision: every product is tcgen05.mma kind::tf32 with fp32 accumulation.

#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"
#include "kda_chunk_ops.cuh"

__device__ unsigned int g_kda_2pass_status;   // nonzero after a bounded wait gave up

namespace {

using namespace sm100;
using namespace kda_chunk;

constexpr int C = 32;
constexpr int D = 128;
constexpr int kThreads = 512;
constexpr uint32_t kPollLimit = 1u << 23;   // mbarrier polls (about half a second)

// Pass-1 output per chunk: Aqk rows then Tb rows, 32 x 128 B each.
constexpr uint32_t kSlot = 8192, OFF_AQK = 0, OFF_TB = 4096;

constexpr int kDecayTile = 0, kDecayLogits = 1, kDecayScalar = 2;

struct Params {
    const __nv_bfloat16 *q, *k, *v;
    const float *g;              // per-channel log-decay (fp32 tile mode)
    const __nv_bfloat16 *z;      // decay logits (gate prologue)
    const float *a_log;
    const float *g_head;         // one log-decay per (token, head) (nullptr: none)
    const float *beta;           // beta, or its logits with the gate prologue
    const float *init;
    const int32_t *cu;
    void *out;
    float *fin;
    float *ckpt;
    int64_t ckpt_every, ckpt_cap;   // chunks between checkpoints; rows allocated
    const __nv_bfloat16 *ogate;
    const float *onorm_w;
    float oeps;
    int N, H;
    int64_t total, seq_len;
    int NC, KMAX;                // pass-2 CTAs; most (sequence, head) pairs of one CTA
    unsigned char *slots;        // [chunks x H][kSlot], chunk-major
    int32_t *chunk_off;          // [N + 1]: first chunk of each sequence (input order)
    int32_t *order;              // [N]: sequences, longest first
    uint32_t *first_step;        // [NC][KMAX + 1]: first step of each pair of a CTA, then the total
};

__device__ __forceinline__ uint32_t off_bf16(int r, int c) {   // TMA tile (SW128), bf16
    return (uint32_t)((c >> 6) * 4096 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ float lds_bf16(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

// ---------------------------------------------------------------------------
// Set-up (one block): chunk offsets of the sequences, their longest-first
// order, and the steps of each pass-2 CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) twopass_setup_kernel(const int32_t *cu, int N, int H,
                                                             int64_t total, int64_t seq_len,
                                                             int NC, int KMAX, int32_t *chunk_off,
                                                             int32_t *order, uint32_t *first_step) {
    __shared__ int32_t part[1024];
    const int t = threadIdx.x, nt = blockDim.x;
    const int per = (N + nt - 1) / nt;
    const int lo = t * per, hi = lo + per < N ? lo + per : N;
    int32_t acc = 0;
    for (int n = lo; n < hi; ++n) {
        int64_t a, b;
        kda::seq_bounds(cu, n, total, seq_len, a, b);
        acc += (int32_t)((b - a + C - 1) / C);
    }
    part[t] = acc;
    __syncthreads();
    if (t == 0) {
        int32_t run = 0;
        for (int i = 0; i < nt; ++i) {
            const int32_t x = part[i];
            part[i] = run;
            run += x;
        }
        chunk_off[N] = run;
    }
    __syncthreads();
    acc = part[t];
    for (int n = lo; n < hi; ++n) {
        chunk_off[n] = acc;
        int64_t a, b;
        kda::seq_bounds(cu, n, total, seq_len, a, b);
        acc += (int32_t)((b - a + C - 1) / C);
    }
    if (cu && N <= nt) {
        if (t < N) {
            int64_t a, b;
            kda::seq_bounds(cu, t, total, seq_len, a, b);
            const int64_t len = b - a;
            int rank = 0;
            for (int m = 0; m < N; ++m) {
                int64_t a2, b2;
                kda::seq_bounds(cu, m, total, seq_len, a2, b2);
                rank += (b2 - a2 > len || (b2 - a2 == len && m < t)) ? 1 : 0;
            }
            order[rank] = t;
        }
    } else {
        for (int i = t; i < N; i += nt) order[i] = i;
    }
    __syncthreads();
    if (t < NC) {
        const int P = N * H;
        uint32_t *fs = first_step + (size_t)t * (KMAX + 1);
        uint32_t s = 0;
        int kp = 0;
        for (int pi = t; pi < P; pi += NC, ++kp) {
            fs[kp] = s;
            int64_t a, b;
            kda::seq_bounds(cu, order[pi / H], total, seq_len, a, b);
            s += (uint32_t)((b - a + C - 1) / C);
        }
        fs[kp] = s;
    }
}

// ---------------------------------------------------------------------------
// Pass 1: T diag(beta) and Aqk of every chunk.
// ---------------------------------------------------------------------------

// A unit: 256 tensor-memory columns (Gram D 64, Gram A 128) and 96 KB of
// shared memory (Gram A staging 64 KB, later the solve's scratch; Gram B 32 KB).
constexpr uint32_t kUnitBytes = 98304;

struct CtlA {
    uint64_t gram[2];
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kSmemA = 2 * kUnitBytes + sizeof(CtlA) + 1024;
static_assert(kSmemA <= 232448, "shared memory budget (pass 1)");

struct Chunk {
    int seq, h, n, L;
    int64_t t0;
};

// Chunk-head i of the slot order: chunk (global chunk index i / H) of head i % H.
__device__ bool decode_chunk(const Params &p, uint32_t i, uint32_t total, Chunk &ck) {
    if (i >= total) return false;
    const int cg = (int)(i / (uint32_t)p.H);
    ck.h = (int)(i % (uint32_t)p.H);
    int lo = 0, hi = p.N - 1;   // the last sequence whose first chunk is <= cg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.chunk_off[mid] <= cg) lo = mid;
        else hi = mid - 1;
    }
    ck.seq = lo;
    ck.n = cg - p.chunk_off[lo];
    int64_t a, b;
    kda::seq_bounds(p.cu, lo, p.total, p.seq_len, a, b);
    ck.t0 = a + (int64_t)ck.n * C;
    const int64_t rem = b - ck.t0;
    ck.L = (int)(rem < C ? rem : C);
    return true;
}

__device__ __noinline__ bool wait_a(CtlA &ctl, uint64_t *bar, uint32_t par) {
    if (mbar_wait_bounded(bar, par, kPollLimit)) return true;
    *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
    atomicOr(&g_kda_2pass_status, 0x200u);
    return false;
}

template <int GMODE>
__global__ void __launch_bounds__(kThreads, 1) kda_intra_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    CtlA &ctl = *reinterpret_cast<CtlA *>(base + 2 * kUnitBytes);
    const int t = threadIdx.x, u = t >> 8, T = t & 255, hx = T >> 7, c = T & 127;
    const int wu = T >> 5, lane = t & 31;
    if (t == 0) {
        mbar_init(&ctl.gram[0], 1);
        mbar_init(&ctl.gram[1], 1);
        fence_mbar_init();
        ctl.abort = 0;
    }
    if ((t >> 5) == 0) {
        tmem_alloc(&ctl.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * (wu & 3)) << 16;
    const uint32_t GD = tb + 256u * (uint32_t)u, GA = GD + 64;
    unsigned char *stg = base + u * kUnitBytes;   // Gram A staging, then the solve's scratch
    unsigned char *gB = stg + 65536;              // Gram B: 4 K-blocks x 64 rows
    const uint32_t bar_id = 1 + u;
    const uint32_t total = (uint32_t)p.chunk_off[p.N] * (uint32_t)p.H;
    const int64_t rs = (int64_t)p.H * D;   // token stride of [T, H, D] tensors
    uint32_t gpar = 0;
    bool ok = true;

    for (uint32_t pr = 2u * blockIdx.x + (uint32_t)u;; pr += 2u * gridDim.x) {
        const uint32_t i0 = 2u * pr;
        // uniform over the unit; also orders the last pair's reads of the
        // staging buffer before this pair overwrites it
        if (named_sync_or(bar_id, 256, !ok || i0 >= total || *(volatile int *)&ctl.abort != 0)) break;
        Chunk ck;
        const bool valid = decode_chunk(p, i0 + (uint32_t)hx, total, ck);
        const int L = valid ? ck.L : 0;

        // ---- phase 1 (thread = channel c of chunk hx): decay prefix, Gram operands ----
        const int64_t e0 = valid ? (ck.t0 * p.H + ck.h) * (int64_t)D + c : 0;
        const int64_t b0i = valid ? ck.t0 * p.H + ck.h : 0;
        float gsc = 0.f;
        if (GMODE == kDecayLogits && valid) gsc = __expf(p.a_log[ck.h]);
        float gam[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float gr = 0.f;
            if (r < L) {
                if (GMODE == kDecayTile) gr = __ldg(p.g + e0 + r * rs);
                else if (GMODE == kDecayLogits) gr = __bfloat162float(__ldg(p.z + e0 + r * rs));
                else gr = p.g_head ? __ldg(p.g_head + b0i + r * p.H) : 0.f;
            }
            gam[r] = gr;
        }
        {
            float run = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                run += (GMODE == kDecayLogits && r < L) ? kda::gate_g(gam[r], gsc) : gam[r];
                gam[r] = run;
            }
        }
        const float g15 = gam[15];
        {
            uint32_t swz[8];
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) swz[k8] = (uint32_t)(((((c & 31) >> 2) ^ k8) << 4) + ((c & 3) << 2));
            unsigned char *stK = stg + (c >> 5) * 16384 + (hx ? 64 : 0) * 128;   // k~ rows of this chunk
            unsigned char *stQ = stK + 32 * 128;                                  // q~ rows
            unsigned char *gBr = gB + (c >> 5) * 8192 + (hx ? 32 : 0) * 128;     // k^ rows
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
                __nv_bfloat16 qr[16], kr[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * h16 + i;
                    const __nv_bfloat16 zero = __float2bfloat16(0.f);
                    qr[i] = r < L ? __ldg(p.q + e0 + r * rs) : zero;
                    kr[i] = r < L ? __ldg(p.k + e0 + r * rs) : zero;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * h16 + i;
                    const uint32_t so = (uint32_t)r * 128 + swz[r & 7];
                    const float qv = __bfloat162float(qr[i]), kv = __bfloat162float(kr[i]);
                    const float x = gam[r] - g15;
                    const float e1 = __expf(x);    // e^{Gamma_r - Gamma_15} in [e^-80, e^75]
                    const float inv = __expf(-x);  // its inverse
                    *reinterpret_cast<float *>(stK + so) = to_tf32(kv * e1);
                    *reinterpret_cast<float *>(stQ + so) = to_tf32(qv * e1);
                    *reinterpret_cast<float *>(gBr + so) = to_tf32(kv * inv);
                }
            }
        }
        fence_proxy_async_smem();   // the Gram B operand is read by the tensor cores
        named_sync(bar_id, 256);

        // ---- phase 2: the Gram A rows into tensor memory (lane = row; warps 0-3
        // channels 0-63, warps 4-7 channels 64-127) ----
        tc_fence_after();
        {
            const int R = 32 * (wu & 3) + lane;
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int kb = 2 * (wu >> 2) + k2;
                const unsigned char *src = stg + kb * 16384 + R * 128;
                float x[32];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(src + ((ch ^ (R & 7)) << 4));
                    x[4 * ch] = v4.x;
                    x[4 * ch + 1] = v4.y;
                    x[4 * ch + 2] = v4.z;
                    x[4 * ch + 3] = v4.w;
                }
                tmem_st32(GA + lane_off + 32 * kb, x);
            }
        }
        tmem_wait_st();
        tc_fence_before();
        named_sync(bar_id, 256);

        // ---- phase 3: Gram = [k~_a ; q~_a ; k~_b ; q~_b] [k^_a ; k^_b]^T (N = 64) ----
        if (T == 0) {
            tc_fence_after();
            const uint64_t dB = sdesc_sw128(smem_u32(gB));
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32_ts(GD, GA + 8 * kk, dB + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                            idesc_tf32(128, 64), kk > 0);
            mma_commit(&ctl.gram[u]);
            ok = wait_a(ctl, &ctl.gram[u], gpar);
        }
        gpar ^= 1u;
        if (named_sync_or(bar_id, 256, !ok || *(volatile int *)&ctl.abort != 0)) break;
        tc_fence_after();

        // ---- phase 4: Tb of each chunk (warps 0 and 6, lane = row), the masked Aqk
        // rows (warps 1 and 7), both into the chunk's slot; the next pair's inputs
        // are prefetched into L2 ----
        {
            Chunk nx;
            const uint32_t inext = 2u * (pr + 2u * gridDim.x) + (uint32_t)hx;
            const int r = c & 31, ln = c >> 5;
            if (decode_chunk(p, inext, total, nx) && r < nx.L) {
                const int64_t row = (nx.t0 + r) * p.H + nx.h;   // (token, head) row
                if (ln < 2) {
                    prefetch_l2(p.q + row * D + 64 * ln);
                    prefetch_l2(p.k + row * D + 64 * ln);
                    if (GMODE == kDecayLogits) prefetch_l2(p.z + row * D + 64 * ln);
                }
                if (GMODE == kDecayTile) prefetch_l2(p.g + row * D + 32 * ln);
            }
        }
        if (wu == 0 || wu == 6) {
            const int xb = wu == 6;   // = hx
            float d[32];
            tmem_ld32(GD + lane_off + 32 * xb, d);
            float br = 0.f;
            if (lane < L) {
                br = __ldg(p.beta + b0i + lane * p.H);
                if (GMODE == kDecayLogits) br = kda::sigmoid_f(br);
            }
            unsigned char *tm = stg + 4096 * xb;
            float(*akkT)[32] = reinterpret_cast<float(*)[32]>(stg + 8192 + 4096 * xb);
            float(*tsc)[16][20] = reinterpret_cast<float(*)[16][20]>(stg + 16384 + 4096 * xb);
            solve_tbeta(d, br, lane, tm, akkT, tsc);
            __syncwarp();
            if (valid) {
                unsigned char *dst = p.slots + (size_t)(i0 + (uint32_t)xb) * kSlot + OFF_TB + lane * 128;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    reinterpret_cast<float4 *>(dst)[e] = reinterpret_cast<const float4 *>(tm + lane * 128)[e];
            }
        } else if (wu == 1 || wu == 7) {
            const int xb = wu == 7;   // = hx
            float d[32];
            tmem_ld32(GD + lane_off + 32 * xb, d);
            if (valid) {
                unsigned char *dst = p.slots + (size_t)(i0 + (uint32_t)xb) * kSlot + OFF_AQK + lane * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float a4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) a4[e] = 4 * ch + e <= lane ? to_tf32(d[4 * ch + e]) : 0.f;
                    *reinterpret_cast<float4 *>(dst + ((ch ^ (lane & 7)) << 4)) =
                        make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            }
        }
        tc_fence_before();
    }
    if ((t & 255) == 0) {   // every MMA issued by this unit has completed (after a stop too)
        tc_fence_after();
        mma_commit(&ctl.gram[u]);
        mbar_wait_bounded(&ctl.gram[u], gpar, kPollLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((t >> 5) == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------------------
// Pass 2: the state recurrence, one (sequence, head) after another.
// ---------------------------------------------------------------------------

// Shared memory (offsets from a 1024-byte aligned base).  Two input stages
// (q, k, v bf16 tiles and the g tile, by TMA) and, per step parity, the X
// group's B operand [gamma Q ; -gamma K] (even) or [-gamma K ; gamma Q] (odd),
// the carry's B operand [Kbar^T ; Aqk] (even) or [Aqk ; Kbar^T] (odd), Tb, and
// e^{Gamma_last}.
constexpr uint32_t IN_Q = 0, IN_K = 8192, IN_V = 16384, IN_G = 24576, kInBytes = 40960;
constexpr uint32_t SB_BX = 2 * kInBytes;          // 2 x 32 KB: 4 K-blocks of 64 rows
constexpr uint32_t SB_BC = SB_BX + 2 * 32768;     // 2 x 20 KB: 160 rows
constexpr uint32_t SB_TB = SB_BC + 2 * 20480;     // 2 x 4 KB: 32 rows
constexpr uint32_t SB_GC = SB_TB + 2 * 4096;      // 2 x 128 floats
constexpr uint32_t SB_CTL = SB_GC + 2 * 512;

// Tensor-memory columns (lane = value index j).  S^T is double-buffered: a step
// of parity p reads S_r(p) and its carry accumulates into S_w(p), which the
// decay pass has filled with S_r Diag(gamma_last).  Each D range below is
// contiguous: X group [X_Q0 | Y0] and [Y1 | X_Q1], carry [S_B | X_Q0] and
// [X_Q1 | S_A].
constexpr uint32_t TM_Y1 = 0, TM_XQ1 = 32, TM_SA = 64, TM_SB = 192, TM_XQ0 = 320, TM_Y0 = 352,
                   TM_U0 = 384, TM_U1 = 416;
__device__ __forceinline__ uint32_t tm_sr(uint32_t p) { return p ? TM_SB : TM_SA; }
__device__ __forceinline__ uint32_t tm_sw(uint32_t p) { return p ? TM_SA : TM_SB; }
__device__ __forceinline__ uint32_t tm_xd(uint32_t p) { return p ? TM_Y1 : TM_XQ0; }
__device__ __forceinline__ uint32_t tm_xq(uint32_t p) { return p ? TM_XQ1 : TM_XQ0; }
__device__ __forceinline__ uint32_t tm_y(uint32_t p) { return p ? TM_Y1 : TM_Y0; }
__device__ __forceinline__ uint32_t tm_u(uint32_t p) { return p ? TM_U1 : TM_U0; }
__device__ __forceinline__ uint32_t tm_cd(uint32_t p) { return p ? TM_XQ1 : TM_SB; }

constexpr uint32_t BAR_ST = 1, BAR_OG = 2;   // named barriers of the state warps (4-7)

struct CtlB {
    uint64_t infull[2], inempty[2], slotfull[2], prepped[2], pre[2];
    uint64_t barx[2], baru[2], barc[2], scaled[2], sready, fin;
    uint32_t tmem_base;
    int abort;
    float ored[4][32];
};
constexpr size_t kSmemB = SB_CTL + sizeof(CtlB) + 1024;
static_assert(kSmemB <= 232448, "shared memory budget (pass 2)");

__device__ __forceinline__ bool aborted(CtlB &ctl) {
    return *reinterpret_cast<volatile int *>(&ctl.abort) != 0;
}
// Bounded wait for an mbarrier phase; gives up early once the CTA has stopped.
// After a few quick polls the thread backs off with a short sleep between polls,
// so a waiting warp takes few issue slots from the working ones.
__device__ __noinline__ bool wait_slow(CtlB &ctl, uint64_t *bar, uint32_t par, unsigned code) {
    for (uint32_t i = 0; i < kPollLimit; ++i) {
        if (mbar_try_wait(bar, par)) return true;
        if (i >= 8) __nanosleep(32);
        if ((i & 255) == 255 && aborted(ctl)) return false;
    }
    *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
    atomicOr(&g_kda_2pass_status, code);
    return false;
}
__device__ __forceinline__ bool wait_bar(CtlB &ctl, uint64_t *bar, uint32_t par, unsigned code) {
    return mbar_try_wait(bar, par) || wait_slow(ctl, bar, par, code);
}
// Lane 0 waits for a phase; the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(CtlB &ctl, uint64_t *bar, uint32_t par, unsigned code) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(ctl, bar, par, code);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ int chain_pairs(const Params &p, int c) {
    const int P = p.N * p.H;
    return (P - c + p.NC - 1) / p.NC;
}


// Step s of a pass-2 CTA: pair kp covers steps [fs[kp], fs[kp + 1]).  Steps
// are visited in increasing order; pairs without chunks are skipped.
struct Walk {
    int kp = -1, seq = 0, h = 0;
    int64_t a = 0, b = 0;
    uint32_t s0 = 0, s1 = 0;
};
__device__ __forceinline__ void walk_to(const Params &p, const uint32_t *fs, int c, uint32_t s,
                                        Walk &w) {
    if (s < w.s1) return;
    do {
        ++w.kp;
        w.s0 = fs[w.kp];
        w.s1 = fs[w.kp + 1];
    } while (s >= w.s1);
    const int pi = c + w.kp * p.NC;
    w.seq = p.order[pi / p.H];
    w.h = pi % p.H;
    kda::seq_bounds(p.cu, w.seq, p.total, p.seq_len, w.a, w.b);
}
__device__ __forceinline__ int chunk_len(const Walk &w, uint32_t s, int64_t &t0) {
    t0 = w.a + (int64_t)(s - w.s0) * C;
    const int64_t rem = w.b - t0;
    return (int)(rem < C ? rem : C);
}

// Warp 0, one thread: the three MMA groups of every step.
__device__ void chain_issuer(const Params &p, unsigned char *base, CtlB &ctl, uint32_t tb, int c,
                             const uint32_t *fs, uint32_t nsteps) {
    Walk w;
    uint32_t npc = 0;
    bool ok = true;
    for (uint32_t s = 0; s < nsteps && ok; ++s) {
        walk_to(p, fs, c, s, w);
        const uint32_t pp = s & 1u, ph = (s >> 1) & 1u;
        if (s == w.s0) {
            if (!(ok = wait_bar(ctl, &ctl.sready, npc & 1u, 0x21u))) break;
            ++npc;
        }
        if (!(ok = wait_bar(ctl, &ctl.prepped[pp], ph, 0x22u))) break;
        if (!(ok = wait_bar(ctl, &ctl.pre[pp], ph, 0x23u))) break;
        tc_fence_after();
        const uint64_t dX = sdesc_sw128(smem_u32(base + SB_BX + pp * 32768));
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_tf32_ts(tb + tm_xd(pp), tb + tm_sr(pp) + 8 * kk,
                        dX + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_tf32(128, 64), 1u);
        mma_commit(&ctl.barx[pp]);
        if (!(ok = wait_bar(ctl, &ctl.slotfull[pp], ph, 0x24u))) break;
        if (!(ok = wait_bar(ctl, &ctl.barx[pp], ph, 0x25u))) break;
        tc_fence_after();
        const uint64_t dT = sdesc_sw128(smem_u32(base + SB_TB + pp * 4096));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_tf32_ts(tb + tm_u(pp), tb + tm_y(pp) + 8 * kk, dT + (uint64_t)((kk * 32) >> 4),
                        idesc_tf32(128, 32), kk > 0);
        mma_commit(&ctl.baru[pp]);
        if (!(ok = wait_bar(ctl, &ctl.baru[pp], ph, 0x26u))) break;
        if (!(ok = wait_bar(ctl, &ctl.scaled[pp], ph, 0x27u))) break;
        tc_fence_after();
        const uint64_t dC = sdesc_sw128(smem_u32(base + SB_BC + pp * 20480));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_tf32_ts(tb + tm_cd(pp), tb + tm_u(pp) + 8 * kk, dC + (uint64_t)((kk * 32) >> 4),
                        idesc_tf32(128, 160), 1u);
        mma_commit(&ctl.barc[pp]);
        if (!(ok = wait_bar(ctl, &ctl.barc[pp], ph, 0x28u))) break;
    }
    mma_commit(&ctl.fin);   // every MMA issued here has completed
    mbar_wait_bounded(&ctl.fin, 0, kPollLimit);
}

// Warp 1, one thread: the TMA loads of each step's q, k, v and g (or z) tiles.
template <int GMODE>
__device__ void chain_loader(const Params &p, unsigned char *base, CtlB &ctl, int c,
                             const uint32_t *fs, uint32_t nsteps, const CUtensorMap *mq,
                             const CUtensorMap *mk, const CUtensorMap *mv, const CUtensorMap *mg) {
    constexpr uint32_t bytes = GMODE == kDecayScalar   ? 3 * 8192
                               : GMODE == kDecayLogits ? 4 * 8192
                                                       : 3 * 8192 + 16384;
    Walk w;
    uint32_t issued = 0;
    for (uint32_t s = 0; s < nsteps; ++s) {
        walk_to(p, fs, c, s, w);
        const uint32_t st = s & 1u;
        if (s >= 2 && !wait_bar(ctl, &ctl.inempty[st], ((s >> 1) - 1) & 1u, 0x29u)) break;
        int64_t t0;
        chunk_len(w, s, t0);
        unsigned char *in = base + st * kInBytes;
        mbar_arrive_expect_tx(&ctl.infull[st], bytes);
        tma_load_3d(in + IN_Q, mq, &ctl.infull[st], 0, (int)t0, 2 * w.h);
        tma_load_3d(in + IN_K, mk, &ctl.infull[st], 0, (int)t0, 2 * w.h);
        tma_load_3d(in + IN_V, mv, &ctl.infull[st], 0, (int)t0, 2 * w.h);
        if (GMODE == kDecayTile) tma_load_3d(in + IN_G, mg, &ctl.infull[st], 0, (int)t0, 4 * w.h);
        if (GMODE == kDecayLogits) tma_load_3d(in + IN_G, mg, &ctl.infull[st], 0, (int)t0, 2 * w.h);
        issued = s + 1;
    }
    // every load issued has landed before the CTA can exit
    for (uint32_t s = issued > 2u ? issued - 2u : 0u; s < issued; ++s)
        mbar_wait_bounded(&ctl.infull[s & 1u], (s >> 1) & 1u, kPollLimit);
}

// Warp 2, one thread: each step's Aqk and Tb from the pass-1 scratch.
__device__ void chain_slots(const Params &p, unsigned char *base, CtlB &ctl, int c,
                            const uint32_t *fs, uint32_t nsteps) {
    Walk w;
    uint32_t issued = 0;
    for (uint32_t s = 0; s < nsteps; ++s) {
        walk_to(p, fs, c, s, w);
        const uint32_t pp = s & 1u;
        // the carry of step s - 2 has read this parity's Aqk rows (and its U group Tb)
        if (s >= 2 && !wait_bar(ctl, &ctl.barc[pp], ((s >> 1) - 1) & 1u, 0x2au)) break;
        const size_t idx = ((size_t)p.chunk_off[w.seq] + (s - w.s0)) * (size_t)p.H + (size_t)w.h;
        const unsigned char *src = p.slots + idx * kSlot;
        mbar_arrive_expect_tx(&ctl.slotfull[pp], kSlot);
        bulk_g2s(base + SB_BC + pp * 20480 + (pp ? 0u : 16384u), src + OFF_AQK, 4096, &ctl.slotfull[pp]);
        bulk_g2s(base + SB_TB + pp * 4096, src + OFF_TB, 4096, &ctl.slotfull[pp]);
        issued = s + 1;
    }
    for (uint32_t s = issued > 2u ? issued - 2u : 0u; s < issued; ++s)
        mbar_wait_bounded(&ctl.slotfull[s & 1u], (s >> 1) & 1u, kPollLimit);
}

// Warps 8-11 (steps of even index, PP = 0) and 12-15 (odd, PP = 1): thread =
// key channel c.  The decay factors of the step's chunk as running products of
// alpha = e^g: e^{Gamma_r} = alpha_0 ... alpha_r going forward (the X group's B
// operand [gamma Q ; -gamma K] or [-gamma K ; gamma Q]) and e^{Gamma_last -
// Gamma_r} = alpha_{r+1} ... alpha_31 going backward (the Kbar^T rows of the
// carry's B operand); both in (0, 1].  The loops carry only running products,
// so they need no per-token register arrays and stay short.
template <int GMODE, int PP>
__device__ __forceinline__ float prep_alpha(const Params &p, const unsigned char *in, int r, int L,
                                            uint32_t ob, uint32_t of, int64_t t0, int h,
                                            float gsc) {
    float gr = 0.f;
    if (r < L) {
        if (GMODE == kDecayTile) gr = *reinterpret_cast<const float *>(in + IN_G + r * 128 + of);
        else if (GMODE == kDecayLogits) gr = kda::gate_g(lds_bf16(in + IN_G + r * 128 + ob), gsc);
        else gr = p.g_head ? __ldg(p.g_head + (t0 + r) * p.H + h) : 0.f;
    }
    return __expf(gr);
}

template <int GMODE, int PP>
__device__ void chain_prep(const Params &p, unsigned char *base, CtlB &ctl, int c0,
                           const uint32_t *fs, uint32_t nsteps) {
    const int c = (((threadIdx.x >> 5) - 8) & 3) * 32 + (threadIdx.x & 31);
    const unsigned char *in = base + PP * kInBytes;
    unsigned char *bx = base + SB_BX + PP * 32768;
    unsigned char *bcr = base + SB_BC + PP * 20480 + (PP ? 32 + c : c) * 128;   // this channel's Kbar^T row
    float *gc = reinterpret_cast<float *>(base + SB_GC + PP * 512);
    constexpr int rowq = PP ? 32 : 0, rowk = PP ? 0 : 32;   // rows of gamma Q and -gamma K in BX
    // byte offsets of channel c in a row r of each layout, for the eight values of r % 8
    uint32_t ob[8], of[8], ox[8];
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
        ob[k8] = (uint32_t)((c >> 6) * 4096 + ((((c & 63) >> 3) ^ k8) << 4) + ((c & 7) << 1));   // bf16 tile
        of[k8] = (uint32_t)((c >> 5) * 4096 + ((((c & 31) >> 2) ^ k8) << 4) + ((c & 3) << 2));   // fp32 tile
        ox[k8] = (uint32_t)((c >> 5) * 8192 + ((((c & 31) >> 2) ^ k8) << 4) + ((c & 3) << 2));   // BX
    }
    Walk w;
    int kp_g = -1;
    float gsc = 0.f;
    for (uint32_t s = PP; s < nsteps; s += 2) {
        walk_to(p, fs, c0, s, w);
        if (GMODE == kDecayLogits && w.kp != kp_g) {
            gsc = __expf(p.a_log[w.h]);
            kp_g = w.kp;
        }
        int64_t t0;
        const int L = chunk_len(w, s, t0);
        if (!warp_wait(ctl, &ctl.infull[PP], (s >> 1) & 1u, 0x2bu)) break;
        if (s >= 2 && !warp_wait(ctl, &ctl.barc[PP], ((s >> 1) - 1) & 1u, 0x2cu)) break;
        float e = 1.f;   // e^{Gamma_r}
#pragma unroll 8
        for (int r = 0; r < C; ++r) {
            e *= prep_alpha<GMODE, PP>(p, in, r, L, ob[r & 7], of[r & 7], t0, w.h, gsc);
            float qv = 0.f, kv = 0.f;
            if (r < L) {
                qv = lds_bf16(in + IN_Q + r * 128 + ob[r & 7]);
                kv = lds_bf16(in + IN_K + r * 128 + ob[r & 7]);
            }
            *reinterpret_cast<float *>(bx + (rowq + r) * 128 + ox[r & 7]) = to_tf32(qv * e);
            *reinterpret_cast<float *>(bx + (rowk + r) * 128 + ox[r & 7]) = to_tf32(-kv * e);
        }
        gc[c] = e;   // e^{Gamma_last}
        float f = 1.f;   // e^{Gamma_last - Gamma_r}
#pragma unroll 4
        for (int r4 = C / 4 - 1; r4 >= 0; --r4) {
            float kb[4];
#pragma unroll
            for (int i = 3; i >= 0; --i) {
                const int r = 4 * r4 + i;
                const float kv = r < L ? lds_bf16(in + IN_K + r * 128 + ob[r & 7]) : 0.f;
                kb[i] = to_tf32(kv * f);
                f *= prep_alpha<GMODE, PP>(p, in, r, L, ob[r & 7], of[r & 7], t0, w.h, gsc);
            }
            *reinterpret_cast<float4 *>(bcr + (((r4 ^ (c & 7)) & 7) << 4)) = make_float4(kb[0], kb[1], kb[2], kb[3]);
        }
        fence_proxy_async_smem();   // the operands are read by the tensor cores
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            mbar_arrive(&ctl.prepped[PP]);
            mbar_arrive(&ctl.inempty[PP]);
        }
    }
}

// Warps 4-7: thread j = value index j = tensor-memory lane.  Initial states,
// the state decay, V^T into the X group's accumulator, the output rows and the
// final states and checkpoints.
template <typename OUT_T, bool OGATE>
__device__ void chain_state(const Params &p, unsigned char *base, CtlB &ctl, uint32_t tb, int c,
                            const uint32_t *fs, uint32_t nsteps) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, q4 = warp & 3;
    const int j = 32 * q4 + lane;
    const uint32_t tl = tb + ((uint32_t)(32 * q4) << 16);
    const int64_t hd = (int64_t)p.H * D;
    const int npairs = chain_pairs(p, c);
    bool ok = true;
    Walk wpre;   // the step being preloaded (may run into the next pair)

    auto preload = [&](uint32_t s2) {   // [0 | V^T] (even) or [V^T | 0] (odd) of step s2
        walk_to(p, fs, c, s2, wpre);
        int64_t t2;
        const int L2 = chunk_len(wpre, s2, t2);
        const uint32_t p2 = s2 & 1u;
        ok = ok && warp_wait(ctl, &ctl.infull[p2], (s2 >> 1) & 1u, 0x30u);
        if (!ok) return;
        const unsigned char *vt = base + p2 * kInBytes + IN_V;
        float x[32];
#pragma unroll
        for (int r = 0; r < C; ++r) x[r] = r < L2 ? lds_bf16(vt + off_bf16(r, j)) : 0.f;
        tmem_st32(tl + tm_y(p2), x);
#pragma unroll
        for (int r = 0; r < C; ++r) x[r] = 0.f;
        tmem_st32(tl + tm_xq(p2), x);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&ctl.pre[p2]);
            mbar_arrive(&ctl.inempty[p2]);
        }
    };

    // the output rows (and a checkpoint) of step s1 of the pair in `w`; its carry is complete
    auto epilogue = [&](const Walk &w, uint32_t s1, int64_t ck_row0, float wj) {
        int64_t t0;
        const int L = chunk_len(w, s1, t0);
        const int n = (int)(s1 - w.s0);
        float og[C];
        if (OGATE) {
#pragma unroll
            for (int r = 0; r < C; ++r)
                og[r] = r < L ? __bfloat162float(__ldg(p.ogate + (t0 + r) * hd + (int64_t)w.h * D + j)) : 0.f;
        }
        float o[32];
        tmem_ld32(tl + tm_xq(s1 & 1u), o);
        if (OGATE) {
            // y_r = Sigmoid(gate_r) o_r / sqrt(mean_j o_rj^2 + eps) w_j: the sum of squares
            // of row r is reduce-scattered in each warp (lane L ends with its warp's sum
            // for row L), then the four warps' sums meet in shared memory
            float a2[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) a2[r] = o[r] * o[r];
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
                const bool up = (lane & sh) != 0;
#pragma unroll
                for (int i = 0; i < sh; ++i) {
                    const float send = up ? a2[i] : a2[i + sh];
                    const float keep = up ? a2[i + sh] : a2[i];
                    a2[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
                }
            }
            ctl.ored[q4][lane] = a2[0];
            named_sync(BAR_OG, 128);
            const float ms = (ctl.ored[0][lane] + ctl.ored[1][lane] + ctl.ored[2][lane] +
                              ctl.ored[3][lane]) * (1.f / D);
            const float rinv = rsqrtf(ms + p.oeps);
            named_sync(BAR_OG, 128);   // every row sum is read before the next step's
#pragma unroll
            for (int r = 0; r < 32; ++r)
                o[r] *= __shfl_sync(0xffffffffu, rinv, r) * wj * kda::sigmoid_f(og[r]);
        }
        OUT_T *dst = reinterpret_cast<OUT_T *>(p.out) + (t0 * p.H + w.h) * (int64_t)D + j;
#pragma unroll
        for (int r = 0; r < C; ++r)
            if (r < L) kda::st_elem(dst + r * hd, o[r]);
        if (p.ckpt && (n + 1) % p.ckpt_every == 0 && L == C) {
            const int64_t ck = ck_row0 + (n + 1) / p.ckpt_every - 1;
            if (ck < p.ckpt_cap) {
                float *dS = p.ckpt + (ck * p.H + w.h) * (int64_t)D * D + j;
#pragma unroll 1
                for (int k0 = 0; k0 < D; k0 += 32) {
                    float x[32];
                    tmem_ld32(tl + tm_sw(s1 & 1u) + k0, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dS[(int64_t)(k0 + i) * D] = x[i];
                }
            }
        }
    };

    uint32_t s = 0;
    for (int kp = 0; kp < npairs && ok; ++kp) {
        const int pi = c + kp * p.NC;
        Walk w;
        w.kp = kp;
        w.seq = p.order[pi / p.H];
        w.h = pi % p.H;
        w.s0 = fs[kp];
        w.s1 = fs[kp + 1];
        kda::seq_bounds(p.cu, w.seq, p.total, p.seq_len, w.a, w.b);
        const int64_t soff = ((int64_t)w.seq * p.H + w.h) * D * D;
        if (w.s1 == w.s0) {   // an empty sequence: the final state is the initial one
            if (p.fin)
                for (int k0 = 0; k0 < D; ++k0)
                    p.fin[soff + (int64_t)k0 * D + j] = p.init ? p.init[soff + (int64_t)k0 * D + j] : 0.f;
            continue;
        }
        // the initial state: S^T row j = column j of S
#pragma unroll 1
        for (int k0 = 0; k0 < D; k0 += 32) {
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = p.init ? p.init[soff + (int64_t)(k0 + i) * D + j] : 0.f;
            tmem_st32(tl + tm_sr(w.s0 & 1u) + k0, x);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.sready);
        if (w.s0 == 0) preload(0);
        const int64_t ck_row0 =
            p.ckpt ? kda::ckpt_first_row(p.cu, w.seq, p.total, p.seq_len, p.ckpt_every * C) : 0;
        float wj = 1.f;
        if (OGATE && p.onorm_w) wj = p.onorm_w[j];
        for (s = w.s0; s < w.s1; ++s) {
            if (named_sync_or(BAR_ST, 128, !ok || aborted(ctl))) {
                ok = false;
                break;
            }
            const uint32_t pp = s & 1u;
            if (s > w.s0 && !(ok = warp_wait(ctl, &ctl.barc[pp ^ 1u], ((s - 1) >> 1) & 1u, 0x31u))) continue;
            if (!(ok = warp_wait(ctl, &ctl.prepped[pp], (s >> 1) & 1u, 0x32u))) continue;
            tc_fence_after();
            // S_w = S_r Diag(e^{Gamma_last}) while the X and U groups read S_r
            {
                const float *gcp = reinterpret_cast<const float *>(base + SB_GC + pp * 512);
#pragma unroll 1
                for (int k0 = 0; k0 < D; k0 += 32) {
                    float x[32];
                    tmem_ld32(tl + tm_sr(pp) + k0, x);
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 g4 = *reinterpret_cast<const float4 *>(gcp + k0 + 4 * i4);
                        x[4 * i4] *= g4.x;
                        x[4 * i4 + 1] *= g4.y;
                        x[4 * i4 + 2] *= g4.z;
                        x[4 * i4 + 3] *= g4.w;
                    }
                    tmem_st32(tl + tm_sw(pp) + k0, x);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.scaled[pp]);
            }
            if (s > w.s0) epilogue(w, s - 1, ck_row0, wj);
            if (s + 1 < nsteps) preload(s + 1);
            tc_fence_before();
        }
        if (!ok) break;
        // the last step of the pair: its output rows and the final state
        if (!(ok = warp_wait(ctl, &ctl.barc[(w.s1 - 1) & 1u], ((w.s1 - 1) >> 1) & 1u, 0x33u))) break;
        tc_fence_after();
        epilogue(w, w.s1 - 1, ck_row0, wj);
        if (p.fin) {
#pragma unroll 1
            for (int k0 = 0; k0 < D; k0 += 32) {
                float x[32];
                tmem_ld32(tl + tm_sw((w.s1 - 1) & 1u) + k0, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) p.fin[soff + (int64_t)(k0 + i) * D + j] = x[i];
            }
        }
        tc_fence_before();
    }
    if (!ok) *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
}

template <typename OUT_T, int GMODE, bool OGATE>
__global__ void __launch_bounds__(kThreads, 1)
kda_chain2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    CtlB &ctl = *reinterpret_cast<CtlB *>(base + SB_CTL);
    const int t = threadIdx.x, warp = t >> 5;
    const int c = (int)blockIdx.x;
    if (t == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.infull[i], 1);
            mbar_init(&ctl.inempty[i], 8);
            mbar_init(&ctl.slotfull[i], 1);
            mbar_init(&ctl.prepped[i], 4);
            mbar_init(&ctl.pre[i], 4);
            mbar_init(&ctl.barx[i], 1);
            mbar_init(&ctl.baru[i], 1);
            mbar_init(&ctl.barc[i], 1);
            mbar_init(&ctl.scaled[i], 4);
        }
        mbar_init(&ctl.sready, 4);
        mbar_init(&ctl.fin, 1);
        fence_mbar_init();
        ctl.abort = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (GMODE != kDecayScalar) prefetch_tmap(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(&ctl.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tmem_base;
    const uint32_t *fs = p.first_step + (size_t)c * (p.KMAX + 1);
    const uint32_t nsteps = fs[chain_pairs(p, c)];
    if (warp == 0) {
        if ((t & 31) == 0) chain_issuer(p, base, ctl, tb, c, fs, nsteps);
        __syncwarp();
    } else if (warp == 1) {
        if ((t & 31) == 0) chain_loader<GMODE>(p, base, ctl, c, fs, nsteps, &tm_q, &tm_k, &tm_v, &tm_g);
        __syncwarp();
    } else if (warp == 2) {
        if ((t & 31) == 0) chain_slots(p, base, ctl, c, fs, nsteps);
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        chain_state<OUT_T, OGATE>(p, base, ctl, tb, c, fs, nsteps);
    } else if (warp >= 12) {
        chain_prep<GMODE, 1>(p, base, ctl, c, fs, nsteps);
    } else if (warp >= 8) {
        chain_prep<GMODE, 0>(p, base, ctl, c, fs, nsteps);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- host side

struct DevInfo {
    int sms = 0;
    cudaMemPool_t pool = nullptr;
    cudaError_t err = cudaSuccess;
};

DevInfo &dev_info(int dev) {
    static DevInfo info[64];
    static std::once_flag once[64];
    std::call_once(once[dev & 63], [dev] {
        DevInfo &d = info[dev & 63];
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) {
            // a pool of this library's own that keeps its memory between calls
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            d.err = cudaMemPoolCreate(&d.pool, &props);
            if (d.err == cudaSuccess) {
                uint64_t keep = UINT64_MAX;
                d.err = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            }
        }
    });
    return info[dev & 63];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename F>
cudaError_t set_smem(F kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int GMODE>
cudaError_t launch_intra(const Params &prm, int grid, cudaStream_t stream) {
    auto kern = kda_intra_kernel<GMODE>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] { attr = set_smem(kern, kSmemA); });
    if (attr != cudaSuccess) return attr;
    kern<<<grid, kThreads, kSmemA, stream>>>(prm);
    return cudaGetLastError();
}

template <typename OUT_T, int GMODE, bool OGATE>
cudaError_t launch_chain(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mg, const Params &prm, cudaStream_t stream) {
    auto kern = kda_chain2_kernel<OUT_T, GMODE, OGATE>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] { attr = set_smem(kern, kSmemB); });
    if (attr != cudaSuccess) return attr;
    kern<<<prm.NC, kThreads, kSmemB, stream>>>(mq, mk, mv, mg, prm);
    return cudaGetLastError();
}

template <typename OUT_T>
cudaError_t launch_chain_out(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                             const CUtensorMap &mg, const Params &prm, int gmode, bool ogate,
                             cudaStream_t stream) {
    if (gmode == kDecayLogits) return launch_chain<OUT_T, kDecayLogits, false>(mq, mk, mv, mg, prm, stream);
    if (gmode == kDecayScalar) return launch_chain<OUT_T, kDecayScalar, false>(mq, mk, mv, mg, prm, stream);
    if constexpr (sizeof(OUT_T) == 2)
        if (ogate) return launch_chain<OUT_T, kDecayTile, true>(mq, mk, mv, mg, prm, stream);
    return launch_chain<OUT_T, kDecayTile, false>(mq, mk, mv, mg, prm, stream);
}

}  // namespace

bool kda_prefill_2pass_supported(const kda::Problem &P) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const DevInfo &d = dev_info(dev);
    return d.err == cudaSuccess && d.sms >= 1 && (int64_t)P.N * P.H <= ((int64_t)1 << 30);
}

cudaError_t kda_launch_prefill_2pass(const kda::Problem &P, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const float *init_state, const int32_t *cu, void *out,
                                     float *final_state, cudaStream_t stream) {
    if (P.N == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DevInfo &di = dev_info(dev);
    if (di.err != cudaSuccess) return di.err;
    const int gmode = P.a_log ? kDecayLogits : P.scalar_decay ? kDecayScalar : kDecayTile;
    CUtensorMap mq, mk, mv, mg;
    if (!kda_make_tile_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !kda_make_tile_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H) ||
        !(gmode == kDecayLogits   ? kda_make_tile_map(&mg, P.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H)
          : gmode == kDecayScalar ? kda_make_tile_map(&mg, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, P.T, P.H)
                                  : kda_make_tile_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, P.T, P.H)))
        return cudaErrorInvalidValue;
    const int pairs = P.N * P.H;
    const int NC = pairs < di.sms ? pairs : di.sms;
    const int KMAX = (pairs + NC - 1) / NC;
    // chunks: sum over sequences of ceil(len / 32) <= T / 32 + N
    const size_t chunks = (size_t)P.T / C + (size_t)P.N;
    size_t off = 0;
    const size_t o_slots = off; off = align256(off + chunks * (size_t)P.H * kSlot);
    const size_t o_coff = off; off = align256(off + ((size_t)P.N + 1) * 4);
    const size_t o_order = off; off = align256(off + (size_t)P.N * 4);
    const size_t o_fs = off; off = align256(off + (size_t)NC * (KMAX + 1) * 4);
    void *ws = nullptr;
    e = cudaMallocFromPoolAsync(&ws, off, di.pool, stream);
    if (e != cudaSuccess) return e;
    unsigned char *w = static_cast<unsigned char *>(ws);
    Params prm = {};
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.k = static_cast<const __nv_bfloat16 *>(k);
    prm.v = static_cast<const __nv_bfloat16 *>(v);
    prm.g = g;
    prm.z = static_cast<const __nv_bfloat16 *>(P.z);
    prm.a_log = P.a_log;
    prm.g_head = P.g_head;
    prm.beta = beta;
    prm.init = init_state;
    prm.cu = cu;
    prm.out = out;
    prm.fin = final_state;
    prm.ckpt = P.ckpt;
    prm.ckpt_every = P.ckpt ? P.ckpt_interval / C : 1;
    prm.ckpt_cap = P.ckpt_capacity;
    prm.ogate = static_cast<const __nv_bfloat16 *>(P.ogate);
    prm.onorm_w = P.onorm_w;
    prm.oeps = P.oeps;
    prm.N = P.N;
    prm.H = P.H;
    prm.total = P.T;
    prm.seq_len = P.seq_len;
    prm.NC = NC;
    prm.KMAX = KMAX;
    prm.slots = w + o_slots;
    prm.chunk_off = reinterpret_cast<int32_t *>(w + o_coff);
    prm.order = reinterpret_cast<int32_t *>(w + o_order);
    prm.first_step = reinterpret_cast<uint32_t *>(w + o_fs);
    twopass_setup_kernel<<<1, 1024, 0, stream>>>(cu, P.N, P.H, (int64_t)P.T, P.seq_len, NC, KMAX,
                                                  prm.chunk_off, prm.order, prm.first_step);
    e = cudaGetLastError();
    if (e == cudaSuccess)
        e = gmode == kDecayLogits   ? launch_intra<kDecayLogits>(prm, di.sms, stream)
            : gmode == kDecayScalar ? launch_intra<kDecayScalar>(prm, di.sms, stream)
                                    : launch_intra<kDecayTile>(prm, di.sms, stream);
    if (e == cudaSuccess)
        e = P.out_dtype == KDA_DTYPE_BF16
                ? launch_chain_out<__nv_bfloat16>(mq, mk, mv, mg, prm, gmode, P.ogate_fused, stream)
                : launch_chain_out<float>(mq, mk, mv, mg, prm, gmode, P.ogate_fused, stream);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

cudaError_t kda_2pass_read_status(unsigned *status) {
    unsigned st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&st, g_kda_2pass_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_kda_2pass_status, &zero, sizeof(unsigned));
    *status |= st;
    return e;
}
