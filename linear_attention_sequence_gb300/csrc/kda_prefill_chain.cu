// kda_prefill_chain.cu -- chunked KDA prefill with the state recurrence and the
// intra-chunk work on different SMs (sm_103a, tcgen05), one cooperative launch.
//
// The chunk form ("Inside Kimi K3", section "Sequence mixing": tokens of a
// chunk in parallel, inclusive diagonal, state carried between chunks;
// "Hybrid Attention", section "But isn't a recurrent update sequential?": a
// triangular solve resolves the in-chunk dependencies), with Gamma the running
// sum of g inside a chunk of C = 32 tokens and gamma = e^Gamma:
//
//   T   = (I + Akk)^{-1},     Tb = T diag(beta)
//   W   = Tb (gamma . K),     U' = Tb V                       (state-independent)
//   U   = U' - W S0
//   O   = (gamma . Q) S0 + Aqk U
//   S_C = Diag(gamma_last) S0 + Kbar^T U,   Kbar_r = e^{Gamma_last - Gamma_r} . k_r
//
// Everything that does not involve the state S0 -- the decay prefix, the
// decay-weighted operands, the Gram matrices Akk and Aqk, the triangular
// solve, W and U' -- is independent from chunk to chunk.  "Intra" CTAs do it
// for any chunk of any (sequence, head), two chunks at a time per unit of
// eight warps, and write each chunk's operands of the state-dependent products
// into a ring of slots in global memory (about 69 KB a chunk; the ring stays in
// L2).  A "chain" CTA owns one (sequence, head) at a time, keeps S^T in tensor
// memory, and per chunk only copies its slot into shared memory (one bulk
// copy) and issues two MMA groups:
//
//   X group  [X_Q | U] = S^T [gamma Q ; -W]^T   onto [0 | U'^T]  (N = 64, K = 128)
//   carry    [S^T | O^T] += U^T [Kbar^T ; Aqk]^T                 (N = 160, K = 32)
//
// with S^T <- S^T Diag(gamma_last) in between, on twelve warps.  The output rows
// are read from tensor memory and stored while the next chunk's X group runs.
//
// Work split.  The grid is one CTA per SM; the first NC CTAs are chains, the
// rest intra CTAs.  (sequence, head) pairs are taken longest first and dealt
// round-robin to the chains; a chain's "steps" are the chunks of its pairs in
// order.  Intra units take (chain, step) items from one atomic counter in step
// order, so the chunks every chain needs next are made first.  Hand-offs
// through global memory: a slot's ready word holds the step it contains (+1),
// written with release semantics after the slot's data; each chain publishes
// how many of its slots it has copied out, and a unit waits for that before it
// overwrites a slot.  Every wait is bounded; one that gives up stops the whole
// grid through a shared abort word and records the device status word.  The
// cooperative launch guarantees that all CTAs are resident at once.
//
// Decay factoring.  Products e^{Gamma_r - Gamma_i} (i <= r) are split around
// the reference Gamma_15: with g >= g_min = -5, |Gamma_r - Gamma_15| <= 80 for
// every token of a 32-token chunk ("Understanding Kimi K3's Attention",
// log-decay bound), so e^{+-(Gamma_r - Gamma_15)} stays inside the fp32/tf32
// normal range and each Gram matrix is one product of bounded factors.
//
// Precision.  Every product is tcgen05.mma kind::tf32 with fp32 accumulation:
// on these inputs u_t and the intra-chunk terms are several times larger than
// o_t, and bf16 operands for any of the Gram, Aqk, U' or S products cost more
// than the 2e-2 error budget.  gamma . K enters W as bf16 (that one is harmless).

#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"
#include "kda_chunk_ops.cuh"

__device__ unsigned int g_kda_chain_status;   // nonzero after a bounded wait gave up

namespace {

using namespace sm100;
using namespace kda_chunk;

constexpr int C = 32;            // tokens per chunk
constexpr int D = 128;           // d_k = d_v
constexpr int kThreads = 512;
constexpr int kRing = 4;         // slots per chain in global memory
constexpr int kStages = 3;       // shared-memory copies of slots in a chain CTA
constexpr uint32_t kPollLimit = 1u << 23;   // mbarrier polls (about half a second)
constexpr uint32_t kSpinLimit = 1u << 22;   // polls of a global word (with back-off)

// Slot layout (bytes).  BX: the X group's B operand, K-major SW128 tf32, 4
// K-blocks of 64 rows x 128 B; rows [gamma Q ; -W] for an even step, [-W ;
// gamma Q] for an odd one.  BC: the carry's B operand, one K-block of 160 rows;
// [Kbar^T ; Aqk] (even) or [Aqk ; Kbar^T] (odd).  UP: U'^T, row j (value j) of
// 32 fp32 with its 16-byte chunk ch at chunk position ch ^ (j % 8).  GC:
// e^{Gamma_last} per key channel.
constexpr uint32_t OFF_BX = 0, OFF_BC = 32768, OFF_UP = 53248, OFF_GC = 69632;
constexpr uint32_t kSlotBytes = 70144;
constexpr uint32_t kSlotStride = 70656;

// Tensor-memory columns of a chain CTA.  S^T (lane = value, column = key
// channel) at 64..191.  Even steps: X region 192..255 = [X_Q | U], carry
// D = [S^T | O^T] at 64 (N = 160).  Odd steps: X region 0..63 = [U | X_Q],
// carry D = [O^T | S^T] at 32.  Both D ranges are contiguous with S^T.
constexpr uint32_t TM_S = 64;

// Intra unit: 256 tensor-memory columns and 96 KB of shared memory each.
//   GD  (64 cols): Gram D (chunk a: lanes 0-63, columns 0-31; chunk b: lanes
//                  64-127, columns 32-63); then W^T_a | U'^T_a.
//   GA (128 cols): Gram A [k~_a ; q~_a ; k~_b ; q~_b] (lanes = rows); then
//                  V^T_a | (gamma K)^T_a | V^T_b | (gamma K)^T_b.
//   WB  (64 cols): W^T_b | U'^T_b.
constexpr uint32_t kUnitBytes = 98304;     // staging 64 KB (Gram A, then Tb/solve scratch) + Gram B 32 KB
constexpr uint32_t kChainBytes = kStages * kSlotStride;
constexpr uint32_t kCtlOff = kChainBytes > 2 * kUnitBytes ? kChainBytes : 2 * kUnitBytes;

constexpr uint32_t BAR_SC = 3, BAR_OG = 4;   // named barriers of the chain CTA (1, 2: intra units)

struct Scratch {
    unsigned char *ring;    // [NC][kRing][kSlotStride]
    uint32_t *ready;        // [NC][kRing]: step + 1 of the slot's content
    uint32_t *progress;     // [NC]: slots copied out so far
    uint32_t *first_step;   // [NC][KMAX + 1]: first step of each pair of the chain, then the total
    int32_t *order;         // [N]: sequences, longest first
    uint32_t *ctrl;         // [0] item counter, [1] abort, [2] most steps of any chain
};

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
    int NC, KMAX;
    Scratch sc;
};

struct Item {
    int chain, seq, h, L;
    uint32_t step;
    int64_t t0;
};
// The items of one unit for one pair, decoded ahead of time by its thread 0.
struct PairItems {
    Item it[2];
    int valid[2];
    int done;   // no item left for this unit
};

struct Ctl {
    uint64_t full[kStages], empty[kStages], barx, barc[2], pre[2], scaled, sready, fin;
    uint64_t gram[2], wu[2];
    uint32_t tmem_base;
    int abort;
    float ored[4][32];
    PairItems items[2][2];   // intra units: [unit][current / next pair]
};
static_assert(kCtlOff + sizeof(Ctl) + 1024 <= 232448, "shared memory budget");

constexpr int kDecayTile = 0, kDecayLogits = 1, kDecayScalar = 2;

__device__ __forceinline__ bool aborted(Ctl &ctl) {
    return *reinterpret_cast<volatile int *>(&ctl.abort) != 0;
}
__device__ __noinline__ void fail(Ctl &ctl, const Params &p, unsigned code) {
    *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
    atomicExch(p.sc.ctrl + 1, 1u);
    atomicOr(&g_kda_chain_status, code);
}
__device__ __forceinline__ bool global_abort(const Params &p) {
    return *reinterpret_cast<volatile const uint32_t *>(p.sc.ctrl + 1) != 0;
}
// Bounded wait for an mbarrier phase; gives up early when the CTA or the grid stops.
__device__ __noinline__ bool wait_slow(Ctl &ctl, const Params &p, uint64_t *bar, uint32_t par,
                                       unsigned code) {
    for (uint32_t i = 0; i < kPollLimit; ++i) {
        if (mbar_try_wait(bar, par)) return true;
        if ((i & 255) == 255) {
            if (aborted(ctl) || global_abort(p)) {
                *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
                return false;
            }
            __nanosleep(64);
        }
    }
    fail(ctl, p, code);
    return false;
}
__device__ __forceinline__ bool wait_bar(Ctl &ctl, const Params &p, uint64_t *bar, uint32_t par,
                                         unsigned code) {
    return mbar_try_wait(bar, par) || wait_slow(ctl, p, bar, par, code);
}
// Bounded poll of a global word: until *w == want (eq) or *w >= want.
__device__ __noinline__ bool poll_word(Ctl &ctl, const Params &p, const uint32_t *w, uint32_t want,
                                       bool eq, unsigned code) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        const uint32_t x = ld_acquire_gpu(w);
        if (eq ? x == want : x >= want) return true;
        if ((i & 7) == 7 && (aborted(ctl) || global_abort(p))) {
            *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
            return false;
        }
        __nanosleep(i < 32 ? 32 : 256);
    }
    fail(ctl, p, code);
    return false;
}

__device__ __forceinline__ float ldg_bf16(const __nv_bfloat16 *p) {
    return __bfloat162float(__ldg(p));
}

// ---------------------------------------------------------------------------
// Which (sequence, head) and chunk a step of a chain is.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int chain_pairs(const Params &p, int c) {
    const int P = p.N * p.H;
    return (P - c + p.NC - 1) / p.NC;
}
__device__ bool decode_item(const Params &p, uint32_t ticket, uint32_t total, Item &it) {
    if (ticket >= total) return false;
    const int c = (int)(ticket % (uint32_t)p.NC);
    const uint32_t s = ticket / (uint32_t)p.NC;
    const int np = chain_pairs(p, c);
    const uint32_t *fs = p.sc.first_step + (size_t)c * (p.KMAX + 1);
    if (s >= fs[np]) return false;
    int lo = 0, hi = np - 1;   // the last pair whose first step is <= s (it has chunks)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (fs[mid] <= s) lo = mid;
        else hi = mid - 1;
    }
    const int pi = c + lo * p.NC;
    it.chain = c;
    it.step = s;
    it.seq = p.sc.order[pi / p.H];
    it.h = pi % p.H;
    int64_t a, b;
    kda::seq_bounds(p.cu, it.seq, p.total, p.seq_len, a, b);
    it.t0 = a + (int64_t)(s - fs[lo]) * C;
    const int64_t rem = b - it.t0;
    it.L = (int)(rem < C ? rem : C);
    return true;
}

// ---------------------------------------------------------------------------
// Setup (one block): clear the hand-off words, order the sequences longest
// first and lay out each chain's steps.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) chain_setup_kernel(const int32_t *cu, int N, int H,
                                                           int64_t total, int64_t seq_len, int NC,
                                                           int KMAX, Scratch sc) {
    const int t = threadIdx.x;
    for (int i = t; i < NC * kRing; i += blockDim.x) sc.ready[i] = 0;
    for (int i = t; i < NC; i += blockDim.x) sc.progress[i] = 0;
    if (t < 4) sc.ctrl[t] = 0;
    if (cu && N <= (int)blockDim.x) {
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
            sc.order[rank] = t;
        }
    } else {
        for (int i = t; i < N; i += blockDim.x) sc.order[i] = i;
    }
    __syncthreads();
    if (t < NC) {
        const int P = N * H;
        uint32_t *fs = sc.first_step + (size_t)t * (KMAX + 1);
        uint32_t acc = 0;
        int k = 0;
        for (int pi = t; pi < P; pi += NC, ++k) {
            fs[k] = acc;
            int64_t a, b;
            kda::seq_bounds(cu, sc.order[pi / H], total, seq_len, a, b);
            acc += (uint32_t)((b - a + C - 1) / C);
        }
        fs[k] = acc;
        atomicMax(sc.ctrl + 2, acc);
    }
}

// ---------------------------------------------------------------------------
// Intra role: two units of eight warps, each making the slots of two chunks.
// Thread (half x, channel c) of a unit: x = chunk a or b, c = key/value channel
// = its tensor-memory lane.
// ---------------------------------------------------------------------------

// Take the next two items for a unit and decode them (thread 0 of the unit).
__device__ void take_items(const Params &p, uint32_t total, PairItems &pi) {
    uint32_t tk;
    do {   // tickets whose chains have run out of steps are skipped
        tk = atomicAdd(p.sc.ctrl + 0, 2u);
        pi.done = tk >= total;
#pragma unroll
        for (int x = 0; x < 2; ++x) pi.valid[x] = decode_item(p, tk + (uint32_t)x, total, pi.it[x]) ? 1 : 0;
    } while (!pi.done && !pi.valid[0] && !pi.valid[1]);
}
// Wait until the items' ring slots have been copied out by their chains.  A unit
// never waits here while it holds slots it has filled but not yet published, so
// the waits cannot form a cycle.
__device__ bool wait_slots(Ctl &ctl, const Params &p, const PairItems &pi) {
    bool ok = true;
#pragma unroll
    for (int x = 0; x < 2; ++x)
        if (ok && pi.valid[x] && pi.it[x].step >= (uint32_t)kRing)
            ok = poll_word(ctl, p, p.sc.progress + pi.it[x].chain, pi.it[x].step - kRing + 1, false,
                           0x10u);
    return ok;
}
__device__ __forceinline__ void publish_items(const Params &p, const PairItems &pi) {
    bool any = false;
#pragma unroll
    for (int x = 0; x < 2; ++x) any |= pi.valid[x] != 0;
    if (!any) return;
    __threadfence();
#pragma unroll
    for (int x = 0; x < 2; ++x)
        if (pi.valid[x])
            st_relaxed_gpu(p.sc.ready + pi.it[x].chain * kRing + pi.it[x].step % kRing,
                           pi.it[x].step + 1);
}

template <int GMODE>
__device__ void intra_role(const Params &p, unsigned char *base, Ctl &ctl, uint32_t tb) {
    const int t = threadIdx.x, u = t >> 8, T = t & 255, hx = T >> 7, c = T & 127;
    const int wu = T >> 5, lane = t & 31;
    const uint32_t lane_off = (uint32_t)(32 * (wu & 3)) << 16;
    const uint32_t tu = tb + 256u * (uint32_t)u;
    const uint32_t GD = tu, GA = tu + 64, WB = tu + 192;
    unsigned char *stg = base + u * kUnitBytes;   // Gram A staging, then Tb / solve scratch
    unsigned char *gB = stg + 65536;              // Gram B: 4 K-blocks x 64 rows
    const uint32_t bar_id = 1 + u;
    const uint32_t total = (uint32_t)p.NC * ld_acquire_gpu(p.sc.ctrl + 2);
    const int64_t rs = (int64_t)p.H * D;   // token stride of [T, H, D] tensors
    uint32_t gpar = 0, wpar = 0;
    PairItems *items = ctl.items[u];        // [2]: current and next pair (by iteration parity)
    bool ok = true;
    if (T == 0) {
        take_items(p, total, items[0]);
        ok = wait_slots(ctl, p, items[0]);
    }
    int cur = 0;

    for (;;) {
        if (named_sync_or(bar_id, 256, !ok || aborted(ctl) || global_abort(p))) break;
        const PairItems &pi = items[cur];
        if (pi.done) break;
        const bool valid = pi.valid[hx] != 0;
        Item it = pi.it[hx];
        const int L = valid ? it.L : 0;
        const int pp = valid ? (int)(it.step & 1u) : 0;
        unsigned char *slot =
            valid ? p.sc.ring + ((size_t)it.chain * kRing + it.step % kRing) * kSlotStride : nullptr;

        // ---- phase 1 (thread = channel c of chunk hx): decay prefix, decay-weighted operands ----
        const int64_t e0 = valid ? (it.t0 * p.H + it.h) * (int64_t)D + c : 0;   // element (t0, h, c)
        const int64_t b0i = valid ? it.t0 * p.H + it.h : 0;                      // beta / g_head index
        float gsc = 0.f;
        if (GMODE == kDecayLogits && valid) gsc = __expf(p.a_log[it.h]);
        float gam[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {   // every load first, then the running sum
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
        const float g15 = gam[15], gl = gam[C - 1];
        const float E15 = __expf(g15), EL15 = __expf(gl - g15);
        {
            // 128-byte swizzle: channel c's float sits in 16-byte chunk ((c % 32) / 4) ^ (row % 8)
            // of its row; rows below are multiples of 8 plus r, so row % 8 = r % 8
            uint32_t swz[8];
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) swz[k8] = (uint32_t)(((((c & 31) >> 2) ^ k8) << 4) + ((c & 3) << 2));
            unsigned char *stK = stg + (c >> 5) * 16384 + (hx ? 64 : 0) * 128;   // k~ rows of this chunk
            unsigned char *stQ = stK + 32 * 128;                                  // q~ rows
            unsigned char *gBr = gB + (c >> 5) * 8192 + (hx ? 32 : 0) * 128;     // k^ rows
            unsigned char *bxQ = valid ? slot + OFF_BX + (c >> 5) * 8192 + (pp ? 32 : 0) * 128 : nullptr;
            const int rowc = pp ? 32 + c : c;   // this channel's row of Kbar^T in BC
            unsigned char *bcR = valid ? slot + OFF_BC + rowc * 128 : nullptr;
            float kb4[4];
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
                __nv_bfloat16 qr[16], kr[16], vr[16];   // 16 tokens' loads in flight together
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * h16 + i;
                    const __nv_bfloat16 zero = __float2bfloat16(0.f);
                    qr[i] = r < L ? __ldg(p.q + e0 + r * rs) : zero;
                    kr[i] = r < L ? __ldg(p.k + e0 + r * rs) : zero;
                    vr[i] = r < L ? __ldg(p.v + e0 + r * rs) : zero;
                }
                uint32_t vpk[8], gkpk[8];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * h16 + i;
                    const uint32_t so = (uint32_t)r * 128 + swz[r & 7];
                    const float qv = __bfloat162float(qr[i]), kv = __bfloat162float(kr[i]);
                    const float x = gam[r] - g15;
                    const float e1 = __expf(x);    // e^{Gamma_r - Gamma_15} in [e^-80, e^75]
                    const float inv = __expf(-x);  // its inverse
                    const float kh = kv * inv;
                    *reinterpret_cast<float *>(stK + so) = to_tf32(kv * e1);
                    *reinterpret_cast<float *>(stQ + so) = to_tf32(qv * e1);
                    *reinterpret_cast<float *>(gBr + so) = to_tf32(kh);
                    const float gm = e1 * E15;     // e^{Gamma_r}
                    if (valid) *reinterpret_cast<float *>(bxQ + so) = to_tf32(qv * gm);
                    const uint32_t gkb = __bfloat16_as_ushort(__float2bfloat16_rn(kv * gm));
                    const uint32_t vb = __bfloat16_as_ushort(vr[i]);
                    if (i & 1) {
                        gkpk[i >> 1] |= gkb << 16;
                        vpk[i >> 1] |= vb << 16;
                    } else {
                        gkpk[i >> 1] = gkb;
                        vpk[i >> 1] = vb;
                    }
                    kb4[r & 3] = to_tf32(kh * EL15);   // k_r e^{Gamma_last - Gamma_r}
                    if ((r & 3) == 3 && valid)
                        *reinterpret_cast<float4 *>(bcR + (((r >> 2) ^ (rowc & 7)) << 4)) =
                            make_float4(kb4[0], kb4[1], kb4[2], kb4[3]);
                }
                // V and gamma K of this channel, packed bf16 pairs, parked in WB until the
                // Gram is done (WB's previous content was read out before the last barrier)
                if (h16 == 0) tc_fence_after();
                tmem_st8(WB + lane_off + 32 * hx + 8 * h16, vpk);
                tmem_st8(WB + lane_off + 32 * hx + 16 + 8 * h16, gkpk);
            }
        }
        if (valid) reinterpret_cast<float *>(slot + OFF_GC)[c] = __expf(gl);
        fence_proxy_async_smem();   // the Gram B operand is read by the tensor cores
        tmem_wait_st();
        tc_fence_before();
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

        // ---- phase 3: Gram = [k~_a ; q~_a ; k~_b ; q~_b] [k^_a ; k^_b]^T (N = 64).  While
        // it runs, thread 0 takes and decodes the next pair and publishes the last one. ----
        if (T == 0) {
            tc_fence_after();
            const uint64_t dB = sdesc_sw128(smem_u32(gB));
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32_ts(GD, GA + 8 * kk, dB + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                            idesc_tf32(128, 64), kk > 0);
            mma_commit(&ctl.gram[u]);
            take_items(p, total, items[cur ^ 1]);   // decoded while the Gram runs
            ok = wait_bar(ctl, p, &ctl.gram[u], gpar, 0x11u);
        }
        gpar ^= 1u;
        if (named_sync_or(bar_id, 256, !ok || aborted(ctl))) break;
        tc_fence_after();

        // ---- phase 4: V^T and (gamma K)^T (tf32) into GA (the Gram has read it); Akk rows
        // solved (warps 0 and 6), Aqk rows stored (warps 1 and 7); the next pair's inputs
        // are prefetched into L2 ----
        {
            float x16[16], x[32];
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
                tmem_ld16(WB + lane_off + 32 * hx + 16 * w2, x16);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t pk = __float_as_uint(x16[i]);
                    x[2 * i] = __uint_as_float(pk << 16);
                    x[2 * i + 1] = __uint_as_float(pk & 0xffff0000u);
                }
                tmem_st32(GA + lane_off + 64 * hx + 32 * w2, x);
            }
        }
        {
            // the next pair's input rows into L2: thread c of half x takes token c % 32 and
            // 128-byte line c / 32 of its q, k, v (two lines each) and g (four lines) rows
            const PairItems &nx = items[cur ^ 1];
            const int r = c & 31, ln = c >> 5;
            if (!nx.done && nx.valid[hx] && r < nx.it[hx].L) {
                const Item &ni = nx.it[hx];
                const int64_t row = (ni.t0 + r) * p.H + ni.h;   // (token, head) row of the next chunk
                if (ln < 2) {
                    prefetch_l2(p.q + row * D + 64 * ln);
                    prefetch_l2(p.k + row * D + 64 * ln);
                    prefetch_l2(p.v + row * D + 64 * ln);
                    if (GMODE == kDecayLogits) prefetch_l2(p.z + row * D + 64 * ln);
                }
                if (GMODE == kDecayTile) prefetch_l2(p.g + row * D + 32 * ln);
            }
        }
        if (wu == 0 || wu == 6) {
            const int xb = wu == 6;
            float d[32];
            tmem_ld32(GD + lane_off + 32 * xb, d);
            float br = 0.f;
            if (lane < L) {
                br = __ldg(p.beta + b0i + lane * p.H);
                if (GMODE == kDecayLogits) br = kda::sigmoid_f(br);
            }
            float(*akkT)[32] = reinterpret_cast<float(*)[32]>(stg + 8192 + 4096 * xb);
            float(*tsc)[16][20] = reinterpret_cast<float(*)[16][20]>(stg + 16384 + 4096 * xb);
            solve_tbeta(d, br, lane, stg + 4096 * xb, akkT, tsc);
        } else if (wu == 1 || wu == 7) {
            const int xb = wu == 7;
            float d[32];
            tmem_ld32(GD + lane_off + 32 * xb, d);
            if (valid) {
                const int row = pp ? lane : 128 + lane;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float a4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) a4[e] = 4 * ch + e <= lane ? to_tf32(d[4 * ch + e]) : 0.f;
                    *reinterpret_cast<float4 *>(slot + OFF_BC + row * 128 + ((ch ^ (row & 7)) << 4)) =
                        make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        named_sync(bar_id, 256);

        // ---- phase 5: W^T = (gamma K)^T Tb^T and U'^T = V^T Tb^T for both chunks ----
        if (T == 0) {
            tc_fence_after();
#pragma unroll
            for (int xb = 0; xb < 2; ++xb) {
                const uint64_t dT = sdesc_sw128(smem_u32(stg + 4096 * xb));
                const uint32_t dw = xb ? WB : GD, av = GA + 64 * xb;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_tf32_ts(dw, av + 32 + 8 * kk, dT + (uint64_t)((kk * 32) >> 4), idesc_tf32(128, 32),
                                kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_tf32_ts(dw + 32, av + 8 * kk, dT + (uint64_t)((kk * 32) >> 4), idesc_tf32(128, 32),
                                kk > 0);
            }
            mma_commit(&ctl.wu[u]);
            ok = wait_bar(ctl, p, &ctl.wu[u], wpar, 0x12u);
        }
        wpar ^= 1u;
        if (named_sync_or(bar_id, 256, !ok || aborted(ctl))) break;
        tc_fence_after();

        // ---- phase 6: -W rows of BX (column c) and U'^T row c into the slot ----
        if (valid) {
            const uint32_t wcol = hx ? WB : GD;
            float w[32];
            tmem_ld32(wcol + lane_off, w);
#pragma unroll
            for (int r = 0; r < C; ++r) st_f(slot, OFF_BX + sw_off(64, pp ? r : 32 + r, c), to_tf32(-w[r]));
            tmem_ld32(wcol + lane_off + 32, w);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<float4 *>(slot + OFF_UP + c * 128 + ((ch ^ (c & 7)) << 4)) =
                    make_float4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
        }
        tc_fence_before();
        named_sync(bar_id, 256);
        // the slots of this pair are complete: thread 0 publishes them while thread 32
        // waits for the next pair's slots
        if (T == 0) publish_items(p, pi);
        if (T == 32 && !items[cur ^ 1].done) ok = wait_slots(ctl, p, items[cur ^ 1]);
        cur ^= 1;
    }
    if (T == 0) {   // every MMA issued by this unit has completed (after a stop too)
        tc_fence_after();
        mma_commit(&ctl.gram[u]);
        mbar_wait_bounded(&ctl.gram[u], gpar, kPollLimit);
    }
}

// ---------------------------------------------------------------------------
// Chain role.  Warp 0 issues the MMAs, warp 1 copies slots in, warps 4-7 load
// states, preload U'^T, store the outputs and, with warps 8-15, scale the state
// (three warps per TMEM lane quarter, 16-column pieces).  Thread j of warps 4-15
// owns TMEM lane j % 128 = value index.
// ---------------------------------------------------------------------------
__device__ void chain_issuer(const Params &p, unsigned char *base, Ctl &ctl, uint32_t tb, int c,
                             int npairs, const uint32_t *fs) {
    uint32_t s = 0, sr_par = 0;
    bool ok = true;
    for (int kp = 0; kp < npairs && ok; ++kp) {
        const uint32_t s_end = fs[kp + 1];
        if (s_end == s) continue;
        ok = wait_bar(ctl, p, &ctl.sready, sr_par, 0x20u);
        sr_par ^= 1u;
        for (; ok && s < s_end; ++s) {
            const int st = (int)(s % kStages);
            const uint32_t pp = s & 1u;
            unsigned char *stage = base + st * kSlotStride;
            if (!(ok = wait_bar(ctl, p, &ctl.full[st], (s / kStages) & 1u, 0x21u))) break;
            // the slot in global memory is free again (its copy has landed: no fence needed)
            st_relaxed_gpu(p.sc.progress + c, s + 1);
            if (!(ok = wait_bar(ctl, p, &ctl.pre[pp], (s >> 1) & 1u, 0x22u))) break;
            tc_fence_after();
            const uint64_t dX = sdesc_sw128(smem_u32(stage + OFF_BX));
            const uint32_t xcol = pp ? 0u : 192u;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32_ts(tb + xcol, tb + TM_S + 8 * kk,
                            dX + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_tf32(128, 64), 1u);
            mma_commit(&ctl.barx);
            if (!(ok = wait_bar(ctl, p, &ctl.barx, s & 1u, 0x23u))) break;
            if (!(ok = wait_bar(ctl, p, &ctl.scaled, s & 1u, 0x24u))) break;
            tc_fence_after();
            const uint64_t dC = sdesc_sw128(smem_u32(stage + OFF_BC));
            const uint32_t dcol = pp ? 32u : 64u, acol = pp ? 0u : 224u;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ts(tb + dcol, tb + acol + 8 * kk, dC + (uint64_t)((kk * 32) >> 4),
                            idesc_tf32(128, 160), 1u);
            mma_commit(&ctl.barc[pp]);
            mma_commit(&ctl.empty[st]);
            if (!(ok = wait_bar(ctl, p, &ctl.barc[pp], (s >> 1) & 1u, 0x25u))) break;
        }
    }
    mma_commit(&ctl.fin);   // every MMA issued here has completed
    mbar_wait_bounded(&ctl.fin, 0, kPollLimit);
}

__device__ void chain_loader(const Params &p, unsigned char *base, Ctl &ctl, int c, uint32_t nsteps) {
    uint32_t issued = 0;
    for (uint32_t s = 0; s < nsteps; ++s) {
        const int st = (int)(s % kStages);
        if (s >= (uint32_t)kStages && !wait_bar(ctl, p, &ctl.empty[st], (s / kStages - 1) & 1u, 0x26u)) break;
        if (!poll_word(ctl, p, p.sc.ready + c * kRing + s % kRing, s + 1, true, 0x27u)) break;
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&ctl.full[st], kSlotBytes);
        bulk_g2s(base + st * kSlotStride, p.sc.ring + ((size_t)c * kRing + s % kRing) * kSlotStride,
                 kSlotBytes, &ctl.full[st]);
        issued = s + 1;
    }
    // every copy issued has landed before the CTA can exit (its consumer may have stopped)
    for (uint32_t s = issued > (uint32_t)kStages ? issued - kStages : 0; s < issued; ++s)
        mbar_wait_bounded(&ctl.full[s % kStages], (s / kStages) & 1u, kPollLimit);
}

// Lane 0 waits for a phase; the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(Ctl &ctl, const Params &p, uint64_t *bar, uint32_t par,
                                          unsigned code) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(ctl, p, bar, par, code);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <typename OUT_T, bool OGATE>
__device__ void chain_epilogue(const Params &p, unsigned char *base, Ctl &ctl, uint32_t tb, int c,
                               int npairs, const uint32_t *fs, uint32_t nsteps) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, q4 = warp & 3;
    const bool lo = warp < 8;   // warps 4-7 (else 8-15: they only scale)
    const int sg = (warp - 4) >> 2;   // scale group: 16-column pieces [3 sg, 3 sg + 3) of S^T (8 in all)
    const int j = 32 * q4 + lane;
    const uint32_t tl = tb + ((uint32_t)(32 * q4) << 16);
    const int64_t hd = (int64_t)p.H * D;
    bool ok = true;

    auto preload = [&](uint32_t s2) {   // [0 | U'^T] (even) or [U'^T | 0] (odd) into the step's X region
        const int st2 = (int)(s2 % kStages);
        ok = ok && warp_wait(ctl, p, &ctl.full[st2], (s2 / kStages) & 1u, 0x30u);
        if (!ok) return;
        const unsigned char *up = base + st2 * kSlotStride + OFF_UP + j * 128;
        float x[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const float4 v4 = *reinterpret_cast<const float4 *>(up + ((ch ^ (j & 7)) << 4));
            x[4 * ch] = v4.x;
            x[4 * ch + 1] = v4.y;
            x[4 * ch + 2] = v4.z;
            x[4 * ch + 3] = v4.w;
        }
        const bool odd = (s2 & 1u) != 0;
        tmem_st32(tl + (odd ? 0u : 224u), x);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.f;
        tmem_st32(tl + (odd ? 32u : 192u), x);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.pre[s2 & 1u]);
    };

    uint32_t s = 0;
    for (int kp = 0; kp < npairs; ++kp) {
        const int pi = c + kp * p.NC;
        const int seq = p.sc.order[pi / p.H], h = pi % p.H;
        int64_t a, b;
        kda::seq_bounds(p.cu, seq, p.total, p.seq_len, a, b);
        const uint32_t s0 = fs[kp], s_end = fs[kp + 1];
        const int64_t soff = ((int64_t)seq * p.H + h) * D * D;
        if (s_end == s0) {   // an empty sequence: the final state is the initial one
            if (lo && p.fin)
                for (int cc = 0; cc < D; ++cc)
                    p.fin[soff + (int64_t)cc * D + j] = p.init ? p.init[soff + (int64_t)cc * D + j] : 0.f;
            continue;
        }
        if (lo) {
            // the initial state: S^T row j = column j of S
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = p.init ? p.init[soff + (int64_t)(c0 + i) * D + j] : 0.f;
                tmem_st32(tl + TM_S + c0, x);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.sready);
            if (s == 0) preload(0);
        }
        const int64_t ck_row0 =
            p.ckpt ? kda::ckpt_first_row(p.cu, seq, p.total, p.seq_len, p.ckpt_every * C) : 0;
        float wj = 1.f;
        if (OGATE && p.onorm_w) wj = p.onorm_w[j];
        for (; s < s_end; ++s) {
            if (named_sync_or(BAR_SC, 384, !ok || aborted(ctl))) {
                ok = false;
                break;
            }
            const int st = (int)(s % kStages);
            const uint32_t pp = s & 1u;
            const unsigned char *stage = base + st * kSlotStride;
            // S^T <- S^T Diag(e^{Gamma_last}) once the X group has read S
            if (!(ok = warp_wait(ctl, p, &ctl.barx, s & 1u, 0x31u))) continue;
            tc_fence_after();
            {
                const float *gc = reinterpret_cast<const float *>(stage + OFF_GC);
#pragma unroll
                for (int pc = 3 * sg; pc < 3 * sg + 3; ++pc) {
                    if (pc >= 8) break;
                    float x[16];
                    tmem_ld16(tl + TM_S + 16 * pc, x);
#pragma unroll
                    for (int i4 = 0; i4 < 4; ++i4) {
                        const float4 g4 = *reinterpret_cast<const float4 *>(gc + 16 * pc + 4 * i4);
                        x[4 * i4] *= g4.x;
                        x[4 * i4 + 1] *= g4.y;
                        x[4 * i4 + 2] *= g4.z;
                        x[4 * i4 + 3] *= g4.w;
                    }
                    tmem_st16(tl + TM_S + 16 * pc, x);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.scaled);
            }
            if (!lo) continue;
            if (s + 1 < nsteps) preload(s + 1);
            // the output rows of step s
            const int n = (int)(s - s0);
            const int64_t t0 = a + (int64_t)n * C;
            const int L = (int)(b - t0 < C ? b - t0 : C);
            float og[C];
            if (OGATE) {
#pragma unroll
                for (int r = 0; r < C; ++r)
                    og[r] = r < L ? ldg_bf16(p.ogate + (t0 + r) * hd + (int64_t)h * D + j) : 0.f;
            }
            if (!(ok = ok && warp_wait(ctl, p, &ctl.barc[pp], (s >> 1) & 1u, 0x32u))) continue;
            tc_fence_after();
            float o[32];
            tmem_ld32(tl + (pp ? 32u : 192u), o);
            if (OGATE) {
                // y_r = Sigmoid(gate_r) o_r / sqrt(mean_j o_rj^2 + eps) w_j: the sum of
                // squares of row r is reduce-scattered in each warp (lane L ends with
                // its warp's sum for row L), then the four warps' sums meet in shared memory
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
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    o[r] *= __shfl_sync(0xffffffffu, rinv, r) * wj * kda::sigmoid_f(og[r]);
            }
            OUT_T *dst = reinterpret_cast<OUT_T *>(p.out) + (t0 * p.H + h) * (int64_t)D + j;
#pragma unroll
            for (int r = 0; r < C; ++r)
                if (r < L) kda::st_elem(dst + r * hd, o[r]);
            // state checkpoint after every ckpt_every full chunks
            if (p.ckpt && (n + 1) % p.ckpt_every == 0 && L == C) {
                const int64_t ck = ck_row0 + (n + 1) / p.ckpt_every - 1;
                if (ck < p.ckpt_cap) {
                    float *dstS = p.ckpt + (ck * p.H + h) * (int64_t)D * D + j;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float x[32];
                        tmem_ld32(tl + TM_S + c0, x);
#pragma unroll
                        for (int i = 0; i < 32; ++i) dstS[(int64_t)(c0 + i) * D] = x[i];
                    }
                }
            }
            if (s + 1 == s_end && p.fin) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float x[32];
                    tmem_ld32(tl + TM_S + c0, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) p.fin[soff + (int64_t)(c0 + i) * D + j] = x[i];
                }
            }
            tc_fence_before();
        }
        if (!ok) break;
    }
    if (!ok) *reinterpret_cast<volatile int *>(&ctl.abort) = 1;
}

template <typename OUT_T, int GMODE, bool OGATE>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_chain_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kCtlOff);
    const int t = threadIdx.x, warp = t >> 5;
    const int c = (int)blockIdx.x;
    const bool chain = c < p.NC;
    if (t == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&ctl.full[i], 1);
            mbar_init(&ctl.empty[i], 1);
        }
        mbar_init(&ctl.barx, 1);
        mbar_init(&ctl.barc[0], 1);
        mbar_init(&ctl.barc[1], 1);
        mbar_init(&ctl.pre[0], 4);
        mbar_init(&ctl.pre[1], 4);
        mbar_init(&ctl.scaled, 12);
        mbar_init(&ctl.sready, 4);
        mbar_init(&ctl.fin, 1);
        mbar_init(&ctl.gram[0], 1);
        mbar_init(&ctl.gram[1], 1);
        mbar_init(&ctl.wu[0], 1);
        mbar_init(&ctl.wu[1], 1);
        fence_mbar_init();
        ctl.abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(&ctl.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tmem_base;
    if (chain) {
        const int npairs = chain_pairs(p, c);
        const uint32_t *fs = p.sc.first_step + (size_t)c * (p.KMAX + 1);
        const uint32_t nsteps = fs[npairs];
        if (warp == 0) {
            if ((t & 31) == 0) chain_issuer(p, base, ctl, tb, c, npairs, fs);
            __syncwarp();
        } else if (warp == 1) {
            if ((t & 31) == 0) chain_loader(p, base, ctl, c, nsteps);
            __syncwarp();
        } else if (warp >= 4) {
            chain_epilogue<OUT_T, OGATE>(p, base, ctl, tb, c, npairs, fs, nsteps);
        }
    } else {
        intra_role<GMODE>(p, base, ctl, tb);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- host side

struct DevInfo {
    int sms = 0;
    bool coop = false;
    cudaMemPool_t pool = nullptr;
    cudaError_t err = cudaSuccess;
};

DevInfo &dev_info(int dev) {
    static DevInfo info[64];
    static std::once_flag once[64];
    std::call_once(once[dev & 63], [dev] {
        DevInfo &d = info[dev & 63];
        int coop = 0;
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        d.coop = coop != 0;
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

constexpr size_t kSmemBytes = kCtlOff + sizeof(Ctl) + 1024;

// Number of chain CTAs for a grid of `sms` CTAs: about 0.63 of the SMs (96 of
// 152), where the measured cost of a chain step and of an intra chunk balance.
int chain_count(int sms, int pairs) {
    int nc = (sms * 96 + 76) / 152;
    if (nc > sms - 1) nc = sms - 1;
    if (nc < 1) nc = 1;
    return pairs < nc ? pairs : nc;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename OUT_T, int GMODE, bool OGATE>
cudaError_t launch_t(const Params &prm, int grid, cudaStream_t stream) {
    auto kern = kda_prefill_chain_kernel<OUT_T, GMODE, OGATE>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <typename OUT_T>
cudaError_t launch_out(const Params &prm, int grid, int gmode, bool ogate, cudaStream_t stream) {
    if (gmode == kDecayLogits) return launch_t<OUT_T, kDecayLogits, false>(prm, grid, stream);
    if (gmode == kDecayScalar) return launch_t<OUT_T, kDecayScalar, false>(prm, grid, stream);
    if constexpr (sizeof(OUT_T) == 2)
        if (ogate) return launch_t<OUT_T, kDecayTile, true>(prm, grid, stream);
    return launch_t<OUT_T, kDecayTile, false>(prm, grid, stream);
}

}  // namespace

bool kda_prefill_chain_supported(const kda::Problem &P, const void *q, const void *k, const void *v,
                                 const float *g, const void *out) {
    auto al16 = [](const void *x) { return ((uintptr_t)x & 15u) == 0; };
    if (!(P.dk == 128 && P.dv == 128 && P.in_dtype == KDA_DTYPE_BF16 && P.T > 0 && P.N > 0))
        return false;
    if (!(al16(q) && al16(k) && al16(v) && (P.scalar_decay || al16(g)) && al16(out))) return false;
    if ((int64_t)P.N * P.H > (int64_t)1 << 30) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const DevInfo &d = dev_info(dev);
    return d.err == cudaSuccess && d.coop && d.sms >= 2;
}

cudaError_t kda_launch_prefill_chain(const kda::Problem &P, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const float *init_state, const int32_t *cu, void *out,
                                     float *final_state, cudaStream_t stream) {
    if (P.N == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DevInfo &di = dev_info(dev);
    if (di.err != cudaSuccess) return di.err;
    const int pairs = P.N * P.H;
    const int grid = di.sms;
    const int NC = chain_count(grid, pairs);
    const int KMAX = (pairs + NC - 1) / NC;
    // scratch: ring, hand-off words, step table, sequence order
    size_t off = 0;
    const size_t o_ring = off; off = align256(off + (size_t)NC * kRing * kSlotStride);
    const size_t o_ready = off; off = align256(off + (size_t)NC * kRing * 4);
    const size_t o_prog = off; off = align256(off + (size_t)NC * 4);
    const size_t o_fs = off; off = align256(off + (size_t)NC * (KMAX + 1) * 4);
    const size_t o_order = off; off = align256(off + (size_t)P.N * 4);
    const size_t o_ctrl = off; off = align256(off + 16);
    void *ws = nullptr;
    e = cudaMallocFromPoolAsync(&ws, off, di.pool, stream);
    if (e != cudaSuccess) return e;
    unsigned char *w = static_cast<unsigned char *>(ws);
    Scratch sc;
    sc.ring = w + o_ring;
    sc.ready = reinterpret_cast<uint32_t *>(w + o_ready);
    sc.progress = reinterpret_cast<uint32_t *>(w + o_prog);
    sc.first_step = reinterpret_cast<uint32_t *>(w + o_fs);
    sc.order = reinterpret_cast<int32_t *>(w + o_order);
    sc.ctrl = reinterpret_cast<uint32_t *>(w + o_ctrl);
    chain_setup_kernel<<<1, 1024, 0, stream>>>(cu, P.N, P.H, (int64_t)P.T, P.seq_len, NC, KMAX, sc);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
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
        prm.sc = sc;
        const int gmode = P.a_log ? kDecayLogits : P.scalar_decay ? kDecayScalar : kDecayTile;
        const bool ogate = P.ogate_fused;
        e = P.out_dtype == KDA_DTYPE_BF16
                ? launch_out<__nv_bfloat16>(prm, grid, gmode, ogate, stream)
                : launch_out<float>(prm, grid, gmode, ogate, stream);
    }
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

cudaError_t kda_chain_read_status(unsigned *status) {
    unsigned st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&st, g_kda_chain_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_kda_chain_status, &zero, sizeof(unsigned));
    *status |= st;
    return e;
}

// ---------------------------------------------------------------- kda_prefill_noalloc
//
// The same kernel with its scratch in a fixed array of this library instead of
// memory taken from a pool: for callers that may not allocate device memory
// during a call -- hosts whose own caching allocator owns all of the GPU's memory
// from start-up (a call that allocates outside it can fail or fragment it), and
// latency-bound services that keep allocation off their serving path.  The
// array holds the ring, hand-off words, step table and sequence order of at
// most kNaChains chains, each with at most kNaPairsPerChain (sequence, head)
// pairs, for batches of at most kNaSeqs sequences: about 5 MB, which every
// device that loads the library keeps until the process exits.

namespace {

constexpr int kNaChains = 16;
constexpr int kNaPairsPerChain = 4096;
constexpr int kNaSeqs = 65536;
constexpr size_t kNaRingOff = 0;
constexpr size_t kNaReadyOff = kNaRingOff + (size_t)kNaChains * kRing * kSlotStride;
constexpr size_t kNaProgOff = kNaReadyOff + 256;
constexpr size_t kNaFsOff = kNaProgOff + 256;
constexpr size_t kNaOrderOff = kNaFsOff + ((size_t)kNaChains * (kNaPairsPerChain + 1) * 4 + 255) / 256 * 256;
constexpr size_t kNaCtrlOff = kNaOrderOff + (size_t)kNaSeqs * 4;
constexpr size_t kNaBytes = kNaCtrlOff + 256;
static_assert(kNaChains * kRing * 4 <= 256 && kNaChains * 4 <= 256, "hand-off words fit their blocks");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

// Per device: the SM count, cooperative-launch support and the device address of
// g_noalloc_scratch (cudaGetSymbolAddress with the device current; the host-side
// name of the array is not a device address).  Done once, by the first call on
// the device.
struct NaDev {
    unsigned char *ptr = nullptr;
    int sms = 0;
    bool coop = false;
    cudaError_t err = cudaSuccess;
};

NaDev &noalloc_dev(int dev) {
    static NaDev info[64];
    static std::once_flag once[64];
    std::call_once(once[dev & 63], [dev] {
        NaDev &d = info[dev & 63];
        int coop = 0;
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        d.coop = coop != 0;
        if (d.err == cudaSuccess) {
            void *p = nullptr;
            d.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            d.ptr = static_cast<unsigned char *>(p);
        }
    });
    return info[dev & 63];
}

}  // namespace

// Does the fixed array hold this call, and does the split kernel take it?
bool kda_prefill_noalloc_fits(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const void *out) {
    auto al16 = [](const void *x) { return ((uintptr_t)x & 15u) == 0; };
    if (!(P.dk == 128 && P.dv == 128 && P.in_dtype == KDA_DTYPE_BF16)) return false;
    if (P.N == 0) return true;   // nothing to run
    if (!(al16(q) && al16(k) && al16(v) && (P.scalar_decay || al16(g)) && al16(out))) return false;
    if (P.N > kNaSeqs) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const NaDev &d = noalloc_dev(dev);
    if (d.err != cudaSuccess || !d.coop || d.sms < 2) return false;
    const int64_t pairs = (int64_t)P.N * P.H;
    int nc = chain_count(d.sms, (int)(pairs < (1 << 30) ? pairs : (1 << 30)));
    if (nc > kNaChains) nc = kNaChains;
    return (pairs + nc - 1) / nc <= kNaPairsPerChain;
}

// Launch the split kernel on the fixed array.  Calls no allocation routine.
cudaError_t kda_launch_prefill_noalloc(const kda::Problem &P, const void *q, const void *k,
                                       const void *v, const float *g, const float *beta,
                                       const float *init_state, const int32_t *cu, void *out,
                                       float *final_state, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    NaDev &d = noalloc_dev(dev);
    if (d.err != cudaSuccess) return d.err;
    const int pairs = P.N * P.H;
    const int grid = d.sms;
    int NC = chain_count(grid, pairs);
    if (NC > kNaChains) NC = kNaChains;
    const int KMAX = (pairs + NC - 1) / NC;
    if (KMAX > kNaPairsPerChain || P.N > kNaSeqs) return cudaErrorInvalidValue;
    Scratch sc;
    sc.ring = d.ptr + kNaRingOff;
    sc.ready = reinterpret_cast<uint32_t *>(d.ptr + kNaReadyOff);
    sc.progress = reinterpret_cast<uint32_t *>(d.ptr + kNaProgOff);
    sc.first_step = reinterpret_cast<uint32_t *>(d.ptr + kNaFsOff);
    sc.order = reinterpret_cast<int32_t *>(d.ptr + kNaOrderOff);
    sc.ctrl = reinterpret_cast<uint32_t *>(d.ptr + kNaCtrlOff);
    // the array keeps the last call's contents: the set-up kernel clears the
    // hand-off words and rewrites the step table before the main kernel reads them
    chain_setup_kernel<<<1, 1024, 0, stream>>>(cu, P.N, P.H, (int64_t)P.T, P.seq_len, NC, KMAX, sc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    Params prm = {};
    prm.q = static_cast<const __nv_bfloat16 *>(q);
    prm.k = static_cast<const __nv_bfloat16 *>(k);
    prm.v = static_cast<const __nv_bfloat16 *>(v);
    prm.g = g;
    prm.beta = beta;
    prm.init = init_state;
    prm.cu = cu;
    prm.out = out;
    prm.fin = final_state;
    prm.ckpt_every = 1;
    prm.N = P.N;
    prm.H = P.H;
    prm.total = P.T;
    prm.seq_len = P.seq_len;
    prm.NC = NC;
    prm.KMAX = KMAX;
    prm.sc = sc;
    return P.out_dtype == KDA_DTYPE_BF16 ? launch_out<__nv_bfloat16>(prm, grid, kDecayTile, false, stream)
                                         : launch_out<float>(prm, grid, kDecayTile, false, stream);
}
