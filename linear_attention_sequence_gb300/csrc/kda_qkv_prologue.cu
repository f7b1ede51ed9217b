// kda_qkv_prologue.cu -- q, k and v from their projections: the short causal
// convolution, Swish, and (q, k) the L2 normalisation.
//
// "Understanding Kimi K3's Attention", symbol table: q_t, k_t =
// L2Norm(Swish(ShortConv(W_{q/k} x_t))) and v_t = Swish(ShortConv(W_v x_t));
// "Inside Kimi K3", section "Sequence mixing: fixed-state KDA alongside global
// MLA": the convolution has width 4; "Hybrid Attention", section "KDA: don't
// write the same information twice": it is causal.  Read as a per-channel
// (depthwise) convolution over the tokens of one sequence, without bias:
//
//   c[t,h,j] = sum_{i=0..3} w[h,j,3-i] x[t-i,h,j]   (inputs before the sequence
//              start come from the carried conv state, else they are 0)
//   y = c Sigmoid(c);   q, k: y / sqrt(sum_j y^2 + eps) over one head's d channels;  v: y
//
// The projections W x stay with the caller.  HBM-bound: every input row is read
// once from DRAM and every output row written once.
//
// Work split.  One warp takes 16 consecutive tokens of one (stream, head) row
// block; lane l holds channels 4l..4l+3 (d = 128) or 2l, 2l+1 (d = 64), so a
// row is one coalesced 256- or 512-byte access.  The warp loads its 16 rows
// and the 3 rows before them up front (19 independent loads in flight), then
// convolves, applies Swish and, for q and k, reduces the row's sum of squares
// across the warp.  The three earlier rows are read again by the warp of the
// previous tile; they come from L2.  A tile that lies inside one sequence
// (nearly all of them) takes a branch-free path that works on 8 tokens at a
// time with packed fp32x2 arithmetic and one reduce-scatter of the 8 row sums
// (17 shuffles instead of 40); tiles that meet a sequence start take a general
// path with the same arithmetic, one token at a time.  A second, small kernel
// writes the conv state out: the last three inputs of every sequence.

#include "kda_common.cuh"

namespace {

constexpr int kTok = 16;          // tokens per warp
constexpr int kWarps = 4;         // warps per block; 4 blocks an SM with bf16 inputs, 3 with fp32
constexpr int kHalo = 3;          // width - 1

struct PrologueArgs {
    const void *x0, *x1, *x2;     // projections of q, k, v: [T, H, d], in_dtype
    void *y0, *y1, *y2;           // q, k, v: [T, H, d], out_dtype
    const float *w;               // [3, H, d, 4]
    const float *cin;             // [N, 3, 3, H, d] or nullptr (zeros)
    const int32_t *cu;            // [N + 1] or nullptr (N equal sequences)
    int64_t T, seq_len;
    int H, N;
    float eps;
};

// ---------------------------------------------------------------------------
// Channel pairs.  The arithmetic runs on two channels at a time with the packed
// fp32 instructions of sm_100-class parts (fma/mul/add .rn.f32x2: each half is
// an ordinary IEEE operation, so the results are those of scalar code).
// ---------------------------------------------------------------------------
typedef unsigned long long u64;

__device__ __forceinline__ u64 pk2(float a, float b) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float lo2(u64 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(u64 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Swish of a pair: c Sigmoid(c) = c / (1 + e^{-c}), with e^{-c} = 2^{-c log2 e}.
// Where the power overflows (c below about -88) the reciprocal of +inf is +0
// and the result is the limit, 0.
__device__ __forceinline__ u64 swish2(u64 c) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    const u64 m = mul2(c, pk2(kNegLog2e, kNegLog2e));
    const u64 den = add2(pk2(ex2_approx(lo2(m)), ex2_approx(hi2(m))), pk2(1.f, 1.f));
    return mul2(c, pk2(rcp_approx(lo2(den)), rcp_approx(hi2(den))));
}

// A row slice as loaded, kept packed until it is used (bf16 stays two
// values a register, which halves the registers of the 19 rows in flight).
template <typename IN_T, int PER> struct Raw;
template <> struct Raw<float, 4> { float4 v; };
template <> struct Raw<float, 2> { float2 v; };
template <> struct Raw<__nv_bfloat16, 4> { uint2 v; };
template <> struct Raw<__nv_bfloat16, 2> { uint32_t v; };

template <typename IN_T, int PER>
__device__ __forceinline__ void load_raw(const IN_T *p, Raw<IN_T, PER> &r) {
    r.v = *reinterpret_cast<const decltype(r.v) *>(p);
}
template <typename IN_T, int PER>
__device__ __forceinline__ void zero_raw(Raw<IN_T, PER> &r) {
    if constexpr (sizeof(r.v) == 16) r.v = make_float4(0.f, 0.f, 0.f, 0.f);
    else if constexpr (sizeof(r.v) == 8 && sizeof(IN_T) == 4) r.v = make_float2(0.f, 0.f);
    else if constexpr (sizeof(r.v) == 8) r.v = make_uint2(0u, 0u);
    else r.v = 0u;
}
// bf16 pair (low half: the lower channel) -> fp32 pair: a bf16 is the top half of an fp32
__device__ __forceinline__ u64 bf16x2_to_pair(uint32_t u) {
    return pk2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
template <typename IN_T, int PER>
__device__ __forceinline__ void to_pairs(const Raw<IN_T, PER> &r, u64 (&x)[PER / 2]) {
    if constexpr (sizeof(IN_T) == 4 && PER == 4) {
        x[0] = pk2(r.v.x, r.v.y);
        x[1] = pk2(r.v.z, r.v.w);
    } else if constexpr (sizeof(IN_T) == 4) {
        x[0] = pk2(r.v.x, r.v.y);
    } else if constexpr (PER == 4) {
        x[0] = bf16x2_to_pair(r.v.x);
        x[1] = bf16x2_to_pair(r.v.y);
    } else {
        x[0] = bf16x2_to_pair(r.v);
    }
}
// PER consecutive fp32 values of a carried conv state, as pairs
template <int PER>
__device__ __forceinline__ void load_state_pairs(const float *p, u64 (&x)[PER / 2]) {
    if constexpr (PER == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        x[0] = pk2(a.x, a.y);
        x[1] = pk2(a.z, a.w);
    } else {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        x[0] = pk2(a.x, a.y);
    }
}

template <int NP>
__device__ __forceinline__ void store_pairs(float *p, const u64 (&o)[NP]) {
    if constexpr (NP == 2)
        *reinterpret_cast<float4 *>(p) = make_float4(lo2(o[0]), hi2(o[0]), lo2(o[1]), hi2(o[1]));
    else
        *reinterpret_cast<float2 *>(p) = make_float2(lo2(o[0]), hi2(o[0]));
}
template <int NP>
__device__ __forceinline__ void store_pairs(__nv_bfloat16 *p, const u64 (&o)[NP]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(lo2(o[0]), hi2(o[0]));
    if constexpr (NP == 2) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo2(o[1]), hi2(o[1]));
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&a);
        u.y = *reinterpret_cast<const uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = u;
    } else {
        *reinterpret_cast<__nv_bfloat162 *>(p) = a;
    }
}

// One token of one lane: the convolution of its channels over four rows
// (oldest first), Swish, and the lane's part of the row's sum of squares.
// Both code paths below go through this one routine, so a token gives the same
// bits whichever path takes it.
template <int NP>
__device__ __forceinline__ float token(const u64 (&w)[NP][4], const u64 (&x0)[NP],
                                       const u64 (&x1)[NP], const u64 (&x2)[NP],
                                       const u64 (&x3)[NP], u64 (&o)[NP]) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        u64 c = mul2(w[p][0], x0[p]);
        c = fma2(w[p][1], x1[p], c);
        c = fma2(w[p][2], x2[p], c);
        c = fma2(w[p][3], x3[p], c);
        o[p] = swish2(c);
    }
    u64 s2 = mul2(o[0], o[0]);
#pragma unroll
    for (int p = 1; p < NP; ++p) s2 = fma2(o[p], o[p], s2);
    return lo2(s2) + hi2(s2);
}

__device__ __forceinline__ int64_t clamp_cu(const int32_t *cu, int n, int64_t T) {
    const int64_t x = cu[n];
    return x < 0 ? 0 : (x > T ? T : x);
}

// The sequence that holds token t and its bounds: with cu, the last n whose
// start is <= t (so empty sequences are skipped); the bounds are clamped like
// everywhere else, so a malformed array never leads to an out-of-range access.
__device__ __forceinline__ void find_seq(const PrologueArgs &a, int64_t t, int &n, int64_t &start,
                                         int64_t &end) {
    if (a.cu) {
        int lo = 0, hi = a.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (clamp_cu(a.cu, mid, a.T) <= t) lo = mid; else hi = mid - 1;
        }
        n = lo;
        start = clamp_cu(a.cu, n, a.T);
        end = clamp_cu(a.cu, n + 1, a.T);
        if (end < start) end = start;
    } else {
        n = (int)(t / a.seq_len);
        start = (int64_t)n * a.seq_len;
        end = start + a.seq_len;
    }
}

template <typename IN_T, typename OUT_T, int PER>
__global__ void __launch_bounds__(32 * kWarps, sizeof(IN_T) == 2 ? 4 : 3)
kda_qkv_prologue_kernel(const PrologueArgs a) {
    constexpr int D = 32 * PER, NP = PER / 2;
    const int64_t wid = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int SH = 3 * a.H;
    const int64_t tile = wid / SH;
    const int64_t t0 = tile * kTok;
    if (t0 >= a.T) return;   // warp-uniform
    const int sh = (int)(wid - tile * SH);
    const int s = sh / a.H, h = sh - s * a.H;
    const IN_T *x = static_cast<const IN_T *>(s == 0 ? a.x0 : s == 1 ? a.x1 : a.x2);
    OUT_T *y = static_cast<OUT_T *>(s == 0 ? a.y0 : s == 1 ? a.y1 : a.y2);
    const int64_t rs = (int64_t)a.H * D;            // elements between consecutive tokens
    const int64_t col = (int64_t)h * D + lane * PER; // this lane's first channel in a row
    const int64_t tend = t0 + kTok < a.T ? t0 + kTok : a.T;

    // rows t0-3 .. tend-1 (rows outside [0, T) are not read)
    Raw<IN_T, PER> xr[kTok + kHalo];
#pragma unroll
    for (int r = 0; r < kTok + kHalo; ++r) {
        const int64_t t = t0 - kHalo + r;
        if (t >= 0 && t < tend) load_raw<IN_T, PER>(x + t * rs + col, xr[r]);
        else zero_raw<IN_T, PER>(xr[r]);
    }
    // taps of this lane's channels as pairs: w2[p][tap] = (w[2p][tap], w[2p+1][tap])
    u64 w2[NP][4];
    {
        const float4 *wp = reinterpret_cast<const float4 *>(a.w + (((int64_t)s * a.H + h) * D + lane * PER) * 4);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const float4 e0 = wp[2 * p], e1 = wp[2 * p + 1];
            w2[p][0] = pk2(e0.x, e1.x);
            w2[p][1] = pk2(e0.y, e1.y);
            w2[p][2] = pk2(e0.z, e1.z);
            w2[p][3] = pk2(e0.w, e1.w);
        }
    }
    const bool normed = s < 2;   // q and k are L2-normalised, v is not
    int n;
    int64_t sa, sb;
    find_seq(a, t0, n, sa, sb);

    if (t0 + kTok <= a.T && t0 - kHalo >= sa && t0 + kTok <= sb) {
        // Fast path: the tile and the three rows before it lie inside one
        // sequence, so every tap reads a loaded row and there is no branch.
        // Two halves of 8 tokens; the tokens of a half interleave.
        constexpr int kH = kTok / 2;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            u64 xf[kH + kHalo][NP];
#pragma unroll
            for (int r = 0; r < kH + kHalo; ++r) to_pairs<IN_T, PER>(xr[half * kH + r], xf[r]);
            u64 o[kH][NP];
            float ss[kH];
#pragma unroll
            for (int i = 0; i < kH; ++i) ss[i] = token<NP>(w2, xf[i], xf[i + 1], xf[i + 2], xf[i + 3], o[i]);
            if (normed) {
                // Row sums of the 8 tokens by reduce-scatter: at each of the
                // first three exchanges a lane keeps half of its tokens and sends
                // the other half, so lane L ends with token 4 b4 + 2 b3 + b2
                // (bits of L).  Every partial is own + partner, the same tree as
                // a butterfly on one token.
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
                float t4[4], t2[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float keep = b4 ? ss[i + 4] : ss[i], send = b4 ? ss[i] : ss[i + 4];
                    t4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float keep = b3 ? t4[i + 2] : t4[i], send = b3 ? t4[i] : t4[i + 2];
                    t2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                float tot;
                {
                    const float keep = b2 ? t2[1] : t2[0], send = b2 ? t2[0] : t2[1];
                    tot = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                tot += __shfl_xor_sync(0xffffffffu, tot, 2);
                tot += __shfl_xor_sync(0xffffffffu, tot, 1);
                const float inv = rsqrtf(tot + a.eps);
#pragma unroll
                for (int i = 0; i < kH; ++i) {
                    const int src = ((i >> 2) & 1) << 4 | ((i >> 1) & 1) << 3 | (i & 1) << 2;
                    const float iv = __shfl_sync(0xffffffffu, inv, src);
                    const u64 iv2 = pk2(iv, iv);
#pragma unroll
                    for (int p = 0; p < NP; ++p) o[i][p] = mul2(o[i][p], iv2);
                }
            }
#pragma unroll
            for (int i = 0; i < kH; ++i) store_pairs<NP>(y + (t0 + half * kH + i) * rs + col, o[i]);
        }
        return;
    }

    // General path: a sequence starts inside the tile or its three earlier
    // rows, or the tile is the last, partial one.
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
        const int64_t t = t0 + i;
        if (t >= tend) break;   // warp-uniform
        if (t >= sb) find_seq(a, t, n, sa, sb);
        const int64_t st = sa > t ? t : sa;   // start of t's sequence (never after t)
        u64 xt[4][NP];
#pragma unroll
        for (int tap = 0; tap < 4; ++tap) {
            const int64_t u = t - 3 + tap;
            if (u >= st) {
                to_pairs<IN_T, PER>(xr[i + tap], xt[tap]);
            } else if (a.cin) {
                // u - st + 3 is in 0..2: u >= t - 3 >= st - 3
                load_state_pairs<PER>(a.cin + ((((int64_t)n * 3 + s) * 3 + (u - st + 3)) * a.H) * D + col,
                                      xt[tap]);
            } else {
#pragma unroll
                for (int p = 0; p < NP; ++p) xt[tap][p] = 0ull;
            }
        }
        u64 o[NP];
        float ss = token<NP>(w2, xt[0], xt[1], xt[2], xt[3], o);
        if (normed) {
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float inv = rsqrtf(ss + a.eps);
            const u64 iv2 = pk2(inv, inv);
#pragma unroll
            for (int p = 0; p < NP; ++p) o[p] = mul2(o[p], iv2);
        }
        store_pairs<NP>(y + t * rs + col, o);
    }
}

// conv_state_out[n, s, p, h, j] = input p of the last three of sequence n
// (entry 0 the oldest); positions before the sequence start come from the
// state in (or are 0).  One thread per element.
template <typename IN_T>
__global__ void __launch_bounds__(256)
kda_conv_state_kernel(const PrologueArgs a, float *__restrict__ cout, int d) {
    const int64_t per_seq = (int64_t)9 * a.H * d;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= per_seq * a.N) return;
    const int n = (int)(idx / per_seq);
    int64_t r = idx - (int64_t)n * per_seq;
    const int s = (int)(r / (3 * (int64_t)a.H * d));
    r -= (int64_t)s * 3 * a.H * d;
    const int p = (int)(r / ((int64_t)a.H * d));
    const int64_t hj = r - (int64_t)p * a.H * d;
    int64_t sa, sb;
    kda::seq_bounds(a.cu, n, a.T, a.seq_len, sa, sb);
    const int64_t u = sb - 3 + p;
    float val = 0.f;
    if (u >= sa) {
        const IN_T *x = static_cast<const IN_T *>(s == 0 ? a.x0 : s == 1 ? a.x1 : a.x2);
        val = kda::ld_elem(x + u * a.H * d + hj);
    } else if (a.cin) {
        // u - sa + 3 = p + length is in 0..2 here
        val = a.cin[(((int64_t)n * 3 + s) * 3 + (u - sa + 3)) * a.H * d + hj];
    }
    cout[idx] = val;
}

template <typename IN_T, typename OUT_T>
cudaError_t launch_typed(const PrologueArgs &a, int d, float *cout, cudaStream_t stream) {
    if (a.T > 0) {
        const int64_t warps = (a.T + kTok - 1) / kTok * 3 * a.H;
        const unsigned blocks = (unsigned)((warps + kWarps - 1) / kWarps);
        if (d == 128)
            kda_qkv_prologue_kernel<IN_T, OUT_T, 4><<<blocks, 32 * kWarps, 0, stream>>>(a);
        else
            kda_qkv_prologue_kernel<IN_T, OUT_T, 2><<<blocks, 32 * kWarps, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (cout && a.N > 0) {
        const int64_t elems = (int64_t)a.N * 9 * a.H * d;
        const unsigned blocks = (unsigned)((elems + 255) / 256);
        kda_conv_state_kernel<IN_T><<<blocks, 256, 0, stream>>>(a, cout, d);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t kda_launch_qkv_prologue(const kda::Problem &P, const void *xq, const void *xk,
                                    const void *xv, const float *w, const float *cin,
                                    const int32_t *cu, void *q, void *k, void *v, float *cout,
                                    float eps, cudaStream_t stream) {
    PrologueArgs a;
    a.x0 = xq; a.x1 = xk; a.x2 = xv;
    a.y0 = q; a.y1 = k; a.y2 = v;
    a.w = w;
    a.cin = cin;
    a.cu = cu;
    a.T = P.T;
    a.seq_len = P.seq_len;
    a.H = P.H;
    a.N = P.N;
    a.eps = eps;
    const bool ib = P.in_dtype == KDA_DTYPE_BF16, ob = P.out_dtype == KDA_DTYPE_BF16;
    if (ib && ob) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, P.dk, cout, stream);
    if (ib) return launch_typed<__nv_bfloat16, float>(a, P.dk, cout, stream);
    if (ob) return launch_typed<float, __nv_bfloat16>(a, P.dk, cout, stream);
    return launch_typed<float, float>(a, P.dk, cout, stream);
}
