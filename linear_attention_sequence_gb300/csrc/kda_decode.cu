// kda_decode.cu -- single-token KDA update of N x H fixed-size fp32 states.
//
// Per (sequence n, head h), following the delta form of the state update
// ("Understanding Kimi K3's Attention", rewritten update equation) and the
// recurrent implementation in "Hybrid Attention" (section "KDA: don't write
// the same information twice"):
//
//   M = Diag(exp g) S            rows of S are key channels
//   p = M^T k,  r = M^T q        two column reductions over d_k
//   u = beta (v - p)
//   S <- M + k u^T               in place
//   o = S^T q = r + u (k . q)    read after the write
//
// The path is HBM-bound (about 0.9 flop per byte).  One CTA owns one
// (n, h) state: each warp streams whole 512-byte rows with 16-byte
// cache-streaming loads, keeps its rows in registers between the read and the
// write, so each state byte crosses HBM exactly once in each direction.
// The column reductions are warp-local partial sums combined through shared
// memory.

#include "kda_common.cuh"

namespace {

constexpr int kThreads = 256;

template <int D, typename IN_T, typename OUT_T>
__global__ void __launch_bounds__(kThreads, 2)
kda_decode_kernel(const IN_T *__restrict__ q, const IN_T *__restrict__ k,
                  const IN_T *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, float *__restrict__ state,
                  OUT_T *__restrict__ out) {
    constexpr int TPR = D / 4;               // threads per row (one float4 each)
    constexpr int RPP = kThreads / TPR;      // rows covered per pass
    constexpr int PASSES = D / RPP;          // passes over the d_k rows
    static_assert(D % RPP == 0, "row split");

    __shared__ float red_p[RPP][D];
    __shared__ float red_r[RPP][D];
    __shared__ float red_kq[RPP];
    __shared__ float s_u[D];

    const int64_t nh = blockIdx.x;           // n * H + h
    const int t = threadIdx.x;
    const int c4 = t % TPR;                  // column group: columns 4*c4 .. 4*c4+3
    const int rg = t / TPR;                  // row group

    const IN_T *qn = q + nh * D;
    const IN_T *kn = k + nh * D;
    const float *gn = g + nh * D;
    float *S = state + nh * (int64_t)D * D;

    float kr[PASSES], qr[PASSES];
    float4 m[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = rg + p * RPP;
        m[p] = __ldcs(reinterpret_cast<const float4 *>(S + (int64_t)i * D) + c4);
    }
    float kq_part = 0.f;
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), rr = pp;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = rg + p * RPP;
        const float a = expf(gn[i]);
        kr[p] = kda::ld_elem(kn + i);
        qr[p] = kda::ld_elem(qn + i);
        kq_part += kr[p] * qr[p];
        m[p].x *= a; m[p].y *= a; m[p].z *= a; m[p].w *= a;
        pp.x += m[p].x * kr[p]; pp.y += m[p].y * kr[p]; pp.z += m[p].z * kr[p]; pp.w += m[p].w * kr[p];
        rr.x += m[p].x * qr[p]; rr.y += m[p].y * qr[p]; rr.z += m[p].z * qr[p]; rr.w += m[p].w * qr[p];
    }
    *reinterpret_cast<float4 *>(&red_p[rg][4 * c4]) = pp;
    *reinterpret_cast<float4 *>(&red_r[rg][4 * c4]) = rr;
    if (c4 == 0) red_kq[rg] = kq_part;
    __syncthreads();

    if (t < D) {
        const int j = t;
        float ps = 0.f, rs = 0.f, kq = 0.f;
#pragma unroll
        for (int x = 0; x < RPP; ++x) {
            ps += red_p[x][j];
            rs += red_r[x][j];
            kq += red_kq[x];
        }
        const float u = beta[nh] * (kda::ld_elem(v + nh * D + j) - ps);
        s_u[j] = u;
        kda::st_elem(out + nh * D + j, rs + u * kq);
    }
    __syncthreads();

    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * c4]);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = rg + p * RPP;
        float4 s;
        s.x = m[p].x + kr[p] * u4.x;
        s.y = m[p].y + kr[p] * u4.y;
        s.z = m[p].z + kr[p] * u4.z;
        s.w = m[p].w + kr[p] * u4.w;
        __stcs(reinterpret_cast<float4 *>(S + (int64_t)i * D) + c4, s);
    }
}

template <int D, typename IN_T, typename OUT_T>
cudaError_t launch(const kda::Problem &P, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, float *state, void *out,
                   cudaStream_t stream) {
    const int64_t blocks = (int64_t)P.N * P.H;
    if (blocks == 0) return cudaSuccess;
    kda_decode_kernel<D, IN_T, OUT_T><<<(unsigned)blocks, kThreads, 0, stream>>>(
        (const IN_T *)q, (const IN_T *)k, (const IN_T *)v, g, beta, state, (OUT_T *)out);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_dtypes(const kda::Problem &P, const void *q, const void *k, const void *v,
                            const float *g, const float *beta, float *state, void *out,
                            cudaStream_t s) {
    const bool in_bf = P.in_dtype == KDA_DTYPE_BF16, out_bf = P.out_dtype == KDA_DTYPE_BF16;
    if (in_bf && out_bf) return launch<D, __nv_bfloat16, __nv_bfloat16>(P, q, k, v, g, beta, state, out, s);
    if (in_bf) return launch<D, __nv_bfloat16, float>(P, q, k, v, g, beta, state, out, s);
    if (out_bf) return launch<D, float, __nv_bfloat16>(P, q, k, v, g, beta, state, out, s);
    return launch<D, float, float>(P, q, k, v, g, beta, state, out, s);
}

}  // namespace

cudaError_t kda_launch_decode(const kda::Problem &P, const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float *state, void *out,
                              cudaStream_t stream) {
    if (P.dk == 128) return dispatch_dtypes<128>(P, q, k, v, g, beta, state, out, stream);
    return dispatch_dtypes<64>(P, q, k, v, g, beta, state, out, stream);
}
