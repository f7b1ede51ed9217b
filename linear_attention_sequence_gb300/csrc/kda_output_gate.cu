// kda_output_gate.cu -- the layer's output gate applied in place to a
// prefill's output.
//
// "Inside Kimi K3", section "Sequence mixing: fixed-state KDA alongside
// global MLA": the layer output is W_o [Sigmoid(W_g x_t) . RMSNorm(o~_t)].
// This kernel forms the bracket from o~ (in `out`) and the gate logits
// W_g x_t, with RMSNorm read as the root-mean-square over one head's d_v
// channels, eps inside the root and an optional per-channel weight:
//
//   y[t,h,j] = Sigmoid(gate[t,h,j]) * o~[t,h,j] / sqrt(mean_j o~^2 + eps) * w[j]
//
// It gates every kda_prefill_output_gated call except those of the split and
// two-pass variants (which gate a bf16 output in their epilogue), and it is the
// public kda_output_gate for the other calls' outputs.  HBM-bound: the row is read and
// written once, the gate read once.  The main kernel gives each warp four
// (token, head) rows and each lane d_v / 32 consecutive channels of them, and
// issues all of a warp's loads before its first reduction, so that enough
// bytes are in flight to stream at the HBM rate; rows whose pointers are not
// aligned for those vector accesses take a one-row-per-warp scalar kernel.

#include "kda_common.cuh"

namespace {

constexpr int kRowsPerBlock = 8;   // scalar kernel: one row per warp
constexpr int kWarpsPerBlock = 8;  // vector kernel
constexpr int kRowsPerWarp = 4;

template <typename G_T, typename OUT_T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
kda_output_gate_kernel(OUT_T *__restrict__ out, const G_T *__restrict__ gate,
                       const float *__restrict__ w, float eps, int64_t rows, int dv) {
    const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;   // whole warps only: the row index is warp-uniform
    OUT_T *o = out + row * dv;
    const G_T *gl = gate + row * dv;
    const int per = dv >> 5;   // 2 or 4 channels per lane
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (i < per) {
            x[i] = kda::ld_elem(o + lane + 32 * i);
            ss += x[i] * x[i];
        }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    const float rinv = rsqrtf(ss / (float)dv + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (i < per) {
            const int j = lane + 32 * i;
            const float wj = w ? w[j] : 1.f;
            kda::st_elem(o + j, kda::sigmoid_f(kda::ld_elem(gl + j)) * x[i] * rinv * wj);
        }
}

// PER consecutive elements at p (PER * sizeof(T) bytes, aligned to that size).
template <int PER>
__device__ __forceinline__ void ld_vec(const __nv_bfloat16 *p, float (&x)[PER]) {
    if constexpr (PER == 4) {
        const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p));
        x[0] = __uint_as_float(u.x << 16);
        x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16);
        x[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const uint32_t u = __ldcs(reinterpret_cast<const unsigned int *>(p));
        x[0] = __uint_as_float(u << 16);
        x[1] = __uint_as_float(u & 0xffff0000u);
    }
}
template <int PER>
__device__ __forceinline__ void ld_vec(const float *p, float (&x)[PER]) {
    if constexpr (PER == 4) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        const float2 v = __ldcs(reinterpret_cast<const float2 *>(p));
        x[0] = v.x; x[1] = v.y;
    }
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
template <int PER>
__device__ __forceinline__ void st_vec(__nv_bfloat16 *p, const float (&y)[PER]) {
    if constexpr (PER == 4) __stcs(reinterpret_cast<uint2 *>(p), make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3])));
    else __stcs(reinterpret_cast<unsigned int *>(p), pack_bf16(y[0], y[1]));
}
template <int PER>
__device__ __forceinline__ void st_vec(float *p, const float (&y)[PER]) {
    if constexpr (PER == 4) __stcs(reinterpret_cast<float4 *>(p), make_float4(y[0], y[1], y[2], y[3]));
    else __stcs(reinterpret_cast<float2 *>(p), make_float2(y[0], y[1]));
}

// kRowsPerWarp rows per warp; lane l holds channels [PER l, PER l + PER) of each.
template <typename G_T, typename OUT_T, int PER>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
kda_output_gate_vec_kernel(OUT_T *__restrict__ out, const G_T *__restrict__ gate,
                           const float *__restrict__ w, float eps, int64_t rows) {
    constexpr int DV = 32 * PER;
    const int lane = threadIdx.x & 31;
    const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kRowsPerWarp;
    float x[kRowsPerWarp][PER], gt[kRowsPerWarp][PER];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t row = row0 + rr;
        if (row < rows) {
            ld_vec<PER>(out + row * DV + PER * lane, x[rr]);
            ld_vec<PER>(gate + row * DV + PER * lane, gt[rr]);
        } else {
#pragma unroll
            for (int i = 0; i < PER; ++i) x[rr][i] = gt[rr][i] = 0.f;
        }
    }
    float wv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) wv[i] = w ? w[PER * lane + i] : 1.f;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) ss += x[rr][i] * x[rr][i];
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
        const float rinv = rsqrtf(ss / (float)DV + eps);
        float y[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) y[i] = kda::sigmoid_f(gt[rr][i]) * x[rr][i] * rinv * wv[i];
        const int64_t row = row0 + rr;
        if (row < rows) st_vec<PER>(out + row * DV + PER * lane, y);
    }
}

template <typename G_T, typename OUT_T>
cudaError_t launch_gate(OUT_T *out, const G_T *gate, const float *w, float eps, int64_t rows, int dv,
                        cudaStream_t stream) {
    const size_t vbytes = (size_t)(dv / 32) * sizeof(G_T) < (size_t)(dv / 32) * sizeof(OUT_T)
                              ? (size_t)(dv / 32) * sizeof(OUT_T)
                              : (size_t)(dv / 32) * sizeof(G_T);
    const bool vec = (dv == 64 || dv == 128) && ((uintptr_t)out % vbytes) == 0 &&
                     ((uintptr_t)gate % vbytes) == 0;
    if (vec) {
        const int64_t per_block = (int64_t)kWarpsPerBlock * kRowsPerWarp;
        const unsigned blocks = (unsigned)((rows + per_block - 1) / per_block);
        if (dv == 128)
            kda_output_gate_vec_kernel<G_T, OUT_T, 4><<<blocks, 32 * kWarpsPerBlock, 0, stream>>>(out, gate, w, eps, rows);
        else
            kda_output_gate_vec_kernel<G_T, OUT_T, 2><<<blocks, 32 * kWarpsPerBlock, 0, stream>>>(out, gate, w, eps, rows);
    } else {
        const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
        kda_output_gate_kernel<<<blocks, 32 * kRowsPerBlock, 0, stream>>>(out, gate, w, eps, rows, dv);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t kda_launch_output_gate(const kda::Problem &P, void *out, cudaStream_t stream) {
    const int64_t rows = (int64_t)P.T * P.H;
    if (rows == 0) return cudaSuccess;
    const bool gbf = P.in_dtype == KDA_DTYPE_BF16, obf = P.out_dtype == KDA_DTYPE_BF16;
    if (gbf && obf)
        return launch_gate((__nv_bfloat16 *)out, (const __nv_bfloat16 *)P.ogate, P.onorm_w, P.oeps, rows, P.dv, stream);
    if (gbf)
        return launch_gate((float *)out, (const __nv_bfloat16 *)P.ogate, P.onorm_w, P.oeps, rows, P.dv, stream);
    if (obf)
        return launch_gate((__nv_bfloat16 *)out, (const float *)P.ogate, P.onorm_w, P.oeps, rows, P.dv, stream);
    return launch_gate((float *)out, (const float *)P.ogate, P.onorm_w, P.oeps, rows, P.dv, stream);
}
