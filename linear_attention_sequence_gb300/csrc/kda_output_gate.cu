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
// written once, the gate read once.  The main kernel gives each warp eight
// (token, head) rows, half a warp per row and d_v / 16 consecutive channels per
// lane (16-byte accesses for bf16 at d_v = 128), and issues all of a warp's loads
// before its first reduction, so that enough bytes are in flight to stream at the
// HBM rate; rows whose pointers are not aligned for those vector accesses take a
// one-row-per-warp scalar kernel.

#include "kda_common.cuh"

namespace {

// The kernels are launched as programmatic dependents of the previous kernel in
// the stream (normally the prefill that wrote `out`): their blocks may be
// scheduled while that kernel drains, and wait here until it has completed and
// its writes are visible.  Launched without that attribute, this is a no-op.
__device__ __forceinline__ void wait_for_producer() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr int kRowsPerBlock = 8;   // scalar kernel: one row per warp
constexpr int kWarpsPerBlock = 8;  // vector kernel
constexpr int kRowsPerWarp = 8;

template <typename G_T, typename OUT_T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
kda_output_gate_kernel(OUT_T *__restrict__ out, const G_T *__restrict__ gate,
                       const float *__restrict__ w, float eps, int64_t rows, int dv) {
    wait_for_producer();
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

// EPL consecutive elements of one row, as loaded (streaming: the row is read once
// and written once): bf16 as 8 or 16 bytes, fp32 as one or two 16-byte vectors.
template <typename T, int EPL> struct Raw;
template <> struct Raw<__nv_bfloat16, 8> { uint4 u; };
template <> struct Raw<__nv_bfloat16, 4> { uint2 u; };
template <> struct Raw<float, 8> { float4 a, b; };
template <> struct Raw<float, 4> { float4 a; };

__device__ __forceinline__ void ld_raw(const __nv_bfloat16 *p, Raw<__nv_bfloat16, 8> &r) { r.u = __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void ld_raw(const __nv_bfloat16 *p, Raw<__nv_bfloat16, 4> &r) { r.u = __ldcs(reinterpret_cast<const uint2 *>(p)); }
__device__ __forceinline__ void ld_raw(const float *p, Raw<float, 8> &r) {
    r.a = __ldcs(reinterpret_cast<const float4 *>(p));
    r.b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
}
__device__ __forceinline__ void ld_raw(const float *p, Raw<float, 4> &r) { r.a = __ldcs(reinterpret_cast<const float4 *>(p)); }
template <typename T, int EPL> __device__ __forceinline__ void zero_raw(Raw<T, EPL> &r) { r = Raw<T, EPL>{}; }

__device__ __forceinline__ void bf16x2(uint32_t u, float &lo, float &hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}
__device__ __forceinline__ void unpack(const Raw<__nv_bfloat16, 8> &r, float (&x)[8]) {
    bf16x2(r.u.x, x[0], x[1]); bf16x2(r.u.y, x[2], x[3]); bf16x2(r.u.z, x[4], x[5]); bf16x2(r.u.w, x[6], x[7]);
}
__device__ __forceinline__ void unpack(const Raw<__nv_bfloat16, 4> &r, float (&x)[4]) {
    bf16x2(r.u.x, x[0], x[1]); bf16x2(r.u.y, x[2], x[3]);
}
__device__ __forceinline__ void unpack(const Raw<float, 8> &r, float (&x)[8]) {
    x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w; x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
}
__device__ __forceinline__ void unpack(const Raw<float, 4> &r, float (&x)[4]) {
    x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w;
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
__device__ __forceinline__ void st_vec(__nv_bfloat16 *p, const float (&y)[8]) {
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                                                    pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7])));
}
__device__ __forceinline__ void st_vec(__nv_bfloat16 *p, const float (&y)[4]) {
    __stcs(reinterpret_cast<uint2 *>(p), make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3])));
}
__device__ __forceinline__ void st_vec(float *p, const float (&y)[8]) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4(y[0], y[1], y[2], y[3]));
    __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(y[4], y[5], y[6], y[7]));
}
__device__ __forceinline__ void st_vec(float *p, const float (&y)[4]) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4(y[0], y[1], y[2], y[3]));
}

// Half a warp per row: lane l holds channels [EPL (l % 16), EPL (l % 16) + EPL) of
// row 2 i + l / 16 of its group of kRowsPerWarp rows.  Every load of the group is
// issued before the first reduction (four shuffles inside the half-warp).
template <typename G_T, typename OUT_T, int EPL>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
kda_output_gate_vec_kernel(OUT_T *__restrict__ out, const G_T *__restrict__ gate,
                           const float *__restrict__ w, float eps, int64_t rows) {
    constexpr int DV = 16 * EPL, NP = kRowsPerWarp / 2;
    wait_for_producer();
    const int lane = threadIdx.x & 31, hl = lane & 15, hr = lane >> 4;
    const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kRowsPerWarp;
    Raw<OUT_T, EPL> ro[NP];
    Raw<G_T, EPL> rg[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const int64_t row = row0 + 2 * i + hr;
        if (row < rows) {
            ld_raw(out + row * DV + EPL * hl, ro[i]);
            ld_raw(gate + row * DV + EPL * hl, rg[i]);
        } else {
            zero_raw(ro[i]);
            zero_raw(rg[i]);
        }
    }
    float wv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) wv[e] = w ? w[EPL * hl + e] : 1.f;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        float x[EPL], gt[EPL];
        unpack(ro[i], x);
        unpack(rg[i], gt);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) ss += x[e] * x[e];
#pragma unroll
        for (int sh = 8; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
        const float rinv = rsqrtf(ss / (float)DV + eps);
        float y[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) y[e] = kda::sigmoid_f(gt[e]) * x[e] * rinv * wv[e];
        const int64_t row = row0 + 2 * i + hr;
        if (row < rows) st_vec(out + row * DV + EPL * hl, y);
    }
}

template <typename G_T, typename OUT_T>
cudaError_t launch_gate(OUT_T *out, const G_T *gate, const float *w, float eps, int64_t rows, int dv,
                        cudaStream_t stream) {
    // the vector kernel's accesses are 16-byte (bf16 at d_v = 128, fp32) or 8-byte
    // (bf16 at d_v = 64) aligned when the row starts are
    auto aligned = [dv](const void *p, size_t elem) {
        const size_t a = (size_t)(dv / 16) * elem < 16 ? (size_t)(dv / 16) * elem : 16;
        return ((uintptr_t)p % a) == 0;
    };
    const bool vec = (dv == 64 || dv == 128) && aligned(out, sizeof(OUT_T)) && aligned(gate, sizeof(G_T)) &&
                     (w == nullptr || ((uintptr_t)w % 4) == 0);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (vec) {
        const int64_t per_block = (int64_t)kWarpsPerBlock * kRowsPerWarp;
        cfg.gridDim = dim3((unsigned)((rows + per_block - 1) / per_block));
        cfg.blockDim = dim3(32 * kWarpsPerBlock);
        if (dv == 128)
            return cudaLaunchKernelEx(&cfg, kda_output_gate_vec_kernel<G_T, OUT_T, 8>, out, gate, w, eps, rows);
        return cudaLaunchKernelEx(&cfg, kda_output_gate_vec_kernel<G_T, OUT_T, 4>, out, gate, w, eps, rows);
    }
    cfg.gridDim = dim3((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock));
    cfg.blockDim = dim3(32 * kRowsPerBlock);
    return cudaLaunchKernelEx(&cfg, kda_output_gate_kernel<G_T, OUT_T>, out, gate, w, eps, rows, dv);
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
