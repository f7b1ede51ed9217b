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
// It serves the calls the prefill kernel cannot fuse: the CUDA-core kernel,
// whose CTAs each hold a 32-channel slice of d_v, and an fp32 output or a
// misaligned gate on the tensor-core path.  One warp per (token, head) row;
// HBM-bound (the row is read and written once, the gate read once).

#include "kda_common.cuh"

namespace {

constexpr int kRowsPerBlock = 8;

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

}  // namespace

cudaError_t kda_launch_output_gate(const kda::Problem &P, void *out, cudaStream_t stream) {
    const int64_t rows = (int64_t)P.T * P.H;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    const dim3 block(32 * kRowsPerBlock);
    const bool gbf = P.in_dtype == KDA_DTYPE_BF16, obf = P.out_dtype == KDA_DTYPE_BF16;
    if (gbf && obf)
        kda_output_gate_kernel<<<blocks, block, 0, stream>>>(
            (__nv_bfloat16 *)out, (const __nv_bfloat16 *)P.ogate, P.onorm_w, P.oeps, rows, P.dv);
    else if (gbf)
        kda_output_gate_kernel<<<blocks, block, 0, stream>>>(
            (float *)out, (const __nv_bfloat16 *)P.ogate, P.onorm_w, P.oeps, rows, P.dv);
    else if (obf)
        kda_output_gate_kernel<<<blocks, block, 0, stream>>>(
            (__nv_bfloat16 *)out, (const float *)P.ogate, P.onorm_w, P.oeps, rows, P.dv);
    else
        kda_output_gate_kernel<<<blocks, block, 0, stream>>>(
            (float *)out, (const float *)P.ogate, P.onorm_w, P.oeps, rows, P.dv);
    return cudaGetLastError();
}
