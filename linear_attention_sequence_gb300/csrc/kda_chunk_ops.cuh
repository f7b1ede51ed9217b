// kda_chunk_ops.cuh -- pieces of the chunk algebra shared by the kernels that
// make the intra-chunk products of many chunks at once (sm_103a): K-major SW128
// operand offsets and the 32 x 32 triangular solve T diag(beta).
#pragma once

#include "sm100_ptx.cuh"

namespace kda_chunk {

using namespace sm100;

// Element (row, k) of a K-major SW128 operand with `rows` rows per 32-element K-block.
__device__ __forceinline__ uint32_t sw_off(int rows, int row, int k) {
    return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) +
                      ((k & 3) << 2));
}
__device__ __forceinline__ void st_f(unsigned char *p, uint32_t off, float x) {
    *reinterpret_cast<float *>(p + off) = x;
}
// T diag(beta) of one chunk from its Gram rows.  Lane r holds d[i] = k~_r . k^_i
// (i = 0..31) and beta_r; the result goes to `tmat` as a K-major SW128 tf32
// operand (row r, element i).  T = (I + A)^{-1} with A[r][i] = beta_r d[i] for
// i < r, by 16 x 16 blocks: the diagonal blocks T11 (lanes 0-15) and T22 (lanes
// 16-31) by forward substitution, one column per lane, then T21 = -T22 (A21 T11).
__device__ __forceinline__ void solve_tbeta(const float (&d)[32], float br, int lane,
                                            unsigned char *tmat, float (*akkT)[32],
                                            float (*tsc)[16][20]) {
#pragma unroll
    for (int m = 0; m < 32; ++m) akkT[m][lane] = m < lane ? br * d[m] : 0.f;
    __syncwarp();
    const int hb = lane >> 4, jj = lane & 15, b0 = 16 * hb;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = i == jj ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
        const float xm = x[m];
        const float4 *row = reinterpret_cast<const float4 *>(&akkT[b0 + m][b0]);
#pragma unroll
        for (int q4 = (m + 1) >> 2; q4 < 4; ++q4) {
            const float4 a4 = row[q4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (4 * q4 + e > m) x[4 * q4 + e] -= av[e] * xm;
        }
    }
    if (hb == 0) {
#pragma unroll
        for (int k = 0; k < 16; ++k) tsc[0][k][jj] = x[k];
    } else {
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4)
            *reinterpret_cast<float4 *>(&tsc[1][jj][4 * i4]) =
                make_float4(x[4 * i4], x[4 * i4 + 1], x[4 * i4 + 2], x[4 * i4 + 3]);
    }
    __syncwarp();
    float mm[8];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) mm[r8] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float tk = tsc[0][k][jj];
        const float4 a0 = *reinterpret_cast<const float4 *>(&akkT[k][16 + 8 * hb]);
        const float4 a1 = *reinterpret_cast<const float4 *>(&akkT[k][20 + 8 * hb]);
        mm[0] += a0.x * tk; mm[1] += a0.y * tk; mm[2] += a0.z * tk; mm[3] += a0.w * tk;
        mm[4] += a1.x * tk; mm[5] += a1.y * tk; mm[6] += a1.z * tk; mm[7] += a1.w * tk;
    }
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) tsc[2][8 * hb + r8][jj] = mm[r8];
    __syncwarp();
    float t21[8];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) t21[r8] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float mk = tsc[2][k][jj];
        const float4 c0 = *reinterpret_cast<const float4 *>(&tsc[1][k][8 * hb]);
        const float4 c1 = *reinterpret_cast<const float4 *>(&tsc[1][k][8 * hb + 4]);
        t21[0] -= c0.x * mk; t21[1] -= c0.y * mk; t21[2] -= c0.z * mk; t21[3] -= c0.w * mk;
        t21[4] -= c1.x * mk; t21[5] -= c1.y * mk; t21[6] -= c1.z * mk; t21[7] -= c1.w * mk;
    }
    const float bd = __shfl_sync(0xffffffffu, br, b0 + jj);
    const float bl = __shfl_sync(0xffffffffu, br, jj);
#pragma unroll
    for (int i = 0; i < 16; ++i) st_f(tmat, sw_off(32, b0 + i, b0 + jj), to_tf32(x[i] * bd));
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) st_f(tmat, sw_off(32, 16 + 8 * hb + r8, jj), to_tf32(t21[r8] * bl));
#pragma unroll
    for (int e = 0; e < 8; ++e) {   // the block T12 (rows 0-15, columns 16-31) is zero
        const int idx = 8 * lane + e;
        st_f(tmat, sw_off(32, idx >> 4, 16 + (idx & 15)), 0.f);
    }
}


// The same blocked solve returning T = (I + A)^{-1} itself (fp32, row r, column
// i of `tout`, rows of `ld` floats) instead of T diag(beta).
__device__ __forceinline__ void solve_t(const float (&d)[32], float br, int lane, float *tout, int ld,
                                        float (*akkT)[32], float (*tsc)[16][20]) {
#pragma unroll
    for (int m = 0; m < 32; ++m) akkT[m][lane] = m < lane ? br * d[m] : 0.f;
    __syncwarp();
    const int hb = lane >> 4, jj = lane & 15, b0 = 16 * hb;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = i == jj ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
        const float xm = x[m];
        const float4 *row = reinterpret_cast<const float4 *>(&akkT[b0 + m][b0]);
#pragma unroll
        for (int q4 = (m + 1) >> 2; q4 < 4; ++q4) {
            const float4 a4 = row[q4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (4 * q4 + e > m) x[4 * q4 + e] -= av[e] * xm;
        }
    }
    if (hb == 0) {
#pragma unroll
        for (int k = 0; k < 16; ++k) tsc[0][k][jj] = x[k];
    } else {
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4)
            *reinterpret_cast<float4 *>(&tsc[1][jj][4 * i4]) =
                make_float4(x[4 * i4], x[4 * i4 + 1], x[4 * i4 + 2], x[4 * i4 + 3]);
    }
    __syncwarp();
    float mm[8];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) mm[r8] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float tk = tsc[0][k][jj];
        const float4 a0 = *reinterpret_cast<const float4 *>(&akkT[k][16 + 8 * hb]);
        const float4 a1 = *reinterpret_cast<const float4 *>(&akkT[k][20 + 8 * hb]);
        mm[0] += a0.x * tk; mm[1] += a0.y * tk; mm[2] += a0.z * tk; mm[3] += a0.w * tk;
        mm[4] += a1.x * tk; mm[5] += a1.y * tk; mm[6] += a1.z * tk; mm[7] += a1.w * tk;
    }
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) tsc[2][8 * hb + r8][jj] = mm[r8];
    __syncwarp();
    float t21[8];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) t21[r8] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float mk = tsc[2][k][jj];
        const float4 c0 = *reinterpret_cast<const float4 *>(&tsc[1][k][8 * hb]);
        const float4 c1 = *reinterpret_cast<const float4 *>(&tsc[1][k][8 * hb + 4]);
        t21[0] -= c0.x * mk; t21[1] -= c0.y * mk; t21[2] -= c0.z * mk; t21[3] -= c0.w * mk;
        t21[4] -= c1.x * mk; t21[5] -= c1.y * mk; t21[6] -= c1.z * mk; t21[7] -= c1.w * mk;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) tout[(b0 + i) * ld + b0 + jj] = x[i];
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) tout[(16 + 8 * hb + r8) * ld + jj] = t21[r8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {   // the block T12 (rows 0-15, columns 16-31) is zero
        const int idx = 8 * lane + e;
        tout[(idx >> 4) * ld + 16 + (idx & 15)] = 0.f;
    }
}

}  // namespace kda_chunk
