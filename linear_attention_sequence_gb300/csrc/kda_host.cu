// kda_host.cu -- host helpers shared by the kernels: TMA tensor maps and the
// device status words.

#include <mutex>

#include "kda_common.cuh"
#include "kda_chunk_ops.cuh"

namespace {

constexpr int C = 32;    // tokens per chunk (the TMA box height)
constexpr int D = 128;   // d_k = d_v of the tensor-core kernels

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

// 3-D view of a [T, H, D] tensor: (element within a 128-byte segment, token,
// segment index along the H*D row); box = one head's segments for C tokens,
// stored segment by segment (C rows of 128 bytes each), 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int64_t T,
              int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int seg = 128 / esize, nseg = D / seg;
    const cuuint64_t dims[3] = {(cuuint64_t)seg, (cuuint64_t)T, (cuuint64_t)H * nseg};
    const cuuint64_t strides[2] = {(cuuint64_t)H * D * esize, 128};
    const cuuint32_t box[3] = {(cuuint32_t)seg, (cuuint32_t)C, (cuuint32_t)nseg};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool kda_tma_available() { return encode_fn() != nullptr; }

// The 3-D TMA view of a [T, H, 128] tensor (box: one head's 128-byte segments
// for 32 tokens, 128-byte swizzle), for the kernels that load chunk tiles.
bool kda_make_tile_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                       int64_t T, int H) {
    return make_map(m, base, dt, esize, T, H);
}

// The TMA view of an fp32 state array [rows, 128] (rows = states x 128 key
// channels): box = 128 rows x 32 columns, 128-byte swizzle, so that four boxes
// give a 128-row K-major SW128 operand (rows = key channel, K = value index).
bool kda_make_state_map(CUtensorMap *m, const float *base, int64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Wait for the stream, then read and clear the status words of every kernel
// family (ORed into *status): bounded waits that gave up, and the backward's
// missing chunk-state rows.
cudaError_t kda_read_device_status(cudaStream_t stream, unsigned *status) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = kda_tc_read_status(status);
    if (e == cudaSuccess) e = kda_chain_read_status(status);
    if (e == cudaSuccess) e = kda_2pass_read_status(status);
    if (e == cudaSuccess) e = kda_bwd_read_status(status);
    if (e == cudaSuccess) e = kda_bwdtc_read_status(status);
    return e;
}
