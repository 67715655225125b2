// Tiled-TMA tensor maps (CUtensorMap) for the pools, per-request contiguous
// regions and prefill queries.  Every map describes rows of 128 16-bit values
// (bf16 or fp16: the copies move bits, so one data type serves both) read as
// boxes of 16 rows x 64 values with 128-byte swizzle (the layout both the
// tcgen05 descriptors and the ldmatrix address math expect).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace pkv {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

bool encode_rows_map(CUtensorMap *m, void *base, long long rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows <= 0) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128 * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *m, const void *q, int rows, int hq) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)hq, (cuuint64_t)rows};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)hq * 128 * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

kv_status pool_tensor_maps(kv_pool *p) {
    if (p->tmaps_ready) return KV_OK;
    if (p->dtype == KV_F32 || p->head_dim != 128) return KV_ERR_UNSUPPORTED;
    const long long rows = (long long)p->num_blocks * p->num_kv_heads * 16;
    if (rows > INT32_MAX) return KV_ERR_UNSUPPORTED;
    if (!encode_rows_map(&p->tmap_k, p->k, rows) || !encode_rows_map(&p->tmap_v, p->v, rows))
        return KV_ERR_CUDA;
    p->tmaps_ready = true;
    return KV_OK;
}

}  // namespace pkv
