// fa_tmap.h -- host-side TMA tensor-map construction.  The driver entry
// point cuTensorMapEncodeTiled is fetched through the runtime
// (cudaGetDriverEntryPoint) so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

namespace fa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// (B*H, T, D) bf16 tensor viewed as a 3-D map {D, T, BH} (innermost first),
// box {64, box_rows, 1}, 128-byte swizzle, out-of-range elements read as 0
// and clipped on store.  Returns false if the driver rejects it.
inline bool make_tmap_bhtd(CUtensorMap* map, const void* base, int BH, int T, int D, int box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
    cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// (BH, T_pad, D) fp32 accumulator viewed as {D, T_pad, BH} with boxes of 32
// columns (128 bytes) x box_rows rows and 128-byte swizzle: the target of the
// fused backward's dQ reduce-adds.
inline bool make_tmap_f32_acc(CUtensorMap* map, const void* base, int BH, int T_pad, int D, int box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T_pad), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(T_pad) * D * 4};
    cuuint32_t box[3] = {32u, static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed variable-length layout (total, H, D) bf16: dimensions (D, H, total)
// with strides (2 B, D*2 B, H*D*2 B), boxes of 64 columns x 1 head x
// box_rows rows.  The box lands in shared memory exactly as a
// 64 x box_rows box of the (B*H, T, D) map does (rows of 128 bytes, 128-byte
// swizzle), so kernels only swap the (row, head) coordinates.  Rows past
// `total` read as zeros.
inline bool make_tmap_packed(CUtensorMap* map, const void* base, int total, int H, int D, int box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fa
