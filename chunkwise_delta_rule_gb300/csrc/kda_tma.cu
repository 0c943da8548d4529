// Host side of the TMA tensor maps for the token-major inputs [Ttot][H][D]. A box may be wider
// than the tensor's rows: the columns past D read as zeros (loads) or are dropped (stores).
// The encode function is taken from the driver through the runtime's
// versioned entry-point query, so the library does not link the driver API.
#include <cudaTypedefs.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int Ttot, int H, int D,
            int box_x, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Ttot};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    const cuuint32_t box[3] = {(cuuint32_t)box_x, 1u, (cuuint32_t)BT};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tmap_rows_bf16(CUtensorMap* m, const void* base, int Ttot, int H, int D) {
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, Ttot, H, D, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_state_f32(CUtensorMap* m, const float* base, int NH, int K, int V) {
    auto fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15) || K % 32 != 0 || V % 32 != 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)K, (cuuint64_t)NH};
    const cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)K * V * 4};
    const cuuint32_t box[3] = {32u, 32u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_rows_f32(CUtensorMap* m, const void* base, int Ttot, int H, int D, int box_x) {
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, Ttot, H, D, box_x > 0 ? box_x : D,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace kda
