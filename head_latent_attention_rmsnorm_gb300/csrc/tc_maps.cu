// tc_maps.cu -- TMA tensor-map encoding for the tensor-core kernels.  The driver's
// cuTensorMapEncodeTiled is reached through the runtime's entry-point query, so the
// library has no link-time dependency on the driver library.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_internal.h"

namespace mla {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

}  // namespace

cudaError_t make_tma_map(CUtensorMap *map, const void *ptr, int rank, const unsigned long long *dims,
                         const unsigned long long *strides, const unsigned *box) {
    std::call_once(g_once, resolve);
    if (!g_encode) return cudaErrorNotSupported;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_operand_map(CUtensorMap *map, const TmaOperand &op, int tile_rows) {
    unsigned br = (unsigned)(op.rows_per_z < tile_rows ? op.rows_per_z : tile_rows);
    unsigned bz = (unsigned)(tile_rows / br);
    if (br > 256 || bz > 256 || (tile_rows % br) != 0) return cudaErrorInvalidValue;
    unsigned long long dims[3] = {(unsigned long long)op.k_extent, (unsigned long long)op.rows,
                                  (unsigned long long)op.z_extent};
    unsigned long long zs = (unsigned long long)op.z_stride;
    if (op.z_extent <= 1) zs = (unsigned long long)op.rows * (unsigned long long)op.row_stride;
    zs = (zs + 15) / 16 * 16;
    unsigned long long strides[2] = {(unsigned long long)op.row_stride, zs};
    unsigned box[3] = {64, br, bz};
    return make_tma_map(map, op.ptr, 3, dims, strides, box);
}

cudaError_t make_operand_map_mn(CUtensorMap *map, const TmaOperand &op) {
    unsigned long long dims[3] = {(unsigned long long)op.k_extent, (unsigned long long)op.rows,
                                  (unsigned long long)(op.z_extent < 1 ? 1 : op.z_extent)};
    unsigned long long zs = (unsigned long long)op.z_stride;
    if (op.z_extent <= 1) zs = (unsigned long long)op.rows * (unsigned long long)op.row_stride;
    zs = (zs + 15) / 16 * 16;
    unsigned long long strides[2] = {(unsigned long long)op.row_stride, zs};
    unsigned box[3] = {64, 64, 1};
    return make_tma_map(map, op.ptr, 3, dims, strides, box);
}

}  // namespace mla
