// gemm_w8a8.cu -- instantiation of the MMQ tensor-core kernel for one weight type (see gemm.cuh).
#include "gemm.cuh"
#include "internal.h"

namespace mmq {

cudaError_t run_gemm_w8a8(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s) {
    if (mode == MODE_DEBUG) return launch_gemm<WT_W8A8, MODE_DEBUG, false>(p, grid_y, s);
    if (moe) return cudaErrorNotSupported;             // MUL_MAT_ID is defined for the block types
    return launch_gemm<WT_W8A8, MODE_PROD, false>(p, grid_y, s);
}

MMQ_DEFINE_ERROR_READER(w8a8)

}  // namespace mmq
