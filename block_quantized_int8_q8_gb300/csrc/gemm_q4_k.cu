// gemm_q4_k.cu -- instantiation of the MMQ tensor-core kernel for one weight type (see gemm.cuh).
#include "gemm.cuh"
#include "internal.h"

namespace mmq {

cudaError_t run_gemm_q4_k(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s) {
    if (mode == MODE_DEBUG) return launch_gemm<WT_Q4_K, MODE_DEBUG, false>(p, grid_y, s);
    if (moe) return launch_gemm<WT_Q4_K, MODE_PROD, true>(p, grid_y, s);
    return launch_gemm<WT_Q4_K, MODE_PROD, false>(p, grid_y, s);
}

MMQ_DEFINE_ERROR_READER(q4_k)

}  // namespace mmq
