// gemm_iq1_m.cu -- instantiation of the MMQ tensor-core kernel for one weight type (see gemm.cuh).
#include "gemm.cuh"
#include "internal.h"

namespace mmq {

cudaError_t run_gemm_iq1_m(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s) {
    if (mode == MODE_DEBUG) return launch_gemm<WT_IQ1_M, MODE_DEBUG, false>(p, grid_y, s);
    if (moe) return launch_gemm<WT_IQ1_M, MODE_PROD, true>(p, grid_y, s);
    return launch_gemm<WT_IQ1_M, MODE_PROD, false>(p, grid_y, s);
}

MMQ_DEFINE_ERROR_READER(iq1_m)

}  // namespace mmq
