// gemv.h -- the few-token path of the block types (gemv.cu): host launcher.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mmq {

// Largest token count the matrix-vector kernel takes; larger M run on the tile kernels (every type: q6_K,
// the heaviest decode per value, still beats its tile path at 5-7 tokens and ties it at 8 on the 7B
// FFN-down shape).
constexpr int MMVQ_MAX_M = 8;
inline int mmvq_max_m(int) { return MMVQ_MAX_M; }

// out f32 [M][N] for block-type weights W (raw blocks, N rows of row_bytes) and q8_1 activations Xq
// (int8 codes [M][K] at byte 0, float2 (d, s) [M][K/32] at byte M*K); 1 <= M <= MMVQ_MAX_M, K % 256 == 0.
cudaError_t run_gemv(int wt, const void* W, long long row_bytes, const void* Xq, float* out, long long M, long long N,
                     long long K, cudaStream_t s);

}  // namespace mmq
