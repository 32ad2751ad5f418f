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

// Most (token, slot) pairs run_gemv_id takes: one grid row (gridDim.y) per pair.
constexpr long long kMaxGemvPairs = 65535;

// The same kernel for MUL_MAT_ID at 1 <= M <= MMVQ_MAX_M tokens: W holds n_experts matrices of N rows;
// out f32 [M][slots][N], row (t, j) the product of token t with expert ids[t][j] (no routing pass).
cudaError_t run_gemv_id(int wt, const void* W, long long row_bytes, int n_experts, const void* Xq,
                        const int32_t* ids, int slots, float* out, long long M, long long N, long long K,
                        cudaStream_t s);

// Read and clear the device error bits the MoE mode raises (mmq_read_device_errors gathers every kernel's).
cudaError_t read_clear_errors_gemv(unsigned* bits, cudaStream_t s);

}  // namespace mmq
