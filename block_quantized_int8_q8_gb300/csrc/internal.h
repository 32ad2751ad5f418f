// internal.h -- host-side interface between the C ABI (capi.cu) and the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/mmq.h"

namespace mmq {
struct GemmParams;

// ------------------------------------------------------------------------------------------ shape rules
// One set of rules for every entry point and size helper (include/mmq.h, "Shape rules").
constexpr long long kMaxDim = (1ll << 31) - 1;

inline bool known_type(int t) { return t >= MMQ_Q8_0 && t <= MMQ_Q6_K; }
inline bool block_type(int t) { return (t >= MMQ_Q8_0 && t <= MMQ_IQ1_M) || t == MMQ_Q6_K; }
// Types the general kernel takes (debug partials, mmq_gemm_id_noalloc, shapes the TMA kernel does not).
inline bool general_type(int t) { return t >= MMQ_Q8_0 && t <= MMQ_W8A8; }

// K granule of a weight type: the block types run in 256-k super-stages, W8A8 in 64-k stages.
inline long long k_granule(int t) { return t == MMQ_W8A8 ? 64 : 256; }

// Raw bytes of one weight row of K values (-1 for an unknown type).
inline long long weight_row_bytes(int t, long long K) {
    switch (t) {
        case MMQ_Q8_0: return K / 32 * 34;
        case MMQ_Q4_0: return K / 32 * 18;
        case MMQ_Q4_K: return K / 256 * 144;
        case MMQ_IQ1_M: return K / 256 * 76;
        case MMQ_W8A8: return K;
        case MMQ_Q6_K: return K / 256 * 224;
    }
    return -1;
}

// Shape rules shared by every GEMM entry point: M, N >= 0; K > 0 and a multiple of the type's granule;
// M*K and N*K below 2^31.
inline mmq_status check_shape(int t, long long M, long long N, long long K) {
    if (M < 0 || N < 0 || K <= 0) return MMQ_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return MMQ_ERR_SHAPE;
    if (M * K > kMaxDim || N * K > kMaxDim) return MMQ_ERR_SHAPE;
    return (K % k_granule(t) == 0) ? MMQ_OK : MMQ_ERR_SHAPE;
}

// q8_1 activation buffers (the quantizer's rule): K > 0, K % 64 == 0, M*K below 2^31.
inline bool q8_1_shape_ok(long long M, long long K) {
    return M >= 0 && K > 0 && K % 64 == 0 && M <= kMaxDim && M * K <= kMaxDim;
}

// Record a CUDA failure for mmq_last_cuda_error (the calling host thread's message) and return
// MMQ_ERR_CUDA (capi.cu).
mmq_status record_cuda_failure(cudaError_t e, const char* where);

// q8_1 buffer sections (byte offsets), see include/mmq.h
struct Q81Layout {
    long long ds, h, dT, sT, Mp, total;
};
inline Q81Layout q81_layout(long long M, long long K) {
    Q81Layout L;
    const long long kb = K / 32;
    L.Mp = (M + 3) / 4 * 4;                       // block-major rows padded to 16 bytes
    L.ds = M * K;
    L.h = (M * K + M * kb * 8 + 255) / 256 * 256;
    L.dT = (L.h + 2 * M * K + 255) / 256 * 256;
    L.sT = L.dT + L.Mp * kb * 4;
    L.total = (L.sT + L.Mp * kb * 4 + 255) / 256 * 256;
    return L;
}

// Arguments of the TMA-fed dense kernel (gemm_tma.cu).
struct TmaGemmArgs {
    const void* W;              // raw weights, N rows of w_row_bytes
    const void* xh;             // q8_1 shadow: fp16 codes [M][K]
    const float* dT;            // q8_1 shadow: d, block-major [K/32][Mp]
    const float* sT;            // q8_1 shadow: s, block-major [K/32][Mp]
    float* out;                 // f32 [M][N] (MoE: [M*slots][N])
    long long w_row_bytes;
    long long M, N, K, Mp;      // MoE: M = gathered rows, Mp their block-major pitch
    // MoE mode (work != null): the weights hold E experts of N rows; xh/dT/sT are the gathered operand
    long long E = 1;
    const int* work = nullptr;
    const int* nwork = nullptr;
    const int* gstart = nullptr;
    const int* rowlist = nullptr;
    int max_work = 0;
};
bool tma_gemm_supported(int wt, long long K);
// block_sums: instead of the product, int32 [M][N][K/32] of every 32-k block's exact integer accumulator
// (dense only; `out` then points at the int32 array).
cudaError_t run_gemm_tma(int wt, const TmaGemmArgs& a, cudaStream_t s, bool block_sums = false);
// MoE operand gather (gemm_tma.cu): the fp16 codes and block scales of each work item's token rows,
// copied to rows gstart[w] .. gstart[w] + count - 1 of xg [Rg][K] / dTg, sTg [K/32][Rg]; gstart[w] is
// the 4-aligned prefix sum of the preceding items' counts.  Rg >= M*slots + 3*max_work, Rg % 4 == 0.
struct MoeGatherArgs {
    const int* work;
    const int* nwork;
    const int* rowlist;
    int slots, max_work;
    const void* xh;             // q8_1 shadow of the M tokens
    const float* dT;
    const float* sT;
    long long Mp, K;
    int* gstart;
    void* xg;
    float* dTg;
    float* sTg;
    long long Rg;
    float* out;                 // MoE output [M*slots][N]: rows of tiles split along K are zeroed here
    long long N;
    int sms = 0, kparts = 1;    // set by run_moe_gather
};
cudaError_t run_moe_gather(const MoeGatherArgs& g, int wt, cudaStream_t s);
// Per-channel W8A8 on the TMA-fed kernel (gemm_w8a8_tma.cuh): W = int8 [N][K] + f32 ws[N],
// X = int8 [M][K] + f32 xs[M], out bf16 [M][N]; K % 64 == 0.
cudaError_t run_gemm_w8a8_tma(const void* W, const void* X, void* out, long long M, long long N, long long K,
                              cudaStream_t s);

// Quantizer and shadow preparation (quantize.cu)
cudaError_t run_quantize_q8_1(const float* x, long long M, long long K, void* xq, cudaStream_t s);
cudaError_t run_prepare_q8_1(void* xq, long long M, long long K, cudaStream_t s);

// Dense / MoE / debug GEMM launchers, one per weight type (gemm_<type>.cu).
// mode: 0 production, 1 debug partials.  moe: grouped launch driven by the routing workspace.
cudaError_t run_gemm_q8_0(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s);
cudaError_t run_gemm_q4_0(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s);
cudaError_t run_gemm_q4_k(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s);
cudaError_t run_gemm_iq1_m(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s);
cudaError_t run_gemm_w8a8(const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s);

// MoE routing (route.cu): count, scan into work items, scatter.  Workspace carved by the caller.
struct RouteWorkspace {
    int* counts;     // [E]
    int* offsets;    // [E]
    int* cursor;     // [E]
    int* nwork;      // [1]
    int* work;       // [3 * max_work]
    int* rowlist;    // [M * slots]
    int max_work;
};
cudaError_t run_route(const int32_t* ids, int M, int slots, int E, int tile_n, const RouteWorkspace& ws,
                      cudaStream_t s);
// The same lists from one single-block launch (route.cu), for small problems; writes work, nwork and
// rowlist only.
constexpr int ROUTE_FUSED_MAX_EXPERTS = 1024;
constexpr long long ROUTE_FUSED_MAX_ROWS = 1 << 16;
bool route_fused_supported(long long M, int slots, int E);
cudaError_t run_route_fused(const int32_t* ids, int M, int slots, int E, int tile_n, const RouteWorkspace& ws,
                            cudaStream_t s);

// Per-device once-flags for function attributes (cudaFuncSetAttribute acts on the current device's
// context): the current device's flag in `flags`, or a scratch flag (always false) past 64 devices.
inline bool& device_flag(bool (&flags)[64]) {
    static thread_local bool scratch;
    int dev = 0;
    scratch = false;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return scratch;
    return flags[dev];
}

// Per-translation-unit device error words: read, OR into *bits, clear.
cudaError_t read_clear_errors_quantize(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_route(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_q8_0(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_q4_0(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_q4_k(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_iq1_m(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_w8a8(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_tma(unsigned* bits, cudaStream_t s);
cudaError_t read_clear_errors_selftest(unsigned* bits, cudaStream_t s);
// Device self-test of the bounded waits (selftest.cu): result int32 [4].
cudaError_t run_wait_timeout_selftest(int* result, cudaStream_t s);
}  // namespace mmq

// Defines read_clear_errors_<name> for the translation unit that expands it.
#define MMQ_DEFINE_ERROR_READER(name)                                                               \
    cudaError_t read_clear_errors_##name(unsigned* bits, cudaStream_t s) {                          \
        unsigned v = 0, z = 0;                                                                      \
        cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_mmq_device_errors, sizeof(v), 0,            \
                                                  cudaMemcpyDeviceToHost, s);                       \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                                         \
        if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_mmq_device_errors, &z, sizeof(z), 0,    \
                                                          cudaMemcpyHostToDevice, s);               \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                                         \
        *bits |= v;                                                                                 \
        return e;                                                                                   \
    }
