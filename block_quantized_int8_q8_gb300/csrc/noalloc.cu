// noalloc.cu -- mmq_gemm_id_noalloc: the MoE product for callers that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is unavailable or forbidden -- inside a
// stream-capture region that must not allocate, under an allocator that owns all device memory
// (a framework's caching pool, a serving engine with a fixed memory budget), or in a plugin that is
// handed only its input and output buffers.  mmq_gemm_id needs a caller-supplied workspace for its
// routing lists; this variant keeps that workspace in a file-scope device array instead.
//
// The scratch array is MMQ_NOALLOC_SCRATCH_BYTES (1 MiB) of static device memory: every GPU that
// loads the library holds it until the process exits.  All calls share it and it keeps the last
// call's contents; the routing kernels rewrite every entry they later read (the per-expert counts
// are cleared at the start of each call), so nothing has to be zero on entry.  Two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on the array.
// The array's device address is looked up once per device and kept for the life of the process: it
// assumes the device's primary context, which the CUDA runtime uses, is never torn down and recreated
// (cudaDeviceReset) while the library is in use.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include "../../include/mmq.h"
#include "gemm.cuh"
#include "internal.h"
#include "gemv.h"

using namespace mmq;

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MMQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  The symbol name is a host-side
// stand-in, so the address must come from cudaGetSymbolAddress, once per device, with that device
// current.  This runs on the first call on each device.
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

extern "C" mmq_status mmq_gemm_id_noalloc(mmq_type wtype, const void* W, int n_experts, const void* Xq,
                                          const int32_t* expert_ids, int n_slots, float* out, int64_t M,
                                          int64_t N, int64_t K, mmq_stream_t stream) {
    if (!known_type(wtype)) return MMQ_ERR_INVALID_ARG;
    // the general kernel's block types; W8A8 has no MoE form and Q6_K runs on the TMA-fed kernel only
    if (!block_type(wtype) || !general_type(wtype)) return MMQ_ERR_UNSUPPORTED;
    if (n_experts <= 0 || n_slots <= 0) return MMQ_ERR_INVALID_ARG;
    const mmq_status st = check_shape(wtype, M, N, K);
    if (st != MMQ_OK) return st;
    if (M * n_slots > kMaxDim || (long long)n_experts * N * weight_row_bytes(wtype, K) > (1ll << 40))
        return MMQ_ERR_SHAPE;
    if (M == 0 || N == 0) return MMQ_OK;
    if (!W || !Xq || !expert_ids || !out) return MMQ_ERR_INVALID_ARG;
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(W) || !al(Xq) || !al(out) || !al(expert_ids)) return MMQ_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M <= mmvq_max_m((int)wtype) && M * n_slots <= kMaxGemvPairs) {
        // a few tokens: the matrix-vector kernel reads the ids itself and needs no routing lists
        const cudaError_t e = run_gemv_id((int)wtype, W, weight_row_bytes(wtype, K), n_experts, Xq, expert_ids,
                                          n_slots, out, M, N, K, s);
        return e == cudaSuccess ? MMQ_OK : record_cuda_failure(e, "mmq_gemm_id_noalloc");
    }

    // carve the routing lists out of the scratch array (same layout as the mmq_gemm_id workspace)
    const long long rows = M * n_slots;
    const int max_work = (int)((rows + BN - 1) / BN + n_experts);
    const size_t counts = 0, offsets = counts + round256(4ull * n_experts), cursor = offsets + round256(4ull * n_experts);
    const size_t nwork = cursor + round256(4ull * n_experts), work = nwork + round256(4);
    const size_t rowlist = work + round256(12ull * max_work), total = rowlist + round256(4ull * rows);
    if (total > MMQ_NOALLOC_SCRATCH_BYTES) return MMQ_ERR_WORKSPACE;   // problem too large for the array

    void* base = nullptr;
    cudaError_t e = scratch_for_current_device(&base);
    if (e != cudaSuccess) return record_cuda_failure(e, "mmq_gemm_id_noalloc scratch address");
    uint8_t* sb = static_cast<uint8_t*>(base);
    RouteWorkspace ws;
    ws.counts = reinterpret_cast<int*>(sb + counts);
    ws.offsets = reinterpret_cast<int*>(sb + offsets);
    ws.cursor = reinterpret_cast<int*>(sb + cursor);
    ws.nwork = reinterpret_cast<int*>(sb + nwork);
    ws.work = reinterpret_cast<int*>(sb + work);
    ws.rowlist = reinterpret_cast<int*>(sb + rowlist);
    ws.max_work = max_work;
    e = run_route(expert_ids, (int)M, n_slots, n_experts, BN, ws, s);
    if (e != cudaSuccess) return record_cuda_failure(e, "mmq_gemm_id_noalloc routing");

    GemmParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.xq = static_cast<const int8_t*>(Xq);
    const Q81Layout Lq = q81_layout(M, K);
    p.xds = reinterpret_cast<const float4*>(static_cast<const uint8_t*>(Xq) + Lq.ds);
    p.xh = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(Xq) + Lq.h);
    p.out = out;
    p.w_row_bytes = weight_row_bytes(wtype, K);
    p.w_expert_bytes = p.w_row_bytes * N;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.rowlist = ws.rowlist;
    p.work = ws.work;
    p.nwork = ws.nwork;
    p.slots = n_slots;
    e = cudaErrorInvalidValue;
    switch (wtype) {
        case MMQ_Q8_0: e = run_gemm_q8_0(p, MODE_PROD, true, max_work, s); break;
        case MMQ_Q4_0: e = run_gemm_q4_0(p, MODE_PROD, true, max_work, s); break;
        case MMQ_Q4_K: e = run_gemm_q4_k(p, MODE_PROD, true, max_work, s); break;
        case MMQ_IQ1_M: e = run_gemm_iq1_m(p, MODE_PROD, true, max_work, s); break;
        default: break;
    }
    return e == cudaSuccess ? MMQ_OK : record_cuda_failure(e, "mmq_gemm_id_noalloc");
}
