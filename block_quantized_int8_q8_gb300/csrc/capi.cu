// capi.cu -- the extern "C" boundary of libmmq_gb300.so (declared and documented in include/mmq.h).
// Validates arguments synchronously, carves caller-owned workspaces, and enqueues kernels on the
// caller's stream.  Nothing here allocates, frees or synchronises device memory (except
// mmq_read_device_errors, which synchronises the given stream by design).
#include <cstdint>
#include <cstddef>
#include <cstdio>
#include <cuda_runtime.h>
#include "../../include/mmq.h"
#include "gemm.cuh"
#include "internal.h"
#include "gemv.h"

using namespace mmq;

namespace {
thread_local char g_last_cuda_error[256] = "";
}  // namespace

namespace mmq {
mmq_status record_cuda_failure(cudaError_t e, const char* where) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", where, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return MMQ_ERR_CUDA;
}
}  // namespace mmq

namespace {

mmq_status cuda_fail(cudaError_t e, const char* where) { return record_cuda_failure(e, where); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long weight_row_bytes(mmq_type t, long long K) { return mmq::weight_row_bytes((int)t, K); }
mmq_status check_shape(mmq_type t, long long M, long long N, long long K) { return mmq::check_shape((int)t, M, N, K); }

cudaError_t dispatch(mmq_type t, const GemmParams& p, int mode, bool moe, int grid_y, cudaStream_t s) {
    switch (t) {
        case MMQ_Q8_0: return run_gemm_q8_0(p, mode, moe, grid_y, s);
        case MMQ_Q4_0: return run_gemm_q4_0(p, mode, moe, grid_y, s);
        case MMQ_Q4_K: return run_gemm_q4_k(p, mode, moe, grid_y, s);
        case MMQ_IQ1_M: return run_gemm_iq1_m(p, mode, moe, grid_y, s);
        case MMQ_W8A8: return run_gemm_w8a8(p, mode, moe, grid_y, s);
    }
    return cudaErrorInvalidValue;
}

GemmParams dense_params(mmq_type t, const void* W, const void* Xq, void* out, long long M, long long N,
                        long long K) {
    GemmParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.xq = static_cast<const int8_t*>(Xq);
    const uint8_t* xb = static_cast<const uint8_t*>(Xq);
    if (t == MMQ_W8A8) {
        p.w8_xs = reinterpret_cast<const float*>(xb + M * K);
        p.w8_ws = reinterpret_cast<const float*>(static_cast<const uint8_t*>(W) + N * K);
    } else {
        const Q81Layout L = q81_layout(M, K);
        p.xds = reinterpret_cast<const float4*>(xb + L.ds);
        p.xh = reinterpret_cast<const uint16_t*>(xb + L.h);
    }
    p.out = out;
    p.w_row_bytes = weight_row_bytes(t, K);
    p.w_expert_bytes = p.w_row_bytes * N;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    return p;
}

// mmq_gemm_id workspace: the routing lists, then the gathered MoE operand of the TMA-fed kernel
// (fp16 codes [Rg][K], block-major d and s [K/32][Rg], each work item's rows at a 4-aligned offset).
struct IdLayout {
    size_t counts, offsets, cursor, nwork, work, rowlist, gstart, xg, dTg, sTg, total;
    long long Rg;
    int max_work;
};

IdLayout id_layout(long long M, long long K, int slots, int E) {
    IdLayout L{};
    const long long rows = M * slots;
    L.max_work = (int)((rows + BN - 1) / BN + E);
    L.Rg = (rows + 3ll * L.max_work + 3) / 4 * 4;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    L.counts = take(sizeof(int) * (size_t)E);
    L.offsets = take(sizeof(int) * (size_t)E);
    L.cursor = take(sizeof(int) * (size_t)E);
    L.nwork = take(sizeof(int));
    L.work = take(sizeof(int) * 3 * (size_t)L.max_work);
    L.rowlist = take(sizeof(int) * (size_t)rows);
    L.gstart = take(sizeof(int) * (size_t)L.max_work);
    L.xg = take((size_t)L.Rg * (size_t)K * 2);
    L.dTg = take((size_t)(K / 32) * (size_t)L.Rg * 4);
    L.sTg = take((size_t)(K / 32) * (size_t)L.Rg * 4);
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

const char* mmq_status_string(mmq_status s) {
    switch (s) {
        case MMQ_OK: return "ok";
        case MMQ_ERR_INVALID_ARG: return "invalid argument";
        case MMQ_ERR_SHAPE: return "shape violates the K/M/N rules";
        case MMQ_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MMQ_ERR_UNSUPPORTED: return "unsupported request";
        case MMQ_ERR_CUDA: return "CUDA runtime or launch failure";
        case MMQ_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t mmq_q8_1_bytes(int64_t M, int64_t K) {
    if (!q8_1_shape_ok(M, K)) return 0;                    // exactly where mmq_quantize_q8_1 says MMQ_ERR_SHAPE
    return (size_t)q81_layout(M, K).total;
}

size_t mmq_weight_bytes(mmq_type t, int64_t N, int64_t K) {
    if (!known_type(t) || check_shape(t, 0, N, K) != MMQ_OK) return 0;   // exactly where mmq_gemm says MMQ_ERR_SHAPE
    if (t == MMQ_W8A8) return (size_t)(N * K + 4 * N);
    return (size_t)(N * weight_row_bytes(t, K));
}

size_t mmq_w8a8_act_bytes(int64_t M, int64_t K) {
    if (check_shape(MMQ_W8A8, M, 0, K) != MMQ_OK) return 0;
    return (size_t)(M * K + 4 * M);
}

mmq_status mmq_q8_1_prepare(void* xq, int64_t M, int64_t K, mmq_stream_t stream) {
    if (!q8_1_shape_ok(M, K)) return MMQ_ERR_SHAPE;
    if (M == 0) return MMQ_OK;
    if (!xq) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(xq)) return MMQ_ERR_ALIGN;
    const cudaError_t e = run_prepare_q8_1(xq, M, K, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_q8_1_prepare");
}

mmq_status mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, void* xq, mmq_stream_t stream) {
    if (!q8_1_shape_ok(M, K)) return MMQ_ERR_SHAPE;
    if (M == 0) return MMQ_OK;
    if (!x || !xq) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq)) return MMQ_ERR_ALIGN;
    const cudaError_t e = run_quantize_q8_1(x, M, K, xq, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_quantize_q8_1");
}

mmq_status mmq_gemm(mmq_type wtype, const void* W, const void* Xq, void* out, int64_t M, int64_t N, int64_t K,
                    mmq_stream_t stream) {
    if (!known_type(wtype)) return MMQ_ERR_INVALID_ARG;
    mmq_status st = check_shape(wtype, M, N, K);
    if (st != MMQ_OK) return st;
    if (M == 0 || N == 0) return MMQ_OK;
    if (!W || !Xq || !out) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(out)) return MMQ_ERR_ALIGN;
    if (wtype == MMQ_W8A8 && (((M * K) & 3) || ((N * K) & 3))) return MMQ_ERR_ALIGN;
    if (block_type(wtype) && M <= mmvq_max_m((int)wtype)) {
        // a few tokens: the matrix-vector kernel (gemv.cu), weights read once at memory speed
        const cudaError_t e = run_gemv((int)wtype, W, weight_row_bytes(wtype, K), Xq, static_cast<float*>(out), M, N,
                                       K, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm");
    }
    if (block_type(wtype) && tma_gemm_supported((int)wtype, K)) {
        // the TMA-fed kernel (gemm_tma.cuh); the general kernel covers the remaining shapes
        const Q81Layout L = q81_layout(M, K);
        const uint8_t* xb = static_cast<const uint8_t*>(Xq);
        TmaGemmArgs a{};
        a.W = W;
        a.xh = xb + L.h;
        a.dT = reinterpret_cast<const float*>(xb + L.dT);
        a.sT = reinterpret_cast<const float*>(xb + L.sT);
        a.out = static_cast<float*>(out);
        a.w_row_bytes = weight_row_bytes(wtype, K);
        a.M = M;
        a.N = N;
        a.K = K;
        a.Mp = L.Mp;
        const cudaError_t e = run_gemm_tma((int)wtype, a, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm");
    }
    if (wtype == MMQ_W8A8) {
        const cudaError_t e = run_gemm_w8a8_tma(W, Xq, out, M, N, K, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm");
    }
    if (!general_type(wtype)) return MMQ_ERR_UNSUPPORTED;
    GemmParams p = dense_params(wtype, W, Xq, out, M, N, K);
    const cudaError_t e =
        dispatch(wtype, p, MODE_PROD, false, (int)((M + BN - 1) / BN), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm");
}

mmq_status mmq_gemm_debug_partials(mmq_type wtype, const void* W, const void* Xq, int32_t* partials, int64_t M,
                                   int64_t N, int64_t K, mmq_stream_t stream) {
    if (!known_type(wtype)) return MMQ_ERR_INVALID_ARG;
    if (!general_type(wtype)) return MMQ_ERR_UNSUPPORTED;
    mmq_status st = check_shape(wtype, M, N, K);
    if (st != MMQ_OK) return st;
    if (M == 0 || N == 0) return MMQ_OK;
    if (!W || !Xq || !partials) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(partials)) return MMQ_ERR_ALIGN;
    GemmParams p = dense_params(wtype, W, Xq, nullptr, M, N, K);
    p.partials = partials;
    const cudaError_t e =
        dispatch(wtype, p, MODE_DEBUG, false, (int)((M + BN - 1) / BN), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm_debug_partials");
}

mmq_status mmq_gemm_debug_block_sums(mmq_type wtype, const void* W, const void* Xq, int32_t* sums, int64_t M,
                                     int64_t N, int64_t K, mmq_stream_t stream) {
    if (!known_type(wtype)) return MMQ_ERR_INVALID_ARG;
    mmq_status st = check_shape(wtype, M, N, K);
    if (st != MMQ_OK) return st;
    if (!block_type(wtype) || !tma_gemm_supported((int)wtype, K)) return MMQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return MMQ_OK;
    if (!W || !Xq || !sums) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(sums)) return MMQ_ERR_ALIGN;
    const Q81Layout L = q81_layout(M, K);
    const uint8_t* xb = static_cast<const uint8_t*>(Xq);
    TmaGemmArgs a{};
    a.W = W;
    a.xh = xb + L.h;
    a.dT = reinterpret_cast<const float*>(xb + L.dT);
    a.sT = reinterpret_cast<const float*>(xb + L.sT);
    a.out = reinterpret_cast<float*>(sums);
    a.w_row_bytes = weight_row_bytes(wtype, K);
    a.M = M;
    a.N = N;
    a.K = K;
    a.Mp = L.Mp;
    const cudaError_t e = run_gemm_tma((int)wtype, a, reinterpret_cast<cudaStream_t>(stream), true);
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm_debug_block_sums");
}

size_t mmq_gemm_id_workspace_bytes(int64_t M, int64_t K, int n_slots, int n_experts) {
    if (M < 0 || K < 0 || n_slots <= 0 || n_experts <= 0) return 0;
    return id_layout(M, K, n_slots, n_experts).total;
}

mmq_status mmq_gemm_id(mmq_type wtype, const void* W, int n_experts, const void* Xq, const int32_t* expert_ids,
                       int n_slots, float* out, int64_t M, int64_t N, int64_t K, void* workspace,
                       size_t workspace_bytes, mmq_stream_t stream) {
    if (!block_type(wtype)) return wtype == MMQ_W8A8 ? MMQ_ERR_UNSUPPORTED : MMQ_ERR_INVALID_ARG;
    if (n_experts <= 0 || n_slots <= 0) return MMQ_ERR_INVALID_ARG;
    mmq_status st = check_shape(wtype, M, N, K);
    if (st != MMQ_OK) return st;
    if (M * n_slots > kMaxDim || (long long)n_experts * N * weight_row_bytes(wtype, K) > (1ll << 40))
        return MMQ_ERR_SHAPE;
    if (M == 0 || N == 0) return MMQ_OK;
    if (!W || !Xq || !expert_ids || !out) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(out) || !aligned16(expert_ids)) return MMQ_ERR_ALIGN;
    const IdLayout L = id_layout(M, K, n_slots, n_experts);
    if (!workspace || workspace_bytes < L.total) return MMQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MMQ_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M <= mmvq_max_m((int)wtype) && M * n_slots <= kMaxGemvPairs) {
        // a few tokens: each (token, slot) pair is a one-token product with its expert, read straight
        // from the ids by the matrix-vector kernel (gemv.cu) -- no routing pass, no gather
        const cudaError_t e = run_gemv_id((int)wtype, W, weight_row_bytes(wtype, K), n_experts, Xq, expert_ids,
                                          n_slots, out, M, N, K, s);
        return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm_id");
    }
    uint8_t* wb = static_cast<uint8_t*>(workspace);
    RouteWorkspace ws;
    ws.counts = reinterpret_cast<int*>(wb + L.counts);
    ws.offsets = reinterpret_cast<int*>(wb + L.offsets);
    ws.cursor = reinterpret_cast<int*>(wb + L.cursor);
    ws.nwork = reinterpret_cast<int*>(wb + L.nwork);
    ws.work = reinterpret_cast<int*>(wb + L.work);
    ws.rowlist = reinterpret_cast<int*>(wb + L.rowlist);
    ws.max_work = L.max_work;
    const bool tma = tma_gemm_supported((int)wtype, K) && (long long)n_experts * N < (1ll << 31) && L.Rg < (1ll << 31);
    if (!tma && !general_type(wtype)) return MMQ_ERR_UNSUPPORTED;
    cudaError_t e = (tma && route_fused_supported(M, n_slots, n_experts))
                        ? run_route_fused(expert_ids, (int)M, n_slots, n_experts, BN, ws, s)
                        : run_route(expert_ids, (int)M, n_slots, n_experts, BN, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "mmq_gemm_id routing");
    if (tma) {
        // TMA-fed kernel: gather each work item's token rows, then one CTA per (item, weight-row tile)
        const Q81Layout X = q81_layout(M, K);
        const uint8_t* xb = static_cast<const uint8_t*>(Xq);
        MoeGatherArgs g{};
        g.work = ws.work;
        g.nwork = ws.nwork;
        g.rowlist = ws.rowlist;
        g.slots = n_slots;
        g.max_work = L.max_work;
        g.xh = xb + X.h;
        g.dT = reinterpret_cast<const float*>(xb + X.dT);
        g.sT = reinterpret_cast<const float*>(xb + X.sT);
        g.Mp = X.Mp;
        g.K = K;
        g.gstart = reinterpret_cast<int*>(wb + L.gstart);
        g.xg = wb + L.xg;
        g.dTg = reinterpret_cast<float*>(wb + L.dTg);
        g.sTg = reinterpret_cast<float*>(wb + L.sTg);
        g.Rg = L.Rg;
        g.out = out;
        g.N = N;
        e = run_moe_gather(g, (int)wtype, s);
        if (e != cudaSuccess) return cuda_fail(e, "mmq_gemm_id gather");
        TmaGemmArgs a;
        a.W = W;
        a.xh = g.xg;
        a.dT = g.dTg;
        a.sT = g.sTg;
        a.out = out;
        a.w_row_bytes = weight_row_bytes(wtype, K);
        a.M = L.Rg;
        a.N = N;
        a.K = K;
        a.Mp = L.Rg;
        a.E = n_experts;
        a.work = ws.work;
        a.nwork = ws.nwork;
        a.gstart = g.gstart;
        a.rowlist = ws.rowlist;
        a.max_work = L.max_work;
        e = run_gemm_tma((int)wtype, a, s);
        return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm_id");
    }
    GemmParams p = dense_params(wtype, W, Xq, out, M, N, K);
    p.rowlist = ws.rowlist;
    p.work = ws.work;
    p.nwork = ws.nwork;
    p.slots = n_slots;
    e = dispatch(wtype, p, MODE_PROD, true, L.max_work, s);
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_gemm_id");
}

mmq_status mmq_selftest_bounded_wait(int32_t* result, mmq_stream_t stream) {
    if (!result) return MMQ_ERR_INVALID_ARG;
    if (!aligned16(result)) return MMQ_ERR_ALIGN;
    const cudaError_t e = run_wait_timeout_selftest(result, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_selftest_bounded_wait");
}

mmq_status mmq_read_device_errors(unsigned* bits, mmq_stream_t stream) {
    if (!bits) return MMQ_ERR_INVALID_ARG;
    *bits = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    cudaError_t (*readers[])(unsigned*, cudaStream_t) = {read_clear_errors_quantize, read_clear_errors_route,
                                                         read_clear_errors_q8_0,     read_clear_errors_q4_0,
                                                         read_clear_errors_q4_k,     read_clear_errors_iq1_m,
                                                         read_clear_errors_w8a8,     read_clear_errors_tma,
                                                         read_clear_errors_selftest, read_clear_errors_gemv};
    for (auto r : readers) {
        cudaError_t ei = r(bits, s);
        if (ei != cudaSuccess) e = ei;
    }
    return e == cudaSuccess ? MMQ_OK : cuda_fail(e, "mmq_read_device_errors");
}

const char* mmq_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
