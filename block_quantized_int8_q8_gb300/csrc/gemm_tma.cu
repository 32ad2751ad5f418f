// gemm_tma.cu -- host side of the TMA-fed dense MMQ kernel (gemm_tma.cuh): tensor maps and launch.
//
// Four tensor maps per call, encoded on the host with the driver's cuTensorMapEncodeTiled (looked up
// once through the runtime's driver entry-point query, so the library needs no -lcuda):
//   raw  : the weight bytes [N][row_bytes]; box 128 rows x U*16 bytes (one raw super-stage), of uint8
//          elements where that fits a box dimension (Q4_0, Q4_K, Q6_K), else of uint32 elements (Q8_0,
//          IQ1_M); rows past N read as zeros.  Q6_K's 224-byte
//          super-block is read as a 240-byte box (an odd number of 16-byte units in shared memory).
//   b    : the q8_1 shadow's fp16 codes [M][K]; box 128 tokens x 64 k, 128-byte swizzle (the MMA's
//          K-major operand layout); tokens past M read as zeros.
//   xd/xs: the block-major scales d^T, s^T [K/32][Mp]; box 2 blocks x 128 tokens.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>
#include "gemm_tma.cuh"
#include "gemm_w8a8_tma.cuh"
#include "internal.h"

namespace mmq {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Multiprocessor count of the current device (looked up once per device).
int sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

// Largest K split (4, 2 or 1) of a MoE tail tile: parts are cut at raw super-stage boundaries, so a tile
// splits into at most as many parts as it has super-stages.
int moe_kparts(int wt, long long K) {
    const long long nsup = K / BK / (wt == WT_IQ1_M ? tma::Geom<WT_IQ1_M>::SS : tma::Geom<WT_Q4_0>::SS);
    return nsup >= 4 ? 4 : (nsup >= 2 ? 2 : 1);
}

template <int WT>
cudaError_t launch(const TmaGemmArgs& a, cudaStream_t stream, bool dbg) {
    using L = tma::Smem<WT>;
    constexpr int U = tma::Geom<WT>::U;
    CUtensorMap tm_raw, tm_b, tm_xd, tm_xs;
    const long long wrows = a.E * a.N;      // MoE: every expert's rows, back to back
    {
        // one 2-D box of whole row chunks: bytes where the chunk fits a box dimension (256 elements),
        // else 4-byte elements (Q8_0 272 B, IQ1_M 304 B per row; row strides and chunk offsets are
        // multiples of 16 bytes).  A box of 16-byte units along a third dimension lands the same bytes in
        // the same place but as many more, smaller TMA requests (measured: the 64x256x1024 Q8_0 GEMM 14 %
        // slower, IQ1_M 1-4 % slower).
        const bool words = U * 16 > 256;
        const cuuint64_t dims[2] = {(cuuint64_t)(words ? a.w_row_bytes / 4 : a.w_row_bytes), (cuuint64_t)wrows};
        const cuuint64_t strides[1] = {(cuuint64_t)a.w_row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)(words ? U * 4 : U * 16), (cuuint32_t)BM};
        if (!encode(&tm_raw, words ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.W, dims,
                    strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        const cuuint32_t box[2] = {BK, BN};
        if (!encode(&tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.xh, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.M, (cuuint64_t)(a.K / 32)};
        const cuuint64_t strides[1] = {(cuuint64_t)a.Mp * 4};
        const cuuint32_t box[2] = {BN, 2};
        if (!encode(&tm_xd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.dT, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        if (!encode(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.sT, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    auto kern = tma::mmq_gemm_tma_kernel<WT, false>;
    auto kern_moe = tma::mmq_gemm_tma_kernel<WT, true>;
    auto kern_dbg = tma::mmq_gemm_tma_kernel<WT, false, true>;
    // at most 64 tokens: four converter warps (the same kernel for the types that always use four)
    constexpr int kSmallConv = 4;
    constexpr long long kSmallM = 64;
    auto kern_small = tma::mmq_gemm_tma_kernel<WT, false, false, kSmallConv>;
    static bool configured[64] = {};      // per instantiation and device; the attribute is per function
    bool& done = device_flag(configured);
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern_moe, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern_dbg, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern_small, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
        if (e != cudaSuccess) return e;
        done = true;
    }
    const long long ntn = (a.N + BM - 1) / BM;
    if (dbg) {                              // block sums: one CTA per tile, whole K range
        const long long T = ntn * ((a.M + BN - 1) / BN);
        kern_dbg<<<(unsigned)T, tma::Warps<WT>::kThreads, L::alloc, stream>>>(
            tm_raw, tm_b, tm_xd, tm_xs, a.out, (int)a.M, (int)a.N, (int)a.K, (int)ntn, (int)T, 0, tma::MoeTiles{});
        return cudaGetLastError();
    }
    if (a.work != nullptr) {                // MoE: one CTA per (work item, weight-row tile) + tail parts
        const tma::MoeTiles moe{a.work, a.nwork, a.gstart, a.rowlist, sm_count(), moe_kparts(WT, a.K)};
        const long long ctas = ntn * a.max_work + moe.sms;
        if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;   // beyond the grid's x extent
        kern_moe<<<(unsigned)ctas, tma::Warps<WT>::kThreads, L::alloc, stream>>>(
            tm_raw, tm_b, tm_xd, tm_xs, a.out, (int)a.M, (int)a.N, (int)a.K, (int)ntn, (int)ctas, 0, moe);
        return cudaGetLastError();
    }
    // Small grids: when all tiles fit in half the SMs or fewer, every tile runs as P = 2..16 parts of its K
    // range (P tiles' worth of CTAs, each 1/P of the stages) adding into a zeroed output.
    // Tail split: otherwise, when the last wave of whole tiles would leave at least half the SMs idle, the
    // last token-tile rows run as two K halves each; their output rows are zeroed first.
    const long long ntm = (a.M + BN - 1) / BN, T = ntn * ntm;
    const int sms = sm_count();
    const long long nst = a.K / BK;
    constexpr int SS = tma::Geom<WT>::SS;
    const long long nsup = nst / SS;                           // parts are cut at super-stage boundaries
    long long split_rows = 0;
    int lgp = 1;
    if (sms > 0 && 2 * T <= sms && nsup >= 2) {
        lgp = 1;
        while (lgp < 4 && (T << (lgp + 1)) <= sms && (2ll << lgp) <= nsup) lgp++;
        split_rows = ntm;
    } else if (sms > 0 && T > sms && nsup >= 2) {
        const long long r = T - (T - 1) / sms * sms;          // tiles in the last wave
        if (2 * r <= sms) split_rows = (r + ntn - 1) / ntn;
        if (split_rows >= ntm) split_rows = 0;
    }
    const long long nfull = T - split_rows * ntn;
    if (split_rows > 0) {
        const long long m_begin = (ntm - split_rows) * BN;
        const cudaError_t e = cudaMemsetAsync(a.out + m_begin * a.N, 0, (size_t)((a.M - m_begin) * a.N) * sizeof(float),
                                              stream);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((unsigned)(nfull + (split_rows * ntn << lgp)));
    if (a.M <= kSmallM)
        kern_small<<<grid, tma::Warps<WT, kSmallConv>::kThreads, L::alloc, stream>>>(
            tm_raw, tm_b, tm_xd, tm_xs, a.out, (int)a.M, (int)a.N, (int)a.K, (int)ntn, (int)nfull, lgp, tma::MoeTiles{});
    else
        kern<<<grid, tma::Warps<WT>::kThreads, L::alloc, stream>>>(tm_raw, tm_b, tm_xd, tm_xs, a.out, (int)a.M, (int)a.N,
                                                        (int)a.K, (int)ntn, (int)nfull, lgp, tma::MoeTiles{});
    return cudaGetLastError();
}

// Raw int8 rows [rows][K]; box 128 rows x 64 bytes (one 64-k stage) with the 64-byte swizzle.
bool encode_int8_rows(CUtensorMap* m, const void* base, long long rows, long long K) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {64, 128};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

cudaError_t run_gemm_w8a8_tma(const void* W, const void* X, void* out, long long M, long long N, long long K,
                              cudaStream_t stream) {
    CUtensorMap tm_w, tm_x;
    if (!encode_int8_rows(&tm_w, W, N, K) || !encode_int8_rows(&tm_x, X, M, K)) return cudaErrorInvalidValue;
    const float* ws = reinterpret_cast<const float*>(static_cast<const uint8_t*>(W) + N * K);
    const float* xs = reinterpret_cast<const float*>(static_cast<const uint8_t*>(X) + M * K);
    auto kern = w8tma::mmq_w8a8_tma_kernel;
    static bool configured[64] = {};
    bool& done = device_flag(configured);
    if (!done) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, w8tma::Smem::alloc);
        if (e != cudaSuccess) return e;
        done = true;
    }
    const long long tiles = ((N + BM - 1) / BM) * ((M + BN - 1) / BN);
    kern<<<(unsigned)tiles, w8tma::NTHREADS, w8tma::Smem::alloc, stream>>>(
        tm_w, tm_x, ws, xs, static_cast<__nv_bfloat16*>(out), (int)M, (int)N, (int)K);
    return cudaGetLastError();
}

// MoE gather: block (w, c) copies rows GATHER_ROWS*c .. GATHER_ROWS*(c+1) - 1 of work item w.  The
// item's first gathered row is the 4-aligned sum of the preceding items' counts, so every item starts on
// a 16-byte boundary of the block-major scales (the alignment a TMA box coordinate needs).
constexpr int GATHER_ROWS = 8;          // eight rows per block: enough blocks in flight to fill every SM
__global__ void __launch_bounds__(256) moe_gather_kernel(const MoeGatherArgs g) {
    const int w = blockIdx.x;
    if (w >= *g.nwork) return;
    const int row0 = blockIdx.y * GATHER_ROWS;
    const int count = g.work[3 * w + 2];
    if (row0 >= count) return;
    __shared__ int s_start;
    __shared__ int s_tok[GATHER_ROWS];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int acc = 0;
        for (int i = lane; i < w; i += 32) acc += (g.work[3 * i + 2] + 3) & ~3;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            s_start = acc;
            if (blockIdx.y == 0) g.gstart[w] = acc;
        }
    } else if (threadIdx.x < 32 + GATHER_ROWS) {
        const int j = row0 + lane;
        s_tok[lane] = j < count ? g.rowlist[g.work[3 * w + 1] + j] / g.slots : -1;
    }
    __syncthreads();
    const int nrows = min(GATHER_ROWS, count - row0);
    const long long dst0 = s_start + row0;
    // fp16 codes: thread t copies 16-byte column t (+256...) of eight rows at a time (eight loads in flight)
    const long long kv = g.K / 8;
    const uint4* __restrict__ xh = static_cast<const uint4*>(g.xh);
    uint4* __restrict__ xg = static_cast<uint4*>(g.xg);
    for (long long cidx = threadIdx.x; cidx < kv; cidx += blockDim.x) {
        for (int j0 = 0; j0 < nrows; j0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++)
                if (j0 + u < nrows) v[u] = xh[(long long)s_tok[j0 + u] * kv + cidx];
#pragma unroll
            for (int u = 0; u < 8; u++)
                if (j0 + u < nrows) xg[(dst0 + j0 + u) * kv + cidx] = v[u];
        }
    }
    // outputs of tail tiles computed in K parts (they add into zero): this item's rows, those tiles' columns
    {
        int nf, r;
        const int ntn = (int)((g.N + BM - 1) / BM);
        if (tma::tail_split(*g.nwork * ntn, g.sms, g.kparts, nf, r) > 0) {
            for (int rt = 0; rt < ntn; rt++) {
                if (w * ntn + rt < nf) continue;
                const long long c0 = (long long)rt * BM, nc = min((long long)BM, g.N - c0);
                for (int j = 0; j < nrows; j++) {
                    float* o = g.out + (long long)g.rowlist[g.work[3 * w + 1] + row0 + j] * g.N + c0;
                    for (long long i = threadIdx.x; i < nc; i += blockDim.x) o[i] = 0.f;
                }
            }
        }
    }
    // block scales: lanes over the rows (one 128-byte segment per block index), warps over the blocks,
    // four blocks in flight per lane
    const long long kb = g.K / 32;
    if (lane < nrows) {
        const int tok = s_tok[lane];
        const long long nw = blockDim.x >> 5;
        for (long long b0 = threadIdx.x >> 5; b0 < kb; b0 += 4 * nw) {
            float dv[4], sv[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const long long b = b0 + u * nw;
                if (b < kb) {
                    dv[u] = g.dT[b * g.Mp + tok];
                    sv[u] = g.sT[b * g.Mp + tok];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const long long b = b0 + u * nw;
                if (b < kb) {
                    g.dTg[b * g.Rg + dst0 + lane] = dv[u];
                    g.sTg[b * g.Rg + dst0 + lane] = sv[u];
                }
            }
        }
    }
}

cudaError_t run_moe_gather(const MoeGatherArgs& gin, int wt, cudaStream_t s) {
    MoeGatherArgs g = gin;
    g.sms = sm_count();
    g.kparts = moe_kparts(wt, g.K);
    const dim3 grid((unsigned)g.max_work, (unsigned)((BN + GATHER_ROWS - 1) / GATHER_ROWS));
    moe_gather_kernel<<<grid, 256, 0, s>>>(g);
    return cudaGetLastError();
}

bool tma_gemm_supported(int wt, long long K) {
    if (wt == WT_IQ1_M) return K % 1024 == 0;
    return (wt == WT_Q8_0 || wt == WT_Q4_0 || wt == WT_Q4_K || wt == WT_Q6_K) && K % 256 == 0;
}

cudaError_t run_gemm_tma(int wt, const TmaGemmArgs& a, cudaStream_t s, bool block_sums) {
    switch (wt) {
        case WT_Q8_0: return launch<WT_Q8_0>(a, s, block_sums);
        case WT_Q4_0: return launch<WT_Q4_0>(a, s, block_sums);
        case WT_Q4_K: return launch<WT_Q4_K>(a, s, block_sums);
        case WT_IQ1_M: return launch<WT_IQ1_M>(a, s, block_sums);
        case WT_Q6_K: return launch<WT_Q6_K>(a, s, block_sums);
    }
    return cudaErrorInvalidValue;
}

MMQ_DEFINE_ERROR_READER(tma)

}  // namespace mmq
