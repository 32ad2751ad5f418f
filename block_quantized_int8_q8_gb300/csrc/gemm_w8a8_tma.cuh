// gemm_w8a8_tma.cuh -- TMA-fed per-channel W8A8 GEMM ("INT8 W8A8 GEMM — Prefill", §1-§2):
// I[m,n] = sum_{k<K} x[m,k] * w[n,k] exactly, out = bf16_rne(((float)I * xs[m]) * ws[n]).
//
// One CTA per 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N), all of K:
//   * loader warp (one thread): per 64-k stage, two TMA loads of raw int8 rows (128 weight rows and
//     128 token rows, 64 bytes each) into a four-slot raw ring, with the 64-byte swizzle (16-byte piece p
//     of row r lands at piece p ^ ((r/2) % 4));
//   * eight converter warps (one row per thread: threads 0..127 weight rows, 128..255 token rows):
//     widen the row's 64 int8 values exactly to fp16 (integers |v| <= 127) into the 128B-swizzled
//     K-major operand ring.  Thanks to the swizzle both the raw reads (8 rows of an 8-lane phase cover 8
//     distinct 16-byte bank groups) and the 128B-swizzled operand stores are conflict-free;
//   * MMA warp: four tcgen05.mma kind::f16 (M=128, N=128, K=16) per stage into one of two 1024-k chunk
//     accumulators: |partial sum| < 1024 * 127 * 127 < 2^24, so the f32 accumulator is exact;
//   * eight epilogue warps (two per TMEM lane quarter, 64 tokens each): after every chunk, read it in the
//     16x256b fragment layout, convert exactly to int32 and add; at the end apply the bf16 epilogue in
//     the written order ((float)I * xs) * ws with round-to-nearest steps.
// The epilogue does no per-block work, so the kernel is bound by the MMA and the conversion.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include "gemm_tma.cuh"

namespace mmq {
namespace w8tma {

using tma::mbar_arrive_expect_tx;
using tma::tma_prefetch_desc;

constexpr int STAGES = 4;             // operand ring
constexpr int RAW_SLOTS = 4;          // raw int8 ring (one 64-k stage per slot)
constexpr int CHUNK_STAGES = 16;      // 1024-k chunk accumulators
constexpr int NCB = 2;                // chunk accumulators (128 TMEM columns each)
constexpr int EPI_WARPS = 8;
constexpr int CONV_WARPS = 8;
constexpr int CONV0 = EPI_WARPS;
constexpr int MMA_W = CONV0 + CONV_WARPS;
constexpr int LOAD_W = MMA_W + 1;
constexpr int NTHREADS = (LOAD_W + 1) * 32;
constexpr int RAW_ROW = 64;                               // bytes per row per stage
constexpr int RAW_HALF = 128 * RAW_ROW;                   // weight rows, then token rows
constexpr int RAW_SLOT = 2 * RAW_HALF;

struct Smem {
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + STAGES * A_STAGE_BYTES;
    static constexpr int raw_off = b_off + STAGES * B_STAGE_BYTES;
    static constexpr int bar_off = raw_off + RAW_SLOTS * RAW_SLOT;
    static constexpr int n_bars = 2 * STAGES + 2 * RAW_SLOTS + 2 * NCB + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;     // tmem slot, abort flag
    static constexpr int total = misc_off + 16;
    static constexpr int alloc = total + 1024;
    static_assert(alloc <= 232448, "shared memory budget");
};

struct Bar {
    uint32_t b0;
    __device__ uint32_t full(int i) const { return b0 + 8u * i; }
    __device__ uint32_t empty(int i) const { return b0 + 8u * (STAGES + i); }
    __device__ uint32_t rfull(int i) const { return b0 + 8u * (2 * STAGES + i); }
    __device__ uint32_t rempty(int i) const { return b0 + 8u * (2 * STAGES + RAW_SLOTS + i); }
    __device__ uint32_t accf(int i) const { return b0 + 8u * (2 * STAGES + 2 * RAW_SLOTS + i); }
    __device__ uint32_t acce(int i) const { return b0 + 8u * (2 * STAGES + 2 * RAW_SLOTS + NCB + i); }
    __device__ uint32_t done() const { return b0 + 8u * (2 * STAGES + 2 * RAW_SLOTS + 2 * NCB); }
};

__global__ void __launch_bounds__(NTHREADS, 1)
    mmq_w8a8_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                        const float* __restrict__ ws, const float* __restrict__ xs, __nv_bfloat16* __restrict__ out,
                        int M, int N, int K) {
    using L = Smem;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntn = (N + BM - 1) / BM;
    const int n0 = (blockIdx.x % ntn) * BM, m0 = (blockIdx.x / ntn) * BN;
    const Bar B{sb + L::bar_off};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
    const int nst = K / BK;

    if (warp == MMA_W) {
        if (lane == 0) {
            for (int i = 0; i < STAGES; i++) {
                mbar_init(B.full(i), CONV_WARPS);
                mbar_init(B.empty(i), 1);
            }
            for (int i = 0; i < RAW_SLOTS; i++) {
                mbar_init(B.rfull(i), 1);
                mbar_init(B.rempty(i), CONV_WARPS);
            }
            for (int i = 0; i < NCB; i++) {
                mbar_init(B.accf(i), 1);
                mbar_init(B.acce(i), EPI_WARPS);
            }
            mbar_init(B.done(), 1);
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), NCB * BN);
        tmem_relinquish();
    } else if (warp == LOAD_W && lane == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == LOAD_W) {
        // =========================================================== TMA loader
        if (lane == 0) {
            for (int s = 0; s < nst; s++) {
                const int rs = s % RAW_SLOTS;
                if (!mbar_wait_relaxed(B.rempty(rs), ((s / RAW_SLOTS) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(B.rfull(rs), RAW_SLOT);
                const uint32_t dst = sb + L::raw_off + rs * RAW_SLOT;
                tma::tma_load_2d(dst, &tm_w, BK * s, n0, B.rfull(rs));
                tma::tma_load_2d(dst + RAW_HALF, &tm_x, BK * s, m0, B.rfull(rs));
            }
        }
        __syncwarp();
    } else if (warp >= CONV0 && warp < MMA_W) {
        // =========================================================== converters
        const int ct = (warp - CONV0) * 32 + lane;             // 0..255
        const bool tok = ct >= 128;
        const int row = ct & 127;
        const uint32_t dst0 = sb + (tok ? L::b_off : L::a_off);
        for (int s = 0; s < nst; s++) {
            const int rs = s % RAW_SLOTS, slot = s % STAGES;
            if (!mbar_wait_relaxed(B.rfull(rs), (s / RAW_SLOTS) & 1, abort_flag) ||
                !mbar_wait_relaxed(B.empty(slot), ((s / STAGES) & 1) ^ 1, abort_flag))
                break;
            const uint32_t src = sb + L::raw_off + rs * RAW_SLOT + (tok ? RAW_HALF : 0) + row * RAW_ROW;
            const uint32_t dst = dst0 + slot * A_STAGE_BYTES;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint4 v = ld_shared_u4(src + 16 * (c ^ ((row >> 1) & 3)));   // 64-byte swizzle
                uint32_t h[8];
                s8x4_to_f16x4(v.x, h[0], h[1]);
                s8x4_to_f16x4(v.y, h[2], h[3]);
                s8x4_to_f16x4(v.z, h[4], h[5]);
                s8x4_to_f16x4(v.w, h[6], h[7]);
                st_shared_v4(dst + sw128_off(row, 2 * c), h[0], h[1], h[2], h[3]);
                st_shared_v4(dst + sw128_off(row, 2 * c + 1), h[4], h[5], h[6], h[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B.full(slot));
                mbar_arrive(B.rempty(rs));
            }
        }
    } else if (warp == MMA_W) {
        // =========================================================== MMA issuer
        const uint32_t idesc = idesc_f16_f32(BM, BN);
        for (int s = 0; s < nst; s++) {
            if (*abort_flag) break;
            const int slot = s % STAGES, ch = s / CHUNK_STAGES, cb = ch & (NCB - 1);
            const bool first = s % CHUNK_STAGES == 0;
            const bool last = s % CHUNK_STAGES == CHUNK_STAGES - 1 || s == nst - 1;
            if (!mbar_wait(B.full(slot), (s / STAGES) & 1, abort_flag)) break;
            if (first) mbar_wait(B.acce(cb), ((ch / NCB) & 1) ^ 1, abort_flag);
            tc_fence_after();
            const uint64_t ad0 = sdesc_sw128(sb + L::a_off + slot * A_STAGE_BYTES);
            const uint64_t bd0 = sdesc_sw128(sb + L::b_off + slot * B_STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < 4; j++)
                if (elect_one()) umma_f16(tmem_base + cb * BN, ad0 + 2 * j, bd0 + 2 * j, idesc, (first && j == 0) ? 0u : 1u);
            if (elect_one()) {
                if (last) umma_commit(B.accf(cb));
                umma_commit(B.empty(slot));
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(B.done());
        __syncwarp();
        mbar_wait_final(B.done(), 0);
        __syncwarp();
    } else {
        // =========================================================== epilogue
        // warp: TMEM lane quarter q (weight rows 32q..), tokens 64*ch .. 64*ch+63 as two 32-column groups.
        // 16x256b fragment: per 16-lane half h and column group g, thread t holds rows 16h + 8e + t/4 and
        // tokens 32g + 8j + 2(t%4) + c.
        const int q = warp & 3, ch = warp >> 2;
        const int tq = lane >> 2, tc = lane & 3;
        int32_t acc[2][2][16];                  // [half][group][4e*... ] = v layout: 4j + 2e + c
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int g = 0; g < 2; g++)
#pragma unroll
                for (int r = 0; r < 16; r++) acc[h][g][r] = 0;
        const int nch = (nst + CHUNK_STAGES - 1) / CHUNK_STAGES;
        for (int c2 = 0; c2 < nch; c2++) {
            const int cb = c2 & (NCB - 1);
            if (!mbar_wait(B.accf(cb), (c2 / NCB) & 1, abort_flag)) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; h++) {
#pragma unroll
                for (int g = 0; g < 2; g++) {
                    uint32_t v[16];
                    tmem_ld_16x256b_x4(tmem_base + ((uint32_t)(32 * q + 16 * h) << 16) + cb * BN + 64 * ch + 32 * g, v);
                    tmem_ld_wait(v);
#pragma unroll
                    for (int r = 0; r < 16; r++) acc[h][g][r] += __float2int_rn(__uint_as_float(v[r]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.acce(cb));
        }
        // ---- store: out = bf16(((float)I * xs[m]) * ws[n])
#pragma unroll
        for (int h = 0; h < 2; h++) {
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int n = n0 + 32 * q + 16 * h + 8 * e + tq;
                if (n >= N) continue;
                const float wsn = __ldg(ws + n);
#pragma unroll
                for (int g = 0; g < 2; g++) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
#pragma unroll
                        for (int cc = 0; cc < 2; cc++) {
                            const int m = m0 + 64 * ch + 32 * g + 8 * j + 2 * tc + cc;
                            if (m < M) {
                                const float t = __fmul_rn((float)acc[h][g][4 * j + 2 * e + cc], __ldg(xs + m));
                                out[(long long)m * N + n] = __float2bfloat16_rn(__fmul_rn(t, wsn));
                            }
                        }
                    }
                }
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < tma::ABORT_DRAIN_CYCLES) {
        }
    }
    tc_fence_after();
    if (warp == MMA_W) tmem_dealloc(tmem_base, NCB * BN);
}

}  // namespace w8tma
}  // namespace mmq
