// quantize.cu -- q8_1 activation quantizer for sm_103a.
//
// Per 32-value block: amax = max|x|, d = amax/127, q = round-half-even(x/d) (correctly rounded f32
// division), s = d * sum(q)  ("08 · R1 — int8 MMQ prefill GEMM", §2.2 q8_1 activation pipeline, and
// the §3.2 reference quantizer; f32 scale, the block sum produced in the same pass).
// Output layout (include/mmq.h): int8 q[M][K], float2 (d, s)[M][K/32], then the tensor-core shadow:
// fp16 h[M][K] = q exactly, and the block-major copies d^T, s^T [K/32][Mp] that the TMA-fed GEMM loads
// per 128-token tile.
//
// 4 bytes read per value; 1.25 bytes of q8_1 blocks and 2.25 bytes of shadow (fp16 codes, block-major
// scales) written.  Eight lanes own one block (one float4 each); amax and sum(q) are warp-shuffle
// reductions over the eight lanes; every lane stores its four codes as one 32-bit word, so a warp writes
// 128 contiguous bytes per block quad.  The kernel is issue-bound, so it avoids divisions: d comes from an
// exact FMA correction step (div127), the codes from x * (1/d) with the correctly rounded quotient formed
// only next to a rounding boundary (q8_code_f), and the row and column of a block step forward from one
// division per warp iteration (21.1 -> 16.6 us for 2048 x 4096 values, bit-identical results).
#include <cstdint>
#include "internal.h"
#include <cuda_fp16.h>
#include "mmq_device.cuh"

namespace mmq {

constexpr int QZ_UNROLL = 4;      // blocks per 8-lane group per iteration (loads in flight)

__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// four codes -> four fp16 (exact)
__device__ __forceinline__ uint2 codes_to_f16x4(int q0, int q1, int q2, int q3) {
    const __half2 a = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
    const __half2 b = __halves2half2(__int2half_rn(q2), __int2half_rn(q3));
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// d = amax / 127, correctly rounded, without a division: q0 = amax * r with r the rounded 1/127, then one
// correction step q0 + r * (amax - 127 q0) with the residual formed exactly by an FMA (Markstein's
// correction, "Computation of elementary functions on the IBM RISC System/6000 processor", 1990).  Checked
// equal to the IEEE quotient for every non-negative finite amax (tests/test_div127_exhaustive.py).
__device__ __forceinline__ float div127(float a) {
    constexpr float r = 1.0f / 127.0f;
    const float q0 = __fmul_rn(a, r);
    return __fmaf_rn(__fmaf_rn(-q0, 127.0f, a), r, q0);
}

// The code of x in a block of scale d > 0: round-half-even of the correctly rounded f32 quotient x/d,
// clamped to [-127, 127].  t = x * inv, with inv within 2 ulp of 1/d (__fdividef's bound for normal d),
// lies within |x/d| * (2^-22 + 2^-24) of x/d, and the correctly rounded quotient within |x/d| * 2^-24; for
// |x/d| <= 127.5 the two differ by less than 4.6e-5.  Rounding to an integer only changes at
// half-integers, so when t is more than 1e-4 away from the nearest half-integer, rint(t) is the code the
// definition gives; otherwise (and for subnormal d, where inv is +inf and t not finite) the quotient is
// formed exactly.  The clamp to [-127, 127] can only act on that exact path: for a normal d,
// |x/d| <= 127 / (1 - 2^-24) and |t| stays below 127.5.  In: t, x, d; out: the rounded code as a float
// (an integer in [-127, 127]; a zero code is +0, so its fp16 copy is the integer's).
__device__ __forceinline__ float q8_code_f(float t, float x, float d) {
    float r = rintf(t);
    if (!(fabsf(t - r) <= 0.4999f)) r = fminf(127.0f, fmaxf(-127.0f, rintf(__fdiv_rn(x, d))));
    return __fadd_rn(r, 0.0f);
}

__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float4* __restrict__ x, uint32_t* __restrict__ q,
                                                           float2* __restrict__ ds, uint2* __restrict__ h,
                                                           float* __restrict__ dT,
                                                           float* __restrict__ sT, int kb, int Mp,
                                                           int nblk) {
    const int lane = threadIdx.x & 31, sub = lane & 7, grp = lane >> 3;
    const int warp_id = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    pdl_wait();
    pdl_trigger();
    // one warp iteration covers 4 groups x QZ_UNROLL blocks
    for (int base = warp_id * 4 * QZ_UNROLL; base < nblk; base += nwarps * 4 * QZ_UNROLL) {
        // row and block index of this iteration's first block (one division per iteration; the iteration's
        // 4 * QZ_UNROLL blocks step forward from it)
        const int m_base = base / kb, b_base = base - m_base * kb;
        float4 v[QZ_UNROLL];
#pragma unroll
        for (int u = 0; u < QZ_UNROLL; u++) {
            const int blk = base + u * 4 + grp;
            v[u] = blk < nblk ? ld_stream_f4(x + blk * 8 + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < QZ_UNROLL; u++) {
            const int blk = base + u * 4 + grp;
            float a = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float d = div127(a);
            float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
            if (d != 0.0f) {
                const float inv = d >= 1.17549435e-38f ? __fdividef(1.0f, d) : __int_as_float(0x7f800000);
                r0 = q8_code_f(__fmul_rn(v[u].x, inv), v[u].x, d);
                r1 = q8_code_f(__fmul_rn(v[u].y, inv), v[u].y, d);
                r2 = q8_code_f(__fmul_rn(v[u].z, inv), v[u].z, d);
                r3 = q8_code_f(__fmul_rn(v[u].w, inv), v[u].w, d);
            }
            const int q0 = (int)r0, q1 = (int)r1, q2 = (int)r2, q3 = (int)r3;
            int sum = q0 + q1 + q2 + q3;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if (blk < nblk) {
                q[blk * 8 + sub] = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) |
                                   ((uint32_t)(q2 & 0xff) << 16) | ((uint32_t)(q3 & 0xff) << 24);
                // the codes are integers of magnitude <= 127: exact in fp16
                const __half2 h01 = __floats2half2_rn(r0, r1), h23 = __floats2half2_rn(r2, r3);
                h[blk * 8 + sub] = make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                                              *reinterpret_cast<const uint32_t*>(&h23));
                if (sub == 0) {
                    const float sv = __fmul_rn(d, (float)sum);
                    ds[blk] = make_float2(d, sv);
                    int m = m_base, b = b_base + (blk - base);
                    while (b >= kb) {                  // at most once for rows of 16 blocks or more
                        b -= kb;
                        m++;
                    }
                    dT[b * Mp + m] = d;
                    sT[b * Mp + m] = sv;
                    for (int mm = m + 1; mm < Mp && blk + kb >= nblk; mm++) {   // pad columns: zero
                        dT[b * Mp + mm] = 0.f;
                        sT[b * Mp + mm] = 0.f;
                    }
                }
            }
        }
    }
}

cudaError_t run_quantize_q8_1(const float* x, long long M, long long K, void* xq, cudaStream_t s) {
    const long long nblk = M * K / 32;
    if (nblk == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long warps_needed = (nblk + 4 * QZ_UNROLL - 1) / (4 * QZ_UNROLL);
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = (long long)sms * 8;              // 8 x 256 threads resident per SM
    if (blocks > cap) blocks = cap;
    uint8_t* base = static_cast<uint8_t*>(xq);
    const Q81Layout L = q81_layout(M, K);
    return launch_pdl(quantize_q8_1_kernel, dim3((unsigned)blocks), dim3(256), s,
        reinterpret_cast<const float4*>(x), reinterpret_cast<uint32_t*>(base), reinterpret_cast<float2*>(base + L.ds),
        reinterpret_cast<uint2*>(base + L.h), reinterpret_cast<float*>(base + L.dT),
        reinterpret_cast<float*>(base + L.sT), (int)(K / 32), (int)L.Mp, (int)nblk);
}

// Derived sections from existing q8_1 blocks: eight lanes per block, one 32-bit word of codes each.
__global__ void __launch_bounds__(256) prepare_q8_1_kernel(const uint32_t* __restrict__ q,
                                                          const float2* __restrict__ ds, uint2* __restrict__ h,
                                                          float* __restrict__ dT,
                                                          float* __restrict__ sT, int kb, long long Mp,
                                                          long long nblk) {
    const long long stride = (gridDim.x * (long long)blockDim.x) >> 3;
    const int sub = threadIdx.x & 7;
    for (long long blk = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 3; blk < nblk; blk += stride) {
        const uint32_t w = q[blk * 8 + sub];
        h[blk * 8 + sub] = codes_to_f16x4((int)(int8_t)(w & 0xff), (int)(int8_t)((w >> 8) & 0xff),
                                          (int)(int8_t)((w >> 16) & 0xff), (int)(int8_t)(w >> 24));
        if (sub == 0) {
            const float2 v = ds[blk];
            const long long m = blk / kb, b = blk - m * kb;
            dT[b * Mp + m] = v.x;
            sT[b * Mp + m] = v.y;
            for (long long mm = m + 1; mm < Mp && blk + kb >= nblk; mm++) {   // pad columns: zero
                dT[b * Mp + mm] = 0.f;
                sT[b * Mp + mm] = 0.f;
            }
        }
    }
}

cudaError_t run_prepare_q8_1(void* xq, long long M, long long K, cudaStream_t s) {
    const long long nblk = M * K / 32;
    if (nblk == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (nblk * 8 + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    uint8_t* base = static_cast<uint8_t*>(xq);
    const Q81Layout L = q81_layout(M, K);
    prepare_q8_1_kernel<<<(unsigned)blocks, 256, 0, s>>>(
        reinterpret_cast<const uint32_t*>(base), reinterpret_cast<const float2*>(base + L.ds),
        reinterpret_cast<uint2*>(base + L.h), reinterpret_cast<float*>(base + L.dT),
        reinterpret_cast<float*>(base + L.sT), (int)(K / 32), L.Mp, nblk);
    return cudaGetLastError();
}

MMQ_DEFINE_ERROR_READER(quantize)

}  // namespace mmq
