// gemm.cuh -- block-quantized int8 MMQ on sm_103a tensor cores.
//
// Computes out[m,n] = sum_b scale(m,n,b) * I[m,n,b] with the exact per-block integer dot
// I[m,n,b] = sum_{k in b} xq[m,k] * wq[n,k]  ("A Negative Result on int8 Tensor-Core MMQ", §2;
// "08 · R1 — int8 MMQ prefill GEMM", §2.1 and §3.2).
//
// GB300 design (the pages' kernels target mma.sync on sm_80..sm_121; this one is written for sm_103a):
//   * sm_103a has no tcgen05 int8 MMA kind, and its legacy int8 mma.sync rate is a small fraction of
//     the fp16 tensor rate, so the integer codes are converted EXACTLY to fp16 (integers of magnitude
//     <= 2048 are exact in fp16) and contracted with tcgen05.mma kind::f16 into f32 TMEM
//     accumulators.  Every product is an integer < 2^14 and every partial sum of one block an integer
//     < 2^24, so the f32 accumulator holds the exact int32 block dot.
//   * One CTA computes a 128 (weight rows, MMA M, TMEM lanes) x 128 (tokens, MMA N) tile over all K.
//     Each 32-k block is contracted into its own TMEM accumulator (4 buffers of 128 columns rotate),
//     so the tensor core runs ahead while the epilogue warps rescale the previous blocks.
//   * Warp roles: warps 0-7 epilogue (rescale in registers, store), warps 8-11 producers (load raw
//     weight blocks and q8_1 codes, unpack to fp16 in 128B-swizzled K-major smem tiles), warp 12
//     issues the MMAs (one elected thread) and owns the TMEM allocation.
//   * The f32 scale correction acc += (xd[m,b] * wd[n,b]) * I stays in registers after a tcgen05.ld,
//     never through a shared-memory round trip of the accumulator ("A Negative Result", §2-§4).
//   * IQ1_M: the per-16 sub-scale (2s+1) is folded into the fp16 operand together with the sign fold
//     8g±1 ("CUDA: add IQ1_M to MMQ", Design), giving exact integers |v| <= 135, so one 32-k
//     accumulator carries both halves and the block scale is xd * d/8.
//   * W8A8 ("INT8 W8A8 GEMM — Prefill", §1): no per-block scale; the tensor core accumulates 1024-k
//     chunks (|partial| < 1024*127*128 < 2^24, exact), the epilogue adds them as int32 and applies
//     out = bf16(((float)I * xs[m]) * ws[n]).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "mmq_device.cuh"
#include "internal.h"

namespace mmq {

// Scale-product operands (one 16-byte row per weight row / token per block, K-major, no swizzle).
// The K=16 MMA reads two 8-element K chunks; the leading byte offset is 0 so both chunks are the same
// 16 bytes, every product is counted twice, and the weight-side pieces carry a factor 1/2 (exact).
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)0 << 16;                           // leading byte offset: both K chunks alias
    d |= (uint64_t)(128 >> 4) << 32;                  // stride byte offset: 8 rows x 16 B
    d |= (uint64_t)1 << 46;                           // fixed 0b001 field
    return d;                                         // swizzle mode 0: none
}

// Instruction descriptor, kind::f16 with bf16 A and B, f32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// bf16 record {x1, x1, x2, x2, x3, x3, 0, 0} with x1 + x2 + x3 = d exactly: x1 keeps d's top 16 bits,
// x2 those of the remainder, and the last remainder has at most 8 significant bits.
__device__ __forceinline__ uint4 split3_record(float d) {
    const float x1 = __uint_as_float(__float_as_uint(d) & 0xFFFF0000u);
    const float r1 = __fsub_rn(d, x1);
    const float x2 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
    const float x3 = __fsub_rn(r1, x2);
    const uint32_t h1 = __float_as_uint(x1) >> 16, h2 = __float_as_uint(x2) >> 16, h3 = __float_as_uint(x3) >> 16;
    return make_uint4(h1 | (h1 << 16), h2 | (h2 << 16), h3 | (h3 << 16), 0u);
}

// bf16 record {w1, w2, w1, w2, w1, w2, 0, 0} with w1 + w2 = v exactly (v has at most 16 significant
// bits: an f16 scale, halved); w1 keeps v's top 16 bits.
__device__ __forceinline__ uint4 split2_record(float v) {
    const float w1 = __uint_as_float(__float_as_uint(v) & 0xFFFF0000u);
    const float w2 = __fsub_rn(v, w1);
    const uint32_t h = (__float_as_uint(w1) >> 16) | (__float_as_uint(w2) & 0xFFFF0000u);
    return make_uint4(h, h, h, 0u);
}

enum WType { WT_Q8_0 = 0, WT_Q4_0 = 1, WT_Q4_K = 2, WT_IQ1_M = 3, WT_W8A8 = 4, WT_Q6_K = 5 };
enum Mode { MODE_PROD = 0, MODE_DEBUG = 1 };

constexpr int BM = 128;             // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;             // tokens per tile (MMA N)
constexpr int BK = 64;              // k per pipeline stage: one 128-byte swizzle row of fp16
constexpr int STAGES = 4;           // smem operand pipeline depth
constexpr int SC_STAGES = 6;        // scale ring depth (released by the epilogue, so deeper)
constexpr int RAW_STAGES = 3;       // raw-byte ring filled by cp.async, two stages ahead of conversion
constexpr int NACC = 4;             // TMEM accumulators (BN columns each)
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_PROD_WARPS = 4;
constexpr int PROD_WARP0 = NUM_EPI_WARPS;
constexpr int MMA_WARP = NUM_EPI_WARPS + NUM_PROD_WARPS;
constexpr int NTHREADS = (MMA_WARP + 1) * 32;
constexpr int TMEM_COLS = NACC * BN;  // 512

constexpr int W8A8_CHUNK_K16 = 64;  // 1024-k chunks for the full-K W8A8 dot

constexpr int A_STAGE_BYTES = BM * 128;
constexpr int B_STAGE_BYTES = BN * 128;
constexpr int SC_STAGE_FLOATS = 2 * BM + 2 * BM + 2 * BN + 2 * BN;   // wsc, wmn, xd, xs for 2 blocks

struct GemmParams {
    const uint8_t* W;           // raw weights (expert 0 for MoE); W8A8: int8 [N][K]
    const int8_t* xq;           // activation codes [M][K]
    const float4* xds;          // q8_1 (d, s) pairs [M][K/32], read two blocks at a time
    const float* w8_ws;         // W8A8 per-channel scales [N]
    const float* w8_xs;         // W8A8 per-token scales [M]
    const uint16_t* xh;         // q8_1 shadow: fp16 codes [M][K] (block types)
    void* out;                  // f32 [rows][N] (bf16 for W8A8)
    int32_t* partials;          // debug: int32 [M][N][groups]
    long long w_row_bytes;      // bytes per weight row
    long long w_expert_bytes;   // bytes per expert (MoE)
    int M, N, K;
    // MoE routing (null for dense)
    const int* rowlist;         // (token*slots + slot) grouped by expert
    const int* work;            // work items: {expert, start, count} triples
    const int* nwork;           // number of work items
    int slots;
};

// ------------------------------------------------------------------------------------------ weight unpack
// Raw bytes of one weight row for one 64-k stage, as 32-bit words.
struct RawA {
    uint32_t w[17];
};

// Geometry of one weight row's raw bytes for one 64-k stage, as staged in shared memory.
// kWords: 32-bit words of data; kVec16: copied and read as 16-byte pieces (else 4-byte words);
// kStride: bytes between rows in the raw ring (an odd number of words / 16-byte units, so that one
// thread per row reads without bank conflicts).
template <int WT> struct RawGeom;
template <> struct RawGeom<0> { static constexpr int kWords = 17, kStride = 68, kVec16 = 0; };   // Q8_0: two 34 B blocks
template <> struct RawGeom<1> { static constexpr int kWords = 9, kStride = 36, kVec16 = 0; };    // Q4_0: two 18 B blocks
template <> struct RawGeom<2> { static constexpr int kWords = 12, kStride = 48, kVec16 = 1; };   // Q4_K: header + 32 code bytes
template <> struct RawGeom<3> { static constexpr int kWords = 7, kStride = 28, kVec16 = 0; };    // IQ1_M: 16 code bytes + tail
template <> struct RawGeom<4> { static constexpr int kWords = 16, kStride = 80, kVec16 = 1; };   // W8A8: 64 int8

// Shared-memory layout of one CTA, per weight type.  Block types take the token operand as fp16 rows
// straight from the q8_1 buffer's shadow section (cp.async into the swizzled tile); W8A8 stages its
// int8 activation rows in the raw ring and converts them.
template <int WT, bool SB, bool RING>
struct SmemLayoutT {
    static constexpr bool kW8 = WT == WT_W8A8;
    static constexpr int raw_b = kW8 ? BN * 64 : 0;              // int8 codes per token row
    static constexpr int raw_ds = (SB || RING) ? BN * 16 : 0;    // (d, s) of the stage's two blocks
    static constexpr int raw_a = BM * RawGeom<WT>::kStride;
    static constexpr int raw_stage = (raw_b + raw_ds + raw_a + 127) / 128 * 128;
    static constexpr int sop_block = (BM + BN) * 16;             // weight-side then token-side scale rows
    static constexpr int sop_stage = 2 * sop_block;
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + STAGES * A_STAGE_BYTES;
    static constexpr int sop_off = b_off + STAGES * B_STAGE_BYTES;
    static constexpr int sc_off = sop_off + (SB ? STAGES * sop_stage : 0);
    static constexpr int raw_off = sc_off + (RING ? SC_STAGES * SC_STAGE_FLOATS * 4 : 0);
    static constexpr int orow_off = raw_off + RAW_STAGES * raw_stage;
    static constexpr int trow_off = orow_off + BN * 4;
    static constexpr int bar_off = trow_off + BN * 4;           // 8-byte aligned
    static constexpr int n_bars = 2 * STAGES + 2 * SC_STAGES + 2 * NACC + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;       // tmem slot, abort flag
    static constexpr int total = misc_off + 16;
    static constexpr int alloc = total + 1024;                  // slack for 1024-byte alignment
};

// Global address of word / 16-byte piece `i` of a weight row's raw bytes for stage s.
template <int WT>
__device__ __forceinline__ const uint8_t* raw_a_src(const uint8_t* row, int s, int i) {
    if constexpr (WT == WT_Q8_0) return row + 68 * s + 4 * i;
    else if constexpr (WT == WT_Q4_0) return row + 36 * s + 4 * i;
    else if constexpr (WT == WT_Q4_K) {
        const uint8_t* sb = row + 144 * (s >> 2);
        return i == 0 ? sb : sb + 16 + 32 * (s & 3) + 16 * (i - 1);
    } else if constexpr (WT == WT_IQ1_M) {
        const uint8_t* sb = row + 76 * (s >> 2);
        return i < 4 ? sb + 16 * (s & 3) + 4 * i : sb + 64 + 4 * (i - 4);
    } else {
        return row + 64 * s + 16 * i;
    }
}

__device__ __forceinline__ uint32_t byte_shift2(uint32_t a, uint32_t b) {   // bytes 2..5 of {a, b}
    return __byte_perm(a, b, 0x5432);
}

// Four unsigned bytes (each 0..255) -> two fp16x2 words of (byte - bias).
__device__ __forceinline__ void u8x4_to_f16x4(uint32_t u, uint32_t bias_f16x2, uint32_t& lo, uint32_t& hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias_f16x2));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias_f16x2));
}

// fp16x2 bits of two floats (round to nearest; the callers pass exactly representable values).
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Keep bits 8-9 of each 16-bit half (a 2-bit code placed there by a byte permute) and add the fp16
// exponent of 1024: the halves become 1024 + 256*code exactly.
__device__ __forceinline__ uint32_t lop_or_magic(uint32_t x) {
    return (x & 0x03000300u) | 0x64006400u;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ uint32_t field_le(const uint32_t* words, int pos, int width) {
    const int wi = pos >> 5, off = pos & 31;
    const uint32_t v = __funnelshift_r(words[wi], words[wi + 1], off);
    return v & ((1u << width) - 1u);
}

// Unpack one row's 64-k stage into 32 fp16x2 words (k order) plus the two blocks' scales.
// PROD_FOLD: IQ1_M folds (2s+1) into the values (production); debug keeps 8g±1.
template <int WT, bool PROD_FOLD>
__device__ __forceinline__ void unpack_a(const RawA& r, int s, uint32_t (&h)[32], float (&wsc)[2], float (&wmn)[2]) {
    if constexpr (WT == WT_Q8_0) {
        wsc[0] = half_bits_to_float((uint16_t)(r.w[0] & 0xFFFFu));
        wsc[1] = half_bits_to_float((uint16_t)(r.w[8] >> 16));
        wmn[0] = wmn[1] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) s8x4_to_f16x4(byte_shift2(r.w[j], r.w[j + 1]), h[2 * j], h[2 * j + 1]);
#pragma unroll
        for (int j = 0; j < 8; j++) s8x4_to_f16x4(r.w[9 + j], h[16 + 2 * j], h[16 + 2 * j + 1]);
    } else if constexpr (WT == WT_Q4_0) {
        wsc[0] = half_bits_to_float((uint16_t)(r.w[0] & 0xFFFFu));
        wsc[1] = half_bits_to_float((uint16_t)(r.w[4] >> 16));
        wmn[0] = wmn[1] = 0.f;
        const uint32_t bias = 0x64086408u;                     // 1024 + 8: value = code - 8
#pragma unroll
        for (int blk = 0; blk < 2; blk++) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint32_t nw = blk == 0 ? byte_shift2(r.w[j], r.w[j + 1]) : r.w[5 + j];
                const int base = 16 * blk;                     // fp16x2 word index of the block
                u8x4_to_f16x4(nw & 0x0F0F0F0Fu, bias, h[base + 2 * j], h[base + 2 * j + 1]);
                u8x4_to_f16x4((nw >> 4) & 0x0F0F0F0Fu, bias, h[base + 8 + 2 * j], h[base + 8 + 2 * j + 1]);
            }
        }
    } else if constexpr (WT == WT_Q4_K) {
        const float d = half_bits_to_float((uint16_t)(r.w[0] & 0xFFFFu));
        const float dmin = half_bits_to_float((uint16_t)(r.w[0] >> 16));
        const uint32_t bits[4] = {r.w[1], r.w[2], r.w[3], 0u};
        const int j = s & 3;                                   // sub-blocks 2j, 2j+1
        uint32_t sc[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            sc[i] = field_le(bits, 6 * (2 * j + i), 6);
            wsc[i] = d * (float)sc[i];
            wmn[i] = dmin * (float)field_le(bits, 6 * (8 + 2 * j + i), 6);
        }
        const uint32_t bias = 0x64006400u;                     // unsigned codes 0..15
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const uint32_t nw = r.w[4 + t];
            u8x4_to_f16x4(nw & 0x0F0F0F0Fu, bias, h[2 * t], h[2 * t + 1]);
            u8x4_to_f16x4((nw >> 4) & 0x0F0F0F0Fu, bias, h[16 + 2 * t], h[16 + 2 * t + 1]);
        }
        if constexpr (PROD_FOLD) {
            // fold the 6-bit sub-block scale into the operand: sc * code <= 63 * 15, exact in fp16;
            // the block's weight scale is then the super-block d
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const uint32_t scw = u10x2_to_f16x2(sc[i] | (sc[i] << 16), 0x64006400u);   // (sc, sc) in fp16
#pragma unroll
                for (int t = 0; t < 16; t++) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[16 * i + t]) : "r"(scw));
                wsc[i] = d;
            }
        }
    } else if constexpr (WT == WT_IQ1_M) {
        // operand value v = mult * (8g + sigma), g = code - 1, mult = 2s+1 (production fold) or 1.
        // Two codes of one sign group at a time: a byte permute puts them at bits 8-9 of the two halves
        // of an fp16x2 word, OR-ing in the exponent gives 1024 + 256*code exactly, and one fp16 FMA
        // maps that to mult*(8*code - 8 + sigma) = (1024 + 256*code) * (mult/32) + mult*(sigma - 40).
        // Every intermediate is an integer (or mult/32) well inside fp16's exact range.
        const int j = s & 3;
        const uint32_t signs = (r.w[4] >> (8 * j)) & 0xFFu;    // one bit per 8 values of this stage
        const uint32_t sbits[3] = {(r.w[5] >> 0), r.w[6] & 0xFFFFu, 0u};   // bytes 68..73 of the block
        const float d = half_bits_to_float((uint16_t)(r.w[6] >> 16));
        wsc[0] = wsc[1] = PROD_FOLD ? d * 0.125f : 0.f;
        wmn[0] = wmn[1] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {                          // 16-value sub-scale groups
            const float mult = PROD_FOLD ? (float)(2u * field_le(sbits, 3 * (4 * j + q), 3) + 1u) : 1.f;
            const uint32_t cw = r.w[q];                        // 16 two-bit codes, value 4i+t at byte i
            const uint32_t c0 = cw & 0x03030303u;              // codes 4i
            const uint32_t c1 = (cw >> 2) & 0x03030303u;       // codes 4i+1
            const uint32_t c2 = (cw >> 4) & 0x03030303u;       // codes 4i+2
            const uint32_t c3 = (cw >> 6) & 0x03030303u;       // codes 4i+3
            const uint32_t a2 = f2_to_h2(mult * 0.03125f, mult * 0.03125f);
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {                   // sign groups: values 8hf..8hf+7 of the 16
                const float sig = ((signs >> (2 * q + hf)) & 1u) ? -1.f : 1.f;
                const float bc = mult * (sig - 40.f);
                const uint32_t b2 = f2_to_h2(bc, bc);
#pragma unroll
                for (int ii = 0; ii < 2; ii++) {
                    const int i = 2 * hf + ii;                 // byte of the word: values 4i..4i+3
                    const uint32_t sel = (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12));
                    const uint32_t p01 = lop_or_magic(__byte_perm(c0, c1, sel));
                    const uint32_t p23 = lop_or_magic(__byte_perm(c2, c3, sel));
                    h[8 * q + 2 * i] = hfma2_u32(p01, a2, b2);
                    h[8 * q + 2 * i + 1] = hfma2_u32(p23, a2, b2);
                }
            }
        }
    } else {                                                    // W8A8
        wsc[0] = wsc[1] = 0.f;
        wmn[0] = wmn[1] = 0.f;
#pragma unroll
        for (int j = 0; j < 16; j++) s8x4_to_f16x4(r.w[j], h[2 * j], h[2 * j + 1]);
    }
}

// ------------------------------------------------------------------------------------------ kernel
template <int WT, int MODE>
struct KTraits {
    static constexpr bool kIsW8 = WT == WT_W8A8;
    // k16 MMA steps per accumulator group
    static constexpr int G16 = (MODE == MODE_DEBUG) ? ((WT == WT_IQ1_M) ? 1 : 2) : (kIsW8 ? W8A8_CHUNK_K16 : 2);
    // block types in production: the per-block scale product xd*wd is an MMA outer product (S)
    static constexpr bool kSB = (MODE == MODE_PROD) && !kIsW8;
    // Q4_K's min term -dmin*m_b*s[m,b] is applied from a shared-memory scale ring
    static constexpr bool kScaleRing = kSB && WT == WT_Q4_K;
    static constexpr bool kFold = (MODE == MODE_PROD);
    static constexpr int kNacc = kSB ? 2 : NACC;              // TMEM accumulators in rotation
    static constexpr int kAccCols = kSB ? 2 * BN : BN;        // columns per accumulator: I (and S)
};

template <int WT, int MODE, bool MOE>
__global__ void __launch_bounds__(NTHREADS, 1) mmq_gemm_kernel(const GemmParams p) {
    using T = KTraits<WT, MODE>;
    using SmemLayout = SmemLayoutT<WT, T::kSB, T::kScaleRing>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // align by pointer arithmetic on the __shared__ array so that the compiler keeps the address space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem_s = smem_u32(smem);                   // shared-window address of the tile base
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- tile coordinates
    const int n0 = blockIdx.x * BM;
    int m0 = blockIdx.y * BN, mcount = min(BN, p.M - m0), expert = 0;
    if constexpr (MOE) {
        if ((int)blockIdx.y >= __ldg(p.nwork)) return;        // uniform for the whole CTA
        const int* wi = p.work + 3 * blockIdx.y;
        expert = __ldg(wi);
        m0 = __ldg(wi + 1);
        mcount = __ldg(wi + 2);
    }
    const uint8_t* Wbase = p.W + (long long)expert * p.w_expert_bytes;

    int* orow = reinterpret_cast<int*>(smem + SmemLayout::orow_off);
    int* trow = reinterpret_cast<int*>(smem + SmemLayout::trow_off);
    const uint32_t bar0 = smem_u32(smem + SmemLayout::bar_off);
    auto bar_full = [&](int i) { return bar0 + 8u * i; };
    auto bar_empty = [&](int i) { return bar0 + 8u * (STAGES + i); };
    auto bar_sfull = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
    auto bar_sfree = [&](int i) { return bar0 + 8u * (2 * STAGES + SC_STAGES + i); };
    auto bar_accf = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + i); };
    auto bar_acce = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + NACC + i); };
    const uint32_t bar_done = bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 2 * NACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SmemLayout::misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::misc_off + 4);

    // ---- setup: barriers, TMEM, row maps
    if (warp == MMA_WARP) {
        if (lane == 0) {
            // one arrival per producer warp (an elected lane after the warp's stores are fenced):
            // per-thread arrivals on one barrier word serialise and throttle the whole pipeline
            for (int i = 0; i < STAGES; i++) {
                mbar_init(bar_full(i), NUM_PROD_WARPS);
                mbar_init(bar_empty(i), 1);
            }
            for (int i = 0; i < SC_STAGES; i++) {
                mbar_init(bar_sfull(i), NUM_PROD_WARPS);
                mbar_init(bar_sfree(i), NUM_EPI_WARPS);
            }
            for (int i = 0; i < NACC; i++) {
                mbar_init(bar_accf(i), 1);
                mbar_init(bar_acce(i), NUM_EPI_WARPS);
            }
            mbar_init(bar_done, 1);
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x < BN) {
        const int j = threadIdx.x;
        int tr = -1, orr = -1;
        if (j < mcount) {
            if constexpr (MOE) {
                const int rl = __ldg(p.rowlist + m0 + j);
                tr = rl / p.slots;
                orr = rl;
            } else {
                tr = m0 + j;
                orr = m0 + j;
            }
        }
        trow[j] = tr;
        orow[j] = orr;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nstages = p.K / BK;
    const int nk16 = p.K / 16;
    const int ngroups = (nk16 + T::G16 - 1) / T::G16;
    const int kb32 = p.K / 32;

    if (warp >= PROD_WARP0 && warp < MMA_WARP) {
        // =========================================================== producers
        // Raw bytes arrive by coalesced cp.async into a RAW_STAGES-deep ring (issued two stages
        // ahead, zero-filled for ragged rows); each stage is then unpacked from shared memory into
        // the fp16 operand tiles.  Row maps and layouts: one weight row per thread for the unpack,
        // four threads per token row for the codes.
        using G = RawGeom<WT>;
        const int pt = threadIdx.x - PROD_WARP0 * 32;           // 0..127
        const uint32_t a_smem = smem_s + SmemLayout::a_off;
        const uint32_t b_smem = smem_s + SmemLayout::b_off;
        const uint32_t raw0 = smem_s + SmemLayout::raw_off;
        const uint32_t trow_s = smem_s + SmemLayout::trow_off;
        const uint32_t sop_smem = smem_s + SmemLayout::sop_off;
        const uint8_t* xds_bytes = reinterpret_cast<const uint8_t*>(p.xds);

        // Per-thread copy addresses are fixed for the whole tile: each thread always copies the same
        // token rows / 16-byte chunks and the same weight words; only a per-stage offset changes.
        // token rows (block types): chunk c of rows (pt/8) + 16k, k = 0..7, into the swizzled tile
        const int bc = pt & 7;
        const uint32_t b_dst0 = (uint32_t)sw128_off((uint32_t)(pt >> 3), (uint32_t)bc);   // + 2048*k
        const char* b_src[8];
        uint32_t b_ok = 0;
        if constexpr (!SmemLayout::kW8) {
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int tr = ld_shared_s32(trow_s + 4 * ((pt >> 3) + 16 * k));
                b_src[k] = reinterpret_cast<const char*>(p.xh + (long long)(tr >= 0 ? tr : 0) * p.K + 8 * bc);
                b_ok |= (tr >= 0 ? 1u : 0u) << k;
            }
        }
        // this thread's own token row: scale records / (d, s) pairs / W8A8 int8 codes
        const int my_tr = ld_shared_s32(trow_s + 4 * pt);
        const bool my_ok = my_tr >= 0;
        const long long my_row = my_ok ? my_tr : 0;
        // weight words (or 16-byte pieces) i = pt + 128k: row i / words, offset within the row chunk
        constexpr int AW = G::kVec16 ? G::kWords / 4 : G::kWords;
        uint32_t a_off[AW];
        uint32_t a_ok = 0;
#pragma unroll
        for (int k = 0; k < AW; k++) {
            const int i = pt + 128 * k, row = i / AW, wd = i % AW;
            const bool ok = n0 + row < p.N;
            uint32_t o = (uint32_t)((long long)(ok ? n0 + row : 0) * p.w_row_bytes);
            if constexpr (WT == WT_Q4_K) o += wd ? 16u * wd : 0u;              // header, then code pieces
            else if constexpr (WT == WT_IQ1_M) o += wd < 4 ? 4u * wd : 64u + 4u * (wd - 4);
            else if constexpr (G::kVec16) o += 16u * wd;
            else o += 4u * wd;
            a_off[k] = o;
            a_ok |= (ok ? 1u : 0u) << k;
        }

        auto issue_copies = [&](int s) {
            const uint32_t rb = raw0 + (s % RAW_STAGES) * SmemLayout::raw_stage;
            if constexpr (SmemLayout::kW8) {                    // int8 activation rows: 512 x 16 B
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int i = pt + 128 * k, row = i >> 2, ch = i & 3;
                    const int tr = ld_shared_s32(trow_s + 4 * row);
                    const int8_t* src = p.xq + (long long)(tr >= 0 ? tr : 0) * p.K + 64 * s + 16 * ch;
                    cp_async_16(rb + 16 * i, src, tr >= 0 ? 16u : 0u);
                }
            } else {
                // fp16 token rows go straight into the operand tile once the MMA has released it
                const int slot = s % STAGES;
                mbar_wait(bar_empty(slot), ((s / STAGES) & 1) ^ 1, abort_flag);
                const uint32_t bt = b_smem + slot * B_STAGE_BYTES + b_dst0;
#pragma unroll
                for (int k = 0; k < 8; k++)
                    cp_async_16(bt + 2048 * k, b_src[k] + 128 * s, ((b_ok >> k) & 1) ? 16u : 0u);
                if constexpr (T::kSB || T::kScaleRing) {        // (d, s) of the stage's two blocks
                    const uint8_t* src = xds_bytes + (my_row * kb32 + 2 * s) * 8;
                    cp_async_16(rb + 16 * pt, src, my_ok ? 16u : 0u);
                }
            }
            // weight row chunks of this stage
            const uint32_t ra = rb + SmemLayout::raw_b + SmemLayout::raw_ds;
            uint32_t so_main, so_tail;                          // per-stage source offsets
            if constexpr (WT == WT_Q8_0) so_main = so_tail = 68u * s;
            else if constexpr (WT == WT_Q4_0) so_main = so_tail = 36u * s;
            else if constexpr (WT == WT_Q4_K) { so_tail = 144u * (s >> 2); so_main = so_tail + 16u + 32u * (s & 3) - 16u; }
            else if constexpr (WT == WT_IQ1_M) { so_tail = 76u * (s >> 2); so_main = so_tail + 16u * (s & 3); }
            else so_main = so_tail = 64u * s;
#pragma unroll
            for (int k = 0; k < AW; k++) {
                const int i = pt + 128 * k;
                uint32_t so;
                if constexpr (WT == WT_Q4_K) so = ((i % AW) == 0) ? so_tail : so_main;
                else if constexpr (WT == WT_IQ1_M) so = ((i % AW) < 4) ? so_main : so_tail;
                else so = so_main;
                const uint8_t* src = Wbase + a_off[k] + so;
                const bool ok = (a_ok >> k) & 1;
                if constexpr (G::kVec16) {
                    const uint32_t dst = (WT == WT_W8A8) ? 16u * i + 16u * (uint32_t)(i >> 2) : 16u * i;
                    cp_async_16(ra + dst, src, ok ? 16u : 0u);
                } else {
                    cp_async_4(ra + 4u * i, src, ok ? 4u : 0u);
                }
            }
        };

        auto convert = [&](int s) {
            const int slot = s % STAGES;
            const int sslot = s % SC_STAGES;
            if constexpr (T::kScaleRing) mbar_wait(bar_sfree(sslot), ((s / SC_STAGES) & 1) ^ 1, abort_flag);
            if constexpr (SmemLayout::kW8) mbar_wait(bar_empty(slot), ((s / STAGES) & 1) ^ 1, abort_flag);
            const uint32_t rb = raw0 + (s % RAW_STAGES) * SmemLayout::raw_stage;
            const uint32_t ra = rb + SmemLayout::raw_b + SmemLayout::raw_ds + pt * G::kStride;
            const uint32_t at = a_smem + slot * A_STAGE_BYTES;
            const uint32_t bt = b_smem + slot * B_STAGE_BYTES;
            {
                RawA w;
                if constexpr (G::kVec16) {
#pragma unroll
                    for (int k = 0; k < G::kWords / 4; k++) {
                        const uint4 v = ld_shared_u4(ra + 16 * k);
                        w.w[4 * k] = v.x; w.w[4 * k + 1] = v.y; w.w[4 * k + 2] = v.z; w.w[4 * k + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < G::kWords; k++) w.w[k] = ld_shared_u32(ra + 4 * k);
                }
                uint32_t ha[32];
                float wsc[2], wmn[2];
                unpack_a<WT, T::kFold>(w, s, ha, wsc, wmn);
                if (n0 + pt >= p.N) wsc[0] = wsc[1] = wmn[0] = wmn[1] = 0.f;
#pragma unroll
                for (int c = 0; c < 8; c++)
                    st_shared_v4(at + sw128_off(pt, c), ha[4 * c], ha[4 * c + 1], ha[4 * c + 2], ha[4 * c + 3]);
                if constexpr (T::kSB) {
                    // weight-side scale rows {w1,w2,w1,w2,w1,w2,0,0}, w1 + w2 = wd/2 (the MMA counts
                    // every product twice), and this thread's token row's {x1,x1,x2,x2,x3,x3,0,0},
                    // x1 + x2 + x3 = d, from the staged (d, s) pairs of the two blocks
                    const uint32_t so = sop_smem + slot * SmemLayout::sop_stage + 16 * pt;
                    const float4 dsx = ld_shared_f4(rb + 16 * pt);
#pragma unroll
                    for (int i = 0; i < 2; i++) {
                        const uint4 rec = split2_record(0.5f * wsc[i]);
                        st_shared_v4(so + i * SmemLayout::sop_block, rec.x, rec.y, rec.z, rec.w);
                        const uint4 tr = split3_record(i == 0 ? dsx.x : dsx.z);
                        st_shared_v4(so + i * SmemLayout::sop_block + BM * 16, tr.x, tr.y, tr.z, tr.w);
                    }
                }
                if constexpr (T::kScaleRing) {
                    const float4 ds = ld_shared_f4(rb + 16 * pt);
                    const uint32_t sc = smem_s + SmemLayout::sc_off + sslot * SC_STAGE_FLOATS * 4 + 4 * pt;
                    st_shared_f32(sc + 4 * (0 * BM), wsc[0]);
                    st_shared_f32(sc + 4 * (1 * BM), wsc[1]);
                    st_shared_f32(sc + 4 * (2 * BM), wmn[0]);
                    st_shared_f32(sc + 4 * (3 * BM), wmn[1]);
                    st_shared_f32(sc + 4 * (4 * BM), ds.x);               // xd, block 0
                    st_shared_f32(sc + 4 * (4 * BM + BN), ds.z);          // xd, block 1
                    st_shared_f32(sc + 4 * (4 * BM + 2 * BN), ds.y);      // xs, block 0
                    st_shared_f32(sc + 4 * (4 * BM + 3 * BN), ds.w);      // xs, block 1
                }
            }
            if constexpr (SmemLayout::kW8) {
#pragma unroll
                for (int k = 0; k < 4; k++) {                      // W8A8 activation codes -> fp16
                    const int i = pt + 128 * k, row = i >> 2, ch = i & 3;
                    const uint4 q = ld_shared_u4(rb + 16 * i);
                    uint32_t hb[8];
                    s8x4_to_f16x4(q.x, hb[0], hb[1]);
                    s8x4_to_f16x4(q.y, hb[2], hb[3]);
                    s8x4_to_f16x4(q.z, hb[4], hb[5]);
                    s8x4_to_f16x4(q.w, hb[6], hb[7]);
                    st_shared_v4(bt + sw128_off(row, 2 * ch), hb[0], hb[1], hb[2], hb[3]);
                    st_shared_v4(bt + sw128_off(row, 2 * ch + 1), hb[4], hb[5], hb[6], hb[7]);
                }
            }
            fence_proxy_async_smem();       // this thread's tile stores and landed copies -> tensor core
            __syncwarp();
            if ((threadIdx.x & 31) == 0) {
                mbar_arrive(bar_full(slot));
                if constexpr (T::kScaleRing) mbar_arrive(bar_sfull(sslot));
            }
        };

        // prologue: RAW_STAGES groups (empty ones past the end keep the group count uniform)
#pragma unroll 1
        for (int t = 0; t < RAW_STAGES; t++) {
            if (t < nstages) issue_copies(t);
            cp_async_commit();
        }
#pragma unroll 1
        for (int s = 0; s < nstages; s++) {
            if (s == 0) cp_async_wait<RAW_STAGES - 1>();
            else cp_async_wait<RAW_STAGES - 2>();
            // every producer thread's copies of stage s have landed, and every producer thread has
            // finished unpacking stage s-1, whose raw slot is refilled next
            named_bar_sync(1, NUM_PROD_WARPS * 32);
            if (s >= 1) {
                if (s - 1 + RAW_STAGES < nstages) issue_copies(s - 1 + RAW_STAGES);
                cp_async_commit();
            }
            convert(s);
        }
        cp_async_wait<0>();
    } else if (warp == MMA_WARP) {
        // =========================================================== MMA issuer
        // The whole warp runs the issue loop (warp-uniform control flow keeps the descriptors in the
        // uniform datapath); one elected lane issues each MMA and commit.
        const uint32_t idesc = idesc_f16_f32(BM, BN);
        const uint32_t idesc_s = idesc_bf16_f32(BM, BN);
        const uint32_t a_smem = smem_s + SmemLayout::a_off;
        const uint32_t b_smem = smem_s + SmemLayout::b_off;
        const uint32_t sop_smem = smem_s + SmemLayout::sop_off;
        for (int s = 0; s < nstages; s++) {
            if (*abort_flag) break;
            const int slot = s % STAGES;
            if (!mbar_wait(bar_full(slot), (s / STAGES) & 1, abort_flag)) break;
            tc_fence_after();
            const uint64_t ad0 = sdesc_sw128(a_smem + slot * A_STAGE_BYTES);
            const uint64_t bd0 = sdesc_sw128(b_smem + slot * B_STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int ks = 4 * s + j;
                const int kin = ks % T::G16;
                const int g = ks / T::G16;
                const int buf = g % T::kNacc;
                if (kin == 0) {
                    mbar_wait(bar_acce(buf), ((g / T::kNacc) & 1) ^ 1, abort_flag);
                    tc_fence_after();
                }
                const uint32_t dcol = tmem_base + buf * T::kAccCols;
                // +32 bytes per 16-element K slice: +2 in the descriptor's address field
                if (elect_one()) umma_f16(dcol, ad0 + 2 * j, bd0 + 2 * j, idesc, kin != 0 ? 1u : 0u);
                if (kin == T::G16 - 1 || ks == nk16 - 1) {
                    if constexpr (T::kSB) {
                        // S = wd (x) xd for this block: one bf16 MMA on the scale rows
                        const uint32_t sa = sop_smem + slot * SmemLayout::sop_stage + (j >> 1) * SmemLayout::sop_block;
                        const uint64_t sad = sdesc_rows16(sa), sbd = sdesc_rows16(sa + BM * 16);
                        if (elect_one()) umma_f16(dcol + BN, sad, sbd, idesc_s, 0u);
                    }
                    if (elect_one()) umma_commit(bar_accf(buf));
                }
            }
            if (elect_one()) umma_commit(bar_empty(slot));
            __syncwarp();
        }
        // every MMA and every commit-arrive of this CTA has landed once this barrier flips
        if (elect_one()) umma_commit(bar_done);
        __syncwarp();
        mbar_wait_final(bar_done, 0);
        __syncwarp();
    } else {
        // =========================================================== epilogue
        const int q = warp & 3;                 // TMEM lane quarter
        const int ch = warp >> 2;               // column half: tokens 64*ch .. 64*ch+63
        const int r = 32 * q + lane;            // tile row (weight row n0 + r)
        const int n = n0 + r;
        const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + 64 * ch;

        uint64_t acc2[(MODE == MODE_PROD && !T::kIsW8) ? 32 : 1];   // packed f32 pairs: columns 2t, 2t+1
        int32_t iacc[T::kIsW8 ? 64 : 1];
#pragma unroll
        for (int j = 0; j < (int)(sizeof(acc2) / sizeof(uint64_t)); j++) acc2[j] = 0ull;
        if constexpr (T::kIsW8) {
#pragma unroll
            for (int j = 0; j < 64; j++) iacc[j] = 0;
        }

        for (int g = 0; g < ngroups; g++) {
            const int buf = g % T::kNacc;
            mbar_wait(bar_accf(buf), (g / T::kNacc) & 1, abort_flag);
            tc_fence_after();
            const uint32_t tacc = tbase + buf * T::kAccCols;
            // Q4_K min term: row value dmin*m_b, column values s[m,b] from the scale ring
            uint32_t sc = 0;
            float mn = 0.f;
            int slot = 0, i = 0;
            if constexpr (T::kScaleRing) {
                const int s = g >> 1;
                i = g & 1;
                slot = s % SC_STAGES;
                if (i == 0) mbar_wait(bar_sfull(slot), (s / SC_STAGES) & 1, abort_flag);
                sc = smem_s + SmemLayout::sc_off + slot * SC_STAGE_FLOATS * 4;
                mn = ld_shared_f32(sc + 4 * (2 * BM + i * BM + r));
            }
            const uint64_t nmn2 = f2_pack(-mn, -mn);
            // four quarters of 16 columns: the block's integer dots I and (block types) the scale
            // products S come from TMEM; acc += I * S in packed f32 pairs
#pragma unroll
            for (int qq = 0; qq < 4; qq++) {
                float4 cs[4];
                if constexpr (T::kScaleRing) {
                    const uint32_t xs = sc + 4 * (4 * BM + 2 * BN + i * BN + 64 * ch + 16 * qq);
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++) cs[q4] = ld_shared_f4(xs + 16 * q4);
                }
                uint32_t v[16], w[16];
                tmem_ld16(tacc + 16 * qq, v);
                if constexpr (T::kSB) tmem_ld16(tacc + BN + 16 * qq, w);
                tmem_ld_wait();
                if (qq == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acce(buf));
                }
                if constexpr (MODE == MODE_DEBUG) {
                    if (n < p.N) {
#pragma unroll
                        for (int j = 0; j < 16; j++) {
                            const int col = 64 * ch + 16 * qq + j;
                            if (col < mcount)
                                p.partials[((long long)(m0 + col) * p.N + n) * ngroups + g] =
                                    __float2int_rn(__uint_as_float(v[j]));
                        }
                    }
                } else if constexpr (T::kIsW8) {
#pragma unroll
                    for (int j = 0; j < 16; j++) iacc[16 * qq + j] += __float2int_rn(__uint_as_float(v[j]));
                } else {
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++) {
                        const int j = 4 * q4, a = 8 * qq + 2 * q4;
                        acc2[a] = f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                         f2_pack(__uint_as_float(w[j]), __uint_as_float(w[j + 1])), acc2[a]);
                        acc2[a + 1] = f2_fma(f2_pack(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])),
                                             f2_pack(__uint_as_float(w[j + 2]), __uint_as_float(w[j + 3])), acc2[a + 1]);
                        if constexpr (T::kScaleRing) {
                            acc2[a] = f2_fma(nmn2, f2_pack(cs[q4].x, cs[q4].y), acc2[a]);
                            acc2[a + 1] = f2_fma(nmn2, f2_pack(cs[q4].z, cs[q4].w), acc2[a + 1]);
                        }
                    }
                }
            }
            if constexpr (T::kScaleRing) {
                if (i == 1 || g == ngroups - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_sfree(slot));
                }
            }
        }

        // ---- store
        if constexpr (MODE == MODE_PROD) {
            if (n < p.N) {
                const int* orw = orow + 64 * ch;
                if constexpr (T::kIsW8) {
                    const float wsn = __ldg(p.w8_ws + n);
                    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                    for (int j = 0; j < 64; j++) {
                        const int orr = orw[j];
                        if (orr >= 0) {
                            const float t = __fmul_rn((float)iacc[j], __ldg(p.w8_xs + orr));
                            out[(long long)orr * p.N + n] = __float2bfloat16_rn(__fmul_rn(t, wsn));
                        }
                    }
                } else {
                    float* out = reinterpret_cast<float*>(p.out);
#pragma unroll
                    for (int t = 0; t < 32; t++) {
                        float a0, a1;
                        f2_unpack(acc2[t], a0, a1);
                        const int o0 = orw[2 * t], o1 = orw[2 * t + 1];
                        if (o0 >= 0) out[(long long)o0 * p.N + n] = a0;
                        if (o1 >= 0) out[(long long)o1 * p.N + n] = a1;
                    }
                }
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------------------------------ host launch
template <int WT, int MODE, bool MOE>
cudaError_t launch_gemm(const GemmParams& p, int grid_y, cudaStream_t stream) {
    using T = KTraits<WT, MODE>;
    using SmemLayout = SmemLayoutT<WT, T::kSB, T::kScaleRing>;
    static bool configured[64] = {};       // per instantiation and device
    auto kern = mmq_gemm_kernel<WT, MODE, MOE>;
    bool& done = device_flag(configured);
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemLayout::alloc);
        if (e != cudaSuccess) return e;
        done = true;
    }
    dim3 grid((p.N + BM - 1) / BM, grid_y);
    kern<<<grid, NTHREADS, SmemLayout::alloc, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mmq
