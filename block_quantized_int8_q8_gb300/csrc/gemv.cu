// gemv.cu -- the few-token path (M <= 8) of the block types: a matrix-vector kernel that reads every weight
// byte once at memory speed instead of filling 128-token tensor-core tiles ("CUDA: add IQ1_M to MMQ":
// small batches run on the matrix-vector path; the MMQ tiles win from ~100 tokens on).
//
// One CTA of four warps per group of four weight rows.  Rows are walked in chunks of 32 blocks of 32 values
// (one block per lane), four chunks (one per warp) at a time: each warp stages its chunk of every row in
// shared memory with coalesced cp.async copies -- the whole segment of every row in flight at once --,
// each lane decodes its block to int8 words, forms the exact int32 block dot per token with dp4a ("08 · R1 —
// int8 MMQ prefill GEMM", §2.1: the in-block integer dot is exact), and its f32 term u = (xd * wsc) * I
// (Q4_K: minus dmin*m_b * s; IQ1_M and q6_K: one term per 16-value half).  One thread per (row, token) then
// adds the terms in block order into its running sum ("A Negative Result on int8 Tensor-Core MMQ", §2: the
// blockwise contraction).  Every product and sum is a separate round-to-nearest step in the order written,
// so the output is bit-identical to the blockwise definition computed in that order.  (One warp per row,
// walking its chunks with two in flight, measured 2x slower at one token: two memory round trips per row.)
//
// Decode runs layer after layer, each a quantize launch and this kernel on a few hundred KB to tens of MB
// of weights, so launch gaps matter: both kernels are launched as programmatic dependents.  This kernel's
// CTAs start while the kernel before it finishes, pull the first segment of their first row group into L2
// (a hint with no effect on what loads return), and only then wait for the previous kernel's results;
// measured on a stream of 7B-shaped Q4_0 layers at one token, quantize + GEMV per layer drops from 8.5 to
// 7.7 us (7.3 us with the unrolled copy issue below).
#include <cstdint>
#include <cuda_fp16.h>
#include "gemv.h"
#include "gemm.cuh"
#include "mmq_device.cuh"

namespace mmq {
namespace gemv {

constexpr int WARPS = 4;                 // warps per CTA: one chunk of a segment each
constexpr int RPC = 4;                   // weight rows per CTA
constexpr int CHUNK = 32;                // 32-value blocks per chunk (one per lane)

// Raw bytes of one chunk (32 blocks = 1024 values) per type.
__host__ __device__ constexpr int chunk_bytes(int wt) {
    return wt == WT_Q8_0 ? 32 * 34 : wt == WT_Q4_0 ? 32 * 18 : wt == WT_Q4_K ? 4 * 144 : wt == WT_IQ1_M ? 4 * 76 : 4 * 224;
}
__host__ __device__ constexpr bool per16(int wt) { return wt == WT_IQ1_M || wt == WT_Q6_K; }
// A staging slot: one chunk plus one word that the last block's span read may touch, on 16-byte boundaries.
__host__ __device__ constexpr int stage_words(int wt) { return (chunk_bytes(wt) / 4 + 1 + 3) / 4 * 4; }

// NW consecutive 32-bit words starting at byte offset o of the staged bytes (any alignment): NW + 1
// aligned loads and a funnel shift each.
template <int NW>
__device__ __forceinline__ void st_span(const uint32_t* st, int o, uint32_t (&w)[NW]) {
    const uint32_t* p = st + (o >> 2);
    const int sh = 8 * (o & 3);
    uint32_t prev = p[0];
#pragma unroll
    for (int k = 0; k < NW; k++) {
        const uint32_t nxt = p[k + 1];
        w[k] = __funnelshift_r(prev, nxt, sh);
        prev = nxt;
    }
}
__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// bias_byte: for unsigned bytes u with u + (128 - c) < 256 (so no carry leaves the byte), the int8 value
// u - c is ((u + (128 - c)) ^ 0x80) per byte: one add and one xor for four bytes at once.  Used with c = 8
// (4-bit codes), 32 (6-bit codes) and 9 or 7 (IQ1_M's 8 * code in {0, 8, 16, 24}).

// Decode block j of the staged bytes st: 8 words of int8 values in k order and the scale factors of the
// blockwise definition (per 32 values, or per 16-value half: wsc[0], wsc[1]).  IQ1_M returns 8 * code per
// byte and the sign bits of its four 8-value groups (gsign); the kernel adds each group's offset.
// Super-block types start every record on a 4-byte boundary and read aligned words; Q8_0 and Q4_0 blocks
// are 2-byte aligned.
template <int WT>
__device__ __forceinline__ void decode_block(const uint32_t* st, int j, uint32_t (&w)[8], float (&wsc)[2],
                                             float& wmin, uint32_t& gsign) {
    wmin = 0.f;
    gsign = 0u;
    if constexpr (WT == WT_Q8_0) {                 // f16 d | int8 q[32]
        uint32_t b[9];                             // bytes 34j .. 34j + 35
        st_span<9>(st, 34 * j, b);
        wsc[0] = wsc[1] = half_lo(b[0]);
#pragma unroll
        for (int k = 0; k < 8; k++) w[k] = __funnelshift_r(b[k], b[k + 1], 16);
    } else if constexpr (WT == WT_Q4_0) {          // f16 d | byte i = code i (low) | code i+16 (high); codes
                                                   // unsigned here, the kernel subtracts 8 * sum(q)
        uint32_t b[5];                             // bytes 18j .. 18j + 19
        st_span<5>(st, 18 * j, b);
        wsc[0] = wsc[1] = half_lo(b[0]);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint32_t nw = __funnelshift_r(b[k], b[k + 1], 16);
            w[k] = nw & 0x0F0F0F0Fu;
            w[4 + k] = (nw >> 4) & 0x0F0F0F0Fu;
        }
    } else if constexpr (WT == WT_Q4_K) {          // f16 d | f16 dmin | 12 B six-bit sc, m | 128 B codes
        const uint32_t* rec = st + 36 * (j >> 3);  // 144-byte records
        const int sb = j & 7;
        const uint32_t h0 = rec[0];
        const uint64_t f = (uint64_t)rec[1] | ((uint64_t)rec[2] << 32);  // fields 0..10 (bits 0..63)
        const uint32_t f2 = rec[3];                                      // bits 64..95
        auto field = [&](int pos) -> uint32_t {
            return pos + 6 <= 64 ? (uint32_t)(f >> pos) & 63u
                                 : (pos >= 64 ? (f2 >> (pos - 64)) & 63u
                                              : (uint32_t)((f >> pos) | ((uint64_t)f2 << (64 - pos))) & 63u);
        };
        wsc[0] = wsc[1] = __fmul_rn(half_lo(h0), (float)field(6 * sb));
        wmin = __fmul_rn(half_hi(h0), (float)field(6 * (8 + sb)));
        const uint32_t* codes = rec + 4 + 8 * (sb >> 1);                 // sub-block 2p (low) / 2p+1 (high)
        const int sh = 4 * (sb & 1);
#pragma unroll
        for (int k = 0; k < 8; k++) w[k] = (codes[k] >> sh) & 0x0F0F0F0Fu;
    } else if constexpr (WT == WT_IQ1_M) {         // 64 B codes | 4 B signs | 6 B three-bit s | f16 d
        const uint32_t* rec = st + 19 * (j >> 3);  // 76-byte records
        const int sb = j & 7;
        const uint64_t sbits = (uint64_t)rec[17] | ((uint64_t)rec[18] << 32);   // bytes 68..75
        const float d = half_hi(rec[18]);                                         // bytes 74..75
#pragma unroll
        for (int h = 0; h < 2; h++)
            wsc[h] = __fmul_rn(__fmul_rn(d, (float)(2u * (uint32_t)((sbits >> (3 * (2 * sb + h))) & 7u) + 1u)), 0.125f);
        gsign = (rec[16] >> (4 * sb)) & 15u;                             // one bit per 8 values
#pragma unroll
        for (int p = 0; p < 2; p++) {
            // code word p: byte i holds the 2-bit codes of values 16p + 4i .. + 3 at bits 0-1, 2-3, 4-5,
            // 6-7; a_t = 8 * code of value 4i + t in byte i, then a byte transpose gives the four words
            const uint32_t cw = rec[2 * sb + p];
            const uint32_t a0 = (cw << 3) & 0x18181818u, a1 = (cw << 1) & 0x18181818u;
            const uint32_t a2 = (cw >> 1) & 0x18181818u, a3 = (cw >> 3) & 0x18181818u;
            const uint32_t lo01 = __byte_perm(a0, a1, 0x5140), hi01 = __byte_perm(a0, a1, 0x7362);
            const uint32_t lo23 = __byte_perm(a2, a3, 0x5140), hi23 = __byte_perm(a2, a3, 0x7362);
            const uint32_t v[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                                   __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
#pragma unroll
            for (int i = 0; i < 4; i++) w[4 * p + i] = v[i];           // 8 * code (the kernel adds k_g * S_g)
        }
    } else {                                        // q6_K: int8 sc[16] | f16 d | pad | four 48 B records
        const uint32_t* rec = st + 56 * (j >> 3);  // 224-byte records
        const int sb = j & 7;
        const float d = half_lo(rec[4]);
        const uint32_t scw = rec[sb >> 1] >> (16 * (sb & 1));            // sc of sub-blocks 2sb, 2sb + 1
#pragma unroll
        for (int h = 0; h < 2; h++) wsc[h] = __fmul_rn(d, (float)(int8_t)((scw >> (8 * h)) & 0xFFu));
        const uint32_t* lo = rec + 8 + 12 * (sb >> 1);                   // stage record: 8 low, 4 high words
        const int hh = sb & 1;
#pragma unroll
        for (int k = 0; k < 8; k++) {                                    // values 32hh + 4k .. + 3 of the stage
            const uint32_t l = (lo[k] >> (4 * hh)) & 0x0F0F0F0Fu;
            const uint32_t hi = ((lo[8 + (k & 3)] >> (2 * (2 * hh + (k >> 2)))) & 0x03030303u) << 4;
            w[k] = ((l | hi) + 0x60606060u) ^ 0x80808080u;                // code - 32 (see bias_byte)
        }
    }
}

// CTA of WARPS warps per group of RPC weight rows (grid-stride over row groups); MT tokens.  xq: int8
// codes [MT][K]; xds: (d, s) [MT][K/32].  A row is walked in segments of WARPS chunks: warp w copies chunk
// w of the segment of every row of the group into shared memory (all of the segment's weight bytes in
// flight at once: one memory round trip per segment instead of one per chunk), decodes its chunk's blocks
// (one per lane) and writes each block's f32 term per row and token to shared memory.  Thread t < RPC*MT
// then adds row t/MT's terms for token t%MT in block order, one dependent chain per (row, token).
//
// MoE mode (ID): blockIdx.y is one (token, slot) pair of the MUL_MAT_ID product, each a one-token product
// with its expert's weights: W then holds n_experts matrices of N rows, the pair's expert comes from ids,
// and the output row is token * slots + slot.  An id outside [0, n_experts) sets MMQ_DEVERR_EXPERT_ID and
// leaves the row unwritten; a token listing an expert twice sets MMQ_DEVERR_DUP_EXPERT (both rows are
// still computed), as the routing pass of the tile path does.
template <int WT, int MT, bool ID = false>
__global__ void __launch_bounds__(WARPS * 32) mmvq_kernel(const uint8_t* __restrict__ W_, long long row_bytes,
                                                        const int8_t* __restrict__ xq_,
                                                        const float2* __restrict__ xds_, float* __restrict__ out_,
                                                        int N, int K, const int32_t* __restrict__ ids = nullptr,
                                                        int slots = 1, int n_experts = 1) {
    static_assert(!ID || MT == 1, "the MoE mode runs one token per (token, slot) pair");
    constexpr int TPB = per16(WT) ? 2 : 1;        // terms per block
    constexpr int TSEG = WARPS * CHUNK * TPB;     // terms of one row and token per segment
    static_assert(RPC * MT <= WARPS * 32, "one summing thread per (row, token)");
    __shared__ __align__(16) uint32_t stage[RPC][WARPS][stage_words(WT)];
    constexpr uint32_t kRowStride = WARPS * stage_words(WT) * 4;   // bytes from stage[r][w] to stage[r + 1][w]
    constexpr int kUnits16 = chunk_bytes(WT) / 16, kWords = chunk_bytes(WT) / 4;
    __shared__ __align__(16) float terms[RPC][MT][TSEG];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = K / 32, nchunks = (nb + CHUNK - 1) / CHUNK, nseg = (nchunks + WARPS - 1) / WARPS;
    const bool row16 = (row_bytes & 15) == 0 && (reinterpret_cast<uintptr_t>(W_) & 15) == 0;
    const int sr = threadIdx.x / MT, sm = threadIdx.x % MT;   // summing thread: row sr, token sm
    const uint8_t* W = W_;
    const int8_t* xq = xq_;
    const float2* xds = xds_;
    float* out = out_;
    if (!ID && (long long)blockIdx.x * RPC < N) {
        // the first segment of the first row group's rows into L2 while the kernel before this one
        // finishes (whole rows measured slower for the three-segment q6_K rows: the extra prefetches compete
        // with the previous kernel's traffic)
        const long long n0 = (long long)blockIdx.x * RPC;
        const int prow = (int)min(row_bytes, (long long)WARPS * chunk_bytes(WT));   // the first segment
        const int rows_pf = (int)min((long long)RPC, N - n0);
        const uint8_t* base = W + n0 * row_bytes;
        for (int o = threadIdx.x * 128; o < rows_pf * prow; o += WARPS * 32 * 128) {
            const int r = o / prow, c = o - r * prow;
            prefetch_l2(base + r * row_bytes + c);
        }
    }
    pdl_wait();
    pdl_trigger();
    if constexpr (ID) {
        const int pair = blockIdx.y, t = pair / slots, j = pair - t * slots;
        const int e = ids[pair];
        if (threadIdx.x == 0 && blockIdx.x == 0) {
            unsigned err = (e < 0 || e >= n_experts) ? DEVERR_EXPERT_ID : 0u;
            for (int i = 0; i < j; i++)
                if (ids[(long long)t * slots + i] == e) err |= DEVERR_DUP_EXPERT;
            if (err) atomicOr(&g_mmq_device_errors, err);
        }
        if (e < 0 || e >= n_experts) return;   // uniform over the CTA
        W += (long long)e * N * row_bytes;
        xq += (long long)t * K;
        xds += (long long)t * (K / 32);
        out += (long long)pair * N;
    }
    for (long long g = blockIdx.x; g * RPC < N; g += gridDim.x) {
        const long long n0 = g * RPC;
        const int rows = (int)min((long long)RPC, N - n0);
        float acc = 0.0f;                          // row n0 + sr, token sm (threads below RPC * MT)
        for (int sg = 0; sg < nseg; sg++) {
            const int c = sg * WARPS + warp;       // this warp's chunk
            const int nblk = c < nchunks ? min(CHUNK, nb - c * CHUNK) : 0;
            if (nblk > 0) {
                // every row's chunk c, 16-byte copies that bypass L1 where the rows allow it (the weight
                // stream then does not evict the activations every row reads); the copy loops are unrolled
                // at compile time over a whole chunk's units and predicated (runtime-bounded loops here
                // cost more instructions than the decode)
                const int bytes = nblk * chunk_bytes(WT) / CHUNK;             // whole words: K % 256 == 0
                const uint8_t* src0 = W + n0 * row_bytes + (long long)c * chunk_bytes(WT);
                const uint32_t dst0 = smem_u32(stage[0][warp]);
                if (row16 && (bytes & 15) == 0) {
                    const int units = bytes >> 4;
#pragma unroll
                    for (int r = 0; r < RPC; r++) {
                        if (r < rows) {
#pragma unroll
                            for (int u = 0; u < kUnits16; u += 32) {
                                const int i = u + lane;
                                if (i < units) cp_async_16(dst0 + r * kRowStride + 16 * i, src0 + r * row_bytes + 16 * i, 16);
                            }
                        }
                    }
                } else {
                    const int words = bytes >> 2;
#pragma unroll
                    for (int r = 0; r < RPC; r++) {
                        if (r < rows) {
#pragma unroll
                            for (int u = 0; u < kWords; u += 32) {
                                const int i = u + lane;
                                if (i < words) cp_async_4(dst0 + r * kRowStride + 4 * i, src0 + r * row_bytes + 4 * i, 4);
                            }
                        }
                    }
                }
            }
            cp_async_commit();
            // the block's activations, every token, while the weights are in flight
            int4 x0[MT], x1[MT];
            float2 ds[MT];
            if (lane < nblk) {
                const int b = c * CHUNK + lane;
#pragma unroll
                for (int m = 0; m < MT; m++) {
                    const int4* xp = reinterpret_cast<const int4*>(xq + (long long)m * K + 32 * b);
                    x0[m] = __ldg(xp);
                    x1[m] = __ldg(xp + 1);
                    ds[m] = __ldg(xds + (long long)m * nb + b);
                }
            }
            // Q4_0 codes stay unsigned (0..15): the block dot is sum(code * q) - 8 * sum(q), exact in int32,
            // with 8 * sum(q) formed once per token and shared by the group's rows
            int sq8[MT];
            // IQ1_M, one or two tokens: a value is 8 * code + k_g, k_g = -9 (sign bit of group g set) or
            // -7, so the block dot is dp4a(8 * code, q) + sum_g k_g * S_g with S_g the token's sum over
            // group g, formed once per token and shared by the rows.  More tokens would hold 4 sums each;
            // there the rows add k_g per byte once instead (measured: the sums cost registers from 3 tokens)
            int gs[WT == WT_IQ1_M && MT <= 2 ? MT : 1][4];
            if constexpr (WT == WT_IQ1_M && MT <= 2) {
#pragma unroll
                for (int m = 0; m < MT; m++) {
                    const int e1 = 0x01010101;
                    gs[m][0] = __dp4a(e1, x0[m].y, __dp4a(e1, x0[m].x, 0));
                    gs[m][1] = __dp4a(e1, x0[m].w, __dp4a(e1, x0[m].z, 0));
                    gs[m][2] = __dp4a(e1, x1[m].y, __dp4a(e1, x1[m].x, 0));
                    gs[m][3] = __dp4a(e1, x1[m].w, __dp4a(e1, x1[m].z, 0));
                }
            }
#pragma unroll
            for (int m = 0; m < MT; m++) {
                int t = 0;
                if constexpr (WT == WT_Q4_0) {
                    const int e8 = 0x08080808;
                    t = __dp4a(e8, x0[m].x, t);
                    t = __dp4a(e8, x0[m].y, t);
                    t = __dp4a(e8, x0[m].z, t);
                    t = __dp4a(e8, x0[m].w, t);
                    t = __dp4a(e8, x1[m].x, t);
                    t = __dp4a(e8, x1[m].y, t);
                    t = __dp4a(e8, x1[m].z, t);
                    t = __dp4a(e8, x1[m].w, t);
                }
                sq8[m] = t;
            }
            cp_async_wait<0>();
            __syncwarp();                          // every lane's copies of the chunk have landed
            if (lane < nblk) {
#pragma unroll
                for (int r = 0; r < RPC; r++) {
                    if (r >= rows) break;
                    uint32_t w[8];
                    float wsc[2], wmin;
                    uint32_t gsign;
                    decode_block<WT>(stage[r][warp], lane, w, wsc, wmin, gsign);
                    // IQ1_M: value = 8 * code + k_g, k_g = -9 for a set sign bit of group g, else -7
                    int kg[4] = {0, 0, 0, 0};
                    if constexpr (WT == WT_IQ1_M && MT <= 2) {
#pragma unroll
                        for (int g4 = 0; g4 < 4; g4++) kg[g4] = ((gsign >> g4) & 1u) ? -9 : -7;
                    } else if constexpr (WT == WT_IQ1_M) {
#pragma unroll
                        for (int k = 0; k < 8; k++)     // 8 * code + (-7 | -9) per byte (see bias_byte)
                            w[k] = (w[k] + (((gsign >> (k >> 1)) & 1u) ? 0x77777777u : 0x79797979u)) ^ 0x80808080u;
                    }
#pragma unroll
                    for (int m = 0; m < MT; m++) {
                        int I0 = 0, I1 = WT == WT_Q4_0 ? -sq8[m] : 0;
                        I0 = __dp4a((int)w[0], x0[m].x, I0);
                        I0 = __dp4a((int)w[1], x0[m].y, I0);
                        I0 = __dp4a((int)w[2], x0[m].z, I0);
                        I0 = __dp4a((int)w[3], x0[m].w, I0);
                        I1 = __dp4a((int)w[4], x1[m].x, I1);
                        I1 = __dp4a((int)w[5], x1[m].y, I1);
                        I1 = __dp4a((int)w[6], x1[m].z, I1);
                        I1 = __dp4a((int)w[7], x1[m].w, I1);
                        if constexpr (WT == WT_IQ1_M && MT <= 2) {
                            I0 += kg[0] * gs[m][0] + kg[1] * gs[m][1];
                            I1 += kg[2] * gs[m][2] + kg[3] * gs[m][3];
                        }
                        float* tp = &terms[r][m][(warp * CHUNK + lane) * TPB];
                        if constexpr (per16(WT)) {
                            tp[0] = __fmul_rn(__fmul_rn(ds[m].x, wsc[0]), (float)I0);
                            tp[1] = __fmul_rn(__fmul_rn(ds[m].x, wsc[1]), (float)I1);
                        } else {
                            float u = __fmul_rn(__fmul_rn(ds[m].x, wsc[0]), (float)(I0 + I1));
                            if constexpr (WT == WT_Q4_K) u = __fsub_rn(u, __fmul_rn(wmin, ds[m].y));
                            tp[0] = u;
                        }
                    }
                }
            }
            __syncthreads();                       // the segment's terms of every row are written
            if (threadIdx.x < RPC * MT && sr < rows) {
                // block order: chunk by chunk (warp order), block by block (lane order), halves in order
                const float4* tp = reinterpret_cast<const float4*>(terms[sr][sm]);
                const int nt = TPB * min(nb - sg * WARPS * CHUNK, WARPS * CHUNK);   // a multiple of 8
                for (int q = 0; q < nt / 4; q++) {
                    const float4 v = tp[q];
                    acc = __fadd_rn(acc, v.x);
                    acc = __fadd_rn(acc, v.y);
                    acc = __fadd_rn(acc, v.z);
                    acc = __fadd_rn(acc, v.w);
                }
            }
            __syncthreads();                       // terms and staged chunks are consumed
        }
        if (threadIdx.x < RPC * MT && sr < rows) out[(long long)sm * N + n0 + sr] = acc;
    }
}

template <int WT>
cudaError_t launch_m(dim3 g, dim3 b, cudaStream_t s, const uint8_t* w, long long row_bytes, const int8_t* xq,
                     const float2* xds, float* out, long long M, long long N, long long K) {
    switch (M) {
        case 1: return launch_pdl(mmvq_kernel<WT, 1>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 2: return launch_pdl(mmvq_kernel<WT, 2>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 3: return launch_pdl(mmvq_kernel<WT, 3>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 4: return launch_pdl(mmvq_kernel<WT, 4>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 5: return launch_pdl(mmvq_kernel<WT, 5>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 6: return launch_pdl(mmvq_kernel<WT, 6>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 7: return launch_pdl(mmvq_kernel<WT, 7>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        case 8: return launch_pdl(mmvq_kernel<WT, 8>, g, b, s, w, row_bytes, xq, xds, out, (int)N, (int)K, nullptr, 1, 1);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gemv

cudaError_t run_gemv_id(int wt, const void* W, long long row_bytes, int n_experts, const void* Xq,
                        const int32_t* ids, int slots, float* out, long long M, long long N, long long K,
                        cudaStream_t s) {
    if (M < 1 || M > MMVQ_MAX_M || K % 256 != 0 || slots < 1 || M * slots > kMaxGemvPairs)
        return cudaErrorInvalidValue;
    const long long pairs = M * slots;
    // one CTA per (row group, pair), no grid-stride rounds: capping the grid at 16 CTAs per SM (as the
    // dense launch does) measured 10 % slower for 8 pairs of 384 row groups
    const long long gx = (N + gemv::RPC - 1) / gemv::RPC;
    const uint8_t* w = static_cast<const uint8_t*>(W);
    const int8_t* xq = static_cast<const int8_t*>(Xq);
    const float2* xds = reinterpret_cast<const float2*>(static_cast<const uint8_t*>(Xq) + M * K);
    const dim3 g((unsigned)gx, (unsigned)pairs), b(gemv::WARPS * 32);
    const int iN = (int)N, iK = (int)K;
    switch (wt) {
        case WT_Q8_0: return launch_pdl(gemv::mmvq_kernel<WT_Q8_0, 1, true>, g, b, s, w, row_bytes, xq, xds, out, iN, iK, ids, slots, n_experts);
        case WT_Q4_0: return launch_pdl(gemv::mmvq_kernel<WT_Q4_0, 1, true>, g, b, s, w, row_bytes, xq, xds, out, iN, iK, ids, slots, n_experts);
        case WT_Q4_K: return launch_pdl(gemv::mmvq_kernel<WT_Q4_K, 1, true>, g, b, s, w, row_bytes, xq, xds, out, iN, iK, ids, slots, n_experts);
        case WT_IQ1_M: return launch_pdl(gemv::mmvq_kernel<WT_IQ1_M, 1, true>, g, b, s, w, row_bytes, xq, xds, out, iN, iK, ids, slots, n_experts);
        case WT_Q6_K: return launch_pdl(gemv::mmvq_kernel<WT_Q6_K, 1, true>, g, b, s, w, row_bytes, xq, xds, out, iN, iK, ids, slots, n_experts);
    }
    return cudaErrorInvalidValue;
}

cudaError_t run_gemv(int wt, const void* W, long long row_bytes, const void* Xq, float* out, long long M, long long N,
                     long long K, cudaStream_t s) {
    if (M < 1 || M > MMVQ_MAX_M || K % 256 != 0) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long grid = (N + gemv::RPC - 1) / gemv::RPC;
    if (sms > 0 && grid > (long long)sms * 16) grid = (long long)sms * 16;
    const uint8_t* w = static_cast<const uint8_t*>(W);
    const int8_t* xq = static_cast<const int8_t*>(Xq);
    const float2* xds = reinterpret_cast<const float2*>(static_cast<const uint8_t*>(Xq) + M * K);
    const dim3 g((unsigned)grid), b(gemv::WARPS * 32);
    cudaError_t e = cudaErrorInvalidValue;
    switch (wt) {
        case WT_Q8_0: e = gemv::launch_m<WT_Q8_0>(g, b, s, w, row_bytes, xq, xds, out, M, N, K); break;
        case WT_Q4_0: e = gemv::launch_m<WT_Q4_0>(g, b, s, w, row_bytes, xq, xds, out, M, N, K); break;
        case WT_Q4_K: e = gemv::launch_m<WT_Q4_K>(g, b, s, w, row_bytes, xq, xds, out, M, N, K); break;
        case WT_IQ1_M: e = gemv::launch_m<WT_IQ1_M>(g, b, s, w, row_bytes, xq, xds, out, M, N, K); break;
        case WT_Q6_K: e = gemv::launch_m<WT_Q6_K>(g, b, s, w, row_bytes, xq, xds, out, M, N, K); break;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

MMQ_DEFINE_ERROR_READER(gemv)

}  // namespace mmq
