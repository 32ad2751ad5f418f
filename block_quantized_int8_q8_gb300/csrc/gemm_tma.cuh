// gemm_tma.cuh -- the production MMQ kernel of the block types (dense and MoE): TMA-fed, converter-group
// pipelined, register rescale.
//
// Computes out[m,n] = sum_b wd[n,b] * xd[m,b] * I[m,n,b] (Q4_K: minus dmin*m_b*s[m,b]) with the exact
// per-block integer dot I[m,n,b] = sum_{k in b} xq[m,k] * wq[n,k]  ("A Negative Result on int8
// Tensor-Core MMQ", §2; "08 · R1 — int8 MMQ prefill GEMM", §2.1-§2.2 and §3.2).
//
// Pipeline of one CTA (128 weight rows x 128 tokens, all of K or one part of it):
//   * loader warp (one thread): TMA loads of (a) raw weight bytes, one "super-stage" of 256 k (IQ1_M:
//     1024 k) for the 128 rows, into a two-slot raw ring; (b) the token operand, fp16 codes of the
//     q8_1 shadow, 64 k x 128 tokens with the 128-byte swizzle straight into the MMA operand ring;
//     (c) the tokens' block scales d (Q4_K also s) from the block-major shadow into a scale ring.
//   * a converter group (two warps; four for IQ1_M and q6_K, and for every type on dense grids of at
//     most 64 tokens): each thread takes two weight rows in one unrolled body (one row with four warps),
//     reads its raw bytes from the raw ring (16-byte loads,
//     conflict-free: the row pitch is an odd number of 16-byte units), unpacks them EXACTLY to fp16
//     integers (the unpackers of gemm.cuh; q6_K's below), stores the 128B-swizzled K-major operand row
//     (q6_K: two rows, its sub-block scale split over two exact operands) and the row's block scales.
//   * MMA warp: four tcgen05.mma kind::f16 (M=128, N=128, K=16) per 64-k stage (q6_K: eight) into one
//     of two stage buffers of two 128-column TMEM accumulators; a commit per stage hands it on.
//   * sixteen epilogue warps: tcgen05.ld each finished block and apply acc += I * (xd * wd) in packed
//     f32 pairs in registers ("A Negative Result", §2-§4: no shared-memory round trip of the
//     accumulator).  IQ1_M's per-16 scale (2s+1), Q4_K's 6-bit and q6_K's int8 sub-block scales are
//     folded into the integer operand (exact), so their block scale is the super-block d (IQ1_M: d/8).
// Two stage buffers let the MMAs of stage s+1 run while the epilogue rescales stage s.
#pragma once
#include <cuda.h>
#include "gemm.cuh"

namespace mmq {
namespace tma {

// Operand ring (A converted by the converters, B by TMA): four stages; q6_K carries two A tiles per stage
// (its sub-block scale split over two exactly representable operands) and three stages to fit.
template <int WT> struct Ring {
    static constexpr int kStages = (WT == WT_Q6_K) ? 3 : 4;
    static constexpr int kATiles = (WT == WT_Q6_K) ? 2 : 1;
    static constexpr int kAStage = kATiles * A_STAGE_BYTES;
};
constexpr int SC = 8;                // scale ring depth (converters run up to 4 stages ahead of the
                                     // MMA, the epilogue trails it by up to 2)
constexpr int RAW_SLOTS = 2;
constexpr int NACC = 4;              // 128-column TMEM accumulators: two stage buffers of two blocks
constexpr int NSB = NACC / 2;        // stage buffers handed between the MMA warp and the epilogue
constexpr int EPI_WARPS = 16;         // four per TMEM lane quarter
constexpr int EPI_COLS = BN * 4 / EPI_WARPS;   // tokens per epilogue thread (32)
constexpr int EPI_CHUNKS = EPI_COLS / 16;      // 16-column TMEM loads per block
// Warp roles per weight type: 16 epilogue warps, the converter warps, the MMA warp, the TMA loader warp.
// Two converter warps (two weight rows per thread) serve Q8_0 / Q4_0 / Q4_K and leave 96 registers per
// thread (20 warps; four warps of one row measured slower from 128 tokens on); the unpacks of IQ1_M and
// q6_K are the heaviest per row and get four (22 warps, 80 registers; two warps of two rows measured
// 1.3-1.8x slower).  CV overrides the converter count: dense grids of at most 64 tokens, whose epilogue
// warps are mostly idle, run Q8_0 / Q4_0 / Q4_K with four (Q4_K 16-64 tokens: 12-20 % faster).
template <int WT> constexpr int default_conv() { return (WT == WT_IQ1_M || WT == WT_Q6_K) ? 4 : 2; }
template <int WT, int CV = default_conv<WT>()> struct Warps {
    static constexpr int kConv = CV;
    static constexpr int kRowsPerConv = BM / (kConv * 32);
    static constexpr int kConv0 = EPI_WARPS;
    static constexpr int kMma = kConv0 + kConv;
    static constexpr int kLoad = kMma + 1;
    static constexpr int kThreads = (kLoad + 1) * 32;
};
constexpr long long ABORT_DRAIN_CYCLES = 2000000;   // ~1 ms: lets in-flight TMA writes land after an abort

// Raw super-stage geometry: U 16-byte units per weight row in shared memory (the TMA box width; odd, so
// the converters' 16-byte row reads are conflict-free), UG units per super-stage in global memory, SS 64-k
// operand stages per super-stage.
template <int WT> struct Geom;
template <> struct Geom<WT_Q8_0> { static constexpr int U = 17, UG = 17, SS = 4; };    // 8 blocks x 34 B
template <> struct Geom<WT_Q4_0> { static constexpr int U = 9, UG = 9, SS = 4; };      // 8 blocks x 18 B
template <> struct Geom<WT_Q4_K> { static constexpr int U = 9, UG = 9, SS = 4; };      // one 144 B super-block
template <> struct Geom<WT_IQ1_M> { static constexpr int U = 19, UG = 19, SS = 16; };  // four 76 B super-blocks
// q6_K: one 224 B super-block, read as a 240 B box (the 16 B past it belong to the next super-block or
// are zero-filled past the row end, and are never read)
template <> struct Geom<WT_Q6_K> { static constexpr int U = 15, UG = 14, SS = 4; };

template <int WT> struct Smem {
    static constexpr bool kMin = WT == WT_Q4_K;               // Q4_K min term needs xs and wmn
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + Ring<WT>::kStages * Ring<WT>::kAStage;
    static constexpr int raw_slot = (BM * Geom<WT>::U * 16 + 1023) / 1024 * 1024;
    static constexpr int raw_off = b_off + Ring<WT>::kStages * B_STAGE_BYTES;
    // one scale slot: xd[2][128] (TMA) | xs[2][128] (TMA, Q4_K) | wd[2][128] | wmn[2][128] (Q4_K)
    static constexpr int xd_off = 0;
    static constexpr int xs_off = 1024;
    static constexpr int wd_off = kMin ? 2048 : 1024;
    static constexpr int wmn_off = 3072;
    static constexpr int sc_slot = kMin ? 4096 : 2048;
    static constexpr int sc_off = raw_off + RAW_SLOTS * raw_slot;
    static constexpr int bar_off = sc_off + SC * sc_slot;
    static constexpr int n_bars = 2 * Ring<WT>::kStages + 2 * RAW_SLOTS + 2 * SC + 2 * NSB + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int total = misc_off + 16;
    static constexpr int alloc = total + 1024;                  // slack for 1024-byte alignment
    static_assert(alloc <= 232448, "shared memory budget");
};

// ------------------------------------------------------------------------------------------ TMA
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------------------ raw reads
// Copy NW consecutive 32-bit words starting at byte offset OFF of a raw row record (16-byte aligned
// base) into r[DST..DST+NW), with whole 16-byte loads.
template <int OFF, int NW, int DST>
__device__ __forceinline__ void raw_words(uint32_t rrow, RawA& r) {
    static_assert(OFF % 4 == 0, "word-aligned fields");
    constexpr int c0 = OFF / 16, w0 = (OFF % 16) / 4, nch = (w0 + NW + 3) / 4;
    uint32_t w[4 * nch];
#pragma unroll
    for (int c = 0; c < nch; c++) {
        const uint4 v = ld_shared_u4(rrow + 16 * (c0 + c));
        w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < NW; i++) r.w[DST + i] = w[w0 + i];
}

// The raw words of operand stage J of a super-stage, in the word order the unpackers expect.
template <int WT, int J>
__device__ __forceinline__ void load_raw(uint32_t rrow, RawA& r) {
    if constexpr (WT == WT_Q8_0) {
        raw_words<68 * J, 17, 0>(rrow, r);                     // blocks 2J, 2J+1
    } else if constexpr (WT == WT_Q4_0) {
        raw_words<36 * J, 9, 0>(rrow, r);
    } else if constexpr (WT == WT_Q4_K) {
        raw_words<0, 4, 0>(rrow, r);                           // d, dmin, 12 B of scales
        raw_words<16 + 32 * J, 8, 4>(rrow, r);                 // codes of sub-blocks 2J, 2J+1
    } else if constexpr (WT == WT_IQ1_M) {
        constexpr int sbk = J / 4, jj = J % 4;
        raw_words<76 * sbk + 16 * jj, 4, 0>(rrow, r);          // 64 two-bit codes
        raw_words<76 * sbk + 64, 3, 4>(rrow, r);               // signs, sub-scales, d
    } else {
        raw_words<0, 5, 0>(rrow, r);                           // sc[16], d
        raw_words<32 + 48 * J, 12, 5>(rrow, r);                // stage record: 32 B low nibbles, 16 B high pairs
    }
}

// q6_K, operand stage J of a super-block ("08 · R1 — int8 MMQ prefill GEMM", §2.2: 6-bit grid 0..63
// moved to the signed domain by subtracting 32; scales on 16-element sub-blocks).  The int8 sub-block
// scale sc = 16*sh + sl (sl in 0..15, sh in -8..7) is folded into two operands that fp16 holds exactly:
// A1 = (q-32)*sl, |A1| <= 480, and A2 = (q-32)*16*sh, a multiple of 16 with |A2| <= 4096.  Two MMAs
// add A1.B and A2.B into the block's accumulator, so it holds sum (q-32)*sc*x exactly (|.| <= 32*32*128*127
// < 2^24) and the block scale is the super-block d.  Sub-block g (values 16g..16g+15 of the stage) is
// operand chunks 2g, 2g+1 of both tiles.
template <int J>
__device__ __forceinline__ void q6k_stage_operands(const RawA& r, uint32_t at1, uint32_t at2, int row) {
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const int sc = (int)(int8_t)((r.w[J] >> (8 * g)) & 0xFFu);     // sub-block 4J+g
        const uint32_t m1 = f2_to_h2((float)(sc & 15), (float)(sc & 15));
        const uint32_t m2 = f2_to_h2((float)(16 * (sc >> 4)), (float)(16 * (sc >> 4)));
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 4; k++) {                                   // values 16g+4k .. 16g+4k+3
            const uint32_t lw = g < 2 ? r.w[5 + 4 * g + k] : (r.w[5 + 4 * (g - 2) + k] >> 4);
            const uint32_t code = (lw & 0x0F0F0F0Fu) | (((r.w[13 + k] >> (2 * g)) & 0x03030303u) << 4);
            u8x4_to_f16x4(code, 0x64206420u, h[2 * k], h[2 * k + 1]);  // 1024 + code - 1056 = code - 32
        }
        uint32_t a1[8], a2[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(a1[i]) : "r"(h[i]), "r"(m1));
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(a2[i]) : "r"(h[i]), "r"(m2));
        }
#pragma unroll
        for (int q = 0; q < 2; q++) {
            st_shared_v4(at1 + sw128_off(row, 2 * g + q), a1[4 * q], a1[4 * q + 1], a1[4 * q + 2], a1[4 * q + 3]);
            st_shared_v4(at2 + sw128_off(row, 2 * g + q), a2[4 * q], a2[4 * q + 1], a2[4 * q + 2], a2[4 * q + 3]);
        }
    }
}

// ------------------------------------------------------------------------------------------ kernel
struct Ctx {
    uint32_t sb;             // shared-window address of the 1024-aligned tile base
    uint32_t bar0;
    volatile int* abort_flag;
    int pt;                  // first weight row of this converter thread (rows pt + 32*kConv*i)
    int rows_valid;          // weight rows of the tile below N
    bool ok;
};

template <int WT> struct Bars {
    __device__ static uint32_t full(const Ctx& c, int i) { return c.bar0 + 8u * i; }
    __device__ static uint32_t empty(const Ctx& c, int i) { return c.bar0 + 8u * (Ring<WT>::kStages + i); }
    __device__ static uint32_t rfull(const Ctx& c, int i) { return c.bar0 + 8u * (2 * Ring<WT>::kStages + i); }
    __device__ static uint32_t rempty(const Ctx& c, int i) { return c.bar0 + 8u * (2 * Ring<WT>::kStages + RAW_SLOTS + i); }
    __device__ static uint32_t sfull(const Ctx& c, int i) { return c.bar0 + 8u * (2 * Ring<WT>::kStages + 2 * RAW_SLOTS + i); }
    __device__ static uint32_t sfree(const Ctx& c, int i) {
        return c.bar0 + 8u * (2 * Ring<WT>::kStages + 2 * RAW_SLOTS + SC + i);
    }
    __device__ static uint32_t accf(const Ctx& c, int i) {
        return c.bar0 + 8u * (2 * Ring<WT>::kStages + 2 * RAW_SLOTS + 2 * SC + i);
    }
    __device__ static uint32_t acce(const Ctx& c, int i) {
        return c.bar0 + 8u * (2 * Ring<WT>::kStages + 2 * RAW_SLOTS + 2 * SC + NSB + i);
    }
    __device__ static uint32_t done(const Ctx& c) {
        return c.bar0 + 8u * (2 * Ring<WT>::kStages + 2 * RAW_SLOTS + 2 * SC + 2 * NSB);
    }
};

// Convert operand stage s = t*SS + J of raw super-stage t (this thread: weight rows c.pt + 32*CV*i).
template <int WT, int CV, int J>
__device__ __forceinline__ void convert_stage(Ctx& c, int t, uint32_t raw) {
    using L = Smem<WT>;
    using B = Bars<WT>;
    if (!c.ok) return;
    const int s = t * Geom<WT>::SS + J;
    const int slot = s % Ring<WT>::kStages, ss = s % SC;
    if (!mbar_wait_relaxed(B::empty(c, slot), ((s / Ring<WT>::kStages) & 1) ^ 1, c.abort_flag) ||
        !mbar_wait_relaxed(B::sfree(c, ss), ((s / SC) & 1) ^ 1, c.abort_flag)) {
        c.ok = false;
        return;
    }
    const uint32_t at = c.sb + L::a_off + slot * Ring<WT>::kAStage;
    const uint32_t scs = c.sb + L::sc_off + ss * L::sc_slot;
    // both rows of a 2-row thread in one unrolled body: the second row's raw loads and unpack overlap the
    // first's (measured +9 % on Q4_0, +4 % on Q4_K against one row at a time)
#pragma unroll
    for (int rr = 0; rr < Warps<WT, CV>::kRowsPerConv; rr++) {
        const int row = c.pt + rr * CV * 32;
        RawA r;
        load_raw<WT, J>(raw + row * Geom<WT>::U * 16, r);
        float wsc[2], wmn[2] = {0.f, 0.f};
        if constexpr (WT == WT_Q6_K) {
            q6k_stage_operands<J>(r, at, at + A_STAGE_BYTES, row);
            wsc[0] = wsc[1] = half_bits_to_float((uint16_t)(r.w[4] & 0xFFFFu));   // super-block d
        } else {
            uint32_t h[32];
            // the unpackers use only s % 4 (the stage's place in a 256-value super-block); K ranges start
            // on super-stage boundaries, so the local index gives the same value and keeps it a
            // compile-time one
            unpack_a<WT, true>(r, s, h, wsc, wmn);
#pragma unroll
            for (int q = 0; q < 8; q++)
                st_shared_v4(at + sw128_off(row, q), h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
        }
        if (row >= c.rows_valid) wsc[0] = wsc[1] = wmn[0] = wmn[1] = 0.f;
        st_shared_f32(scs + L::wd_off + 4 * row, wsc[0]);
        st_shared_f32(scs + L::wd_off + 4 * (BM + row), wsc[1]);
        if constexpr (L::kMin) {
            st_shared_f32(scs + L::wmn_off + 4 * row, wmn[0]);
            st_shared_f32(scs + L::wmn_off + 4 * (BM + row), wmn[1]);
        }
    }
    fence_proxy_async_smem();        // the operand row -> tensor core
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        mbar_arrive(B::full(c, slot));
        mbar_arrive(B::sfull(c, ss));
    }
}

template <int WT, int CV, int J, int NJ>
struct ConvUnroll {
    __device__ static __forceinline__ void run(Ctx& c, int t, uint32_t rrow) {
        convert_stage<WT, CV, J>(c, t, rrow);
        ConvUnroll<WT, CV, J + 1, NJ>::run(c, t, rrow);
    }
};
template <int WT, int CV, int NJ>
struct ConvUnroll<WT, CV, NJ, NJ> {
    __device__ static __forceinline__ void run(Ctx&, int, uint32_t) {}
};

template <int WT, int CV>
__device__ __forceinline__ void converter_loop(Ctx& c, int nsuper) {
    using L = Smem<WT>;
    using B = Bars<WT>;
    constexpr int SS = Geom<WT>::SS;
    for (int t = 0; t < nsuper; t++) {
        const int rs = t & 1;
        if (!c.ok || !mbar_wait_relaxed(B::rfull(c, rs), (t >> 1) & 1, c.abort_flag)) {
            c.ok = false;
            return;
        }
        ConvUnroll<WT, CV, 0, SS>::run(c, t, c.sb + L::raw_off + rs * L::raw_slot);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(B::rempty(c, rs));
    }
}

// acc += I * (xd * wd) (Q4_K also -(dmin*m_b) * s[m,b]) for one 16-lane half of a warp's TMEM
// quarter, in the 16x256b fragment layout: v[4j + 2e + c] is row 8e + t/4 of the half, column
// 8j + 2(t%4) + c of the warp's 32 columns.  xd2[j] / xs2[j] hold the two column scales of group j,
// w[e] / mn[e] the row scales.
template <bool MIN>
__device__ __forceinline__ void rescale_half(uint64_t (&acc2)[8], const uint32_t (&v)[16], const uint64_t (&xd2)[4],
                                             const uint64_t (&xs2)[4], const float (&w)[2], const float (&mn)[2]) {
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const uint64_t w2 = f2_pack(w[e], w[e]);
        const uint64_t nmn2 = f2_pack(-mn[e], -mn[e]);
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int a = 4 * e + jj, r = 4 * jj + 2 * e;
            acc2[a] = f2_fma(f2_pack(__uint_as_float(v[r]), __uint_as_float(v[r + 1])), f2_mul(xd2[jj], w2), acc2[a]);
            if constexpr (MIN) acc2[a] = f2_fma(nmn2, xs2[jj], acc2[a]);
        }
    }
}

// MoE (MUL_MAT_ID) mode of the kernel: work item w = (expert, first rowlist entry, row count <= 128)
// as the routing pass lists them, and the item's first row in the gathered operand (a multiple of 4).
struct MoeTiles {
    const int* work;         // [3 * max_work]: expert, start, count; null in dense mode
    const int* nwork;        // number of valid items
    const int* gstart;       // [max_work]
    const int* rowlist;      // (token, slot) row of each routed entry, grouped by expert
    int sms;                 // multiprocessors (one CTA each)
    int kparts;              // largest K split (1, 2 or 4) that keeps whole raw super-stages per part
};

// Tail split of T tiles over `sms` one-CTA-per-SM slots: when the last wave holds r tiles and P*r CTAs
// still fit in one wave, those r tiles are computed as P parts of their K range each (P = 4 or 2, at
// most kparts).  The first nf = T - r tiles run whole.  Returns log2(P) (0: no split).
__host__ __device__ __forceinline__ int tail_split(int T, int sms, int kparts, int& nf, int& r) {
    nf = T;
    r = 0;
    if (sms <= 0 || T <= sms) return 0;
    const int rr = T - (T - 1) / sms * sms;
    const int lg = (kparts >= 4 && 4 * rr <= sms) ? 2 : ((kparts >= 2 && 2 * rr <= sms) ? 1 : 0);
    if (lg > 0) {
        nf = T - rr;
        r = rr;
    }
    return lg;
}

// DBG: instead of the rescale, the epilogue stores every 32-k block's exact integer accumulator (the weights'
// integer sub-scales folded in, as the converters fold them) to int32 [M][N][K/32] at `out`; dense, whole
// K range per CTA.
template <int WT, bool MOE, bool DBG = false, int CV = default_conv<WT>()>
__global__ void __launch_bounds__(Warps<WT, CV>::kThreads, 1)
    mmq_gemm_tma_kernel(const __grid_constant__ CUtensorMap tm_raw, const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_xd, const __grid_constant__ CUtensorMap tm_xs,
                        float* __restrict__ out, int M, int N, int K, int ntn, int nfull, int lgp,
                        const MoeTiles moe) {
    using L = Smem<WT>;
    using B = Bars<WT>;
    using W = Warps<WT, CV>;
    constexpr int U = Geom<WT>::U, UG = Geom<WT>::UG, SS = Geom<WT>::SS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tile of this CTA (weight-row tiles fastest).  Dense: CTAs past the first nfull take the remaining
    // tiles in groups of 2^lgp, each CTA one part of its tile's K range, all adding into a zeroed output
    // (with two parts the f32 result does not depend on their order).  MoE: CTA (item, weight-row tile)
    // multiplies expert e's rows by the item's gathered token rows; CTAs of items past the routed count
    // leave at once.
    int tile = blockIdx.x, part = -1, lgparts = 1;
    int n0, m0, wrow, mvalid, rl0 = 0;
    if constexpr (MOE) {
        // the tile count is known on the device only: CTAs past the tiles (and their tail parts) leave
        int nf, r;
        lgparts = tail_split(*moe.nwork * ntn, moe.sms, moe.kparts, nf, r);
        if (tile >= nf) {
            const int ci = tile - nf;
            if (ci >= (r << lgparts)) return;                  // uniform over the CTA, nothing set up yet
            tile = nf + (ci >> lgparts);
            part = ci & ((1 << lgparts) - 1);
        }
        const int w = tile / ntn;
        n0 = (tile % ntn) * BM;
        wrow = moe.work[3 * w] * N + n0;
        rl0 = moe.work[3 * w + 1];
        mvalid = moe.work[3 * w + 2];
        m0 = moe.gstart[w];
    } else {
        if (tile >= nfull) {
            const int ci = tile - nfull;
            tile = nfull + (ci >> lgp);
            part = ci & ((1 << lgp) - 1);
            lgparts = lgp;
        }
        n0 = (tile % ntn) * BM;
        m0 = (tile / ntn) * BN;
        wrow = n0;
        mvalid = M - m0;
    }
    // K range of this CTA: all stages, or part `part` of 2^lgparts, cut at raw super-stage boundaries
    int nstages = K / BK, s0 = 0;
    if (part >= 0) {
        const int nsup = K / BK / SS;
        const int t0 = (part * nsup) >> lgparts, t1 = ((part + 1) * nsup) >> lgparts;
        s0 = t0 * SS;
        nstages = (t1 - t0) * SS;
    }

    Ctx c;
    c.sb = smem_u32(smem);
    c.bar0 = c.sb + L::bar_off;
    c.abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
    c.pt = 0;
    c.rows_valid = N - n0;
    c.ok = true;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);

    if (warp == W::kMma) {
        if (lane == 0) {
            for (int i = 0; i < Ring<WT>::kStages; i++) {
                mbar_init(B::full(c, i), W::kConv + 1);     // converter warps + the B load
                mbar_init(B::empty(c, i), 1);
            }
            for (int i = 0; i < RAW_SLOTS; i++) {
                mbar_init(B::rfull(c, i), 1);
                mbar_init(B::rempty(c, i), W::kConv);
            }
            for (int i = 0; i < SC; i++) {
                mbar_init(B::sfull(c, i), W::kConv + 1);    // converter warps + the scale load
                mbar_init(B::sfree(c, i), EPI_WARPS);
            }
            for (int i = 0; i < NSB; i++) {
                mbar_init(B::accf(c, i), 1);
                mbar_init(B::acce(c, i), EPI_WARPS);
            }
            mbar_init(B::done(c), 1);
            *c.abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), NACC * BN);
        tmem_relinquish();
    } else if (warp == W::kLoad && lane == 0) {
        tma_prefetch_desc(&tm_raw);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_xd);
        if constexpr (L::kMin) tma_prefetch_desc(&tm_xs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == W::kLoad) {
        // =========================================================== TMA loader
        if (lane == 0) {
            for (int s = 0; s < nstages; s++) {
                if (s % SS == 0) {
                    const int t = s / SS, rs = t & 1;
                    if (!mbar_wait_relaxed(B::rempty(c, rs), ((t >> 1) & 1) ^ 1, c.abort_flag)) break;
                    mbar_arrive_expect_tx(B::rfull(c, rs), BM * U * 16);
                    if constexpr (U * 16 <= 256)
                        tma_load_2d(c.sb + L::raw_off + rs * L::raw_slot, &tm_raw, (t + s0 / SS) * UG * 16, wrow,
                                    B::rfull(c, rs));
                    else
                        tma_load_2d(c.sb + L::raw_off + rs * L::raw_slot, &tm_raw, (t + s0 / SS) * UG * 4, wrow,
                                    B::rfull(c, rs));
                }
                const int slot = s % Ring<WT>::kStages;
                if (!mbar_wait_relaxed(B::empty(c, slot), ((s / Ring<WT>::kStages) & 1) ^ 1, c.abort_flag)) break;
                mbar_arrive_expect_tx(B::full(c, slot), B_STAGE_BYTES);
                tma_load_2d(c.sb + L::b_off + slot * B_STAGE_BYTES, &tm_b, BK * (s + s0), m0, B::full(c, slot));
                const int ss = s % SC;
                if (!mbar_wait_relaxed(B::sfree(c, ss), ((s / SC) & 1) ^ 1, c.abort_flag)) break;
                const uint32_t scs = c.sb + L::sc_off + ss * L::sc_slot;
                mbar_arrive_expect_tx(B::sfull(c, ss), L::kMin ? 2048u : 1024u);
                tma_load_2d(scs + L::xd_off, &tm_xd, m0, 2 * (s + s0), B::sfull(c, ss));
                if constexpr (L::kMin) tma_load_2d(scs + L::xs_off, &tm_xs, m0, 2 * (s + s0), B::sfull(c, ss));
            }
        }
        __syncwarp();
    } else if (warp >= W::kConv0 && warp < W::kMma) {
        // =========================================================== converters
        c.pt = (warp - W::kConv0) * 32 + lane;
        converter_loop<WT, CV>(c, nstages / SS);
    } else if (warp == W::kMma) {
        // =========================================================== MMA issuer
        const uint32_t idesc = idesc_f16_f32(BM, BN);
        const uint32_t a_smem = c.sb + L::a_off;
        const uint32_t b_smem = c.sb + L::b_off;
        for (int s = 0; s < nstages; s++) {
            if (*c.abort_flag) break;
            const int slot = s % Ring<WT>::kStages;
            const int sb = s & (NSB - 1);      // stage buffer: accumulators 2*sb (block 2s), 2*sb+1 (block 2s+1)
            if (!mbar_wait(B::full(c, slot), (s / Ring<WT>::kStages) & 1, c.abort_flag)) break;
            mbar_wait(B::acce(c, sb), ((s / NSB) & 1) ^ 1, c.abort_flag);
            tc_fence_after();
            const uint64_t ad0 = sdesc_sw128(a_smem + slot * Ring<WT>::kAStage);
            const uint64_t bd0 = sdesc_sw128(b_smem + slot * B_STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int buf = 2 * sb + (j >> 1);
                // +32 bytes per 16-element K slice: +2 in the descriptor's address field
                if (elect_one()) umma_f16(tmem_base + buf * BN, ad0 + 2 * j, bd0 + 2 * j, idesc, j & 1);
                if constexpr (Ring<WT>::kATiles == 2) {       // q6_K: second operand tile, same block
                    const uint64_t ad1 = sdesc_sw128(a_smem + slot * Ring<WT>::kAStage + A_STAGE_BYTES);
                    if (elect_one()) umma_f16(tmem_base + buf * BN, ad1 + 2 * j, bd0 + 2 * j, idesc, 1u);
                }
            }
            if (elect_one()) {
                umma_commit(B::accf(c, sb));
                umma_commit(B::empty(c, slot));
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(B::done(c));
        __syncwarp();
        mbar_wait_final(B::done(c), 0);
        __syncwarp();
    } else {
        // =========================================================== epilogue
        // Each warp owns TMEM lane quarter q (weight rows 32q..32q+31) and tokens 32cq..32cq+31, read in
        // the 16x256b fragment layout: per 16-lane half h, thread t holds rows 16h + 8e + t/4 (e = 0, 1)
        // and tokens 8j + 2(t%4) + {0, 1} (j = 0..3).  A thread thus needs 4 row scales and 8 token
        // scales per block (two-lane-group loads, no whole-warp broadcast of the token scales).
        const int q = warp & 3;
        const int cq = warp >> 2;
        const int tq = lane >> 2, tc = lane & 3;
        const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + EPI_COLS * cq;
        // a warp whose token columns all lie past the tile's valid columns (a partly filled MoE tile, the
        // last dense token tile) only takes part in the hand-offs
        const bool active = EPI_COLS * cq < mvalid;
        uint64_t acc[2][8];                     // [half][4e + j]: packed f32 pair, tokens 8j + 2tc + {0, 1}
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int a = 0; a < 8; a++) acc[h][a] = 0ull;
        for (int s = 0; s < (active ? 0 : nstages); s++) {      // idle warp: hand-offs only
            const int sb = s & (NSB - 1), ss = s % SC;
            if (!mbar_wait(B::sfull(c, ss), (s / SC) & 1, c.abort_flag)) break;
            if (!mbar_wait(B::accf(c, sb), (s / NSB) & 1, c.abort_flag)) break;
            tc_fence_after();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B::acce(c, sb));
                mbar_arrive(B::sfree(c, ss));
            }
        }
        for (int s = 0; s < (active ? nstages : 0); s++) {
            const int sb = s & (NSB - 1), ss = s % SC;
            if (!mbar_wait(B::sfull(c, ss), (s / SC) & 1, c.abort_flag)) break;
            if (!mbar_wait(B::accf(c, sb), (s / NSB) & 1, c.abort_flag)) break;
            tc_fence_after();
            const uint32_t scs = c.sb + L::sc_off + ss * L::sc_slot;
            const uint32_t tacc = tb + 2 * sb * BN;
            // four chunks (block i, half h) in one software pipeline: the TMEM load of chunk k+1 is in
            // flight while chunk k is rescaled
            uint32_t va[16], vb[16];
            tmem_ld_16x256b_x4(tacc, va);
            tmem_ld_wait(va);
            uint64_t xd2[4], xs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int i = k >> 1, h = k & 1;                       // block of the stage, lane half
                const int kn = k + 1;
                uint32_t(&cur)[16] = (k & 1) ? vb : va;
                uint32_t(&nxt)[16] = (k & 1) ? va : vb;
                if (kn < 4) tmem_ld_16x256b_x4(tacc + (kn >> 1) * BN + ((uint32_t)(16 * (kn & 1)) << 16), nxt);
                if constexpr (DBG) {
                    int* dbg = reinterpret_cast<int*>(out);
                    const long long nb = K / 32, bglob = 2 * (s + s0) + i;
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int n = n0 + 32 * q + 16 * h + 8 * e + tq;
#pragma unroll
                        for (int jj = 0; jj < 4; jj++)
#pragma unroll
                            for (int c2 = 0; c2 < 2; c2++) {
                                const int col = EPI_COLS * cq + 8 * jj + 2 * tc + c2;
                                if (n < N && col < mvalid)
                                    dbg[((long long)(m0 + col) * N + n) * nb + bglob] =
                                        __float2int_rn(__uint_as_float(cur[4 * jj + 2 * e + c2]));
                            }
                    }
                } else {
                    if (h == 0) {                                      // token scales of block i
#pragma unroll
                        for (int jj = 0; jj < 4; jj++) {
                            const uint32_t col = EPI_COLS * cq + 8 * jj + 2 * tc;
                            const float2 x = ld_shared_f2(scs + L::xd_off + 4 * (i * BN + col));
                            xd2[jj] = f2_pack(x.x, x.y);
                            if constexpr (L::kMin) {
                                const float2 y = ld_shared_f2(scs + L::xs_off + 4 * (i * BN + col));
                                xs2[jj] = f2_pack(y.x, y.y);
                            }
                        }
                    }
                    float w[2], mn[2] = {0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int row = 32 * q + 16 * h + 8 * e + tq;
                        w[e] = ld_shared_f32(scs + L::wd_off + 4 * (i * BM + row));
                        if constexpr (L::kMin) mn[e] = ld_shared_f32(scs + L::wmn_off + 4 * (i * BM + row));
                    }
                    rescale_half<L::kMin>(acc[h], cur, xd2, xs2, w, mn);
                }
                if (kn < 4) tmem_ld_wait(nxt);
                if (kn == 3) {
                    tc_fence_before();          // every TMEM read of this stage buffer is complete
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B::acce(c, sb));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B::sfree(c, ss));
        }
        // ---- store: rows n0 + 32q + 16h + 8e + tq, token columns 32cq + 8j + 2tc + {0, 1} below mvalid;
        // output row of a column: m0 + column (dense) or its rowlist entry (MoE)
      if constexpr (!DBG) {
        int orow[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int col = EPI_COLS * cq + 8 * (i >> 1) + 2 * tc + (i & 1);
            if constexpr (MOE)
                orow[i] = col >= mvalid ? -1 : moe.rowlist[rl0 + col];
            else
                orow[i] = col >= mvalid ? -1 : m0 + col;
        }
#pragma unroll
        for (int h = 0; h < 2; h++) {
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int n = n0 + 32 * q + 16 * h + 8 * e + tq;
                if (n >= N) continue;
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    float a0, a1;
                    f2_unpack(acc[h][4 * e + jj], a0, a1);
                    const int r0 = orow[2 * jj], r1 = orow[2 * jj + 1];
                    if (part < 0) {
                        if (r0 >= 0) out[(long long)r0 * N + n] = a0;
                        if (r1 >= 0) out[(long long)r1 * N + n] = a1;
                    } else {
                        if (r0 >= 0) atomicAdd(out + (long long)r0 * N + n, a0);
                        if (r1 >= 0) atomicAdd(out + (long long)r1 * N + n, a1);
                    }
                }
            }
        }
      }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (*c.abort_flag) {
        // a wait gave up: give any TMA copy still in flight time to land before the CTA's shared
        // memory is released
        const long long t0 = clock64();
        while (clock64() - t0 < ABORT_DRAIN_CYCLES) {
        }
    }
    tc_fence_after();
    if (warp == W::kMma) tmem_dealloc(tmem_base, NACC * BN);
}

}  // namespace tma
}  // namespace mmq
