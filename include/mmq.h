/*
 * mmq.h -- C ABI of the GB300 (sm_103a) block-quantized int8 MMQ library (libmmq_gb300.so).
 *
 * MMQ is the block-quantized integer matrix multiply that governs LLM prefill:
 *
 *     out[m,n] = sum_kb (xs[m,kb] * wd[n,kb]) * sum_{k in kb} xq[m,k] * wq[n,k]
 *
 * ("When the Product Won't Collapse: A Negative Result on int8 Tensor-Core MMQ", §2, the blockwise
 * contraction; "08 · R1 — int8 MMQ prefill GEMM", §2.1-§2.2).  Activations are quantized per 32-k block
 * to q8_1 (int8 codes, an f32 scale d and an f32 block sum s = d * sum(q)); weights stay in their raw
 * block formats and are unpacked to integer tiles inside the kernel; each 32-k block is an exact
 * integer dot and its f32 scale correction is applied in registers.
 *
 * Conventions for every entry point:
 *   - M = tokens (activation rows), N = weight rows (output features), K = reduction length.
 *   - All buffer pointers are DEVICE pointers owned by the caller.  The library allocates, frees and
 *     synchronises nothing; every call only enqueues kernels on `stream` (0 = the legacy default
 *     stream) and returns.  Buffers must not overlap unless stated.
 *   - Stream order is kept.  The quantizer and the few-token (M <= 8) product launch as programmatic
 *     dependents: their CTAs may start while the previous kernel in the stream is still running, but
 *     they read and write no global memory until it has completed (the few-token kernel only issues L2
 *     prefetch hints for its weights before that point, which cannot change what any load returns).
 *   - Pointers must be 16-byte aligned.
 *   - Argument errors are reported synchronously as a status code and nothing is enqueued.
 *     Launch failures are reported as MMQ_ERR_CUDA.  Conditions that can only be seen on the device
 *     (an expert id out of range, an internal pipeline wait that exceeded its time limit) set bits in
 *     a device-resident error word that mmq_read_device_errors() returns and clears.
 *
 * Byte layouts (this library's; the pages give block sizes, not bit layouts):
 *   q8_1 activations (mmq_q8_1_bytes(M,K) bytes), five sections:
 *       int8 q[M][K]                    at byte 0            the q8_1 codes
 *       float2 ds[M][K/32] = (d, s)     at byte M*K          per-block scale and block sum
 *       fp16 h[M][K]                    at byte H = round_up(M*K + 8*M*K/32, 256)
 *                                                            h = q exactly (tensor-core operand)
 *       f32 dT[K/32][Mp], sT[K/32][Mp]  at byte T = round_up(H + 2*M*K, 256) and T + 4*Mp*K/32,
 *                                                            Mp = M rounded up to 4: d and s
 *                                                            block-major (the GEMM's 128-token boxes)
 *       The first two sections are the q8_1 blocks (40 B per 32 values); the last three are derived
 *       from them (mmq_q8_1_prepare) so that the GEMM reads tensor-core-ready operands.
 *   Q8_0  34 B / 32 values : f16 d | int8 q[32]                        value = d*q
 *   Q4_0  18 B / 32 values : f16 d | 16 B, byte i = code i (low nibble) | code i+16 (high nibble)
 *                            value = d*(code-8)
 *   Q4_K 144 B / 256 values: f16 d | f16 dmin | 12 B little-endian bit stream of 16 six-bit fields
 *                            (sc[0..7] then m[0..7]) | 128 B codes, byte 32j+i = code 64j+i (low
 *                            nibble) | code 64j+32+i (high nibble); sub-block b = values 32b..32b+31;
 *                            value = d*sc_b*code - dmin*m_b
 *   IQ1_M 76 B / 256 values: 64 B 2-bit codes (value i at bits 2(i%4) of byte i/4, g = code-1 in
 *                            {-1,0,1}) | 4 B sign bits (bit j of the little-endian word covers values
 *                            8j..8j+7; 0 -> delta=+1/8, 1 -> delta=-1/8) | 6 B little-endian bit stream
 *                            of 16 three-bit sub-scales s (s_h covers values 16h..16h+15) | f16 d;
 *                            value = d*(2s+1)*(g+delta)
 *   Q6_K 224 B / 256 values: int8 sc[16] (sc_h covers values 16h..16h+15) | f16 d | 14 B zero | four
 *                            48 B stage records j = 0..3: 32 B, byte i = low nibble of code 64j+i |
 *                            low nibble of code 64j+32+i << 4; 16 B, byte i = high 2 bits of codes
 *                            64j+i, 64j+16+i, 64j+32+i, 64j+48+i at bits 0-1, 2-3, 4-5, 6-7;
 *                            code in 0..63, value = d*sc_h*(code-32)  ("08 · R1", §2.2: 6-bit grid,
 *                            signed domain by subtracting 32, scales on 16-element sub-blocks)
 *   W8A8 weights           : int8 W[N][K] followed by f32 ws[N]        (mmq_weight_bytes)
 *   W8A8 activations       : int8 X[M][K] followed by f32 xs[M]        (mmq_w8a8_act_bytes)
 *   Weights are row-major over N: row n is its K/values-per-block blocks back to back.
 *
 * Shape rules: M >= 0, N >= 0 (any value; tails are masked; M == 0 or N == 0 is a no-op).  K > 0 and
 * K % 256 == 0 for the block types (Q8_0, Q4_0, Q4_K, IQ1_M, Q6_K: the kernels stage raw weights in
 * 256-value super-stages); K % 64 == 0 for W8A8 and for q8_1 activation buffers (64-value stages).
 * M*K and N*K below 2^31.  Every size helper returns 0 for exactly the shapes its entry point rejects
 * with MMQ_ERR_SHAPE (mmq_weight_bytes: mmq_gemm's rule for the type; mmq_q8_1_bytes:
 * mmq_quantize_q8_1's; mmq_w8a8_act_bytes: W8A8's).
 * Q6_K runs on the TMA-fed kernel only: mmq_gemm and mmq_gemm_id take it; mmq_gemm_debug_partials
 * and mmq_gemm_id_noalloc return MMQ_ERR_UNSUPPORTED for it (as they do for W8A8).
 */
#ifndef MMQ_GB300_H
#define MMQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (identical type). */
typedef struct CUstream_st* mmq_stream_t;

typedef enum {
    MMQ_Q8_0 = 0,
    MMQ_Q4_0 = 1,
    MMQ_Q4_K = 2,
    MMQ_IQ1_M = 3,
    MMQ_W8A8 = 4,
    MMQ_Q6_K = 5
} mmq_type;

typedef enum {
    MMQ_OK = 0,
    MMQ_ERR_INVALID_ARG = 1,   /* null pointer, unknown type, negative size */
    MMQ_ERR_SHAPE = 2,         /* K (or M, N) violates the shape rules above */
    MMQ_ERR_ALIGN = 3,         /* a pointer is not 16-byte aligned */
    MMQ_ERR_UNSUPPORTED = 4,   /* valid request the library does not implement */
    MMQ_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
    MMQ_ERR_WORKSPACE = 6      /* workspace pointer null or smaller than required */
} mmq_status;

/* Device-side error bits returned by mmq_read_device_errors(). */
#define MMQ_DEVERR_TIMEOUT     1u  /* a pipeline wait exceeded its limit; the kernel ended early */
#define MMQ_DEVERR_EXPERT_ID   2u  /* an expert id was outside [0, n_experts); that row was skipped */
#define MMQ_DEVERR_DUP_EXPERT  4u  /* a token listed the same expert twice */

/* Human-readable name of a status code (static string, never NULL). */
const char* mmq_status_string(mmq_status s);

/* Name and description of the CUDA error behind the most recent MMQ_ERR_CUDA returned on the calling
 * host thread ("" if none).  The string stays valid until the next failing call on that thread. */
const char* mmq_last_cuda_error(void);

/* Bytes of a q8_1 activation buffer for an [M][K] matrix, all sections (0 unless K > 0, K % 64 == 0). */
size_t mmq_q8_1_bytes(int64_t M, int64_t K);

/* Bytes of a raw weight buffer of type t with N rows of K values (W8A8: N*K + 4*N).  0 for an unknown
 * type or a shape mmq_gemm rejects (K % 256 for the block types, K % 64 for W8A8). */
size_t mmq_weight_bytes(mmq_type t, int64_t N, int64_t K);

/* Bytes of a W8A8 activation buffer: M*K + 4*M (0 unless K > 0, K % 64 == 0). */
size_t mmq_w8a8_act_bytes(int64_t M, int64_t K);

/*
 * mmq_quantize_q8_1 -- activation quantizer ("08 · R1", §2.2 and the §3.2 reference quantizer).
 * x   : f32 [M][K], row-major, device.
 * xq  : output q8_1 buffer of mmq_q8_1_bytes(M, K) bytes, device.
 * Per row and 32-value block: amax = max|x|; d = amax/127 (f32, round to nearest); q = round-half-even
 * of the correctly rounded f32 x/d, clamped to [-127,127]; s = d*(float)sum(q).  amax == 0 gives
 * d = 0, q = 0, s = 0.  Inputs must be finite.  K % 64 == 0.  Writes all five sections.
 */
mmq_status mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, void* xq, mmq_stream_t stream);

/*
 * mmq_q8_1_prepare -- fill the derived sections (h, dT, sT) of a q8_1 buffer from its q and ds
 * sections, for callers that produce q8_1 blocks themselves.  mmq_quantize_q8_1 already does this.
 * Exact: h = q as fp16; dT, sT are d and s transposed (pad columns up to Mp zero).
 */
mmq_status mmq_q8_1_prepare(void* xq, int64_t M, int64_t K, mmq_stream_t stream);

/*
 * mmq_gemm -- dense MMQ product ("A Negative Result on int8 Tensor-Core MMQ", §2; "08 · R1", §3.2
 * per-block correction; "CUDA: add IQ1_M to MMQ", Design, for IQ1_M; "INT8 W8A8 GEMM — Prefill",
 * §1, for W8A8).
 * W   : raw weights of type wtype, N rows (mmq_weight_bytes(wtype, N, K) bytes).
 * Xq  : q8_1 activations from mmq_quantize_q8_1 (block types) or a W8A8 activation buffer.
 * out : f32 [M][N] row-major for the block types; bf16 [M][N] for W8A8.
 * Block types: out[m,n] = sum_b scale_b * I_b with the exact int32 block dot I_b and the f32 scale
 * products of the layouts above (Q4_K adds -dmin*m_b*s[m,b]; IQ1_M has per-16 scales d(2s+1)/8).
 * W8A8: I = exact int32 dot over the full K, out = bf16_rne(((float)I * xs[m]) * ws[n]).
 * Summation order: for M <= 8 tokens (block types) the block terms are added in block order, so out equals
 * the blockwise definition evaluated in that order bit for bit; larger M runs on the tensor-core kernels,
 * which may add them in another f32 order (and, for K split over CTAs, with atomics), within 1e-3 of the
 * output scale.  W8A8 is bit-exact at every M.
 */
mmq_status mmq_gemm(mmq_type wtype, const void* W, const void* Xq, void* out,
                    int64_t M, int64_t N, int64_t K, mmq_stream_t stream);

/*
 * mmq_gemm_debug_block_sums -- the production (TMA-fed) kernel's exact integer accumulators.
 * Instead of the product, writes sums[m][n][b] (int32 [M][N][K/32]) = the 32-k block dot of token row m
 * and weight row n with the weights' integer sub-scale factors folded in, as the kernel's converters fold
 * them: Q8_0 q, Q4_0 code-8, Q4_K sc_b*code, IQ1_M (2s+1)*(8g+-1) per 16 values, Q6_K sc_h*(code-32) per
 * 16 values ("08 · R1", §2.1: the in-block integer dot is exact; §2.2 for the K-quant sub-scales).  For
 * parity checks of the tensor-core path, bit for bit; block types on shapes the TMA-fed kernel takes
 * (K % 256 == 0; IQ1_M K % 1024 == 0), else MMQ_ERR_UNSUPPORTED.  sums is caller-owned, 16-byte aligned.
 */
mmq_status mmq_gemm_debug_block_sums(mmq_type wtype, const void* W, const void* Xq, int32_t* sums,
                                     int64_t M, int64_t N, int64_t K, mmq_stream_t stream);

/*
 * mmq_gemm_id -- MoE MUL_MAT_ID ("CUDA: add IQ1_M to MMQ", PR description): each token times each of
 * its routed experts.
 * W          : n_experts expert weight matrices of type wtype (block types only), back to back, each
 *              N rows of K values.
 * Xq         : q8_1 activations for M tokens.
 * expert_ids : int32 [M][n_slots], device; ids[t][j] in [0, n_experts), distinct per token.
 * out        : f32 [M][n_slots][N]; out[t][j][:] = W_{ids[t][j]} applied to token t.
 * workspace  : caller-owned device scratch of at least mmq_gemm_id_workspace_bytes(M, K, n_slots,
 *              n_experts) bytes, 16-byte aligned; its contents on entry do not matter.  It holds the
 *              routing lists and, for the TMA-fed kernel, a gathered copy of the routed token rows
 *              (fp16 codes and block scales, about 2*K + K/4 bytes per (token, slot) row).
 * Routing (count, scan, scatter), the gather and the grouped product run on the device with no host
 * synchronisation.  Out-of-range ids set MMQ_DEVERR_EXPERT_ID and their rows are left unwritten.
 * For M <= 8 tokens (and M*n_slots <= 65535) the call runs one matrix-vector kernel instead, which reads
 * the ids itself: each (token, slot) row is a one-token product with its expert, summed in the blockwise
 * definition's order, and the workspace is not touched (it is still required and checked).
 */
size_t mmq_gemm_id_workspace_bytes(int64_t M, int64_t K, int n_slots, int n_experts);
mmq_status mmq_gemm_id(mmq_type wtype, const void* W, int n_experts, const void* Xq,
                       const int32_t* expert_ids, int n_slots, float* out,
                       int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                       mmq_stream_t stream);

/*
 * mmq_gemm_id_noalloc -- mmq_gemm_id for callers that cannot allocate device memory.  The pages have
 * no counterpart: it exists for integrations where cudaMalloc is not available or not allowed (code
 * inside a memory-budgeted serving engine or a framework's caching allocator, plugins that are given
 * only their input and output buffers), which cannot provide mmq_gemm_id's workspace.
 * Arguments and results are those of mmq_gemm_id without the workspace.  The routing lists live in a
 * file-scope device array of MMQ_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the
 * library until the process exits; the call itself allocates nothing.  It runs the general kernel on
 * the token rows in place (no gathered copy); for M <= 8 tokens, the matrix-vector kernel of
 * mmq_gemm_id, which uses no routing lists.  Problems whose routing lists need more than the array
 * (per-expert counts, offsets and cursors, 12 bytes per work item with ceil(M*n_slots/128) + n_experts
 * items, 4 bytes per (token, slot) row, each list rounded up to 256 bytes) are rejected with
 * MMQ_ERR_WORKSPACE.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture.  All calls share the array: calls whose kernels may overlap on the GPU (unordered streams)
 * race and must be serialised by the caller.
 */
#define MMQ_NOALLOC_SCRATCH_BYTES (1u << 20)
mmq_status mmq_gemm_id_noalloc(mmq_type wtype, const void* W, int n_experts, const void* Xq,
                               const int32_t* expert_ids, int n_slots, float* out,
                               int64_t M, int64_t N, int64_t K, mmq_stream_t stream);

/*
 * mmq_gemm_debug_partials -- debug mode: the exact per-group integer dots the tensor-core path
 * computes ("08 · R1", §2.1: the in-block int8 dot is exact in int32).
 * partials : int32 [M][N][K/G], G = 16 for IQ1_M (per-16 halves, values 8g±1), else 32; for W8A8 the
 *            groups are 32-k chunks of the full-K dot.
 */
mmq_status mmq_gemm_debug_partials(mmq_type wtype, const void* W, const void* Xq, int32_t* partials,
                                   int64_t M, int64_t N, int64_t K, mmq_stream_t stream);

/*
 * mmq_read_device_errors -- synchronises `stream`, returns the device error bits accumulated by all
 * previous calls on the current device (MMQ_DEVERR_*) and clears them.  Returns MMQ_ERR_CUDA if the
 * read fails.
 */
mmq_status mmq_read_device_errors(unsigned* bits, mmq_stream_t stream);

/*
 * mmq_selftest_bounded_wait -- device self-test of the bounded pipeline waits.  Two CTAs each wait on a
 * shared-memory mbarrier that nothing arrives at, one with the polling wait and one with the sleeping
 * wait the pipelines use.  Each wait must give up after the library's time limit (~2 s), raise its CTA's
 * abort flag, record MMQ_DEVERR_TIMEOUT and return; the kernel then exits normally.
 * result : int32 [4], device, 16-byte aligned: per CTA {wait completed (0 expected), abort flag (1)}.
 * Enqueues on `stream`; read the error bits with mmq_read_device_errors afterwards.
 */
mmq_status mmq_selftest_bounded_wait(int32_t* result, mmq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MMQ_GB300_H */
