/*
 * mmq_peaks.h -- throughput probes used by the benchmark to state the roofline denominators that the
 * MMQ metric is quoted against (libmmq_peaks.so, built next to libmmq_gb300.so).
 *
 * "% of GB300 int8 peak" needs the int8 tensor rate of this part.  On sm_103a the tcgen05 MMA has no
 * int8 kind (ptxas rejects .kind::i8 for sm_103a), so the only int8 tensor-core path is the legacy
 * warp-level mma.sync.m16n8k32.s8 ("08 · R1 — int8 MMQ prefill GEMM", §2.1 names this instruction);
 * mmq_peak_int8_mma_sync measures its dense rate.  mmq_peak_ffma measures the FP32 FMA rate that
 * bounds the per-block f32 rescale.
 *
 * Both run one kernel over every SM of the current device on `stream`, synchronise it, and return the
 * rate through *out (TOPS for int8, TFLOP/s for FP32).  They allocate a 64-byte device scratch buffer
 * internally (cudaMalloc/cudaFree); they are measurement utilities, not part of the compute path.
 * Return 0 on success, a non-zero CUDA error code otherwise.
 */
#ifndef MMQ_PEAKS_H
#define MMQ_PEAKS_H
#ifdef __cplusplus
extern "C" {
#endif
int mmq_peak_int8_mma_sync(double* out_tops, int iters, void* stream);
int mmq_peak_ffma(double* out_tflops, int iters, void* stream);
#ifdef __cplusplus
}
#endif
#endif
