// peaks.cu -- dense int8 mma.sync and FP32 FMA throughput probes (declared in include/mmq_peaks.h).
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/mmq_peaks.h"

namespace {

// Eight independent m16n8k32 s8 accumulator chains per warp keep the tensor pipe busy.
__global__ void __launch_bounds__(512) int8_mma_kernel(int* sink, int iters) {
    int c[8][4];
#pragma unroll
    for (int j = 0; j < 8; j++)
#pragma unroll
        for (int i = 0; i < 4; i++) c[j][i] = 0;
    const int a0 = threadIdx.x, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3, b0 = a0 * 3, b1 = a0 * 5;
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int j = 0; j < 8; j++)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};\n"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    if (s == 0x7fffffff) sink[0] = s;
}

__global__ void __launch_bounds__(1024) ffma_kernel(float* sink, int iters, float a, float b) {
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; i++) r[i] = threadIdx.x * 1e-3f + i;
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int u = 0; u < 16; u++)
#pragma unroll
            for (int i = 0; i < 8; i++) r[i] = fmaf(r[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) s += r[i];
    if (s == 1234.5f) sink[0] = s;
}

template <typename F>
int time_kernel(F launch, cudaStream_t s, double* ms_out) {
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    launch();                                   // warm-up
    cudaEventRecord(e0, s);
    launch();
    cudaEventRecord(e1, s);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *ms_out = ms;
    return (int)err;
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace

extern "C" int mmq_peak_int8_mma_sync(double* out_tops, int iters, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* sink = nullptr;
    if (cudaMalloc(&sink, 64) != cudaSuccess) return (int)cudaGetLastError();
    const int blocks = sm_count() * 2, threads = 512;
    double ms = 0;
    int err = time_kernel([&] { int8_mma_kernel<<<blocks, threads, 0, s>>>(sink, iters); }, s, &ms);
    if (err == 0) err = (int)cudaGetLastError();
    cudaFree(sink);
    const double ops = (double)blocks * (threads / 32) * iters * 8 * (16.0 * 8 * 32 * 2);
    *out_tops = err == 0 && ms > 0 ? ops / (ms * 1e-3) / 1e12 : 0.0;
    return err;
}

extern "C" int mmq_peak_ffma(double* out_tflops, int iters, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* sink = nullptr;
    if (cudaMalloc(&sink, 64) != cudaSuccess) return (int)cudaGetLastError();
    const int blocks = sm_count() * 2, threads = 1024;
    double ms = 0;
    int err = time_kernel([&] { ffma_kernel<<<blocks, threads, 0, s>>>(sink, iters, 0.9999f, 1e-4f); }, s, &ms);
    if (err == 0) err = (int)cudaGetLastError();
    cudaFree(sink);
    const double flops = (double)blocks * threads * iters * 16 * 8 * 2;
    *out_tflops = err == 0 && ms > 0 ? flops / (ms * 1e-3) / 1e12 : 0.0;
    return err;
}
