// route.cu -- MoE routing for MUL_MAT_ID ("CUDA: add IQ1_M to MMQ", PR description: each token times
// each of its routed experts).  Three small kernels build, on the device and without any host
// synchronisation, the list of (token, slot) rows grouped by expert and the work items (expert,
// first row, row count <= tile width) that the grouped GEMM walks.
#include <cstdint>
#include "internal.h"
#include "mmq_device.cuh"

namespace mmq {

__global__ void route_count_kernel(const int32_t* __restrict__ ids, int M, int slots, int E, int* counts,
                                   int* cursor) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= M) return;
    unsigned err = 0;
    for (int j = 0; j < slots; j++) {
        const int e = ids[(long long)t * slots + j];
        if (e < 0 || e >= E) {
            err |= DEVERR_EXPERT_ID;
            continue;
        }
        for (int i = 0; i < j; i++)
            if (ids[(long long)t * slots + i] == e) err |= DEVERR_DUP_EXPERT;
        atomicAdd(counts + e, 1);
    }
    if (err) atomicOr(&g_mmq_device_errors, err);
}

// One thread: exclusive scan of the per-expert counts and the work-item list.
__global__ void route_scan_kernel(const int* __restrict__ counts, int E, int tile_n, int max_work, int* offsets,
                                  int* cursor, int* work, int* nwork) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int off = 0, nw = 0;
    for (int e = 0; e < E; e++) {
        const int c = counts[e];
        offsets[e] = off;
        cursor[e] = 0;
        for (int st = 0; st < c && nw < max_work; st += tile_n) {
            work[3 * nw + 0] = e;
            work[3 * nw + 1] = off + st;
            work[3 * nw + 2] = min(tile_n, c - st);
            nw++;
        }
        off += c;
    }
    *nwork = nw;
}

__global__ void route_scatter_kernel(const int32_t* __restrict__ ids, int M, int slots, int E,
                                     const int* __restrict__ offsets, int* cursor, int* rowlist) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= (long long)M * slots) return;
    const int e = ids[i];
    if (e < 0 || e >= E) return;
    const int pos = offsets[e] + atomicAdd(cursor + e, 1);
    rowlist[pos] = (int)i;
}

__global__ void route_zero_kernel(int* counts, int E) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = 0;
}

cudaError_t run_route(const int32_t* ids, int M, int slots, int E, int tile_n, const RouteWorkspace& ws,
                      cudaStream_t s) {
    route_zero_kernel<<<1, 256, 0, s>>>(ws.counts, E);
    route_count_kernel<<<(M + 127) / 128, 128, 0, s>>>(ids, M, slots, E, ws.counts, ws.cursor);
    route_scan_kernel<<<1, 32, 0, s>>>(ws.counts, E, tile_n, ws.max_work, ws.offsets, ws.cursor, ws.work, ws.nwork);
    const long long rows = (long long)M * slots;
    route_scatter_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(ids, M, slots, E, ws.offsets, ws.cursor,
                                                                        ws.rowlist);
    return cudaGetLastError();
}

MMQ_DEFINE_ERROR_READER(route)

}  // namespace mmq
