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

// Single-block routing for problems of up to ROUTE_FUSED_MAX_ROWS (token, slot) rows and
// ROUTE_FUSED_MAX_EXPERTS experts: count, scan and scatter in one launch with the counters in shared
// memory.  Same lists and error bits as the three-kernel route above.
constexpr int RF_THREADS = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        warp_tot[lane] = ti - t;                    // exclusive warp offsets
        if (lane == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    const int r = warp_tot[warp] + inc - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(RF_THREADS) route_fused_kernel(const int32_t* __restrict__ ids, int M, int slots,
                                                                 int E, int tile_n, int max_work, int* work,
                                                                 int* nwork, int* rowlist) {
    __shared__ int cnt[ROUTE_FUSED_MAX_EXPERTS], off[ROUTE_FUSED_MAX_EXPERTS], cur[ROUTE_FUSED_MAX_EXPERTS];
    __shared__ int warp_tot[33];
    for (int e = threadIdx.x; e < E; e += RF_THREADS) {
        cnt[e] = 0;
        cur[e] = 0;
    }
    __syncthreads();
    unsigned err = 0;
    for (int t = threadIdx.x; t < M; t += RF_THREADS) {
        for (int j = 0; j < slots; j++) {
            const int e = ids[(long long)t * slots + j];
            if (e < 0 || e >= E) {
                err |= DEVERR_EXPERT_ID;
                continue;
            }
            for (int i = 0; i < j; i++)
                if (ids[(long long)t * slots + i] == e) err |= DEVERR_DUP_EXPERT;
            atomicAdd(&cnt[e], 1);
        }
    }
    if (err) atomicOr(&g_mmq_device_errors, err);
    __syncthreads();
    // E <= RF_THREADS: thread e scans expert e's row count and its number of work items
    const int e = threadIdx.x;
    const int c = e < E ? cnt[e] : 0;
    int tot_rows, tot_items;
    const int o = block_exclusive_scan(c, warp_tot, tot_rows);
    const int ni = (c + tile_n - 1) / tile_n;
    const int oi = block_exclusive_scan(ni, warp_tot, tot_items);
    if (e < E) {
        off[e] = o;
        for (int i = 0; i < ni && oi + i < max_work; i++) {
            work[3 * (oi + i) + 0] = e;
            work[3 * (oi + i) + 1] = o + i * tile_n;
            work[3 * (oi + i) + 2] = min(tile_n, c - i * tile_n);
        }
    }
    if (threadIdx.x == 0) *nwork = min(tot_items, max_work);
    __syncthreads();
    for (int i = threadIdx.x; i < M * slots; i += RF_THREADS) {
        const int ex = ids[i];
        if (ex < 0 || ex >= E) continue;
        rowlist[off[ex] + atomicAdd(&cur[ex], 1)] = i;
    }
}

bool route_fused_supported(long long M, int slots, int E) {
    return E <= ROUTE_FUSED_MAX_EXPERTS && M * slots <= ROUTE_FUSED_MAX_ROWS;
}

cudaError_t run_route_fused(const int32_t* ids, int M, int slots, int E, int tile_n, const RouteWorkspace& ws,
                            cudaStream_t s) {
    route_fused_kernel<<<1, RF_THREADS, 0, s>>>(ids, M, slots, E, tile_n, ws.max_work, ws.work, ws.nwork, ws.rowlist);
    return cudaGetLastError();
}

MMQ_DEFINE_ERROR_READER(route)

}  // namespace mmq
