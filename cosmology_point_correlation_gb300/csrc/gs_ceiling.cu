// gs_ceiling.cu -- measured ceilings of the counting kernels' inner loops.
//
// The triangle count is not bound by HBM: its rows are re-read from L2 and
// every closed triangle costs one shared-memory atomic add into a histogram.
// This probe measures how many such adds an SM retires per second when the
// adds do nothing else, with the address pattern of the count: each lane adds
// 1 to a counter of a histogram of `ncfg` 32-bit entries in shared memory,
// `lanes_active` lanes of every warp taking part. The count's adds per second
// divided by this rate is how close the count is to the atomic ceiling.

#include <algorithm>

#include "gs_internal.cuh"

constexpr int CEIL_THREADS = 512;
constexpr int CEIL_ADDR = 16;            // addresses held per thread, cycled

// PATTERN 0: independent pseudo-random counters in [0, ncfg) per lane;
// 1: lane l of every warp uses counter l + 32 q (no two lanes share a bank);
// 2: every lane uses counter 0 (all lanes of a warp on one address).
template <int PATTERN>
__global__ void __launch_bounds__(CEIL_THREADS, 2)
k_smem_atomic_rate(int ncfg, int lanes_active, int iters, unsigned long long *sink)
{
    extern __shared__ unsigned s_h[];
    for (int t = threadIdx.x; t < ncfg; t += CEIL_THREADS) s_h[t] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    unsigned addr[CEIL_ADDR];
    uint32_t x = (blockIdx.x * CEIL_THREADS + threadIdx.x) * 0x9E3779B1u + 0x7f4a7c15u;
#pragma unroll
    for (int q = 0; q < CEIL_ADDR; ++q) {
        x = x * 1664525u + 1013904223u;
        addr[q] = PATTERN == 0 ? (x >> 8) % (unsigned)ncfg
                : PATTERN == 1 ? (unsigned)(lane + 32 * q) % (unsigned)ncfg : 0u;
    }
    if (lane < lanes_active) {
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int q = 0; q < CEIL_ADDR; ++q) atomicAdd(&s_h[addr[q]], 1u);
        }
    }
    __syncthreads();
    unsigned long long v = 0;
    for (int t = threadIdx.x; t < ncfg; t += CEIL_THREADS) v += s_h[t];
    if (v) atomicAdd(sink, v);           // keeps the adds observable; equals the adds made
}

extern "C" gs_status gs_measure_smem_atomics(int ncfg, int pattern, int lanes_active, double *lane_adds_per_s,
                                             void *cuda_stream)
{
    GS_ENTRY();
    if (!lane_adds_per_s || ncfg < 32 || ncfg > 27648 || pattern < 0 || pattern > 2 || lanes_active < 1 ||
        lanes_active > 32)
        return gs_set_error(GS_ERR_ARG, "ncfg in [32, 27648], pattern in 0..2, lanes_active in 1..32");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    auto kern = pattern == 0 ? k_smem_atomic_rate<0> : pattern == 1 ? k_smem_atomic_rate<1> : k_smem_atomic_rate<2>;
    const size_t dyn = sizeof(unsigned) * (size_t)ncfg;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    const int grid = gs_sm_count() * 2;
    unsigned long long *sink = nullptr, got = 0;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    GS_TRY_CUDA(gs_malloc_async(&sink, sizeof(unsigned long long), st));
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    int iters = 64;
    float ms = 0.f;
    // grow the run until it takes at least 20 ms (the first launches also warm up)
    for (int round = 0; e == cudaSuccess && round < 12; ++round) {
        e = cudaMemsetAsync(sink, 0, sizeof(unsigned long long), st);
        if (e == cudaSuccess) e = cudaEventRecord(e0, st);
        if (e == cudaSuccess) {
            kern<<<grid, CEIL_THREADS, dyn, st>>>(ncfg, lanes_active, iters, sink);
            gs_note_launch();
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) e = cudaEventRecord(e1, st);
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
        if (e == cudaSuccess) e = cudaMemcpy(&got, sink, sizeof(got), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess || ms >= 20.f) break;
        iters *= 2;
    }
    const double adds = (double)grid * (CEIL_THREADS / 32) * lanes_active * (double)iters * CEIL_ADDR;
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFreeAsync(sink, st);
    if (e != cudaSuccess) return gs_set_error(GS_ERR_CUDA, "atomic-rate probe: %s", cudaGetErrorString(e));
    if ((double)got != adds) return gs_set_error(GS_ERR_INTERNAL, "atomic-rate probe lost adds");
    *lane_adds_per_s = adds / (ms * 1e-3);
    return GS_OK;
}
