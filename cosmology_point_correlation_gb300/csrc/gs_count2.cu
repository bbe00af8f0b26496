// gs_count2.cu -- internal 2pCF pair counts on the graph (GRAMSCI v2, §III.3:
// the two-point function is computed on the same graph and radial bins as the
// higher-order counts, in one sweep of the graph).
//
// Every unordered pair {i, j} appears twice in the symmetric CSR (once in each
// row), so the pair count of bin b is half the number of edge bytes equal to b.
// The kernel streams the bin bytes with 16-byte vector loads into per-warp
// shared-memory histograms (fewer same-address collisions than one per block)
// and adds them into the caller's histogram once per block.

#include <algorithm>

#include "gs_internal.cuh"

constexpr int C2_THREADS = 256;
constexpr int C2_WARPS = C2_THREADS / 32;

__global__ void __launch_bounds__(C2_THREADS)
k_count2(const uint8_t *__restrict__ bin, int64_t n_edges, int nb, unsigned long long *__restrict__ hist)
{
    __shared__ unsigned s_h[C2_WARPS][256];
    const int warp = threadIdx.x >> 5;
    for (int t = threadIdx.x; t < C2_WARPS * 256; t += C2_THREADS) (&s_h[0][0])[t] = 0u;
    __syncthreads();
    unsigned *h = s_h[warp];
    // whole 16-byte vectors first (the bin array starts 256-byte aligned)
    const int64_t nvec = n_edges >> 4;
    const uint4 *v = reinterpret_cast<const uint4 *>(bin);
    for (int64_t q = (int64_t)blockIdx.x * C2_THREADS + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * C2_THREADS) {
        const uint4 x = __ldg(v + q);
        const unsigned w[4] = { x.x, x.y, x.z, x.w };
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int b = 0; b < 4; ++b) atomicAdd(&h[(w[k] >> (8 * b)) & 0xffu], 1u);
    }
    for (int64_t e = (nvec << 4) + (int64_t)blockIdx.x * C2_THREADS + threadIdx.x; e < n_edges;
         e += (int64_t)gridDim.x * C2_THREADS)
        atomicAdd(&h[bin[e]], 1u);
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += C2_THREADS) {
        unsigned long long s = 0;
        for (int w = 0; w < C2_WARPS; ++w) s += s_h[w][b];
        if (s) atomicAdd(hist + b, s);
    }
}

__global__ void k_halve(unsigned long long *__restrict__ hist, int nb)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < nb) hist[b] >>= 1;
}

extern "C" gs_status gs_count_2pcf(gs_graph_t g, uint64_t *hist_dev, void *cuda_stream)
{
    gs_clear_error();
    if (!g || !hist_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    GS_TRY_CUDA(cudaMemsetAsync(hist_dev, 0, sizeof(uint64_t) * g->nb, st));
    if (g->n_edges == 0) return GS_OK;
    // a per-warp u32 counter receives at most (edges per warp) adds: bound the
    // grid so that no warp sees 2^32 edges
    const int64_t min_blocks = g->n_edges / ((int64_t)C2_WARPS << 31) + 1;
    const int grid = (int)std::max<int64_t>(std::min<int64_t>((g->n_edges + 4095) / 4096,
                                                              (int64_t)gs_sm_count() * 8), min_blocks);
    k_count2<<<grid, C2_THREADS, 0, st>>>(g->bin, g->n_edges, g->nb, (unsigned long long *)hist_dev);
    gs_note_launch();
    k_halve<<<(g->nb + 255) / 256, 256, 0, st>>>((unsigned long long *)hist_dev, g->nb);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}
