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
    // bytes up to the first 16-byte boundary, then whole 16-byte vectors, then the tail
    const int64_t mis = (int64_t)((16 - ((uintptr_t)bin & 15)) & 15);
    const int64_t head = mis < n_edges ? mis : n_edges;
    for (int64_t e = (int64_t)blockIdx.x * C2_THREADS + threadIdx.x; e < head; e += (int64_t)gridDim.x * C2_THREADS)
        atomicAdd(&h[bin[e]], 1u);
    bin += head;
    n_edges -= head;
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

// Add the bin bytes [bin, bin + n) into hist.
static gs_status count2_bytes(const uint8_t *bin, int64_t n, int nb, unsigned long long *hist, cudaStream_t st)
{
    if (n == 0) return GS_OK;
    // a per-warp u32 counter receives at most (edges per warp) adds: bound the
    // grid so that no warp sees 2^32 edges
    const int64_t min_blocks = n / ((int64_t)C2_WARPS << 31) + 1;
    const int grid = (int)std::max<int64_t>(std::min<int64_t>((n + 4095) / 4096, (int64_t)gs_sm_count() * 8),
                                            min_blocks);
    k_count2<<<grid, C2_THREADS, 0, st>>>(bin, n, nb, hist);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

extern "C" gs_status gs_count_2pcf(gs_graph_t g, uint64_t *hist_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !hist_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    GS_TRY_CUDA(cudaMemsetAsync(hist_dev, 0, sizeof(uint64_t) * g->nb, st));
    if (g->n_edges == 0) return GS_OK;
    unsigned long long *hist = (unsigned long long *)hist_dev;
    if (g->n_win == 0) {
        gs_status s = count2_bytes(g->bin, g->n_edges, g->nb, hist, st);
        if (s != GS_OK) return s;
    } else {
        for (int w = 0; w < g->n_win; ++w) {             // one staged window at a time
            const int64_t e0 = g->win_e0[w], e1 = g->win_e0[w + 1];
            if (e1 == e0) continue;
            int64_t off = 0;
            gs_status s = gs_stage_window(g, w, 0, st, &off);
            if (s == GS_OK) s = count2_bytes(g->s_bin[0] + (e0 - off), e1 - e0, g->nb, hist, st);
            if (s != GS_OK) return s;
        }
    }
    k_halve<<<(g->nb + 255) / 256, 256, 0, st>>>(hist, g->nb);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}
