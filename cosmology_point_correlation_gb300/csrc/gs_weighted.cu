// gs_weighted.cu -- point weights and the weighted 2pCF (GRAMSCI v2 §II.1 and
// §III.3: counts accumulated with signed, normalised data-minus-random
// weights, so that the pair sum is the Landy-Szalay numerator DD - 2DR + RR
// and xi = (signed pair sum) / RR).
//
// Weights are int16 fixed-point values (a caller scales real weights by 2^F).
// A pair contributes w_i w_j (|.| <= 2^30); sums are kept exactly as 128-bit
// integers (gs_add128). Integer addition is associative, so the result does
// not depend on the order in which threads add. The weighted 3pCF is a mode
// of the triangle kernel (gs_count3.cu).

#include <algorithm>

#include "gs_internal.cuh"

__global__ void k_gather_weights(const int4 *__restrict__ pts, const int16_t *__restrict__ w_in, int64_t n,
                                 int16_t *__restrict__ w)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x)
        w[p] = w_in[pts[p].w];
}

extern "C" gs_status gs_graph_set_weights(gs_graph_t g, const int16_t *w_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || (g->n > 0 && !w_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (!g->w) GS_TRY_CUDA(gs_malloc(&g->w, sizeof(int16_t) * (size_t)std::max<int64_t>(g->n, 1)));
    if (g->n == 0) return GS_OK;
    const int grid = (int)std::min<int64_t>((g->n + 255) / 256, (int64_t)gs_sm_count() * 16);
    k_gather_weights<<<grid, 256, 0, st>>>(g->pts, w_dev, g->n, g->w);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

// ---------------------------------------------------------------- weighted 2pCF

constexpr int W2_THREADS = 256;
constexpr int W2_WARPS = W2_THREADS / 32;
constexpr int W2_LANE_BINS = 32;     // lane-private sums up to this many bins

// A warp per hub i: w_i w_j over the forward entries j > i of row i.
// Lane-private int64 sums s[warp][bin][lane] (plain adds, no conflicts: the
// bank depends on the lane only). A lane adds at most E/64 + (its warp's hubs)
// terms of |.| <= 2^30; with E < 2^36 (the host's condition) that is below
// 2^32 terms, so the int64 sums are exact. At the end the block adds its
// 32 x warps values per bin into 128 bits, then into the global sums.
__global__ void __launch_bounds__(W2_THREADS)
k_count2w_lanes(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd, const int32_t *__restrict__ nbr,
                const uint8_t *__restrict__ bin, int64_t off, const int16_t *__restrict__ w, int64_t i0, int64_t i1,
                int nb, unsigned long long *__restrict__ out)
{
    extern __shared__ long long s_lane[];             // [W2_WARPS][nb][32]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = threadIdx.x; t < W2_WARPS * nb * 32; t += W2_THREADS) s_lane[t] = 0;
    __syncthreads();
    long long *mine = s_lane + (size_t)warp * nb * 32 + lane;
    const int64_t w0 = ((int64_t)blockIdx.x * W2_THREADS + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * W2_THREADS) >> 5;
    for (int64_t i = i0 + w0; i < i1; i += nw) {
        const long long wi = w[i];
        const int64_t p1 = row_ptr[i + 1];
        for (int64_t p = row_ptr[i] + fwd[i] + lane; p < p1; p += 32) mine[32 * bin[p - off]] += wi * w[nbr[p - off]];
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += W2_THREADS) {
        unsigned long long lo = 0, hi = 0;
        for (int q = 0; q < W2_WARPS; ++q)
            for (int l = 0; l < 32; ++l) {
                const long long v = s_lane[((size_t)q * nb + b) * 32 + l];
                const unsigned long long u = (unsigned long long)v;
                lo += u;
                hi += (lo < u ? 1ull : 0ull) + (v < 0 ? ~0ull : 0ull);
            }
        if (lo | hi) gs_add128w(out + 2 * b, lo, hi);
    }
}

// Any number of bins: 128-bit sums per block in shared memory (gs_add128).
__global__ void __launch_bounds__(W2_THREADS)
k_count2w(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd, const int32_t *__restrict__ nbr,
          const uint8_t *__restrict__ bin, int64_t off, const int16_t *__restrict__ w, int64_t i0, int64_t i1, int nb,
          unsigned long long *__restrict__ out)
{
    __shared__ unsigned long long s_acc[2 * 256];
    for (int t = threadIdx.x; t < 2 * 256; t += W2_THREADS) s_acc[t] = 0ull;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * W2_THREADS + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * W2_THREADS) >> 5;
    for (int64_t i = i0 + w0; i < i1; i += nw) {
        const long long wi = w[i];
        const int64_t p1 = row_ptr[i + 1];
        for (int64_t p = row_ptr[i] + fwd[i] + lane; p < p1; p += 32)
            gs_add128(s_acc + 2 * bin[p - off], wi * w[nbr[p - off]]);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += W2_THREADS)
        if (s_acc[2 * b] | s_acc[2 * b + 1]) gs_add128w(out + 2 * b, s_acc[2 * b], s_acc[2 * b + 1]);
}

extern "C" gs_status gs_count_2pcf_weighted(gs_graph_t g, int64_t *sums_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !sums_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (!g->w) return gs_set_error(GS_ERR_ARG, "no weights: call gs_graph_set_weights first");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    GS_TRY_CUDA(cudaMemsetAsync(sums_dev, 0, sizeof(int64_t) * 2 * g->nb, st));
    if (g->n_edges == 0) return GS_OK;
    const bool lanes = g->nb <= W2_LANE_BINS && g->n_edges < (1ll << 36);
    const size_t dyn = lanes ? sizeof(long long) * W2_WARPS * 32 * (size_t)g->nb : 0;
    if (lanes) GS_TRY_CUDA(cudaFuncSetAttribute(k_count2w_lanes, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    // hubs [i0, i1) with their rows at (nbr, bin) - off
    auto launch = [&](int64_t i0, int64_t i1, const int32_t *nbr, const uint8_t *bin, int64_t off) -> gs_status {
        const int grid = (int)std::min<int64_t>((i1 - i0 + W2_WARPS - 1) / W2_WARPS, (int64_t)gs_sm_count() * 8);
        if (grid < 1) return GS_OK;
        if (lanes)
            k_count2w_lanes<<<grid, W2_THREADS, dyn, st>>>(g->row_ptr, g->fwd, nbr, bin, off, g->w, i0, i1, g->nb,
                                                            (unsigned long long *)sums_dev);
        else
            k_count2w<<<grid, W2_THREADS, 0, st>>>(g->row_ptr, g->fwd, nbr, bin, off, g->w, i0, i1, g->nb,
                                                   (unsigned long long *)sums_dev);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
        return GS_OK;
    };
    if (g->n_win == 0) return launch(0, g->n, g->nbr, g->bin, 0);
    for (int w = 0; w < g->n_win; ++w) {              // one staged window of hub rows at a time
        if (g->win_e0[w + 1] == g->win_e0[w]) continue;
        int64_t off = 0;
        gs_status s = gs_stage_window(g, w, 0, st, &off);
        if (s == GS_OK) s = launch(g->win_row[w], g->win_row[w + 1], g->s_nbr[0], g->s_bin[0], off);
        if (s != GS_OK) return s;
    }
    return GS_OK;
}
