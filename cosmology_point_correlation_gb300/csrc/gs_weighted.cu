// gs_weighted.cu -- weighted 2pCF and 3pCF with signed integer weights, exact
// (GRAMSCI v2 §II.1 and §III.3: counts accumulated with signed, normalised
// data-minus-random weights, so that the pair sum is the Landy-Szalay
// numerator DD - 2DR + RR and xi = (signed pair sum) / RR).
//
// Weights are int16 fixed-point values (a caller scales real weights by 2^F).
// A pair contributes w_i w_j (|.| <= 2^30), a triangle w_i w_j w_k
// (|.| <= 2^45); sums are kept exactly in 128-bit integers: a low word added
// with a 64-bit atomic, its carry and the sign extension added to the high
// word. Integer addition is associative, so the result does not depend on
// the order in which threads add.
//
// Weighted 3pCF: the hub's forward row goes into a shared hash table holding
// each key's bin and weight. For one spoke j (bin b_ij fixed) a warp sums the
// weights w_k of its hits per (b_ik, b_jk) in a per-warp nb x nb int32 array
// (at most 2048 hits of |w| <= 2^15 per spoke and chunk: no overflow); at the
// end of the spoke every non-zero entry S is added as w_i w_j S to the block's
// 128-bit accumulator of its configuration.

#include <algorithm>

#include "gs_internal.cuh"

constexpr int W3_THREADS = 512;
constexpr int W3_WARPS = W3_THREADS / 32;
constexpr int W3_TABLE_LOG = 13;
constexpr int W3_TABLE = 1 << W3_TABLE_LOG;
constexpr int W3_CHUNK = W3_TABLE / 4;
constexpr int W3_EMPTY = -1;
constexpr int W3_MAX_BINS = 40;              // per-warp nb x nb sums in shared memory
constexpr int W3_SMEM_ACC_MAX = 5120;        // configurations with shared 128-bit accumulators

// v added to the 128-bit integer (lo, hi) at p (global or shared memory).
__device__ __forceinline__ void add128(unsigned long long *p, long long v)
{
    const unsigned long long u = (unsigned long long)v;
    const unsigned long long old = atomicAdd(p, u);
    const unsigned long long hi = (old + u < old ? 1ull : 0ull) + (v < 0 ? ~0ull : 0ull);
    if (hi) atomicAdd(p + 1, hi);
}

// Add a 128-bit value (lo, hi) to the 128-bit integer at p.
__device__ __forceinline__ void add128w(unsigned long long *p, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long old = atomicAdd(p, lo);
    const unsigned long long h = hi + (old + lo < old ? 1ull : 0ull);
    if (h) atomicAdd(p + 1, h);
}

__global__ void k_gather_weights(const int4 *__restrict__ pts, const int16_t *__restrict__ w_in, int64_t n,
                                 int16_t *__restrict__ w)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x)
        w[p] = w_in[pts[p].w];
}

extern "C" gs_status gs_graph_set_weights(gs_graph_t g, const int16_t *w_dev, void *cuda_stream)
{
    gs_clear_error();
    if (!g || (g->n > 0 && !w_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (!g->w) GS_TRY_CUDA(cudaMalloc(&g->w, sizeof(int16_t) * (size_t)std::max<int64_t>(g->n, 1)));
    if (g->n == 0) return GS_OK;
    const int grid = (int)std::min<int64_t>((g->n + 255) / 256, (int64_t)gs_sm_count() * 16);
    k_gather_weights<<<grid, 256, 0, st>>>(g->pts, w_dev, g->n, g->w);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

// ---------------------------------------------------------------- weighted 2pCF

// A warp per hub i: w_i w_j over the forward entries j > i of row i, into the
// block's 128-bit sums (shared), then into the global sums.
__global__ void __launch_bounds__(256)
k_count2w(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd, const int32_t *__restrict__ nbr,
          const uint8_t *__restrict__ bin, const int16_t *__restrict__ w, int64_t n, int nb,
          unsigned long long *__restrict__ out)
{
    __shared__ unsigned long long s_acc[2 * 256];
    for (int t = threadIdx.x; t < 2 * 256; t += blockDim.x) s_acc[t] = 0ull;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = w0; i < n; i += nw) {
        const long long wi = w[i];
        const int64_t p1 = row_ptr[i + 1];
        for (int64_t p = row_ptr[i] + fwd[i] + lane; p < p1; p += 32)
            add128(s_acc + 2 * bin[p], wi * w[nbr[p]]);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += blockDim.x)
        if (s_acc[2 * b] | s_acc[2 * b + 1]) add128w(out + 2 * b, s_acc[2 * b], s_acc[2 * b + 1]);
}

extern "C" gs_status gs_count_2pcf_weighted(gs_graph_t g, int64_t *sums_dev, void *cuda_stream)
{
    gs_clear_error();
    if (!g || !sums_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    if (!g->w) return gs_set_error(GS_ERR_ARG, "no weights: call gs_graph_set_weights first");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    GS_TRY_CUDA(cudaMemsetAsync(sums_dev, 0, sizeof(int64_t) * 2 * g->nb, st));
    if (g->n_edges == 0) return GS_OK;
    const int grid = (int)std::min<int64_t>((g->n + 7) / 8, (int64_t)gs_sm_count() * 8);
    k_count2w<<<grid, 256, 0, st>>>(g->row_ptr, g->fwd, g->nbr, g->bin, g->w, g->n, g->nb,
                                    (unsigned long long *)sums_dev);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

// ---------------------------------------------------------------- weighted 3pCF

struct W3Args {
    const int64_t *row_ptr;
    const int32_t *fwd;
    const int32_t *nbr;
    const uint8_t *bin;
    const int16_t *w;
    const uint16_t *cfg3;         // [nb][nb][nb] configuration of (z, x, y)
    int64_t hub_begin, hub_end;
    int nb, ncfg;
    unsigned long long *out;      // [ncfg][2] 128-bit sums
    unsigned long long *cursor;
};

template <bool SMEM_ACC>
__global__ void __launch_bounds__(W3_THREADS)
k_count3w(W3Args a)
{
    // dynamic: keys [W3_TABLE] i32, bins [W3_TABLE] u8, weights [W3_TABLE] i16,
    // per-warp sums [W3_WARPS][nb*nb] i32, then (SMEM_ACC) [ncfg][2] u64
    extern __shared__ unsigned long long s_dyn64[];
    __shared__ long long s_hub;
    __shared__ int s_next;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = a.nb, nb2 = nb * nb;
    int32_t *s_key = (int32_t *)s_dyn64;
    uint8_t *s_bin = (uint8_t *)(s_key + W3_TABLE);
    int16_t *s_w = (int16_t *)(s_bin + W3_TABLE);
    int *s_sum = (int *)(s_w + W3_TABLE) + warp * nb2;
    unsigned long long *s_acc = (unsigned long long *)((int *)(s_w + W3_TABLE) + ((W3_WARPS * nb2 + 1) & ~1));
    unsigned long long *acc = SMEM_ACC ? s_acc : a.out;

    for (int t = lane; t < nb2; t += 32) s_sum[t] = 0;
    if (SMEM_ACC)
        for (int t = threadIdx.x; t < 2 * a.ncfg; t += W3_THREADS) s_acc[t] = 0ull;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        const long long i = s_hub;
        if (i >= a.hub_end) break;
        const long long wi = a.w[i];
        const int64_t f0 = a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        for (int c0 = 0; c0 < f; c0 += W3_CHUNK) {
            const int c1 = min(f, c0 + W3_CHUNK), cn = c1 - c0;
            if (c1 < 2) break;
            int lg = 6;
            while ((1 << lg) < 4 * cn) ++lg;
            const int tsize = 1 << lg, shift = 32 - lg, mask = tsize - 1;
            for (int t = threadIdx.x; t < tsize; t += W3_THREADS) s_key[t] = W3_EMPTY;
            __syncthreads();
            for (int t = threadIdx.x; t < cn; t += W3_THREADS) {
                const int32_t k = a.nbr[f0 + c0 + t];
                uint32_t h = gs_hash(k, shift);
                while (atomicCAS(&s_key[h], W3_EMPTY, k) != W3_EMPTY) h = (h + 1) & mask;
                s_bin[h] = a.bin[f0 + c0 + t];
                s_w[h] = a.w[k];
            }
            if (threadIdx.x == 0) s_next = 0;
            __syncthreads();
            const int32_t kmax = a.nbr[f0 + c1 - 1];
            const int32_t kfirst = a.nbr[f0 + c0];
            for (;;) {
                int s = 0;
                if (lane == 0) s = atomicAdd(&s_next, 1);
                s = __shfl_sync(0xffffffffu, s, 0);
                if (s >= c1 - 1) break;
                const int32_t j = a.nbr[f0 + s];
                const int bij = a.bin[f0 + s];
                const long long wij = wi * a.w[j];
                const int64_t pe = a.row_ptr[j + 1];
                int64_t p0 = a.row_ptr[j] + a.fwd[j];
                if (s + 1 < c0) {                                  // later chunk: start at kfirst
                    int64_t lo = p0, hi = pe;
                    while (lo < hi) {
                        const int64_t mid = (lo + hi) >> 1;
                        if (a.nbr[mid] < kfirst) lo = mid + 1; else hi = mid;
                    }
                    p0 = lo;
                }
                for (int64_t p = p0; p < pe; p += 32) {
                    const int64_t q = p + lane;
                    const int32_t k = q < pe ? a.nbr[q] : 0x7fffffff;
                    if (k <= kmax) {
                        uint32_t h = gs_hash(k, shift);
                        int32_t key;
                        while ((key = s_key[h]) != k && key != W3_EMPTY) h = (h + 1) & mask;
                        if (key == k) atomicAdd(&s_sum[s_bin[h] * nb + a.bin[q]], (int)s_w[h]);
                    }
                    if (__shfl_sync(0xffffffffu, k, 31) > kmax) break;
                }
                __syncwarp();
                // w_i w_j S into the 128-bit sum of configuration (b_ij, b_ik, b_jk)
                const uint16_t *cz = a.cfg3 + (size_t)bij * nb2;
                for (int t = lane; t < nb2; t += 32) {
                    const int v = s_sum[t];
                    if (v) {
                        s_sum[t] = 0;
                        add128(acc + 2 * (size_t)__ldg(cz + t), wij * v);
                    }
                }
                __syncwarp();
            }
            __syncthreads();
        }
    }
    if (SMEM_ACC) {
        __syncthreads();
        for (int t = threadIdx.x; t < a.ncfg; t += W3_THREADS)
            if (s_acc[2 * t] | s_acc[2 * t + 1]) add128w(a.out + 2 * t, s_acc[2 * t], s_acc[2 * t + 1]);
    }
}

extern "C" gs_status gs_count_3pcf_weighted(gs_graph_t g, int64_t *sums_dev, int64_t hub_begin, int64_t hub_end,
                                            void *cuda_stream)
{
    gs_clear_error();
    if (!g || !sums_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    if (!g->w) return gs_set_error(GS_ERR_ARG, "no weights: call gs_graph_set_weights first");
    if (g->nb > W3_MAX_BINS || !g->cfg3)
        return gs_set_error(GS_ERR_ARG, "the weighted 3pCF supports at most %d bins", W3_MAX_BINS);
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int ncfg = (int)gs_ncfg3(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(sums_dev, 0, sizeof(int64_t) * 2 * ncfg, st));
    if (hub_end == hub_begin || g->n_edges == 0) return GS_OK;
    GS_TRY_CUDA(cudaMemsetAsync(g->work, 0, sizeof(unsigned long long), st));
    W3Args a{};
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.w = g->w;
    a.cfg3 = g->cfg3;
    a.hub_begin = hub_begin;
    a.hub_end = hub_end;
    a.nb = g->nb;
    a.ncfg = ncfg;
    a.out = (unsigned long long *)sums_dev;
    a.cursor = g->work;
    const int nb2 = g->nb * g->nb;
    const bool smem = ncfg <= W3_SMEM_ACC_MAX;
    const size_t dyn = (size_t)W3_TABLE * (4 + 1 + 2) + sizeof(int) * (size_t)((W3_WARPS * nb2 + 1) & ~1) +
                       (smem ? sizeof(unsigned long long) * 2 * ncfg : 0);
    auto kern = smem ? k_count3w<true> : k_count3w<false>;
    int per_sm = 0;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, W3_THREADS, dyn));
    if (per_sm < 1) return gs_set_error(GS_ERR_CAPACITY, "weighted 3pCF workspace does not fit in shared memory");
    const int grid = (int)std::min<int64_t>((int64_t)gs_sm_count() * per_sm, hub_end - hub_begin);
    kern<<<grid, W3_THREADS, dyn, st>>>(a);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}
