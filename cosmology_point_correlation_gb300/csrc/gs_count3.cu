// gs_count3.cu -- 3pCF triangle histogram (GRAMSCI v2, §II.2 and §III.1).
//
// Every unordered triangle {i, j, k} with i < j < k (internal numbering) is
// found once, at hub i: j is a forward spoke of i (j in N(i), j > i) and k
// lies both in the hub tail {k in N(i) : k > j} and in N(j). The paper finds
// that intersection with a two-pointer merge-walk over the two sorted lists
// (§III.1). On the GPU the same set intersection is done hub-first:
//
//   * one thread block owns one hub at a time (the paper's "one gang per hub"
//     rule, §III.5.2); it loads the hub's forward row into a shared-memory
//     hash table (node id -> bin b_ik);
//   * each warp takes a spoke j and streams the forward part of N(j) with
//     coalesced loads, 32 entries per step; every lane probes the table for
//     its entry k, and a hit is a closed triangle with bins (b_ij, b_ik, b_jk);
//   * the walk over N(j) stops at the largest hub key, because both lists are
//     sorted (Eq.(1));
//   * hits go to a per-block uint32 shared-memory histogram, flushed into the
//     caller's uint64 histogram with one global atomic per non-zero bin
//     before any counter could overflow and when the block exits.
//
// Rows longer than the table are processed in chunks of the hub row: chunk
// [c0, c1) holds the k candidates, every spoke at position s < c1 - 1 is
// walked over keys in (max(j, F[c0] - 1), F[c1 - 1]].
//
// Hubs are handed out in increasing internal order from a global counter, so
// the blocks resident at any moment work on neighbouring hubs whose spoke
// rows overlap and stay in L2.

#include <algorithm>

#include "gs_internal.cuh"

constexpr int C3_THREADS = 256;
constexpr int C3_WARPS = C3_THREADS / 32;
constexpr int C3_TABLE_LOG = 12;                 // 4096 slots
constexpr int C3_TABLE = 1 << C3_TABLE_LOG;
constexpr int C3_CHUNK = C3_TABLE / 2;           // load factor <= 1/2
constexpr int C3_SMEM_HIST_MAX = 12288;          // configurations kept in shared memory
constexpr int C3_EMPTY = -1;

struct C3Args {
    const int64_t *row_ptr;
    const int32_t *fwd;
    const int32_t *nbr;
    const uint8_t *bin;
    int64_t hub_begin, hub_end;
    int nb;
    int ncfg;
    unsigned long long *ghist;
    unsigned long long *cursor;   // next hub to hand out
};

// Flush the shared histogram into the global one and clear it.
__device__ __forceinline__ void c3_flush(unsigned *sh, int ncfg, unsigned long long *gh)
{
    for (int t = threadIdx.x; t < ncfg; t += C3_THREADS) {
        const unsigned v = sh[t];
        if (v) {
            atomicAdd(gh + t, (unsigned long long)v);
            sh[t] = 0;
        }
    }
}

template <bool SMEM_HIST>
__global__ void __launch_bounds__(C3_THREADS)
k_count3(C3Args a)
{
    extern __shared__ unsigned s_hist[];            // [ncfg] when SMEM_HIST
    __shared__ int32_t s_key[C3_TABLE];
    __shared__ uint8_t s_bin[C3_TABLE];
    __shared__ int s_lex_a[256];                    // idx3 = s_lex_a[lo] + s_lex_b[mid] + hi
    __shared__ int s_lex_b[256];
    __shared__ long long s_hub;
    __shared__ unsigned long long s_pending;        // hits bound since the last flush

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = a.nb;
    // gs_idx3(a, b, c) = F(a) - G(a) + G(b) - b + c with F(a) = gs_idx3(a, a, a) and
    // G(t) = t nb - t (t - 1) / 2, split into two per-bin tables.
    for (int t = threadIdx.x; t < nb; t += C3_THREADS) {
        const int64_t Gt = (int64_t)t * nb - (int64_t)t * (t - 1) / 2;
        s_lex_a[t] = (int)(gs_idx3(nb, t, t, t) - Gt);
        s_lex_b[t] = (int)(Gt - t);
    }
    if (SMEM_HIST)
        for (int t = threadIdx.x; t < a.ncfg; t += C3_THREADS) s_hist[t] = 0;
    for (int t = threadIdx.x; t < C3_TABLE; t += C3_THREADS) s_key[t] = C3_EMPTY;
    if (threadIdx.x == 0) s_pending = 0;
    __syncthreads();

    for (;;) {
        __syncthreads();                                     // everyone has read the last s_hub
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        const long long i = s_hub;
        if (i >= a.hub_end) break;

        const int64_t f0 = a.row_ptr[i] + a.fwd[i];          // forward row F = nbr[f0, f1)
        const int f = (int)(a.row_ptr[i + 1] - f0);
        for (int c0 = 0; c0 < f; c0 += C3_CHUNK) {           // chunks of candidate keys
            const int c1 = min(f, c0 + C3_CHUNK);
            const int cn = c1 - c0;
            int lg = 6;                                      // table of 2^lg >= 2 cn slots
            while ((1 << lg) < 2 * cn) ++lg;
            const int tsize = 1 << lg, shift = 32 - lg, mask = tsize - 1;

            if (SMEM_HIST) {
                // bound on the hits of this chunk: every spoke before c1 can close
                // at most cn triangles
                const unsigned long long bound = (unsigned long long)c1 * cn;
                if (s_pending + bound > 0xffffffffull) {     // block-uniform
                    __syncthreads();
                    c3_flush(s_hist, a.ncfg, a.ghist);
                    __syncthreads();
                    if (threadIdx.x == 0) s_pending = 0;
                }
                __syncthreads();
                if (threadIdx.x == 0) s_pending += bound;
            }
            for (int t = threadIdx.x; t < cn; t += C3_THREADS) {
                const int32_t k = a.nbr[f0 + c0 + t];
                uint32_t h = gs_hash(k, shift);
                while (atomicCAS(&s_key[h], C3_EMPTY, k) != C3_EMPTY) h = (h + 1) & mask;
                s_bin[h] = a.bin[f0 + c0 + t];
            }
            __syncthreads();

            const int32_t kmax = a.nbr[f0 + c1 - 1];
            const int32_t kfirst = a.nbr[f0 + c0];
            for (int s = warp; s < c1 - 1; s += C3_WARPS) {
                const int32_t j = a.nbr[f0 + s];
                const int bij = a.bin[f0 + s];
                const int64_t rj1 = a.row_ptr[j + 1];
                int64_t p;
                if (s + 1 >= c0) {
                    p = a.row_ptr[j] + a.fwd[j];                   // first entry > j
                } else {
                    // first entry >= kfirst in N(j) (lower bound; only for later chunks)
                    int64_t lo = a.row_ptr[j] + a.fwd[j], hi = rj1;
                    while (lo < hi) {
                        const int64_t mid = (lo + hi) >> 1;
                        if (a.nbr[mid] < kfirst) lo = mid + 1; else hi = mid;
                    }
                    p = lo;
                }
                for (; p < rj1; p += 32) {
                    const int64_t q = p + lane;
                    int32_t k = 0x7fffffff;
                    int bjk = 0;
                    if (q < rj1) {
                        k = a.nbr[q];
                        bjk = a.bin[q];
                    }
                    if (k <= kmax) {
                        uint32_t h = gs_hash(k, shift);
                        int32_t key;
                        while ((key = s_key[h]) != k && key != C3_EMPTY) h = (h + 1) & mask;
                        if (key == k) {
                            const int bik = s_bin[h];
                            const int lo = min(bij, min(bik, bjk));
                            const int hi = max(bij, max(bik, bjk));
                            const int mid = bij + bik + bjk - lo - hi;
                            const int idx = s_lex_a[lo] + s_lex_b[mid] + hi;
                            if (SMEM_HIST) atomicAdd(&s_hist[idx], 1u);
                            else atomicAdd(a.ghist + idx, 1ull);
                        }
                    }
                    // the row is sorted: stop once the last lane's key passes kmax
                    if (__shfl_sync(0xffffffffu, k, 31) > kmax) break;
                }
            }
            __syncthreads();
            for (int t = threadIdx.x; t < tsize; t += C3_THREADS) s_key[t] = C3_EMPTY;
            __syncthreads();
        }
    }
    if (SMEM_HIST) {
        __syncthreads();
        c3_flush(s_hist, a.ncfg, a.ghist);
    }
}

extern "C" gs_status gs_count_3pcf(gs_graph_t g, uint64_t *hist_dev, int64_t hub_begin, int64_t hub_end,
                                   void *cuda_stream)
{
    gs_clear_error();
    if (!g || !hist_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int ncfg = (int)gs_ncfg3(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(hist_dev, 0, sizeof(uint64_t) * ncfg, st));
    if (hub_end == hub_begin || g->n_edges == 0) return GS_OK;
    GS_TRY_CUDA(cudaMemsetAsync(g->work, 0, sizeof(unsigned long long), st));

    C3Args a;
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.hub_begin = hub_begin;
    a.hub_end = hub_end;
    a.nb = g->nb;
    a.ncfg = ncfg;
    a.ghist = (unsigned long long *)hist_dev;
    a.cursor = g->work;

    // shared-memory histogram unless it is too large or a chunk's hit bound
    // (spokes x chunk) could overflow a 32-bit counter
    const bool smem = ncfg <= C3_SMEM_HIST_MAX && (int64_t)g->max_degree * C3_CHUNK < (1ll << 31);
    const size_t dyn = smem ? sizeof(unsigned) * ncfg : 0;
    int per_sm = 0;
    if (smem) {
        GS_TRY_CUDA(cudaFuncSetAttribute(k_count3<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
        GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_count3<true>, C3_THREADS, dyn));
    } else {
        GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_count3<false>, C3_THREADS, 0));
    }
    per_sm = std::max(per_sm, 1);
    const int64_t hubs = hub_end - hub_begin;
    const int grid = (int)std::min<int64_t>((int64_t)gs_sm_count() * per_sm, hubs);
    if (smem) k_count3<true><<<grid, C3_THREADS, dyn, st>>>(a);
    else k_count3<false><<<grid, C3_THREADS, 0, st>>>(a);
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}
