// gs_build.cu -- fixed-radius neighbour graph on the GPU (GRAMSCI v2, §II.1 and
// §III.5.1): cell list, counting sort by cell, two-pass (count, fill) neighbour
// search writing index-sorted CSR rows with a radial-bin byte per edge.
//
// The paper builds the graph on the CPU with a kd-tree; here a uniform cell
// grid with cell side >= r_max makes the search a scan of <= 27 neighbour
// cells, which the GPU does with coalesced, shared-memory-staged candidate
// tiles. Rows come out sorted (Eq.(1)) with no sort pass: points are numbered
// in cell order and the neighbour cells of a point are visited in increasing
// cell id, so the candidates are met in increasing index order.

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gs_internal.cuh"

// ---------------------------------------------------------------- errors

static thread_local char g_msg[512] = "";

gs_status gs_set_error(gs_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

extern "C" const char *gs_last_error(void) { return g_msg; }

static thread_local int t_depth = 0;                 // public calls in progress on this thread
static thread_local int64_t t_alloc_ordinal = 0;     // allocations since the outermost one began
static std::atomic<uint64_t> g_allocs{ 0 };

gs_call_scope::gs_call_scope(const char *name)
{
    nvtxRangePushA(name);
    if (t_depth++ == 0) {
        g_msg[0] = 0;
        t_alloc_ordinal = 0;
    }
}

gs_call_scope::~gs_call_scope()
{
    --t_depth;
    nvtxRangePop();
}

cudaError_t gs_alloc_gate()
{
    g_allocs.fetch_add(1, std::memory_order_relaxed);
    const int64_t k = ++t_alloc_ordinal;
    const char *env = getenv("GS_FAULT");
    if (env && !strncmp(env, "alloc:", 6) && atoll(env + 6) == k) return cudaErrorMemoryAllocation;
    return cudaSuccess;
}

extern "C" uint64_t gs_alloc_calls(void) { return g_allocs.load(); }

gs_status gs_checked_begin(gs_graph_t g, cudaStream_t st)
{
#ifdef GS_CHECKED
    GS_TRY_CUDA(cudaMemsetAsync(g->chk, 0, sizeof(unsigned), st));
#else
    (void)g;
    (void)st;
#endif
    return GS_OK;
}

gs_status gs_checked_end(gs_graph_t g, cudaStream_t st, const char *what)
{
#ifdef GS_CHECKED
    unsigned h = 0;
    GS_TRY_CUDA(cudaMemcpyAsync(&h, g->chk, sizeof(unsigned), cudaMemcpyDeviceToHost, st));
    GS_TRY_CUDA(cudaStreamSynchronize(st));
    if (h) return gs_set_error(GS_ERR_INTERNAL, "%s: device bounds checks failed at sites 0x%x", what, h);
#else
    (void)g;
    (void)st;
    (void)what;
#endif
    return GS_OK;
}

static std::atomic<uint64_t> g_launches{ 0 };

void gs_note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

extern "C" uint64_t gs_kernel_launches(void) { return g_launches.load(); }

int gs_sm_count()
{
    static int cache[64] = { 0 };
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (!cache[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 1;
    }
    return cache[dev];
}

// ---------------------------------------------------------------- exclusive scan
//
// Three phases over tiles of SCAN_TILE elements: per-tile scan writing tile
// totals, a one-block scan of the totals, then a uniform add.

constexpr int SCAN_THREADS = 256;
constexpr int SCAN_ITEMS = 8;
constexpr int SCAN_TILE = SCAN_THREADS * SCAN_ITEMS;

template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T *total)
{
    __shared__ T warp_sums[SCAN_THREADS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T w = lane < SCAN_THREADS / 32 ? warp_sums[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < SCAN_THREADS / 32) warp_sums[lane] = w;
    }
    __syncthreads();
    T prefix = (warp > 0 ? warp_sums[warp - 1] : T(0)) + x - v;
    *total = warp_sums[SCAN_THREADS / 32 - 1];
    __syncthreads();
    return prefix;
}

template <typename Tout>
__global__ void __launch_bounds__(SCAN_THREADS)
k_scan_tiles(const int32_t *__restrict__ in, Tout *__restrict__ out, Tout *__restrict__ tile_sums,
             int64_t n)
{
    const int64_t base = (int64_t)blockIdx.x * SCAN_TILE + (int64_t)threadIdx.x * SCAN_ITEMS;
    Tout v[SCAN_ITEMS];
    Tout s = 0;
#pragma unroll
    for (int k = 0; k < SCAN_ITEMS; ++k) {
        v[k] = (base + k < n) ? (Tout)in[base + k] : Tout(0);
        s += v[k];
    }
    Tout total;
    Tout run = block_exclusive_scan<Tout>(s, &total);
#pragma unroll
    for (int k = 0; k < SCAN_ITEMS; ++k) {
        if (base + k < n) out[base + k] = run;
        run += v[k];
    }
    if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

template <typename Tout>
__global__ void __launch_bounds__(SCAN_THREADS)
k_scan_sums(Tout *__restrict__ sums, int64_t ntiles, Tout *__restrict__ grand_total)
{
    Tout carry = 0;
    for (int64_t b = 0; b < ntiles; b += SCAN_TILE) {
        const int64_t base = b + (int64_t)threadIdx.x * SCAN_ITEMS;
        Tout v[SCAN_ITEMS];
        Tout s = 0;
#pragma unroll
        for (int k = 0; k < SCAN_ITEMS; ++k) {
            v[k] = (base + k < ntiles) ? sums[base + k] : Tout(0);
            s += v[k];
        }
        Tout total;
        Tout run = block_exclusive_scan<Tout>(s, &total) + carry;
#pragma unroll
        for (int k = 0; k < SCAN_ITEMS; ++k) {
            if (base + k < ntiles) sums[base + k] = run;
            run += v[k];
        }
        carry += total;
    }
    if (threadIdx.x == 0) *grand_total = carry;
}

template <typename Tout>
__global__ void __launch_bounds__(SCAN_THREADS)
k_scan_add(Tout *__restrict__ out, const Tout *__restrict__ tile_sums, int64_t n)
{
    const int64_t base = (int64_t)blockIdx.x * SCAN_TILE + (int64_t)threadIdx.x * SCAN_ITEMS;
    const Tout add = tile_sums[blockIdx.x];
#pragma unroll
    for (int k = 0; k < SCAN_ITEMS; ++k)
        if (base + k < n) out[base + k] += add;
}

template <typename Tout>
static gs_status scan_impl(const int32_t *in, Tout *out, int64_t n, cudaStream_t st)
{
    if (n == 0) {
        GS_TRY_CUDA(cudaMemsetAsync(out, 0, sizeof(Tout), st));
        return GS_OK;
    }
    const int64_t ntiles = (n + SCAN_TILE - 1) / SCAN_TILE;
    Tout *sums = nullptr;
    GS_TRY_CUDA(gs_malloc_async(&sums, sizeof(Tout) * ntiles, st));
    k_scan_tiles<Tout><<<(unsigned)ntiles, SCAN_THREADS, 0, st>>>(in, out, sums, n);
    gs_note_launch();
    k_scan_sums<Tout><<<1, SCAN_THREADS, 0, st>>>(sums, ntiles, out + n);
    gs_note_launch();
    k_scan_add<Tout><<<(unsigned)ntiles, SCAN_THREADS, 0, st>>>(out, sums, n);
    gs_note_launch();
    cudaError_t e = cudaGetLastError();
    cudaFreeAsync(sums, st);
    if (e != cudaSuccess) return gs_set_error(GS_ERR_CUDA, "scan launch failed: %s", cudaGetErrorString(e));
    return GS_OK;
}

gs_status gs_scan_i32_to_i64(const int32_t *in, int64_t *out, int64_t n, cudaStream_t st)
{
    return scan_impl<int64_t>(in, out, n, st);
}

gs_status gs_scan_i32_to_i32(const int32_t *in, int32_t *out, int64_t n, cudaStream_t st)
{
    return scan_impl<int32_t>(in, out, n, st);
}

// ---------------------------------------------------------------- cell sort

// Cell of each point and its arrival slot in that cell; flags coordinates
// outside [0, box).
__global__ void k_cell_assign(const int32_t *__restrict__ xyz, int64_t n, int box, int ncell,
                              int32_t *__restrict__ cell, int32_t *__restrict__ slot,
                              int32_t *__restrict__ cell_count, int32_t *__restrict__ err)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        int x = xyz[3 * i], y = xyz[3 * i + 1], z = xyz[3 * i + 2];
        bool ok = x >= 0 && x < box && y >= 0 && y < box && z >= 0 && z < box;
        if (!ok) {
            atomicOr(err, 1);
            x = y = z = 0;
        }
        int cx = (int)((long long)x * ncell / box);
        int cy = (int)((long long)y * ncell / box);
        int cz = (int)((long long)z * ncell / box);
        int c = (cx * ncell + cy) * ncell + cz;
        cell[i] = c;
        slot[i] = atomicAdd(&cell_count[c], 1);
    }
}

__global__ void k_cell_scatter(const int32_t *__restrict__ cell, const int32_t *__restrict__ slot,
                               const int32_t *__restrict__ cell_start, int64_t n,
                               int32_t *__restrict__ tmp)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        tmp[cell_start[cell[i]] + slot[i]] = (int32_t)i;
}

// Put each cell's points in increasing input index (the atomic slots above
// arrive in arbitrary order). One warp per cell, rank sort: each element's
// new position is the number of smaller ids in its cell.
__global__ void k_cell_order(const int32_t *__restrict__ cell_start, int ncells,
                             const int32_t *__restrict__ tmp, int32_t *__restrict__ perm)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t c = w0; c < ncells; c += nw) {
        const int s0 = cell_start[c], s1 = cell_start[c + 1];
        for (int a = s0 + lane; a < s1; a += 32) {
            const int e = tmp[a];
            int r = 0;
            for (int b = s0; b < s1; ++b) r += tmp[b] < e;
            perm[s0 + r] = e;
        }
    }
}

__global__ void k_gather_points(const int32_t *__restrict__ xyz, const int32_t *__restrict__ perm,
                                int64_t n, int4 *__restrict__ pts, int32_t *__restrict__ inv)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n;
         p += (int64_t)gridDim.x * blockDim.x) {
        const int i = perm[p];
        pts[p] = make_int4(xyz[3 * (int64_t)i], xyz[3 * (int64_t)i + 1], xyz[3 * (int64_t)i + 2], i);
        inv[i] = (int32_t)p;
    }
}

// ---------------------------------------------------------------- neighbour search
//
// NB_SPLIT blocks per home cell (blockIdx.y), each taking every NB_SPLIT-th
// batch of NB_HOME home points, so that the grid holds several waves of
// blocks and the cells of a clustered catalogue, which differ widely in size,
// leave no long tail. A block stages its home points and, range by range, up
// to NB_CAND candidate points in shared memory; each warp tests its home
// points against the staged tile, 32 candidates per step, and (FILL pass)
// writes hits in candidate order with a ballot prefix count. Neighbour cells
// are visited in increasing id, merged into contiguous index ranges (a z-run
// of three cells is one range unless it wraps). PERIODIC and LOWER (a lower
// edge e_0 > 0) are compile-time, so the common open or periodic box with
// e_0 = 0 pays for neither test it does not need.

constexpr int NB_THREADS = 256;
constexpr int NB_HOME = 256;
constexpr int NB_SPLIT = 4;
constexpr int NB_CAND = 1024;

template <bool FILL, bool PERIODIC, bool LOWER>
__global__ void __launch_bounds__(NB_THREADS)
k_neighbors(const int4 *__restrict__ pts, const int32_t *__restrict__ cell_start, int ncell,
            int box, int periodic, long long e0sq, long long rsq,
            const long long *__restrict__ esq, int nb,
            int32_t *__restrict__ deg, int32_t *__restrict__ fwd,
            const int64_t *__restrict__ row_ptr, int32_t *__restrict__ nbr,
            uint8_t *__restrict__ bin, unsigned *__restrict__ max_deg, int cell0, int64_t woff,
            unsigned *__restrict__ chk, int64_t cap)
{
    __shared__ int4 s_home[NB_HOME];
    __shared__ int s_cnt[NB_HOME];
    __shared__ int s_lo[NB_HOME];
    __shared__ int4 s_cand[NB_CAND];
    __shared__ long long s_esq[256];
    __shared__ int s_r0[27], s_r1[27];
    __shared__ int s_nr;

    // cells [cell0, cell0 + gridDim.x); FILL writes edge e at nbr[e - woff]
    const int c = cell0 + blockIdx.x;
    const int h0 = cell_start[c], h1 = cell_start[c + 1];
    if (h0 + (int)blockIdx.y * NB_HOME >= h1) return;        // no batch of this cell for this block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = NB_THREADS / 32;

    if (FILL)
        for (int t = threadIdx.x; t <= nb; t += NB_THREADS) s_esq[t] = esq[t];
    if (threadIdx.x == 0) {
        const int cx = c / (ncell * ncell), cy = (c / ncell) % ncell, cz = c % ncell;
        int ids[27];
        int m = 0;
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz) {
                    int x = cx + dx, y = cy + dy, z = cz + dz;
                    if (periodic) {
                        x = (x + ncell) % ncell;
                        y = (y + ncell) % ncell;
                        z = (z + ncell) % ncell;
                    } else if (x < 0 || x >= ncell || y < 0 || y >= ncell || z < 0 || z >= ncell) {
                        continue;
                    }
                    ids[m++] = (x * ncell + y) * ncell + z;
                }
        for (int a = 1; a < m; ++a)        // insertion sort, m <= 27
            for (int b = a; b > 0 && ids[b - 1] > ids[b]; --b) {
                int t = ids[b];
                ids[b] = ids[b - 1];
                ids[b - 1] = t;
            }
        int nr = 0, prev = -2;
        for (int a = 0; a < m; ++a) {
            if (ids[a] == prev) continue;  // duplicate cell (fewer than 3 cells per axis)
            if (ids[a] == prev + 1) {
                s_r1[nr - 1] = cell_start[ids[a] + 1];
            } else {
                s_r0[nr] = cell_start[ids[a]];
                s_r1[nr] = cell_start[ids[a] + 1];
                ++nr;
            }
            prev = ids[a];
        }
        s_nr = nr;
    }
    __syncthreads();
    const int nr = s_nr;

    for (int hb = h0 + (int)blockIdx.y * NB_HOME; hb < h1; hb += NB_SPLIT * NB_HOME) {
        const int hn = min(NB_HOME, h1 - hb);
        for (int t = threadIdx.x; t < hn; t += NB_THREADS) {
            s_home[t] = pts[hb + t];
            s_cnt[t] = 0;
            s_lo[t] = 0;
        }
        __syncthreads();
        for (int r = 0; r < nr; ++r) {
            for (int cb = s_r0[r]; cb < s_r1[r]; cb += NB_CAND) {
                const int cn = min(NB_CAND, s_r1[r] - cb);
                for (int t = threadIdx.x; t < cn; t += NB_THREADS) s_cand[t] = pts[cb + t];
                __syncthreads();
                for (int hp = warp; hp < hn; hp += nwarps) {
                    const int p = hb + hp;
                    const int4 P = s_home[hp];
                    int cnt = s_cnt[hp];
                    int lo = s_lo[hp];
                    const int64_t rowp = FILL ? row_ptr[p] : 0;
                    for (int t0 = 0; t0 < cn; t0 += 32) {
                        const int t = t0 + lane;
                        bool hit = false;
                        long long d2 = 0;
                        if (t < cn) {
                            const int4 Q = s_cand[t];
                            const int dx = gs_delta(P.x, Q.x, box, PERIODIC);
                            const int dy = gs_delta(P.y, Q.y, box, PERIODIC);
                            const int dz = gs_delta(P.z, Q.z, box, PERIODIC);
                            d2 = gs_norm2(dx, dy, dz);
                            hit = (cb + t != p) && (!LOWER || d2 >= e0sq) && d2 < rsq;
                        }
                        const unsigned m = __ballot_sync(0xffffffffu, hit);
                        if (FILL && hit) {
                            const int64_t pos = rowp + cnt + __popc(m & gs_lanemask_lt()) - woff;
                            int lo_b = 0, hi_b = nb;       // e_lo^2 <= d2 < e_hi^2
                            while (hi_b - lo_b > 1) {
                                const int mid = (lo_b + hi_b) >> 1;
                                if (s_esq[mid] <= d2) lo_b = mid; else hi_b = mid;
                            }
                            // checked builds: the edge lies in its own row and in the array
                            if (GS_DCHECK(pos >= 0 && pos < cap && pos + woff < row_ptr[p + 1], chk, GS_SITE_NB_ROW)) {
                                nbr[pos] = cb + t;
                                bin[pos] = (uint8_t)lo_b;
                            }
                        }
                        cnt += __popc(m);
                        if (!FILL) {
                            // neighbours below p: the step lies below p, above it, or
                            // straddles it (lanes below p - cb - t0 < 32)
                            if (cb + t0 + 31 < p) lo += __popc(m);
                            else if (cb + t0 < p) lo += __popc(m & ((1u << (p - cb - t0)) - 1u));
                        }
                    }
                    if (lane == 0) {
                        s_cnt[hp] = cnt;
                        s_lo[hp] = lo;
                    }
                }
                __syncthreads();
            }
        }
        if (!FILL) {
            for (int t = threadIdx.x; t < hn; t += NB_THREADS) {
                deg[hb + t] = s_cnt[t];
                fwd[hb + t] = s_lo[t];
                atomicMax(max_deg, (unsigned)s_cnt[t]);
                atomicMax(max_deg + 1, (unsigned)(s_cnt[t] - s_lo[t]));
            }
        }
        __syncthreads();
    }
}

// The neighbour kernel of a pass (count or fill), box type and lower edge.
using NeighborsKernel = decltype(&k_neighbors<false, false, false>);

static NeighborsKernel neighbors_kernel(bool fill, bool periodic, bool lower)
{
    if (fill)
        return periodic ? (lower ? k_neighbors<true, true, true> : k_neighbors<true, true, false>)
                        : (lower ? k_neighbors<true, false, true> : k_neighbors<true, false, false>);
    return periodic ? (lower ? k_neighbors<false, true, true> : k_neighbors<false, true, false>)
                    : (lower ? k_neighbors<false, false, true> : k_neighbors<false, false, false>);
}

// ---------------------------------------------------------------- build

static int choose_ncell(int64_t box, int64_t rmax, int64_t n)
{
    int64_t nc = rmax > 0 ? box / rmax : 1;
    if (nc < 1) nc = 1;
    // keep the cell table no larger than the point count (and within 2^24 cells)
    while (nc > 1 && (nc * nc * nc > std::max<int64_t>(n, 1) || nc * nc * nc > (1ll << 24))) --nc;
    return (int)nc;
}

static void free_graph_arrays(gs_graph *g)
{
    if (!g) return;
    cudaFree(g->pts);
    cudaFree(g->inv);
    cudaFree(g->row_ptr);
    cudaFree(g->fwd);
    cudaFree(g->nbr);
    cudaFree(g->bin);
    cudaFree(g->work);
    cudaFree(g->err);
    cudaFree(g->chk);
    cudaFree(g->cfg3);
    cudaFree(g->cfg6);
    cudaFree(g->w);
    cudaFreeHost(g->h_nbr);
    cudaFreeHost(g->h_bin);
    for (int k = 0; k < GS_SLOTS; ++k) {
        cudaFree(g->s_nbr[k]);
        cudaFree(g->s_bin[k]);
    }
    delete[] g->win_row;
    delete[] g->win_e0;
    delete[] g->win_maxnbr;
    delete[] g->win_pair;
    delete[] g->win_first;
}

extern "C" void gs_graph_free(gs_graph_t g)
{
    if (!g) return;
    cudaDeviceSynchronize();
    free_graph_arrays(g);
    delete g;
}

static gs_status validate_build(const int32_t *coords, int64_t n, int64_t box, int periodic,
                                int64_t rmax, const int64_t *edges, int nb, gs_graph_t *out)
{
    if (!out) return gs_set_error(GS_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (n < 0 || n >= 2147483647ll) return gs_set_error(GS_ERR_ARG, "n = %lld outside [0, 2^31-1)", (long long)n);
    if (n > 0 && !coords) return gs_set_error(GS_ERR_ARG, "coords_dev is NULL");
    if (box < 1 || box > (1ll << 30)) return gs_set_error(GS_ERR_ARG, "box_lu = %lld outside [1, 2^30]", (long long)box);
    if (nb < 1 || nb > 255) return gs_set_error(GS_ERR_ARG, "nbins = %d outside [1, 255]", nb);
    if (!edges) return gs_set_error(GS_ERR_ARG, "edges_lu is NULL");
    if (edges[0] < 0) return gs_set_error(GS_ERR_ARG, "edges_lu[0] < 0");
    for (int k = 0; k < nb; ++k)
        if (edges[k + 1] <= edges[k]) return gs_set_error(GS_ERR_ARG, "edges_lu not strictly increasing at %d", k);
    if (edges[nb] != rmax) return gs_set_error(GS_ERR_ARG, "r_max_lu != edges_lu[nbins]");
    if (rmax > (1ll << 31)) return gs_set_error(GS_ERR_ARG, "r_max_lu too large");
    if (periodic && 2 * rmax > box) return gs_set_error(GS_ERR_ARG, "periodic box needs 2*r_max_lu <= box_lu");
    return GS_OK;
}

// Row windows over whole cells, each holding at most window_edges edges (a
// single larger cell gets a window of its own). Fills the graph's window
// tables; returns the first cell of every window and, last, the cell count.
static std::vector<int> plan_windows(gs_graph *g, const std::vector<int32_t> &cs, const std::vector<int64_t> &rp,
                                     int64_t window_edges)
{
    const int ncells = (int)cs.size() - 1;
    std::vector<int> wc(1, 0);
    for (int c = 0; c < ncells;) {
        int c1 = c + 1;
        while (c1 < ncells && rp[cs[c1 + 1]] - rp[cs[c]] <= window_edges) ++c1;
        wc.push_back(c1);
        c = c1;
    }
    const int nw = (int)wc.size() - 1;
    g->n_win = nw;
    g->win_row = new int64_t[nw + 1];
    g->win_e0 = new int64_t[nw + 1];
    g->win_maxnbr = new int32_t[nw];
    g->win_cap = GS_EDGE_PAD;
    for (int w = 0; w <= nw; ++w) {
        g->win_row[w] = cs[wc[w]];
        g->win_e0[w] = rp[g->win_row[w]];
    }
    for (int w = 0; w < nw; ++w) {
        g->win_maxnbr[w] = -1;
        g->win_cap = std::max(g->win_cap, g->win_e0[w + 1] + GS_EDGE_PAD - (g->win_e0[w] & ~(int64_t)3));
    }
    return wc;
}

// first[w] = the smallest i - r0 over the rows i in [r0, r1) that have a
// forward neighbour in window w (0xffffffff: none); edges staged at
// nbr - off; win_row on the device, nw + 1 entries.
__global__ void k_window_pairs(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd,
                               const int32_t *__restrict__ nbr, int64_t off, int64_t r0, int64_t r1,
                               const int64_t *__restrict__ win_row, int nw, unsigned *__restrict__ first)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = r0 + w0; i < r1; i += nwarp)
        for (int64_t p = row_ptr[i] + fwd[i] + lane; p < row_ptr[i + 1]; p += 32) {
            const int64_t k = nbr[p - off];
            int lo = 0, hi = nw;                         // window of k: win_row[lo] <= k < win_row[lo + 1]
            while (hi - lo > 1) {
                const int m = (lo + hi) >> 1;
                if (win_row[m] <= k) lo = m; else hi = m;
            }
            const unsigned r = (unsigned)(i - r0);
            if (r < first[lo]) atomicMin(first + lo, r);
        }
}

gs_status gs_stage_window(gs_graph_t g, int w, int slot, cudaStream_t st, int64_t *off)
{
    const int64_t a = g->win_e0[w] & ~(int64_t)3;
    const int64_t b = g->win_e0[w + 1] + GS_EDGE_PAD;       // the host arrays hold E + GS_EDGE_PAD entries
    GS_TRY_CUDA(cudaMemcpyAsync(g->s_nbr[slot], g->h_nbr + a, sizeof(int32_t) * (size_t)(b - a),
                                cudaMemcpyHostToDevice, st));
    GS_TRY_CUDA(cudaMemcpyAsync(g->s_bin[slot], g->h_bin + a, (size_t)(b - a), cudaMemcpyHostToDevice, st));
    *off = a;
    return GS_OK;
}

gs_status gs_stage_set(gs_graph_t g, int *held, int64_t *off, const int *need, int n, int *slot, cudaStream_t st)
{
    bool used[GS_SLOTS] = {};
    for (int q = 0; q < n; ++q) {
        slot[q] = -1;
        for (int k = 0; k < GS_SLOTS; ++k)
            if (held[k] == need[q]) slot[q] = k;
        if (slot[q] >= 0) used[slot[q]] = true;
    }
    for (int q = 0; q < n; ++q) {
        if (slot[q] >= 0) continue;
        int k = 0;
        while (used[k]) ++k;                 // n <= GS_SLOTS distinct windows: a free slot exists
        gs_status s = gs_stage_window(g, need[q], k, st, &off[k]);
        if (s != GS_OK) return s;
        held[k] = need[q];
        used[k] = true;
        for (int r = q; r < n; ++r)          // the same window asked for twice
            if (need[r] == need[q]) slot[r] = k;
    }
    return GS_OK;
}

// Edge budget of a graph: window_edges > 0 forces row windows of that size;
// 0 keeps the CSR on the device unless it would not fit, and then uses windows
// of an eighth of the free memory each (three staging slots); the environment
// variable GS_WINDOW_EDGES, when set to a positive count, overrides 0.
static int64_t choose_window_edges(int64_t window_edges, int64_t n_edges)
{
    if (window_edges > 0) return window_edges;
    if (const char *env = getenv("GS_WINDOW_EDGES")) {
        const long long v = atoll(env);
        if (v > 0) return v;
    }
    size_t fr = 0, tot = 0;
    if (cudaMemGetInfo(&fr, &tot) != cudaSuccess) return 0;
    const size_t need = 5 * (size_t)(n_edges + GS_EDGE_PAD) + ((size_t)256 << 20);
    if (need <= fr) return 0;
    return std::max<int64_t>((int64_t)(fr / 8 / 5), (int64_t)1 << 20);     // 5 B per edge
}

static gs_status build_impl(const int32_t *coords_dev, int64_t n, int64_t box_lu, int periodic,
                            int64_t r_max_lu, const int64_t *edges_lu, int nbins, int64_t window_edges,
                            void *cuda_stream, gs_graph_t *out)
{
    GS_ENTRY();
    gs_status s = validate_build(coords_dev, n, box_lu, periodic, r_max_lu, edges_lu, nbins, out);
    if (s != GS_OK) return s;
    if (window_edges < 0) return gs_set_error(GS_ERR_ARG, "window_edges < 0");
    cudaStream_t st = (cudaStream_t)cuda_stream;

    gs_graph *g = new gs_graph();
    memset(g, 0, sizeof(*g));
    cudaGetDevice(&g->device);
    g->n = n;
    g->box_lu = box_lu;
    g->periodic = periodic ? 1 : 0;
    g->nb = nbins;
    for (int k = 0; k <= nbins; ++k) g->edges[k] = edges_lu[k];
    g->ncell = choose_ncell(box_lu, r_max_lu, n);
    const int ncells = g->ncell * g->ncell * g->ncell;

    int32_t *cell = nullptr, *slot = nullptr, *cell_count = nullptr, *cell_start = nullptr;
    int32_t *tmp = nullptr, *perm = nullptr, *deg = nullptr;
    long long *esq = nullptr;
    unsigned *maxd = nullptr;
    int64_t *wrow_dev = nullptr;
    unsigned *pair_dev = nullptr;
    const int sms = gs_sm_count();
    const int grid1 = (int)std::min<int64_t>(std::max<int64_t>((n + 255) / 256, 1), (int64_t)sms * 16);

#define GS_BUILD_CUDA(call)                                                                  \
    do {                                                                                     \
        cudaError_t e_ = (call);                                                             \
        if (e_ != cudaSuccess) {                                                             \
            s = gs_set_error(e_ == cudaErrorMemoryAllocation ? GS_ERR_NOMEM : GS_ERR_CUDA,   \
                             "%s failed: %s", #call, cudaGetErrorString(e_));                \
            goto fail;                                                                       \
        }                                                                                    \
    } while (0)

    {
        const size_t nn = (size_t)std::max<int64_t>(n, 1);
        GS_BUILD_CUDA(gs_malloc(&g->pts, sizeof(int4) * nn));
        GS_BUILD_CUDA(gs_malloc(&g->inv, sizeof(int32_t) * nn));
        GS_BUILD_CUDA(gs_malloc(&g->row_ptr, sizeof(int64_t) * (nn + 1)));
        GS_BUILD_CUDA(gs_malloc(&g->fwd, sizeof(int32_t) * nn));
        GS_BUILD_CUDA(gs_malloc(&g->work, sizeof(unsigned long long) * 4));
        GS_BUILD_CUDA(gs_malloc(&g->err, sizeof(int32_t)));
        GS_BUILD_CUDA(gs_malloc(&g->chk, sizeof(unsigned)));
        GS_BUILD_CUDA(cudaMemset(g->chk, 0, sizeof(unsigned)));
        if (nbins <= 40) {
            // configuration index of every (z, x, y) bin triple, for the 3pCF kernel
            std::vector<uint16_t> h((size_t)nbins * nbins * nbins);
            for (int z = 0; z < nbins; ++z)
                for (int x = 0; x < nbins; ++x)
                    for (int y = 0; y < nbins; ++y) {
                        int v[3] = { x, y, z };
                        std::sort(v, v + 3);
                        h[((size_t)z * nbins + x) * nbins + y] = (uint16_t)gs_idx3(nbins, v[0], v[1], v[2]);
                    }
            GS_BUILD_CUDA(gs_malloc(&g->cfg3, sizeof(uint16_t) * h.size()));
            GS_BUILD_CUDA(cudaMemcpy(g->cfg3, h.data(), sizeof(uint16_t) * h.size(), cudaMemcpyHostToDevice));
        }
        GS_BUILD_CUDA(gs_malloc_async(&cell, sizeof(int32_t) * nn, st));
        GS_BUILD_CUDA(gs_malloc_async(&slot, sizeof(int32_t) * nn, st));
        GS_BUILD_CUDA(gs_malloc_async(&tmp, sizeof(int32_t) * nn, st));
        GS_BUILD_CUDA(gs_malloc_async(&perm, sizeof(int32_t) * nn, st));
        GS_BUILD_CUDA(gs_malloc_async(&deg, sizeof(int32_t) * nn, st));
        GS_BUILD_CUDA(gs_malloc_async(&cell_count, sizeof(int32_t) * ncells, st));
        GS_BUILD_CUDA(gs_malloc_async(&cell_start, sizeof(int32_t) * (ncells + 1), st));
        GS_BUILD_CUDA(gs_malloc_async(&esq, sizeof(long long) * 256, st));
        GS_BUILD_CUDA(gs_malloc_async(&maxd, 2 * sizeof(unsigned), st));

        long long hesq[256];
        for (int k = 0; k <= nbins; ++k) hesq[k] = (long long)edges_lu[k] * edges_lu[k];
        GS_BUILD_CUDA(cudaMemcpyAsync(esq, hesq, sizeof(long long) * (nbins + 1), cudaMemcpyHostToDevice, st));
        GS_BUILD_CUDA(cudaMemsetAsync(cell_count, 0, sizeof(int32_t) * ncells, st));
        GS_BUILD_CUDA(cudaMemsetAsync(g->err, 0, sizeof(int32_t), st));
        GS_BUILD_CUDA(cudaMemsetAsync(maxd, 0, 2 * sizeof(unsigned), st));

        if (n > 0) {
            k_cell_assign<<<grid1, 256, 0, st>>>(coords_dev, n, (int)box_lu, g->ncell, cell, slot,
                                                 cell_count, g->err);
            gs_note_launch();
            GS_BUILD_CUDA(cudaGetLastError());
        }
        s = gs_scan_i32_to_i32(cell_count, cell_start, ncells, st);
        if (s != GS_OK) goto fail;
        if (n > 0) {
            k_cell_scatter<<<grid1, 256, 0, st>>>(cell, slot, cell_start, n, tmp);
            gs_note_launch();
            const int gw = (int)std::min<int64_t>(((int64_t)ncells * 32 + 255) / 256, (int64_t)sms * 32);
            k_cell_order<<<gw, 256, 0, st>>>(cell_start, ncells, tmp, perm);
            gs_note_launch();
            k_gather_points<<<grid1, 256, 0, st>>>(coords_dev, perm, n, g->pts, g->inv);
            gs_note_launch();
            neighbors_kernel(false, g->periodic, edges_lu[0] > 0)<<<dim3(ncells, NB_SPLIT), NB_THREADS, 0, st>>>(
                g->pts, cell_start, g->ncell, (int)box_lu, g->periodic,
                (long long)edges_lu[0] * edges_lu[0], (long long)r_max_lu * r_max_lu, esq, nbins,
                deg, g->fwd, nullptr, nullptr, nullptr, maxd, 0, 0, g->chk, 0);
            gs_note_launch();
            GS_BUILD_CUDA(cudaGetLastError());
        }
        s = gs_scan_i32_to_i64(deg, g->row_ptr, n, st);
        if (s != GS_OK) goto fail;

        int32_t herr = 0;
        unsigned hmax[2] = { 0, 0 };
        GS_BUILD_CUDA(cudaMemcpyAsync(&g->n_edges, g->row_ptr + n, sizeof(int64_t), cudaMemcpyDeviceToHost, st));
        GS_BUILD_CUDA(cudaMemcpyAsync(&herr, g->err, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
        GS_BUILD_CUDA(cudaMemcpyAsync(hmax, maxd, 2 * sizeof(unsigned), cudaMemcpyDeviceToHost, st));
        GS_BUILD_CUDA(cudaStreamSynchronize(st));
        if (herr) {
            s = gs_set_error(GS_ERR_ARG, "a coordinate lies outside [0, box_lu)");
            goto fail;
        }
        g->max_degree = (int32_t)hmax[0];
        g->max_forward = (int32_t)hmax[1];

        const size_t ne = (size_t)(g->n_edges + GS_EDGE_PAD);
        const int64_t wedges = choose_window_edges(window_edges, g->n_edges);
        g->nbr_len = (int64_t)ne;
        if (wedges == 0) {
            GS_BUILD_CUDA(gs_malloc(&g->nbr, sizeof(int32_t) * ne));
            GS_BUILD_CUDA(gs_malloc(&g->bin, ne));
            GS_BUILD_CUDA(cudaMemsetAsync(g->nbr + g->n_edges, 0xff, sizeof(int32_t) * GS_EDGE_PAD, st));
            GS_BUILD_CUDA(cudaMemsetAsync(g->bin + g->n_edges, 0, GS_EDGE_PAD, st));
            if (n > 0 && g->n_edges > 0) {
                neighbors_kernel(true, g->periodic, edges_lu[0] > 0)<<<dim3(ncells, NB_SPLIT), NB_THREADS, 0, st>>>(
                    g->pts, cell_start, g->ncell, (int)box_lu, g->periodic,
                    (long long)edges_lu[0] * edges_lu[0], (long long)r_max_lu * r_max_lu, esq, nbins,
                    nullptr, nullptr, g->row_ptr, g->nbr, g->bin, nullptr, 0, 0, g->chk, (int64_t)ne);
                gs_note_launch();
                GS_BUILD_CUDA(cudaGetLastError());
            }
        } else {
            // row windows: rows filled one window at a time into a device slot,
            // then copied to pinned host memory
            std::vector<int32_t> hcs((size_t)ncells + 1);
            std::vector<int64_t> hrp((size_t)n + 1);
            GS_BUILD_CUDA(cudaMemcpyAsync(hcs.data(), cell_start, sizeof(int32_t) * hcs.size(),
                                          cudaMemcpyDeviceToHost, st));
            GS_BUILD_CUDA(cudaMemcpyAsync(hrp.data(), g->row_ptr, sizeof(int64_t) * hrp.size(),
                                          cudaMemcpyDeviceToHost, st));
            GS_BUILD_CUDA(cudaStreamSynchronize(st));
            const std::vector<int> wc = plan_windows(g, hcs, hrp, wedges);
            GS_BUILD_CUDA(gs_malloc_host(&g->h_nbr, sizeof(int32_t) * ne));
            GS_BUILD_CUDA(gs_malloc_host(&g->h_bin, ne));
            memset(g->h_nbr + g->n_edges, 0xff, sizeof(int32_t) * GS_EDGE_PAD);
            memset(g->h_bin + g->n_edges, 0, GS_EDGE_PAD);
            g->nbr_len = g->win_cap;
            for (int k = 0; k < GS_SLOTS; ++k) {
                GS_BUILD_CUDA(gs_malloc(&g->s_nbr[k], sizeof(int32_t) * (size_t)g->win_cap));
                GS_BUILD_CUDA(gs_malloc(&g->s_bin[k], (size_t)g->win_cap));
            }
            const int nw = g->n_win;
            g->win_pair = new uint8_t[(size_t)nw * nw]();
            g->win_first = new int64_t[(size_t)nw * nw]();
            std::vector<unsigned> hpair((size_t)nw * nw, 0u);
            GS_BUILD_CUDA(gs_malloc_async(&wrow_dev, sizeof(int64_t) * (nw + 1), st));
            GS_BUILD_CUDA(gs_malloc_async(&pair_dev, sizeof(unsigned) * (size_t)nw * nw, st));
            GS_BUILD_CUDA(cudaMemcpyAsync(wrow_dev, g->win_row, sizeof(int64_t) * (nw + 1), cudaMemcpyHostToDevice, st));
            GS_BUILD_CUDA(cudaMemsetAsync(pair_dev, 0xff, sizeof(unsigned) * (size_t)nw * nw, st));
            for (int w = 0; w < g->n_win; ++w) {
                const int cell0 = wc[w], cell1 = wc[w + 1];
                const int64_t e0 = g->win_e0[w], e1 = g->win_e0[w + 1];
                if (e1 > e0) {
                    const int64_t a = e0 & ~(int64_t)3;
                    neighbors_kernel(true, g->periodic, edges_lu[0] > 0)<<<dim3(cell1 - cell0, NB_SPLIT), NB_THREADS, 0, st>>>(
                        g->pts, cell_start, g->ncell, (int)box_lu, g->periodic,
                        (long long)edges_lu[0] * edges_lu[0], (long long)r_max_lu * r_max_lu, esq, nbins,
                        nullptr, nullptr, g->row_ptr, g->s_nbr[0], g->s_bin[0], nullptr, cell0, a, g->chk, g->win_cap);
                    gs_note_launch();
                    GS_BUILD_CUDA(cudaGetLastError());
                    GS_BUILD_CUDA(cudaMemcpyAsync(g->h_nbr + e0, g->s_nbr[0] + (e0 - a), sizeof(int32_t) * (e1 - e0),
                                                  cudaMemcpyDeviceToHost, st));
                    GS_BUILD_CUDA(cudaMemcpyAsync(g->h_bin + e0, g->s_bin[0] + (e0 - a), (size_t)(e1 - e0),
                                                  cudaMemcpyDeviceToHost, st));
                    const int64_t rows = g->win_row[w + 1] - g->win_row[w];
                    const int gp = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)sms * 8);
                    k_window_pairs<<<gp, 256, 0, st>>>(g->row_ptr, g->fwd, g->s_nbr[0], a, g->win_row[w],
                                                       g->win_row[w + 1], wrow_dev, nw, pair_dev + (size_t)w * nw);
                    gs_note_launch();
                    GS_BUILD_CUDA(cudaGetLastError());
                }
            }
            GS_BUILD_CUDA(cudaMemcpyAsync(hpair.data(), pair_dev, sizeof(unsigned) * hpair.size(),
                                          cudaMemcpyDeviceToHost, st));
            GS_BUILD_CUDA(cudaStreamSynchronize(st));
            for (size_t q = 0; q < hpair.size(); ++q) {
                g->win_pair[q] = hpair[q] != 0xffffffffu ? 1 : 0;
                g->win_first[q] = g->win_row[q / nw] + (g->win_pair[q] ? (int64_t)hpair[q] : 0);
            }
            for (int w = 0; w < g->n_win; ++w)        // rows are sorted: the last entry is the row's largest
                for (int64_t i = g->win_row[w]; i < g->win_row[w + 1]; ++i)
                    if (hrp[i + 1] > hrp[i]) g->win_maxnbr[w] = std::max(g->win_maxnbr[w], g->h_nbr[hrp[i + 1] - 1]);
        }
    }
    if (GS_CHECKED_BUILD) {                                   // the fill kernels' bounds checks
        s = gs_checked_end(g, st, "graph build");
        if (s != GS_OK) goto fail;
    }
    cudaFreeAsync(cell, st);
    cudaFreeAsync(slot, st);
    cudaFreeAsync(tmp, st);
    cudaFreeAsync(perm, st);
    cudaFreeAsync(deg, st);
    cudaFreeAsync(cell_count, st);
    cudaFreeAsync(cell_start, st);
    cudaFreeAsync(esq, st);
    cudaFreeAsync(maxd, st);
    cudaFreeAsync(wrow_dev, st);
    cudaFreeAsync(pair_dev, st);
    *out = g;
    return GS_OK;

fail:
    cudaStreamSynchronize(st);
    cudaFree(cell);
    cudaFree(slot);
    cudaFree(tmp);
    cudaFree(perm);
    cudaFree(deg);
    cudaFree(cell_count);
    cudaFree(cell_start);
    cudaFree(esq);
    cudaFree(maxd);
    cudaFree(wrow_dev);
    cudaFree(pair_dev);
    free_graph_arrays(g);
    delete g;
    return s;
#undef GS_BUILD_CUDA
}

// ---------------------------------------------------------------- export

// Degree of output row t: input point ids[t] (or t when ids is NULL).
__global__ void k_input_degrees(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ inv,
                                const int32_t *__restrict__ ids, int64_t n, int32_t *__restrict__ deg_in)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int p = inv[ids ? ids[i] : i];
        deg_in[i] = (int32_t)(row_ptr[p + 1] - row_ptr[p]);
    }
}

constexpr int EX_THREADS = 256;
constexpr int EX_SMEM = 4096;   // rows up to this length are sorted in shared memory

// One block per input row: map neighbour ids to input numbering and sort the
// row by them (bitonic in shared memory, rank sort for longer rows).
__global__ void __launch_bounds__(EX_THREADS)
k_export_rows(const int4 *__restrict__ pts, const int32_t *__restrict__ inv, const int32_t *__restrict__ ids,
              const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ nbr,
              const uint8_t *__restrict__ bin, int64_t off, int64_t p_lo, int64_t p_hi, int64_t n,
              const int64_t *__restrict__ out_ptr, int32_t *__restrict__ out_nbr, uint8_t *__restrict__ out_bin)
{
    // rows of internal index p in [p_lo, p_hi) only; their edges at (nbr, bin) - off
    __shared__ unsigned long long s_kv[EX_SMEM];
    for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int p = inv[ids ? ids[i] : i];
        if (p < p_lo || p >= p_hi) continue;             // block-uniform
        const int64_t r0 = row_ptr[p] - off;
        const int len = (int)(row_ptr[p + 1] - row_ptr[p]);
        const int64_t o0 = out_ptr[i];
        if (len <= EX_SMEM) {
            int pw = 1;
            while (pw < len) pw <<= 1;
            for (int t = threadIdx.x; t < pw; t += EX_THREADS)
                s_kv[t] = t < len ? (((unsigned long long)(unsigned)pts[nbr[r0 + t]].w << 8) | bin[r0 + t])
                                  : ~0ull;
            __syncthreads();
            for (int k = 2; k <= pw; k <<= 1)
                for (int j = k >> 1; j > 0; j >>= 1) {
                    for (int t = threadIdx.x; t < pw; t += EX_THREADS) {
                        const int u = t ^ j;
                        if (u > t) {
                            const bool up = (t & k) == 0;
                            const unsigned long long a = s_kv[t], b = s_kv[u];
                            if ((a > b) == up) {
                                s_kv[t] = b;
                                s_kv[u] = a;
                            }
                        }
                    }
                    __syncthreads();
                }
            for (int t = threadIdx.x; t < len; t += EX_THREADS) {
                out_nbr[o0 + t] = (int32_t)(s_kv[t] >> 8);
                out_bin[o0 + t] = (uint8_t)(s_kv[t] & 0xff);
            }
            __syncthreads();
        } else {
            for (int t = threadIdx.x; t < len; t += EX_THREADS) {
                const int e = pts[nbr[r0 + t]].w;
                int r = 0;
                for (int u = 0; u < len; ++u) r += pts[nbr[r0 + u]].w < e;
                out_nbr[o0 + r] = e;
                out_bin[o0 + r] = bin[r0 + t];
            }
        }
    }
}

// Rows of the input points ids[0..count) (all points in input order when ids is
// NULL), neighbour ids in input numbering, each row sorted.
static gs_status export_rows(gs_graph_t g, const int32_t *ids, int64_t count, int64_t *row_ptr_dev,
                             int32_t *nbr_dev, uint8_t *bin_dev, cudaStream_t st)
{
    if (count == 0) {
        GS_TRY_CUDA(cudaMemsetAsync(row_ptr_dev, 0, sizeof(int64_t), st));
        return GS_OK;
    }
    int32_t *deg_in = nullptr;
    GS_TRY_CUDA(gs_malloc_async(&deg_in, sizeof(int32_t) * count, st));
    const int sms = gs_sm_count();
    const int grid = (int)std::min<int64_t>((count + 255) / 256, (int64_t)sms * 16);
    k_input_degrees<<<grid, 256, 0, st>>>(g->row_ptr, g->inv, ids, count, deg_in);
    gs_note_launch();
    gs_status s = gs_scan_i32_to_i64(deg_in, row_ptr_dev, count, st);
    cudaFreeAsync(deg_in, st);
    if (s != GS_OK) return s;
    if (nbr_dev && g->n_edges > 0) {
        const int gridr = (int)std::min<int64_t>(count, (int64_t)sms * 8);
        if (g->n_win == 0) {
            k_export_rows<<<gridr, EX_THREADS, 0, st>>>(g->pts, g->inv, ids, g->row_ptr, g->nbr, g->bin, 0, 0, g->n,
                                                        count, row_ptr_dev, nbr_dev, bin_dev);
            gs_note_launch();
        }
        for (int w = 0; w < g->n_win; ++w) {            // windowed: the rows of one staged window at a time
            if (g->win_e0[w + 1] == g->win_e0[w]) continue;
            int64_t off = 0;
            s = gs_stage_window(g, w, 0, st, &off);
            if (s != GS_OK) return s;
            k_export_rows<<<gridr, EX_THREADS, 0, st>>>(g->pts, g->inv, ids, g->row_ptr, g->s_nbr[0], g->s_bin[0],
                                                        off, g->win_row[w], g->win_row[w + 1], count, row_ptr_dev,
                                                        nbr_dev, bin_dev);
            gs_note_launch();
        }
    }
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

extern "C" gs_status gs_graph_export_csr(gs_graph_t g, int64_t *row_ptr_dev, int32_t *nbr_dev,
                                         uint8_t *bin_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !row_ptr_dev || (g->n_edges > 0 && (!nbr_dev || !bin_dev)))
        return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    return export_rows(g, nullptr, g->n, row_ptr_dev, nbr_dev, bin_dev, (cudaStream_t)cuda_stream);
}

extern "C" gs_status gs_graph_export_rows(gs_graph_t g, const int32_t *ids_dev, int64_t count,
                                          int64_t *row_ptr_dev, int32_t *nbr_dev, uint8_t *bin_dev,
                                          void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !row_ptr_dev || (count > 0 && !ids_dev) || (nbr_dev && !bin_dev))
        return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (count < 0) return gs_set_error(GS_ERR_ARG, "negative row count");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    gs_status s = gs_check_ids(g, ids_dev, count, st);
    if (s != GS_OK) return s;
    return export_rows(g, ids_dev, count, row_ptr_dev, nbr_dev, bin_dev, st);
}

__global__ void k_perm(const int4 *__restrict__ pts, int64_t n, int32_t *__restrict__ perm)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n;
         p += (int64_t)gridDim.x * blockDim.x)
        perm[p] = pts[p].w;
}

extern "C" gs_status gs_graph_export_perm(gs_graph_t g, int32_t *perm_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || (g->n > 0 && !perm_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (g->n == 0) return GS_OK;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int grid = (int)std::min<int64_t>((g->n + 255) / 256, (int64_t)gs_sm_count() * 16);
    k_perm<<<grid, 256, 0, st>>>(g->pts, g->n, perm_dev);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

// Per-graph work statistics: sum C(f,2), sum b*f, max f (see gramsci_gb.h).
__global__ void k_graph_stats(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd,
                              int64_t n, unsigned long long *__restrict__ acc)
{
    unsigned long long tail = 0, walk = 0;
    unsigned fmax = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const unsigned long long d = (unsigned long long)(row_ptr[i + 1] - row_ptr[i]);
        const unsigned long long b = (unsigned long long)fwd[i], f = d - b;
        tail += f * (f - (f > 0)) / 2;
        walk += b * f;
        fmax = max(fmax, (unsigned)f);
    }
    for (int o = 16; o > 0; o >>= 1) {
        tail += __shfl_down_sync(0xffffffffu, tail, o);
        walk += __shfl_down_sync(0xffffffffu, walk, o);
        fmax = max(fmax, __shfl_down_sync(0xffffffffu, fmax, o));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(acc, tail);
        atomicAdd(acc + 1, walk);
        atomicMax(acc + 2, (unsigned long long)fmax);
    }
}

extern "C" gs_status gs_graph_stats(gs_graph_t g, gs_graph_stats_t *out, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !out) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    unsigned long long *acc = nullptr, h[3] = { 0, 0, 0 };
    GS_TRY_CUDA(gs_malloc_async(&acc, sizeof(h), st));
    cudaError_t e = cudaMemsetAsync(acc, 0, sizeof(h), st);
    if (e == cudaSuccess && g->n > 0) {
        const int grid = (int)std::min<int64_t>((g->n + 255) / 256, (int64_t)gs_sm_count() * 8);
        k_graph_stats<<<grid, 256, 0, st>>>(g->row_ptr, g->fwd, g->n, acc);
        gs_note_launch();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(h, acc, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFreeAsync(acc, st);
    if (e != cudaSuccess) return gs_set_error(GS_ERR_CUDA, "graph stats failed: %s", cudaGetErrorString(e));
    out->n = g->n;
    out->n_edges = g->n_edges;
    out->max_degree = g->max_degree;
    out->max_forward = (int32_t)h[2];
    out->cells_per_axis = g->ncell;
    out->reserved = 0;
    out->hub_tail = (int64_t)h[0];
    out->spoke_walk = (int64_t)h[1];
    return GS_OK;
}

// Per-hub work of the 3pCF walk, one warp per hub of [r0, r1): f_i and
// w_i = sum over the forward spokes j of i of f_j. Row entries are read at
// e - off (the staged window of a windowed graph, else the device CSR).
__global__ void k_hub_work(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ fwd,
                           const int32_t *__restrict__ nbr, int64_t off, int64_t r0, int64_t r1,
                           int32_t *__restrict__ f_out, int64_t *__restrict__ w_out)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = r0 + (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < r1; i += warps) {
        const int64_t p0 = row_ptr[i] + fwd[i], pe = row_ptr[i + 1];
        long long s = 0;
        for (int64_t p = p0 + lane; p < pe; p += 32) {
            const int32_t j = nbr[p - off];
            s += (row_ptr[j + 1] - row_ptr[j]) - fwd[j];
        }
        for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
        if (lane == 0) {
            if (f_out) f_out[i] = (int32_t)(pe - p0);
            w_out[i] = s;
        }
    }
}

extern "C" gs_status gs_graph_hub_work(gs_graph_t g, int32_t *fwd_dev, int64_t *walk_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || (g->n > 0 && !walk_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    gs_status s = gs_check_device(g);
    if (s != GS_OK || g->n == 0) return s;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int grid = (int)std::min<int64_t>((g->n + 7) / 8, (int64_t)gs_sm_count() * 8);
    if (g->n_win == 0) {
        k_hub_work<<<grid, 256, 0, st>>>(g->row_ptr, g->fwd, g->nbr, 0, 0, g->n, fwd_dev, walk_dev);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
        return GS_OK;
    }
    // windowed: stage each window's rows in turn; the spokes' degrees are on the device
    for (int w = 0; w < g->n_win; ++w) {
        if (g->win_row[w + 1] == g->win_row[w]) continue;
        int64_t off = 0;
        s = gs_stage_window(g, w, 0, st, &off);
        if (s != GS_OK) return s;
        k_hub_work<<<grid, 256, 0, st>>>(g->row_ptr, g->fwd, g->s_nbr[0], off, g->win_row[w], g->win_row[w + 1],
                                         fwd_dev, walk_dev);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }
    return GS_OK;
}

gs_status gs_check_device(gs_graph_t g)
{
    int dev = -1;
    GS_TRY_CUDA(cudaGetDevice(&dev));
    if (dev != g->device)
        return gs_set_error(GS_ERR_ARG, "the graph lives on device %d but device %d is current", g->device, dev);
    return GS_OK;
}

extern "C" gs_status gs_graph_info(gs_graph_t g, int64_t *n, int64_t *n_edges, int32_t *max_degree)
{
    GS_ENTRY();
    if (!g) return gs_set_error(GS_ERR_ARG, "graph is NULL");
    if (n) *n = g->n;
    if (n_edges) *n_edges = g->n_edges;
    if (max_degree) *max_degree = g->max_degree;
    return GS_OK;
}

extern "C" gs_status gs_build_graph(const int32_t *coords_dev, int64_t n, int64_t box_lu, int periodic,
                                    int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                                    void *cuda_stream, gs_graph_t *out)
{
    return build_impl(coords_dev, n, box_lu, periodic, r_max_lu, edges_lu, nbins, 0, cuda_stream, out);
}

extern "C" gs_status gs_build_graph_windowed(const int32_t *coords_dev, int64_t n, int64_t box_lu, int periodic,
                                             int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                                             int64_t window_edges, void *cuda_stream, gs_graph_t *out)
{
    GS_ENTRY();
    if (window_edges < 1) return gs_set_error(GS_ERR_ARG, "window_edges must be >= 1");
    return build_impl(coords_dev, n, box_lu, periodic, r_max_lu, edges_lu, nbins, window_edges, cuda_stream, out);
}

extern "C" gs_status gs_graph_windows(gs_graph_t g, int32_t *n_windows, int64_t *window_edges_max)
{
    GS_ENTRY();
    if (!g) return gs_set_error(GS_ERR_ARG, "graph is NULL");
    int64_t m = 0;
    for (int w = 0; w < g->n_win; ++w) m = std::max(m, g->win_e0[w + 1] - g->win_e0[w]);
    if (n_windows) *n_windows = g->n_win;
    if (window_edges_max) *window_edges_max = g->n_win ? m : g->n_edges;
    return GS_OK;
}
