// gs_internal.cuh -- shared definitions of the sm_103a library (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gramsci_gb.h"

// ---------------------------------------------------------------- the graph

// Device staging slots of a windowed graph.
constexpr int GS_SLOTS = 3;

// HBM layout of one graph (N points, E directed edges):
//   pts      int4   [N]    x, y, z and the input index, points sorted by cell
//                          (16-byte rows: one aligned vector load per point)
//   inv      int32  [N]    input index -> internal index
//   row_ptr  int64  [N+1]  CSR offsets (E may exceed 2^31, GRAMSCI §III.5.1)
//   fwd      int32  [N]    offset in row i of the first neighbour > i
//   nbr      int32  [E]    neighbour ids (internal), strictly increasing per row
//   bin      uint8  [E]    radial bin of each edge
// Internal index = position in cell order, so a hub's neighbours are a few
// contiguous index ranges and consecutive hubs share most of their spokes
// (L2 reuse in the counting kernels).
struct gs_graph {
    int device;
    int64_t n;
    int64_t box_lu;
    int periodic;
    int nb;
    int64_t edges[256];
    int64_t n_edges;
    int32_t max_degree;
    int32_t max_forward;       // largest |{j in N(i) : j > i}|
    int ncell;                 // cells per axis
    int4 *pts;
    int32_t *inv;
    int64_t *row_ptr;
    int32_t *fwd;
    int32_t *nbr;
    uint8_t *bin;
    unsigned long long *work;  // 4 device counters used by the count kernels
    int32_t *err;              // device error word of the build kernels
    unsigned *chk;             // device check word of checked builds (see GS_DCHECK)
    int64_t nbr_len;           // entries of nbr / bin (E + GS_EDGE_PAD), or of a staging slot when windowed
    uint16_t *cfg3;            // [nb][nb][nb] idx3(sort(x, y, z)) at (z, x, y), nb <= 40; or NULL
    int32_t *cfg6;             // [nb^6] six-bin 4pCF configuration and orientation (built on first use)
    int ncfg6;
    int16_t *w;                // [N] point weights in internal order (set by gs_graph_set_weights), or NULL

    // Row windows (§III.5.3 out-of-core operation). With n_win > 0 the edge
    // arrays live in pinned host memory (h_nbr, h_bin, padded like nbr / bin)
    // and nbr / bin are NULL. Window w holds the rows [win_row[w], win_row[w+1])
    // (whole cells), i.e. the edges [win_e0[w], win_e0[w+1]); win_maxnbr[w] is
    // the largest neighbour id in those rows (-1 if none). A window is staged
    // into one of two device slots from edge (win_e0[w] & ~3) on, through
    // win_e0[w+1] + GS_EDGE_PAD, so 16-byte vector reads stay aligned and in
    // bounds.
    int n_win;
    int64_t *win_row;          // host [n_win + 1]
    int64_t *win_e0;           // host [n_win + 1]
    int32_t *win_maxnbr;       // host [n_win]
    uint8_t *win_pair;         // host [n_win][n_win]: 1 if a row of window h has a forward neighbour in window w
    int64_t *win_first;        // host [n_win][n_win]: the first such row of window h (when win_pair is 1)
    int32_t *h_nbr;
    uint8_t *h_bin;
    int64_t win_cap;           // edges a staging slot holds
    int32_t *s_nbr[GS_SLOTS];  // device staging slots (three: a hub window, a spoke window and
    uint8_t *s_bin[GS_SLOTS];  // the next tile's window, copied while the current tile runs)
};

// Copy window w of a windowed graph into staging slot `slot` (asynchronously
// on st); *off is the global edge index of the slot's first entry (a multiple
// of 4).
gs_status gs_stage_window(gs_graph_t g, int w, int slot, cudaStream_t st, int64_t *off);

// Make the windows need[0..n) (n <= GS_SLOTS) resident in the staging slots,
// stream-ordered on st: a window already held (held[k] == window) is reused,
// others are copied into slots this call does not need. On return slot[q] is
// the slot of need[q] and off[slot[q]] its first edge. held / off persist
// across calls of one query (initialise held to -1).
gs_status gs_stage_set(gs_graph_t g, int *held, int64_t *off, const int *need, int n, int *slot, cudaStream_t st);

// Is there an edge between a row of window h and a row of window c (either
// direction)?
inline bool gs_windows_adjacent(gs_graph_t g, int h, int c)
{
    return g->win_pair[(size_t)h * g->n_win + c] || g->win_pair[(size_t)c * g->n_win + h];
}

// ---------------------------------------------------------------- errors

gs_status gs_set_error(gs_status s, const char *fmt, ...);

// A public entry point in progress on this thread. The outermost one (calls
// nest: gs_3pcf_from_host calls gs_build_graph) clears the thread's error
// message and restarts the allocation ordinal that fault injection counts.
// Every one opens an NVTX range named after the call, so a profiler's
// timeline shows the graph build and each count as a phase (NVTX is
// header-only and costs nothing when no tool is attached).
struct gs_call_scope {
    explicit gs_call_scope(const char *name);
    ~gs_call_scope();
};
#define GS_ENTRY() gs_call_scope gs_scope_(__func__)

// Every device and pinned-host allocation of the library passes this gate
// first. It counts the allocation (gs_alloc_calls) and, when the environment
// variable GS_FAULT holds "alloc:N", fails the N-th allocation of the current
// outermost call with cudaErrorMemoryAllocation without allocating anything,
// so that the NOMEM path of every allocation site can be exercised on the host.
cudaError_t gs_alloc_gate();

template <typename T>
inline cudaError_t gs_malloc(T **p, size_t bytes)
{
    const cudaError_t e = gs_alloc_gate();
    return e != cudaSuccess ? e : cudaMalloc((void **)p, bytes);
}

template <typename T>
inline cudaError_t gs_malloc_async(T **p, size_t bytes, cudaStream_t st)
{
    const cudaError_t e = gs_alloc_gate();
    return e != cudaSuccess ? e : cudaMallocAsync((void **)p, bytes, st);
}

template <typename T>
inline cudaError_t gs_malloc_host(T **p, size_t bytes)
{
    const cudaError_t e = gs_alloc_gate();
    return e != cudaSuccess ? e : cudaMallocHost((void **)p, bytes);
}

#define GS_TRY_CUDA(call)                                                              \
    do {                                                                               \
        cudaError_t e_ = (call);                                                       \
        if (e_ != cudaSuccess) {                                                       \
            return gs_set_error(e_ == cudaErrorMemoryAllocation ? GS_ERR_NOMEM : GS_ERR_CUDA, \
                                "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                                __FILE__, __LINE__);                                   \
        }                                                                              \
    } while (0)

// Count one kernel launch (reported by gs_kernel_launches).
void gs_note_launch();

// Entries of padding after the last edge of nbr / bin: a warp may read whole
// 16-byte vectors up to 256 entries past a row's end without leaving the
// allocation (the 3pCF walk reads every 256-entry step that starts in a row
// whole).
constexpr int64_t GS_EDGE_PAD = 256;

// GS_ERR_ARG unless the current device is the one the graph was built on
// (every pointer a count passes to its kernels belongs to that device).
gs_status gs_check_device(gs_graph_t g);

#define GS_TRY_DEVICE(g)                                                               \
    do {                                                                               \
        gs_status s_ = gs_check_device(g);                                             \
        if (s_ != GS_OK) return s_;                                                    \
    } while (0)

// GS_ERR_ARG unless every one of `count` device input indices lies in [0, n);
// synchronises st.
gs_status gs_check_ids(gs_graph_t g, const int32_t *ids, int64_t count, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int gs_sm_count();

// Exclusive scan of n int32 values; out has n+1 entries (out[n] = total).
gs_status gs_scan_i32_to_i64(const int32_t *in, int64_t *out, int64_t n, cudaStream_t st);
gs_status gs_scan_i32_to_i32(const int32_t *in, int32_t *out, int64_t n, cudaStream_t st);

// ---------------------------------------------------------------- checked builds
//
// A build compiled with -DGS_CHECKED (libgramsci_gb_checked.so) tests the
// indices of the hot kernels' shared-memory and global accesses. A failed
// test sets bit `site` of the graph's check word and the access is skipped;
// the entry point reads the word after its kernels (synchronising its
// stream) and returns GS_ERR_INTERNAL naming the sites. In the regular build
// every test is the constant true and the word is never read.
#ifdef GS_CHECKED
constexpr bool GS_CHECKED_BUILD = true;
__device__ __forceinline__ bool gs_dcheck(bool ok, unsigned *word, int site)
{
    if (!ok) atomicOr(word, 1u << site);
    return ok;
}
#define GS_DCHECK(ok, word, site) gs_dcheck((ok), (word), (site))
#else
constexpr bool GS_CHECKED_BUILD = false;
#define GS_DCHECK(ok, word, site) true
#endif

// Check sites (bits of the check word).
enum {
    GS_SITE_NB_ROW = 0,        // k_neighbors: an edge written outside its row
    GS_SITE_C3M_MAP_W = 1,     // k_count3m: byte-map or segment-table write
    GS_SITE_C3M_MAP_R = 2,     // k_count3m: byte-map read
    GS_SITE_C3M_HIST = 3,      // k_count3m: histogram counter
    GS_SITE_C3M_ROW = 4,       // k_count3m: spoke-row read
    GS_SITE_C3_BITMAP = 5,     // k_count3: bitmap, rank or bin read
    GS_SITE_C3_HIST = 6,       // k_count3: histogram counter
    GS_SITE_C4_BITS = 7,       // k_count4_*: adjacency bits or spoke vector
    GS_SITE_C4_HIST = 8        // k_count4_*: histogram counter
};

// Clear the check word before a count's kernels, and read it after them
// (checked builds only; both are no-ops otherwise).
gs_status gs_checked_begin(gs_graph_t g, cudaStream_t st);
gs_status gs_checked_end(gs_graph_t g, cudaStream_t st, const char *what);

// ---------------------------------------------------------------- device helpers

// Minimum-image (periodic) or raw displacement component b - a; |b - a| < 2^30.
__device__ __forceinline__ int gs_delta(int a, int b, int box, int periodic)
{
    int d = b - a;
    if (periodic) {
        d -= (2 * d >= box) ? box : 0;
        d += (2 * d < -box) ? box : 0;
    }
    return d;
}

__device__ __forceinline__ long long gs_norm2(int dx, int dy, int dz)
{
    return (long long)dx * dx + (long long)dy * dy + (long long)dz * dz;
}

// Packed lexicographic index of a sorted bin triple a <= b <= c over nb bins:
// (#triples with first bin < a) + (#with first bin a and second bin < b) + (c - b).
__host__ __device__ __forceinline__ int64_t gs_idx3(int nb, int a, int b, int c)
{
    auto tet = [](int64_t m) { return m * (m + 1) * (m + 2) / 6; };
    auto g = [nb](int64_t t) { return t * nb - t * (t - 1) / 2; };
    return tet(nb) - tet(nb - a) + g(b) - g(a) + (c - b);
}

// Packed lexicographic index of a strictly increasing triple a < b < c.
__host__ __device__ __forceinline__ int64_t gs_idx4(int nb, int a, int b, int c)
{
    auto c3 = [](int64_t m) { return m * (m - 1) * (m - 2) / 6; };
    auto h = [nb](int64_t t) { return t * (nb - 1) - t * (t - 1) / 2; };
    return c3(nb) - c3(nb - a) + h(b) - h(a + 1) + (c - b - 1);
}

__host__ __device__ __forceinline__ int64_t gs_ncfg3(int nb) { return (int64_t)nb * (nb + 1) * (nb + 2) / 6; }
__host__ __device__ __forceinline__ int64_t gs_ncfg4(int nb) { return (int64_t)nb * (nb - 1) * (nb - 2) / 6; }

// Multiplicative hash of a node id into a table of 2^(32 - shift) slots.
__device__ __forceinline__ uint32_t gs_hash(int32_t key, int shift)
{
    return ((uint32_t)key * 0x9E3779B1u) >> shift;
}

// Position of the n-th set bit (n from 0) of x, which has more than n set
// bits: a binary search on the popcounts of the lower halves.
__device__ __forceinline__ int gs_nth_bit(unsigned x, int n)
{
    int pos = 0, c;
    c = __popc(x & 0xffffu);
    if (n >= c) { n -= c; pos += 16; x >>= 16; }
    c = __popc(x & 0xffu);
    if (n >= c) { n -= c; pos += 8; x >>= 8; }
    c = __popc(x & 0xfu);
    if (n >= c) { n -= c; pos += 4; x >>= 4; }
    c = __popc(x & 0x3u);
    if (n >= c) { n -= c; pos += 2; x >>= 2; }
    return pos + (n >= (int)(x & 1u));
}

__device__ __forceinline__ unsigned gs_lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// v added to the 128-bit two's-complement integer (low word p[0], high word
// p[1]) in global or shared memory: the low word takes v with a 64-bit atomic,
// the high word the carry out of it plus the sign extension of v.
__device__ __forceinline__ void gs_add128(unsigned long long *p, long long v)
{
    const unsigned long long u = (unsigned long long)v;
    const unsigned long long old = atomicAdd(p, u);
    const unsigned long long hi = (old + u < old ? 1ull : 0ull) + (v < 0 ? ~0ull : 0ull);
    if (hi) atomicAdd(p + 1, hi);
}

// The 128-bit value (lo, hi) added to the 128-bit integer at p.
__device__ __forceinline__ void gs_add128w(unsigned long long *p, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long old = atomicAdd(p, lo);
    const unsigned long long h = hi + (old + lo < old ? 1ull : 0ull);
    if (h) atomicAdd(p + 1, h);
}

// v added to the 128-bit two's-complement integer held in four 32-bit words
// q[0..3], least significant first, with 32-bit atomics: each word takes its
// part of v plus the carry out of the word below (computed from the value the
// atomic returned); words whose addend is zero are skipped. The carries of
// concurrent adds each count once, so the sum of all adds is exact mod 2^128.
__device__ __forceinline__ void gs_add128_u32(unsigned *q, long long v)
{
    const unsigned long long u = (unsigned long long)v;
    const unsigned ext = v < 0 ? 0xffffffffu : 0u;
    const unsigned part[4] = { (unsigned)u, (unsigned)(u >> 32), ext, ext };
    unsigned carry = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const unsigned long long add = (unsigned long long)part[k] + carry;   // <= 2^32
        const unsigned lo = (unsigned)add;
        carry = (unsigned)(add >> 32);                                      // 1 only when lo == 0
        if (lo) {
            const unsigned old = atomicAdd(q + k, lo);
            carry = (old + lo < old) ? 1u : 0u;
        }
    }
}
