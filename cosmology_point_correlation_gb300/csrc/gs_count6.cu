// gs_count6.cu -- six-edge-bin 4pCF with parity channels (GRAMSCI v2, §II.2:
// tetrahedra whose six pairs are all neighbours; §III.2, Eq.(3): handedness;
// §V.2: tetrahedron configurations, 276 of them for 4 radial bins).
//
// Every tetrahedron {i, j1, j2, j3} with i < j1 < j2 < j3 (internal order) is
// found once, at hub i, from its forward row F = {j in N(i) : j > i}:
//   1. F is staged in shared memory (ids; spoke vectors x_j - x_i with the
//      hub bin, one int4 per spoke) with a hash table id -> position;
//   2. warps walk the forward part of each spoke's row N(j) and, for every
//      entry that is also in F, set bit (s, t) of an adjacency bit-matrix and
//      store the spoke-spoke bin in a byte matrix;
//   3. cliques (s1 < s2 < s3) come from the AND of two bit rows; the six bins
//      (b_ij1, b_ij2, b_ij3, b_j1j2, b_j1j3, b_j2j3) index a per-graph table
//      holding the configuration and the parity of a vertex ordering that
//      turns this labelling into the configuration's smallest tuple (0 when
//      orderings of both parities do: an achiral configuration); the odd
//      channel adds that parity times sign(det[r_j1; r_j2; r_j3]).
// Hubs with up to 128 forward neighbours run in a 128-slot shared-memory
// kernel (four blocks per SM), up to C6_M in a 256-slot one, larger hubs in a
// kernel with a global workspace slice and 1024-thread blocks; all keep their
// histograms in shared memory. A warp takes a row s1 and its lanes one pair
// (s1, s2) each; per word of the bit rows the lanes either walk their own
// pairs' tetrahedra or, when those are uneven, deal them out 32 at a time, as
// the parity kernel does. In the weighted mode (several atomics per
// tetrahedron) warps take rows s1 from a counter and deal sooner.
//
// Windowed graphs (§III.5.3): tiles (hub window, spoke windows c1 <= c2) as
// for the parity count; only tetrahedra whose two lowest spokes lie in c1 and
// c2 are counted in a tile, so each is counted once.
//
// Weighted counts (§II.1 signed weights): each tetrahedron adds
// W = w_i w_j1 w_j2 w_j3 (|W| <= 2^60) to the even channel and sign x W to
// the odd one, into exact 128-bit sums: per block in shared memory as four
// 32-bit words (gs_add128_u32) when the configurations fit, else straight
// into the global (low, high) pairs.

#include <algorithm>
#include <array>
#include <type_traits>
#include <vector>

#include "gs_internal.cuh"

constexpr int C6_THREADS = 256;
constexpr int C6_LARGE_THREADS = 1024;       // hubs above C6_M: few and large, a wide block each
constexpr int C6_M = 256;                   // forward degree kept in shared memory
constexpr int C6_M_SMALL = 128;             // hubs up to this degree run in a lighter kernel (more blocks per SM)
constexpr int C6_SMEM_HIST_MAX = 4096;
constexpr int C6_SMEM_W_MAX = 2500;         // weighted: configurations with shared 128-bit sums (nb <= 6)
constexpr int C6_EMPTY = -1;
constexpr int C6_MAX_BINS = 10;             // the tuple table holds nb^6 entries
constexpr int64_t C6_SMALL_R = 32768;       // r_max (lattice units) below which cross products fit in int32
// Unweighted shared-memory histogram: three u32 counters per configuration,
// the tetrahedra of negative, zero and positive signed volume, so that a
// tetrahedron is one add (even = their sum, odd = positive - negative).
constexpr int C6_HIST_WORDS = 3;

struct C6Args {
    const int4 *pts;
    const int64_t *row_ptr;
    const int32_t *fwd;
    const int32_t *nbr;
    const uint8_t *bin;
    const int32_t *cfg6;          // [nb^6] (configuration << 2) | (orientation parity + 1)
    int64_t hub_begin, hub_end;
    int box, periodic, nb, ncfg;
    unsigned long long *even;
    long long *odd;
    unsigned long long *cursor;
    int f_lo;                     // small paths: hubs with f_lo < f <= M
    int big_m;                    // large path: forward degree the slices hold
    char *scratch;
    size_t scratch_stride;
    // weighted counts: weights in internal order; 128-bit sums [ncfg][2]
    const int16_t *w;
    unsigned long long *weven, *wodd;
    // windowed graphs: hub rows at hnbr / hbin (edge e at e - hoff); spoke rows
    // of ids in [a_lo, a_hi) at anbr / abin - aoff, of ids in [b_lo, b_hi) at
    // bnbr / bbin - boff (the same window when a_lo == b_lo)
    const int32_t *hnbr, *anbr, *bnbr;
    const uint8_t *hbin, *abin, *bbin;
    int64_t hoff, aoff, boff;
    int32_t a_lo, a_hi, b_lo, b_hi;
};

// First position of a sorted row whose id is >= key.
__device__ __forceinline__ int c6_lower(const int32_t *row, int m, int32_t key)
{
    int lo = 0, hi = m;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (row[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

struct C6Space {
    int32_t *key;      // hash table
    int32_t *pos;
    int32_t *row;      // [f] ids
    uint8_t *hb;       // [f] hub bins
    int4 *v;           // [f] spoke vector x_s - x_i and hub bin (.w)
    unsigned *bits;    // [f][W]
    uint8_t *sbin;     // [f][f] spoke-spoke bins (valid where the bit is set)
    int16_t *ww;       // [f] spoke weights (weighted counts)
    int *next;         // shared counter handing out the rows s1 of the tetrahedron search
};

// SMALLR: r_max below C6_SMALL_R lattice units, so a spoke-pair cross product
// fits in int32 (components |r| <= 32767: |y1 z2 - z1 y2| < 2^31) and the
// volume is three 32 x 32 -> 64-bit products instead of 64-bit arithmetic.
template <int NT, bool SMEM_HIST, bool WEIGHTED, bool WINDOWED, bool SMALLR = false>
__device__ __forceinline__ void c6_hub(const C6Args &a, const C6Space &w, long long i, int64_t f0, int f,
                                       int tlog, unsigned *s_cnt, unsigned *s_w128)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t *F = WINDOWED ? a.hnbr + (f0 - a.hoff) : a.nbr + f0;       // forward row and its bins
    const uint8_t *FB = WINDOWED ? a.hbin + (f0 - a.hoff) : a.bin + f0;
    // spokes walked: positions [pa0, pa1) (window c1) and [pb0, pb1) (c2 when
    // it differs); tetrahedra take s1 in [pa0, pa1), s2 in [q2_lo, q2_hi)
    int pa0 = 0, pa1 = f, pb0 = 0, pb1 = 0, q2_lo = 0, q2_hi = f;
    if (WINDOWED) {                                            // the same values in every thread
        pa0 = c6_lower(F, f, a.a_lo);
        pa1 = c6_lower(F, f, a.a_hi);
        q2_lo = pa0;
        q2_hi = pa1;
        if (a.b_lo != a.a_lo) {
            pb0 = q2_lo = c6_lower(F, f, a.b_lo);
            pb1 = q2_hi = c6_lower(F, f, a.b_hi);
        }
        if (pa0 >= pa1 || q2_lo >= q2_hi || pa0 >= q2_hi - 1) return;   // nothing in this tile
    }
    const int W = (f + 31) >> 5;
    const int tsize = 1 << tlog, shift = 32 - tlog, mask = tsize - 1;
    const int4 P = a.pts[i];
    const int nb = a.nb;

    for (int t = threadIdx.x; t < f; t += NT) {
        const int32_t k = F[t];
        w.row[t] = k;
        const int b = FB[t];
        w.hb[t] = (uint8_t)b;
        const int4 Q = a.pts[k];
        w.v[t] = make_int4(gs_delta(P.x, Q.x, a.box, a.periodic), gs_delta(P.y, Q.y, a.box, a.periodic),
                           gs_delta(P.z, Q.z, a.box, a.periodic), b);
        if (WEIGHTED) w.ww[t] = a.w[k];
        uint32_t h = gs_hash(k, shift);
        while (atomicCAS(&w.key[h], C6_EMPTY, k) != C6_EMPTY) h = (h + 1) & mask;
        w.pos[h] = t;
    }
    for (int t = threadIdx.x; t < f * W; t += NT) w.bits[t] = 0u;
    __syncthreads();

    if (threadIdx.x == 0) *w.next = pa0;                       // read after the barrier below
    const int32_t kmax = w.row[f - 1];
    const int na = pa1 - pa0, nab = na + (pb1 - pb0);
    for (int u = warp; u < nab; u += (NT / 32)) {
        const bool in_a = u < na;
        const int s = in_a ? pa0 + u : pb0 + (u - na);
        if (s >= f - 1) continue;                              // no position above the last
        const int32_t *SN = WINDOWED ? (in_a ? a.anbr : a.bnbr) : a.nbr;
        const uint8_t *SB = WINDOWED ? (in_a ? a.abin : a.bbin) : a.bin;
        const int64_t soff = WINDOWED ? (in_a ? a.aoff : a.boff) : 0;
        const int32_t j = w.row[s];
        const int64_t pe = a.row_ptr[j + 1];
        for (int64_t p = a.row_ptr[j] + a.fwd[j]; p < pe; p += 32) {
            const int64_t q = p + lane;
            const int32_t k = q < pe ? SN[q - soff] : 0x7fffffff;
            if (k <= kmax) {
                uint32_t h = gs_hash(k, shift);
                int32_t key;
                while ((key = w.key[h]) != k && key != C6_EMPTY) h = (h + 1) & mask;
                if (key == k) {
                    const int t = w.pos[h];
                    atomicOr(&w.bits[(size_t)s * W + (t >> 5)], 1u << (t & 31));
                    w.sbin[(size_t)s * f + t] = SB[q - soff];
                }
            }
            if (__shfl_sync(0xffffffffu, k, 31) > kmax) break;
        }
    }
    __syncthreads();

    const long long wi = WEIGHTED ? (long long)a.w[i] : 0;
    const int s1_end = min(pa1, f - 2), s2_end = min(q2_hi, f - 1);
    // A warp per s1, its lanes over 32 candidate spokes s2 at a time, one pair
    // (s1, s2) per lane with its cross product in registers. For each word of
    // the bit rows: when the lanes' tetrahedra are even enough (the largest
    // count at most C6_WALK_ROUNDS times the rounds that dealing them out would
    // take) each lane walks the common bits of its own pair; else the counts are
    // prefix-summed and the tetrahedra handed out 32 at a time with the owner's
    // pair data, so that all lanes stay busy however unevenly the tetrahedra are
    // spread over the pairs. Dealing costs a prefix sum, an owner search and the
    // pair's shuffles per round; a weighted tetrahedron costs two 128-bit
    // atomics, so dealing pays off sooner there.
    constexpr int C6_WALK_ROUNDS = WEIGHTED ? 2 : 3;
    using CT = typename std::conditional<SMALLR, int, long long>::type;
    struct Pair {
        int s2, b02, b12;
        CT cx, cy, cz;
        long long w12;
    };
    // rows s1: weighted, from the shared counter (low rows, with the most
    // candidates, first); unweighted, where rows are cheap, strided by warp
    auto next_row = [&](int prev) {
        if (!WEIGHTED) return prev < 0 ? pa0 + warp : prev + (NT / 32);
        int r = 0;
        if (lane == 0) r = atomicAdd(w.next, 1);
        return __shfl_sync(0xffffffffu, r, 0);
    };
    for (int s1 = next_row(-1); s1 < s1_end; s1 = next_row(s1)) {
        const unsigned *row1 = w.bits + (size_t)s1 * W;
        const int4 r1 = w.v[s1];
        const int b01 = r1.w;
        const CT x1 = r1.x, y1 = r1.y, z1 = r1.z;
        const long long w1 = WEIGHTED ? wi * w.ww[s1] : 0;
        auto make_pair = [&](int s2) {
            Pair p;
            p.s2 = s2;
            const int4 r2 = w.v[s2];
            p.b02 = r2.w;
            p.b12 = w.sbin[(size_t)s1 * f + s2];
            const CT x2 = r2.x, y2 = r2.y, z2 = r2.z;
            p.cx = y1 * z2 - z1 * y2;
            p.cy = z1 * x2 - x1 * z2;
            p.cz = x1 * y2 - y1 * x2;
            p.w12 = WEIGHTED ? w1 * w.ww[s2] : 0;                          // |.| <= 2^45
            return p;
        };
        // one tetrahedron (i, s1, s2, s3)
        auto tetra = [&](const Pair &p, int s3) {
            const int4 r3 = w.v[s3];
            const int b03 = r3.w;
            const int b13 = w.sbin[(size_t)s1 * f + s3], b23 = w.sbin[(size_t)p.s2 * f + s3];
            const int pk = ((((b01 * nb + p.b02) * nb + b03) * nb + p.b12) * nb + b13) * nb + b23;
            const int v = __ldg(a.cfg6 + pk);
            const int ci = v >> 2, par = (v & 3) - 1;
            const long long d = (long long)p.cx * r3.x + (long long)p.cy * r3.y + (long long)p.cz * r3.z;
            const int sg = par * ((d > 0) - (d < 0));
            if (WEIGHTED) {
                const long long W4 = p.w12 * w.ww[s3];                    // |.| <= 2^60
                if (SMEM_HIST) {
                    gs_add128_u32(s_w128 + 8 * ci, W4);
                    if (sg) gs_add128_u32(s_w128 + 8 * ci + 4, sg * W4);
                } else {
                    gs_add128(a.weven + 2 * ci, W4);
                    if (sg) gs_add128(a.wodd + 2 * ci, sg * W4);
                }
            } else if (SMEM_HIST) {
                atomicAdd(&s_cnt[(sg + 1) * a.ncfg + ci], 1u);       // the counter of the volume's sign
            } else {
                atomicAdd(a.even + ci, 1ull);
                if (sg) atomicAdd((unsigned long long *)(a.odd + ci), (unsigned long long)(long long)sg);
            }
        };
        for (int c2 = max(s1 + 1, q2_lo); c2 < s2_end; c2 += 32) {        // warp-uniform
            const int s2 = c2 + lane;
            const bool valid = s2 < s2_end && ((row1[s2 >> 5] >> (s2 & 31)) & 1u);
            if (!__any_sync(0xffffffffu, valid)) continue;
            const unsigned *row2 = w.bits + (size_t)(valid ? s2 : s1) * W;
            const Pair p = make_pair(valid ? s2 : s1);                 // an idle lane's pair is never used
            for (int wd = c2 >> 5; wd < W; ++wd) {
                unsigned common = 0u;
                if (valid && wd >= (s2 >> 5)) {
                    common = row1[wd] & row2[wd];
                    if (wd == (s2 >> 5)) common &= ~((2u << (s2 & 31)) - 1u);   // s3 > s2
                }
                const int cnt = __popc(common);
                const int all = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
                if (all == 0) continue;                            // no tetrahedron in this word
                const int most = (int)__reduce_max_sync(0xffffffffu, (unsigned)cnt);
                if (most <= C6_WALK_ROUNDS * ((all + 31) >> 5)) {
                    for (unsigned cm = common; cm; cm &= cm - 1) tetra(p, (wd << 5) + __ffs(cm) - 1);
                    continue;
                }
                int inc = cnt;                                     // inclusive prefix over lanes
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                for (int k = 0; k < all; k += 32) {
                    const int q = k + lane;
                    int owner = 0;                                 // first lane whose prefix exceeds q
#pragma unroll
                    for (int step = 16; step > 0; step >>= 1)
                        if (__shfl_sync(0xffffffffu, inc, owner + step - 1) <= q) owner += step;
                    const unsigned cm = __shfl_sync(0xffffffffu, common, owner);
                    const int first = __shfl_sync(0xffffffffu, inc - cnt, owner);
                    Pair o;                                        // the owner's pair
                    o.s2 = __shfl_sync(0xffffffffu, p.s2, owner);
                    o.b02 = __shfl_sync(0xffffffffu, p.b02, owner);
                    o.b12 = __shfl_sync(0xffffffffu, p.b12, owner);
                    o.cx = __shfl_sync(0xffffffffu, p.cx, owner);
                    o.cy = __shfl_sync(0xffffffffu, p.cy, owner);
                    o.cz = __shfl_sync(0xffffffffu, p.cz, owner);
                    o.w12 = WEIGHTED ? __shfl_sync(0xffffffffu, p.w12, owner) : 0;
                    if (q < all) tetra(o, (wd << 5) + gs_nth_bit(cm, q - first));
                }
            }
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < tsize; t += NT) w.key[t] = C6_EMPTY;
}

// Add the unweighted shared counters into the caller's histograms (even =
// negative + zero + positive volume, odd = positive - negative) and clear them.
template <int NT>
__device__ __forceinline__ void c6_flush(unsigned *sc, int ncfg, unsigned long long *ge, long long *go)
{
    for (int t = threadIdx.x; t < ncfg; t += NT) {
        const unsigned neg = sc[t], zero = sc[ncfg + t], pos = sc[2 * ncfg + t];
        const unsigned long long e = (unsigned long long)neg + zero + pos;
        const long long o = (long long)pos - (long long)neg;
        if (e) atomicAdd(ge + t, e);
        if (o) atomicAdd((unsigned long long *)(go + t), (unsigned long long)o);
        sc[t] = 0u;
        sc[ncfg + t] = 0u;
        sc[2 * ncfg + t] = 0u;
    }
}

// Hubs with max(3, a.f_lo + 1) .. M forward neighbours, workspace in shared
// memory. M = 128 keeps the per-block footprint near 25 KB (about four
// resident blocks per SM); M = 256 takes the rarer hubs up to C6_M.
template <int M, bool SMEM_HIST, bool WEIGHTED, bool WINDOWED, bool SMALLR = false>
__global__ void __launch_bounds__(C6_THREADS, M <= C6_M_SMALL ? 4 : 2)
k_count6_small(C6Args a)
{
    // dynamic: bits [M*M/32], sbin [M*M], then (SMEM_HIST) the counters
    // [3][ncfg], or (WEIGHTED) the 128-bit sums [ncfg][2][4] u32
    extern __shared__ unsigned s_dyn[];
    __shared__ int32_t s_key[2 * M];
    __shared__ int32_t s_pos[2 * M];
    __shared__ int32_t s_row[M];
    __shared__ uint8_t s_hb[M];
    __shared__ int4 s_v[M];
    __shared__ int16_t s_ww[M];
    __shared__ long long s_hub;
    __shared__ int s_next;
    __shared__ unsigned long long s_pending;

    unsigned *s_bits = s_dyn;
    uint8_t *s_sbin = (uint8_t *)(s_bits + M * (M / 32));
    unsigned *s_cnt = (unsigned *)(s_sbin + M * M);
    unsigned *s_w128 = s_cnt;
    if (SMEM_HIST && WEIGHTED)
        for (int t = threadIdx.x; t < 8 * a.ncfg; t += C6_THREADS) s_w128[t] = 0;
    else if (SMEM_HIST)
        for (int t = threadIdx.x; t < C6_HIST_WORDS * a.ncfg; t += C6_THREADS) s_cnt[t] = 0u;
    for (int t = threadIdx.x; t < 2 * M; t += C6_THREADS) s_key[t] = C6_EMPTY;
    if (threadIdx.x == 0) s_pending = 0;
    C6Space w{ s_key, s_pos, s_row, s_hb, s_v, s_bits, s_sbin, s_ww, &s_next };

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        const long long i = s_hub;
        if (i >= a.hub_end) break;
        const int64_t f0 = a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        if (f < 3 || f <= a.f_lo || f > M) continue;
        if (SMEM_HIST && !WEIGHTED) {
            const unsigned long long bound = (unsigned long long)f * (f - 1) * (f - 2) / 6;
            if (s_pending + bound > 0x7fffffffull) {
                c6_flush<C6_THREADS>(s_cnt, a.ncfg, a.even, a.odd);
                __syncthreads();
                if (threadIdx.x == 0) s_pending = 0;
            }
            __syncthreads();
            if (threadIdx.x == 0) s_pending += bound;
        }
        int tlog = 4;
        while ((1 << tlog) < 2 * f) ++tlog;
        c6_hub<C6_THREADS, SMEM_HIST, WEIGHTED, WINDOWED, SMALLR>(a, w, i, f0, f, tlog, s_cnt, s_w128);
    }
    if (SMEM_HIST && WEIGHTED) {
        __syncthreads();
        for (int t = threadIdx.x; t < 2 * a.ncfg; t += C6_THREADS) {
            const unsigned *q = s_w128 + 4 * t;
            const unsigned long long lo = q[0] | ((unsigned long long)q[1] << 32);
            const unsigned long long hi = q[2] | ((unsigned long long)q[3] << 32);
            unsigned long long *dst = (t & 1) ? a.wodd + 2 * (t >> 1) : a.weven + 2 * (t >> 1);
            if (lo | hi) gs_add128w(dst, lo, hi);
        }
    } else if (SMEM_HIST) {
        __syncthreads();
        c6_flush<C6_THREADS>(s_cnt, a.ncfg, a.even, a.odd);
    }
}

// Hubs with more than C6_M forward neighbours: workspace in a global slice,
// one wide block per hub; the histograms stay in shared memory as in the
// small kernels (global atomics on a few hundred configurations would
// serialise in L2).
template <bool SMEM_HIST, bool WEIGHTED, bool WINDOWED>
__global__ void __launch_bounds__(C6_LARGE_THREADS, 1)
k_count6_large(C6Args a)
{
    // dynamic (SMEM_HIST): the counters [3][ncfg], or (WEIGHTED) the 128-bit sums [ncfg][2][4] u32
    extern __shared__ unsigned s_dyn[];
    __shared__ long long s_hub;
    __shared__ int s_next;
    __shared__ unsigned long long s_pending;
    unsigned *s_cnt = s_dyn;
    unsigned *s_w128 = s_dyn;
    if (SMEM_HIST && WEIGHTED)
        for (int t = threadIdx.x; t < 8 * a.ncfg; t += C6_LARGE_THREADS) s_w128[t] = 0;
    else if (SMEM_HIST)
        for (int t = threadIdx.x; t < C6_HIST_WORDS * a.ncfg; t += C6_LARGE_THREADS) s_cnt[t] = 0u;
    if (threadIdx.x == 0) s_pending = 0;
    const int M = a.big_m;
    int tlog = 4;
    while ((1 << tlog) < 2 * M) ++tlog;
    const int WM = (M + 31) >> 5;
    char *base = a.scratch + (size_t)blockIdx.x * a.scratch_stride;
    C6Space w;
    w.v = (int4 *)base;                                   // slices start 256-byte aligned
    w.key = (int32_t *)(w.v + M);
    w.pos = w.key + (1 << tlog);
    w.row = w.pos + (1 << tlog);
    w.bits = (unsigned *)(w.row + M);
    w.hb = (uint8_t *)(w.bits + (size_t)M * WM);
    w.sbin = w.hb + M;
    w.ww = (int16_t *)(w.sbin + (size_t)M * M);          // M + M*M is even: 2-byte aligned
    w.next = &s_next;
    for (int t = threadIdx.x; t < (1 << tlog); t += C6_LARGE_THREADS) w.key[t] = C6_EMPTY;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        const long long i = s_hub;
        if (i >= a.hub_end) break;
        const int64_t f0 = a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        if (f <= C6_M) continue;
        int tl = 4;
        while ((1 << tl) < 2 * f) ++tl;
        const unsigned long long bound = (unsigned long long)f * (f - 1) * (f - 2) / 6;
        if (SMEM_HIST && !WEIGHTED && bound > 0x7fffffffull) {
            // one hub could overflow the 32-bit shared counters: global atomics
            c6_hub<C6_LARGE_THREADS, false, false, WINDOWED>(a, w, i, f0, f, tl, nullptr, nullptr);
            continue;
        }
        if (SMEM_HIST && !WEIGHTED) {
            if (s_pending + bound > 0x7fffffffull) {
                c6_flush<C6_LARGE_THREADS>(s_cnt, a.ncfg, a.even, a.odd);
                __syncthreads();
                if (threadIdx.x == 0) s_pending = 0;
            }
            __syncthreads();
            if (threadIdx.x == 0) s_pending += bound;
        }
        c6_hub<C6_LARGE_THREADS, SMEM_HIST, WEIGHTED, WINDOWED>(a, w, i, f0, f, tl, s_cnt, s_w128);
    }
    if (SMEM_HIST && WEIGHTED) {
        __syncthreads();
        for (int t = threadIdx.x; t < 2 * a.ncfg; t += C6_LARGE_THREADS) {
            const unsigned *q = s_w128 + 4 * t;
            const unsigned long long lo = q[0] | ((unsigned long long)q[1] << 32);
            const unsigned long long hi = q[2] | ((unsigned long long)q[3] << 32);
            unsigned long long *dst = (t & 1) ? a.wodd + 2 * (t >> 1) : a.weven + 2 * (t >> 1);
            if (lo | hi) gs_add128w(dst, lo, hi);
        }
    } else if (SMEM_HIST) {
        __syncthreads();
        c6_flush<C6_LARGE_THREADS>(s_cnt, a.ncfg, a.even, a.odd);
    }
}

static size_t c6_large_stride(int M)
{
    int tlog = 4;
    while ((1 << tlog) < 2 * M) ++tlog;
    const size_t WM = (size_t)(M + 31) / 32;
    const size_t bytes = 16 * (size_t)M + sizeof(int32_t) * (2 * ((size_t)1 << tlog) + (size_t)M) +
                         sizeof(unsigned) * M * WM + M + (size_t)M * M + sizeof(int16_t) * M;
    return (bytes + 255) & ~(size_t)255;
}

// Host table over all nb^6 bin tuples t = (b01, b02, b03, b12, b13, b23) of a
// labelled tetrahedron: the configuration (rank of the smallest relabelling
// among all smallest tuples, in lexicographic order) and the parity of a
// relabelling reaching it, 0 if relabellings of both parities do.
static std::vector<int32_t> c6_table(int nb, int *ncfg_out)
{
    // vertex permutations and the edge permutation each induces: relabelled
    // tuple u[e] = t[edge(perm[a], perm[b])] for edge e = (a, b)
    static const int ea[6] = { 0, 0, 0, 1, 1, 2 }, eb[6] = { 1, 2, 3, 2, 3, 3 };
    int eid[4][4];
    for (int e = 0; e < 6; ++e) eid[ea[e]][eb[e]] = eid[eb[e]][ea[e]] = e;
    std::vector<std::array<int, 6>> emap;
    std::vector<int> par;
    int p[4] = { 0, 1, 2, 3 };
    std::sort(p, p + 4);
    do {
        std::array<int, 6> m;
        for (int e = 0; e < 6; ++e) m[e] = eid[p[ea[e]]][p[eb[e]]];
        emap.push_back(m);
        int inv = 0;
        for (int x = 0; x < 4; ++x)
            for (int y = x + 1; y < 4; ++y) inv += p[x] > p[y];
        par.push_back(inv & 1);
    } while (std::next_permutation(p, p + 4));

    size_t nt = 1;
    for (int k = 0; k < 6; ++k) nt *= (size_t)nb;
    std::vector<int32_t> canon(nt), orient(nt);
    auto pack = [nb](const int *u) {
        size_t q = 0;
        for (int k = 0; k < 6; ++k) q = q * (size_t)nb + (size_t)u[k];
        return q;
    };
    int t[6];
    for (size_t q = 0; q < nt; ++q) {
        size_t r = q;
        for (int k = 5; k >= 0; --k) {
            t[k] = (int)(r % (size_t)nb);
            r /= (size_t)nb;
        }
        size_t best = (size_t)-1;
        bool ev = false, od = false;
        for (size_t g = 0; g < emap.size(); ++g) {
            int u[6];
            for (int e = 0; e < 6; ++e) u[e] = t[emap[g][e]];
            const size_t pu = pack(u);           // packed order = lexicographic order
            if (pu < best) {
                best = pu;
                ev = !par[g];
                od = par[g];
            } else if (pu == best) {
                (par[g] ? od : ev) = true;
            }
        }
        canon[q] = (int32_t)best;
        orient[q] = (ev && od) ? 0 : (ev ? 1 : -1);
    }
    // configuration numbers: canonical tuples in increasing packed order
    std::vector<int32_t> rank(nt, -1);
    int n = 0;
    for (size_t q = 0; q < nt; ++q)
        if ((size_t)canon[q] == q) rank[q] = n++;
    std::vector<int32_t> out(nt);
    for (size_t q = 0; q < nt; ++q) out[q] = (rank[canon[q]] << 2) | (orient[q] + 1);
    *ncfg_out = n;
    return out;
}

static gs_status c6_prepare(gs_graph_t g)
{
    if (g->cfg6) return GS_OK;
    int n = 0;
    std::vector<int32_t> t = c6_table(g->nb, &n);
    int32_t *d = nullptr;
    GS_TRY_CUDA(gs_malloc(&d, sizeof(int32_t) * t.size()));
    cudaError_t e = cudaMemcpy(d, t.data(), sizeof(int32_t) * t.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(d);
        return gs_set_error(GS_ERR_CUDA, "copy of the configuration table failed: %s", cudaGetErrorString(e));
    }
    g->cfg6 = d;
    g->ncfg6 = n;
    return GS_OK;
}

extern "C" gs_status gs_config_tuple_4pcf6(int nbins, int64_t config, int32_t *tuple_host)
{
    GS_ENTRY();
    if (nbins < 1 || nbins > C6_MAX_BINS || !tuple_host) return gs_set_error(GS_ERR_ARG, "bad argument");
    int n = 0;
    static thread_local int cached_nb = 0;
    static thread_local std::vector<int64_t> canon_packed;
    if (cached_nb != nbins) {
        std::vector<int32_t> t = c6_table(nbins, &n);
        canon_packed.assign((size_t)n, 0);
        size_t nt = t.size();
        std::vector<int32_t> first(n, -1);
        // the smallest packed tuple of each configuration is the canonical one
        for (size_t q = 0; q < nt; ++q) {
            const int c = t[q] >> 2;
            if (first[c] < 0) {
                first[c] = (int32_t)q;
                canon_packed[c] = (int64_t)q;
            }
        }
        cached_nb = nbins;
    }
    if (config < 0 || config >= (int64_t)canon_packed.size()) return gs_set_error(GS_ERR_ARG, "configuration out of range");
    int64_t q = canon_packed[config];
    for (int k = 5; k >= 0; --k) {
        tuple_host[k] = (int32_t)(q % nbins);
        q /= nbins;
    }
    return GS_OK;
}

extern "C" int64_t gs_config_count_4pcf6(int nbins)
{
    if (nbins < 1 || nbins > C6_MAX_BINS) return -1;
    const int64_t b = nbins;
    return (b * b * b * b * b * b + 9 * b * b * b * b + 14 * b * b) / 24;
}

// Blocks of the large-hub kernel for a launch over `hubs` hubs (its
// workspace is capped at 2 GiB), and the workspace they need (0 when no hub
// has more than C6_M forward neighbours).
static int c6_large_blocks(gs_graph_t g, int64_t hubs)
{
    const size_t budget = (size_t)2 << 30;
    return (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>((int64_t)gs_sm_count() * 2, hubs),
                                                       (int64_t)(budget / c6_large_stride(g->max_forward))));
}

static size_t c6_scratch_bytes(gs_graph_t g, int64_t hubs)
{
    if (g->max_forward <= C6_M || hubs <= 0 || g->n_edges == 0) return 0;
    return c6_large_stride(g->max_forward) * (size_t)c6_large_blocks(g, hubs);
}

// Launch the small-hub and large-hub kernels over [hub_begin, hub_end) of a
// prepared argument block (outputs already cleared).
static gs_status c6_launch(gs_graph_t g, C6Args a, bool windowed, cudaStream_t st)
{
    const int64_t hubs = a.hub_end - a.hub_begin;
    const int sms = gs_sm_count();
    const int ncfg = a.ncfg;
    const bool weighted = a.w != nullptr;
    const bool smem = weighted ? ncfg <= C6_SMEM_W_MAX : ncfg <= C6_SMEM_HIST_MAX;
    const size_t acc = weighted ? 32 * (size_t)ncfg : sizeof(unsigned) * C6_HIST_WORDS * (size_t)ncfg;
    const bool small_r = g->edges[g->nb] < C6_SMALL_R;    // int32 cross products (the resident shared-memory kernels)
    // the two shared-memory kernels: hubs of forward degree 3..128, then 129..256
    for (int pass = 0; pass < 2; ++pass) {
        const int m = pass ? C6_M : C6_M_SMALL;
        if (pass && g->max_forward <= C6_M_SMALL) break;
        const size_t dyn = sizeof(unsigned) * m * (m / 32) + (size_t)m * m + (smem ? acc : 0);
        using K = decltype(&k_count6_small<C6_M, true, true, true>);
        auto pick = [&](auto mtag) -> K {
            constexpr int MM = decltype(mtag)::value;
            if (windowed)
                return weighted ? (smem ? k_count6_small<MM, true, true, true> : k_count6_small<MM, false, true, true>)
                                : (smem ? k_count6_small<MM, true, false, true> : k_count6_small<MM, false, false, true>);
            if (smem && small_r)
                return weighted ? k_count6_small<MM, true, true, false, true> : k_count6_small<MM, true, false, false, true>;
            return weighted ? (smem ? k_count6_small<MM, true, true, false> : k_count6_small<MM, false, true, false>)
                            : (smem ? k_count6_small<MM, true, false, false> : k_count6_small<MM, false, false, false>);
        };
        const K kern = pass ? pick(std::integral_constant<int, C6_M>()) : pick(std::integral_constant<int, C6_M_SMALL>());
        int per_sm = 0;
        GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
        GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C6_THREADS, dyn));
        if (per_sm < 1) return gs_set_error(GS_ERR_CAPACITY, "4pCF workspace of %zu bytes does not fit in shared memory", dyn);
        GS_TRY_CUDA(cudaMemsetAsync(a.cursor, 0, sizeof(unsigned long long), st));
        a.f_lo = pass ? C6_M_SMALL : 0;
        kern<<<(int)std::min<int64_t>((int64_t)sms * per_sm, hubs), C6_THREADS, dyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }

    const int M = g->max_forward;              // bounds the large path's slices
    if (M > C6_M) {
        // a.scratch: the caller's workspace of c6_scratch_bytes(g, hubs) bytes
        const size_t stride = c6_large_stride(M);
        const int gl = c6_large_blocks(g, hubs);
        GS_TRY_CUDA(cudaMemsetAsync(a.cursor, 0, sizeof(unsigned long long), st));
        a.big_m = M;
        a.scratch_stride = stride;
        const size_t bdyn = smem ? acc : 0;
        decltype(&k_count6_large<true, true, true>) big;
        if (windowed)
            big = weighted ? (smem ? k_count6_large<true, true, true> : k_count6_large<false, true, true>)
                           : (smem ? k_count6_large<true, false, true> : k_count6_large<false, false, true>);
        else
            big = weighted ? (smem ? k_count6_large<true, true, false> : k_count6_large<false, true, false>)
                           : (smem ? k_count6_large<true, false, false> : k_count6_large<false, false, false>);
        GS_TRY_CUDA(cudaFuncSetAttribute(big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bdyn));
        big<<<gl, C6_LARGE_THREADS, bdyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }
    return GS_OK;
}

// The hubs [hub_begin, hub_end): one pass on a device-resident graph; on a
// windowed graph one pass per tile (hub window h, spoke windows c1 <= c2 that
// hold forward neighbours of window h), the three windows staged.
static gs_status c6_run(gs_graph_t g, C6Args a, int64_t hub_begin, int64_t hub_end, cudaStream_t st)
{
    if (!g->n_win) {
        a.hub_begin = hub_begin;
        a.hub_end = hub_end;
        return c6_launch(g, a, false, st);
    }
    int held[GS_SLOTS];
    int64_t off[GS_SLOTS] = {};
    for (int k = 0; k < GS_SLOTS; ++k) held[k] = -1;
    for (int h = 0; h < g->n_win; ++h) {
        const int64_t b0 = std::max(hub_begin, g->win_row[h]), b1 = std::min(hub_end, g->win_row[h + 1]);
        if (b0 >= b1 || g->win_e0[h + 1] == g->win_e0[h]) continue;
        std::vector<int> fw;
        for (int c = h; c < g->n_win; ++c)
            if (g->win_e0[c + 1] > g->win_e0[c] && g->win_pair[(size_t)h * g->n_win + c]) fw.push_back(c);
        for (size_t x = 0; x < fw.size(); ++x)
            for (size_t y = x; y < fw.size(); ++y) {
                const int need[3] = { h, fw[x], fw[y] };
                int slot[3];
                gs_status s = gs_stage_set(g, held, off, need, 3, slot, st);
                if (s != GS_OK) return s;
                a.hnbr = g->s_nbr[slot[0]];
                a.hbin = g->s_bin[slot[0]];
                a.hoff = off[slot[0]];
                a.anbr = g->s_nbr[slot[1]];
                a.abin = g->s_bin[slot[1]];
                a.aoff = off[slot[1]];
                a.bnbr = g->s_nbr[slot[2]];
                a.bbin = g->s_bin[slot[2]];
                a.boff = off[slot[2]];
                a.a_lo = (int32_t)g->win_row[fw[x]];
                a.a_hi = (int32_t)g->win_row[fw[x] + 1];
                a.b_lo = (int32_t)g->win_row[fw[y]];
                a.b_hi = (int32_t)g->win_row[fw[y] + 1];
                a.hub_begin = b0;
                a.hub_end = b1;
                s = c6_launch(g, a, true, st);
                if (s != GS_OK) return s;
            }
    }
    return GS_OK;
}

static gs_status c6_check(gs_graph_t g, int64_t hub_begin, int64_t hub_end)
{
    if (g->nb > C6_MAX_BINS)
        return gs_set_error(GS_ERR_ARG, "the six-bin 4pCF supports at most %d bins", C6_MAX_BINS);
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    if (g->edges[g->nb] >= (1ll << 20))
        return gs_set_error(GS_ERR_ARG, "the 4pCF needs r_max_lu < 2^20 for an exact int64 volume");
    return c6_prepare(g);
}

static C6Args c6_args(gs_graph_t g, int64_t hub_begin, int64_t hub_end)
{
    C6Args a{};
    a.pts = g->pts;
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.cfg6 = g->cfg6;
    a.hub_begin = hub_begin;
    a.hub_end = hub_end;
    a.box = (int)g->box_lu;
    a.periodic = g->periodic;
    a.nb = g->nb;
    a.ncfg = g->ncfg6;
    a.cursor = g->work + 3;
    return a;
}

// A count with its workspace allocated before any output is written: then
// the outputs (out_bytes each) are cleared and the tiles run.
static gs_status c6_count(gs_graph_t g, C6Args a, void *even_dev, void *odd_dev, size_t out_bytes,
                          int64_t hub_begin, int64_t hub_end, cudaStream_t st)
{
    char *scratch = nullptr;
    const size_t sbytes = c6_scratch_bytes(g, hub_end - hub_begin);
    if (sbytes) GS_TRY_CUDA(gs_malloc_async(&scratch, sbytes, st));
    gs_status s = GS_OK;
    cudaError_t e = cudaMemsetAsync(even_dev, 0, out_bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(odd_dev, 0, out_bytes, st);
    if (e != cudaSuccess) s = gs_set_error(GS_ERR_CUDA, "clearing the histograms failed: %s", cudaGetErrorString(e));
    if (s == GS_OK && hub_end > hub_begin && g->n_edges > 0) {
        a.scratch = scratch;
        s = c6_run(g, a, hub_begin, hub_end, st);
    }
    if (scratch) cudaFreeAsync(scratch, st);
    return s;
}

extern "C" gs_status gs_count_4pcf6(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev, int64_t hub_begin,
                                    int64_t hub_end, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !even_dev || !odd_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    gs_status s = c6_check(g, hub_begin, hub_end);
    if (s != GS_OK) return s;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    C6Args a = c6_args(g, hub_begin, hub_end);
    a.even = (unsigned long long *)even_dev;
    a.odd = (long long *)odd_dev;
    return c6_count(g, a, even_dev, odd_dev, sizeof(uint64_t) * g->ncfg6, hub_begin, hub_end, st);
}

extern "C" gs_status gs_count_4pcf6_weighted(gs_graph_t g, int64_t *even_dev, int64_t *odd_dev, int64_t hub_begin,
                                             int64_t hub_end, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !even_dev || !odd_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (!g->w) return gs_set_error(GS_ERR_ARG, "no weights: call gs_graph_set_weights first");
    gs_status s = c6_check(g, hub_begin, hub_end);
    if (s != GS_OK) return s;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    C6Args a = c6_args(g, hub_begin, hub_end);
    a.w = g->w;
    a.weven = (unsigned long long *)even_dev;
    a.wodd = (unsigned long long *)odd_dev;
    return c6_count(g, a, even_dev, odd_dev, sizeof(int64_t) * 2 * g->ncfg6, hub_begin, hub_end, st);
}
