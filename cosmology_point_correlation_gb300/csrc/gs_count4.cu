// gs_count4.cu -- parity-decomposed 4pCF (GRAMSCI v2, §III.1.1 and §III.2).
//
// For every hub i and every triple of spokes j1 < j2 < j3 in N(i) that are
// pairwise adjacent, the paper's three-way merge (§III.1.1, Eq.(2)) finds j3
// in hub tail ∩ N(j1) ∩ N(j2). Here the same triples come from one adjacency
// bit-matrix per hub: row s of the matrix holds, as bits, the positions t > s
// of the hub row whose node is also a neighbour of spoke s. The three-way
// intersection for (s1, s2) is then the AND of rows s1 and s2 above s2 --
// m/32 word operations instead of a pointer walk.
//
// Per hub, one thread block:
//   1. stages the hub row (ids; spoke vectors x_s - x_i, minimum image, with
//      the hub bin, as one int4 per spoke), one bitset of positions per hub
//      bin, and a hash table id -> row position in shared memory;
//   2. builds the bit-matrix: each warp walks the forward part of N(j) for one
//      spoke j (coalesced), probing the table;
//   3. clique search: warps take rows s1 from a counter, lanes take candidate
//      spokes s2 with bit (s1, s2) set and a hub bin other than s1's. The
//      third spokes of a pair are the AND of rows s1 and s2 above s2, less the
//      bitsets of the two bins already used; the warp prefix-sums the lanes'
//      counts word by word and deals the cliques out 32 at a time. A clique
//      adds 1 to even and sign(V) to odd at its sorted bin triple, with
//      V = det[r_1; r_2; r_3] of the bin-ordered spokes (Eq.(3)) obtained as
//      (r_s1 x r_s2) . r_s3 times the sign of the sorting permutation, in
//      exact int64 (V == 0 adds 0: the degenerate rule of §III.2).
// Hubs of degree <= C4_M run entirely in shared memory; rarer hubs of higher
// degree run in a second kernel whose per-block workspace lives in a global
// scratch slice. Both keep uint32 / int32 histograms in shared memory (a hub
// whose clique bound exceeds 2^31 adds straight to global memory).
//
// Windowed graphs (§III.5.3: tiles over pairs of search windows c1 <= c2):
// a tile stages the hub window and windows c1, c2; the bit rows of spokes in
// c1 and c2 are built, and only cliques s1 < s2 < s3 with s1 in c1 and s2 in
// c2 are counted. The rows of s1 and s2 give all three bits, and the windows
// of s1 <= s2 fix one tile, so every clique is counted once.

#include <algorithm>
#include <mutex>
#include <type_traits>
#include <vector>

#include "gs_internal.cuh"

constexpr int C4_THREADS = 256;
constexpr int C4_WARPS = C4_THREADS / 32;
constexpr int C4_M = 512;                   // largest hub degree kept in shared memory
constexpr int C4_WORDS = C4_M / 32;
constexpr int C4_TABLE = 2 * C4_M;
constexpr int C4_SMEM_HIST_MAX = 8192;
// Shared-memory histogram: three u32 counters per configuration, the cliques
// of negative, zero and positive volume, so that a clique is one add (the
// even count is their sum, the odd sum positive minus negative).
constexpr int C4_HIST_WORDS = 3;
constexpr int C4_EMPTY = -1;

struct C4Args {
    const int4 *pts;
    const int64_t *row_ptr;
    const int32_t *fwd;
    const int32_t *nbr;
    const uint8_t *bin;
    int64_t hub_begin, hub_end;
    int box, periodic;
    int nb, ncfg;
    unsigned long long *even;
    long long *odd;
    unsigned long long *cursor;
    // hub-list mode: hubs [0, hub_end) of this list, given by input index
    const int32_t *hubs;
    const int32_t *inv;
    // large-hub path
    int big_m;                    // largest degree the scratch slices hold
    char *scratch;                // gridDim.x slices of scratch_stride bytes
    size_t scratch_stride;
    // windowed graphs: hub rows at hnbr / hbin (edge e at e - hoff); spoke rows
    // of ids in [a_lo, a_hi) at anbr - aoff, of ids in [b_lo, b_hi) at
    // bnbr - boff (the same window when a_lo == b_lo)
    const int32_t *hnbr, *anbr, *bnbr;
    const uint8_t *hbin;
    int64_t hoff, aoff, boff;
    int32_t a_lo, a_hi, b_lo, b_hi;
    unsigned *chk;                // checked builds: the graph's check word
};

// Bins up to which the clique's packed index and bin-sorting parity come from
// one table of nb^3 entries (in the shared memory of the per-bin index tables).
constexpr int C4_TAB_BINS = 10;
// r_max (lattice units) up to which a spoke-pair cross product fits in int32:
// components |r| <= 32767, so |y1 z2 - z1 y2| <= 2 * 32767^2 < 2^31
constexpr int64_t C4_SMALL_R = 32768;
static_assert(C4_TAB_BINS * C4_TAB_BINS * C4_TAB_BINS * 2 <= 512 * 4, "the u16 table must fit the index tables' space");

// First position of a sorted row whose id is >= key.
__device__ __forceinline__ int c4_lower(const int32_t *row, int m, int32_t key)
{
    int lo = 0, hi = m;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (row[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Workspace of one hub: either shared memory or a global scratch slice.
struct HubSpace {
    int32_t *key;      // hash table (tsize slots)
    int32_t *pos;      // row position of each table slot
    int32_t *row;      // [m] neighbour ids
    uint8_t *hb;       // [m] hub bins
    int4 *v;           // [m] spoke vector x_s - x_i and hub bin (.w)
    unsigned *bits;    // [m][W] adjacency bits
    unsigned *bm;      // [nb][W] positions of each hub bin, as bits (zero between hubs)
    int *next;         // shared counter handing out the rows s1 of the clique search
};

template <bool SMEM_HIST, bool WINDOWED, bool SMALLR>
__device__ __forceinline__ void c4_hub(const C4Args &a, const HubSpace &w, long long i, int m,
                                       int tlog, unsigned *s_cnt,
                                       const int *lex_a, const int *lex_b)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r0 = a.row_ptr[i];
    const int32_t *R = WINDOWED ? a.hnbr + (r0 - a.hoff) : a.nbr + r0;     // the hub row and its bins
    const uint8_t *RB = WINDOWED ? a.hbin + (r0 - a.hoff) : a.bin + r0;
    // spokes whose rows are walked: positions [pa0, pa1) (window c1) and
    // [pb0, pb1) (window c2 when it differs); cliques take s1 in [pa0, pa1) and
    // s2 in [q2_lo, q2_hi)
    int pa0 = 0, pa1 = m, pb0 = 0, pb1 = 0, q2_lo = 0, q2_hi = m;
    if (WINDOWED) {                                            // the same values in every thread
        pa0 = c4_lower(R, m, a.a_lo);
        pa1 = c4_lower(R, m, a.a_hi);
        q2_lo = pa0;
        q2_hi = pa1;
        if (a.b_lo != a.a_lo) {
            pb0 = q2_lo = c4_lower(R, m, a.b_lo);
            pb1 = q2_hi = c4_lower(R, m, a.b_hi);
        }
        if (pa0 >= pa1 || q2_lo >= q2_hi || pa0 >= q2_hi - 1) return;   // no clique in this tile
    }
    const int W = (m + 31) >> 5;
    const int tsize = 1 << tlog, shift = 32 - tlog, mask = tsize - 1;
    const int4 P = a.pts[i];

    // 1. stage the row and the table
    for (int t = threadIdx.x; t < m; t += C4_THREADS) {
        const int32_t k = R[t];
        w.row[t] = k;
        const int b = RB[t];
        w.hb[t] = (uint8_t)b;
        const int4 Q = a.pts[k];
        w.v[t] = make_int4(gs_delta(P.x, Q.x, a.box, a.periodic), gs_delta(P.y, Q.y, a.box, a.periodic),
                           gs_delta(P.z, Q.z, a.box, a.periodic), b);
        atomicOr(&w.bm[b * W + (t >> 5)], 1u << (t & 31));
        uint32_t h = gs_hash(k, shift);
        while (atomicCAS(&w.key[h], C4_EMPTY, k) != C4_EMPTY) h = (h + 1) & mask;
        w.pos[h] = t;
    }
    for (int t = threadIdx.x; t < m * W; t += C4_THREADS) w.bits[t] = 0u;
    __syncthreads();

    // 2. adjacency among the spokes: bit (s, t) for t > s
    if (threadIdx.x == 0) *w.next = pa0;                       // read after the barrier below
    const int32_t kmax = w.row[m - 1];
    const int na = pa1 - pa0, nab = na + (pb1 - pb0);
    for (int u = warp; u < nab; u += C4_WARPS) {
        const bool in_a = u < na;
        const int s = in_a ? pa0 + u : pb0 + (u - na);
        if (s >= m - 1) continue;                              // no position above the last
        const int32_t *SN = WINDOWED ? (in_a ? a.anbr : a.bnbr) : a.nbr;
        const int64_t soff = WINDOWED ? (in_a ? a.aoff : a.boff) : 0;
        const int32_t j = w.row[s];
        const int64_t pe = a.row_ptr[j + 1];
        for (int64_t p = a.row_ptr[j] + a.fwd[j]; p < pe; p += 32) {
            const int64_t q = p + lane;
            const int32_t k = q < pe ? SN[q - soff] : 0x7fffffff;
            if (k <= kmax) {
                uint32_t h = gs_hash(k, shift);
                int32_t key;
                while ((key = w.key[h]) != k && key != C4_EMPTY) h = (h + 1) & mask;
                if (key == k) {
                    const int t = w.pos[h];
                    if (GS_DCHECK(t > s && t < m, a.chk, GS_SITE_C4_BITS))
                        atomicOr(&w.bits[(size_t)s * W + (t >> 5)], 1u << (t & 31));
                }
            }
            if (__shfl_sync(0xffffffffu, k, 31) > kmax) break;
        }
    }
    __syncthreads();

    // 3. cliques (s1 < s2 < s3), distinct hub bins. Warps take rows s1 from a
    // shared counter (low rows, with the most candidates, first) and 32
    // candidates s2 at a time (one per lane). For each word of the bit rows the
    // lanes' common bits (s3 > s2) are counted, prefix-summed across the warp
    // and handed out 32 at a time, so that all lanes work on cliques however
    // unevenly they are spread over the pairs (s1, s2). The volume is taken in
    // position order, D = (r_s1 x r_s2) . r_s3 with the cross product once per
    // pair, and V of the bin-ordered spokes is D times the sign of the
    // permutation that sorts (b1, b2, b3).
    const int s1_end = min(pa1, m - 2), s2_end = min(q2_hi, m - 1);
    for (;;) {
        int s1 = 0;
        if (lane == 0) s1 = atomicAdd(w.next, 1);
        s1 = __shfl_sync(0xffffffffu, s1, 0);
        if (s1 >= s1_end) break;
        const int4 r1 = w.v[s1];
        const int b1 = r1.w, x1 = r1.x, y1 = r1.y, z1 = r1.z;
        const unsigned *bm1 = w.bm + b1 * W;
        const unsigned *row1 = w.bits + (size_t)s1 * W;
        // cross products in int32 when r_max < C4_SMALL_R, else int64
        using CT = typename std::conditional<SMALLR, int, long long>::type;
        // s3's hub bin differs from b1 and b2 (the common bits were masked)
        auto clique = [&](int b2, CT cx, CT cy, CT cz, int s3) {
            if (!GS_DCHECK(s3 > s1 && s3 < m, a.chk, GS_SITE_C4_BITS)) return;
            const int4 r3 = w.v[s3];
            const int b3 = r3.w;
            const long long d = (long long)cx * r3.x + (long long)cy * r3.y + (long long)cz * r3.z;   // |d| < 3 * 2^60
            int sg = (d > 0) - (d < 0);
            int idx;
            if (a.nb <= C4_TAB_BINS) {                             // block-uniform
                // lex_a holds the table: (idx4 << 1) | parity of the sorting permutation
                const int e = reinterpret_cast<const uint16_t *>(lex_a)[(b1 * a.nb + b2) * a.nb + b3];
                idx = e >> 1;
                if (e & 1) sg = -sg;
            } else {
                if (((b1 > b2) + (b1 > b3) + (b2 > b3)) & 1) sg = -sg;
                const int lo = min(b1, min(b2, b3)), hi = max(b1, max(b2, b3));
                idx = lex_a[lo] + lex_b[b1 + b2 + b3 - lo - hi] + hi;
            }
            if (!GS_DCHECK(idx >= 0 && idx < a.ncfg, a.chk, GS_SITE_C4_HIST)) return;
            if (SMEM_HIST) {
                // one add, into the counter of the volume's sign
                atomicAdd(&s_cnt[(sg + 1) * a.ncfg + idx], 1u);
            } else {
                atomicAdd(a.even + idx, 1ull);
                if (sg) atomicAdd((unsigned long long *)(a.odd + idx), (unsigned long long)(long long)sg);
            }
        };
        for (int c2 = max(s1 + 1, q2_lo); c2 < s2_end; c2 += 32) {        // warp-uniform
            const int s2 = c2 + lane;
            bool valid = s2 < s2_end && ((row1[s2 >> 5] >> (s2 & 31)) & 1u);
            int b2 = 0;
            CT cx = 0, cy = 0, cz = 0;
            if (valid) {
                const int4 r2 = w.v[s2];
                b2 = r2.w;
                valid = b2 != b1;
                const int x2 = r2.x, y2 = r2.y, z2 = r2.z;                       // r_s1 x r_s2, |.| < 2^41
                cx = (CT)y1 * z2 - (CT)z1 * y2;
                cy = (CT)z1 * x2 - (CT)x1 * z2;
                cz = (CT)x1 * y2 - (CT)y1 * x2;
            }
            if (!__any_sync(0xffffffffu, valid)) continue;
            const unsigned *row2 = w.bits + (size_t)(valid ? s2 : s1) * W;
            const unsigned *bm2 = w.bm + b2 * W;
            for (int wd = c2 >> 5; wd < W; ++wd) {
                unsigned common = 0u;
                if (valid && wd >= (s2 >> 5)) {                // s3 adjacent to both, hub bin not b1 or b2
                    common = row1[wd] & row2[wd] & ~(bm1[wd] | bm2[wd]);
                    if (wd == (s2 >> 5)) common &= ~((2u << (s2 & 31)) - 1u);   // keep s3 > s2
                }
                if (!__ballot_sync(0xffffffffu, common != 0u)) continue;   // no clique in this word
                const int cnt = __popc(common);
                // When the lanes' cliques in this word are even enough (the largest
                // count at most twice the rounds that dealing them out would take),
                // each lane takes its own, with its pair data in its registers;
                // else they are dealt out 32 at a time
                const int all = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
                const int most = (int)__reduce_max_sync(0xffffffffu, (unsigned)cnt);
                if (most <= 2 * ((all + 31) >> 5)) {
                    for (unsigned cm = common; cm; cm &= cm - 1) clique(b2, cx, cy, cz, (wd << 5) + __ffs(cm) - 1);
                    continue;
                }
                int inc = cnt;                                     // inclusive prefix over lanes
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                const int total = __shfl_sync(0xffffffffu, inc, 31);
                for (int k = 0; k < total; k += 32) {
                    const int q = k + lane;
                    int owner = 0;                                 // first lane whose prefix exceeds q
#pragma unroll
                    for (int step = 16; step > 0; step >>= 1)
                        if (__shfl_sync(0xffffffffu, inc, owner + step - 1) <= q) owner += step;
                    const unsigned cm = __shfl_sync(0xffffffffu, common, owner);
                    const int first = __shfl_sync(0xffffffffu, inc - cnt, owner);
                    const int o_b2 = __shfl_sync(0xffffffffu, b2, owner);
                    const CT ocx = __shfl_sync(0xffffffffu, cx, owner);
                    const CT ocy = __shfl_sync(0xffffffffu, cy, owner);
                    const CT ocz = __shfl_sync(0xffffffffu, cz, owner);
                    if (q < total) clique(o_b2, ocx, ocy, ocz, (wd << 5) + gs_nth_bit(cm, q - first));
                }
            }
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < tsize; t += C4_THREADS) w.key[t] = C4_EMPTY;
    for (int t = threadIdx.x; t < a.nb * W; t += C4_THREADS) w.bm[t] = 0u;
}

// gs_idx4(a, b, c) = F4(a) - H(a + 1) + H(b) + c - b - 1 with
// H(t) = t (nb - 1) - t (t - 1) / 2 and F4(a) = gs_idx4(a, a + 1, a + 2),
// split into two per-bin tables: idx4 = lex_a[a] + lex_b[b] + c. For
// nb <= C4_TAB_BINS the space of both (contiguous) holds instead one u16 per
// ordered triple (b1, b2, b3) of distinct bins: (idx4 of the sorted triple
// << 1) | the parity of the permutation that sorts it.
__device__ __forceinline__ void c4_lex_tables(int nb, int *lex_a, int *lex_b)
{
    if (nb <= C4_TAB_BINS) {
        uint16_t *tab = reinterpret_cast<uint16_t *>(lex_a);
        for (int t = threadIdx.x; t < nb * nb * nb; t += C4_THREADS) {
            const int x = t / (nb * nb), y = (t / nb) % nb, z = t % nb;
            if (x == y || x == z || y == z) continue;
            const int lo = min(x, min(y, z)), hi = max(x, max(y, z)), mid = x + y + z - lo - hi;
            tab[t] = (uint16_t)((gs_idx4(nb, lo, mid, hi) << 1) | (((x > y) + (x > z) + (y > z)) & 1));
        }
        return;
    }
    for (int t = threadIdx.x; t < nb; t += C4_THREADS) {
        const int64_t h1 = (int64_t)(t + 1) * (nb - 1) - (int64_t)(t + 1) * t / 2;
        const int64_t h0 = (int64_t)t * (nb - 1) - (int64_t)t * (t - 1) / 2;
        lex_a[t] = (int)(gs_idx4(nb, t, t + 1, t + 2) - h1);
        lex_b[t] = (int)(h0 - t - 1);
    }
}

// Add the shared counters into the caller's histograms and clear them: even =
// negative + zero + positive volume, odd = positive - negative.
__device__ __forceinline__ void c4_flush(unsigned *sc, int ncfg, unsigned long long *ge, long long *go)
{
    for (int t = threadIdx.x; t < ncfg; t += C4_THREADS) {
        const unsigned neg = sc[t], zero = sc[ncfg + t], pos = sc[2 * ncfg + t];
        const unsigned long long e = (unsigned long long)neg + zero + pos;
        const long long o = (long long)pos - (long long)neg;
        if (e) atomicAdd(ge + t, (unsigned long long)e);
        if (o) atomicAdd((unsigned long long *)(go + t), (unsigned long long)o);
        sc[t] = 0u;
        sc[ncfg + t] = 0u;
        sc[2 * ncfg + t] = 0u;
    }
}

// Hubs of degree 3..C4_M, workspace in shared memory; histograms in shared
// memory too unless there are too many configurations.
template <bool SMEM_HIST, bool HUB_LIST, bool WINDOWED, bool SMALLR>
__global__ void __launch_bounds__(C4_THREADS, 4)
k_count4_small(C4Args a)
{
    extern __shared__ unsigned s_dyn[];         // bits [C4_M * C4_WORDS], bin masks [nb * C4_WORDS], counters [3][ncfg]
    __shared__ int32_t s_key[C4_TABLE];
    __shared__ int32_t s_pos[C4_TABLE];
    __shared__ int32_t s_row[C4_M];
    __shared__ uint8_t s_hb[C4_M];
    __shared__ int4 s_v[C4_M];
    __shared__ int s_lex[512];                  // lex_a, lex_b (or the u16 table; see c4_lex_tables)
    int *s_lex_a = s_lex, *s_lex_b = s_lex + 256;
    __shared__ long long s_hub;
    __shared__ unsigned long long s_pending;
    __shared__ int s_next;

    unsigned *s_bits = s_dyn;
    unsigned *s_bm = s_dyn + C4_M * C4_WORDS;                 // [nb][C4_WORDS]
    unsigned *s_cnt = s_bm + a.nb * C4_WORDS;
    c4_lex_tables(a.nb, s_lex_a, s_lex_b);
    if (SMEM_HIST)
        for (int t = threadIdx.x; t < C4_HIST_WORDS * a.ncfg; t += C4_THREADS) s_cnt[t] = 0u;
    for (int t = threadIdx.x; t < C4_TABLE; t += C4_THREADS) s_key[t] = C4_EMPTY;
    if (threadIdx.x == 0) s_pending = 0;
    HubSpace w{ s_key, s_pos, s_row, s_hb, s_v, s_bits, s_bm, &s_next };
    for (int t = threadIdx.x; t < a.nb * C4_WORDS; t += C4_THREADS) s_bm[t] = 0u;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        if (s_hub >= a.hub_end) break;
        const long long i = HUB_LIST ? (long long)a.inv[a.hubs[s_hub]] : s_hub;
        const int m = (int)(a.row_ptr[i + 1] - a.row_ptr[i]);
        if (m < 3 || m > C4_M) continue;
        if (SMEM_HIST) {
            // C(m, 3) bounds the cliques of this hub
            const unsigned long long bound = (unsigned long long)m * (m - 1) * (m - 2) / 6;
            if (s_pending + bound > 0x7fffffffull) {
                c4_flush(s_cnt, a.ncfg, a.even, a.odd);
                __syncthreads();
                if (threadIdx.x == 0) s_pending = 0;
            }
            __syncthreads();
            if (threadIdx.x == 0) s_pending += bound;
        }
        int tlog = 4;
        while ((1 << tlog) < 2 * m) ++tlog;
        c4_hub<SMEM_HIST, WINDOWED, SMALLR>(a, w, i, m, tlog, s_cnt, s_lex_a, s_lex_b);
    }
    if (SMEM_HIST) {
        __syncthreads();
        c4_flush(s_cnt, a.ncfg, a.even, a.odd);
    }
}

// Hubs of degree > C4_M: workspace in a global scratch slice per block;
// histograms in shared memory (SMEM_HIST) as in the small kernel, except for
// a hub whose clique bound could overflow the 32-bit counters, which adds
// straight to global memory.
template <bool SMEM_HIST, bool HUB_LIST, bool WINDOWED, bool SMALLR>
__global__ void __launch_bounds__(C4_THREADS, 4)
k_count4_large(C4Args a)
{
    extern __shared__ unsigned s_dyn[];             // (SMEM_HIST) counters [3][ncfg]
    __shared__ int s_lex[512];                  // lex_a, lex_b (or the u16 table; see c4_lex_tables)
    int *s_lex_a = s_lex, *s_lex_b = s_lex + 256;
    __shared__ long long s_hub;
    __shared__ int s_next;
    __shared__ unsigned long long s_pending;
    unsigned *s_cnt = s_dyn;
    c4_lex_tables(a.nb, s_lex_a, s_lex_b);
    if (SMEM_HIST)
        for (int t = threadIdx.x; t < C4_HIST_WORDS * a.ncfg; t += C4_THREADS) s_cnt[t] = 0u;
    if (threadIdx.x == 0) s_pending = 0;

    const int M = a.big_m;
    int tlog = 4;
    while ((1 << tlog) < 2 * M) ++tlog;
    const int WM = (M + 31) >> 5;
    char *base = a.scratch + (size_t)blockIdx.x * a.scratch_stride;
    HubSpace w;
    w.v = (int4 *)base;                                   // slices start 256-byte aligned
    w.key = (int32_t *)(w.v + M);
    w.pos = w.key + (1 << tlog);
    w.row = w.pos + (1 << tlog);
    w.bits = (unsigned *)(w.row + M);
    w.bm = w.bits + (size_t)M * WM;
    w.hb = (uint8_t *)(w.bm + (size_t)a.nb * WM);
    for (int t = threadIdx.x; t < a.nb * WM; t += C4_THREADS) w.bm[t] = 0u;
    w.next = &s_next;
    for (int t = threadIdx.x; t < (1 << tlog); t += C4_THREADS) w.key[t] = C4_EMPTY;

    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        if (s_hub >= a.hub_end) break;
        const long long i = HUB_LIST ? (long long)a.inv[a.hubs[s_hub]] : s_hub;
        const int m = (int)(a.row_ptr[i + 1] - a.row_ptr[i]);
        if (m <= C4_M) continue;
        int tl = 4;
        while ((1 << tl) < 2 * m) ++tl;
        const unsigned long long bound = (unsigned long long)m * (m - 1) * (m - 2) / 6;
        if (!SMEM_HIST || bound > 0x7fffffffull) {
            c4_hub<false, WINDOWED, SMALLR>(a, w, i, m, tl, nullptr, s_lex_a, s_lex_b);
            continue;
        }
        if (s_pending + bound > 0x7fffffffull) {
            c4_flush(s_cnt, a.ncfg, a.even, a.odd);
            __syncthreads();
            if (threadIdx.x == 0) s_pending = 0;
        }
        __syncthreads();
        if (threadIdx.x == 0) s_pending += bound;
        c4_hub<SMEM_HIST, WINDOWED, SMALLR>(a, w, i, m, tl, s_cnt, s_lex_a, s_lex_b);
    }
    if (SMEM_HIST) {
        __syncthreads();
        c4_flush(s_cnt, a.ncfg, a.even, a.odd);
    }
}

// Bytes of one large-hub workspace slice (hubs of degree up to M), a multiple
// of 256: spoke vectors, hash table, row, bit-matrix, bin masks, hub bins.
static size_t c4_large_stride(int M, int nb)
{
    int tlog = 4;
    while ((1 << tlog) < 2 * M) ++tlog;
    const size_t WM = (size_t)(M + 31) / 32;
    const size_t bytes = 16 * (size_t)M + sizeof(int32_t) * (2 * ((size_t)1 << tlog) + (size_t)M) +
                         sizeof(unsigned) * ((size_t)M * WM + (size_t)nb * WM) + (size_t)M;
    return (bytes + 255) & ~(size_t)255;
}

// The kernel instantiations by shared histogram, hub list, windows and the
// width of the cross products.
using C4Kernel = void (*)(C4Args);

template <bool S, bool L, bool W>
static C4Kernel c4_pick(bool large, bool sr)
{
    if (large) return sr ? k_count4_large<S, L, W, true> : k_count4_large<S, L, W, false>;
    return sr ? k_count4_small<S, L, W, true> : k_count4_small<S, L, W, false>;
}

static C4Kernel c4_kernel(bool large, bool smem, bool list, bool win, gs_graph_t g)
{
    const bool sr = g->edges[g->nb] <= C4_SMALL_R;
    if (smem) {
        if (list) return win ? c4_pick<true, true, true>(large, sr) : c4_pick<true, true, false>(large, sr);
        return win ? c4_pick<true, false, true>(large, sr) : c4_pick<true, false, false>(large, sr);
    }
    if (list) return win ? c4_pick<false, true, true>(large, sr) : c4_pick<false, true, false>(large, sr);
    return win ? c4_pick<false, false, true>(large, sr) : c4_pick<false, false, false>(large, sr);
}

// Both kernels over the hubs [a.hub_begin, a.hub_end) (outputs accumulate).
static gs_status c4_launch(gs_graph_t g, C4Args a, bool windowed, cudaStream_t st)
{
    const int64_t hubs = a.hub_end - a.hub_begin;
    const int sms = gs_sm_count();
    const bool smem = a.ncfg <= C4_SMEM_HIST_MAX;
    const size_t dyn = sizeof(unsigned) * ((size_t)C4_M * C4_WORDS + (size_t)a.nb * C4_WORDS +
                                           (smem ? C4_HIST_WORDS * (size_t)a.ncfg : 0));
    const C4Kernel kern = c4_kernel(false, smem, false, windowed, g);
    int per_sm = 0;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C4_THREADS, dyn));
    per_sm = std::max(per_sm, 1);
    GS_TRY_CUDA(cudaMemsetAsync(g->work + 1, 0, 2 * sizeof(unsigned long long), st));
    a.cursor = g->work + 1;
    const int grid = (int)std::min<int64_t>((int64_t)sms * per_sm, hubs);
    kern<<<grid, C4_THREADS, dyn, st>>>(a);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());

    if (g->max_degree > C4_M) {
        // a.scratch: the caller's workspace of c4_scratch_bytes(g, hubs) bytes
        const int M = g->max_degree;
        a.cursor = g->work + 2;
        a.big_m = M;
        a.scratch_stride = c4_large_stride(M, g->nb);
        const int gl = (int)std::min<int64_t>((int64_t)sms * 2, hubs);
        const size_t ldyn = smem ? sizeof(unsigned) * C4_HIST_WORDS * (size_t)a.ncfg : 0;
        const C4Kernel big = c4_kernel(true, smem, false, windowed, g);
        GS_TRY_CUDA(cudaFuncSetAttribute(big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ldyn));
        big<<<gl, C4_THREADS, ldyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }
    return GS_OK;
}

// Workspace of the large-hub kernel for a launch over at most `hubs` hubs
// (0 when no hub has more than C4_M neighbours).
static size_t c4_scratch_bytes(gs_graph_t g, int64_t hubs)
{
    if (g->max_degree <= C4_M || hubs <= 0) return 0;
    return c4_large_stride(g->max_degree, g->nb) * (size_t)std::min<int64_t>((int64_t)gs_sm_count() * 2, hubs);
}

static gs_status c4_count(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev, int64_t hub_begin,
                          int64_t hub_end, char *scratch, cudaStream_t st);

extern "C" gs_status gs_count_4pcf_parity(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev,
                                          int64_t hub_begin, int64_t hub_end, void *cuda_stream)
{
    GS_ENTRY();
    if (!g) return gs_set_error(GS_ERR_ARG, "graph is NULL");
    GS_TRY_DEVICE(g);
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    if (g->edges[g->nb] >= (1ll << 20))
        return gs_set_error(GS_ERR_ARG, "parity 4pCF needs r_max_lu < 2^20 for an exact int64 volume");
    const int64_t ncfg = gs_ncfg4(g->nb);
    if (ncfg <= 0) return GS_OK;
    if (!even_dev || !odd_dev) return gs_set_error(GS_ERR_ARG, "NULL histogram");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    // the large-hub workspace is allocated before any output is written
    char *scratch = nullptr;
    const size_t sbytes = g->n_edges > 0 ? c4_scratch_bytes(g, hub_end - hub_begin) : 0;
    if (sbytes) GS_TRY_CUDA(gs_malloc_async(&scratch, sbytes, st));
    gs_status s = gs_checked_begin(g, st);
    if (s == GS_OK) s = c4_count(g, (uint64_t *)even_dev, odd_dev, hub_begin, hub_end, scratch, st);
    if (s == GS_OK) s = gs_checked_end(g, st, "parity 4pCF count");
    if (scratch) cudaFreeAsync(scratch, st);
    return s;
}

// The parity count once its workspace is in hand: clear the outputs, then
// one launch (device-resident graph) or one per window tile.
static gs_status c4_count(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev, int64_t hub_begin,
                          int64_t hub_end, char *scratch, cudaStream_t st)
{
    const int64_t ncfg = gs_ncfg4(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(even_dev, 0, sizeof(uint64_t) * ncfg, st));
    GS_TRY_CUDA(cudaMemsetAsync(odd_dev, 0, sizeof(int64_t) * ncfg, st));
    if (hub_end == hub_begin || g->n_edges == 0) return GS_OK;

    C4Args a{};
    a.pts = g->pts;
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.hub_begin = hub_begin;
    a.hub_end = hub_end;
    a.box = (int)g->box_lu;
    a.periodic = g->periodic;
    a.nb = g->nb;
    a.ncfg = (int)ncfg;
    a.even = (unsigned long long *)even_dev;
    a.odd = (long long *)odd_dev;
    a.chk = g->chk;
    a.scratch = scratch;
    if (!g->n_win) return c4_launch(g, a, false, st);

    // windowed: tiles (hub window h, spoke windows c1 <= c2), both adjacent to h
    int held[GS_SLOTS];
    int64_t off[GS_SLOTS] = {};
    for (int k = 0; k < GS_SLOTS; ++k) held[k] = -1;
    for (int h = 0; h < g->n_win; ++h) {
        const int64_t b0 = std::max(hub_begin, g->win_row[h]), b1 = std::min(hub_end, g->win_row[h + 1]);
        if (b0 >= b1 || g->win_e0[h + 1] == g->win_e0[h]) continue;
        std::vector<int> adj;
        for (int c = 0; c < g->n_win; ++c)
            if (g->win_e0[c + 1] > g->win_e0[c] && gs_windows_adjacent(g, h, c)) adj.push_back(c);
        for (size_t x = 0; x < adj.size(); ++x)
            for (size_t y = x; y < adj.size(); ++y) {
                const int need[3] = { h, adj[x], adj[y] };
                int slot[3];
                gs_status s = gs_stage_set(g, held, off, need, 3, slot, st);
                if (s != GS_OK) return s;
                a.hnbr = g->s_nbr[slot[0]];
                a.hbin = g->s_bin[slot[0]];
                a.hoff = off[slot[0]];
                a.anbr = g->s_nbr[slot[1]];
                a.aoff = off[slot[1]];
                a.bnbr = g->s_nbr[slot[2]];
                a.boff = off[slot[2]];
                a.a_lo = (int32_t)g->win_row[adj[x]];
                a.a_hi = (int32_t)g->win_row[adj[x] + 1];
                a.b_lo = (int32_t)g->win_row[adj[y]];
                a.b_hi = (int32_t)g->win_row[adj[y] + 1];
                a.hub_begin = b0;
                a.hub_end = b1;
                s = c4_launch(g, a, true, st);
                if (s != GS_OK) return s;
            }
    }
    return GS_OK;
}

static gs_status c4_count_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count, uint64_t *even_dev,
                               int64_t *odd_dev, char *scratch, cudaStream_t st);

extern "C" gs_status gs_count_4pcf_parity_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count,
                                               uint64_t *even_dev, int64_t *odd_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || (count > 0 && !hubs_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (count < 0) return gs_set_error(GS_ERR_ARG, "negative hub count");
    if (g->n_win) return gs_set_error(GS_ERR_ARG, "the parity 4pCF needs a device-resident graph (this one is windowed)");
    if (g->edges[g->nb] >= (1ll << 20))
        return gs_set_error(GS_ERR_ARG, "parity 4pCF needs r_max_lu < 2^20 for an exact int64 volume");
    const int64_t ncfg = gs_ncfg4(g->nb);
    if (ncfg <= 0) return GS_OK;
    if (!even_dev || !odd_dev) return gs_set_error(GS_ERR_ARG, "NULL histogram");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    gs_status s = gs_check_ids(g, hubs_dev, count, st);
    if (s != GS_OK) return s;
    // the large-hub workspace is allocated before any output is written
    char *scratch = nullptr;
    const size_t sbytes = g->n_edges > 0 ? c4_scratch_bytes(g, count) : 0;
    if (sbytes) GS_TRY_CUDA(gs_malloc_async(&scratch, sbytes, st));
    s = gs_checked_begin(g, st);
    if (s == GS_OK) s = c4_count_hubs(g, hubs_dev, count, (uint64_t *)even_dev, odd_dev, scratch, st);
    if (s == GS_OK) s = gs_checked_end(g, st, "parity 4pCF hub-list count");
    if (scratch) cudaFreeAsync(scratch, st);
    return s;
}

static gs_status c4_count_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count, uint64_t *even_dev,
                               int64_t *odd_dev, char *scratch, cudaStream_t st)
{
    const int64_t ncfg = gs_ncfg4(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(even_dev, 0, sizeof(uint64_t) * ncfg, st));
    GS_TRY_CUDA(cudaMemsetAsync(odd_dev, 0, sizeof(int64_t) * ncfg, st));
    if (count == 0 || g->n_edges == 0) return GS_OK;
    GS_TRY_CUDA(cudaMemsetAsync(g->work + 1, 0, 2 * sizeof(unsigned long long), st));

    C4Args a{};
    a.pts = g->pts;
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.hub_begin = 0;
    a.hub_end = count;
    a.hubs = hubs_dev;
    a.inv = g->inv;
    a.box = (int)g->box_lu;
    a.periodic = g->periodic;
    a.nb = g->nb;
    a.ncfg = (int)ncfg;
    a.even = (unsigned long long *)even_dev;
    a.odd = (long long *)odd_dev;
    a.chk = g->chk;
    a.scratch = scratch;

    const int sms = gs_sm_count();
    const bool smem = ncfg <= C4_SMEM_HIST_MAX;
    const size_t dyn = sizeof(unsigned) * ((size_t)C4_M * C4_WORDS + (size_t)g->nb * C4_WORDS +
                                           (smem ? C4_HIST_WORDS * ncfg : 0));
    const C4Kernel kern = c4_kernel(false, smem, true, false, g);
    int per_sm = 0;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C4_THREADS, dyn));
    per_sm = std::max(per_sm, 1);
    a.cursor = g->work + 1;
    kern<<<(int)std::min<int64_t>((int64_t)sms * per_sm, count), C4_THREADS, dyn, st>>>(a);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    if (g->max_degree > C4_M) {
        const int M = g->max_degree;
        size_t stride = c4_large_stride(M, g->nb);
        const int gl = (int)std::min<int64_t>((int64_t)sms * 2, count);
        a.cursor = g->work + 2;
        a.big_m = M;
        a.scratch_stride = stride;
        const size_t ldyn = smem ? sizeof(unsigned) * C4_HIST_WORDS * (size_t)ncfg : 0;
        const C4Kernel big = c4_kernel(true, smem, true, false, g);
        GS_TRY_CUDA(cudaFuncSetAttribute(big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ldyn));
        big<<<gl, C4_THREADS, ldyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }
    return GS_OK;
}

// ---------------------------------------------------------------- fixed-workspace variant
//
// gs_count_4pcf_parity_static runs the same two kernels as gs_count_4pcf_parity
// but takes every piece of scratch memory it needs -- the two work cursors and
// the per-block workspace of hubs with more than C4_M neighbours -- from the
// file-scope device array below instead of cudaMallocAsync / graph memory.
// The array is part of the library image: every GPU that loads the library
// holds GS_C4_STATIC_BYTES of device memory for it until the process exits.

constexpr size_t GS_C4_STATIC_BYTES = (size_t)16 << 20;     // 16 MiB
constexpr size_t GS_C4_STATIC_HEAD = 256;                     // two cursors, padded

static __device__ __align__(256) unsigned char g_c4_static[GS_C4_STATIC_BYTES];

static std::mutex g_c4_static_mu;
static char *g_c4_static_base[64];                            // per device

// Device address of g_c4_static on the current device. Host code may not use
// the symbol itself (it names a host-side stand-in), so the address is looked
// up once per device with that device current and cached.
static gs_status c4_static_base(char **out)
{
    int dev = 0;
    GS_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return gs_set_error(GS_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_c4_static_mu);
    if (!g_c4_static_base[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_c4_static);
        if (e != cudaSuccess || !p)
            return gs_set_error(GS_ERR_CUDA, "cudaGetSymbolAddress of the static workspace failed: %s",
                                cudaGetErrorString(e));
        g_c4_static_base[dev] = (char *)p;
    }
    *out = g_c4_static_base[dev];
    return GS_OK;
}

extern "C" gs_status gs_count_4pcf_parity_static(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev,
                                                 int64_t hub_begin, int64_t hub_end, void *cuda_stream)
{
    GS_ENTRY();
    if (!g) return gs_set_error(GS_ERR_ARG, "graph is NULL");
    GS_TRY_DEVICE(g);
    if (g->n_win) return gs_set_error(GS_ERR_ARG, "the parity 4pCF needs a device-resident graph (this one is windowed)");
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    if (g->edges[g->nb] >= (1ll << 20))
        return gs_set_error(GS_ERR_ARG, "parity 4pCF needs r_max_lu < 2^20 for an exact int64 volume");
    const int64_t ncfg = gs_ncfg4(g->nb);
    if (ncfg <= 0) return GS_OK;
    if (!even_dev || !odd_dev) return gs_set_error(GS_ERR_ARG, "NULL histogram");

    // workspace of one block for the largest hub; refuse before writing anything
    const int M = g->max_degree;
    size_t stride = 0;
    if (M > C4_M) {
        stride = c4_large_stride(M, g->nb);
        if (stride > GS_C4_STATIC_BYTES - GS_C4_STATIC_HEAD)
            return gs_set_error(GS_ERR_CAPACITY,
                                "a hub of degree %d needs %zu bytes of workspace; the static workspace holds %zu "
                                "(use gs_count_4pcf_parity)", M, stride, GS_C4_STATIC_BYTES - GS_C4_STATIC_HEAD);
    }
    char *base = nullptr;
    gs_status s = c4_static_base(&base);
    if (s != GS_OK) return s;

    cudaStream_t st = (cudaStream_t)cuda_stream;
    GS_TRY_CUDA(cudaMemsetAsync(even_dev, 0, sizeof(uint64_t) * ncfg, st));
    GS_TRY_CUDA(cudaMemsetAsync(odd_dev, 0, sizeof(int64_t) * ncfg, st));
    if (hub_end == hub_begin || g->n_edges == 0) return GS_OK;
    unsigned long long *cursors = (unsigned long long *)base;
    GS_TRY_CUDA(cudaMemsetAsync(cursors, 0, 2 * sizeof(unsigned long long), st));   // left over from the last call
    s = gs_checked_begin(g, st);
    if (s != GS_OK) return s;

    C4Args a{};
    a.pts = g->pts;
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.nbr = g->nbr;
    a.bin = g->bin;
    a.hub_begin = hub_begin;
    a.hub_end = hub_end;
    a.box = (int)g->box_lu;
    a.periodic = g->periodic;
    a.nb = g->nb;
    a.ncfg = (int)ncfg;
    a.even = (unsigned long long *)even_dev;
    a.odd = (long long *)odd_dev;
    a.chk = g->chk;

    const int64_t hubs = hub_end - hub_begin;
    const int sms = gs_sm_count();
    const bool smem = ncfg <= C4_SMEM_HIST_MAX;
    const size_t dyn = sizeof(unsigned) * ((size_t)C4_M * C4_WORDS + (size_t)g->nb * C4_WORDS +
                                           (smem ? C4_HIST_WORDS * ncfg : 0));
    const C4Kernel kern = c4_kernel(false, smem, false, false, g);
    int per_sm = 0;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C4_THREADS, dyn));
    per_sm = std::max(per_sm, 1);
    a.cursor = cursors;
    const int grid = (int)std::min<int64_t>((int64_t)sms * per_sm, hubs);
    kern<<<grid, C4_THREADS, dyn, st>>>(a);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());

    if (M > C4_M) {
        const int64_t slices = (int64_t)((GS_C4_STATIC_BYTES - GS_C4_STATIC_HEAD) / stride);
        const int gl = (int)std::min<int64_t>(std::min<int64_t>((int64_t)sms * 2, hubs), slices);
        a.cursor = cursors + 1;
        a.big_m = M;
        a.scratch = base + GS_C4_STATIC_HEAD;
        a.scratch_stride = stride;
        const size_t ldyn = smem ? sizeof(unsigned) * C4_HIST_WORDS * (size_t)ncfg : 0;
        const C4Kernel big = c4_kernel(true, smem, false, false, g);
        GS_TRY_CUDA(cudaFuncSetAttribute(big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ldyn));
        big<<<gl, C4_THREADS, ldyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
    }
    return gs_checked_end(g, st, "parity 4pCF count (fixed workspace)");
}
