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
// Weighted counts (§II.1: signed per-point weights) use the same walk: the
// chunk also holds each key's weight and a hit adds w_j w_k (|.| <= 2^30) to
// the block's int64 sum T[config] of the current hub (two 32-bit words with
// a carry, so that a hit costs one 32-bit shared atomic). A pass over at most
// C3_SPOKES spokes of one chunk closes at most 2^24 triangles, so |T| stays
// below 2^54; after each pass the block adds w_i T, an exact 128-bit product,
// into its own 128-bit slice of a global scratch array (no atomics: each
// configuration has one owner thread), and a second kernel sums the slices.
//
// Long rows are processed in chunks of the hub row: chunk [c0, c1) holds the
// k candidates, every spoke at position s < c1 - 1 is walked over keys in
// (max(j, F[c0] - 1), F[c1 - 1]]; a spoke of an earlier chunk first finds its
// starting entry by binary search. A bitmap chunk holds up to C3_CHUNK_BM
// keys (C3_CHUNK_BM_W weighted), a hash chunk C3_CHUNK.
//
// Hubs are handed out in increasing internal order from a global counter, so
// the blocks resident at any moment work on neighbouring hubs whose spoke
// rows overlap and stay in L2.

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <utility>
#include <vector>

#include "gs_internal.cuh"

constexpr int C3_THREADS = 512;
constexpr int C3_MAX_BLOCKS_PER_SM = 2;          // __launch_bounds__ of k_count3
constexpr int C3_WARPS = C3_THREADS / 32;
constexpr int C3_TABLE_LOG = 13;                 // 8192 slots
constexpr int C3_TABLE = 1 << C3_TABLE_LOG;
constexpr int C3_CHUNK = C3_TABLE / 4;           // hash mode: keys per chunk (load factor <= 1/4)
constexpr int C3_CHUNK_BM = 8192;                // bitmap mode: keys per chunk
constexpr int C3_CHUNK_BM_W = 4096;              // bitmap mode, weighted (2 more bytes per key)
constexpr int C3_SPOKES = 4096;                  // spokes grouped per pass
constexpr int C3_SPAN_BITS = 1 << 18;            // bitmap mode: key span of a chunk
constexpr int C3_SPAN_WORDS = C3_SPAN_BITS / 32;
constexpr int C3_BM_WORDS = C3_SPAN_WORDS + 4;   // + a zero guard word that out-of-range probes read
// bytes of the candidate-key region: the larger of the two modes
constexpr int C3_REGION_BITMAP = C3_BM_WORDS * 4 + C3_SPAN_WORDS * 2 + C3_CHUNK_BM;
constexpr int C3_REGION_HASH = C3_TABLE * 5;
constexpr int C3_REGION = ((C3_REGION_BITMAP > C3_REGION_HASH ? C3_REGION_BITMAP : C3_REGION_HASH) + 15) & ~15;
// weighted: the chunk's weights follow the bins (int16 per key / per slot)
constexpr int C3_REGION_BITMAP_W = C3_BM_WORDS * 4 + C3_SPAN_WORDS * 2 + C3_CHUNK_BM_W * 3;
constexpr int C3_REGION_HASH_W = C3_TABLE * 7;
constexpr int C3_REGION_W = ((C3_REGION_BITMAP_W > C3_REGION_HASH_W ? C3_REGION_BITMAP_W : C3_REGION_HASH_W) + 15) & ~15;
constexpr int C3_SMEM_HIST_MAX = 12288;          // configurations kept in shared memory (nbins <= 40)
constexpr int C3_WEIGHTED_MAX_BINS = 40;
constexpr int C3_EMPTY = -1;

struct C3Args {
    const int64_t *row_ptr;
    const int32_t *fwd;
    // edge arrays: hub rows from (hnbr, hbin), spoke rows from (snbr, sbin);
    // global edge e sits at index e - hoff (e - soff). A device-resident graph
    // passes its own arrays with offset 0; a windowed graph (§III.5.3) the
    // staged hub and spoke windows, and only spokes j in [s_lo, s_hi) are walked
    const int32_t *hnbr, *snbr;
    const uint8_t *hbin, *sbin;
    int64_t hoff, soff;
    int windowed;
    int32_t s_lo, s_hi;
    int64_t hub_begin, hub_end;
    int nb;
    int ncfg;
    int hs;                       // byte-map walk: row stride of the b_ik index of its histogram (>= nb)
    unsigned long long *ghist;
    unsigned long long *cursor;   // next hub to hand out
    const uint16_t *cfg3;         // [nb][nb][nb] configuration index of (z, x, y) (SMEM_HIST)
    // hub-list mode: hubs given by input index; every triangle incident to a
    // listed hub is counted for it (the whole row is staged, not its forward part)
    const int32_t *hubs;          // [nhubs] input indices, or NULL
    const int32_t *inv;           // input -> internal index
    // weighted counts: weights in internal order; per-block 128-bit sums
    // [gridDim.x][ncfg][2] (low, high)
    const int16_t *w;
    unsigned long long *gsum;
    unsigned long long *slices;   // weighted: the caller's scratch of c3_slice_bytes() bytes
    unsigned *chk;                // checked builds: the graph's check word
    int64_t nbr_len;              // entries readable at snbr / sbin (checked builds)
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

// Configuration index of the sorted triple of (x, y, z), from the per-bin tables
// lex_a / lex_b: idx3(lo, mid, hi) = lex_a[lo] + lex_b[mid] + hi.
__device__ __forceinline__ int c3_index(int x, int y, int z, const int *lex_a, const int *lex_b)
{
    const int lo = min(x, min(y, z));
    const int hi = max(x, max(y, z));
    const int mid = x + y + z - lo - hi;
    return lex_a[lo] + lex_b[mid] + hi;
}

// Copy the z-slice of the configuration table (nb x nb u16) into this warp's
// shared-memory table.
__device__ __forceinline__ void c3_fill_tab(uint16_t *tab, const uint16_t *cfg3, int nb, int z)
{
    const int lane = threadIdx.x & 31;
    const uint16_t *src = cfg3 + (size_t)z * nb * nb;
    __syncwarp();
    for (int t = lane; t < nb * nb; t += 32) tab[t] = __ldg(src + t);
    __syncwarp();
}

// Exclusive block-wide scan of one int per thread (C3_THREADS threads).
__device__ __forceinline__ int c3_block_scan(int v, int *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < C3_WARPS ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < C3_WARPS) s_warp[lane] = w;
    }
    __syncthreads();
    const int r = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    __syncthreads();
    return r;
}

// Grouped walk, for graphs whose rows hold a few hundred entries: there a
// spoke's walk is one or two steps, and its time is the latency of the loads
// that start it (the spoke, its row bounds, its first step). So a warp walks
// four spokes at a time, eight lanes each: lane l of a group reads entries
// 4l .. 4l+3 of a 32-entry step, and four spokes' loads are in flight per warp.
// The four spokes' bins b_ij differ, so configurations come from the whole
// table [b_ij][b_ik][b_jk] in shared memory. Probes and hits are as in the
// one-spoke-per-warp walk of k_count3.
__device__ __forceinline__ void c3_walk_grouped(const C3Args &a, const int32_t *F, const uint8_t *FB, int sb,
                                                int ns, int c0, int32_t kfirst, int32_t kmax, int span,
                                                bool bmode, int shift, int mask, const unsigned *s_bm,
                                                const uint16_t *s_rank, const uint8_t *s_cbin,
                                                const int32_t *s_key, const uint8_t *s_bin, unsigned *s_hist,
                                                const uint16_t *s_full, int *s_next)
{
    const int lane = threadIdx.x & 31, grp = lane >> 3, gl = lane & 7;
    const int nb = a.nb;
    for (;;) {
        int li = 0;
        if (lane == 0) li = atomicAdd(s_next, 4);
        li = __shfl_sync(0xffffffffu, li, 0);
        if (li >= ns) break;
        li += grp;
        // this group's spoke j and the part [p0, pe) of N(j) it walks
        int64_t p0 = 0, pe = 0;
        int bij = 0;
        if (li < ns) {
            const int s = sb + li;
            const int32_t j = F[s];
            bij = FB[s];
            pe = a.row_ptr[j + 1];
            if (s + 1 >= c0) {
                p0 = a.row_ptr[j] + a.fwd[j];                  // first entry > j
            } else {
                int64_t lo = a.row_ptr[j] + a.fwd[j], hi = pe;  // first entry >= kfirst
                while (lo < hi) {
                    const int64_t mid = (lo + hi) >> 1;
                    if (a.snbr[mid] < kfirst) lo = mid + 1; else hi = mid;
                }
                p0 = lo;
            }
        }
        const int64_t pa = p0 & ~(int64_t)3;
        const int head = (int)(p0 - pa);
        const int total = p0 < pe ? head + (int)(pe - p0) : 0;
        const int4 *vk = reinterpret_cast<const int4 *>(a.snbr + pa) + gl;
        const uint32_t *vb = reinterpret_cast<const uint32_t *>(a.sbin + pa) + gl;
        const uint16_t *ztab = s_full + bij * nb * nb;
        int4 kk = make_int4(0, 0, 0, 0);
        uint32_t bb = 0;
        bool go = total > 0;                                   // the same in the eight lanes of a group
        if (go) {
            kk = __ldg(vk);
            bb = __ldg(vb);
        }
        for (int base = 0; __any_sync(0xffffffffu, go); base += 32) {
            const bool more = go && base + 32 < total;
            int4 kn = kk;
            uint32_t bn = bb;
            if (more) {                                        // next step in flight
                vk += 8;
                vb += 8;
                kn = __ldg(vk);
                bn = __ldg(vb);
            }
            if (go) {
                unsigned vmask = 0xfu;
                if (base == 0 || base + 32 > total) {
                    const int r0 = base + 4 * gl;
                    if (head > r0) vmask &= (0xfu << min(head - r0, 4)) & 0xfu;
                    if (total - r0 < 4) vmask &= (1u << max(total - r0, 0)) - 1u;
                }
                const int k[4] = { kk.x, kk.y, kk.z, kk.w };
                if (bmode) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kv = ((vmask >> e) & 1u) ? k[e] : kfirst - 1;
                        const unsigned o = min((unsigned)(kv - kfirst), (unsigned)span);
                        const unsigned w = s_bm[o >> 5];
                        if ((w >> (o & 31u)) & 1u) {
                            const int rank = s_rank[o >> 5] + __popc(w & ((1u << (o & 31u)) - 1u));
                            atomicAdd(&s_hist[ztab[s_cbin[rank] * nb + ((bb >> (8 * e)) & 0xffu)]], 1u);
                        }
                    }
                } else {
                    uint32_t h[4];
                    int32_t key[4];
                    unsigned pend = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        h[e] = gs_hash(k[e], shift);
                        key[e] = s_key[h[e]];
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) pend |= (unsigned)(key[e] != k[e] && key[e] != C3_EMPTY) << e;
                    while (pend) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if ((pend >> e) & 1u) {
                                h[e] = (h[e] + 1) & mask;
                                key[e] = s_key[h[e]];
                                if (key[e] == k[e] || key[e] == C3_EMPTY) pend &= ~(1u << e);
                            }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (((vmask >> e) & 1u) && key[e] == k[e])
                            atomicAdd(&s_hist[ztab[s_bin[h[e]] * nb + ((bb >> (8 * e)) & 0xffu)]], 1u);
                }
            }
            // rows are sorted: a group stops once its step's last key passes kmax
            const int last = __shfl_sync(0xffffffffu, kk.w, lane | 7);
            go = more && last <= kmax;
            kk = kn;
            bb = bn;
        }
    }
}

template <bool SMEM_HIST, bool HUB_LIST, bool WEIGHTED, bool WINDOWED, bool GROUPED = false>
__global__ void __launch_bounds__(C3_THREADS, C3_MAX_BLOCKS_PER_SM)
k_count3(C3Args a)
{
    // dynamic: the candidate-key region [C3_REGION bytes] (bitmap mode: bitmap,
    // per-pair ranks, chunk bins; hash mode: keys, bins), then (SMEM_HIST only)
    // the histogram [ncfg] u32 and one nb x nb u16 table per warp.
    // WEIGHTED: the region [C3_REGION_W bytes] also holds the weights (bitmap
    // mode: [C3_CHUNK_BM_W] after the bins; hash mode: [C3_TABLE] after the bins),
    // then the pass sums T [ncfg] int64
    extern __shared__ unsigned s_dyn[];
    __shared__ uint16_t s_order[C3_SPOKES];         // spoke positions grouped by b_ij
    __shared__ int s_next;                          // next entry of s_order to hand out
    __shared__ int s_bucket[257];
    __shared__ int s_lex_a[256];
    __shared__ int s_lex_b[256];
    __shared__ int s_warp[C3_WARPS];
    __shared__ long long s_hub;
    __shared__ unsigned long long s_pending;        // bound on hits since the last flush
    __shared__ int s_q[2];                          // windowed: spoke positions [q_lo, q_hi) of F

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = a.nb;
    // bitmap mode
    unsigned *s_bm = (unsigned *)s_dyn;                               // [C3_BM_WORDS] bits
    uint16_t *s_rank = (uint16_t *)(s_bm + C3_BM_WORDS);              // [C3_SPAN_WORDS] bits before the word
    constexpr int CHUNK_BM = WEIGHTED ? C3_CHUNK_BM_W : C3_CHUNK_BM;
    uint8_t *s_cbin = (uint8_t *)(s_rank + C3_SPAN_WORDS);            // [CHUNK_BM] bins in key order
    // hash mode
    int32_t *s_key = (int32_t *)s_dyn;
    uint8_t *s_bin = (uint8_t *)(s_key + C3_TABLE);
    unsigned *s_hist = (unsigned *)((char *)s_dyn + C3_REGION);
    uint16_t *tab = (uint16_t *)(s_hist + ((a.ncfg + 3) & ~3)) + warp * nb * nb;
    int tab_z = -1;
    // GROUPED: the whole configuration table [nb][nb][nb] in place of the per-warp tables
    uint16_t *s_full = (uint16_t *)(s_hist + ((a.ncfg + 3) & ~3));
    // weighted
    int16_t *s_cw = (int16_t *)(s_cbin + CHUNK_BM);                   // [CHUNK_BM] weights in key order
    int16_t *s_hw = (int16_t *)(s_bin + C3_TABLE);                    // [C3_TABLE] weights per slot
    unsigned long long *s_T = (unsigned long long *)((char *)s_dyn + C3_REGION_W);

    // idx3(a, b, c) = F(a) - G(a) + G(b) - b + c with F(a) = idx3(a, a, a) and
    // G(t) = t nb - t (t - 1) / 2, split into two per-bin tables.
    for (int t = threadIdx.x; t < nb; t += C3_THREADS) {
        const int64_t Gt = (int64_t)t * nb - (int64_t)t * (t - 1) / 2;
        s_lex_a[t] = (int)(gs_idx3(nb, t, t, t) - Gt);
        s_lex_b[t] = (int)(Gt - t);
    }
    if (WEIGHTED) {
        for (int t = threadIdx.x; t < a.ncfg; t += C3_THREADS) s_T[t] = 0ull;
    } else if (SMEM_HIST) {
        for (int t = threadIdx.x; t < a.ncfg; t += C3_THREADS) s_hist[t] = 0;
        if (GROUPED)
            for (int t = threadIdx.x; t < nb * nb * nb; t += C3_THREADS) s_full[t] = __ldg(a.cfg3 + t);
    }
    if (threadIdx.x == 0) s_pending = 0;
    __syncthreads();

    for (;;) {
        __syncthreads();                                     // everyone has read the last s_hub
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        if (s_hub >= a.hub_end) break;
        // forward row F = nbr[f0, f0 + f); in hub-list mode the whole row
        const long long i = HUB_LIST ? (long long)a.inv[a.hubs[s_hub]] : s_hub;
        const int64_t f0 = HUB_LIST ? a.row_ptr[i] : a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        const int64_t hoff = WINDOWED ? a.hoff : 0;
        const int32_t *F = a.hnbr + (f0 - hoff);            // the hub's row and its bins
        const uint8_t *FB = a.hbin + (f0 - hoff);
        const long long wi = WEIGHTED ? (long long)a.w[i] : 0;
        // spokes whose rows are walked: positions [q_lo, q_hi) of F (all of F
        // unless the graph is windowed; rows are sorted, so a window is a range)
        int q_lo = 0, q_hi = f;
        if (WINDOWED) {
            if (threadIdx.x == 0) {
                int lo = 0, hi = f;
                while (lo < hi) { const int m = (lo + hi) >> 1; if (F[m] < a.s_lo) lo = m + 1; else hi = m; }
                s_q[0] = lo;
                hi = f;
                while (lo < hi) { const int m = (lo + hi) >> 1; if (F[m] < a.s_hi) lo = m + 1; else hi = m; }
                s_q[1] = lo;
            }
            __syncthreads();
            q_lo = s_q[0];
            q_hi = s_q[1];
        }
        for (int c0 = 0, c1 = 0; c0 < f; c0 = c1) {         // chunks of candidate keys
            // a bitmap chunk of up to CHUNK_BM keys when their span fits, else a
            // C3_CHUNK-key chunk (bitmap if its span fits, else hash); block-uniform
            c1 = min(f, c0 + CHUNK_BM);
            bool bmode = (int64_t)F[c1 - 1] - F[c0] + 1 <= C3_SPAN_BITS;
            if (!bmode) {
                c1 = min(f, c0 + C3_CHUNK);
                bmode = (int64_t)F[c1 - 1] - F[c0] + 1 <= C3_SPAN_BITS;
            }
            const int cn = c1 - c0;
            if (c1 < 2) break;                               // a lone key closes nothing
            const int s_end = min(c1 - 1, q_hi);             // spokes [q_lo, s_end) meet this chunk
            if (s_end <= q_lo) continue;                     // block-uniform
            const int32_t kmax = F[c1 - 1];
            const int32_t kfirst = F[c0];
            const int64_t span64 = (int64_t)kmax - kfirst + 1;
            const int span = (int)(span64 < C3_SPAN_BITS ? span64 : C3_SPAN_BITS);
            int lg = 6;                                      // hash mode: 2^lg >= 4 cn slots
            while ((1 << lg) < 4 * cn) ++lg;
            const int tsize = 1 << lg, shift = 32 - lg, mask = tsize - 1;

            if (SMEM_HIST && !WEIGHTED) {
                // bound on the hits of this chunk: every spoke before c1 closes at
                // most cn triangles
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
            if (bmode) {
                // exact bitmap of the chunk's keys over [kfirst, kmax], the rank of
                // every 64-bit pair, and the chunk's bins in key order
                const int nwords = (span + 31) >> 5;
                // the word holding offset `span` stays zero: probes clamp to it
                for (int t = threadIdx.x; t <= nwords; t += C3_THREADS) s_bm[t] = 0u;
                __syncthreads();
                for (int t = threadIdx.x; t < cn; t += C3_THREADS) {
                    const int off = F[c0 + t] - kfirst;
                    atomicOr(s_bm + (off >> 5), 1u << (off & 31));
                    s_cbin[t] = FB[c0 + t];
                    if (WEIGHTED) s_cw[t] = a.w[off + kfirst];
                }
                __syncthreads();
                const int per = (nwords + C3_THREADS - 1) / C3_THREADS;
                const int q0 = threadIdx.x * per;
                int cnt = 0;
                for (int q = q0; q < min(nwords, q0 + per); ++q) cnt += __popc(s_bm[q]);
                int run = c3_block_scan(cnt, s_warp);
                for (int q = q0; q < min(nwords, q0 + per); ++q) {
                    s_rank[q] = (uint16_t)run;
                    run += __popc(s_bm[q]);
                }
            } else {
                for (int t = threadIdx.x; t < tsize; t += C3_THREADS) s_key[t] = C3_EMPTY;
                __syncthreads();
                for (int t = threadIdx.x; t < cn; t += C3_THREADS) {
                    const int32_t k = F[c0 + t];
                    uint32_t h = gs_hash(k, shift);
                    while (atomicCAS(&s_key[h], C3_EMPTY, k) != C3_EMPTY) h = (h + 1) & mask;
                    s_bin[h] = FB[c0 + t];
                    if (WEIGHTED) s_hw[h] = a.w[k];
                }
            }

            // spokes s in [sb, se) of [q_lo, s_end), at most C3_SPOKES at a time
            for (int sb = q_lo; sb < s_end; sb += C3_SPOKES) {
                const int se = min(s_end, sb + C3_SPOKES);
                const int ns = se - sb;
                if (GROUPED) {
                    if (threadIdx.x == 0) s_next = 0;
                    __syncthreads();
                    c3_walk_grouped(a, F, FB, sb, ns, c0, kfirst, kmax, span, bmode, shift, mask,
                                    s_bm, s_rank, s_cbin, s_key, s_bin, s_hist, s_full, &s_next);
                } else {
                    // counting sort of the spokes by b_ij, so that a warp's spokes
                    // share their bin and its configuration table changes rarely
                    for (int t = threadIdx.x; t <= nb; t += C3_THREADS) s_bucket[t] = 0;
                    __syncthreads();
                    for (int t = threadIdx.x; t < ns; t += C3_THREADS) atomicAdd(&s_bucket[FB[sb + t] + 1], 1);
                    __syncthreads();
                    if (warp == 0) {
                        int carry = 0;
                        for (int b0 = 0; b0 <= nb; b0 += 32) {
                            const int v = b0 + lane <= nb ? s_bucket[b0 + lane] : 0;
                            int x = v;
    #pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const int y = __shfl_up_sync(0xffffffffu, x, o);
                                if (lane >= o) x += y;
                            }
                            if (b0 + lane <= nb) s_bucket[b0 + lane] = carry + x;   // inclusive: bucket b starts at s_bucket[b]
                            carry += __shfl_sync(0xffffffffu, x, 31);
                        }
                    }
                    __syncthreads();
                    for (int t = threadIdx.x; t < ns; t += C3_THREADS) {
                        const int b = FB[sb + t];
                        s_order[atomicAdd(&s_bucket[b], 1)] = (uint16_t)t;
                    }
                    if (threadIdx.x == 0) s_next = 0;
                    __syncthreads();

                    for (;;) {
                        int li = 0;
                        if (lane == 0) li = atomicAdd(&s_next, 1);
                        li = __shfl_sync(0xffffffffu, li, 0);
                        if (li >= ns) break;
                        const int s = sb + s_order[li];
                        const int32_t j = F[s];
                        const int bij = FB[s];
                        if (SMEM_HIST && !WEIGHTED && bij != tab_z) {
                            c3_fill_tab(tab, a.cfg3, nb, bij);
                            tab_z = bij;
                        }
                        const int64_t pe = a.row_ptr[j + 1];
                        int64_t p0;
                        if (s + 1 >= c0) {
                            p0 = a.row_ptr[j] + a.fwd[j];                  // first entry > j
                        } else {
                            // first entry >= kfirst in N(j) (lower bound; only for later chunks)
                            int64_t lo = a.row_ptr[j] + a.fwd[j], hi = pe;
                            while (lo < hi) {
                                const int64_t mid = (lo + hi) >> 1;
                                if (a.snbr[mid - (WINDOWED ? a.soff : 0)] < kfirst) lo = mid + 1; else hi = mid;
                            }
                            p0 = lo;
                        }
                        if (p0 >= pe) continue;
                        const int wj = WEIGHTED ? (int)a.w[j] : 0;
                        // one triangle with sides (b_ij, b_ik, b_jk) and third vertex weight wk
                        auto hit = [&](int bik, int bjk, int wk) {
                            if (WEIGHTED) {
                                // T[c] += w_j w_k (|.| <= 2^30) as a 64-bit integer held in two
                                // 32-bit words: add to the low word, then the carry out of it
                                // plus the sign extension to the high word (zero, and skipped,
                                // for most adds)
                                unsigned *q = reinterpret_cast<unsigned *>(s_T + c3_index(bij, bik, bjk, s_lex_a, s_lex_b));
                                const int p = wj * wk;
                                const unsigned old = atomicAdd(q, (unsigned)p);
                                const unsigned up = (old + (unsigned)p < old ? 1u : 0u) + (p < 0 ? ~0u : 0u);
                                if (up) atomicAdd(q + 1, up);
                            }
                            else if (SMEM_HIST) {
                                const int c = tab[bik * nb + bjk];
                                if (GS_DCHECK(bik < nb && bjk < nb && c < a.ncfg, a.chk, GS_SITE_C3_HIST))
                                    atomicAdd(&s_hist[c], 1u);
                            }
                            else atomicAdd(a.ghist + c3_index(bij, bik, bjk, s_lex_a, s_lex_b), 1ull);
                        };
                        // Walk nbr[p0, pe) in aligned 128-entry steps: lane l reads entries
                        // 4l .. 4l+3 of the step as one int4 and their bins as one word.
                        const int64_t pa = p0 & ~(int64_t)3;
                        const int head = (int)(p0 - pa);
                        const int total = head + (int)(pe - p0);
                        const int64_t soff = WINDOWED ? a.soff : 0;
                        const int4 *vk = reinterpret_cast<const int4 *>(a.snbr + (pa - soff)) + lane;
                        const uint32_t *vb = reinterpret_cast<const uint32_t *>(a.sbin + (pa - soff)) + lane;
                        int4 kk = __ldg(vk);                            // step 0, then prefetch
                        uint32_t bb = __ldg(vb);
                        for (int base = 0; base < total; base += 128) {
                            vk += 32;
                            vb += 32;
                            int4 kn = kk;
                            uint32_t bn = bb;
                            if (base + 128 < total) {                  // next step in flight
                                kn = __ldg(vk);
                                bn = __ldg(vb);
                            }
                            unsigned vmask = 0xfu;
                            if (base == 0 || base + 128 > total) {     // first / last step only
                                const int r0 = base + 4 * lane;
                                if (head > r0) vmask &= (0xfu << min(head - r0, 4)) & 0xfu;
                                if (total - r0 < 4) vmask &= (1u << max(total - r0, 0)) - 1u;
                            }
                            const int k[4] = { kk.x, kk.y, kk.z, kk.w };
                            if (bmode) {
                                // entries outside [p0, pe) (first and last step) become kfirst - 1;
                                // every offset outside [0, span) clamps to the zero guard bit at span
                                int kv[4] = { k[0], k[1], k[2], k[3] };
                                if (vmask != 0xfu) {
    #pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        if (!((vmask >> e) & 1u)) kv[e] = kfirst - 1;
                                }
    #pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const unsigned o = min((unsigned)(kv[e] - kfirst), (unsigned)span);
                                    const unsigned w = s_bm[o >> 5];
                                    if ((w >> (o & 31u)) & 1u) {
                                        const int rank = s_rank[o >> 5] + __popc(w & ((1u << (o & 31u)) - 1u));
                                        if (GS_DCHECK(rank < cn, a.chk, GS_SITE_C3_BITMAP))
                                            hit(s_cbin[rank], (bb >> (8 * e)) & 0xffu, WEIGHTED ? s_cw[rank] : 0);
                                    }
                                }
                            } else {
                                uint32_t h[4];
                                int32_t key[4];
                                unsigned pend = 0;
    #pragma unroll
                                for (int e = 0; e < 4; ++e) {          // first probes, all in flight
                                    h[e] = gs_hash(k[e], shift);
                                    key[e] = s_key[h[e]];
                                }
    #pragma unroll
                                for (int e = 0; e < 4; ++e) pend |= (unsigned)(key[e] != k[e] && key[e] != C3_EMPTY) << e;
                                while (pend) {                         // collisions
    #pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        if ((pend >> e) & 1u) {
                                            h[e] = (h[e] + 1) & mask;
                                            key[e] = s_key[h[e]];
                                            if (key[e] == k[e] || key[e] == C3_EMPTY) pend &= ~(1u << e);
                                        }
                                }
    #pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (((vmask >> e) & 1u) && key[e] == k[e])
                                        hit(s_bin[h[e]], (bb >> (8 * e)) & 0xffu, WEIGHTED ? s_hw[h[e]] : 0);
                            }
                            // rows are sorted: stop once the step's last key passes kmax
                            if (__shfl_sync(0xffffffffu, kk.w, 31) > kmax) break;
                            kk = kn;
                            bb = bn;
                        }
                    }
                }
                __syncthreads();
                if (WEIGHTED) {
                    // slice[t] += w_i T[t] (128-bit); thread t owns configuration t
                    unsigned long long *slice = a.gsum + 2 * (size_t)a.ncfg * blockIdx.x;
                    for (int t = threadIdx.x; t < a.ncfg; t += C3_THREADS) {
                        const long long v = (long long)s_T[t];
                        if (v) {
                            s_T[t] = 0ull;
                            const unsigned long long lo = (unsigned long long)(wi * v);
                            const unsigned long long hi = (unsigned long long)__mul64hi(wi, v);
                            const unsigned long long l0 = slice[2 * t];
                            slice[2 * t] = l0 + lo;
                            slice[2 * t + 1] += hi + (l0 + lo < l0 ? 1ull : 0ull);
                        }
                    }
                }
            }
        }
    }
    if (SMEM_HIST && !WEIGHTED) {
        __syncthreads();
        c3_flush(s_hist, a.ncfg, a.ghist);
    }
}

// ---------------------------------------------------------------- byte-map walk
//
// The walk for long rows, one spoke per warp, with fewer instructions per
// triangle than the bitmap-and-rank lookup of k_count3. The count is bound by
// instruction issue: there a closed triangle costs a membership probe, a rank,
// a bin load, a configuration-table load and the atomic. Here:
//
//   * the chunk's keys are held as a byte map: the key span is cut into
//     segments of C3M_SEG ids, a segment table gives each segment that holds
//     a key a slot of C3M_SEG bytes, and byte k of a slot is b_ik (C3M_ABSENT
//     when k is not a key). A probe is two dependent shared loads and yields
//     the bin together with the membership;
//   * hits go to an unsorted histogram H[b_ij][b_ik][b_jk] of nb^3 counters,
//     addressed with two multiply-adds, so no configuration table is read per
//     triangle and spokes need not be grouped by bin. The block folds the
//     permutations of each sorted triple into the caller's histogram when a
//     counter could overflow and when it exits.
//
// A chunk ends before the first key that would need more segment slots than
// the block holds, or that lies C3M_SPAN_SEGS segments or more past the first
// key's segment. So every chunk is a byte-map chunk (there is no hash mode):
// a forward row that wraps a periodic box simply runs as two chunks.
constexpr int C3M_SEG_LOG = 10;
constexpr int C3M_SEG = 1 << C3M_SEG_LOG;        // ids per segment
constexpr int C3M_SPAN_SEGS = 256;               // segments a chunk may span (2^18 ids)
constexpr int C3M_SEG_TABLE = C3M_SPAN_SEGS + 16;  // + the guard entry (0: the absent slot), padded
// Catalogues of at most C3M_ABS_SEGS segments of ids index the segment table by
// the absolute segment k >> C3M_SEG_LOG: no subtraction and no clamp per probe
// (an entry outside its row is replaced by the guard id, whose segment is absent).
constexpr int C3M_ABS_SEGS = 2048;               // ids below 2^21
constexpr int C3M_SEG_TABLE_ABS = C3M_ABS_SEGS + 16;
constexpr int C3M_KEYS_PER_THREAD = 8;           // chunk keys per thread
constexpr int C3M_MIN_SLOTS = 24;                // fewest segment slots worth a launch
constexpr int C3M_MAX_SLOTS = 255;               // slot numbers are bytes
constexpr int C3M_MAX_BINS = 32;                 // nb^3 u32 counters must fit beside the map
constexpr unsigned C3M_ABSENT = 0xffu;

// Exclusive scan of one int per thread over a block of THREADS threads; *total
// receives the sum.
template <int THREADS>
__device__ __forceinline__ int c3m_block_scan(int v, int *s_warp, int *total)
{
    constexpr int WARPS = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < WARPS ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < WARPS) s_warp[lane] = w;
    }
    __syncthreads();
    const int r = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[WARPS - 1];
    __syncthreads();
    return r;
}

// Fold the unsorted counters into the caller's sorted-triple histogram and
// clear them: the thread that meets the sorted triple x <= y <= z sums its
// distinct permutations (cfg3 at (x, y, z) is its packed index).
template <int THREADS>
__device__ __forceinline__ void c3m_flush(unsigned *h, int nb, int hs, const uint16_t *cfg3, unsigned long long *gh)
{
    const int nb2 = nb * nb, n3 = nb2 * nb;
    for (int u = threadIdx.x; u < n3; u += THREADS) {
        const int x = u / nb2, y = (u / nb) % nb, z = u % nb;
        if (x > y || y > z) continue;
        const int p[6] = { (x * nb + y) * hs + z, (x * nb + z) * hs + y, (y * nb + x) * hs + z,
                           (y * nb + z) * hs + x, (z * nb + x) * hs + y, (z * nb + y) * hs + x };
        unsigned long long v = 0;
#pragma unroll
        for (int q = 0; q < 6; ++q) {
            bool dup = false;
#pragma unroll
            for (int r = 0; r < q; ++r) dup |= p[r] == p[q];
            if (!dup) {
                v += h[p[q]];
                h[p[q]] = 0;
            }
        }
        if (v) atomicAdd(gh + __ldg(cfg3 + u), v);
    }
}

// The part [*p0, *pe) of N(j) that spoke s (j = F[s]) walks against the chunk
// starting at c0 (first key kfirst): from the first entry beyond j, or, for a
// spoke of an earlier chunk, from the first entry >= kfirst (binary search).
// First position of the sorted row F[0, f) whose id is >= key, found by the 32
// lanes of a warp together: each round probes 32 evenly spaced positions, so
// a row of up to 32^r entries takes r + 1 dependent loads.
__device__ __forceinline__ int c3m_warp_lower_bound(const int32_t *F, int f, int32_t key)
{
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = f;                                      // the answer lies in [lo, hi]
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) >> 5;
        const int p = lo + lane * step;
        const int c = __popc(__ballot_sync(0xffffffffu, p < hi && F[p] < key));   // probes below key
        const int nlo = c > 0 ? lo + (c - 1) * step + 1 : lo;
        hi = min(hi, lo + c * step);
        lo = nlo;
    }
    const int p = lo + lane;
    return lo + __popc(__ballot_sync(0xffffffffu, p < hi && F[p] < key));
}

// Spoke rows are read at e - soff (a staged window of a windowed graph, else 0).
__device__ __forceinline__ void c3m_spoke_range(const C3Args &a, int64_t soff, int32_t j, int s, int c0,
                                                int32_t kfirst, int64_t *p0, int64_t *pe)
{
    *pe = a.row_ptr[j + 1];
    if (s + 1 >= c0) {
        *p0 = a.row_ptr[j] + a.fwd[j];
    } else {
        int64_t lo = a.row_ptr[j] + a.fwd[j], hi = *pe;
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (a.snbr[mid - soff] < kfirst) lo = mid + 1; else hi = mid;
        }
        *p0 = lo;
    }
}

// Probe N row entries against the chunk's byte map and count the hits into
// H[b_ij][b_ik][b_jk] at (b_ij nb + b_ik) hs + b_jk (hb = b_ij nb hs; bins of
// entries 4q .. 4q+3 in bb[q]).
// ABS: the segment table is indexed by the absolute segment of k (kbase 0,
// every k below the guard id), so the offset needs no clamp.
// The segment slots of all N entries are loaded first, then their bin bytes,
// then the adds are issued: the two dependent shared loads of one entry
// overlap those of the others. The adds touch only the histogram, which
// nothing in the walk reads (it is read after a block barrier), so they carry
// no memory clobber and the loads may be scheduled around them.
template <bool ABS, int N>
__device__ __forceinline__ void c3m_probe(const int *k, const uint32_t *bb, int32_t kbase, unsigned guard,
                                          const uint8_t *s_seg, const uint8_t *s_map, unsigned *s_h, int hb,
                                          int nb, int hs, const C3Args &a, int nslots)
{
#ifdef GS_CHECKED
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const unsigned o = ABS ? (unsigned)k[e] : min((unsigned)(k[e] - kbase), guard);
        const unsigned sl = s_seg[o >> C3M_SEG_LOG];
        if (!GS_DCHECK(sl <= (unsigned)nslots, a.chk, GS_SITE_C3M_MAP_R)) continue;
        const unsigned b = s_map[(sl << C3M_SEG_LOG) | (o & (C3M_SEG - 1))];
        if (b == C3M_ABSENT) continue;
        const int idx = hb + (int)b * hs + (int)((bb[e >> 2] >> (8 * (e & 3))) & 0xffu);
        if (GS_DCHECK(b < (unsigned)nb && idx >= 0 && idx < nb * nb * hs, a.chk, GS_SITE_C3M_HIST))
            atomicAdd(s_h + idx, 1u);
    }
#else
    (void)a;
    (void)nslots;
    (void)nb;
    unsigned o[N], v[N];
#pragma unroll
    for (int e = 0; e < N; ++e) o[e] = ABS ? (unsigned)k[e] : min((unsigned)(k[e] - kbase), guard);
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = s_seg[o[e] >> C3M_SEG_LOG];
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = s_map[v[e] * C3M_SEG + (o[e] & (C3M_SEG - 1))];
    const unsigned h0 = (unsigned)__cvta_generic_to_shared(s_h) + 4u * (unsigned)hb;
    const unsigned nb4 = 4u * (unsigned)hs;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        // a predicated reduction, no branch: a lane whose entry is absent adds nothing
        const unsigned addr = h0 + v[e] * nb4 + 4u * __byte_perm(bb[e >> 2], 0u, 0x4440u + (unsigned)(e & 3));
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 255;\n\t@p red.shared.add.u32 [%1], 1;\n\t}"
                     :: "r"(v[e]), "r"(addr));
    }
#endif
}

// One 256-entry step of a spoke's walk in the one-spoke-per-warp form: cur
// holds the step's entries (lane l: 4l .. 4l+3 in k0/b0, 128+4l .. in k1/b1);
// the next step, when it starts before the row's end, is loaded into nxt.
// Entries outside the row (the first step's head, the last step's tail)
// become kout, an id of an absent segment. True when the spoke's walk ends:
// at the row's end, or once a loaded key passes kmax (rows are sorted, so no
// later entry is a key of the chunk).
struct C3MStep {
    int4 k0, k1;
    uint32_t b0, b1;
};

template <bool ABS>
__device__ __forceinline__ bool c3m_step(const C3MStep &cur, C3MStep &nxt, const int4 *&vk, const uint32_t *&vb,
                                         int base, int total_e, int head, int lane, int32_t kmax, int32_t kout,
                                         int32_t kbase, unsigned guard, const uint8_t *s_seg, const uint8_t *s_map,
                                         unsigned *s_h, int hb, int nb, int hs, const C3Args &a, int nslots)
{
    const bool more = base + 256 < total_e;                  // the same in every lane
    if (more) {
        vk += 64;
        vb += 64;
        nxt.k0 = __ldg(vk);
        nxt.b0 = __ldg(vb);
        nxt.k1 = __ldg(vk + 32);
        nxt.b1 = __ldg(vb + 32);
    }
    int k[8] = { cur.k0.x, cur.k0.y, cur.k0.z, cur.k0.w, cur.k1.x, cur.k1.y, cur.k1.z, cur.k1.w };
    const uint32_t bb[2] = { cur.b0, cur.b1 };
    if (base == 0 || !more) {
        const unsigned r0 = (unsigned)(base + 4 * lane - head), len = (unsigned)(total_e - head);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            k[e] = r0 + e < len ? k[e] : kout;
            k[4 + e] = r0 + 128 + e < len ? k[4 + e] : kout;
        }
    }
    // once the first half's last key passes kmax, the second half holds no key
    // (lane 31 holds it; a vote, not a shuffle: shuffles take slots of the
    // shared-memory pipe that the probes use)
    if (__any_sync(0xffffffffu, lane == 31 && cur.k0.w > kmax)) {
        c3m_probe<ABS, 4>(k, bb, kbase, guard, s_seg, s_map, s_h, hb, nb, hs, a, nslots);
        return true;
    }
    c3m_probe<ABS, 8>(k, bb, kbase, guard, s_seg, s_map, s_h, hb, nb, hs, a, nslots);
    return !more || __any_sync(0xffffffffu, lane == 31 && cur.k1.w > kmax);
}

// Four spokes per warp, eight lanes each (for rows of a few hundred entries,
// where a spoke's walk is one or two steps and its time is the latency of the
// loads that start it): lane l of a group reads entries 4l .. 4l+3 of a
// 32-entry step of its spoke's row. Each group stops once its step passes kmax.
template <bool ABS>
__device__ __forceinline__ void c3m_walk_grouped(const C3Args &a, int64_t soff, const int32_t *F, const uint8_t *FB,
                                                 int s_lo, int s_end, int c0, int32_t kfirst, int32_t kbase,
                                                 int32_t kmax, unsigned guard, const uint8_t *s_seg,
                                                 const uint8_t *s_map, unsigned *s_h, int *s_next, int nslots)
{
    const int lane = threadIdx.x & 31, grp = lane >> 3, gl = lane & 7;
    const int nb = a.nb, hs = a.hs, nbhs = nb * hs;
    const int32_t kout = ABS ? (int32_t)guard : kbase - 1;   // an id whose segment is absent
    for (;;) {
        int li = 0;
        if (lane == 0) li = s_lo + atomicAdd(s_next, 4);
        li = __shfl_sync(0xffffffffu, li, 0);
        if (li >= s_end) break;
        const int s = li + grp;
        int64_t p0 = 0, pe = 0;
        int hb = 0;
        if (s < s_end) {
            c3m_spoke_range(a, soff, F[s], s, c0, kfirst, &p0, &pe);
            hb = FB[s] * nbhs;
        }
        const int64_t pa = p0 & ~(int64_t)3;
        const int head = (int)(p0 - pa);
        const int total = p0 < pe ? head + (int)(pe - p0) : 0;
        const int4 *vk = reinterpret_cast<const int4 *>(a.snbr + (pa - soff)) + gl;
        const uint32_t *vb = reinterpret_cast<const uint32_t *>(a.sbin + (pa - soff)) + gl;
        int4 kk = make_int4(0, 0, 0, 0);
        uint32_t bb = 0;
        // checked builds: the group's last vector of the row lies in the readable array
        bool go = total > 0 && GS_DCHECK((pa - soff) + (((total + 31) >> 5) << 5) <= a.nbr_len, a.chk, GS_SITE_C3M_ROW);
        if (go) {
            kk = __ldg(vk);
            bb = __ldg(vb);
        }
        for (int base = 0; __any_sync(0xffffffffu, go); base += 32) {
            const bool more = go && base + 32 < total;
            int4 kn = kk;
            uint32_t bn = bb;
            if (more) {                                      // next step in flight
                vk += 8;
                vb += 8;
                kn = __ldg(vk);
                bn = __ldg(vb);
            }
            if (go) {
                int k[4] = { kk.x, kk.y, kk.z, kk.w };
                if (base == 0 || base + 32 > total) {
                    const unsigned r0 = (unsigned)(base + 4 * gl - head), len = (unsigned)(total - head);
#pragma unroll
                    for (int e = 0; e < 4; ++e) k[e] = r0 + e < len ? k[e] : kout;
                }
                c3m_probe<ABS, 4>(k, &bb, kbase, guard, s_seg, s_map, s_h, hb, nb, hs, a, nslots);
            }
            // rows are sorted: a group stops once its step's last key passes kmax
            const int last = __shfl_sync(0xffffffffu, kk.w, lane | 7);
            go = more && last <= kmax;
            kk = kn;
            bb = bn;
        }
    }
}

template <int THREADS, bool GROUPED, bool WINDOWED, bool ABS>
__global__ void __launch_bounds__(THREADS, THREADS >= 1024 ? 1 : 2)
k_count3m(C3Args a, int nslots)
{
    constexpr int WARPS = THREADS / 32;
    constexpr int KPT = C3M_KEYS_PER_THREAD;
    constexpr int MAX_KEYS = THREADS * KPT;
    // dynamic: segment table [C3M_SEG_TABLE] u8, map [(nslots + 1) * C3M_SEG] u8
    // (slot 0: the all-absent segment), histogram [nb][nb][hs] u32
    extern __shared__ unsigned s_dyn[];
    __shared__ int s_next;
    __shared__ int s_cut;
    __shared__ int s_warp[WARPS];
    __shared__ long long s_hub;
    __shared__ unsigned long long s_pending;        // bound on the counts added since the last flush
    __shared__ int s_q[2];                          // windowed: spoke positions [q_lo, q_hi) of F

    const int lane = threadIdx.x & 31;
    const int nb = a.nb, hs = a.hs, nbhs = nb * hs, nh = nb * nbhs;
    const int64_t soff = WINDOWED ? a.soff : 0;
    // the segment table and the map first, at fixed offsets (their probes need
    // no base register), then the histogram
    constexpr int SEG_TABLE = ABS ? C3M_SEG_TABLE_ABS : C3M_SEG_TABLE;
    constexpr int SPAN_SEGS = ABS ? C3M_ABS_SEGS : C3M_SPAN_SEGS;
    uint8_t *s_seg = reinterpret_cast<uint8_t *>(s_dyn);
    uint8_t *s_map = s_seg + SEG_TABLE;
    unsigned *s_h = reinterpret_cast<unsigned *>(s_map + (size_t)(nslots + 1) * C3M_SEG);

    for (int t = threadIdx.x; t < nh; t += THREADS) s_h[t] = 0;
    for (int t = threadIdx.x; t < C3M_SEG / 16; t += THREADS)
        reinterpret_cast<uint4 *>(s_map)[t] = make_uint4(~0u, ~0u, ~0u, ~0u);
    if (threadIdx.x == 0) s_pending = 0;

    for (;;) {
        __syncthreads();                                     // everyone has read the last s_hub
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        if (s_hub >= a.hub_end) break;
        const long long i = s_hub;
        const int64_t f0 = a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        if (f < 2) continue;                                 // fewer than two forward keys close nothing
        const int64_t hoff = WINDOWED ? a.hoff : 0;
        const int32_t *F = a.hnbr + (f0 - hoff);             // the hub's forward row and its bins
        const uint8_t *FB = a.hbin + (f0 - hoff);
        // spokes whose rows are walked: positions [q_lo, q_hi) of F (all of F
        // unless the graph is windowed; rows are sorted, so a window is a range)
        int q_lo = 0, q_hi = f;
        if (WINDOWED) {
            if (threadIdx.x < 32) {
                // rows are sorted: the tile's spokes [s_lo, s_hi) are one range of F
                const int lo = F[f - 1] < a.s_lo ? f : c3m_warp_lower_bound(F, f, a.s_lo);
                const int hi = lo >= f ? f : c3m_warp_lower_bound(F, f, a.s_hi);
                if (threadIdx.x == 0) {
                    s_q[0] = lo;
                    s_q[1] = hi;
                }
            }
            __syncthreads();
            q_lo = s_q[0];
            q_hi = s_q[1];
            if (q_lo >= q_hi || q_lo >= f - 1) continue;     // no spoke of this tile (block-uniform)
        }
        for (int c0 = 0, c1 = 0; c0 < f; c0 = c1) {
            // ---- the chunk [c0, c1); thread t owns keys c0 + KPT t .. + KPT - 1
            const int32_t kbase = ABS ? 0 : F[c0] & ~(C3M_SEG - 1);
            const int cap = min(f, c0 + MAX_KEYS);
            const int t0 = c0 + threadIdx.x * KPT;
            int32_t key[KPT];
            unsigned starts = 0;                             // bit q: key q opens a segment
            int32_t prev = (t0 > c0 && t0 < cap) ? (F[t0 - 1] - kbase) >> C3M_SEG_LOG : -1;
#pragma unroll
            for (int q = 0; q < KPT; ++q) {
                key[q] = t0 + q < cap ? F[t0 + q] : 0;
                const int32_t sg = (key[q] - kbase) >> C3M_SEG_LOG;
                if (t0 + q < cap && sg != prev) starts |= 1u << q;
                prev = sg;
            }
            if (threadIdx.x == 0) s_cut = cap;
            int total = 0;
            // slot of a key = the number of segments opened from c0 through it
            const int sbase = c3m_block_scan<THREADS>(__popc(starts), s_warp, &total);
            {
                int slot = sbase;
#pragma unroll
                for (int q = 0; q < KPT; ++q) {
                    if (t0 + q >= cap) break;
                    slot += (starts >> q) & 1u;
                    if (slot > nslots || ((key[q] - kbase) >> C3M_SEG_LOG) >= SPAN_SEGS) {
                        atomicMin(&s_cut, t0 + q);           // slots and segments grow with q
                        break;
                    }
                }
            }
            // clear the segment table and the slots the chunk can use
            for (int t = threadIdx.x; t < SEG_TABLE; t += THREADS) s_seg[t] = 0;
            {
                const int nclear = min(nslots, total);
                uint4 *m = reinterpret_cast<uint4 *>(s_map + C3M_SEG);
                for (int t = threadIdx.x; t < nclear * (C3M_SEG / 16); t += THREADS)
                    m[t] = make_uint4(~0u, ~0u, ~0u, ~0u);
            }
            __syncthreads();
            c1 = s_cut;
            {
                int slot = sbase;
#pragma unroll
                for (int q = 0; q < KPT; ++q) {
                    if (t0 + q >= c1) break;
                    slot += (starts >> q) & 1u;
                    const int off = key[q] - kbase;
                    if (!GS_DCHECK(slot >= 1 && slot <= nslots && off >= 0 && (off >> C3M_SEG_LOG) < SPAN_SEGS,
                                   a.chk, GS_SITE_C3M_MAP_W))
                        continue;
                    if ((starts >> q) & 1u) s_seg[off >> C3M_SEG_LOG] = (uint8_t)slot;
                    s_map[(slot << C3M_SEG_LOG) | (off & (C3M_SEG - 1))] = FB[t0 + q];
                }
            }
            const int s_end = min(c1 - 1, q_hi);             // spokes [q_lo, s_end) meet this chunk
            const int cn = c1 - c0;
            // bound on the counts of this chunk: every spoke before c1 closes at
            // most cn triangles; flush first if a counter could pass 2^32 - 1
            const unsigned long long bound = (unsigned long long)c1 * cn;
            const bool flush = s_pending + bound > 0xffffffffull;   // the same in every thread
            __syncthreads();                                 // s_pending read; the map is written
            if (flush) {
                c3m_flush<THREADS>(s_h, nb, hs, a.cfg3, a.ghist);
                __syncthreads();
            }
            if (threadIdx.x == 0) {
                s_pending = (flush ? 0ull : s_pending) + bound;
                s_next = 0;
            }
            __syncthreads();
            if (s_end <= q_lo) continue;
            const int32_t kmax = F[c1 - 1];
            const int32_t kfirst = F[c0];
            const unsigned guard = (unsigned)SPAN_SEGS << C3M_SEG_LOG;   // an id of the absent guard segment
            const int32_t kout = ABS ? (int32_t)guard : kbase - 1;      // what entries outside the row become

            if (GROUPED) {
                c3m_walk_grouped<ABS>(a, soff, F, FB, q_lo, s_end, c0, kfirst, kbase, kmax, guard, s_seg, s_map,
                                      s_h, &s_next, nslots);
            } else {
                // ---- spokes, one per warp, handed out in row order
                for (;;) {
                    int s = 0;
                    if (lane == 0) s = q_lo + atomicAdd(&s_next, 1);
                    s = __shfl_sync(0xffffffffu, s, 0);
                    if (s >= s_end) break;
                    int64_t p0, pe;
                    c3m_spoke_range(a, soff, F[s], s, c0, kfirst, &p0, &pe);
                    const int hb = FB[s] * nbhs;
                    if (p0 >= pe) continue;
                    // walk nbr[p0, pe) in aligned 256-entry steps: lane l reads entries
                    // 4l .. 4l+3 and 128+4l .. 128+4l+3 of a step as two int4 and their
                    // bins as two words (the arrays hold GS_EDGE_PAD = 256 entries past
                    // the last row, so a step that starts before the row's end is read
                    // whole); two step buffers take turns, the next step in flight
                    const int64_t pa = p0 & ~(int64_t)3;
                    const int head = (int)(p0 - pa);
                    const int total_e = head + (int)(pe - p0);
                    // checked builds: the walk's last loaded step lies in the readable array
                    if (!GS_DCHECK((pa - soff) + (((total_e + 255) >> 8) << 8) <= a.nbr_len, a.chk, GS_SITE_C3M_ROW))
                        continue;
                    const int4 *vk = reinterpret_cast<const int4 *>(a.snbr + (pa - soff)) + lane;
                    const uint32_t *vb = reinterpret_cast<const uint32_t *>(a.sbin + (pa - soff)) + lane;
                    C3MStep A, B;
                    A.k0 = __ldg(vk);
                    A.b0 = __ldg(vb);
                    A.k1 = __ldg(vk + 32);
                    A.b1 = __ldg(vb + 32);
                    for (int base = 0;; base += 512) {
                        if (c3m_step<ABS>(A, B, vk, vb, base, total_e, head, lane, kmax, kout, kbase, guard, s_seg,
                                          s_map, s_h, hb, nb, hs, a, nslots))
                            break;
                        if (c3m_step<ABS>(B, A, vk, vb, base + 256, total_e, head, lane, kmax, kout, kbase, guard,
                                          s_seg, s_map, s_h, hb, nb, hs, a, nslots))
                            break;
                    }
                }
            }
            __syncthreads();                                 // the chunk's map is no longer read
        }
    }
    __syncthreads();
    c3m_flush<THREADS>(s_h, nb, hs, a.cfg3, a.ghist);
}

// ---------------------------------------------------------------- weighted byte-map walk
//
// The weighted 3pCF (for every configuration the exact sum of w_i w_j w_k over
// its triangles, §II.1) on the byte-map walk, for device-resident graphs with
// at most C3M_MAX_BINS bins; k_count3<..., WEIGHTED> (bitmap walk) serves the
// rest. The chunk's keys are held as in k_count3m (a byte map of their bins)
// and, in a parallel map with the same slots, as their int16 weights. A hit
// adds w_j w_k (|.| <= 2^30) to the hub's sum T[c], c read from the nb^3
// configuration table in shared memory; T[c] is an int64 held as two 32-bit
// words, one shared add on the low word and a second, on the high word, only
// on a carry or borrow. A hub closes at most f (f - 1) / 2 triangles, and
// the kernel serves graphs whose forward rows hold fewer than 2^16 keys, so
// |T| < 2^61. After the hub's last chunk the block adds w_i T[c], an exact
// 128-bit product, into its own slice (each configuration has one owner
// thread, no atomics) and clears T; k_sum128_slices adds the slices. Spokes
// are walked one per warp in 256-entry steps.

// T[c] += p for the (low, high) word pair q of an int64 sum.
__device__ __forceinline__ void c3w_add64(unsigned *q, int p)
{
    const unsigned pu = (unsigned)p;
    const unsigned old = atomicAdd(q, pu);
    const unsigned up = (old + pu < old ? 1u : 0u) + (p < 0 ? ~0u : 0u);   // carry, plus the sign extension
    if (up) atomicAdd(q + 1, up);
}

// Probe the eight entries of a step (lane l: 4l .. 4l+3 in k[0..3], 128+4l ..
// in k[4..7], their bins in bb[0], bb[1]); a hit adds w_j w_k to T.
template <bool ABS>
__device__ __forceinline__ void c3w_probe8(const int *k, const uint32_t *bb, int32_t kbase, unsigned guard,
                                           const uint8_t *s_seg, const uint8_t *s_map, const int16_t *s_wmap,
                                           const uint16_t *s_cfg, unsigned *s_T, int hb, int nb, int wj,
                                           const C3Args &a, int nslots)
{
    unsigned o[8], sl[8], v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = ABS ? (unsigned)k[e] : min((unsigned)(k[e] - kbase), guard);
#pragma unroll
    for (int e = 0; e < 8; ++e) sl[e] = s_seg[o[e] >> C3M_SEG_LOG];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (!GS_DCHECK(sl[e] <= (unsigned)nslots, a.chk, GS_SITE_C3M_MAP_R)) sl[e] = 0;
        v[e] = s_map[sl[e] * C3M_SEG + (o[e] & (C3M_SEG - 1))];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (v[e] == C3M_ABSENT) continue;
        const int bjk = (int)((bb[e >> 2] >> (8 * (e & 3))) & 0xffu);
        const int u = hb + (int)v[e] * nb + bjk;
        if (!GS_DCHECK(v[e] < (unsigned)nb && u >= 0 && u < nb * nb * nb, a.chk, GS_SITE_C3M_HIST)) continue;
        const int c = s_cfg[u];
        const int wk = s_wmap[sl[e] * C3M_SEG + (o[e] & (C3M_SEG - 1))];
        if (GS_DCHECK(c < a.ncfg, a.chk, GS_SITE_C3M_HIST)) c3w_add64(s_T + 2 * c, wj * wk);
    }
}

template <int THREADS, bool ABS>
__global__ void __launch_bounds__(THREADS, 1)
k_count3mw(C3Args a, int nslots)
{
    constexpr int WARPS = THREADS / 32;
    constexpr int KPT = C3M_KEYS_PER_THREAD;
    constexpr int MAX_KEYS = THREADS * KPT;
    constexpr int SEG_TABLE = ABS ? C3M_SEG_TABLE_ABS : C3M_SEG_TABLE;
    constexpr int SPAN_SEGS = ABS ? C3M_ABS_SEGS : C3M_SPAN_SEGS;
    // dynamic: pass sums T [ncfg rounded up to even] x (low, high) u32, weight
    // map [(nslots + 1) * C3M_SEG] i16, configuration table [nb^3 rounded up
    // to a multiple of 8] u16, segment table [SEG_TABLE] u8, bin map
    // [(nslots + 1) * C3M_SEG] u8 (slot 0: the all-absent segment)
    extern __shared__ unsigned s_dyn[];
    __shared__ int s_next;
    __shared__ int s_cut;
    __shared__ int s_warp[WARPS];
    __shared__ long long s_hub;

    const int lane = threadIdx.x & 31;
    const int nb = a.nb, nb2 = nb * nb, n3 = nb2 * nb, ncfg = a.ncfg;
    unsigned *s_T = s_dyn;
    int16_t *s_wmap = reinterpret_cast<int16_t *>(s_T + 2 * ((ncfg + 1) & ~1));
    uint16_t *s_cfg = reinterpret_cast<uint16_t *>(s_wmap + (size_t)(nslots + 1) * C3M_SEG);
    uint8_t *s_seg = reinterpret_cast<uint8_t *>(s_cfg + ((n3 + 7) & ~7));
    uint8_t *s_map = s_seg + SEG_TABLE;
    unsigned long long *slice = a.gsum + 2 * (size_t)ncfg * blockIdx.x;

    for (int t = threadIdx.x; t < 2 * ncfg; t += THREADS) s_T[t] = 0u;
    for (int t = threadIdx.x; t < n3; t += THREADS) s_cfg[t] = __ldg(a.cfg3 + t);
    for (int t = threadIdx.x; t < C3M_SEG / 16; t += THREADS)
        reinterpret_cast<uint4 *>(s_map)[t] = make_uint4(~0u, ~0u, ~0u, ~0u);

    for (;;) {
        __syncthreads();                                     // everyone has read the last s_hub; T is folded
        if (threadIdx.x == 0) s_hub = (long long)atomicAdd(a.cursor, 1ull) + a.hub_begin;
        __syncthreads();
        if (s_hub >= a.hub_end) break;
        const long long i = s_hub;
        const int64_t f0 = a.row_ptr[i] + a.fwd[i];
        const int f = (int)(a.row_ptr[i + 1] - f0);
        if (f < 2) continue;                                 // fewer than two forward keys close nothing
        const int32_t *F = a.hnbr + f0;                      // the hub's forward row and its bins
        const uint8_t *FB = a.hbin + f0;
        for (int c0 = 0, c1 = 0; c0 < f; c0 = c1) {
            // ---- the chunk [c0, c1): keys, segment slots and the two maps, as in k_count3m
            const int32_t kbase = ABS ? 0 : F[c0] & ~(C3M_SEG - 1);
            const int cap = min(f, c0 + MAX_KEYS);
            const int t0 = c0 + threadIdx.x * KPT;
            int32_t key[KPT];
            unsigned starts = 0;
            int32_t prev = (t0 > c0 && t0 < cap) ? (F[t0 - 1] - kbase) >> C3M_SEG_LOG : -1;
#pragma unroll
            for (int q = 0; q < KPT; ++q) {
                key[q] = t0 + q < cap ? F[t0 + q] : 0;
                const int32_t sg = (key[q] - kbase) >> C3M_SEG_LOG;
                if (t0 + q < cap && sg != prev) starts |= 1u << q;
                prev = sg;
            }
            if (threadIdx.x == 0) s_cut = cap;
            int total = 0;
            const int sbase = c3m_block_scan<THREADS>(__popc(starts), s_warp, &total);
            {
                int slot = sbase;
#pragma unroll
                for (int q = 0; q < KPT; ++q) {
                    if (t0 + q >= cap) break;
                    slot += (starts >> q) & 1u;
                    if (slot > nslots || ((key[q] - kbase) >> C3M_SEG_LOG) >= SPAN_SEGS) {
                        atomicMin(&s_cut, t0 + q);
                        break;
                    }
                }
            }
            for (int t = threadIdx.x; t < SEG_TABLE; t += THREADS) s_seg[t] = 0;
            {
                const int nclear = min(nslots, total);
                uint4 *m = reinterpret_cast<uint4 *>(s_map + C3M_SEG);
                for (int t = threadIdx.x; t < nclear * (C3M_SEG / 16); t += THREADS)
                    m[t] = make_uint4(~0u, ~0u, ~0u, ~0u);
            }
            __syncthreads();
            c1 = s_cut;
            {
                int slot = sbase;
#pragma unroll
                for (int q = 0; q < KPT; ++q) {
                    if (t0 + q >= c1) break;
                    slot += (starts >> q) & 1u;
                    const int off = key[q] - kbase;
                    if (!GS_DCHECK(slot >= 1 && slot <= nslots && off >= 0 && (off >> C3M_SEG_LOG) < SPAN_SEGS,
                                   a.chk, GS_SITE_C3M_MAP_W))
                        continue;
                    if ((starts >> q) & 1u) s_seg[off >> C3M_SEG_LOG] = (uint8_t)slot;
                    const int at = (slot << C3M_SEG_LOG) | (off & (C3M_SEG - 1));
                    s_map[at] = FB[t0 + q];
                    s_wmap[at] = a.w[key[q]];
                }
            }
            if (threadIdx.x == 0) s_next = 0;
            __syncthreads();                                 // the maps are written
            const int s_end = c1 - 1;                        // spokes [0, s_end) meet this chunk
            const int32_t kmax = F[c1 - 1];
            const int32_t kfirst = F[c0];
            const unsigned guard = (unsigned)SPAN_SEGS << C3M_SEG_LOG;
            const int32_t kout = ABS ? (int32_t)guard : kbase - 1;
            for (;;) {
                int s = 0;
                if (lane == 0) s = atomicAdd(&s_next, 1);
                s = __shfl_sync(0xffffffffu, s, 0);
                if (s >= s_end) break;
                const int32_t j = F[s];
                int64_t p0, pe;
                c3m_spoke_range(a, 0, j, s, c0, kfirst, &p0, &pe);
                if (p0 >= pe) continue;
                const int hb = FB[s] * nb2;
                const int wj = a.w[j];
                const int64_t pa = p0 & ~(int64_t)3;
                const int head = (int)(p0 - pa);
                const int total_e = head + (int)(pe - p0);
                if (!GS_DCHECK(pa + (((total_e + 255) >> 8) << 8) <= a.nbr_len, a.chk, GS_SITE_C3M_ROW)) continue;
                const int4 *vk = reinterpret_cast<const int4 *>(a.snbr + pa) + lane;
                const uint32_t *vb = reinterpret_cast<const uint32_t *>(a.sbin + pa) + lane;
                int4 k0 = __ldg(vk), k1 = __ldg(vk + 32);
                uint32_t b0 = __ldg(vb), b1 = __ldg(vb + 32);
                for (int base = 0;; base += 256) {
                    const bool more = base + 256 < total_e;
                    int4 n0 = k0, n1 = k1;
                    uint32_t nb0 = b0, nb1 = b1;
                    if (more) {                              // the next step in flight
                        vk += 64;
                        vb += 64;
                        n0 = __ldg(vk);
                        n1 = __ldg(vk + 32);
                        nb0 = __ldg(vb);
                        nb1 = __ldg(vb + 32);
                    }
                    int k[8] = { k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w };
                    const uint32_t bb[2] = { b0, b1 };
                    if (base == 0 || !more) {                // entries outside the row: an absent segment
                        const unsigned r0 = (unsigned)(base + 4 * lane - head), len = (unsigned)(total_e - head);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            k[e] = r0 + e < len ? k[e] : kout;
                            k[4 + e] = r0 + 128 + e < len ? k[4 + e] : kout;
                        }
                    }
                    c3w_probe8<ABS>(k, bb, kbase, guard, s_seg, s_map, s_wmap, s_cfg, s_T, hb, nb, wj, a, nslots);
                    // rows are sorted: stop once the step's last key passes kmax
                    if (!more || __any_sync(0xffffffffu, lane == 31 && k1.w > kmax)) break;
                    k0 = n0;
                    k1 = n1;
                    b0 = nb0;
                    b1 = nb1;
                }
            }
            __syncthreads();                                 // the chunk's maps are no longer read
        }
        // slice[c] += w_i T[c] (128-bit); thread t owns configurations t, t + THREADS, ...
        const long long wi = a.w[i];
        for (int t = threadIdx.x; t < ncfg; t += THREADS) {
            const long long v = (long long)(((unsigned long long)s_T[2 * t + 1] << 32) | s_T[2 * t]);
            if (v) {
                s_T[2 * t] = 0u;
                s_T[2 * t + 1] = 0u;
                const unsigned long long lo = (unsigned long long)(wi * v);
                const unsigned long long hi = (unsigned long long)__mul64hi(wi, v);
                const unsigned long long l0 = slice[2 * t];
                slice[2 * t] = l0 + lo;
                slice[2 * t + 1] += hi + (l0 + lo < l0 ? 1ull : 0ull);
            }
        }
    }
}

// out[c] += sum over the slices of slice[c], 128-bit (low, high) words.
__global__ void k_sum128_slices(const unsigned long long *__restrict__ slices, int nslices, int ncfg,
                                unsigned long long *__restrict__ out)
{
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < ncfg; c += gridDim.x * blockDim.x) {
        unsigned long long lo = out[2 * c], hi = out[2 * c + 1];
        for (int b = 0; b < nslices; ++b) {
            const unsigned long long l = slices[2 * ((size_t)b * ncfg + c)];
            const unsigned long long h = slices[2 * ((size_t)b * ncfg + c) + 1];
            lo += l;
            hi += h + (lo < l ? 1ull : 0ull);
        }
        out[2 * c] = lo;
        out[2 * c + 1] = hi;
    }
}

// Walk mode of the unweighted, device-resident count: one spoke per warp for
// long rows, four spokes per warp (c3_walk_grouped) when the mean degree is at
// most C3_GROUPED_MAX_DEGREE. The environment variable GS_COUNT3_WALK = "warp"
// or "group" overrides the choice.
constexpr int64_t C3_GROUPED_MAX_DEGREE = 1024;

static int count3_walk_override()
{
    const char *env = getenv("GS_COUNT3_WALK");
    if (!env) return -1;
    if (!strcmp(env, "warp")) return 0;
    if (!strcmp(env, "group")) return 1;
    if (!strcmp(env, "map")) return 2;
    if (!strcmp(env, "mapgroup")) return 3;
    return -1;
}

// Shape of a byte-map walk launch: 512-thread blocks two per SM when the
// histogram leaves room for C3M_MIN_SLOTS segment slots each, else one
// 1024-thread block per SM; as many slots as fit. False when neither fits
// (e.g. nb > C3M_MAX_BINS).
using C3MKernel = void (*)(C3Args, int);

template <bool W, bool A>
static C3MKernel c3m_kernel(int threads, bool grouped)
{
    return threads == 512 ? (grouped ? k_count3m<512, true, W, A> : k_count3m<512, false, W, A>)
                          : (grouped ? k_count3m<1024, true, W, A> : k_count3m<1024, false, W, A>);
}

// The absolute segment table serves graphs whose ids lie below 2^21.
static bool c3m_abs(gs_graph_t g) { return g->n <= (int64_t)C3M_ABS_SEGS * C3M_SEG; }

static C3MKernel c3m_kernel(gs_graph_t g, int threads, bool grouped, bool windowed)
{
    if (c3m_abs(g))
        return windowed ? c3m_kernel<true, true>(threads, grouped) : c3m_kernel<false, true>(threads, grouped);
    return windowed ? c3m_kernel<true, false>(threads, grouped) : c3m_kernel<false, false>(threads, grouped);
}

// Threads, map slots and dynamic shared memory of a byte-map launch whose
// histogram and segment table take `fixed` bytes; false when fewer than
// C3M_MIN_SLOTS slots fit.
static bool plan_count3m_slots(gs_graph_t g, bool grouped, bool windowed, size_t fixed, int *threads, int *slots,
                               size_t *dyn)
{
    int dev = 0, smem_sm = 0, smem_block = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (int variant = 0; variant < 2; ++variant) {
        const int t = variant == 0 ? 512 : 1024;
        const int want = variant == 0 ? 2 : 1;                   // resident blocks per SM
        const C3MKernel kern = c3m_kernel(g, t, grouped, windowed);
        // per block: the SM's shared memory split, less 1 KB reserved and 2 KB of static data
        const long long room = std::min<long long>(smem_block, smem_sm / want - 1024) - 2048;
        int sl = (int)std::min<long long>(C3M_MAX_SLOTS, (room - (long long)fixed) / C3M_SEG - 1);
        while (sl >= C3M_MIN_SLOTS) {
            const size_t d = fixed + (size_t)(sl + 1) * C3M_SEG;
            int per = 0;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d);
            if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, t, d);
            if (e != cudaSuccess) {
                cudaGetLastError();
                per = 0;
            }
            if (per >= want) {
                *threads = t;
                *slots = sl;
                *dyn = d;
                return true;
            }
            sl -= 4;
        }
    }
    return false;
}

// Row stride of the b_ik index of the byte-map walk's histogram. A warp's
// adds share b_ij and spread over (b_ik, b_jk); the counter's bank is
// (hs b_ik + b_jk) mod 32. With hs = nb = 30 (the BAO-scale bins) many pairs
// collide (30 = -2 mod 32); a stride of 5 mod 32 spreads them. Modelled on
// the one-spoke walk's adds over a scaled BAO-scale catalogue (15 of 32 lanes
// hit): 1.58 wavefronts per add instruction with hs = 30, 1.07 with hs = 37;
// on a uniform catalogue (8.5 hitting lanes) the stride made no difference.
// So the one-spoke walk (dense rows) takes the padded stride while its
// histogram leaves room for enough map slots; the four-spokes-per-warp walk
// keeps hs = nb.
static int c3m_padded_stride(int nb) { return nb + ((5 - nb) & 31); }

static bool plan_count3m(gs_graph_t g, bool grouped, bool windowed, int *threads, int *slots, size_t *dyn, int *hs)
{
    if (g->nb > C3M_MAX_BINS || !g->cfg3) return false;
    for (int pad = grouped ? 1 : 0; pad < 2; ++pad) {
        const int h = pad == 0 ? c3m_padded_stride(g->nb) : g->nb;
        const int nh = g->nb * g->nb * h;
        const size_t fixed =
            sizeof(unsigned) * (size_t)((nh + 3) & ~3) + (c3m_abs(g) ? C3M_SEG_TABLE_ABS : C3M_SEG_TABLE);
        if (plan_count3m_slots(g, grouped, windowed, fixed, threads, slots, dyn)) {
            *hs = h;
            return true;
        }
    }
    return false;
}

// Shared-memory size of the four-spokes-per-warp walk (the whole nb^3
// configuration table replaces the per-warp tables); false unless two blocks
// fit on an SM (one when the walk is forced) or the histogram is global.
static bool plan_count3g(gs_graph_t g, bool forced, size_t *dyn)
{
    const int ncfg = (int)gs_ncfg3(g->nb);
    const bool smem = ncfg <= C3_SMEM_HIST_MAX && g->cfg3 && (int64_t)g->max_degree * C3_CHUNK_BM < (1ll << 31);
    if (!smem) return false;
    const size_t d = C3_REGION + sizeof(unsigned) * ((ncfg + 3) & ~3) + sizeof(uint16_t) * (size_t)g->nb * g->nb * g->nb;
    auto kg = k_count3<true, false, false, false, true>;
    int per = 0;
    // a table too large for one block (nb near 40) is refused here: the
    // one-spoke walk runs instead, and the refusal is cleared
    cudaError_t e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kg, C3_THREADS, d);
    if (e != cudaSuccess) {
        cudaGetLastError();
        per = 0;
    }
    *dyn = d;
    return per >= 2 || (forced && per >= 1);
}

// The walk an unweighted count takes: 2 = byte map, one spoke per warp (long
// rows: mean degree above C3_GROUPED_MAX_DEGREE); 3 = byte map, four spokes
// per warp (short rows); when the byte map does not fit (more than
// C3M_MAX_BINS bins) 1 = bitmap, four spokes per warp (device-resident
// graphs) or 0 = bitmap, one spoke per warp. GS_COUNT3_WALK overrides the
// choice.
static int count3_walk(gs_graph_t g)
{
    int mode = count3_walk_override();
    const bool long_rows = g->n_edges > C3_GROUPED_MAX_DEGREE * g->n;
    int t, sl, hs;
    size_t d;
    if (mode < 0) mode = long_rows ? 2 : 3;
    if (mode >= 2 && plan_count3m(g, mode == 3, g->n_win > 0, &t, &sl, &d, &hs)) return mode;
    if (g->n_win) return 0;                                  // the bitmap walk of windowed tiles
    if (mode == 1 || mode == 3 || (mode == 2 && !long_rows)) return plan_count3g(g, mode == 1, &d) ? 1 : 0;
    return 0;
}

extern "C" int gs_count3_walk(gs_graph_t g)
{
    GS_ENTRY();
    if (!g) return -1;
    if (gs_check_device(g) != GS_OK) return -1;
    return count3_walk(g);
}

// Shared memory of the weighted byte-map walk (1024-thread blocks, one per
// SM): false when it does not apply (more than C3M_MAX_BINS bins, forward rows
// of 2^16 keys or more, GS_COUNT3_WALK naming a bitmap walk) or fewer than
// C3M_MIN_SLOTS segment slots fit beside the sums and the configuration table.
static bool plan_count3mw(gs_graph_t g, int *slots, size_t *dyn)
{
    const int mode = count3_walk_override();
    if (mode == 0 || mode == 1) return false;
    if (g->nb > C3M_MAX_BINS || !g->cfg3 || g->max_forward >= 65536) return false;
    const int n3 = g->nb * g->nb * g->nb, ncfg = (int)gs_ncfg3(g->nb);
    const size_t fixed = 8 * (size_t)((ncfg + 1) & ~1) + 2 * (size_t)((n3 + 7) & ~7) +
                         (c3m_abs(g) ? C3M_SEG_TABLE_ABS : C3M_SEG_TABLE);
    int dev = 0, smem_sm = 0, smem_block = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const auto kern = c3m_abs(g) ? k_count3mw<1024, true> : k_count3mw<1024, false>;
    // the SM's shared memory, less 1 KB reserved and 2 KB of static data; 3 bytes per id of a slot
    const long long room = std::min<long long>(smem_block, smem_sm - 1024) - 2048;
    for (int sl = (int)std::min<long long>(C3M_MAX_SLOTS, (room - (long long)fixed) / (3 * C3M_SEG) - 1);
         sl >= C3M_MIN_SLOTS; sl -= 4) {
        const size_t d = fixed + 3 * (size_t)(sl + 1) * C3M_SEG;
        int per = 0;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, 1024, d);
        if (e != cudaSuccess) {
            cudaGetLastError();
            per = 0;
        }
        if (per >= 1) {
            *slots = sl;
            *dyn = d;
            return true;
        }
    }
    return false;
}

static gs_status launch_count3(gs_graph_t g, C3Args a, int64_t hubs, cudaStream_t st)
{
    const int ncfg = a.ncfg;
    const int nb2 = g->nb * g->nb;
    const bool list = a.hubs != nullptr;
    const bool weighted = a.w != nullptr;
    bool smem;
    size_t dyn;
    const bool win = a.windowed != 0;
    decltype(&k_count3<true, true, false, false>) kern;
    if (weighted && !win && !list) {
        int slots = 0;
        size_t dm = 0;
        if (plan_count3mw(g, &slots, &dm)) {
            // one 128-bit slice per block, then their sum added to the output
            unsigned long long *out = a.gsum, *slices = a.slices;
            const int grid = (int)std::min<int64_t>((int64_t)gs_sm_count(), hubs);
            GS_TRY_CUDA(cudaMemsetAsync(slices, 0, 16 * (size_t)ncfg * grid, st));
            GS_TRY_CUDA(cudaMemsetAsync(a.cursor, 0, sizeof(unsigned long long), st));
            a.gsum = slices;
            (c3m_abs(g) ? k_count3mw<1024, true> : k_count3mw<1024, false>)<<<grid, 1024, dm, st>>>(a, slots);
            gs_note_launch();
            GS_TRY_CUDA(cudaGetLastError());
            k_sum128_slices<<<(ncfg + 255) / 256, 256, 0, st>>>(slices, grid, ncfg, out);
            gs_note_launch();
            GS_TRY_CUDA(cudaGetLastError());
            return GS_OK;
        }
    }
    if (weighted) {
        smem = true;
        dyn = C3_REGION_W + sizeof(unsigned long long) * (size_t)ncfg;
        kern = win ? k_count3<true, false, true, true> : k_count3<true, false, true, false>;
    } else {
        const int walk = !list ? count3_walk(g) : 0;
        if (walk >= 2) {
            const bool grouped = walk == 3;
            int threads = 0, slots = 0;
            size_t dm = 0;
            if (!plan_count3m(g, grouped, win, &threads, &slots, &dm, &a.hs))
                return gs_set_error(GS_ERR_INTERNAL, "byte-map walk plan");
            const int grid = (int)std::min<int64_t>((int64_t)gs_sm_count() * (threads == 512 ? 2 : 1), hubs);
            GS_TRY_CUDA(cudaMemsetAsync(a.cursor, 0, sizeof(unsigned long long), st));
            c3m_kernel(g, threads, grouped, win)<<<grid, threads, dm, st>>>(a, slots);
            gs_note_launch();
            GS_TRY_CUDA(cudaGetLastError());
            return GS_OK;
        }
        // shared-memory histogram unless it is too large or a chunk's hit bound
        // (spokes x chunk) could overflow a 32-bit counter
        smem = ncfg <= C3_SMEM_HIST_MAX && g->cfg3 && (int64_t)g->max_degree * C3_CHUNK_BM < (1ll << 31);
        dyn = C3_REGION + (smem ? sizeof(unsigned) * ((ncfg + 3) & ~3) + sizeof(uint16_t) * C3_WARPS * nb2 : 0);
        if (win)
            kern = smem ? k_count3<true, false, false, true> : k_count3<false, false, false, true>;
        else
            kern = smem ? (list ? k_count3<true, true, false, false> : k_count3<true, false, false, false>)
                        : (list ? k_count3<false, true, false, false> : k_count3<false, false, false, false>);
        if (walk == 1) {
            size_t dg = 0;
            plan_count3g(g, true, &dg);
            kern = k_count3<true, false, false, false, true>;
            dyn = dg;
        }
    }
    int per_sm = 0;
    GS_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn));
    GS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C3_THREADS, dyn));
    if (per_sm < 1) return gs_set_error(GS_ERR_CAPACITY, "3pCF workspace of %zu bytes does not fit in shared memory", dyn);
    const int grid = (int)std::min<int64_t>((int64_t)gs_sm_count() * std::min(per_sm, C3_MAX_BLOCKS_PER_SM), hubs);
    GS_TRY_CUDA(cudaMemsetAsync(a.cursor, 0, sizeof(unsigned long long), st));
    if (!weighted) {
        kern<<<grid, C3_THREADS, dyn, st>>>(a);
        gs_note_launch();
        GS_TRY_CUDA(cudaGetLastError());
        return GS_OK;
    }
    // weighted: one 128-bit slice per block (in the caller's scratch, which
    // holds C3_MAX_BLOCKS_PER_SM slices per SM), then their sum added to the output
    unsigned long long *out = a.gsum, *slices = a.slices;
    const size_t bytes = 16 * (size_t)ncfg * grid;
    GS_TRY_CUDA(cudaMemsetAsync(slices, 0, bytes, st));
    a.gsum = slices;
    kern<<<grid, C3_THREADS, dyn, st>>>(a);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    k_sum128_slices<<<(ncfg + 255) / 256, 256, 0, st>>>(slices, grid, ncfg, out);
    gs_note_launch();
    GS_TRY_CUDA(cudaGetLastError());
    return GS_OK;
}

// Scratch of the weighted count: a 128-bit slice per configuration for every
// block that can be resident (k_count3 is launched with at most
// C3_MAX_BLOCKS_PER_SM blocks per SM).
static size_t c3_slice_bytes(gs_graph_t g)
{
    return 16 * (size_t)gs_ncfg3(g->nb) * (size_t)gs_sm_count() * C3_MAX_BLOCKS_PER_SM;
}

// The hubs [hub_begin, hub_end): one launch on a device-resident graph; on a
// windowed graph one launch per (hub window h, spoke window w >= h) tile that
// holds work. A triangle (i < j < k) is closed in the tile of i's and j's
// windows only, so the tiles add up to the full histogram (§III.5.3).
// Windows are staged into three device slots on a copy stream: a window
// already in a slot is not copied again (the spoke window of tile (h, h+1) is
// the hub window of (h+1, h+1)), and the next tile's missing window is copied
// into the free slot while the current tile runs. Outputs accumulate; the
// caller clears them first.
static gs_status run_count3(gs_graph_t g, C3Args a, int64_t hub_begin, int64_t hub_end, cudaStream_t st)
{
    if (g->n_win == 0) {
        a.hub_begin = hub_begin;
        a.hub_end = hub_end;
        return launch_count3(g, a, hub_end - hub_begin, st);
    }
    std::vector<std::pair<int, int>> tiles;
    for (int h = 0; h < g->n_win; ++h) {
        if (std::max(hub_begin, g->win_row[h]) >= std::min(hub_end, g->win_row[h + 1])) continue;
        if (g->win_e0[h + 1] == g->win_e0[h]) continue;
        for (int w = h; w < g->n_win; ++w)
            if (g->win_pair[(size_t)h * g->n_win + w] && g->win_e0[w + 1] > g->win_e0[w]) tiles.push_back({ h, w });
    }
    if (tiles.empty()) return GS_OK;

    cudaStream_t cs = nullptr;
    cudaEvent_t start = nullptr, fin = nullptr, ready[GS_SLOTS] = {}, done[GS_SLOTS] = {};
    int held[GS_SLOTS];
    int64_t off[GS_SLOTS] = {};
    for (int k = 0; k < GS_SLOTS; ++k) held[k] = -1;
    gs_status s = GS_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&fin, cudaEventDisableTiming);
    for (int k = 0; k < GS_SLOTS && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&ready[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[k], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventRecord(start, st);     // slots are free once earlier work on st is done
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, start, 0);

    auto slot_of = [&](int w) {
        for (int k = 0; k < GS_SLOTS; ++k)
            if (held[k] == w) return k;
        return -1;
    };
    // copy window w into slot k once the last tile that read slot k is done
    auto stage_into = [&](int k, int w) {
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, done[k], 0);
        if (e == cudaSuccess && s == GS_OK) s = gs_stage_window(g, w, k, cs, &off[k]);
        if (e == cudaSuccess && s == GS_OK) e = cudaEventRecord(ready[k], cs);
        held[k] = w;
    };
    // a slot other than keep0 / keep1, preferring one whose window the tile
    // after t does not need
    auto victim = [&](int keep0, int keep1, size_t t) {
        for (int pass = 0; pass < 2; ++pass)
            for (int k = 0; k < GS_SLOTS; ++k) {
                if (k == keep0 || k == keep1) continue;
                const bool wanted = t + 1 < tiles.size() &&
                                    (held[k] == tiles[t + 1].first || held[k] == tiles[t + 1].second);
                if (pass == 1 || !wanted) return k;
            }
        return -1;
    };

    a.windowed = 1;
    for (size_t t = 0; t < tiles.size() && e == cudaSuccess && s == GS_OK; ++t) {
        const int h = tiles[t].first, w = tiles[t].second;
        int sh = slot_of(h);
        if (sh < 0) stage_into(sh = victim(slot_of(w), -1, t), h);
        int sw = slot_of(w);
        if (sw < 0) stage_into(sw = victim(sh, -1, t), w);
        if (e != cudaSuccess || s != GS_OK) break;
        e = cudaStreamWaitEvent(st, ready[sh], 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ready[sw], 0);
        if (e != cudaSuccess) break;
        a.hnbr = g->s_nbr[sh];
        a.hbin = g->s_bin[sh];
        a.hoff = off[sh];
        a.snbr = g->s_nbr[sw];
        a.sbin = g->s_bin[sw];
        a.soff = off[sw];
        a.s_lo = (int32_t)g->win_row[w];
        a.s_hi = (int32_t)g->win_row[w + 1];
        // hubs of window h before the first one with a forward neighbour in w hold no work
        a.hub_begin = std::max(hub_begin, g->win_first[(size_t)h * g->n_win + w]);
        a.hub_end = std::min(hub_end, g->win_row[h + 1]);
        if (a.hub_begin >= a.hub_end) {
            e = cudaEventRecord(done[sh], st);
            if (e == cudaSuccess) e = cudaEventRecord(done[sw], st);
            continue;
        }
        s = launch_count3(g, a, a.hub_end - a.hub_begin, st);
        if (s != GS_OK) break;
        e = cudaEventRecord(done[sh], st);
        if (e == cudaSuccess) e = cudaEventRecord(done[sw], st);
        // prefetch the next tile's missing windows into slots this tile does not read
        if (t + 1 < tiles.size())
            for (int q = 0; q < 2; ++q) {
                const int x = q ? tiles[t + 1].second : tiles[t + 1].first;
                const int y = q ? tiles[t + 1].first : tiles[t + 1].second;
                if (slot_of(x) >= 0) continue;
                for (int k = 0; k < GS_SLOTS; ++k)
                    if (k != sh && k != sw && k != slot_of(y)) {
                        stage_into(k, x);
                        break;
                    }
            }
    }
    // the caller's stream waits for the last copies; then release the helpers
    if (e == cudaSuccess) e = cudaEventRecord(fin, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, fin, 0);
    for (int k = 0; k < GS_SLOTS; ++k) {
        if (ready[k]) cudaEventDestroy(ready[k]);
        if (done[k]) cudaEventDestroy(done[k]);
    }
    if (start) cudaEventDestroy(start);
    if (fin) cudaEventDestroy(fin);
    if (cs) cudaStreamDestroy(cs);
    if (s != GS_OK) return s;
    if (e != cudaSuccess) return gs_set_error(GS_ERR_CUDA, "windowed 3pCF: %s", cudaGetErrorString(e));
    return GS_OK;
}

static C3Args count3_args(gs_graph_t g, uint64_t *hist_dev)
{
    C3Args a{};
    a.row_ptr = g->row_ptr;
    a.fwd = g->fwd;
    a.hnbr = a.snbr = g->nbr;
    a.hbin = a.sbin = g->bin;
    a.hoff = a.soff = 0;
    a.windowed = 0;
    a.s_lo = 0;
    a.s_hi = 0x7fffffff;
    a.nb = g->nb;
    a.ncfg = (int)gs_ncfg3(g->nb);
    a.ghist = (unsigned long long *)hist_dev;
    a.cursor = g->work;
    a.cfg3 = g->cfg3;
    a.inv = g->inv;
    a.chk = g->chk;
    a.nbr_len = g->nbr_len;
    return a;
}

extern "C" gs_status gs_count_3pcf(gs_graph_t g, uint64_t *hist_dev, int64_t hub_begin, int64_t hub_end,
                                   void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !hist_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int ncfg = (int)gs_ncfg3(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(hist_dev, 0, sizeof(uint64_t) * ncfg, st));
    if (hub_end == hub_begin || g->n_edges == 0) return GS_OK;
    gs_status s = gs_checked_begin(g, st);
    if (s == GS_OK) s = run_count3(g, count3_args(g, hist_dev), hub_begin, hub_end, st);
    if (s == GS_OK) s = gs_checked_end(g, st, "3pCF count");
    return s;
}

// Range check of a device list of input indices, one flag word for the host.
__global__ void k_check_ids(const int32_t *__restrict__ ids, int64_t count, int64_t n, int32_t *__restrict__ err)
{
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < count;
         t += (int64_t)gridDim.x * blockDim.x)
        if (ids[t] < 0 || ids[t] >= n) atomicOr(err, 1);
}

gs_status gs_check_ids(gs_graph_t g, const int32_t *ids, int64_t count, cudaStream_t st)
{
    if (count == 0) return GS_OK;
    GS_TRY_CUDA(cudaMemsetAsync(g->err, 0, sizeof(int32_t), st));
    const int grid = (int)std::min<int64_t>((count + 255) / 256, (int64_t)gs_sm_count() * 4);
    k_check_ids<<<grid, 256, 0, st>>>(ids, count, g->n, g->err);
    gs_note_launch();
    int32_t h = 0;
    GS_TRY_CUDA(cudaMemcpyAsync(&h, g->err, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    GS_TRY_CUDA(cudaStreamSynchronize(st));
    if (h) return gs_set_error(GS_ERR_ARG, "a hub index lies outside [0, n)");
    return GS_OK;
}

extern "C" gs_status gs_count_3pcf_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count,
                                        uint64_t *hist_dev, void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !hist_dev || (count > 0 && !hubs_dev)) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (count < 0) return gs_set_error(GS_ERR_ARG, "negative hub count");
    if (g->n_win) return gs_set_error(GS_ERR_ARG, "hub lists need a device-resident graph (this one is windowed)");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    gs_status s = gs_check_ids(g, hubs_dev, count, st);
    if (s != GS_OK) return s;
    const int ncfg = (int)gs_ncfg3(g->nb);
    GS_TRY_CUDA(cudaMemsetAsync(hist_dev, 0, sizeof(uint64_t) * ncfg, st));
    if (count == 0 || g->n_edges == 0) return GS_OK;
    C3Args a = count3_args(g, hist_dev);
    a.hub_begin = 0;
    a.hub_end = count;
    a.hubs = hubs_dev;
    s = gs_checked_begin(g, st);
    if (s == GS_OK) s = launch_count3(g, a, count, st);
    if (s == GS_OK) s = gs_checked_end(g, st, "3pCF hub-list count");
    return s;
}

extern "C" gs_status gs_count_3pcf_weighted(gs_graph_t g, int64_t *sums_dev, int64_t hub_begin, int64_t hub_end,
                                            void *cuda_stream)
{
    GS_ENTRY();
    if (!g || !sums_dev) return gs_set_error(GS_ERR_ARG, "NULL argument");
    GS_TRY_DEVICE(g);
    if (!g->w) return gs_set_error(GS_ERR_ARG, "no weights: call gs_graph_set_weights first");
    if (g->nb > C3_WEIGHTED_MAX_BINS)
        return gs_set_error(GS_ERR_ARG, "the weighted 3pCF supports at most %d bins", C3_WEIGHTED_MAX_BINS);
    if (hub_begin < 0 || hub_end > g->n || hub_begin > hub_end)
        return gs_set_error(GS_ERR_ARG, "hub range [%lld, %lld) outside [0, %lld]", (long long)hub_begin,
                            (long long)hub_end, (long long)g->n);
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const int ncfg = (int)gs_ncfg3(g->nb);
    const bool work = hub_end > hub_begin && g->n_edges > 0;
    // the per-block slices are allocated before any output is written
    unsigned long long *slices = nullptr;
    if (work) GS_TRY_CUDA(gs_malloc_async(&slices, c3_slice_bytes(g), st));
    gs_status s = GS_OK;
    const cudaError_t e = cudaMemsetAsync(sums_dev, 0, sizeof(int64_t) * 2 * ncfg, st);
    if (e != cudaSuccess) s = gs_set_error(GS_ERR_CUDA, "clearing the sums failed: %s", cudaGetErrorString(e));
    if (s == GS_OK && work) {
        C3Args a = count3_args(g, nullptr);
        a.w = g->w;
        a.gsum = (unsigned long long *)sums_dev;
        a.slices = slices;
        s = gs_checked_begin(g, st);
        if (s == GS_OK) s = run_count3(g, a, hub_begin, hub_end, st);
        if (s == GS_OK) s = gs_checked_end(g, st, "weighted 3pCF count");
    }
    if (slices) cudaFreeAsync(slices, st);
    return s;
}
