/*
 * gramsci_gb.h -- C ABI of libgramsci_gb.so: graph-based 3pCF and
 * parity-decomposed 4pCF counting on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the GRAMSCI v2 paper, "Fast Graph-based Higher-Order
 * Clustering Statistics on the GPU":
 *   - gs_build_graph: the fixed-radius neighbour graph of §II.1 (all j with
 *     |x_i - x_j| < r_max), stored as sorted adjacency lists (Eq.(1)) with a
 *     radial-bin byte per neighbour, flattened to CSR (§III.5.1: 64-bit row
 *     offsets, 32-bit neighbour ids, 8-bit bins).
 *   - gs_count_3pcf: the triangle count of §II.2 / §III.1 (hub, spoke and a
 *     third point adjacent to both), binned by the sorted side bins
 *     b1 <= b2 <= b3 and packed lexicographically (§V.1, Fig.8 key).
 *   - gs_count_4pcf_parity: the parity-decomposed 4pCF of §III.2: per hub and
 *     triple of mutually adjacent spokes, an even count and an odd sum of the
 *     sign of V = (r_ij1 x r_ij2) . r_ij3 (Eq.(3)), V == 0 adding 0 to odd.
 *
 * Data model (all integer, all exact):
 *   - Coordinates are int32 lattice positions (1 lattice unit = 1/1024
 *     h^-1 Mpc in the intended use) in [0, box_lu) on each axis, row-major
 *     [n][3] (x, y, z).
 *   - periodic != 0: separations use the minimum image in a cube of side
 *     box_lu (delta -= box if 2*delta >= box, delta += box if 2*delta < -box).
 *   - Bin edges e_0 < e_1 < ... < e_nb in lattice units; a pair i != j is an
 *     edge iff e_0^2 <= d^2 < e_nb^2, its bin the b with e_b^2 <= d^2 <
 *     e_{b+1}^2. d^2 is computed in int64.
 *   - 3pCF: every unordered triangle {i, j, k} whose three sides are edges
 *     adds 1 at index idx3(sort(b_ij, b_ik, b_jk)), the rank of the sorted
 *     triple among all b1 <= b2 <= b3 in lexicographic order
 *     (gs_config_count_3pcf(nb) = C(nb+2, 3) entries).
 *   - parity 4pCF: for each hub i and each set of three spokes {j, k, l} in
 *     N(i) that are pairwise adjacent and whose hub bins are pairwise
 *     distinct, the spokes are ordered by hub bin (b1 < b2 < b3),
 *     V = det[r_is1; r_is2; r_is3] with r_is = x_s - x_i (minimum image), and
 *     even[idx4] += 1, odd[idx4] += sign(V) where idx4 ranks b1 < b2 < b3 in
 *     lexicographic order (gs_config_count_4pcf(nb) = C(nb, 3) entries).
 *
 * Conventions:
 *   - "_dev" pointers are CUDA device pointers on the current device; the
 *     caller owns and allocates them. Host pointers are marked "_host".
 *   - Every call runs on `cuda_stream` (a cudaStream_t; NULL = the legacy
 *     default stream). gs_build_graph synchronises that stream once (to read
 *     the edge total); the count and export calls are asynchronous.
 *   - Outputs are overwritten, never accumulated.
 *   - A graph keeps one work cursor per count kind, so count calls on the
 *     same graph must not overlap in time (issue them on one stream);
 *     different graphs are independent.
 *   - On any non-OK status no output has been written by this call (except
 *     where noted), everything the call allocated is freed, and
 *     gs_last_error() returns a message for the calling thread.
 *   - Limits: 0 <= n < 2^31 - 1; 1 <= box_lu <= 2^30; 1 <= nbins <= 255;
 *     periodic boxes need 2 * r_max_lu <= box_lu; the parity 4pCF needs
 *     r_max_lu < 2^20 (so that the int64 volume is exact).
 */
#ifndef GRAMSCI_GB_H
#define GRAMSCI_GB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gs_graph *gs_graph_t;   /* opaque; owns all device memory of one graph */

typedef enum {
    GS_OK = 0,
    GS_ERR_ARG = 1,        /* invalid argument (sizes, edges, coordinates out of range, ...) */
    GS_ERR_NOMEM = 2,      /* a device allocation failed */
    GS_ERR_CUDA = 3,       /* a CUDA runtime call or kernel launch failed */
    GS_ERR_CAPACITY = 4,   /* the graph exceeds a documented size limit */
    GS_ERR_INTERNAL = 5    /* a device-side consistency check failed */
} gs_status;

/* Build the neighbour graph of n points (§II.1, Eq.(1); CSR layout §III.5.1).
 *   coords_dev  int32 [n][3], device, caller-owned; values in [0, box_lu)
 *   n           number of points (0 allowed: empty graph)
 *   box_lu      cube side in lattice units
 *   periodic    1 = minimum-image separations, 0 = open box
 *   r_max_lu    must equal edges_lu[nbins]
 *   edges_lu    int64 [nbins+1], HOST, strictly increasing, edges_lu[0] >= 0
 *   nbins       1..255
 *   out         receives the new graph handle (free with gs_graph_free)
 * The coordinates are copied; coords_dev may be freed after the call returns.
 * The edge arrays normally live in device memory. When they would not fit in
 * the free device memory, or when the environment variable GS_WINDOW_EDGES
 * holds a positive edge count, the graph is built windowed instead (pinned
 * host memory, see gs_build_graph_windowed); gs_graph_windows tells which.
 * Errors: GS_ERR_ARG for bad arguments or a coordinate outside [0, box_lu)
 * (checked on the device, reported at the call's one synchronisation),
 * GS_ERR_NOMEM, GS_ERR_CUDA. On error *out is set to NULL. */
gs_status gs_build_graph(const int32_t *coords_dev, int64_t n, int64_t box_lu, int periodic,
                         int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                         void *cuda_stream, gs_graph_t *out);

/* Triangle histogram of the 3pCF (§II.2 hub-and-spoke enumeration, §III.1
 * set intersection of the hub's and the spoke's sorted lists).
 *   hist_dev    uint64 [gs_config_count_3pcf(nbins)], device, overwritten
 *   hub_begin, hub_end  half-open range of hubs in the graph's internal order
 *               (points sorted by cell); [0, n) gives the full histogram.
 *               Each triangle is counted at its lowest internal index, so the
 *               histograms of disjoint ranges that cover [0, n) sum exactly
 *               to the full one.
 * The spoke walk depends on the graph (gs_count3_walk); the environment
 * variable GS_COUNT3_WALK = "map", "mapgroup", "group" or "warp" overrides the choice
 * (read at each call). The histogram is the same for every walk.
 * Errors: GS_ERR_ARG (NULL pointers, range outside [0, n]), GS_ERR_CUDA. */
gs_status gs_count_3pcf(gs_graph_t g, uint64_t *hist_dev, int64_t hub_begin, int64_t hub_end,
                        void *cuda_stream);

/* The spoke walk gs_count_3pcf takes on this graph (host query, no device
 * work). The hub's keys and their bins are held in shared memory either as a
 * byte map (a bin byte per id of the key span, in 1024-id segments; hits go
 * to an unsorted nb^3 histogram) or as a bitmap with ranks (hits go to the
 * sorted-triple histogram through a configuration table):
 *   2 = byte map, one spoke per warp (long rows: mean degree above 1024)
 *   3 = byte map, four spokes per warp (short rows)
 *   1 = bitmap, four spokes per warp, and 0 = bitmap, one spoke per warp,
 *       when the byte map does not fit (more than 32 bins; windowed graphs
 *       then take 0)
 * Windowed graphs run the same walks on their tiles. GS_COUNT3_WALK = "map",
 * "mapgroup", "warp" or "group" overrides the choice, as for the count. -1
 * for a NULL graph or one of another device. */
int gs_count3_walk(gs_graph_t g);

/* Parity-decomposed 4pCF histograms (§III.1.1 three-way intersection,
 * §III.2 Eq.(3), degenerate volumes add 0 to odd).
 *   even_dev    uint64 [gs_config_count_4pcf(nbins)], device, overwritten
 *   odd_dev     int64  [gs_config_count_4pcf(nbins)], device, overwritten
 *   hub_begin, hub_end  half-open hub range in internal order, as above;
 *               every hub's contribution is independent of the others.
 * For nbins < 3 there are no configurations and nothing is written.
 * Errors: GS_ERR_ARG (NULL pointers, bad range, r_max_lu >= 2^20),
 * GS_ERR_NOMEM (scratch for hubs of very high degree), GS_ERR_CUDA. */
gs_status gs_count_4pcf_parity(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev,
                               int64_t hub_begin, int64_t hub_end, void *cuda_stream);

/* The parity-4pCF count of gs_count_4pcf_parity, without any device memory
 * allocation inside the call. The paper has no counterpart: this entry point
 * is for callers that cannot call cudaMalloc / cudaMallocAsync -- for example
 * a latency-critical pipeline where cudaMalloc and cudaFree would synchronise
 * the whole device and stall other streams, or a service that reserves all of
 * its device memory once at start-up and forbids later allocations.
 * gs_count_4pcf_parity allocates a per-block workspace for hubs of more than
 * 512 neighbours; this variant instead uses a fixed 16 MiB workspace that is
 * compiled into the library (a static device array: every GPU that loads the
 * library holds those 16 MiB until the process exits), plus its own two work
 * cursors kept in the same array.
 *   Arguments, outputs and results are those of gs_count_4pcf_parity.
 *   Limit: one workspace slice must fit a hub of the graph's largest degree
 *   (16 MiB hold degree 11,392 at 8 bins); otherwise GS_ERR_CAPACITY is returned
 *   before anything is written.
 *   Set-up: the first call on each device looks up the workspace's device
 *   address (cudaGetSymbolAddress) with that device current and caches it;
 *   make that first call before any stream capture.
 *   Sharing: all calls share the one workspace. The call clears what must
 *   start at zero, but calls whose kernels overlap on the GPU (different
 *   streams, different threads) race on it: serialise them. */
gs_status gs_count_4pcf_parity_static(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev,
                                      int64_t hub_begin, int64_t hub_end, void *cuda_stream);

/* Hub-and-spoke triangle counts of selected hubs (§II.2 literally: for hub
 * i, every pair of neighbours j < k of i that are neighbours of each other).
 * Each triangle incident to a listed hub is counted once for that hub, so a
 * triangle is seen from each of its listed vertices (over all n hubs the
 * result is 3 x gs_count_3pcf). Same kernel as gs_count_3pcf, with the
 * whole hub row staged instead of its forward part.
 *   hubs_dev   int32 [count], device, INPUT indices in [0, n); repeats count
 *              again
 *   hist_dev   uint64 [gs_config_count_3pcf(nbins)], device, overwritten
 * Synchronises cuda_stream once (index check). Errors: GS_ERR_ARG (NULL,
 * negative count, an index outside [0, n)), GS_ERR_CUDA. */
gs_status gs_count_3pcf_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count,
                             uint64_t *hist_dev, void *cuda_stream);

/* Parity-4pCF contribution of selected hubs (INPUT indices), as
 * gs_count_4pcf_parity restricted to those hubs; the same kernels.
 * Synchronises cuda_stream once (index check). Errors as gs_count_3pcf_hubs
 * plus those of gs_count_4pcf_parity. */
gs_status gs_count_4pcf_parity_hubs(gs_graph_t g, const int32_t *hubs_dev, int64_t count,
                                    uint64_t *even_dev, int64_t *odd_dev, void *cuda_stream);

/* Six-edge-bin 4pCF with parity channels (§II.2 tetrahedra: four points whose
 * six pairs are all neighbours; §III.2 Eq.(3) handedness; §V.2
 * configurations). Every tetrahedron counts once. Its configuration is the
 * lexicographically smallest bin tuple (b01, b02, b03, b12, b13, b23) over the
 * 24 orderings (v0, v1, v2, v3) of its vertices (b_ab: bin of the pair
 * v_a v_b); configurations are numbered in lexicographic order of those
 * tuples (gs_config_count_4pcf6(nb) = (nb^6 + 9 nb^4 + 14 nb^2) / 24 of them,
 * 276 for 4 bins). even[c] counts the tetrahedra of configuration c; odd[c]
 * sums sign(det[x_v1 - x_v0; x_v2 - x_v0; x_v3 - x_v0]) for an ordering that
 * reaches the smallest tuple, with 0 when orderings of both permutation
 * parities reach it (an achiral configuration) or when the volume is 0.
 *   even_dev  uint64 [gs_config_count_4pcf6(nbins)], device, overwritten
 *   odd_dev   int64  [gs_config_count_4pcf6(nbins)], device, overwritten
 *   hub_begin, hub_end  internal-order hub range; a tetrahedron belongs to
 *             its lowest internal index, so disjoint ranges add exactly.
 * The first call on a graph builds a table of nb^6 entries (synchronously).
 * Limits: nbins <= 10, r_max_lu < 2^20. Errors: GS_ERR_ARG, GS_ERR_NOMEM,
 * GS_ERR_CUDA. */
gs_status gs_count_4pcf6(gs_graph_t g, uint64_t *even_dev, int64_t *odd_dev,
                         int64_t hub_begin, int64_t hub_end, void *cuda_stream);
int64_t gs_config_count_4pcf6(int nbins);

/* Weighted six-bin 4pCF (§II.1 signed weights, §III.3: NNNN of the
 * estimator NNNN / RRRR): per configuration, the exact sums over tetrahedra
 * of W = w_i w_j w_k w_l (even) and of s W (odd), s the tetrahedron's odd
 * sign of gs_count_4pcf6 (+1, -1 or 0). Weights from gs_graph_set_weights.
 *   even_dev, odd_dev  int64 [2 * gs_config_count_4pcf6(nbins)], device,
 *             overwritten: 128-bit sums as (low, high) word pairs
 *   hub_begin, hub_end  as for gs_count_4pcf6
 * Limits and errors as gs_count_4pcf6, plus GS_ERR_ARG when no weights are
 * set. */
gs_status gs_count_4pcf6_weighted(gs_graph_t g, int64_t *even_dev, int64_t *odd_dev,
                                  int64_t hub_begin, int64_t hub_end, void *cuda_stream);

/* The smallest bin tuple (b01, b02, b03, b12, b13, b23) of six-bin 4pCF
 * configuration `config` (host call, no device work): tuple_host int32 [6].
 * Errors: GS_ERR_ARG (nbins outside 1..10, config out of range). */
gs_status gs_config_tuple_4pcf6(int nbins, int64_t config, int32_t *tuple_host);

/* Internal 2pCF pair counts: the number of unordered pairs {i, j} in each
 * radial bin, from one sweep of the graph's bin bytes (§III.3: the two-point
 * function on the same graph and binning as the higher-order counts).
 *   hist_dev   uint64 [nbins], device, overwritten
 * Asynchronous. Errors: GS_ERR_ARG (NULL), GS_ERR_CUDA. */
gs_status gs_count_2pcf(gs_graph_t g, uint64_t *hist_dev, void *cuda_stream);

/* Point weights for the weighted counts (§II.1: counts accumulated with
 * signed, normalised data-minus-random weights, the Landy-Szalay and
 * Szapudi-Szalay estimators). The weights are int16 fixed-point values: a
 * caller scales real weights by 2^F (|w| <= 32767), and the sums below are
 * then exact integers in units of 2^(2F) (pairs) and 2^(3F) (triangles).
 *   w_dev  int16 [n], device, in INPUT order; copied (gathered into the
 *          graph's internal order), so the caller may free it afterwards.
 * Asynchronous on cuda_stream; the first call allocates 2n bytes on the
 * graph. Errors: GS_ERR_ARG (NULL), GS_ERR_NOMEM, GS_ERR_CUDA. */
gs_status gs_graph_set_weights(gs_graph_t g, const int16_t *w_dev, void *cuda_stream);

/* Weighted 2pCF: per radial bin, the sum over unordered pairs {i, j} of
 * w_i w_j, exact (§III.3: with data weights summing to +1 and random
 * weights to -1 this is the Landy-Szalay numerator DD - 2DR + RR).
 *   sums_dev  int64 [2 * nbins], device, overwritten: bin b holds a 128-bit
 *             two's-complement integer as (low word at 2b, high word at 2b+1)
 * Asynchronous. Errors: GS_ERR_ARG (NULL, no weights set), GS_ERR_CUDA. */
gs_status gs_count_2pcf_weighted(gs_graph_t g, int64_t *sums_dev, void *cuda_stream);

/* Weighted 3pCF: per sorted-bin configuration (packed index of
 * gs_config_index_3pcf), the sum over triangles {i, j, k} of w_i w_j w_k,
 * exact (§II.1, §II.2: the hub-and-spoke triangle count with each triangle
 * weighted by its three vertex weights).
 *   sums_dev  int64 [2 * gs_config_count_3pcf(nbins)], device, overwritten,
 *             128-bit sums as (low, high) word pairs
 *   hub_begin, hub_end  internal-order hub range, as for gs_count_3pcf
 * Device-resident graphs with at most 32 bins take the byte-map walk (the
 * hub's keys as a byte map of their bins and a parallel map of their
 * weights), others the bitmap walk; GS_COUNT3_WALK = "warp" or "group" asks
 * for the bitmap walk. The call allocates 32 bytes per configuration and SM
 * of scratch (per-block 128-bit slices) before writing sums_dev.
 * Limits: nbins <= 40. Errors: GS_ERR_ARG (NULL, no weights set, nbins,
 * range), GS_ERR_NOMEM, GS_ERR_CAPACITY, GS_ERR_CUDA. */
gs_status gs_count_3pcf_weighted(gs_graph_t g, int64_t *sums_dev, int64_t hub_begin, int64_t hub_end,
                                 void *cuda_stream);

/* Sizes of a built graph (host outputs; any pointer may be NULL).
 *   n           number of points
 *   n_edges     directed edges, sum of degrees (= 2 x pairs)
 *   max_degree  largest |N(i)|
 * Host data only, no device work. Errors: GS_ERR_ARG (NULL graph). */
gs_status gs_graph_info(gs_graph_t g, int64_t *n, int64_t *n_edges, int32_t *max_degree);

/* Work statistics of a built graph (the merge-walk work of §III.1), in the
 * graph's internal order, where f_i = |{j in N(i): j > i}| (forward degree)
 * and b_i = deg_i - f_i:
 *   hub_tail    sum_i C(f_i, 2): hub-tail entries the merge-walk of §III.1
 *               reads over all forward spokes (also the number of candidate
 *               third vertices)
 *   spoke_walk  sum over forward edges (i, j) of f_j = sum_j b_j f_j: spoke-row
 *               entries the merge-walk reads
 *   max_forward largest f_i
 * Computed on the device; the call synchronises cuda_stream. Errors:
 * GS_ERR_ARG (NULL, graph of another device), GS_ERR_NOMEM (24 bytes
 * of scratch), GS_ERR_CUDA. */
typedef struct {
    int64_t n;
    int64_t n_edges;
    int32_t max_degree;
    int32_t max_forward;
    int32_t cells_per_axis;
    int32_t reserved;
    int64_t hub_tail;
    int64_t spoke_walk;
} gs_graph_stats_t;

gs_status gs_graph_stats(gs_graph_t g, gs_graph_stats_t *out, void *cuda_stream);

/* Per-hub work of the 3pCF count, in the graph's internal (hub) order: the
 * forward degree f_i and the spoke-row length of hub i's merge-walks,
 * w_i = sum over the forward spokes j of i of f_j (§III.1: the entries of
 * N(j) beyond j that the intersections of hub i read). The prefix sum of
 * w_i splits [0, n) into contiguous hub ranges of equal work, the partition
 * of the counts across devices (§IV.7: hub windows, no communication).
 *   fwd_dev   int32 [n] or NULL, device, overwritten
 *   walk_dev  int64 [n], device, overwritten
 * Asynchronous (a windowed graph stages its windows one at a time).
 * Errors: GS_ERR_ARG (NULL, graph of another device), GS_ERR_CUDA. */
gs_status gs_graph_hub_work(gs_graph_t g, int32_t *fwd_dev, int64_t *walk_dev, void *cuda_stream);

/* The graph of gs_build_graph with its edge arrays in pinned HOST memory,
 * split into row windows of at most window_edges directed edges (whole cells;
 * a larger cell gets a window of its own). This is the out-of-core mode of
 * §III.5.3 for graphs larger than device memory. The graph holds three
 * device slots of the largest window's size. A 3pCF query runs one tile per
 * (hub window, spoke window >= it) pair that holds work, with the two windows
 * staged in slots; a window already in a slot is not copied again, and the
 * next tile's missing window is copied on a second stream while the current
 * tile runs. The 4pCF counts run one tile per (hub window, spoke windows
 * c1 <= c2) triple. Every triangle and clique lands in exactly one tile, so
 * results equal those of the resident graph bit for bit. gs_build_graph
 * itself switches to this mode when the CSR does not fit in free device
 * memory, or when the environment variable GS_WINDOW_EDGES holds a positive
 * edge count.
 *   window_edges  >= 1
 * Windowed graphs support every count (plain and weighted), the exports,
 * stats and info; the hub-list counts and gs_count_4pcf_parity_static return
 * GS_ERR_ARG. Needs 5 B per edge of host memory. Errors: as gs_build_graph. */
gs_status gs_build_graph_windowed(const int32_t *coords_dev, int64_t n, int64_t box_lu, int periodic,
                                  int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                                  int64_t window_edges, void *cuda_stream, gs_graph_t *out);

/* Row windows of a graph (§III.5.3; host outputs, either pointer may be
 * NULL): n_windows = 0 for a device-resident graph; window_edges_max = the
 * largest window's edge count (all edges when resident). Host data only.
 * Errors: GS_ERR_ARG (NULL graph). */
gs_status gs_graph_windows(gs_graph_t g, int32_t *n_windows, int64_t *window_edges_max);

/* Number of CUDA kernels this library has launched in this process so far
 * (all threads, all devices). */
uint64_t gs_kernel_launches(void);

/* Number of device and pinned-host allocations this library has attempted in
 * this process so far (all threads). A call that allocates nothing leaves it
 * unchanged.
 * Fault injection for tests: when the environment variable GS_FAULT holds
 * "alloc:N" (N >= 1), the N-th allocation inside each public call (counted
 * from the start of the outermost call on the calling thread) fails without
 * allocating, and the call returns GS_ERR_NOMEM having freed what it had
 * allocated. The variable is read at every allocation. */
uint64_t gs_alloc_calls(void);

/* The graph as CSR in INPUT numbering, rows sorted by neighbour id (Eq.(1)).
 *   row_ptr_dev int64 [n+1], device
 *   nbr_dev     int32 [n_edges], device
 *   bin_dev     uint8 [n_edges], device
 * Asynchronous on cuda_stream. Errors: GS_ERR_ARG, GS_ERR_NOMEM, GS_ERR_CUDA. */
gs_status gs_graph_export_csr(gs_graph_t g, int64_t *row_ptr_dev, int32_t *nbr_dev,
                              uint8_t *bin_dev, void *cuda_stream);

/* Selected rows N(i) of the graph (§II.1, Eq.(1)) in INPUT numbering, each
 * sorted.
 *   ids_dev     int32 [count], device, input indices in [0, n)
 *   row_ptr_dev int64 [count+1], device: offsets of the output rows
 *   nbr_dev     int32 [row_ptr_dev[count]] or NULL, device
 *   bin_dev     uint8 [row_ptr_dev[count]], device (needed when nbr_dev is set)
 * With nbr_dev NULL only row_ptr_dev is written, so a caller can size the
 * row arrays first. Synchronises cuda_stream once (index check). Errors:
 * GS_ERR_ARG (NULL, negative count, an index outside [0, n), graph of another
 * device), GS_ERR_NOMEM, GS_ERR_CUDA. */
gs_status gs_graph_export_rows(gs_graph_t g, const int32_t *ids_dev, int64_t count,
                               int64_t *row_ptr_dev, int32_t *nbr_dev, uint8_t *bin_dev,
                               void *cuda_stream);

/* Internal order (the cell order of the §II.1 neighbour search):
 * perm_dev int32 [n], device; perm_dev[p] = input index of the point the
 * graph numbers p (the hub order of the count calls). Asynchronous. Errors:
 * GS_ERR_ARG (NULL, graph of another device), GS_ERR_CUDA. */
gs_status gs_graph_export_perm(gs_graph_t g, int32_t *perm_dev, void *cuda_stream);

/* Number of histogram entries: C(nbins+2, 3) and C(nbins, 3); -1 if nbins is
 * outside 1..255. */
int64_t gs_config_count_3pcf(int nbins);
int64_t gs_config_count_4pcf(int nbins);

/* Packed index of a configuration (host-side, same formula as the device):
 * idx3 of b1 <= b2 <= b3, idx4 of b1 < b2 < b3; -1 if the triple is not in
 * that form or out of range. */
int64_t gs_config_index_3pcf(int nbins, int b1, int b2, int b3);
int64_t gs_config_index_4pcf(int nbins, int b1, int b2, int b3);

/* One call from host arrays to a host histogram: copies coords_host to the
 * device, builds the graph, counts, copies the result back and frees
 * everything, all on cuda_stream; returns once the result is in host memory.
 * Arguments as for gs_build_graph; hist_host / even_host / odd_host are host
 * arrays of the sizes above (pinned memory makes the copies faster).
 * Errors: those of gs_build_graph and of the count, GS_ERR_ARG for a NULL
 * histogram, GS_ERR_NOMEM, GS_ERR_CUDA; the host outputs are written only
 * after the count succeeded. */
gs_status gs_3pcf_from_host(const int32_t *coords_host, int64_t n, int64_t box_lu, int periodic,
                            int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                            uint64_t *hist_host, void *cuda_stream);
gs_status gs_4pcf_parity_from_host(const int32_t *coords_host, int64_t n, int64_t box_lu,
                                   int periodic, int64_t r_max_lu, const int64_t *edges_lu,
                                   int nbins, uint64_t *even_host, int64_t *odd_host,
                                   void *cuda_stream);

/* Measured ceiling of the counts' histogram adds (a measurement aid for the
 * roofline of the triangle count, whose every closed triangle is one
 * shared-memory atomic add of 1 into a histogram; §III.5.2 accumulates into
 * per-gang histograms the same way). Launches two 512-thread blocks per SM
 * that do nothing but such adds into a histogram of ncfg 32-bit counters in
 * shared memory, lanes_active lanes of each warp taking part, and returns
 * the lane-adds retired per second on the whole device.
 *   pattern  0: pseudo-random counters (the count's pattern), 1: one bank
 *            per lane (no conflicts), 2: one counter for all lanes
 * Synchronises cuda_stream; runs for about 20 ms. Errors: GS_ERR_ARG
 * (ncfg outside [32, 27648], pattern, lanes_active outside 1..32),
 * GS_ERR_NOMEM, GS_ERR_CUDA. */
gs_status gs_measure_smem_atomics(int ncfg, int pattern, int lanes_active, double *lane_adds_per_s,
                                  void *cuda_stream);

/* Release a graph and its device memory (NULL is a no-op). Synchronises the
 * device before freeing. */
void gs_graph_free(gs_graph_t g);

/* Message for the calling thread's last non-OK status ("" if none). */
const char *gs_last_error(void);

/* Library version string; it ends in ", checked)" for the checked build
 * (libgramsci_gb_checked.so: the same sources compiled with GS_CHECKED, whose
 * graph build, 3pCF and parity-4pCF kernels test the indices of their memory
 * accesses, skip an access that fails, and make the call return
 * GS_ERR_INTERNAL naming the failed check sites; its calls synchronise their
 * stream to read the check word). */
const char *gs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GRAMSCI_GB_H */
