/*
 * gs_oracle.c -- the CPU oracle for graph-based 3pCF and parity-4pCF counts.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
 * loads or calls this file; only the tests, the smoke check and the timed CPU
 * baseline of the benchmark do. It shares no code, header, table or constant
 * with the CUDA library.
 *
 * It is a plain, slow, obviously correct restatement of what the GRAMSCI v2
 * paper ("Fast Graph-based Higher-Order Clustering Statistics on the GPU")
 * computes, in exact integer arithmetic on lattice coordinates:
 *
 *   - graph: brute force over all pairs (the definition that the kd-tree
 *     search of §II.1 reaches faster), rows sorted by index as Eq.(1)
 *     requires, each neighbour stored with its radial-bin byte (§II.1);
 *   - 3pCF: the hub-and-spoke loop of §II.2, counting each unordered
 *     triangle once (at its lowest-index vertex), with the closing side
 *     re-tested from coordinates instead of a graph lookup;
 *   - parity 4pCF: the signed volume of Eq.(3) over every hub and spoke
 *     triple whose three spoke-spoke pairs are also neighbours (§III.2),
 *     with zero volume given zero odd weight (§III.2, degenerate rule);
 *   - six-bin 4pCF: every tetrahedron once, at its smallest S4-relabelled
 *     bin tuple, with the handedness of Eq.(3) (§II.2, §III.2, §V.2);
 *   - weighted 2pCF, 3pCF and six-bin 4pCF: the same sums with each pair,
 *     triangle or tetrahedron weighted by the product of its signed integer
 *     point weights (§II.1, §III.3), exact in 128 bits;
 *   - brute force over all triples / quadruples, with no graph at all.
 *
 * Conventions (readings where the paper is silent):
 *   - lattice coordinates in [0, box); periodic boxes use the minimum image
 *     (delta -= box if 2*delta >= box, delta += box if 2*delta < -box);
 *   - a pair (i != j) is an edge iff e_0^2 <= d^2 < e_nb^2, with bin b the one
 *     for which e_b^2 <= d^2 < e_{b+1}^2 (half-open bins on squared integers);
 *   - 3pCF bins are sorted b1 <= b2 <= b3 and packed lexicographically;
 *     4pCF spokes are ordered by hub bin b1 < b2 < b3 (distinct bins only),
 *     packed lexicographically, and the volume uses r_is = x_s - x_i with
 *     the spokes in that bin order; odd += sign(V), sign(0) = 0.
 *
 * Parallelism: hubs are shared among pthreads through an atomic cursor; each
 * thread owns a private histogram and the integer histograms are summed at
 * the end, so the result does not depend on the thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>
#include <stdatomic.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* threads                                                                   */

static int g_threads = 0;

int oracle_set_threads(int t) { g_threads = t; return g_threads; }

int oracle_threads(void)
{
    if (g_threads > 0) return g_threads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

typedef void (*hub_fn)(void *ctx, int tid, int64_t i);

typedef struct {
    void *ctx;
    hub_fn fn;
    int64_t n;
    int64_t chunk;
    _Atomic int64_t next;
} pool_t;

typedef struct { pool_t *p; int tid; } worker_arg_t;

static void *worker(void *arg)
{
    worker_arg_t *w = (worker_arg_t *)arg;
    pool_t *p = w->p;
    for (;;) {
        int64_t s = atomic_fetch_add(&p->next, p->chunk);
        if (s >= p->n) break;
        int64_t e = s + p->chunk < p->n ? s + p->chunk : p->n;
        for (int64_t i = s; i < e; ++i) p->fn(p->ctx, w->tid, i);
    }
    return NULL;
}

/* Run fn(ctx, tid, i) for every i in [begin, end) on nt threads. */
static void parallel_for(int64_t begin, int64_t end, int nt, hub_fn fn, void *ctx)
{
    pool_t p;
    p.ctx = ctx; p.fn = fn; p.n = end; p.chunk = 4;
    atomic_init(&p.next, begin);
    if (nt <= 1) {
        worker_arg_t w = { &p, 0 };
        worker(&w);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    worker_arg_t *wa = (worker_arg_t *)malloc(sizeof(worker_arg_t) * (size_t)nt);
    for (int t = 0; t < nt; ++t) {
        wa[t].p = &p; wa[t].tid = t;
        pthread_create(&th[t], NULL, worker, &wa[t]);
    }
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
    free(th);
    free(wa);
}

/* ------------------------------------------------------------------------ */
/* the pair rule                                                             */

typedef struct {
    const int32_t *xyz;   /* [n][3] */
    int64_t n;
    int64_t box;
    int periodic;
    const int64_t *edges; /* [nb+1] lattice units */
    int nb;
} cat_t;

/* Component of the displacement x_b - x_a along one axis. */
static int64_t axis_delta(int64_t a, int64_t b, int64_t box, int periodic)
{
    int64_t d = b - a;
    if (periodic) {
        if (2 * d >= box) d -= box;
        else if (2 * d < -box) d += box;
    }
    return d;
}

static void displacement(const cat_t *c, int64_t a, int64_t b, int64_t r[3])
{
    for (int ax = 0; ax < 3; ++ax)
        r[ax] = axis_delta(c->xyz[3 * a + ax], c->xyz[3 * b + ax], c->box, c->periodic);
}

static int64_t dist2(const cat_t *c, int64_t a, int64_t b)
{
    int64_t r[3];
    displacement(c, a, b, r);
    return r[0] * r[0] + r[1] * r[1] + r[2] * r[2];
}

/* Radial bin of the pair (a, b), or -1 when it is not an edge. */
static int pair_bin(const cat_t *c, int64_t a, int64_t b)
{
    if (a == b) return -1;
    int64_t d2 = dist2(c, a, b);
    for (int k = 0; k < c->nb; ++k) {
        int64_t lo = c->edges[k], hi = c->edges[k + 1];
        if (lo * lo <= d2 && d2 < hi * hi) return k;
    }
    return -1;
}

/* ------------------------------------------------------------------------ */
/* configuration indices by enumeration                                      */

/* Lexicographic rank of every sorted triple b1 <= b2 <= b3, as a dense nb^3 table. */
static int32_t *table3(int nb)
{
    int32_t *t = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb * nb * nb);
    int32_t c = 0;
    for (int a = 0; a < nb; ++a)
        for (int b = a; b < nb; ++b)
            for (int d = b; d < nb; ++d)
                t[((size_t)a * nb + b) * nb + d] = c++;
    return t;
}

/* Lexicographic rank of every strictly increasing triple b1 < b2 < b3. */
static int32_t *table4(int nb)
{
    int32_t *t = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb * nb * nb);
    int32_t c = 0;
    for (int a = 0; a < nb; ++a)
        for (int b = a + 1; b < nb; ++b)
            for (int d = b + 1; d < nb; ++d)
                t[((size_t)a * nb + b) * nb + d] = c++;
    return t;
}

int64_t oracle_nconfig3(int nb) { return (int64_t)nb * (nb + 1) * (nb + 2) / 6; }
int64_t oracle_nconfig4(int nb) { return (int64_t)nb * (nb - 1) * (nb - 2) / 6; }

static void sort3(int v[3])
{
    int t;
    if (v[0] > v[1]) { t = v[0]; v[0] = v[1]; v[1] = t; }
    if (v[1] > v[2]) { t = v[1]; v[1] = v[2]; v[2] = t; }
    if (v[0] > v[1]) { t = v[0]; v[0] = v[1]; v[1] = t; }
}

/* ------------------------------------------------------------------------ */
/* graph by brute force over all pairs                                       */

typedef struct {
    cat_t c;
    int64_t *deg;
    const int64_t *row_ptr;
    int32_t *nbr;
    uint8_t *bin;
} graph_ctx_t;

static void degree_hub(void *vctx, int tid, int64_t i)
{
    (void)tid;
    graph_ctx_t *g = (graph_ctx_t *)vctx;
    int64_t d = 0;
    for (int64_t j = 0; j < g->c.n; ++j)
        if (pair_bin(&g->c, i, j) >= 0) ++d;
    g->deg[i] = d;
}

static void fill_hub(void *vctx, int tid, int64_t i)
{
    (void)tid;
    graph_ctx_t *g = (graph_ctx_t *)vctx;
    int64_t p = g->row_ptr[i];
    for (int64_t j = 0; j < g->c.n; ++j) {          /* j ascending: rows come out sorted */
        int b = pair_bin(&g->c, i, j);
        if (b >= 0) { g->nbr[p] = (int32_t)j; g->bin[p] = (uint8_t)b; ++p; }
    }
}

/* deg[i] = |N(i)|; returns the directed edge total sum(deg). */
int64_t oracle_graph_degrees(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                             const int64_t *edges, int nb, int64_t *deg)
{
    graph_ctx_t g = { { xyz, n, box, periodic, edges, nb }, deg, NULL, NULL, NULL };
    parallel_for(0, n, oracle_threads(), degree_hub, &g);
    int64_t e = 0;
    for (int64_t i = 0; i < n; ++i) e += deg[i];
    return e;
}

/* Fill rows [row_ptr[i], row_ptr[i+1]) with sorted neighbour ids and bins. */
void oracle_graph_fill(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                       const int64_t *edges, int nb, const int64_t *row_ptr,
                       int32_t *nbr, uint8_t *bin)
{
    graph_ctx_t g = { { xyz, n, box, periodic, edges, nb }, NULL, row_ptr, nbr, bin };
    parallel_for(0, n, oracle_threads(), fill_hub, &g);
}

/* One row N(i) by brute force; returns its length. nbr/bin hold up to n entries. */
int64_t oracle_row(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                   const int64_t *edges, int nb, int64_t i, int32_t *nbr, uint8_t *bin)
{
    cat_t c = { xyz, n, box, periodic, edges, nb };
    int64_t p = 0;
    for (int64_t j = 0; j < n; ++j) {
        int b = pair_bin(&c, i, j);
        if (b >= 0) { nbr[p] = (int32_t)j; bin[p] = (uint8_t)b; ++p; }
    }
    return p;
}

/* ------------------------------------------------------------------------ */
/* 3pCF: hub-and-spoke loop over the graph                                   */

typedef struct {
    cat_t c;
    const int64_t *row_ptr;
    const int32_t *nbr;
    const uint8_t *bin;
    const int32_t *t3;
    int64_t ncfg;
    uint64_t *hist;        /* [threads][ncfg] */
} tri_ctx_t;

static void tri_hub(void *vctx, int tid, int64_t i)
{
    tri_ctx_t *t = (tri_ctx_t *)vctx;
    uint64_t *h = t->hist + (size_t)tid * (size_t)t->ncfg;
    int nb = t->c.nb;
    for (int64_t a = t->row_ptr[i]; a < t->row_ptr[i + 1]; ++a) {
        int64_t j = t->nbr[a];
        if (j <= i) continue;                      /* spoke j > hub i */
        for (int64_t b = a + 1; b < t->row_ptr[i + 1]; ++b) {
            int64_t k = t->nbr[b];                 /* k > j since the row is sorted */
            int bjk = pair_bin(&t->c, j, k);       /* closing side, from coordinates */
            if (bjk < 0) continue;
            int v[3] = { t->bin[a], t->bin[b], bjk };
            sort3(v);
            h[t->t3[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += 1;
        }
    }
}

static void reduce_u64(uint64_t *out, const uint64_t *parts, int nt, int64_t m)
{
    memset(out, 0, sizeof(uint64_t) * (size_t)m);
    for (int t = 0; t < nt; ++t)
        for (int64_t x = 0; x < m; ++x) out[x] += parts[(size_t)t * m + x];
}

static void reduce_i64(int64_t *out, const int64_t *parts, int nt, int64_t m)
{
    memset(out, 0, sizeof(int64_t) * (size_t)m);
    for (int t = 0; t < nt; ++t)
        for (int64_t x = 0; x < m; ++x) out[x] += parts[(size_t)t * m + x];
}

/* hist[C(nb+2,3)]: triangles per sorted bin triple, hubs i in [hub_begin, hub_end). */
void oracle_3pcf_range(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                       const int64_t *edges, int nb, const int64_t *row_ptr,
                       const int32_t *nbr, const uint8_t *bin,
                       int64_t hub_begin, int64_t hub_end, uint64_t *hist)
{
    int nt = oracle_threads();
    tri_ctx_t t;
    t.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    t.row_ptr = row_ptr; t.nbr = nbr; t.bin = bin;
    t.t3 = table3(nb);
    t.ncfg = oracle_nconfig3(nb);
    t.hist = (uint64_t *)calloc((size_t)nt * (size_t)t.ncfg, sizeof(uint64_t));
    if (hub_end > hub_begin) parallel_for(hub_begin, hub_end, nt, tri_hub, &t);
    reduce_u64(hist, t.hist, nt, t.ncfg);
    free(t.hist);
    free((void *)t.t3);
}

void oracle_3pcf(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                 const int64_t *edges, int nb, const int64_t *row_ptr,
                 const int32_t *nbr, const uint8_t *bin, uint64_t *hist)
{
    oracle_3pcf_range(xyz, n, box, periodic, edges, nb, row_ptr, nbr, bin, 0, n, hist);
}

/* ------------------------------------------------------------------------ */
/* parity 4pCF: every hub, every spoke triple forming a clique               */

typedef struct {
    cat_t c;
    const int64_t *row_ptr;
    const int32_t *nbr;
    const uint8_t *bin;
    const int32_t *t4;
    int64_t ncfg;
    uint64_t *even;       /* [threads][ncfg] */
    int64_t *odd;         /* [threads][ncfg] */
} quad_ctx_t;

/* Signed volume (r1 x r2) . r3, Eq.(3). */
static int64_t triple_product(const int64_t r1[3], const int64_t r2[3], const int64_t r3[3])
{
    int64_t cx = r1[1] * r2[2] - r1[2] * r2[1];
    int64_t cy = r1[2] * r2[0] - r1[0] * r2[2];
    int64_t cz = r1[0] * r2[1] - r1[1] * r2[0];
    return cx * r3[0] + cy * r3[1] + cz * r3[2];
}

/* Add one (hub, spoke triple) to the even and odd channels. The spokes are
 * put in hub-bin order before the volume is taken. */
static void add_clique(const cat_t *c, const int32_t *t4, uint64_t *even, int64_t *odd,
                       int64_t hub, const int64_t s[3], const int b[3])
{
    if (b[0] == b[1] || b[0] == b[2] || b[1] == b[2]) return;
    int order[3] = { 0, 1, 2 };
    for (int x = 0; x < 3; ++x)
        for (int y = x + 1; y < 3; ++y)
            if (b[order[y]] < b[order[x]]) { int tmp = order[x]; order[x] = order[y]; order[y] = tmp; }
    int64_t r[3][3];
    for (int q = 0; q < 3; ++q) displacement(c, hub, s[order[q]], r[q]);
    int64_t v = triple_product(r[0], r[1], r[2]);
    int nb = c->nb;
    int idx = t4[((size_t)b[order[0]] * nb + b[order[1]]) * nb + b[order[2]]];
    even[idx] += 1;
    odd[idx] += (v > 0) - (v < 0);
}

static void quad_hub(void *vctx, int tid, int64_t i)
{
    quad_ctx_t *q = (quad_ctx_t *)vctx;
    uint64_t *ev = q->even + (size_t)tid * (size_t)q->ncfg;
    int64_t *od = q->odd + (size_t)tid * (size_t)q->ncfg;
    int64_t r0 = q->row_ptr[i], r1 = q->row_ptr[i + 1];
    for (int64_t a = r0; a < r1; ++a)
        for (int64_t b = a + 1; b < r1; ++b) {
            if (pair_bin(&q->c, q->nbr[a], q->nbr[b]) < 0) continue;
            for (int64_t d = b + 1; d < r1; ++d) {
                if (pair_bin(&q->c, q->nbr[a], q->nbr[d]) < 0) continue;
                if (pair_bin(&q->c, q->nbr[b], q->nbr[d]) < 0) continue;
                int64_t s[3] = { q->nbr[a], q->nbr[b], q->nbr[d] };
                int bb[3] = { q->bin[a], q->bin[b], q->bin[d] };
                add_clique(&q->c, q->t4, ev, od, i, s, bb);
            }
        }
}

/* even/odd[C(nb,3)] over hubs i in [hub_begin, hub_end). */
void oracle_4pcf_parity_range(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                              const int64_t *edges, int nb, const int64_t *row_ptr,
                              const int32_t *nbr, const uint8_t *bin,
                              int64_t hub_begin, int64_t hub_end,
                              uint64_t *even, int64_t *odd)
{
    int nt = oracle_threads();
    quad_ctx_t q;
    q.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    q.row_ptr = row_ptr; q.nbr = nbr; q.bin = bin;
    q.t4 = table4(nb < 3 ? 3 : nb);
    q.ncfg = oracle_nconfig4(nb);
    size_t m = q.ncfg > 0 ? (size_t)q.ncfg : 1;
    q.even = (uint64_t *)calloc((size_t)nt * m, sizeof(uint64_t));
    q.odd = (int64_t *)calloc((size_t)nt * m, sizeof(int64_t));
    if (q.ncfg > 0) {
        if (hub_end > hub_begin) parallel_for(hub_begin, hub_end, nt, quad_hub, &q);
        reduce_u64(even, q.even, nt, q.ncfg);
        reduce_i64(odd, q.odd, nt, q.ncfg);
    }
    free(q.even); free(q.odd);
    free((void *)q.t4);
}

void oracle_4pcf_parity(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                        const int64_t *edges, int nb, const int64_t *row_ptr,
                        const int32_t *nbr, const uint8_t *bin, uint64_t *even, int64_t *odd)
{
    oracle_4pcf_parity_range(xyz, n, box, periodic, edges, nb, row_ptr, nbr, bin, 0, n, even, odd);
}

/* Per-hub work with rows found by brute force over all points (no graph):
 * for sampled checks at full size. Each thread keeps its own row buffer. */
typedef struct {
    cat_t c;
    const int64_t *hubs;
    const int32_t *t;       /* configuration table (3pCF: table3, 4pCF: table4) */
    int64_t ncfg;
    uint64_t *even;         /* [threads][ncfg] (3pCF: the histogram) */
    int64_t *odd;           /* [threads][ncfg] (4pCF only) */
    int32_t **row;          /* [threads][n] */
    uint8_t **rb;           /* [threads][n] */
} hubs_ctx_t;

/* Every triangle {i, j, k} with j, k in N(i), j < k, (j, k) an edge: the
 * hub-and-spoke loop of §II.2 without the forward restriction. */
static void tri_listed_hub(void *vctx, int tid, int64_t h)
{
    hubs_ctx_t *x = (hubs_ctx_t *)vctx;
    const cat_t *c = &x->c;
    int64_t i = x->hubs[h];
    int32_t *row = x->row[tid];
    uint8_t *rb = x->rb[tid];
    uint64_t *hist = x->even + (size_t)tid * (size_t)x->ncfg;
    int nb = c->nb;
    int64_t m = oracle_row(c->xyz, c->n, c->box, c->periodic, c->edges, nb, i, row, rb);
    for (int64_t a = 0; a < m; ++a)
        for (int64_t b = a + 1; b < m; ++b) {
            int bjk = pair_bin(c, row[a], row[b]);
            if (bjk < 0) continue;
            int v[3] = { rb[a], rb[b], bjk };
            sort3(v);
            hist[x->t[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += 1;
        }
}

static void quad_listed_hub(void *vctx, int tid, int64_t h)
{
    hubs_ctx_t *x = (hubs_ctx_t *)vctx;
    const cat_t *c = &x->c;
    int64_t i = x->hubs[h];
    int32_t *row = x->row[tid];
    uint8_t *rb = x->rb[tid];
    uint64_t *ev = x->even + (size_t)tid * (size_t)x->ncfg;
    int64_t *od = x->odd + (size_t)tid * (size_t)x->ncfg;
    int64_t m = oracle_row(c->xyz, c->n, c->box, c->periodic, c->edges, c->nb, i, row, rb);
    for (int64_t a = 0; a < m; ++a)
        for (int64_t b = a + 1; b < m; ++b) {
            if (pair_bin(c, row[a], row[b]) < 0) continue;
            for (int64_t d = b + 1; d < m; ++d) {
                if (pair_bin(c, row[a], row[d]) < 0) continue;
                if (pair_bin(c, row[b], row[d]) < 0) continue;
                int64_t sp[3] = { row[a], row[b], row[d] };
                int bb[3] = { rb[a], rb[b], rb[d] };
                add_clique(c, x->t, ev, od, i, sp, bb);
            }
        }
}

static void run_listed(hubs_ctx_t *x, int64_t nh, hub_fn fn, int nt)
{
    size_t nn = (size_t)(x->c.n > 0 ? x->c.n : 1);
    x->row = (int32_t **)malloc(sizeof(int32_t *) * (size_t)nt);
    x->rb = (uint8_t **)malloc(sizeof(uint8_t *) * (size_t)nt);
    for (int t = 0; t < nt; ++t) {
        x->row[t] = (int32_t *)malloc(sizeof(int32_t) * nn);
        x->rb[t] = (uint8_t *)malloc(nn);
    }
    parallel_for(0, nh, nt, fn, x);
    for (int t = 0; t < nt; ++t) { free(x->row[t]); free(x->rb[t]); }
    free(x->row); free(x->rb);
}

/* 3pCF triangles incident to each listed hub (input indices), summed. */
void oracle_3pcf_hubs(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                      const int64_t *edges, int nb, const int64_t *hubs, int64_t nh, uint64_t *hist)
{
    int nt = oracle_threads();
    hubs_ctx_t x;
    memset(&x, 0, sizeof(x));
    x.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    x.hubs = hubs;
    x.t = table3(nb);
    x.ncfg = oracle_nconfig3(nb);
    x.even = (uint64_t *)calloc((size_t)nt * (size_t)x.ncfg, sizeof(uint64_t));
    run_listed(&x, nh, tri_listed_hub, nt);
    reduce_u64(hist, x.even, nt, x.ncfg);
    free(x.even);
    free((void *)x.t);
}

/* Parity-4pCF contribution of the listed hubs only, each row found by brute
 * force over all points (no graph needed: for sampled checks at full size). */
void oracle_4pcf_parity_hubs(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                             const int64_t *edges, int nb, const int64_t *hubs, int64_t nh,
                             uint64_t *even, int64_t *odd)
{
    int64_t ncfg = oracle_nconfig4(nb);
    if (ncfg <= 0) return;
    int nt = oracle_threads();
    hubs_ctx_t x;
    memset(&x, 0, sizeof(x));
    x.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    x.hubs = hubs;
    x.t = table4(nb);
    x.ncfg = ncfg;
    x.even = (uint64_t *)calloc((size_t)nt * (size_t)ncfg, sizeof(uint64_t));
    x.odd = (int64_t *)calloc((size_t)nt * (size_t)ncfg, sizeof(int64_t));
    run_listed(&x, nh, quad_listed_hub, nt);
    reduce_u64(even, x.even, nt, ncfg);
    reduce_i64(odd, x.odd, nt, ncfg);
    free(x.even); free(x.odd);
    free((void *)x.t);
}

/* ------------------------------------------------------------------------ */
/* brute force with no graph                                                 */

typedef struct {
    cat_t c;
    const int32_t *t;
    int64_t ncfg;
    uint64_t *hist;
    int64_t *odd;
} brute_ctx_t;

static void brute3_i(void *vctx, int tid, int64_t i)
{
    brute_ctx_t *b = (brute_ctx_t *)vctx;
    uint64_t *h = b->hist + (size_t)tid * (size_t)b->ncfg;
    int nb = b->c.nb;
    for (int64_t j = i + 1; j < b->c.n; ++j) {
        int bij = pair_bin(&b->c, i, j);
        if (bij < 0) continue;
        for (int64_t k = j + 1; k < b->c.n; ++k) {
            int bik = pair_bin(&b->c, i, k);
            if (bik < 0) continue;
            int bjk = pair_bin(&b->c, j, k);
            if (bjk < 0) continue;
            int v[3] = { bij, bik, bjk };
            sort3(v);
            h[b->t[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += 1;
        }
    }
}

/* O(N^3) over all unordered triples i < j < k. */
void oracle_brute3(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                   const int64_t *edges, int nb, uint64_t *hist)
{
    int nt = oracle_threads();
    brute_ctx_t b;
    b.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    b.t = table3(nb);
    b.ncfg = oracle_nconfig3(nb);
    b.hist = (uint64_t *)calloc((size_t)nt * (size_t)b.ncfg, sizeof(uint64_t));
    b.odd = NULL;
    parallel_for(0, n, nt, brute3_i, &b);
    reduce_u64(hist, b.hist, nt, b.ncfg);
    free(b.hist);
    free((void *)b.t);
}

static void brute4_i(void *vctx, int tid, int64_t i)
{
    brute_ctx_t *b = (brute_ctx_t *)vctx;
    uint64_t *ev = b->hist + (size_t)tid * (size_t)b->ncfg;
    int64_t *od = b->odd + (size_t)tid * (size_t)b->ncfg;
    int64_t n = b->c.n;
    for (int64_t j = 0; j < n; ++j) {
        int bij = pair_bin(&b->c, i, j);
        if (bij < 0) continue;
        for (int64_t k = j + 1; k < n; ++k) {
            int bik = pair_bin(&b->c, i, k);
            if (bik < 0 || pair_bin(&b->c, j, k) < 0) continue;
            for (int64_t l = k + 1; l < n; ++l) {
                int bil = pair_bin(&b->c, i, l);
                if (bil < 0 || pair_bin(&b->c, j, l) < 0 || pair_bin(&b->c, k, l) < 0) continue;
                int64_t s[3] = { j, k, l };
                int bb[3] = { bij, bik, bil };
                add_clique(&b->c, b->t, ev, od, i, s, bb);
            }
        }
    }
}

/* O(N^4): every hub i and every triple j < k < l of other points. */
void oracle_brute4(const int32_t *xyz, int64_t n, int64_t box, int periodic,
                   const int64_t *edges, int nb, uint64_t *even, int64_t *odd)
{
    int nt = oracle_threads();
    brute_ctx_t b;
    b.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    b.t = table4(nb < 3 ? 3 : nb);
    b.ncfg = oracle_nconfig4(nb);
    if (b.ncfg <= 0) { free((void *)b.t); return; }
    b.hist = (uint64_t *)calloc((size_t)nt * (size_t)b.ncfg, sizeof(uint64_t));
    b.odd = (int64_t *)calloc((size_t)nt * (size_t)b.ncfg, sizeof(int64_t));
    parallel_for(0, n, nt, brute4_i, &b);
    reduce_u64(even, b.hist, nt, b.ncfg);
    reduce_i64(odd, b.odd, nt, b.ncfg);
    free(b.hist); free(b.odd);
    free((void *)b.t);
}

/* ------------------------------------------------------------------------ */
/* six-edge-bin 4pCF with parity channels                                    */
/*
 * A tetrahedron is four points whose six pairs are all edges; each counts
 * once. Its configuration is the lexicographically smallest tuple
 * (b01, b02, b03, b12, b13, b23) over the 24 orderings (v0, v1, v2, v3) of its
 * vertices, where b_ab is the bin of the pair (v_a, v_b); configurations are
 * numbered in lexicographic order of their smallest tuples. The odd channel
 * adds sign(V) with V = det[x_v1 - x_v0; x_v2 - x_v0; x_v3 - x_v0] for an
 * ordering that reaches the smallest tuple -- and 0 when orderings of both
 * permutation parities reach it (an achiral configuration: the sign would
 * depend on labels) or when V = 0. (GRAMSCI v2 §II.2 tetrahedra, §III.2
 * Eq.(3); 276 configurations for 4 bins, §V.2.)
 */

/* the 24 orderings of (0,1,2,3) and their parities, generated by swaps */
static int g_perm[24][4];
static int g_perm_par[24];
static int g_perm_ready = 0;

static void make_perms(void)
{
    if (g_perm_ready) return;
    int c = 0;
    for (int a = 0; a < 4; ++a)
        for (int b = 0; b < 4; ++b)
            for (int d = 0; d < 4; ++d)
                for (int e = 0; e < 4; ++e) {
                    if (a == b || a == d || a == e || b == d || b == e || d == e) continue;
                    int p[4] = { a, b, d, e };
                    int inv = 0;
                    for (int x = 0; x < 4; ++x)
                        for (int y = x + 1; y < 4; ++y) inv += p[x] > p[y];
                    for (int x = 0; x < 4; ++x) g_perm[c][x] = p[x];
                    g_perm_par[c] = inv & 1;
                    ++c;
                }
    g_perm_ready = 1;
}

/* bins of the six pairs of an ordered 4-tuple of points */
static int tuple_of(const int bm[4][4], const int *o, int t[6])
{
    t[0] = bm[o[0]][o[1]]; t[1] = bm[o[0]][o[2]]; t[2] = bm[o[0]][o[3]];
    t[3] = bm[o[1]][o[2]]; t[4] = bm[o[1]][o[3]]; t[5] = bm[o[2]][o[3]];
    return 0;
}

static int cmp6(const int *a, const int *b)
{
    for (int k = 0; k < 6; ++k) {
        if (a[k] < b[k]) return -1;
        if (a[k] > b[k]) return 1;
    }
    return 0;
}

/* smallest tuple over all orderings; *par = parity of a minimal ordering
 * relative to (0,1,2,3), *chiral = 0 if minimal orderings of both parities
 * exist; best_order receives one minimal ordering */
static void canonical(const int bm[4][4], int best[6], int *chiral, int best_order[4])
{
    make_perms();
    int seen_even = 0, seen_odd = 0;
    int have = 0;
    for (int q = 0; q < 24; ++q) {
        int t[6];
        tuple_of(bm, g_perm[q], t);
        int c = have ? cmp6(t, best) : -1;
        if (c < 0) {
            memcpy(best, t, sizeof(t));
            for (int x = 0; x < 4; ++x) best_order[x] = g_perm[q][x];
            seen_even = !g_perm_par[q];
            seen_odd = g_perm_par[q];
            have = 1;
        } else if (c == 0) {
            if (g_perm_par[q]) seen_odd = 1; else seen_even = 1;
        }
    }
    *chiral = !(seen_even && seen_odd);
}

/* number of configurations for nb bins, and the index of a canonical tuple:
 * rank among all canonical tuples in lexicographic order (by enumeration) */
static int64_t six_count_and_index(int nb, const int *want)
{
    int64_t rank = 0;
    int t[6];
    for (t[0] = 0; t[0] < nb; ++t[0])
    for (t[1] = 0; t[1] < nb; ++t[1])
    for (t[2] = 0; t[2] < nb; ++t[2])
    for (t[3] = 0; t[3] < nb; ++t[3])
    for (t[4] = 0; t[4] < nb; ++t[4])
    for (t[5] = 0; t[5] < nb; ++t[5]) {
        /* is t its own smallest relabelling? rebuild the pair matrix */
        int bm[4][4];
        bm[0][1] = bm[1][0] = t[0]; bm[0][2] = bm[2][0] = t[1]; bm[0][3] = bm[3][0] = t[2];
        bm[1][2] = bm[2][1] = t[3]; bm[1][3] = bm[3][1] = t[4]; bm[2][3] = bm[3][2] = t[5];
        int best[6], ch, ord[4];
        canonical(bm, best, &ch, ord);
        if (cmp6(best, t) != 0) continue;
        if (want && cmp6(want, t) == 0) return rank;
        ++rank;
    }
    return want ? -1 : rank;
}

int64_t oracle_nconfig6(int nb) { return six_count_and_index(nb, NULL); }

/* Dense table: configuration index of every canonical tuple, by packed tuple. */
static int32_t *six_index_table(int nb)
{
    size_t nt = 1;
    for (int k = 0; k < 6; ++k) nt *= (size_t)nb;
    int32_t *tab = (int32_t *)malloc(sizeof(int32_t) * nt);
    for (size_t x = 0; x < nt; ++x) tab[x] = -1;
    int32_t rank = 0;
    int t[6];
    for (t[0] = 0; t[0] < nb; ++t[0])
    for (t[1] = 0; t[1] < nb; ++t[1])
    for (t[2] = 0; t[2] < nb; ++t[2])
    for (t[3] = 0; t[3] < nb; ++t[3])
    for (t[4] = 0; t[4] < nb; ++t[4])
    for (t[5] = 0; t[5] < nb; ++t[5]) {
        int bm[4][4];
        bm[0][1] = bm[1][0] = t[0]; bm[0][2] = bm[2][0] = t[1]; bm[0][3] = bm[3][0] = t[2];
        bm[1][2] = bm[2][1] = t[3]; bm[1][3] = bm[3][1] = t[4]; bm[2][3] = bm[3][2] = t[5];
        int best[6], ch, ord[4];
        canonical(bm, best, &ch, ord);
        if (cmp6(best, t) != 0) continue;
        size_t p = 0;
        for (int k = 0; k < 6; ++k) p = p * (size_t)nb + (size_t)t[k];
        tab[p] = rank++;
    }
    return tab;
}

/* Configuration index of the tetrahedron of points q[0..3] (catalogue
 * indices) and its odd-channel sign: sign(V) for an ordering reaching the
 * smallest tuple, 0 if the configuration is achiral or V = 0. */
static int tetra_class(const cat_t *c, const int32_t *tab, const int64_t q[4], int *sign)
{
    int bm[4][4];
    for (int a = 0; a < 4; ++a)
        for (int b = a + 1; b < 4; ++b) bm[a][b] = bm[b][a] = pair_bin(c, q[a], q[b]);
    int best[6], chiral, ord[4];
    canonical(bm, best, &chiral, ord);
    size_t p = 0;
    for (int k = 0; k < 6; ++k) p = p * (size_t)c->nb + (size_t)best[k];
    *sign = 0;
    if (chiral) {
        int64_t r[3][3];
        for (int k = 0; k < 3; ++k) displacement(c, q[ord[0]], q[ord[k + 1]], r[k]);
        int64_t v = triple_product(r[0], r[1], r[2]);
        *sign = (v > 0) - (v < 0);
    }
    return tab[p];
}

/* One tetrahedron of points q[0..3]. */
static void add_tetra(const cat_t *c, const int32_t *tab, const int64_t q[4], uint64_t *even, int64_t *odd)
{
    int sg;
    int idx = tetra_class(c, tab, q, &sg);
    even[idx] += 1;
    odd[idx] += sg;
}

typedef struct {
    cat_t c;
    const int64_t *row_ptr;
    const int32_t *nbr;
    const int32_t *tab;
    int64_t ncfg;
    uint64_t *even;
    int64_t *odd;
} six_ctx_t;

/* hub i = the lowest-index vertex; j < k < l forward neighbours, pairwise adjacent */
static void six_hub(void *vctx, int tid, int64_t i)
{
    six_ctx_t *x = (six_ctx_t *)vctx;
    uint64_t *ev = x->even + (size_t)tid * (size_t)x->ncfg;
    int64_t *od = x->odd + (size_t)tid * (size_t)x->ncfg;
    int64_t r0 = x->row_ptr[i], r1 = x->row_ptr[i + 1];
    for (int64_t a = r0; a < r1; ++a) {
        if (x->nbr[a] <= i) continue;
        for (int64_t b = a + 1; b < r1; ++b) {
            if (pair_bin(&x->c, x->nbr[a], x->nbr[b]) < 0) continue;
            for (int64_t d = b + 1; d < r1; ++d) {
                if (pair_bin(&x->c, x->nbr[a], x->nbr[d]) < 0) continue;
                if (pair_bin(&x->c, x->nbr[b], x->nbr[d]) < 0) continue;
                int64_t q[4] = { i, x->nbr[a], x->nbr[b], x->nbr[d] };
                add_tetra(&x->c, x->tab, q, ev, od);
            }
        }
    }
}

void oracle_4pcf6(const int32_t *xyz, int64_t n, int64_t box, int periodic, const int64_t *edges, int nb,
                  const int64_t *row_ptr, const int32_t *nbr, int64_t hub_begin, int64_t hub_end,
                  uint64_t *even, int64_t *odd)
{
    int nt = oracle_threads();
    six_ctx_t x;
    x.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    x.row_ptr = row_ptr; x.nbr = nbr;
    x.tab = six_index_table(nb);
    x.ncfg = oracle_nconfig6(nb);
    x.even = (uint64_t *)calloc((size_t)nt * (size_t)x.ncfg, sizeof(uint64_t));
    x.odd = (int64_t *)calloc((size_t)nt * (size_t)x.ncfg, sizeof(int64_t));
    if (hub_end > hub_begin) parallel_for(hub_begin, hub_end, nt, six_hub, &x);
    reduce_u64(even, x.even, nt, x.ncfg);
    reduce_i64(odd, x.odd, nt, x.ncfg);
    free(x.even); free(x.odd);
    free((void *)x.tab);
}

/* O(N^4 / 24): every set of four points whose six pairs are edges. */
void oracle_brute4six(const int32_t *xyz, int64_t n, int64_t box, int periodic, const int64_t *edges, int nb,
                      uint64_t *even, int64_t *odd)
{
    cat_t c = { xyz, n, box, periodic, edges, nb };
    int32_t *tab = six_index_table(nb);
    int64_t ncfg = oracle_nconfig6(nb);
    memset(even, 0, sizeof(uint64_t) * (size_t)ncfg);
    memset(odd, 0, sizeof(int64_t) * (size_t)ncfg);
    for (int64_t a = 0; a < n; ++a)
        for (int64_t b = a + 1; b < n; ++b) {
            if (pair_bin(&c, a, b) < 0) continue;
            for (int64_t d = b + 1; d < n; ++d) {
                if (pair_bin(&c, a, d) < 0 || pair_bin(&c, b, d) < 0) continue;
                for (int64_t e = d + 1; e < n; ++e) {
                    if (pair_bin(&c, a, e) < 0 || pair_bin(&c, b, e) < 0 || pair_bin(&c, d, e) < 0) continue;
                    int64_t q[4] = { a, b, d, e };
                    add_tetra(&c, tab, q, even, odd);
                }
            }
        }
    free(tab);
}

/* The configuration index of one canonical tuple, -1 if it is not canonical. */
int64_t oracle_config_index6(int nb, const int32_t *t)
{
    int w[6];
    for (int k = 0; k < 6; ++k) w[k] = t[k];
    return six_count_and_index(nb, w);
}

/* ------------------------------------------------------------------------ */
/* weighted 2pCF and 3pCF (signed integer weights, exact)                    */
/*
 * GRAMSCI v2 §II.1 / §III.3: counts are accumulated with signed per-point
 * weights (data positive, randoms negative), so that the pair sum is the
 * Landy-Szalay numerator DD - 2DR + RR. Here the weights are integers (a
 * caller scales real weights by 2^F); sums are exact, in 128 bits, written
 * as two int64 words per bin (low word, then high word).
 */

static void put128(__int128 v, int64_t *out)
{
    out[0] = (int64_t)(uint64_t)v;               /* low 64 bits */
    out[1] = (int64_t)(v >> 64);                  /* high 64 bits, signed */
}

/* sum over unordered pairs {i, j} in bin b of w_i w_j */
void oracle_2pcf_weighted(const int32_t *xyz, int64_t n, int64_t box, int periodic, const int64_t *edges, int nb,
                          const int16_t *w, int64_t *out)
{
    cat_t c = { xyz, n, box, periodic, edges, nb };
    __int128 *acc = (__int128 *)calloc((size_t)nb, sizeof(__int128));
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = i + 1; j < n; ++j) {
            int b = pair_bin(&c, i, j);
            if (b >= 0) acc[b] += (__int128)w[i] * w[j];
        }
    for (int b = 0; b < nb; ++b) put128(acc[b], out + 2 * b);
    free(acc);
}

typedef struct {
    cat_t c;
    const int64_t *row_ptr;
    const int32_t *nbr;
    const uint8_t *bin;
    const int16_t *w;
    const int32_t *t3;
    int64_t ncfg;
    __int128 *acc;          /* [threads][ncfg] */
} wtri_ctx_t;

static void wtri_hub(void *vctx, int tid, int64_t i)
{
    wtri_ctx_t *t = (wtri_ctx_t *)vctx;
    __int128 *h = t->acc + (size_t)tid * (size_t)t->ncfg;
    int nb = t->c.nb;
    for (int64_t a = t->row_ptr[i]; a < t->row_ptr[i + 1]; ++a) {
        int64_t j = t->nbr[a];
        if (j <= i) continue;
        for (int64_t b = a + 1; b < t->row_ptr[i + 1]; ++b) {
            int64_t k = t->nbr[b];
            int bjk = pair_bin(&t->c, j, k);
            if (bjk < 0) continue;
            int v[3] = { t->bin[a], t->bin[b], bjk };
            sort3(v);
            h[t->t3[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += (__int128)t->w[i] * t->w[j] * t->w[k];
        }
    }
}

/* sum over triangles {i, j, k} in each sorted-bin configuration of w_i w_j w_k */
void oracle_3pcf_weighted(const int32_t *xyz, int64_t n, int64_t box, int periodic, const int64_t *edges, int nb,
                          const int64_t *row_ptr, const int32_t *nbr, const uint8_t *bin, const int16_t *w,
                          int64_t *out)
{
    int nt = oracle_threads();
    wtri_ctx_t t;
    t.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    t.row_ptr = row_ptr; t.nbr = nbr; t.bin = bin; t.w = w;
    t.t3 = table3(nb);
    t.ncfg = oracle_nconfig3(nb);
    t.acc = (__int128 *)calloc((size_t)nt * (size_t)t.ncfg, sizeof(__int128));
    parallel_for(0, n, nt, wtri_hub, &t);
    for (int64_t x = 0; x < t.ncfg; ++x) {
        __int128 s = 0;
        for (int q = 0; q < nt; ++q) s += t.acc[(size_t)q * t.ncfg + x];
        put128(s, out + 2 * x);
    }
    free(t.acc);
    free((void *)t.t3);
}

/* Weighted six-bin 4pCF: per configuration, the sum over tetrahedra
 * {i, j, k, l} of W = w_i w_j w_k w_l (even) and of sign x W (odd), with the
 * sign of the unweighted odd channel; exact 128-bit sums, (low, high) words. */
typedef struct {
    cat_t c;
    const int64_t *row_ptr;
    const int32_t *nbr;
    const int32_t *tab;
    const int16_t *w;
    int64_t ncfg;
    __int128 *even;         /* [threads][ncfg] */
    __int128 *odd;
} wsix_ctx_t;

static void wsix_hub(void *vctx, int tid, int64_t i)
{
    wsix_ctx_t *x = (wsix_ctx_t *)vctx;
    __int128 *ev = x->even + (size_t)tid * (size_t)x->ncfg;
    __int128 *od = x->odd + (size_t)tid * (size_t)x->ncfg;
    int64_t r0 = x->row_ptr[i], r1 = x->row_ptr[i + 1];
    for (int64_t a = r0; a < r1; ++a) {
        if (x->nbr[a] <= i) continue;
        for (int64_t b = a + 1; b < r1; ++b) {
            if (pair_bin(&x->c, x->nbr[a], x->nbr[b]) < 0) continue;
            for (int64_t d = b + 1; d < r1; ++d) {
                if (pair_bin(&x->c, x->nbr[a], x->nbr[d]) < 0) continue;
                if (pair_bin(&x->c, x->nbr[b], x->nbr[d]) < 0) continue;
                int64_t q[4] = { i, x->nbr[a], x->nbr[b], x->nbr[d] };
                int sg;
                int idx = tetra_class(&x->c, x->tab, q, &sg);
                __int128 W = (__int128)x->w[q[0]] * x->w[q[1]] * x->w[q[2]] * x->w[q[3]];
                ev[idx] += W;
                od[idx] += sg * W;
            }
        }
    }
}

void oracle_4pcf6_weighted(const int32_t *xyz, int64_t n, int64_t box, int periodic, const int64_t *edges, int nb,
                           const int64_t *row_ptr, const int32_t *nbr, const int16_t *w,
                           int64_t hub_begin, int64_t hub_end, int64_t *even, int64_t *odd)
{
    int nt = oracle_threads();
    wsix_ctx_t x;
    x.c = (cat_t){ xyz, n, box, periodic, edges, nb };
    x.row_ptr = row_ptr; x.nbr = nbr; x.w = w;
    x.tab = six_index_table(nb);
    x.ncfg = oracle_nconfig6(nb);
    x.even = (__int128 *)calloc((size_t)nt * (size_t)x.ncfg, sizeof(__int128));
    x.odd = (__int128 *)calloc((size_t)nt * (size_t)x.ncfg, sizeof(__int128));
    if (hub_end > hub_begin) parallel_for(hub_begin, hub_end, nt, wsix_hub, &x);
    for (int64_t k = 0; k < x.ncfg; ++k) {
        __int128 se = 0, so = 0;
        for (int q = 0; q < nt; ++q) {
            se += x.even[(size_t)q * x.ncfg + k];
            so += x.odd[(size_t)q * x.ncfg + k];
        }
        put128(se, even + 2 * k);
        put128(so, odd + 2 * k);
    }
    free(x.even); free(x.odd);
    free((void *)x.tab);
}
