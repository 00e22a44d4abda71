/*
 * CPU ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct all-pairs / single-source shortest paths on
 * a dense distance matrix.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this; the library never does.  It shares no code,
 * header or constant generator with the CUDA path.
 *
 * Problem (blocked Floyd-Warshall thesis page, 1library.co excerpt,
 * section 4.6; Johnson/Dijkstra page, CEUR Vol-1631 pp.105-112, the
 * notation paragraph): a weighted directed graph given as an n x n matrix,
 * W[i][j] the weight of arc i->j, "no arc" encoded as INF, 0 on the diagonal,
 * weights >= 0.  Output D[i][j] = minimum over all directed paths i ~> j of
 * the sum of arc weights, INF if there is none.
 *
 * int32 encoding: INF = 0x3FFFFFFF.  Entries >= INF are read as INF.  All
 * sums are formed in int64 and a sum is only kept when it is below the value
 * it replaces, so a path whose length reaches INF is reported as INF (the
 * encoding cannot hold it).  Floating point: computed in double, +inf for
 * "no arc".
 *
 * Functions:
 *   oracle_fw_i32 / oracle_fw_f64  -- the Floyd-Warshall recurrence as the
 *       thesis page restates it (section 4.6, phase descriptions): for each
 *       intermediate vertex k in order, D[i][j] = min(D[i][j], D[i][k]+D[k][j]).
 *       No tiling.  With threads > 1 the i-loop of one k runs in parallel; that
 *       is exact because row k and column k do not change during step k
 *       (D[k][k] = 0).
 *   oracle_dijkstra_* -- Dijkstra from given sources with a binary heap
 *       (Johnson/Dijkstra page, the sequential Dijkstra operators init,
 *       ExtractMin and RelaxEdge).  reverse != 0 runs it on the reversed graph,
 *       which gives columns D[:, s] instead of rows.
 *   oracle_bfs_hops -- breadth-first hop counts (reachability).
 *   oracle_bellman_ford_i32 -- single-source Bellman-Ford (Johnson/Dijkstra
 *       page, the RelaxEdges/BellmanFord operators and the negative-cycle
 *       condition cnc): |V| - 1 rounds relaxing every arc, stopping early when a
 *       round changes nothing, then one more round to detect a negative cycle.
 *   oracle_johnson_i32 -- Johnson's APSP as the same page lays it out: extend
 *       the graph with a vertex s and 0-weight arcs s->v, Bellman-Ford from s
 *       gives h, reweight w'(u,v) = w(u,v) + h(u) - h(v) >= 0, Dijkstra from
 *       every vertex on w', and map back D(i,j) = D'(i,j) + h(j) - h(i).
 *       Handles negative arc weights; reports a negative cycle.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define O_INF 0x3FFFFFFFLL

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ---------------- Floyd-Warshall ---------------- */

int oracle_fw_i32(int32_t* d, int64_t n, int64_t ld, int threads) {
    if (n < 0 || ld < n || (n > 0 && !d)) return -1;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            if (d[i * ld + j] > O_INF) d[i * ld + j] = (int32_t)O_INF;
    (void)threads;
    for (int64_t k = 0; k < n; ++k) {
        const int32_t* rowk = d + k * ld;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)
        for (int64_t i = 0; i < n; ++i) {
            int32_t* rowi = d + i * ld;
            int64_t dik = rowi[k];
            if (dik >= O_INF) continue; /* no path i ~> k yet */
            for (int64_t j = 0; j < n; ++j) {
                int64_t dkj = rowk[j];
                if (dkj >= O_INF) continue; /* no path k ~> j yet */
                int64_t s = dik + dkj;
                if (s < (int64_t)rowi[j]) rowi[j] = (int32_t)s;
            }
        }
    }
    return 0;
}

/* Steps k in [k_begin, k_end) only (used to time a bounded sample). */
int oracle_fw_i32_steps(int32_t* d, int64_t n, int64_t ld, int64_t k_begin, int64_t k_end, int threads) {
    if (n < 0 || ld < n || k_begin < 0 || k_end > n || (n > 0 && !d)) return -1;
    (void)threads;
    for (int64_t k = k_begin; k < k_end; ++k) {
        const int32_t* rowk = d + k * ld;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)
        for (int64_t i = 0; i < n; ++i) {
            int32_t* rowi = d + i * ld;
            int64_t dik = rowi[k];
            if (dik >= O_INF) continue;
            for (int64_t j = 0; j < n; ++j) {
                int64_t dkj = rowk[j];
                if (dkj >= O_INF) continue;
                int64_t s = dik + dkj;
                if (s < (int64_t)rowi[j]) rowi[j] = (int32_t)s;
            }
        }
    }
    return 0;
}

int oracle_fw_f64(double* d, int64_t n, int64_t ld, int threads) {
    if (n < 0 || ld < n || (n > 0 && !d)) return -1;
    (void)threads;
    for (int64_t k = 0; k < n; ++k) {
        const double* rowk = d + k * ld;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)
        for (int64_t i = 0; i < n; ++i) {
            double* rowi = d + i * ld;
            double dik = rowi[k];
            if (isinf(dik)) continue;
            for (int64_t j = 0; j < n; ++j) {
                double s = dik + rowk[j];
                if (s < rowi[j]) rowi[j] = s;
            }
        }
    }
    return 0;
}

/* Steps k in [k_begin, k_end) of oracle_fw_f64 only (to time a bounded
 * sample of an fp32 workload). */
int oracle_fw_f64_steps(double* d, int64_t n, int64_t ld, int64_t k_begin, int64_t k_end, int threads) {
    if (n < 0 || ld < n || k_begin < 0 || k_end > n || (n > 0 && !d)) return -1;
    (void)threads;
    for (int64_t k = k_begin; k < k_end; ++k) {
        const double* rowk = d + k * ld;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)
        for (int64_t i = 0; i < n; ++i) {
            double* rowi = d + i * ld;
            double dik = rowi[k];
            if (isinf(dik)) continue;
            for (int64_t j = 0; j < n; ++j) {
                double s = dik + rowk[j];
                if (s < rowi[j]) rowi[j] = s;
            }
        }
    }
    return 0;
}

/* ---------------- graph in adjacency form ---------------- */

typedef struct {
    int64_t n;
    int64_t* off;  /* n + 1 */
    int32_t* dst;  /* arcs */
    double* wf;    /* weights as double */
    int64_t* wi;   /* weights as int64 */
} o_graph;

static void o_graph_free(o_graph* g) {
    free(g->off); free(g->dst); free(g->wf); free(g->wi);
    memset(g, 0, sizeof(*g));
}

/* kind: 0 = int32 matrix, 1 = float32 matrix.  reverse: arcs j->i for W[i][j]. */
static int o_graph_build(o_graph* g, const void* w, int kind, int64_t n, int64_t ld, int reverse) {
    memset(g, 0, sizeof(*g));
    g->n = n;
    g->off = (int64_t*)calloc((size_t)n + 1, sizeof(int64_t));
    if (!g->off) return -1;
    const int32_t* wi32 = (const int32_t*)w;
    const float* wf32 = (const float*)w;
#define O_HAS_ARC(i, j) ((i) != (j) && (kind == 0 ? (int64_t)wi32[(i) * ld + (j)] < O_INF \
                                                  : !isinf(wf32[(i) * ld + (j)])))
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            if (O_HAS_ARC(i, j)) g->off[(reverse ? j : i) + 1]++;
    for (int64_t v = 0; v < n; ++v) g->off[v + 1] += g->off[v];
    int64_t m = g->off[n];
    g->dst = (int32_t*)malloc(sizeof(int32_t) * (size_t)(m ? m : 1));
    g->wf = (double*)malloc(sizeof(double) * (size_t)(m ? m : 1));
    g->wi = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m ? m : 1));
    int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n ? n : 1));
    if (!g->dst || !g->wf || !g->wi || !fill) { free(fill); o_graph_free(g); return -1; }
    memcpy(fill, g->off, sizeof(int64_t) * (size_t)n);
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            if (O_HAS_ARC(i, j)) {
                int64_t from = reverse ? j : i, to = reverse ? i : j;
                int64_t e = fill[from]++;
                g->dst[e] = (int32_t)to;
                if (kind == 0) { g->wi[e] = wi32[i * ld + j]; g->wf[e] = (double)wi32[i * ld + j]; }
                else { g->wf[e] = (double)wf32[i * ld + j]; g->wi[e] = 0; }
            }
#undef O_HAS_ARC
    free(fill);
    return 0;
}

/* ---------------- binary heap of (key, vertex) ---------------- */

typedef struct { double key; int64_t ikey; int32_t v; } o_item;
typedef struct { o_item* a; int64_t size, cap; int integer; } o_heap;

static int o_less(const o_heap* h, const o_item* x, const o_item* y) {
    return h->integer ? (x->ikey < y->ikey) : (x->key < y->key);
}

static int o_push(o_heap* h, o_item it) {
    if (h->size == h->cap) {
        int64_t nc = h->cap ? 2 * h->cap : 1024;
        o_item* na = (o_item*)realloc(h->a, sizeof(o_item) * (size_t)nc);
        if (!na) return -1;
        h->a = na; h->cap = nc;
    }
    int64_t c = h->size++;
    h->a[c] = it;
    while (c > 0) {                      /* sift up */
        int64_t p = (c - 1) / 2;
        if (!o_less(h, &h->a[c], &h->a[p])) break;
        o_item t = h->a[c]; h->a[c] = h->a[p]; h->a[p] = t;
        c = p;
    }
    return 0;
}

static o_item o_pop(o_heap* h) {
    o_item top = h->a[0];
    h->a[0] = h->a[--h->size];
    int64_t c = 0;
    for (;;) {                           /* sift down */
        int64_t l = 2 * c + 1, r = l + 1, m = c;
        if (l < h->size && o_less(h, &h->a[l], &h->a[m])) m = l;
        if (r < h->size && o_less(h, &h->a[r], &h->a[m])) m = r;
        if (m == c) break;
        o_item t = h->a[c]; h->a[c] = h->a[m]; h->a[m] = t;
        c = m;
    }
    return top;
}

/* One Dijkstra run: init (all INF, source 0), then repeatedly take the
 * unsettled vertex of least tentative distance (ExtractMin) and relax its
 * out-arcs (RelaxEdge).  Stale heap entries are skipped. */
static int o_dijkstra_one(const o_graph* g, int64_t src, int integer, int64_t* di, double* df,
                          unsigned char* settled) {
    int64_t n = g->n;
    o_heap h = {0, 0, 0, integer};
    for (int64_t v = 0; v < n; ++v) { di[v] = INT64_MAX; df[v] = INFINITY; settled[v] = 0; }
    di[src] = 0; df[src] = 0.0;
    o_item s0 = {0.0, 0, (int32_t)src};
    if (o_push(&h, s0)) return -1;
    while (h.size > 0) {
        o_item it = o_pop(&h);
        int64_t u = it.v;
        if (settled[u]) continue;
        settled[u] = 1;
        for (int64_t e = g->off[u]; e < g->off[u + 1]; ++e) {
            int64_t v = g->dst[e];
            if (integer) {
                int64_t nd = di[u] + g->wi[e];
                if (nd < di[v]) {
                    di[v] = nd;
                    o_item x = {0.0, nd, (int32_t)v};
                    if (o_push(&h, x)) { free(h.a); return -1; }
                }
            } else {
                double nd = df[u] + g->wf[e];
                if (nd < df[v]) {
                    df[v] = nd;
                    o_item x = {nd, 0, (int32_t)v};
                    if (o_push(&h, x)) { free(h.a); return -1; }
                }
            }
        }
    }
    free(h.a);
    return 0;
}

static int o_dijkstra_rows(const void* w, int kind, int64_t n, int64_t ld, const int32_t* sources,
                           int64_t ns, int reverse, int32_t* out_i, double* out_f, int threads) {
    if (n < 0 || ld < n || ns < 0 || (n > 0 && !w)) return -1;
    for (int64_t s = 0; s < ns; ++s)
        if (sources[s] < 0 || sources[s] >= n) return -1;
    o_graph g;
    if (o_graph_build(&g, w, kind, n, ld, reverse)) return -2;
    int err = 0;
    (void)threads;
#pragma omp parallel num_threads(threads > 0 ? threads : 1) if (threads > 1)
    {
        int64_t* di = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n ? n : 1));
        double* df = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1));
        unsigned char* st = (unsigned char*)malloc((size_t)(n ? n : 1));
        if (!di || !df || !st) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t s = 0; s < ns; ++s) {
                if (o_dijkstra_one(&g, sources[s], kind == 0, di, df, st)) {
#pragma omp atomic write
                    err = -2;
                    continue;
                }
                for (int64_t v = 0; v < n; ++v) {
                    if (kind == 0) out_i[s * n + v] = (int32_t)(di[v] < O_INF ? di[v] : O_INF);
                    else out_f[s * n + v] = df[v];
                }
            }
        }
        free(di); free(df); free(st);
    }
    o_graph_free(&g);
    return err;
}

/* Rows (or, with reverse, columns) of D for an int32 matrix; out is ns x n,
 * INF for unreachable (and for path lengths that reach INF). */
int oracle_dijkstra_i32(const int32_t* w, int64_t n, int64_t ld, const int32_t* sources, int64_t ns,
                        int reverse, int32_t* out, int threads) {
    return o_dijkstra_rows(w, 0, n, ld, sources, ns, reverse, out, NULL, threads);
}

/* Same for an fp32 matrix, accumulated in double; +inf for unreachable. */
int oracle_dijkstra_f32(const float* w, int64_t n, int64_t ld, const int32_t* sources, int64_t ns,
                        int reverse, double* out, int threads) {
    return o_dijkstra_rows(w, 1, n, ld, sources, ns, reverse, NULL, out, threads);
}

/* Breadth-first hop counts from src over arcs W[i][j] < INF (int32 matrix);
 * -1 where unreachable. */
int oracle_bfs_hops_i32(const int32_t* w, int64_t n, int64_t ld, int64_t src, int32_t* hops) {
    if (n <= 0 || ld < n || src < 0 || src >= n || !w || !hops) return -1;
    int32_t* q = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
    if (!q) return -2;
    for (int64_t v = 0; v < n; ++v) hops[v] = -1;
    int64_t qh = 0, qt = 0;
    hops[src] = 0; q[qt++] = (int32_t)src;
    while (qh < qt) {
        int64_t u = q[qh++];
        for (int64_t v = 0; v < n; ++v)
            if (v != u && (int64_t)w[u * ld + v] < O_INF && hops[v] < 0) {
                hops[v] = hops[u] + 1;
                q[qt++] = (int32_t)v;
            }
    }
    free(q);
    return 0;
}

/* ---------------- Bellman-Ford and Johnson ---------------- */

/* Distances from src over arcs W[u][v] < INF (u != v), int64 arithmetic.
 * out[v] = distance, or INF when v is unreachable.  Returns 0, or 1 when a
 * negative cycle is reachable from src (out is then undefined), or < 0 on
 * bad arguments. */
int oracle_bellman_ford_i32(const int32_t* w, int64_t n, int64_t ld, int64_t src, int64_t* out) {
    if (n <= 0 || ld < n || src < 0 || src >= n || !w || !out) return -1;
    const int64_t UNSET = INT64_MAX;
    for (int64_t v = 0; v < n; ++v) out[v] = UNSET;
    out[src] = 0;
    for (int64_t round = 0; round < n - 1; ++round) {        /* |V| - 1 rounds */
        int changed = 0;
        for (int64_t u = 0; u < n; ++u) {
            if (out[u] == UNSET) continue;
            for (int64_t v = 0; v < n; ++v) {
                if (v == u || (int64_t)w[u * ld + v] >= O_INF) continue;
                const int64_t nd = out[u] + w[u * ld + v];
                if (nd < out[v]) { out[v] = nd; changed = 1; }
            }
        }
        if (!changed) break;
    }
    for (int64_t u = 0; u < n; ++u) {                        /* cnc: any arc still relaxable? */
        if (out[u] == UNSET) continue;
        for (int64_t v = 0; v < n; ++v)
            if (v != u && (int64_t)w[u * ld + v] < O_INF && out[u] + w[u * ld + v] < out[v]) return 1;
    }
    for (int64_t v = 0; v < n; ++v) if (out[v] == UNSET) out[v] = O_INF;
    return 0;
}

/* Johnson's method for the rows of the sources (all rows when sources is
 * NULL).  Row s of out (ns x n, int32, INF for unreachable) holds the
 * distances from sources[s].  Returns 0, 1 on a negative cycle, < 0 on bad
 * arguments or allocation failure. */
static int o_johnson(const int32_t* w, int64_t n, int64_t ld, const int32_t* sources, int64_t ns, int32_t* out,
                     int threads) {
    if (n <= 0 || ld < n || !w || !out) return -1;
    if (!sources) ns = n;
    for (int64_t s = 0; sources && s < ns; ++s)
        if (sources[s] < 0 || sources[s] >= n) return -1;
    /* extendGraph + BellmanFord(s): s reaches every v directly with weight 0. */
    int64_t* h = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
    if (!h) return -2;
    for (int64_t v = 0; v < n; ++v) h[v] = 0;                /* after the arcs s->v */
    h[n] = 0;                                                /* s itself */
    for (int64_t round = 0; round < n; ++round) {            /* |V'| - 1 = n rounds */
        int changed = 0;
        for (int64_t u = 0; u < n; ++u)
            for (int64_t v = 0; v < n; ++v) {
                if (v == u || (int64_t)w[u * ld + v] >= O_INF) continue;
                const int64_t nd = h[u] + w[u * ld + v];
                if (nd < h[v]) { h[v] = nd; changed = 1; }
            }
        if (!changed) break;
    }
    for (int64_t u = 0; u < n; ++u)                          /* cnc */
        for (int64_t v = 0; v < n; ++v)
            if (v != u && (int64_t)w[u * ld + v] < O_INF && h[u] + w[u * ld + v] < h[v]) {
                free(h);
                return 1;
            }
    /* UpdateWeights: w'(u,v) = w(u,v) + h(u) - h(v), kept in the adjacency form */
    o_graph g;
    if (o_graph_build(&g, w, 0, n, ld, 0)) { free(h); return -2; }
    for (int64_t u = 0; u < n; ++u)
        for (int64_t e = g.off[u]; e < g.off[u + 1]; ++e) g.wi[e] += h[u] - h[g.dst[e]];
    int err = 0;
    (void)threads;
#pragma omp parallel num_threads(threads > 0 ? threads : 1) if (threads > 1)
    {
        int64_t* di = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
        double* df = (double*)malloc(sizeof(double) * (size_t)n);
        unsigned char* st = (unsigned char*)malloc((size_t)n);
        if (!di || !df || !st) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t q = 0; q < ns; ++q) {
                const int64_t i = sources ? sources[q] : q;
                if (o_dijkstra_one(&g, i, 1, di, df, st)) {  /* D(i) on w' */
#pragma omp atomic write
                    err = -2;
                    continue;
                }
                for (int64_t j = 0; j < n; ++j) {            /* to(): D(i,j) = D'(i,j) + h(j) - h(i) */
                    if (di[j] == INT64_MAX) { out[q * n + j] = (int32_t)O_INF; continue; }
                    const int64_t d = di[j] + h[j] - h[i];
                    out[q * n + j] = (int32_t)(d < O_INF ? d : O_INF);
                }
            }
        }
        free(di); free(df); free(st);
    }
    o_graph_free(&g);
    free(h);
    return err;
}

/* All-pairs distances by Johnson's method.  out is n x n (int32, INF for
 * unreachable).  Returns 0, 1 on a negative cycle, < 0 on bad arguments or
 * allocation failure. */
int oracle_johnson_i32(const int32_t* w, int64_t n, int64_t ld, int32_t* out, int threads) {
    return o_johnson(w, n, ld, NULL, n, out, threads);
}

/* The same for the rows of the ns given sources only (out is ns x n). */
int oracle_johnson_rows_i32(const int32_t* w, int64_t n, int64_t ld, const int32_t* sources, int64_t ns,
                            int32_t* out, int threads) {
    if (!sources || ns < 0) return -1;
    return o_johnson(w, n, ld, sources, ns, out, threads);
}

/* ---------------- Dijkstra on a CSR graph ----------------
 *
 * The same binary-heap Dijkstra (Johnson/Dijkstra page, the sequential
 * Dijkstra operators) read straight from a CSR arc list: the arcs leaving u
 * are row_ptr[u] .. row_ptr[u+1]-1, heads col[], weights w[] (all >= 0).
 * Self-loops and parallel arcs are allowed.  out (ns x n, int32) gets the
 * distance from sources[s], INF for unreachable, and distances at or above
 * INF read as INF.  Returns 0, -1 on bad arguments (including a negative
 * weight or a head out of range), -2 on allocation failure. */
static int o_dijkstra_csr_one(const int64_t* row_ptr, const int32_t* col, const int32_t* w, int64_t n,
                              int64_t src, int64_t* di, unsigned char* settled) {
    o_heap h = {0, 0, 0, 1};
    for (int64_t v = 0; v < n; ++v) { di[v] = INT64_MAX; settled[v] = 0; }
    di[src] = 0;
    o_item s0 = {0.0, 0, (int32_t)src};
    if (o_push(&h, s0)) return -2;
    while (h.size > 0) {
        o_item it = o_pop(&h);
        const int64_t u = it.v;
        if (settled[u]) continue;
        settled[u] = 1;
        for (int64_t e = row_ptr[u]; e < row_ptr[u + 1]; ++e) {
            const int64_t v = col[e];
            const int64_t nd = di[u] + w[e];
            if (nd < di[v]) {
                di[v] = nd;
                o_item x = {0.0, nd, (int32_t)v};
                if (o_push(&h, x)) { free(h.a); return -2; }
            }
        }
    }
    free(h.a);
    return 0;
}

int oracle_dijkstra_csr_i32(const int64_t* row_ptr, const int32_t* col, const int32_t* w, int64_t n,
                            const int32_t* sources, int64_t ns, int32_t* out, int threads) {
    if (n <= 0 || ns < 0 || !row_ptr || !sources || !out || row_ptr[0] != 0) return -1;
    for (int64_t v = 0; v < n; ++v)
        if (row_ptr[v + 1] < row_ptr[v]) return -1;
    const int64_t m = row_ptr[n];
    if (m > 0 && (!col || !w)) return -1;
    for (int64_t e = 0; e < m; ++e)
        if (w[e] < 0 || col[e] < 0 || col[e] >= n) return -1;
    for (int64_t s = 0; s < ns; ++s)
        if (sources[s] < 0 || sources[s] >= n) return -1;
    int err = 0;
    (void)threads;
#pragma omp parallel num_threads(threads > 0 ? threads : 1) if (threads > 1)
    {
        int64_t* di = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
        unsigned char* st = (unsigned char*)malloc((size_t)n);
        if (!di || !st) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t s = 0; s < ns; ++s) {
                if (o_dijkstra_csr_one(row_ptr, col, w, n, sources[s], di, st)) {
#pragma omp atomic write
                    err = -2;
                    continue;
                }
                int32_t* row = out + s * n;
                for (int64_t v = 0; v < n; ++v) row[v] = (int32_t)(di[v] < O_INF ? di[v] : O_INF);
            }
        }
        free(di); free(st);
    }
    return err;
}
