/*
 * Seeded synthetic graph generators, shared by the tests, the bench and the
 * oracle's pins.  This file holds no shortest-path arithmetic: it only draws
 * dense distance matrices (INF for no edge, 0 on the diagonal).
 *
 * Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), written from its published
 * definition.  SplitMix64 seeded with s produces, as its t-th output (t >= 1),
 * mix(s + t * GAMMA).  Because of that closed form every draw below is
 * addressed by its position t in the stream, so rows can be generated in any
 * order (or in parallel) and the result is the same on every machine.
 *
 * Workloads (shapes follow the pages' workloads):
 *   - directed Erdos-Renyi G(n, p): for every ordered pair (i, j), i != j,
 *     stream position 2*(i*n + j) + 1 decides presence (u < p, u uniform on
 *     [0,1) with 53 bits) and position 2*(i*n + j) + 2 draws the weight.
 *   - Barabasi-Albert preferential attachment with beta edges per new vertex,
 *     each undirected edge stored as two arcs (m ~ 2*beta*n), after the
 *     betweenness-centrality page (arXiv 1409.7764, section IV, the synthetic
 *     graph paragraph).  Seed graph and draw order are our own reading; the
 *     page only names the model and its parameter.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t gen_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* t-th output (t >= 1) of SplitMix64 seeded with `seed`. */
uint64_t graphgen_splitmix64_at(uint64_t seed, uint64_t t) {
    return gen_mix(seed + t * GEN_GAMMA);
}

/* Uniform double on [0, 1) with 53 random bits. */
static inline double gen_unit(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* Integer in [lo, hi] from the top 32 bits (multiply-shift, no rejection). */
static inline int32_t gen_int(uint64_t x, int32_t lo, int32_t hi) {
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
    return (int32_t)((int64_t)lo + (int64_t)(((x >> 32) * span) >> 32));
}

/* Weight in (0, 1] on a 2^-24 grid: 1 - k * 2^-24 with k uniform in [0, 2^24). */
static inline float gen_unit_weight_f32(uint64_t x) {
    uint64_t k = x >> 40;
    return (float)(1.0 - (double)k * (1.0 / 16777216.0));
}

/* Directed ER graph, int32 weights uniform in [wlo, whi]; absent edges get
 * `inf`; diagonal 0.  Rows [row_begin, row_end) of an n x n matrix written at
 * out + (i - row_begin) * ld.  Columns n..ld-1 are not touched. */
void graphgen_er_i32(int32_t* out, int64_t n, int64_t ld, int64_t row_begin, int64_t row_end,
                     double p, int32_t wlo, int32_t whi, int32_t inf, uint64_t seed) {
    for (int64_t i = row_begin; i < row_end; ++i) {
        int32_t* row = out + (i - row_begin) * ld;
        for (int64_t j = 0; j < n; ++j) {
            if (i == j) { row[j] = 0; continue; }
            uint64_t t = 2u * (uint64_t)(i * n + j) + 1u;
            if (gen_unit(graphgen_splitmix64_at(seed, t)) < p)
                row[j] = gen_int(graphgen_splitmix64_at(seed, t + 1u), wlo, whi);
            else
                row[j] = inf;
        }
    }
}

/* Directed ER graph, fp32 weights in (0, 1]; absent edges get +inf. */
void graphgen_er_f32(float* out, int64_t n, int64_t ld, int64_t row_begin, int64_t row_end,
                     double p, uint64_t seed) {
    const float inf = __builtin_inff();
    for (int64_t i = row_begin; i < row_end; ++i) {
        float* row = out + (i - row_begin) * ld;
        for (int64_t j = 0; j < n; ++j) {
            if (i == j) { row[j] = 0.0f; continue; }
            uint64_t t = 2u * (uint64_t)(i * n + j) + 1u;
            if (gen_unit(graphgen_splitmix64_at(seed, t)) < p)
                row[j] = gen_unit_weight_f32(graphgen_splitmix64_at(seed, t + 1u));
            else
                row[j] = inf;
        }
    }
}

/* Barabasi-Albert edge list.  Vertices 0..beta-1 start with no edges.  Vertex
 * v = beta links to all of them; every later vertex v links to beta distinct
 * existing vertices drawn with probability proportional to their degree
 * (uniform picks from the list of all edge endpoints so far, duplicates
 * redrawn).  Target draws use stream positions 1, 2, 3, ... in order.
 * Writes (u, v) pairs with u = new vertex into edges[2*e], edges[2*e+1].
 * Returns the number of undirected edges (beta * (n - beta)), or -1 on bad
 * arguments / allocation failure.  `edges` must hold 2*beta*(n-beta) ints. */
int64_t graphgen_ba_edges(int32_t* edges, int64_t n, int32_t beta, uint64_t seed) {
    if (beta < 1 || n <= beta) return -1;
    int64_t m = (int64_t)beta * (n - beta);
    int32_t* ends = (int32_t*)malloc(sizeof(int32_t) * (size_t)(2 * m));
    int32_t* pick = (int32_t*)malloc(sizeof(int32_t) * (size_t)beta);
    if (!ends || !pick) { free(ends); free(pick); return -1; }
    int64_t nends = 0, e = 0;
    uint64_t t = 1;
    for (int64_t v = beta; v < n; ++v) {
        int npick = 0;
        if (v == beta) {
            for (int32_t q = 0; q < beta; ++q) pick[npick++] = q;
        } else {
            while (npick < beta) {
                uint64_t x = graphgen_splitmix64_at(seed, t++);
                int32_t cand = ends[(int64_t)(((x >> 32) * (uint64_t)nends) >> 32)];
                int dup = 0;
                for (int q = 0; q < npick; ++q) dup |= (pick[q] == cand);
                if (!dup) pick[npick++] = cand;
            }
        }
        for (int q = 0; q < npick; ++q) {
            edges[2 * e] = (int32_t)v;
            edges[2 * e + 1] = pick[q];
            ++e;
            ends[nends++] = (int32_t)v;
            ends[nends++] = pick[q];
        }
    }
    free(ends);
    free(pick);
    return e;
}

/* Dense int32 matrix of a BA graph: every undirected edge {u, v} becomes arcs
 * u->v and v->u, each with its own weight uniform in [wlo, whi] drawn at
 * stream position 2^40 + (u*n + v) (independent per direction; far past the
 * positions the target draws use).  Absent arcs are `inf`, diagonal 0.
 * Returns the number of arcs, or -1 on failure. */
int64_t graphgen_ba_i32(int32_t* out, int64_t n, int64_t ld, int32_t beta, int32_t wlo,
                        int32_t whi, int32_t inf, uint64_t seed) {
    if (beta < 1 || n <= beta) return -1;
    int64_t m = (int64_t)beta * (n - beta);
    int32_t* edges = (int32_t*)malloc(sizeof(int32_t) * (size_t)(2 * m));
    if (!edges) return -1;
    if (graphgen_ba_edges(edges, n, beta, seed) != m) { free(edges); return -1; }
    for (int64_t i = 0; i < n; ++i) {
        int32_t* row = out + i * ld;
        for (int64_t j = 0; j < n; ++j) row[j] = (i == j) ? 0 : inf;
    }
    const uint64_t base = 1ULL << 40;
    for (int64_t e = 0; e < m; ++e) {
        int64_t u = edges[2 * e], v = edges[2 * e + 1];
        out[u * ld + v] = gen_int(graphgen_splitmix64_at(seed, base + (uint64_t)(u * n + v)), wlo, whi);
        out[v * ld + u] = gen_int(graphgen_splitmix64_at(seed, base + (uint64_t)(v * n + u)), wlo, whi);
    }
    free(edges);
    return 2 * m;
}

/* Directed ER graph with some negative arc weights but no negative cycle:
 * w(i, j) = w0(i, j) + p(i) - p(j), where w0 is uniform in [wlo, whi]
 * (wlo >= 0) and p is a vertex potential uniform in [0, pmax] drawn at stream
 * position 2^41 + i.  Every cycle's weight is the sum of its w0 >= 0.
 * Presence and w0 use the same stream positions as graphgen_er_i32. */
void graphgen_er_potential_i32(int32_t* out, int64_t n, int64_t ld, int64_t row_begin,
                               int64_t row_end, double p, int32_t wlo, int32_t whi, int32_t pmax,
                               int32_t inf, uint64_t seed) {
    const uint64_t pbase = 1ULL << 41;
    for (int64_t i = row_begin; i < row_end; ++i) {
        int32_t* row = out + (i - row_begin) * ld;
        const int32_t pi = gen_int(graphgen_splitmix64_at(seed, pbase + (uint64_t)i), 0, pmax);
        for (int64_t j = 0; j < n; ++j) {
            if (i == j) { row[j] = 0; continue; }
            uint64_t t = 2u * (uint64_t)(i * n + j) + 1u;
            if (gen_unit(graphgen_splitmix64_at(seed, t)) < p) {
                const int32_t pj = gen_int(graphgen_splitmix64_at(seed, pbase + (uint64_t)j), 0, pmax);
                row[j] = gen_int(graphgen_splitmix64_at(seed, t + 1u), wlo, whi) + pi - pj;
            } else {
                row[j] = inf;
            }
        }
    }
}

/* ---------------- R-MAT (sparse, CSR) ----------------
 *
 * The Delta-stepping page measures on R-MAT graphs of scale 17..23 (2^scale
 * vertices) with 32 arcs per vertex on average.  It names the model but not
 * its parameters; this recipe takes the usual Graph500 quadrant
 * probabilities (a, b, c, d) = (0.57, 0.19, 0.19, 0.05).
 *
 * Arc e (0 <= e < m) descends `scale` levels of the adjacency matrix: at
 * level l the draw at stream position e * 64 + l + 1 picks a quadrant, which
 * fixes one bit of the tail and one of the head.  Its weight is drawn at
 * position 2^44 + e.  Vertex ids then go through the bijection
 * v -> (v * 0x9E3779B1 + 0x7F4A7C15) mod 2^scale (odd multiplier), so that
 * the high-degree vertices do not all sit at the lowest ids.  Self-loops and
 * parallel arcs are kept: the arc list is what the model draws.
 *
 * graphgen_rmat_arcs fills tail/head/weight for arcs [e_begin, e_end).
 * graphgen_csr_from_arcs is a stable counting sort of those arcs by tail:
 * row_ptr (n + 1), then col/w in arc order within each row. */
static inline uint32_t rmat_scramble(uint32_t v, int scale) {
    const uint32_t mask = scale >= 32 ? 0xFFFFFFFFu : ((1u << scale) - 1u);
    return (uint32_t)((v * 0x9E3779B1u + 0x7F4A7C15u) & mask);
}

void graphgen_rmat_arcs(int32_t* tail, int32_t* head, int32_t* weight, int64_t e_begin, int64_t e_end,
                        int32_t scale, double a, double b, double c, int32_t wlo, int32_t whi, uint64_t seed) {
    for (int64_t e = e_begin; e < e_end; ++e) {
        uint32_t u = 0, v = 0;
        for (int l = 0; l < scale; ++l) {
            const double r = gen_unit(graphgen_splitmix64_at(seed, (uint64_t)e * 64u + (uint64_t)l + 1u));
            const uint32_t bu = r >= a + b ? 1u : 0u;           /* quadrants c and d: lower half */
            const uint32_t bv = (r >= a && r < a + b) || r >= a + b + c ? 1u : 0u;  /* b and d: right half */
            u = (u << 1) | bu;
            v = (v << 1) | bv;
        }
        const int64_t k = e - e_begin;
        tail[k] = (int32_t)rmat_scramble(u, scale);
        head[k] = (int32_t)rmat_scramble(v, scale);
        weight[k] = gen_int(graphgen_splitmix64_at(seed, (1ULL << 44) + (uint64_t)e), wlo, whi);
    }
}

/* Stable counting sort by tail.  row_ptr must hold n + 1 entries. */
int graphgen_csr_from_arcs(const int32_t* tail, const int32_t* head, const int32_t* weight, int64_t m, int64_t n,
                           int64_t* row_ptr, int32_t* col, int32_t* w) {
    memset(row_ptr, 0, sizeof(int64_t) * (size_t)(n + 1));
    for (int64_t e = 0; e < m; ++e) {
        if (tail[e] < 0 || tail[e] >= n || head[e] < 0 || head[e] >= n) return -1;
        row_ptr[tail[e] + 1]++;
    }
    for (int64_t v = 0; v < n; ++v) row_ptr[v + 1] += row_ptr[v];
    int64_t* cur = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n ? n : 1));
    if (!cur) return -2;
    memcpy(cur, row_ptr, sizeof(int64_t) * (size_t)n);
    for (int64_t e = 0; e < m; ++e) {
        const int64_t p = cur[tail[e]]++;
        col[p] = head[e];
        w[p] = weight[e];
    }
    free(cur);
    return 0;
}
