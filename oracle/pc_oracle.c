/*
 * pc_oracle.c -- the ORACLE for dense point-cloud neighbor search.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * It is the plain, slow, obviously correct CPU statement of the operator
 * definitions on the mps-pointops 0.5.0 project page, section "The operators
 * in equations", and of the mps-pointops "Numerical contracts" page, section
 * "Selection and output".  Every function below names the passage it follows.
 *
 * Arithmetic: IEEE-754 binary32, round to nearest even, each operation rounded
 * separately.  The file must be compiled with -ffp-contract=off and without
 * -ffast-math (aarch64 GCC contracts a*b+c into an FMA by default, which would
 * change the rounding that the selection rules depend on).  Subnormals are
 * kept.  The squared distance is summed in the order ((dx*dx + dy*dy) + dz*dz),
 * the order the project page's "How the kernels work" section gives for FPS
 * and kNN; the "Numerical contracts" page fixes the Ball Query threshold as
 * fl32(fl32(r) * fl32(r)) with a strict "<".
 *
 * Inputs are finite float32 coordinates, row-major [B, N, 3]; indices int64.
 */
#define _POSIX_C_SOURCE 200809L  /* pthread barriers under -std=c11 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

#if defined(__FAST_MATH__)
#error "the oracle must not be built with fast-math"
#endif

/* Status codes of the oracle's own entry points. */
#define ORC_OK 0
#define ORC_BAD_ARGUMENT 1
#define ORC_NO_MEMORY 2

/*
 * Squared distance s = sum_{d=0..2} (a_d - b_d)^2.
 * Project page, "The operators in equations" (the shared squared distance);
 * summation order ((dx^2 + dy^2) + dz^2) from "How the kernels work".
 * Each statement below is one float32 operation.
 */
float orc_s32(const float *a, const float *b)
{
    float dx = a[0] - b[0];
    float dy = a[1] - b[1];
    float dz = a[2] - b[2];
    float xx = dx * dx;
    float yy = dy * dy;
    float zz = dz * dz;
    float sxy = xx + yy;
    return sxy + zz;
}

/*
 * Ball Query threshold R2 = fl32(fl32(r) * fl32(r)).
 * Project page, "Ball Query: first K within a radius"; "Numerical contracts",
 * "Selection and output" (r32 = fl32(r); R2_dense = fl32(r32 * r32)).
 */
float orc_radius_threshold(double radius)
{
    float r32 = (float)radius;
    float r2 = r32 * r32;
    return r2;
}

/*
 * Farthest point sampling, one call for all B clouds.
 * Project page, "Farthest point sampling":
 *   c_0 = start_idx,
 *   m_j(t) = min_{0<=u<=t} s(x_j, x_{c_u}),
 *   c_{t+1} = the smallest j with m_j(t) = max_l m_l(t).
 * The running minimum is the literal min over the selected centers, started
 * from the first center (no sentinel).  The scan for the maximum keeps the
 * first j that reaches it, which is the smallest index on an exact tie.  Once
 * every m_j is 0 the rule itself yields j = 0, so the slots after exhaustion
 * repeat index 0 (project page, "Contracts": furthest_point_sample).
 */
int orc_fps(const float *xyz, int64_t B, int64_t N, int64_t npoint,
            int64_t start_idx, int64_t *out_idx)
{
    if (B < 0 || N < 1 || npoint < 1 || start_idx < 0 || start_idx >= N)
        return ORC_BAD_ARGUMENT;
    float *m = (float *)malloc((size_t)N * sizeof(float));
    if (!m) return ORC_NO_MEMORY;
    for (int64_t b = 0; b < B; ++b) {
        const float *x = xyz + (size_t)b * (size_t)N * 3;
        int64_t *sel = out_idx + (size_t)b * (size_t)npoint;
        int64_t c = start_idx;
        sel[0] = c;
        for (int64_t j = 0; j < N; ++j)
            m[j] = orc_s32(x + 3 * j, x + 3 * c);
        for (int64_t t = 1; t < npoint; ++t) {
            /* c_t = smallest j attaining max_l m_l */
            int64_t best = 0;
            for (int64_t j = 1; j < N; ++j)
                if (m[j] > m[best]) best = j;
            c = best;
            sel[t] = c;
            /* m_j = min(m_j, s(x_j, x_c)) */
            for (int64_t j = 0; j < N; ++j) {
                float s = orc_s32(x + 3 * j, x + 3 * c);
                if (s < m[j]) m[j] = s;
            }
        }
    }
    free(m);
    return ORC_OK;
}

/*
 * Farthest point sampling with the points of each step split over T host
 * threads (the all-core CPU baseline).  Same definition as orc_fps (project
 * page, "Farthest point sampling"), same arithmetic per point: thread t owns
 * the points [lo_t, hi_t) of a contiguous split in increasing order; in each
 * step it updates m_j = min(m_j, s(x_j, x_c)) for its points and keeps the
 * first j of its range attaining its maximum; after a barrier one thread takes
 * the largest of those maxima, scanning the threads in increasing order and
 * replacing only on a strictly larger value, which is the smallest index
 * attaining the global maximum; a second barrier publishes the new center.
 */
typedef struct {
    const float *x;
    float *m;
    int64_t N, npoint, T;
    int64_t *sel;            /* out_idx of the current cloud */
    int64_t c;               /* current center */
    float *best_v;           /* [T] */
    int64_t *best_j;         /* [T] */
    pthread_barrier_t *bar;
} orc_fps_shared;

typedef struct {
    orc_fps_shared *sh;
    int64_t t;
} orc_fps_task;

static void *orc_fps_worker(void *arg)
{
    orc_fps_task *task = (orc_fps_task *)arg;
    orc_fps_shared *sh = task->sh;
    const int64_t t = task->t, T = sh->T, N = sh->N;
    const int64_t lo = N * t / T, hi = N * (t + 1) / T;
    const float *x = sh->x;
    float *m = sh->m;
    for (int64_t step = 0; step < sh->npoint; ++step) {
        const int64_t c = sh->c;
        /* m_j = s(x_j, x_{c_0}) on the first step, min with s(x_j, x_c) after */
        float bv = 0.0f;
        int64_t bj = -1;
        for (int64_t j = lo; j < hi; ++j) {
            float s = orc_s32(x + 3 * j, x + 3 * c);
            if (step == 0 || s < m[j]) m[j] = s;
            if (bj < 0 || m[j] > bv) {
                bv = m[j];
                bj = j;
            }
        }
        sh->best_v[t] = bv;
        sh->best_j[t] = bj;
        pthread_barrier_wait(sh->bar);
        if (t == 0 && step + 1 < sh->npoint) {
            int64_t best = -1;
            float v = 0.0f;
            for (int64_t u = 0; u < T; ++u)
                if (sh->best_j[u] >= 0 && (best < 0 || sh->best_v[u] > v)) {
                    v = sh->best_v[u];
                    best = sh->best_j[u];
                }
            sh->c = best;
            sh->sel[step + 1] = best;
        }
        pthread_barrier_wait(sh->bar);
    }
    return NULL;
}

int orc_fps_threads(const float *xyz, int64_t B, int64_t N, int64_t npoint,
                    int64_t start_idx, int64_t nthreads, int64_t *out_idx)
{
    if (B < 0 || N < 1 || npoint < 1 || start_idx < 0 || start_idx >= N ||
        nthreads < 1 || nthreads > 1024)
        return ORC_BAD_ARGUMENT;
    const int64_t T = nthreads;
    float *m = (float *)malloc((size_t)N * sizeof(float));
    float *bv = (float *)malloc((size_t)T * sizeof(float));
    int64_t *bj = (int64_t *)malloc((size_t)T * sizeof(int64_t));
    pthread_t *th = (pthread_t *)malloc((size_t)T * sizeof(pthread_t));
    orc_fps_task *tasks = (orc_fps_task *)malloc((size_t)T * sizeof(orc_fps_task));
    if (!m || !bv || !bj || !th || !tasks) {
        free(m); free(bv); free(bj); free(th); free(tasks);
        return ORC_NO_MEMORY;
    }
    pthread_barrier_t bar;
    pthread_barrier_init(&bar, NULL, (unsigned)T);
    int rc = ORC_OK;
    for (int64_t b = 0; b < B && rc == ORC_OK; ++b) {
        orc_fps_shared sh = {xyz + (size_t)b * (size_t)N * 3, m, N, npoint, T,
                             out_idx + (size_t)b * (size_t)npoint, start_idx,
                             bv, bj, &bar};
        sh.sel[0] = start_idx;
        int64_t started = 0;
        for (int64_t t = 1; t < T; ++t) {
            tasks[t].sh = &sh;
            tasks[t].t = t;
            if (pthread_create(&th[t], NULL, orc_fps_worker, &tasks[t]) != 0) break;
            ++started;
        }
        if (started != T - 1) {
            /* cannot run short of threads: the barrier counts T */
            for (int64_t t = 1; t <= started; ++t) pthread_cancel(th[t]);
            rc = ORC_NO_MEMORY;
            break;
        }
        tasks[0].sh = &sh;
        tasks[0].t = 0;
        orc_fps_worker(&tasks[0]);
        for (int64_t t = 1; t < T; ++t) pthread_join(th[t], NULL);
    }
    pthread_barrier_destroy(&bar);
    free(m); free(bv); free(bj); free(th); free(tasks);
    return rc;
}

/*
 * m_j for a given set of centers: min over the centers u of s(x_j, x_{c_u}).
 * The FPS running minimum of the project page's "Farthest point sampling"
 * equation, evaluated for chosen points j only.  Used by the at-scale property
 * checks (the selected center must attain the maximum of m).
 */
int orc_min_dist_to_set(const float *x, int64_t N, const int64_t *centers,
                        int64_t ncenters, const int64_t *points,
                        int64_t npoints, float *out)
{
    if (N < 1 || ncenters < 1) return ORC_BAD_ARGUMENT;
    for (int64_t i = 0; i < npoints; ++i) {
        int64_t j = points[i];
        if (j < 0 || j >= N) return ORC_BAD_ARGUMENT;
        float m = 0.0f;
        for (int64_t u = 0; u < ncenters; ++u) {
            int64_t c = centers[u];
            if (c < 0 || c >= N) return ORC_BAD_ARGUMENT;
            float s = orc_s32(x + 3 * j, x + 3 * c);
            if (u == 0 || s < m) m = s;
        }
        out[i] = m;
    }
    return ORC_OK;
}

/* One (squared distance, index) candidate of the kNN sort. */
typedef struct {
    float s;
    int64_t j;
} orc_pair;

/* Lexicographic order on (s, j): "sort by squared distance and then input
 * index" (project page, "k nearest neighbors"). */
static int orc_pair_cmp(const void *pa, const void *pb)
{
    const orc_pair *a = (const orc_pair *)pa;
    const orc_pair *b = (const orc_pair *)pb;
    if (a->s < b->s) return -1;
    if (a->s > b->s) return 1;
    if (a->j < b->j) return -1;
    if (a->j > b->j) return 1;
    return 0;
}

/*
 * kNN for a list of query rows.  Row r = b*Q + i names query i of cloud b.
 * Project page, "k nearest neighbors":
 *   pi_bi = argsort_j (s_bij, j),  I_bik = pi_bi[k],  D_bik = sqrt(s_bi,I_bik).
 * "Numerical contracts": the smallest k distances, exact ties to the smaller
 * reference index, Euclidean distances returned.  The sort is the C library's
 * qsort over all N candidates; k <= N ("Contracts": knn).  sqrtf is the
 * correctly rounded IEEE square root.
 * Outputs: out_dist[nrows*k] float32, out_idx[nrows*k] int64, row-major.
 */
int orc_knn_rows(const float *query, int64_t B, int64_t Q, const float *ref,
                 int64_t N, int64_t k, const int64_t *rows, int64_t nrows,
                 float *out_dist, int64_t *out_idx)
{
    if (B < 0 || Q < 0 || N < 1 || k < 1 || k > N) return ORC_BAD_ARGUMENT;
    orc_pair *cand = (orc_pair *)malloc((size_t)N * sizeof(orc_pair));
    if (!cand) return ORC_NO_MEMORY;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) {
            free(cand);
            return ORC_BAD_ARGUMENT;
        }
        int64_t b = row / Q;
        const float *q = query + (size_t)row * 3;
        const float *x = ref + (size_t)b * (size_t)N * 3;
        for (int64_t j = 0; j < N; ++j) {
            cand[j].s = orc_s32(q, x + 3 * j);
            cand[j].j = j;
        }
        qsort(cand, (size_t)N, sizeof(orc_pair), orc_pair_cmp);
        for (int64_t t = 0; t < k; ++t) {
            out_dist[r * k + t] = sqrtf(cand[t].s);
            out_idx[r * k + t] = cand[t].j;
        }
    }
    free(cand);
    return ORC_OK;
}

/*
 * Ball Query for a list of query rows.  Row r = b*Q + i names query i of
 * cloud b.  Project page, "Ball Query: first K within a radius":
 *   R2 = fl32(fl32(r) * fl32(r)),
 *   J_bi = [ j in 0..N-1 : s_bij < R2 ] in input order,
 *   (I, S)_bik = (J_bi[k], s_bi,J_bi[k]) for k < min(K, |J_bi|), else (-1, 0).
 * "Numerical contracts", "Selection and output": accept iff s32 < R2 (strict).
 * Outputs: out_dist2[nrows*K] float32, out_idx[nrows*K] int64, row-major.
 * N = 0 is allowed and gives padding only.
 */
int orc_ball_query_rows(const float *query, int64_t B, int64_t Q,
                        const float *ref, int64_t N, double radius, int64_t K,
                        const int64_t *rows, int64_t nrows, float *out_dist2,
                        int64_t *out_idx)
{
    if (B < 0 || Q < 0 || N < 0 || K < 1) return ORC_BAD_ARGUMENT;
    float R2 = orc_radius_threshold(radius);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) return ORC_BAD_ARGUMENT;
        int64_t b = row / Q;
        const float *q = query + (size_t)row * 3;
        const float *x = ref + (size_t)b * (size_t)N * 3;
        int64_t cnt = 0;
        for (int64_t j = 0; j < N && cnt < K; ++j) {
            float s = orc_s32(q, x + 3 * j);
            if (s < R2) {
                out_idx[r * K + cnt] = j;
                out_dist2[r * K + cnt] = s;
                ++cnt;
            }
        }
        for (; cnt < K; ++cnt) {
            out_idx[r * K + cnt] = -1;
            out_dist2[r * K + cnt] = 0.0f;
        }
    }
    return ORC_OK;
}

/*
 * Number of (query, reference) pairs the first-K Ball Query rule has to
 * examine for each row: the position of the K-th accepted reference plus one,
 * or N when fewer than K references are accepted.  Used to count the
 * algorithmic work of a Ball Query launch; it follows the same definition as
 * orc_ball_query_rows.
 */
int orc_ball_query_scan_len(const float *query, int64_t B, int64_t Q,
                            const float *ref, int64_t N, double radius,
                            int64_t K, const int64_t *rows, int64_t nrows,
                            int64_t *out_len)
{
    if (B < 0 || Q < 0 || N < 0 || K < 1) return ORC_BAD_ARGUMENT;
    float R2 = orc_radius_threshold(radius);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) return ORC_BAD_ARGUMENT;
        int64_t b = row / Q;
        const float *q = query + (size_t)row * 3;
        const float *x = ref + (size_t)b * (size_t)N * 3;
        int64_t cnt = 0, j = 0;
        for (; j < N && cnt < K; ++j)
            if (orc_s32(q, x + 3 * j) < R2) ++cnt;
        out_len[r] = j;
    }
    return ORC_OK;
}

/* Pairwise squared distances s32(a_i, b_i) for n point pairs (test helper). */
void orc_s32_pairs(const float *a, const float *b, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_s32(a + 3 * i, b + 3 * i);
}

/* ------------------------------------------------------------------------
 * Per-cloud valid lengths.  The project page's Chamfer contract ("Roadmap",
 * Phase 4: "lengths mask padding in forward and backward") and its
 * PyTorch3D-style Ball Query ("lengths1, lengths2") restrict cloud b to its
 * first qlen[b] queries and first rlen[b] references.  Reading taken: a
 * length outside [0, Q] (or [0, N]) is clamped to that range; rows past the
 * query length and slots past the available references hold (-1, 0), the
 * padding convention of "Ball Query: first K within a radius".
 * ---------------------------------------------------------------------- */
static int64_t orc_clamp_len(const int64_t *len, int64_t b, int64_t full)
{
    if (!len) return full;
    if (len[b] < 0) return 0;
    return len[b] > full ? full : len[b];
}

/*
 * kNN with lengths, optionally returning the squared distance.  Project
 * page, "k nearest neighbors": pi = argsort_j (s_bij, j) over the valid
 * references j < rlen[b]; D = sqrt(s), or s itself when `squared` is set
 * (the Chamfer operator's squared-L2 nearest distance, "Roadmap" Phase 4).
 * The first min(k, rlen[b]) entries are real; the rest are (-1, 0).
 */
int orc_knn_masked_rows(const float *query, int64_t B, int64_t Q,
                        const float *ref, int64_t N, int64_t k,
                        const int64_t *qlen, const int64_t *rlen, int squared,
                        const int64_t *rows, int64_t nrows, float *out_dist,
                        int64_t *out_idx)
{
    if (B < 0 || Q < 0 || N < 0 || k < 1) return ORC_BAD_ARGUMENT;
    orc_pair *cand = (orc_pair *)malloc((size_t)(N > 0 ? N : 1) * sizeof(orc_pair));
    if (!cand) return ORC_NO_MEMORY;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) {
            free(cand);
            return ORC_BAD_ARGUMENT;
        }
        int64_t b = row / Q, i = row % Q;
        int64_t nq = orc_clamp_len(qlen, b, Q);
        int64_t nr = orc_clamp_len(rlen, b, N);
        int64_t real = 0;
        if (i < nq) {
            const float *q = query + (size_t)row * 3;
            const float *x = ref + (size_t)b * (size_t)N * 3;
            for (int64_t j = 0; j < nr; ++j) {
                cand[j].s = orc_s32(q, x + 3 * j);
                cand[j].j = j;
            }
            qsort(cand, (size_t)nr, sizeof(orc_pair), orc_pair_cmp);
            real = k < nr ? k : nr;
        }
        for (int64_t t = 0; t < k; ++t) {
            if (t < real) {
                out_dist[r * k + t] = squared ? cand[t].s : sqrtf(cand[t].s);
                out_idx[r * k + t] = cand[t].j;
            } else {
                out_dist[r * k + t] = 0.0f;
                out_idx[r * k + t] = -1;
            }
        }
    }
    free(cand);
    return ORC_OK;
}

/*
 * Ball Query with lengths.  Project page, "Ball Query: first K within a
 * radius", over the valid references j < rlen[b]; query rows i >= qlen[b]
 * are padding in full ("PyTorch3D-style Ball Query": lengths1, lengths2).
 */
int orc_ball_query_masked_rows(const float *query, int64_t B, int64_t Q,
                               const float *ref, int64_t N,
                               const int64_t *qlen, const int64_t *rlen,
                               double radius, int64_t K, const int64_t *rows,
                               int64_t nrows, float *out_dist2,
                               int64_t *out_idx)
{
    if (B < 0 || Q < 0 || N < 0 || K < 1) return ORC_BAD_ARGUMENT;
    float R2 = orc_radius_threshold(radius);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) return ORC_BAD_ARGUMENT;
        int64_t b = row / Q, i = row % Q;
        int64_t nq = orc_clamp_len(qlen, b, Q);
        int64_t nr = orc_clamp_len(rlen, b, N);
        int64_t cnt = 0;
        if (i < nq) {
            const float *q = query + (size_t)row * 3;
            const float *x = ref + (size_t)b * (size_t)N * 3;
            for (int64_t j = 0; j < nr && cnt < K; ++j) {
                float s = orc_s32(q, x + 3 * j);
                int accept = s < R2;
                if (accept) {
                    out_idx[r * K + cnt] = j;
                    out_dist2[r * K + cnt] = s;
                    ++cnt;
                }
            }
        }
        for (; cnt < K; ++cnt) {
            out_dist2[r * K + cnt] = 0.0f;
            out_idx[r * K + cnt] = (int64_t)-1;
        }
    }
    return ORC_OK;
}

/*
 * Gather of neighbor coordinates: out[b,i,t,:] = x[b, idx[b,i,t], :], and
 * (0, 0, 0) where idx = -1.  Project page, "PyTorch3D-style Ball Query":
 * return_nn gives the neighbor coordinates, "with zero coordinates in knn
 * where idx = -1".  Any other index outside [0, N) is an error.
 */
int orc_gather_points(const float *x, int64_t B, int64_t N,
                      const int64_t *idx, int64_t Q, int64_t K, float *out)
{
    if (B < 0 || N < 0 || Q < 0 || K < 0) return ORC_BAD_ARGUMENT;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t e = 0; e < Q * K; ++e) {
            int64_t j = idx[b * Q * K + e];
            float *o = out + (size_t)(b * Q * K + e) * 3;
            if (j == -1) {
                o[0] = o[1] = o[2] = 0.0f;
            } else if (j < 0 || j >= N) {
                return ORC_BAD_ARGUMENT;
            } else {
                const float *p = x + (size_t)(b * N + j) * 3;
                o[0] = p[0];
                o[1] = p[1];
                o[2] = p[2];
            }
        }
    return ORC_OK;
}

/*
 * three_interpolate forward (project page, Quick start and "Roadmap" Phase 2:
 * PointNet++ feature propagation with externally computed weights):
 *   out[b,c,i] = sum_{t=0..2} w[b,i,t] * f[b,c,idx[b,i,t]]
 * features f [B,C,M], idx [B,n,3] int64, w [B,n,3], out [B,C,n].
 * Reading taken: float32, each product and sum rounded separately, summed
 * in the order ((w0 f0 + w1 f1) + w2 f2); idx = -1 (padding) reads the
 * feature as 0; any other index outside [0, M) is an error.
 */
int orc_three_interpolate(const float *f, int64_t B, int64_t C, int64_t M,
                          const int64_t *idx, const float *w, int64_t n,
                          float *out)
{
    if (B < 0 || C < 0 || M < 0 || n < 0) return ORC_BAD_ARGUMENT;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t i = 0; i < n; ++i)
            for (int t = 0; t < 3; ++t) {
                int64_t m = idx[(b * n + i) * 3 + t];
                if (m != -1 && (m < 0 || m >= M)) return ORC_BAD_ARGUMENT;
            }
    for (int64_t b = 0; b < B; ++b)
        for (int64_t c = 0; c < C; ++c) {
            const float *fr = f + (size_t)(b * C + c) * (size_t)M;
            for (int64_t i = 0; i < n; ++i) {
                const int64_t *id = idx + (b * n + i) * 3;
                const float *wi = w + (b * n + i) * 3;
                float term[3];
                for (int t = 0; t < 3; ++t) {
                    float v = id[t] == -1 ? 0.0f : fr[id[t]];
                    term[t] = wi[t] * v;
                }
                float s01 = term[0] + term[1];
                out[(b * C + c) * n + i] = s01 + term[2];
            }
        }
    return ORC_OK;
}

/*
 * three_interpolate backward ("Roadmap" Phase 2: "accumulates backward
 * gradients into input features"): with upstream gradient g [B,C,n],
 *   grad_f[b,c,m] = sum over (i, t) with idx[b,i,t] = m of w[b,i,t] g[b,c,i].
 * The sum is accumulated in float32 from 0 in increasing (i, t) order, each
 * product and addition rounded; the pages allow any summation order (the
 * GPU accumulates atomically), so parity is to a bound on the order.
 */
int orc_three_interpolate_backward(const float *g, int64_t B, int64_t C,
                                   int64_t n, const int64_t *idx,
                                   const float *w, int64_t M, float *grad_f)
{
    if (B < 0 || C < 0 || M < 0 || n < 0) return ORC_BAD_ARGUMENT;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t i = 0; i < n; ++i)
            for (int t = 0; t < 3; ++t) {
                int64_t m = idx[(b * n + i) * 3 + t];
                if (m != -1 && (m < 0 || m >= M)) return ORC_BAD_ARGUMENT;
            }
    memset(grad_f, 0, (size_t)(B * C * M) * sizeof(float));
    for (int64_t b = 0; b < B; ++b)
        for (int64_t c = 0; c < C; ++c) {
            float *gr = grad_f + (size_t)(b * C + c) * (size_t)M;
            const float *gi = g + (size_t)(b * C + c) * (size_t)n;
            for (int64_t i = 0; i < n; ++i)
                for (int t = 0; t < 3; ++t) {
                    int64_t m = idx[(b * n + i) * 3 + t];
                    if (m == -1) continue;
                    float p = w[(b * n + i) * 3 + t] * gi[i];
                    gr[m] = gr[m] + p;
                }
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * kNN in D dimensions (project page, "Roadmap", Phase 2: kNN in arbitrary
 * dimension for feature-space neighbour search, with "direct
 * dimension-by-dimension distance accumulation as the numerical baseline"):
 *   s = fl(... fl(fl(t_0 + t_1) + t_2) ... + t_{D-1}),  t_d = fl(fl(q_d - x_d)^2),
 * accumulated in increasing d, each operation a separately rounded float32
 * operation (for D = 3 this is exactly s32).  Selection as "k nearest
 * neighbors": the first k of the lexicographic (s, j) order; D = sqrt(s)
 * or s itself when `squared` is set.  query [B, Q, D], ref [B, N, D].
 * ---------------------------------------------------------------------- */
float orc_sd(const float *a, const float *b, int64_t D)
{
    float s = 0.0f;
    for (int64_t d = 0; d < D; ++d) {
        float t = a[d] - b[d];
        float t2 = t * t;
        s = s + t2;
    }
    return s;
}

int orc_knn_d_rows(const float *query, int64_t B, int64_t Q, const float *ref,
                   int64_t N, int64_t D, int64_t k, int squared,
                   const int64_t *rows, int64_t nrows, float *out_dist,
                   int64_t *out_idx)
{
    if (B < 0 || Q < 0 || N < 1 || D < 1 || k < 1 || k > N) return ORC_BAD_ARGUMENT;
    orc_pair *cand = (orc_pair *)malloc((size_t)N * sizeof(orc_pair));
    if (!cand) return ORC_NO_MEMORY;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        if (row < 0 || row >= B * Q) {
            free(cand);
            return ORC_BAD_ARGUMENT;
        }
        int64_t b = row / Q;
        const float *q = query + (size_t)row * (size_t)D;
        const float *x = ref + (size_t)b * (size_t)N * (size_t)D;
        for (int64_t j = 0; j < N; ++j) {
            cand[j].s = orc_sd(q, x + (size_t)j * (size_t)D, D);
            cand[j].j = j;
        }
        qsort(cand, (size_t)N, sizeof(orc_pair), orc_pair_cmp);
        for (int64_t t = 0; t < k; ++t) {
            float sd = cand[t].s;
            out_dist[r * k + t] = squared ? sd : sqrtf(sd);
            out_idx[r * k + t] = cand[t].j;
        }
    }
    free(cand);
    return ORC_OK;
}
