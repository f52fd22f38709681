/*
 * pointcloud.h -- C ABI of the GB300 (sm_103a) dense point-cloud neighbor
 * search library (libpointcloud.so).
 *
 * Three operators over dense, batched float32 clouds, with the selection rules
 * of the mps-pointops 0.5.0 project page ("The operators in equations",
 * "Contracts") and the mps-pointops "Numerical contracts" page ("Selection and
 * output"):
 *
 *   squared distance  s(i,j) = ((dx*dx + dy*dy) + dz*dz), dx = q_x - x_x, ...
 *                     every operation a separately rounded float32 operation
 *                     (round to nearest even, no FMA contraction, subnormals
 *                     kept).  All three operators select on this value.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: coordinates are row-major [B, N, 3] float32 (x, y, z of a point
 *    adjacent; clouds adjacent); outputs are row-major as stated per call.
 *  - Memory: every pointer argument named *xyz, *query, *ref, *out_* is a
 *    DEVICE pointer (cudaMalloc / caching-allocator / managed memory) on the
 *    current CUDA device, owned by the caller.  The library never frees or
 *    keeps a caller pointer.  Coordinates must be 4-byte aligned, int64
 *    outputs 8-byte aligned.  Inputs and outputs must not overlap.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Every call only enqueues work on that stream and
 *    returns; results are ready when the stream reaches that point.  Calls
 *    on one stream run in order; calls on different streams share nothing
 *    except the library's device status word (see pc_device_status).
 *  - Errors: arguments are validated on the host before anything is
 *    enqueued; a rejected call enqueues nothing and returns a status code.
 *    There is no silent fallback to another device or to the CPU.
 *    pc_last_error_message() gives a one-line reason for the last failing
 *    call on the calling host thread.
 *  - Inputs must be finite.  Ball Query never accepts a NaN distance; FPS and
 *    kNN results for non-finite coordinates are unspecified.
 *  - Sizes: B, N, Q >= 0 with N < 2^31 and every output size < 2^62 elements.
 *  - Scratch memory: calls that need scratch (stated per call) take it,
 *    stream-ordered on the call's stream, from a memory pool the library
 *    creates per device on first use (cudaMemPoolCreate +
 *    cudaMallocFromPoolAsync) and return it there after their kernels.  The
 *    pool keeps up to 256 MiB reserved between calls, so a caller that
 *    synchronizes after every call does not pay for mapping the memory again
 *    each time; where the device has no memory pools the device's default
 *    pool (cudaMallocAsync) is used.  pc_fps_grid_static allocates nothing.
 */
#ifndef POINTCLOUD_H
#define POINTCLOUD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum pc_status {
    PC_OK = 0,
    PC_ERR_INVALID_ARGUMENT = 1, /* a size, pointer or parameter is invalid  */
    PC_ERR_UNSUPPORTED = 2,      /* valid, but beyond what the library runs  */
    PC_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed     */
    PC_ERR_DEVICE_TIMEOUT = 4,   /* a bounded device-side wait ran out       */
    PC_ERR_NO_DEVICE = 5         /* no usable sm_103 device is current       */
} pc_status;

/* Static, NUL-terminated name of a status code ("PC_OK", ...). */
const char *pc_status_string(int status);

/* One-line reason for the last non-OK status returned on this host thread
 * (empty string if none).  The pointer stays valid until the next call that
 * fails on this thread. */
const char *pc_last_error_message(void);

/* Library version as 10000*major + 100*minor + patch. */
int pc_version(void);

/*
 * Farthest point sampling.
 * Project page, "Farthest point sampling": c_0 = start_idx; with
 * m_j(t) = min_{u<=t} s(x_j, x_{c_u}), the next center is the smallest j
 * attaining max_l m_l(t).  "Contracts": once every point is taken the
 * remaining slots repeat index 0.  The same start index is used for every
 * cloud.
 *
 *   xyz        [B, N, 3] float32, device.
 *   out_idx    [B, npoint] int64, device; written in full.
 *   npoint     >= 1 (npoint > N is allowed).  0 <= start_idx < N when B > 0.
 *   workspace  device scratch of at least pc_fps_workspace_bytes(B, N,
 *              npoint) bytes, 256-byte aligned, or NULL.  When the chosen
 *              schedule needs scratch and workspace is NULL the library takes
 *              it from the library's stream-ordered scratch pool (see
 *              "Scratch memory" above) and
 *              frees it after the launch on the same stream.  A workspace must
 *              not be shared by calls that may run concurrently.
 *
 * Schedules (chosen from B and N): one thread block per cloud, one thread
 * block cluster per cloud (distributed shared memory), or -- for clouds too
 * large for one cluster -- a cooperative grid of clusters per cloud: the
 * blocks of each cluster send their lists of best points to the cluster's
 * first block through distributed shared memory, which publishes the
 * cluster's summary (up to 128 listed points and a bound, 4128 bytes per
 * cluster and round parity) through the workspace, and every block
 * certifies the same run of centers from all clusters' summaries (the
 * rounds of pc_fps_set_batched; with rounds off, one tagged key and the
 * point's coordinates per cluster and step; with cluster_size 1 in
 * pc_fps_ex, one level: one 64-bit key per block and step).  Only the grid
 * schedule uses scratch; the cluster and grid schedules bound their device-side waits: if a wait runs out the kernel
 * stops, writes -1 into the remaining out_idx slots of that cloud and raises
 * the device status word (PC_ERR_DEVICE_TIMEOUT).
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT, PC_ERR_UNSUPPORTED (cloud too large
 * for the on-chip schedules), PC_ERR_CUDA or PC_ERR_NO_DEVICE.
 */
int pc_fps(const float *xyz, int64_t B, int64_t N, int64_t npoint,
           int64_t start_idx, int64_t *out_idx, void *workspace,
           size_t workspace_bytes, void *stream);

/* Scratch bytes pc_fps needs for these sizes (0 when no scratch is used). */
size_t pc_fps_workspace_bytes(int64_t B, int64_t N, int64_t npoint);

/* FPS schedule selectors for pc_fps_ex. */
typedef enum pc_fps_strategy {
    PC_FPS_AUTO = 0,
    PC_FPS_BLOCK = 1,   /* one thread block per cloud                        */
    PC_FPS_CLUSTER = 2, /* one thread block cluster per cloud                */
    PC_FPS_GRID = 3     /* cooperative grid, workspace exchange (see above)  */
} pc_fps_strategy;

/* pc_fps with an explicit schedule (results are identical for every
 * schedule).  `cluster_size` (0 = automatic) is the cluster of
 * PC_FPS_CLUSTER (1..16) or the cluster of the two-level PC_FPS_GRID (1 = one
 * level, 2..16; blocks_per_cloud must then be a multiple of it);
 * `blocks_per_cloud` (0 = automatic) applies to PC_FPS_GRID.  The workspace
 * size for PC_FPS_GRID with cluster_size 0 is pc_fps_workspace_bytes_ex. */
int pc_fps_ex(const float *xyz, int64_t B, int64_t N, int64_t npoint,
              int64_t start_idx, int64_t *out_idx, void *workspace,
              size_t workspace_bytes, int strategy, int cluster_size,
              int blocks_per_cloud, void *stream);

size_t pc_fps_workspace_bytes_ex(int64_t B, int64_t N, int64_t npoint,
                                 int strategy, int blocks_per_cloud);

/* The schedule pc_fps_ex would run for these sizes and arguments on the
 * current device: *out_strategy (PC_FPS_BLOCK, _CLUSTER or _GRID),
 * *out_cluster_size (blocks per thread block cluster; 1 for PC_FPS_BLOCK and
 * for the one-level grid) and *out_blocks_per_cloud.  Nothing is enqueued.
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT (B or N < 1, null outputs),
 * PC_ERR_UNSUPPORTED (no schedule fits) or PC_ERR_NO_DEVICE. */
int pc_fps_plan(int64_t B, int64_t N, int strategy, int cluster_size,
                int blocks_per_cloud, int *out_strategy, int *out_cluster_size,
                int *out_blocks_per_cloud);

/*
 * pc_fps_grid_static: pc_fps with the PC_FPS_GRID schedule for callers that
 * cannot allocate device memory at call time (for instance a host program
 * that has given all device memory to its own pool, so cudaMalloc would fail
 * or break its accounting, or a real-time loop with a fixed footprint).  The
 * mps-pointops pages have no counterpart of this entry point.
 *
 * The grid schedule's exchange scratch is a fixed array of 16384 64-bit
 * words (128 KiB) inside the library, present on every device that loads
 * the library until the process exits; the call allocates nothing.  The
 * two-level grid runs in rounds when its summaries fit in the array (B * 2 *
 * clusters per cloud slots of 4128 bytes), else one center per step.  Limit:
 * the step-by-step schedule needs B * max(2 * blocks_per_cloud, 32 *
 * clusters per cloud) words (one 128-byte line per cluster and step parity
 * with two levels; 2 words per block with one level, when blocks_per_cloud
 * is not a multiple of 4), at most 16384 in all, and the blocks are bounded
 * by the SM count; larger requests return PC_ERR_INVALID_ARGUMENT.  Arguments and results are
 * those of pc_fps_ex with strategy PC_FPS_GRID and cluster_size 0
 * (blocks_per_cloud 0 = automatic).
 *
 * The first call on a device (while it is current) looks up the array's
 * device address with cudaGetSymbolAddress; make that first call before any
 * stream capture.  The address is cached for the life of the process: after
 * a cudaDeviceReset the entry point must not be called again.  Devices with
 * ordinals of 64 and above get PC_ERR_UNSUPPORTED.  Every call on a device
 * uses the same array, and each call
 * clears the words it needs (stream-ordered) before its kernel.  Calls whose
 * work may overlap on the GPU (different streams without ordering between
 * them) race on the array and must not be issued.
 */
int pc_fps_grid_static(const float *xyz, int64_t B, int64_t N, int64_t npoint,
                       int64_t start_idx, int64_t *out_idx,
                       int blocks_per_cloud, void *stream);

/*
 * k nearest neighbors.
 * Project page, "k nearest neighbors": for each query, candidates sorted by
 * (s, j) -- squared distance, then reference index -- and the first k
 * returned with Euclidean distance D = sqrt(s) (correctly rounded float32
 * square root).  "Numerical contracts": exact ties go to the smaller index.
 *
 *   query     [B, Q, 3] float32, device.   ref [B, N, 3] float32, device.
 *   out_dist  [B, Q, k] float32, device.   out_idx [B, Q, k] int64, device.
 *             Row (b, i) lists the k neighbors of query i of cloud b in
 *             increasing (s, j) order; indices are into cloud b of ref.
 *   k         1 <= k <= N ("Contracts": k <= N), and k <= 256.
 *
 * Scratch: with at least 16,384 references and 4,096 queries per cloud and
 * 2 <= k <= 32 the call first puts the points in a spatial order.  It takes
 * that scratch -- ordered copies of the references (and of the queries
 * unless they are the references), 16 bytes a point; cell tables of about
 * 640 KB per cloud; a seed heap of k 8-byte keys per query; with few queries
 * against many references, up to 8 parts' k keys per query -- from the
 * library's stream-ordered scratch pool on `stream` and frees it there
 * after its kernels; an allocation failure returns PC_ERR_CUDA.  Results do
 * not depend on the path taken.
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT (k > N, k < 1, bad pointer ...),
 * PC_ERR_UNSUPPORTED (k > 256), PC_ERR_CUDA or PC_ERR_NO_DEVICE.
 */
int pc_knn(const float *query, int64_t B, int64_t Q, const float *ref,
           int64_t N, int64_t k, float *out_dist, int64_t *out_idx,
           void *stream);

/*
 * kNN with per-cloud valid lengths and a choice of returned distance.
 * Same selection as pc_knn (project page, "k nearest neighbors"), restricted
 * per cloud b to queries i < query_lengths[b] and references
 * j < ref_lengths[b] (the lengths masks of the project page's Chamfer and
 * PyTorch3D-style contracts, "Roadmap" Phase 4 and "PyTorch3D-style Ball
 * Query").
 *
 *   query_lengths, ref_lengths  [B] int64, device, or NULL (= Q, = N).
 *              Values are clamped to [0, Q] and [0, N].
 *   k          1 <= k <= 256; k > N is allowed here.
 *   flags      0, or PC_KNN_SQUARED to return the squared distance s
 *              instead of sqrt(s).
 *   Rows i >= query_lengths[b], and slots past the cloud's valid reference
 *   count, hold (index -1, distance 0).  Other outputs as pc_knn.
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT, PC_ERR_UNSUPPORTED, PC_ERR_CUDA or
 * PC_ERR_NO_DEVICE.
 */
#define PC_KNN_SQUARED 1
int pc_knn_ex(const float *query, int64_t B, int64_t Q, const float *ref,
              int64_t N, int64_t k, const int64_t *query_lengths,
              const int64_t *ref_lengths, int flags, float *out_dist,
              int64_t *out_idx, void *stream);

/*
 * Ball Query: the first K references in input order inside the radius.
 * Project page, "Ball Query: first K within a radius"; "Numerical
 * contracts", "Selection and output":
 *   R2 = fl32(fl32(r) * fl32(r)); reference j is accepted iff s < R2
 *   (strict); the first K accepted j in increasing order are returned with
 *   their squared distances; unused slots hold (index -1, distance 0).
 *
 *   query      [B, Q, 3] float32, device.  ref [B, N, 3] float32, device.
 *   radius     finite and > 0 (rounded to float32 by the library).
 *   K          >= 1.  N = 0 is allowed (all slots padded).
 *   out_dist2  [B, Q, K] float32, device.  out_idx [B, Q, K] int64, device.
 *
 * Scratch: with few queries against many references (under 24 queries per
 * warp of the GPU-wide launch and at least 64 tiles of 256 references) the
 * references are split into P <= 8 parts that run side by side and whose
 * first-K hits are then joined in part order; that takes P * B * Q * (12 K
 * + 4) bytes (at most 1 GiB) from the library's stream-ordered scratch pool
 * on `stream`, freed there after the merge; an allocation
 * failure returns PC_ERR_CUDA.  Results do not depend on the path taken.
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT, PC_ERR_CUDA or PC_ERR_NO_DEVICE.
 */
int pc_ball_query(const float *query, int64_t B, int64_t Q, const float *ref,
                  int64_t N, double radius, int64_t K, float *out_dist2,
                  int64_t *out_idx, void *stream);

/*
 * Ball Query with per-cloud valid lengths: pc_ball_query restricted per cloud
 * b to queries i < query_lengths[b] and references j < ref_lengths[b]
 * (project page, "PyTorch3D-style Ball Query": lengths1, lengths2).
 *
 *   query_lengths, ref_lengths  [B] int64, device, or NULL (= Q, = N).
 *              Values are clamped to [0, Q] and [0, N].
 *   Rows i >= query_lengths[b] hold (index -1, distance 0) in every slot.
 *   Other arguments and outputs as pc_ball_query.
 */
int pc_ball_query_ex(const float *query, int64_t B, int64_t Q,
                     const float *ref, int64_t N, const int64_t *query_lengths,
                     const int64_t *ref_lengths, double radius, int64_t K,
                     float *out_dist2, int64_t *out_idx, void *stream);

/*
 * kNN and Ball Query of the same queries against the same references in one
 * call: the results of pc_knn(query, ref, k) and pc_ball_query(query, ref,
 * radius, K), bit for bit (project page, "k nearest neighbors" and "Ball
 * Query: first K within a radius"; "Numerical contracts").  A
 * set-abstraction layer asks both of one cloud; both read every (query,
 * reference) pair's squared distance, and here each pair is filtered and,
 * where it may matter to either, computed once.
 *
 *   query      [B, Q, 3] float32, device.  ref [B, N, 3] float32, device.
 *   k          1 <= k <= N, k <= 256.  knn_dist / knn_idx [B, Q, k]: as
 *              pc_knn's out_dist (Euclidean) / out_idx.
 *   radius     finite and > 0; K >= 1.  bq_dist2 / bq_idx [B, Q, K]: as
 *              pc_ball_query's out_dist2 / out_idx.
 *
 * One fused pass runs where pc_knn_ball_query_plan says so: 2 <= k <= 32,
 * K <= 64, at least 16,384 references and 4,096 queries per cloud, B <= 64,
 * R2 = fl32(fl32(r)^2) > 0, and the references are not split into parts
 * (enough queries to fill the GPU).  Otherwise the call runs pc_knn's and
 * pc_ball_query's kernels one after the other.  The fused pass takes
 * pc_knn's ordered-path scratch plus B * Q * (8 K + 16) bytes from the
 * library's stream-ordered scratch pool on `stream`; an allocation failure
 * returns PC_ERR_CUDA.  A wait that runs out (PC_ERR_DEVICE_TIMEOUT in the
 * status word, pc_device_status) leaves the stopped queries' rows of both
 * outputs at index -1 (kNN distances unspecified there, as pc_knn; Ball
 * Query distances 0).
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT, PC_ERR_UNSUPPORTED, PC_ERR_CUDA or
 * PC_ERR_NO_DEVICE.
 */
int pc_knn_ball_query(const float *query, int64_t B, int64_t Q, const float *ref,
                      int64_t N, int64_t k, float *knn_dist, int64_t *knn_idx,
                      double radius, int64_t K, float *bq_dist2, int64_t *bq_idx,
                      void *stream);

/*
 * Whether pc_knn_ball_query with these sizes runs the fused pass on the
 * current device: *out_fused = 1 (fused) or 0 (pc_knn's and pc_ball_query's
 * kernels).  Arguments are checked as by pc_knn_ball_query.  Returns PC_OK,
 * PC_ERR_INVALID_ARGUMENT, PC_ERR_UNSUPPORTED or PC_ERR_NO_DEVICE.
 */
int pc_knn_ball_query_plan(int64_t B, int64_t Q, int64_t N, int64_t k, double radius,
                           int64_t K, int *out_fused);

/*
 * Exact grid-accelerated kNN and Ball Query.
 * mps-pointops project page, "Roadmap" (Phase 4: spatial acceleration
 * structures, a uniform grid or BVH, for large clouds): the same operators
 * as pc_knn and pc_ball_query -- same squared-distance arithmetic, same
 * (s, j) order, same strict radius test, same padding -- computed from a
 * uniform grid over each reference cloud, so that a query examines only the
 * cells that can hold its answer.  Results are identical to pc_knn and
 * pc_ball_query for finite inputs.
 *
 * A grid is caller-owned device memory of pc_grid_bytes(B, N) bytes,
 * 256-byte aligned.  pc_grid_build fills it from ref [B, N, 3] (enqueued on
 * `stream`; the points are copied into the grid, so ref may change
 * afterwards); the query calls read it and may run any number of times, on
 * any stream ordered after the build.  A grid must not be rebuilt while a
 * query that reads it may still run.
 *
 *   pc_knn_grid:         1 <= k <= N, k <= 256; outputs as pc_knn.
 *   pc_ball_query_grid:  radius finite and > 0, 1 <= K <= 256; outputs as
 *                        pc_ball_query.  N = 0 gives padding only.
 * B, N must be the values the grid was built with.
 */
size_t pc_grid_bytes(int64_t B, int64_t N);

int pc_grid_build(const float *ref, int64_t B, int64_t N, void *grid,
                  size_t grid_bytes, void *stream);

int pc_knn_grid(const float *query, int64_t B, int64_t Q, const void *grid,
                int64_t N, int64_t k, float *out_dist, int64_t *out_idx,
                void *stream);

int pc_ball_query_grid(const float *query, int64_t B, int64_t Q,
                       const void *grid, int64_t N, double radius, int64_t K,
                       float *out_dist2, int64_t *out_idx, void *stream);

/*
 * kNN in D dimensions (feature-space neighbour search).  Project page,
 * "Roadmap", Phase 2: "direct dimension-by-dimension distance accumulation":
 *   s = fl(... fl(fl(t_0 + t_1) + t_2) ... + t_{D-1}),  t_d = fl(fl(q_d - x_d)^2),
 * accumulated in increasing d, every operation a separately rounded float32
 * operation (D = 3 gives the s32 of pc_knn).  Selection as pc_knn: the first
 * k of the (s, j) lexicographic order; distance sqrt(s), or s with
 * PC_KNN_SQUARED.
 *
 *   query [B, Q, D], ref [B, N, D] float32, device.  1 <= k <= N, k <= 32,
 *   1 <= D <= 256 (PC_ERR_UNSUPPORTED above).
 *   out_dist [B, Q, k] float32, out_idx [B, Q, k] int64, device.
 */
int pc_knn_d(const float *query, int64_t B, int64_t Q, const float *ref,
             int64_t N, int64_t D, int64_t k, int flags, float *out_dist,
             int64_t *out_idx, void *stream);

/* ------------------------------------------------------------------------
 * Chamfer distance, PointNet++ feature propagation, neighbor gather.
 * ---------------------------------------------------------------------- */

typedef enum pc_reduction {
    PC_REDUCTION_NONE = 0,
    PC_REDUCTION_SUM = 1,
    PC_REDUCTION_MEAN = 2
} pc_reduction;

/*
 * Bidirectional squared-L2 Chamfer distance, forward.  Project page, "Quick
 * start" (chamfer_distance) and "Roadmap", Phase 4:
 *   L = sum_i |x_i - y_a(i)|^2 + sum_j |y_j - x_b(j)|^2,
 * a(i) the nearest valid point of y to x_i and b(j) the nearest valid point
 * of x to y_j, found exactly as pc_knn_ex with k = 1 (smallest s, ties to the
 * smaller index).
 *
 *   x [B, P1, 3], y [B, P2, 3]  float32, device.
 *   x_lengths, y_lengths  [B] int64, device, or NULL; clamped to [0, P].
 *              Points past a cloud's length are neither queries nor
 *              references.
 *   weights    [B] float32, device, or NULL: each cloud's loss is scaled.
 *   point_reduction  PC_REDUCTION_SUM or PC_REDUCTION_MEAN (a cloud's sum
 *              divided by max(length, 1)).
 *   batch_reduction  PC_REDUCTION_NONE (out_loss [B]), SUM or MEAN (out_loss
 *              [1]; MEAN divides by B).
 *   single_directional  nonzero: only the x -> y term (out_*_y unused).
 *   out_dist_x [B, P1] float32, out_idx_x [B, P1] int64: squared distance and
 *              index of each x point's nearest y point ((0, -1) for masked
 *              points and for clouds without valid y points).
 *   out_dist_y, out_idx_y  [B, P2], the other direction.
 *   out_loss   float32, device, or NULL (no reduction).  Sums are formed in
 *              float64 in a fixed order and rounded once to float32.
 * Launches: one kNN kernel (both directions), then with out_loss one
 * reduction block per cloud and, for a batch SUM or MEAN, one more block
 * (the clouds' losses in stream-ordered scratch of B doubles).
 *
 * Returns PC_OK, PC_ERR_INVALID_ARGUMENT, PC_ERR_UNSUPPORTED, PC_ERR_CUDA or
 * PC_ERR_NO_DEVICE.
 */
int pc_chamfer(const float *x, int64_t B, int64_t P1, const float *y,
               int64_t P2, const int64_t *x_lengths, const int64_t *y_lengths,
               const float *weights, int point_reduction, int batch_reduction,
               int single_directional, float *out_dist_x, int64_t *out_idx_x,
               float *out_dist_y, int64_t *out_idx_y, float *out_loss,
               void *stream);

/*
 * three_interpolate, forward.  Project page, "Quick start" and "Roadmap",
 * Phase 2 (PointNet++ feature propagation with externally computed weights):
 *   out[b,c,i] = (w0 f[b,c,m0] + w1 f[b,c,m1]) + w2 f[b,c,m2],
 *   (m_t, w_t) = (idx[b,i,t], weight[b,i,t]); float32, each product and sum
 *   rounded separately in that order.
 *
 *   features [B, C, M] float32, idx [B, n, 3] int64, weight [B, n, 3]
 *   float32, out [B, C, n] float32; all device.
 *   idx = -1 reads the feature as 0 (padding).  Any other index outside
 *   [0, M) is also read as 0 and sets PC_ERR_INVALID_ARGUMENT in the device
 *   status word (pc_device_status).
 */
int pc_three_interpolate(const float *features, int64_t B, int64_t C,
                         int64_t M, const int64_t *idx, const float *weight,
                         int64_t n, float *out, void *stream);

/*
 * three_interpolate, backward ("Roadmap", Phase 2: gradients accumulated into
 * the input features):
 *   grad_features[b,c,m] = sum over (i, t) with idx[b,i,t] = m of
 *                          weight[b,i,t] * grad_out[b,c,i].
 * grad_features [B, C, M] is overwritten.  For M <= 16384 and n <= 8192 each
 * sum is formed from 0 in increasing (i, t) order, every product and
 * addition rounded to float32 (deterministic; bit-identical run to run): three
 * kernels build and sort a per-cloud list of the entries of every known
 * point, in stream-ordered scratch (the library's pool, 8 bytes per entry plus
 * M + 1 ints per cloud), then sum each list in order.  Larger sizes zero
 * grad_features and accumulate with float32 atomic adds, whose summation
 * order is not fixed ("Numerical contracts", "Differentiation": the order
 * may vary).  Index rules as pc_three_interpolate.
 */
int pc_three_interpolate_backward(const float *grad_out, int64_t B, int64_t C,
                                  int64_t n, const int64_t *idx,
                                  const float *weight, int64_t M,
                                  float *grad_features, void *stream);

/*
 * Neighbor coordinates for a [B, Q, K] index tensor (project page,
 * "PyTorch3D-style Ball Query": return_nn, zero coordinates where idx = -1):
 *   out[b,q,t,:] = xyz[b, idx[b,q,t], :], or (0, 0, 0) for idx = -1.
 *   xyz [B, N, 3] float32, idx [B, Q, K] int64, out [B, Q, K, 3] float32;
 *   device.  Other out-of-range indices give zeros and set
 *   PC_ERR_INVALID_ARGUMENT in the device status word.
 */
int pc_gather_points(const float *xyz, int64_t B, int64_t N,
                     const int64_t *idx, int64_t Q, int64_t K, float *out,
                     void *stream);

/*
 * Device status word.  Kernels that wait on other thread blocks bound every
 * wait; when a wait runs out they record PC_ERR_DEVICE_TIMEOUT here (the
 * first error wins) and return instead of hanging.  This call synchronizes
 * `stream`, copies the word of the current device to *out_status (PC_OK if
 * nothing was recorded) and, if `reset` is non-zero, clears it.
 */
int pc_device_status(void *stream, int reset, int32_t *out_status);

/*
 * Bound on each device-side wait, in nanoseconds (default 2e9).  Applies to
 * launches enqueued after the call, on every device.  Values below 1000 are
 * raised to 1000.
 *
 * Testing hooks, so that every bounded wait can be made to run out without
 * a fault: pc_debug_set_stall(mask) applies to launches enqueued after the
 * call (0 restores normal operation):
 *   PC_STALL_FPS_GRID     block 0 of each cloud of a PC_FPS_GRID launch
 *                         withholds its first exchange word: every block's
 *                         wait for that step runs out;
 *   PC_STALL_FPS_CLUSTER  block 0 of the first cloud of a PC_FPS_CLUSTER
 *                         launch withholds its first candidate: every block
 *                         of that cluster runs out its wait for that step;
 *   PC_STALL_TILE_STREAM  the producer warp of the first thread block of a
 *                         brute-force kNN or Ball Query launch never issues
 *                         its first tile's copy (nothing is left in flight):
 *                         the producer and that block's consumers run out
 *                         their waits.
 * Each ends as a real timeout does: PC_ERR_DEVICE_TIMEOUT in the status
 * word, -1 in the outputs the stopped blocks did not finish.
 * pc_debug_set_fps_grid_stall(e) sets or clears PC_STALL_FPS_GRID alone.
 */
#define PC_STALL_FPS_GRID 1
#define PC_STALL_FPS_CLUSTER 2
#define PC_STALL_TILE_STREAM 4
void pc_set_wait_timeout_ns(uint64_t ns);
void pc_debug_set_stall(int mask);
void pc_debug_set_fps_grid_stall(int enable);

/*
 * Concurrency hint: the number of SMs that work running at the same time on
 * another stream occupies (default 0).  The brute-force kNN (one block per
 * SM) and Ball Query (two blocks per SM) size their grids for one wave; with
 * a reserve of n they plan for (SM count - n) SMs (at least 1), so that none
 * of their blocks waits for the other work to finish.
 * Results do not depend on it.  Applies to launches enqueued after the call,
 * on every device; negative values count as 0.
 */
void pc_set_sm_reserve(int sms);

/*
 * FPS of the CLUSTER and two-level GRID schedules in rounds (default on):
 * per exchange between the blocks of a cloud, a run of several centers is
 * certified from each warp's listed points and the bound of its other
 * points (project page, "Farthest point sampling": the same centers as one
 * step at a time); in the grid each cluster first summarizes its blocks'
 * lists.
 * pc_fps_set_batched(0) makes every exchange take one center, 1 restores
 * the rounds; applies to launches enqueued after the call on every device.
 * Returns the previous setting.
 */
int pc_fps_set_batched(int enable);

/* The number of SMs an FPS launch of these sizes occupies while it runs (its
 * resident thread blocks, at most the SM count), or 0 when the sizes have no
 * schedule or there is no device.  npoint does not change it. */
int pc_fps_sm_count(int64_t B, int64_t N, int64_t npoint);

#ifdef __cplusplus
}
#endif

#endif /* POINTCLOUD_H */
