/*
 * nbody.h - C ABI of the GB300 (sm_103a) all-pairs softened-gravity library.
 *
 * What it computes
 *   Softened all-pairs acceleration, G = 1 ("CUDA N-Body Simulation",
 *   §1.2 Gravitational Softening, the softened equation):
 *       a_i = sum_{j=0}^{n-1} m_j (x_j - x_i) / (|x_j - x_i|^2 + eps2)^(3/2)
 *   The j = i term is zero because x_i - x_i = 0 while eps2 > 0 (same
 *   section, the remark after bodyInteractions).  One pair costs the 20
 *   conventional FLOP counted in the comments of bodybodyinteraction
 *   ("Cuda Nbody Notes").
 *
 *   Leapfrog kick/drift step ("CUDA N-Body Simulation", §1.3 Numerical Time
 *   Integration, the two update equations):
 *       a_i = A_i(x(t))                 for every body, from the same x(t)
 *       v_i <- v_i + (dt/2) a_i         half-step velocity kick
 *       x_i <- x_i + dt v_i             full-step drift with the kicked v
 *   The section keeps the kicked velocity across launches and shows no
 *   closing half-kick; a step here is exactly the two updates above.
 *
 * Data layout (all arrays are float4 rows, 16-byte aligned, row i = body i;
 * "CUDA N-Body Simulation" §2.2 Data Structures and Memory Alignment):
 *   pos_mass  (x, y, z, m)      FP32; m is never modified.
 *   vel       (vx, vy, vz, w)   FP32; w is never read or modified.
 *   accel     (ax, ay, az, 0)   FP32; written, w set to 0
 *                               ("Cuda Nbody Notes", calculate_forces).
 *
 * Pointers are DEVICE pointers on the calling thread's current CUDA device
 * (cudaMalloc / cudaMallocAsync / managed memory); host pointers are
 * rejected with NBODY_EINVAL.  The caller owns every array it passes.  The
 * library owns only what it keeps per (device, stream): a status word and
 * its cached scratch (the second buffer of the positions where one kernel
 * both reads and drifts them, the split-j partial sums and the pair path's
 * action and reaction sums).  Both
 * come from stream-ordered allocation (cudaMallocAsync on the call's stream)
 * on the stream's first use and when a larger call needs more, and are
 * freed by nbody_release().
 *
 * Execution is asynchronous: a call validates its arguments, enqueues its
 * kernels on the stream and returns.  NBODY_OK means "enqueued"; a device
 * side failure (a bounded wait that expired) is recorded in the stream's
 * status word and reported by nbody_sync() on that stream.  Results are
 * bitwise deterministic for a given (n, path, split, device model, library
 * build): every sum runs in a fixed order and no atomics take part in any
 * reduction.  Calls on different streams use different scratch and status
 * words and may run concurrently; the caller orders calls that share a
 * stream, as usual.  Within a call, each kernel is launched as a
 * programmatic dependent of the library kernel before it on the stream: its
 * launch overlaps that kernel's last CTAs, and it waits for that kernel to
 * complete before it touches memory.  The library's kernels allow their
 * dependents' launch as they start, so a kernel of the caller's that is
 * itself launched with programmatic stream serialization right after a call
 * must wait for its prerequisite grid (cudaGridDependencySynchronize)
 * before it reads the call's outputs; any other work enqueued after a call
 * is ordered as for any stream.
 *
 * Errors (every entry point returns one of these codes):
 *   NBODY_EINVAL    n < 0 or n > 2^31-1; eps2 not finite or <= 0; dt not
 *                   finite; steps < 0; a NULL, misaligned (not 16-byte) or
 *                   non-device pointer; accel overlapping pos_mass or vel;
 *                   pos_mass overlapping vel; unknown path; split < 0.
 *                   Nothing is enqueued.
 *   NBODY_ENOMEM    scratch allocation failed.  Nothing is enqueued.
 *   NBODY_ECUDA     no usable CUDA device, or a launch failed.
 *   NBODY_ETIMEOUT  (nbody_sync only) a kernel's bounded wait for a tile
 *                   copy expired; the kernel stopped and its outputs are
 *                   undefined.  The CUDA context stays usable.
 *   NBODY_EBOUNDS   (nbody_sync only, index-checked builds only) an index
 *                   into a scratch or output array fell outside what the
 *                   host allocated; the access was skipped, the outputs are
 *                   undefined.  The release build has no such checks.
 *   n == 0 and steps == 0 are valid no-ops that return NBODY_OK.
 *
 * Positions, masses and velocities are not checked: a non-finite value
 * gives non-finite results for every body whose sum it enters (all of them,
 * for a non-finite source), as in the pages' kernels.  Zero and negative
 * masses are valid.
 */
#ifndef NBODY_H
#define NBODY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nbody_status {
    NBODY_OK = 0,
    NBODY_EINVAL = 1,
    NBODY_ENOMEM = 2,
    NBODY_ECUDA = 3,
    NBODY_ETIMEOUT = 4,
    /* Index-checked builds only (compiled with NBODY_BOUNDS_CHECK): a
       device-side index check failed and the access was skipped. */
    NBODY_EBOUNDS = 5
} nbody_status;

/* Force-pass path for the *_with entry points. */
typedef enum nbody_path {
    /* Library's choice: the warp-split kernel below n = 16384, the
       pair-symmetric kernel from there on (NBODY_PATH_PAIRS); the one-sided
       tiled kernel with its (i-block, j-tile) units divided evenly over one
       wave of CTAs (stream-K) if the pair path's scratch cannot be
       allocated. */
    NBODY_PATH_AUTO = 0,
    /* One CTA per i-block over the whole j range; no second pass.  The
       pages' tiled design ("CUDA N-Body Simulation" §3.1). */
    NBODY_PATH_TILED = 1,
    /* The j range of every i-block is cut into `split` slices handled by
       different CTAs; a second pass sums the slices in fixed order
       ("CUDA N-Body Simulation" §3.2-3.3, without the N x N matrix). */
    NBODY_PATH_SPLIT = 2,
    /* Small-n kernel: the 32 lanes of a warp share target bodies and
       stride over sources; lanes combine by warp shuffles, warps through
       shared memory in fixed order, CTAs through the second pass. */
    NBODY_PATH_WARP = 3,
    /* Pair-symmetric tiled kernel: every pair of bodies in different
       i-blocks is evaluated once and serves both bodies (Newton's third
       law: the term body i adds to a_j is the negative of the one body j
       adds to a_i with m_j replaced by m_i, bit for bit in FP32), about 2/3
       of the FP32 work of the one-sided paths.  The reactions on a tile's
       sources are summed over the CTA's targets in fixed order and stored
       per (i-block, tile) unit; the second pass adds them to the action in
       block order.  Scratch: about 8 n^2 / B bytes of reaction sums for B
       targets per i-block (2.1 to 2.5 GB at n = 2^20); where that exceeds
       1 GiB (or NBODY_PAIRS_MAX_BYTES) the pass runs in chunks of
       consecutive i-blocks whose sums fit, each chunk's sums folded into a
       per-body accumulator (16 B per body) before the next chunk (two more
       launches per chunk, one at the end).  AUTO takes this path from
       n = 16384 on, and falls back to NBODY_PATH_SPLIT's plan if its
       scratch cannot be allocated; nbody_last_plan tells which ran. */
    NBODY_PATH_PAIRS = 4
} nbody_path;

/*
 * accel[i] = (a_i, 0) for every i < n, a_i as defined above.
 *   pos_mass  in   n rows (x, y, z, m); only read.
 *   accel     out  n rows; must not overlap pos_mass.
 *   n         number of bodies, 0 <= n <= 2^31 - 1.
 *   eps2      softening length squared, finite and > 0.
 * Enqueued on the legacy default stream.
 */
int nbody_accel(const float *pos_mass, float *accel, int64_t n, float eps2);

/* nbody_accel on an explicit stream (a cudaStream_t; NULL = legacy stream). */
int nbody_accel_on_stream(const float *pos_mass, float *accel, int64_t n,
                          float eps2, void *cuda_stream);

/*
 * `steps` leapfrog kick/drift steps, updated in place from the caller's
 * point of view.
 *   pos_mass  in/out  n rows; xyz advanced, m unchanged.
 *   vel       in/out  n rows; xyz kicked, w unchanged.
 *   accel     out     n rows; the accelerations of the last step, i.e. at
 *                     the positions before its drift (w = 0).
 *   eps2, dt          finite; eps2 > 0.  steps >= 0.
 * Within a step every acceleration uses the start-of-step positions (the
 * new positions go to a second buffer), so no body sees a half-updated
 * neighbour.
 */
int nbody_leapfrog_step(float *pos_mass, float *vel, float *accel, int64_t n,
                        float eps2, float dt, int steps);

int nbody_leapfrog_step_on_stream(float *pos_mass, float *vel, float *accel,
                                  int64_t n, float eps2, float dt, int steps,
                                  void *cuda_stream);

/*
 * The two calls above with an explicit force-pass path (nbody_path) and,
 * for NBODY_PATH_SPLIT / NBODY_PATH_WARP, the number of j slices per
 * i-block (`split` = 0 lets the library choose).  Every path computes the
 * same sums in a different fixed order.
 */
int nbody_accel_with(const float *pos_mass, float *accel, int64_t n,
                     float eps2, int path, int split, void *cuda_stream);

int nbody_leapfrog_step_with(float *pos_mass, float *vel, float *accel,
                             int64_t n, float eps2, float dt, int steps,
                             int path, int split, void *cuda_stream);

/*
 * `steps` kick-drift-kick leapfrog steps: per step
 *     v <- v + (dt/2) a(x(t));  x <- x + dt v;  v <- v + (dt/2) a(x(t + dt)),
 * the closed, time-symmetric form of the staggered leapfrog that
 * "CUDA N-Body Simulation" §1.3 names (the pages' own step, above, stops
 * after the drift).  The closing half kick of each step is fused with the
 * opening half kick of the next, so a call costs steps + 1 force passes.
 *   pos_mass, vel  in/out as for nbody_leapfrog_step.
 *   accel          out: the accelerations at the final positions.
 * Arguments, errors and paths as for nbody_leapfrog_step_with.
 */
int nbody_leapfrog_kdk_on_stream(float *pos_mass, float *vel, float *accel,
                                 int64_t n, float eps2, float dt, int steps,
                                 void *cuda_stream);

int nbody_leapfrog_kdk_with(float *pos_mass, float *vel, float *accel,
                            int64_t n, float eps2, float dt, int steps,
                            int path, int split, void *cuda_stream);

/*
 * The point shaders of "CUDA N-Body Simulation" §4.3 (vertex and fragment
 * shader of the mass-coloured GL_POINTS view) as a kernel writing into
 * device buffers, for use without any graphics API:
 *   ndc[i]  = (p_x, p_y, p_z, 1),  p_c = 2 (c - (-max_c)) / (max_c - (-max_c)) - 1
 *   rgba[i] = (w, 1 - w, 0, 1),    w = (m - min_w) / (max_w - min_w),
 * i.e. GLSL mix(green, red, w); nothing is clamped, as in the shaders.
 *   pos_mass   in   n rows (x, y, z, m).
 *   ndc, rgba  out  n float4 rows each; must not overlap each other or pos_mass.
 *   max_x, max_y, max_z  finite, > 0 (the view box half-widths).
 *   min_w, max_w         finite, max_w > min_w (the mass range).
 * Errors as for nbody_accel; n == 0 is a no-op.
 */
int nbody_render_points(const float *pos_mass, float *ndc, float *rgba,
                        int64_t n, float max_x, float max_y, float max_z,
                        float min_w, float max_w, void *cuda_stream);

/*
 * 2-D cutoff neighbour list over all pairs, without atomics: the neighbour-
 * list example of "CUDA编程（九）原子函数的合理使用" §3 in its atomic-free form
 * (every pair (i, j), j != i, tested by the thread of i, which alone writes
 * the list of i).  In single precision, each operation rounded separately:
 *     x12 = x[j] - x[i], y12 = y[j] - y[i], d2 = x12*x12 + y12*y12,
 *     j is a neighbour of i when d2 < cutoff*cutoff (cutoff*cutoff rounded
 *     to float).
 *   x, y    in   n floats each (4-byte aligned device arrays).
 *   nn      out  n int32: number of neighbours of each point (not capped).
 *   nl      out  max_neighbors * n int32, transposed as on the page:
 *                nl[k * n + i] = k-th neighbour of i in ascending index
 *                order for k < min(nn[i], max_neighbors), -1 for the other
 *                k < max_neighbors.  nn[i] > max_neighbors means the list of
 *                i was truncated.  May be NULL when max_neighbors == 0.
 *   cutoff  finite, > 0, with cutoff*cutoff a normal float.
 * nn and nl must not overlap each other or x, y.  Errors as for
 * nbody_accel; n == 0 is a no-op.  Deterministic: no atomics.
 */
int nbody_neighbors_2d(const float *x, const float *y, int64_t n, float cutoff,
                       int max_neighbors, int32_t *nn, int32_t *nl,
                       void *cuda_stream);

/*
 * Layouts of the velocity and acceleration arrays for the *_layout entry
 * points ("CUDA N-Body Simulation" §3.5 compares float4 and float3 forms).
 * Positions stay float4 rows (x, y, z, m) in every layout.
 */
typedef enum nbody_layout {
    NBODY_ROWS4 = 0,   /* n rows of float4; accel.w = 0, vel.w kept; 16-byte aligned */
    NBODY_ROWS3 = 1,   /* n rows of 3 floats (12 bytes); 4-byte aligned */
    NBODY_BLOCKS3 = 2  /* x[0..n), then y[0..n), then z[0..n); 4-byte aligned */
} nbody_layout;

/*
 * nbody_accel_on_stream writing accel in `layout` (12n bytes for the
 * three-float layouts).  Same accelerations, bit for bit, as NBODY_ROWS4.
 */
int nbody_accel_layout(const float *pos_mass, float *accel, int64_t n,
                       float eps2, int layout, void *cuda_stream);

/*
 * nbody_leapfrog_step_on_stream with vel and accel in `layout`.  Same
 * results, bit for bit, as NBODY_ROWS4 (apart from the w column, which the
 * three-float layouts do not have).
 */
int nbody_leapfrog_step_layout(float *pos_mass, float *vel, float *accel,
                               int64_t n, float eps2, float dt, int steps,
                               int layout, void *cuda_stream);

/*
 * Wait for the stream, then report and clear its status word: NBODY_OK,
 * NBODY_ETIMEOUT (or NBODY_EBOUNDS in the checked build) if a kernel this
 * library enqueued on that stream recorded a failure since the last
 * nbody_sync on it, or NBODY_ECUDA if the stream reported a CUDA error.
 * Failures of kernels on other streams are not reported here.  The status
 * of nbody_accel_noalloc, whose calls share one status word per device, is
 * reported on the stream of its last call.  Call it with the stream's
 * device current.
 */
int nbody_sync(void *cuda_stream);

/*
 * The plan of the last force pass this library enqueued on the stream (the
 * fields of nbody_plan), which differs from nbody_plan's answer where AUTO
 * chose the pair path and its scratch could not be allocated: the call then
 * ran NBODY_PATH_SPLIT's one-sided plan.  Returns NBODY_EINVAL if no force
 * pass has run on the stream (since nbody_release).  Needs the stream's
 * device current.
 */
int nbody_last_plan(void *cuda_stream, int64_t *out, int len);

/*
 * Largest n that nbody_accel_noalloc accepts.
 */
#define NBODY_NOALLOC_MAX_N 65536

/*
 * nbody_accel without any memory allocation (the paper has no counterpart;
 * this entry point exists for callers of this library).
 *
 * Some callers cannot allocate GPU memory at the point where they need the
 * accelerations: hosts that hand every byte of device memory to their own
 * pool and forbid other allocations, and real-time or certified loops that
 * ban allocation after start-up because cudaMalloc may block or synchronise
 * the device.  This call computes the same accelerations as
 * nbody_accel_on_stream, with the same argument rules, but keeps its
 * working memory (the split-j partial sums, and a status word for its
 * bounded waits) in fixed arrays that the library holds on every GPU that
 * loads it, until the process exits: 6 MiB of device memory.  It calls no
 * allocation routine of CUDA, PyTorch or the C/C++ runtime.
 *
 *   n must be <= NBODY_NOALLOC_MAX_N; larger n returns NBODY_EINVAL and
 *   enqueues nothing.  All other arguments as for nbody_accel_on_stream.
 *
 * The first call on a device looks up that device's copy of the arrays
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture.  All calls on a device share the arrays, which
 * keep whatever the last call left in them; every call writes each slot it
 * reads before reading it, so nothing needs clearing.  Two calls whose
 * kernels overlap on the same GPU (for example on two streams without
 * ordering between them) race on the arrays and give wrong results; order
 * them (same stream, or an event).  nbody_sync on the stream of the last
 * call reports an expired wait of these calls.
 */
int nbody_accel_noalloc(const float *pos_mass, float *accel, int64_t n,
                        float eps2, void *cuda_stream);

/*
 * Describe the launch plan a force pass over n bodies would use on the
 * current device.  out[0..len) receives, as far as len allows:
 *   [0] path actually used (nbody_path value)   [1] grid (CTAs)
 *   [2] threads per CTA                         [3] target bodies per CTA
 *   [4] source bodies per tile                  [5] tiles over n
 *   [6] work units (i-blocks x tiles; for NBODY_PATH_PAIRS the (i-block,
 *       tile) units from each block's own first tile on)
 *   [7] 1 if a second pass runs
 *   [8] kernel launches of one nbody_accel call (pair path in chunks:
 *       2 per chunk + 1)
 *   [9] kernel launches of one nbody_leapfrog_step call with steps = 1
 *  [10] streaming multiprocessors on the device
 *  [11] bytes of reaction sums the pair path keeps (0 on the other paths)
 *  [12] chunks of i-blocks the pair pass runs in (1 on the other paths)
 * This is the plan before any scratch is allocated; see nbody_last_plan.
 * Returns NBODY_OK, NBODY_EINVAL or NBODY_ECUDA.
 */
int nbody_plan(int64_t n, int path, int split, int64_t *out, int len);

/*
 * Rows of this build's kernel tables (for tests and tuning sweeps; the
 * NBODY_TILED_CONFIG / NBODY_PAIRS_CONFIG / NBODY_WARP_CONFIG environment
 * variables select a row by its index).  which = 0: the one-sided tiled
 * kernel, 1: the pair-symmetric kernel, 2: the small-n warp kernel.
 * out[0..len) receives, as far as len allows:
 *   [0] rows in the table
 *   [1] target bodies per thread (warp kernel: per CTA)
 *   [2] threads per CTA
 *   [3] sources per tile (warp kernel: sources each thread loads ahead)
 *   [4] tiled: 1 for the mixed rsqrt/logarithmic loop; pairs: 1 for running
 *       sums in shared memory; warp kernel: 1 for lanes combined by a
 *       reduce-scatter, 0 for a butterfly
 *   [5] pairs: the reaction scheme (0 warp butterfly over batches, 1 and 2
 *       lane rotation with one or two groups, 3 and 4 the same with loads one
 *       step ahead, scalar carries and duplicated groups); others: 0.
 * The release build holds only the rows its plans use; the tuning build
 * (compiled with NBODY_TUNING_TABLE) appends the others.  Needs no device.
 * Returns NBODY_OK or NBODY_EINVAL (unknown table or row).
 */
int nbody_table(int which, int row, int64_t *out, int len);

/*
 * Measurement hooks.  Every kernel launch of the library is counted.  While
 * enabled (nonzero), every force-kernel launch is also bracketed by a pair
 * of CUDA events recorded on its own stream (which costs host time per
 * launch: time calls with profiling off, and the force kernels in a
 * separate profiled run).  nbody_profile_read waits for the recorded events
 * and returns, since the last read, the summed force-kernel time in
 * milliseconds, the number of force-kernel launches and the number of all
 * kernel launches; then it starts a new interval.  Any output pointer may
 * be NULL.  Not thread-safe with concurrent calls on other host threads.
 */
int nbody_profile_enable(int enable);
int nbody_profile_read(double *force_ms, int64_t *force_launches,
                       int64_t *kernel_launches);

/*
 * Phase clocks of the pair-symmetric kernel, in the profiling build only
 * (compiled with NBODY_PHASE_CLOCKS; build(phases=True)): waits for the
 * device, then returns and clears the SM cycles its warps spent, summed over
 * every warp of every launch since the last read, in out[0..len):
 *   [0] the tile copy's wait and the first CTA barrier
 *   [1] issuing the next copy, expanding the tile, the second barrier
 *   [2] the arithmetic of tiles of a CTA's own i-block
 *   [3] the arithmetic of the other tiles (the lane rotation and reaction rows)
 *   [4] the third barrier, the warps' reaction sums and the row's store
 *   [5] folding the per-tile sums into the running sums
 *   [6] everything else (target loads, segment epilogues, set-up)
 * Other builds return NBODY_EINVAL.
 */
int nbody_phase_read(int64_t *out, int len);

/* Text of a status code (static storage; never NULL). */
const char *nbody_strerror(int status);

/* Free all cached scratch on every device (synchronises those devices). */
void nbody_release(void);

/*
 * Failure-detection check: runs the one-sided tiled kernel and the pair
 * kernel, each on a tiny private problem with its first tile copy
 * deliberately never issued and a wait limit of `timeout_ms`, calling
 * nbody_sync on the stream after each.  A correct build returns
 * NBODY_ETIMEOUT (both kernels gave up and returned; the context stays
 * usable); otherwise the first other status.  Its buffers are the stream's
 * scratch.
 */
int nbody_selftest_timeout(int timeout_ms, void *cuda_stream);

/*
 * The same two kernels enqueued on the stream without waiting: their
 * expired waits stay in that stream's status word until nbody_sync on it
 * (NBODY_ETIMEOUT once both have run).  Returns NBODY_OK when enqueued.
 */
int nbody_selftest_timeout_enqueue(int timeout_ms, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* NBODY_H */
