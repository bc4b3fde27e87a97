/*
 * FP64 CPU oracle for the all-pairs softened-gravity acceleration and the
 * leapfrog kick/drift step that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  The GPU library never links, loads or calls this
 * file, and shares no source with it.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it.
 *
 * It is deliberately plain: an outer loop over target bodies i and an inner
 * loop over source bodies j in ascending order, every operation in IEEE
 * double, no blocking and no reordering.  It is built with
 * -ffp-contract=off, so no multiply-add is fused and results are the same on
 * every host.  OpenMP splits only the independent outer loop.
 *
 * Sources (page, section):
 *   "CUDA N-Body Simulation" (LienoPC/N-BodySimulation README)
 *     §1.2 Gravitational Softening: the softened sum over all j with G = 1,
 *          r_ij = x_j - x_i, and the remark that the self term is zero.
 *     §1.3 Numerical Time Integration: the half-step velocity kick with
 *          a(x(t)) followed by the full-step drift with the kicked velocity;
 *          accelerations come from the coordinates at the start of the step.
 *          The same section names the scheme a staggered leapfrog; its
 *          textbook closed form (kick-drift-kick) adds the second half-kick
 *          with a(x(t + dt)) and is given as oracle_leapfrog_kdk.
 *   "Cuda Nbody Notes": the per-pair interaction (r, |r|^2 + eps^2, the
 *          inverse 3/2 power, the mass factor, the accumulation).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of OpenMP threads a call with `requested` threads would use. */
int oracle_threads(int requested)
{
#ifdef _OPENMP
    return requested > 0 ? requested : omp_get_max_threads();
#else
    (void)requested;
    return 1;
#endif
}

/*
 * Softened acceleration on one target body i, G = 1:
 *   a_i = sum_{j=0}^{n-1} m_j (x_j - x_i) / (|x_j - x_i|^2 + eps2)^(3/2)
 * ("CUDA N-Body Simulation" §1.2).  The j = i term has r = 0 and adds exactly
 * zero while eps2 > 0.  pos_mass rows are (x, y, z, m).
 */
static void accel_of_body(const double *pm, int64_t n, double eps2, int64_t i,
                          double a[3])
{
    const double xi = pm[4 * i + 0];
    const double yi = pm[4 * i + 1];
    const double zi = pm[4 * i + 2];
    double ax = 0.0, ay = 0.0, az = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double rx = pm[4 * j + 0] - xi;
        const double ry = pm[4 * j + 1] - yi;
        const double rz = pm[4 * j + 2] - zi;
        const double d = rx * rx + ry * ry + rz * rz + eps2;
        const double w = pm[4 * j + 3] / (d * sqrt(d));
        ax += w * rx;
        ay += w * ry;
        az += w * rz;
    }
    a[0] = ax;
    a[1] = ay;
    a[2] = az;
}

/*
 * Accelerations of the bodies listed in idx[0..n_idx) (all n bodies in order
 * when idx is NULL, in which case n_idx must equal n), each summed over every
 * one of the n source bodies.  acc is n_idx rows of (ax, ay, az).
 * Returns the number of threads used, or -1 on a bad argument.
 */
int oracle_accel(const double *pos_mass, int64_t n, double eps2,
                 const int64_t *idx, int64_t n_idx, double *acc, int threads)
{
    if (n < 0 || n_idx < 0 || (idx == NULL && n_idx != n))
        return -1;
    if (n_idx > 0 && (pos_mass == NULL || acc == NULL))
        return -1;
    if (idx != NULL)
        for (int64_t k = 0; k < n_idx; ++k)
            if (idx[k] < 0 || idx[k] >= n)
                return -1;
    const int nt = oracle_threads(threads);
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
    for (int64_t k = 0; k < n_idx; ++k) {
        const int64_t i = idx ? idx[k] : k;
        accel_of_body(pos_mass, n, eps2, i, acc + 3 * k);
    }
    return nt;
}

/*
 * `steps` leapfrog kick/drift steps in place ("CUDA N-Body Simulation" §1.3):
 *   for every body:  a_i = A_i(x(t))           (all from the same x(t))
 *   then for every body:
 *       v_i <- v_i + (dt/2) a_i
 *       x_i <- x_i + dt v_i
 * Masses (pos_mass column 3) are never changed.  pos_mass is n rows of
 * (x, y, z, m), vel n rows of (vx, vy, vz), acc n rows of (ax, ay, az); on
 * return acc holds the accelerations of the last step, i.e. at the positions
 * before its drift.  Returns the number of threads used, or -1 on a bad
 * argument.
 */
int oracle_leapfrog(double *pos_mass, double *vel, double *acc, int64_t n,
                    double eps2, double dt, int steps, int threads)
{
    if (n < 0 || steps < 0)
        return -1;
    if (n > 0 && (pos_mass == NULL || vel == NULL || acc == NULL))
        return -1;
    const int nt = oracle_threads(threads);
    for (int s = 0; s < steps; ++s) {
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
        for (int64_t i = 0; i < n; ++i)
            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t i = 0; i < n; ++i) {
            for (int c = 0; c < 3; ++c) {
                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];
                pos_mass[4 * i + c] = pos_mass[4 * i + c] + dt * vel[3 * i + c];
            }
        }
    }
    return nt;
}

/*
 * One step of oracle_leapfrog for the bodies idx[0..m) only ("CUDA N-Body
 * Simulation" §1.3): a_i = A_i(x(t)) over all n sources, then
 *     v_i <- v_i + (dt/2) a_i,   x_i <- x_i + dt v_i.
 * A body's step needs only its own acceleration, so each row equals the
 * full step's.  pos_mass: n rows (x, y, z, m), vel: n rows (vx, vy, vz);
 * pos_out m rows (x, y, z, m), vel_out and acc_out m rows of 3.  Returns
 * the threads used, or -1 on a bad argument.
 */
int oracle_step_sampled(const double *pos_mass, const double *vel, int64_t n, double eps2,
                        double dt, const int64_t *idx, int64_t m, double *pos_out,
                        double *vel_out, double *acc_out, int threads)
{
    if (n < 0 || m < 0 || (m > 0 && (idx == NULL || pos_mass == NULL || vel == NULL ||
                                     pos_out == NULL || vel_out == NULL || acc_out == NULL)))
        return -1;
    const int nt = oracle_accel(pos_mass, n, eps2, idx, m, acc_out, threads);
    if (nt < 0)
        return -1;
    for (int64_t k = 0; k < m; ++k) {
        const int64_t i = idx[k];
        for (int c = 0; c < 3; ++c) {
            vel_out[3 * k + c] = vel[3 * i + c] + 0.5 * dt * acc_out[3 * k + c];
            pos_out[4 * k + c] = pos_mass[4 * i + c] + dt * vel_out[3 * k + c];
        }
        pos_out[4 * k + 3] = pos_mass[4 * i + 3];
    }
    return nt;
}

/*
 * `steps` kick-drift-kick leapfrog steps in place, the closed form of the
 * staggered leapfrog named in "CUDA N-Body Simulation" §1.3:
 *   a = A(x(t))                       (once, before the first step)
 *   per step, for every body:
 *       v_i <- v_i + (dt/2) a_i       half kick with a(x(t))
 *       x_i <- x_i + dt v_i           drift
 *   then a = A(x(t + dt)) for every body, and for every body:
 *       v_i <- v_i + (dt/2) a_i       half kick with a(x(t + dt))
 * steps + 1 evaluations of A.  On return acc holds A at the final positions
 * (untouched when steps is 0).  Returns the threads used or -1.
 */
int oracle_leapfrog_kdk(double *pos_mass, double *vel, double *acc, int64_t n,
                        double eps2, double dt, int steps, int threads)
{
    if (n < 0 || steps < 0)
        return -1;
    if (n > 0 && (pos_mass == NULL || vel == NULL || acc == NULL))
        return -1;
    const int nt = oracle_threads(threads);
    if (steps == 0)
        return nt;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
    for (int64_t i = 0; i < n; ++i)
        accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);
    for (int s = 0; s < steps; ++s) {
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t i = 0; i < n; ++i) {
            for (int c = 0; c < 3; ++c) {
                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];
                pos_mass[4 * i + c] = pos_mass[4 * i + c] + dt * vel[3 * i + c];
            }
        }
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
        for (int64_t i = 0; i < n; ++i)
            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t i = 0; i < n; ++i)
            for (int c = 0; c < 3; ++c)
                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];
    }
    return nt;
}

/*
 * CPU restatement of the point shaders of "CUDA N-Body Simulation" §4.3
 * (GLSL Shader Pipeline and Mass-Normalized Color Mapping), per body:
 *   vertex:   weight = (m - min_w) / (max_w - min_w)
 *             p_c    = 2 (c - (-max_c)) / (max_c - (-max_c)) - 1,  c = x, y, z
 *             ndc    = (p_x, p_y, p_z, 1)
 *   fragment: colour = mix(green, red, weight), GLSL mix(a, b, t) = a (1-t) + b t,
 *             green = (0, 1, 0), red = (1, 0, 0); rgba = (colour, 1)
 * No clamping: the shaders apply none.  ndc and rgba are n rows of 4 doubles.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_render_points(const double *pos_mass, int64_t n, double max_x, double max_y,
                         double max_z, double min_w, double max_w, double *ndc, double *rgba)
{
    if (n < 0 || (n > 0 && (pos_mass == NULL || ndc == NULL || rgba == NULL)))
        return -1;
    const double lim[3] = {max_x, max_y, max_z};
    const double green[3] = {0.0, 1.0, 0.0};
    const double red[3] = {1.0, 0.0, 0.0};
    for (int64_t i = 0; i < n; ++i) {
        const double weight = (pos_mass[4 * i + 3] - min_w) / (max_w - min_w);
        for (int c = 0; c < 3; ++c) {
            ndc[4 * i + c] = 2.0 * (pos_mass[4 * i + c] - (-lim[c])) / (lim[c] - (-lim[c])) - 1.0;
            rgba[4 * i + c] = green[c] * (1.0 - weight) + red[c] * weight;
        }
        ndc[4 * i + 3] = 1.0;
        rgba[4 * i + 3] = 1.0;
    }
    return 0;
}

/*
 * 2-D cutoff neighbour list, all pairs, without atomics ("CUDA编程（九）原子函数
 * 的合理使用" §3, the neighbour-list example: the version that tests every pair
 * (n1, n2), n2 != n1, and writes only the lists of n1).  In the page's single
 * precision: x12 = x[n2] - x[n1], y12 = y[n2] - y[n1],
 * d2 = x12 * x12 + y12 * y12, neighbour when d2 < cutoff * cutoff (all float,
 * every operation rounded separately: this file is built with
 * -ffp-contract=off).  nn[n1] = number of neighbours; nl[k * n + n1] = the
 * k-th neighbour in ascending index order for k < min(nn[n1], mn), -1 for the
 * remaining k < mn (the page's transposed layout).  With idx, only the
 * targets idx[0..n_idx) are listed (row k of nl then has n_idx entries);
 * idx NULL means all n targets in order.  Returns 0 or -1.
 */
int oracle_neighbors_2d(const float *x, const float *y, int64_t n, float cutoff, int mn,
                        const int64_t *idx, int64_t n_idx, int32_t *nn, int32_t *nl,
                        int threads)
{
    if (n < 0 || mn < 0 || n_idx < 0 || (idx == NULL && n_idx != n))
        return -1;
    if (n_idx > 0 && (x == NULL || y == NULL || nn == NULL || (mn > 0 && nl == NULL)))
        return -1;
    if (idx != NULL)
        for (int64_t k = 0; k < n_idx; ++k)
            if (idx[k] < 0 || idx[k] >= n)
                return -1;
    const float cutoff_square = cutoff * cutoff;
    const int nt = oracle_threads(threads);
#pragma omp parallel for schedule(dynamic, 64) num_threads(nt)
    for (int64_t k = 0; k < n_idx; ++k) {
        const int64_t n1 = idx ? idx[k] : k;
        const float x1 = x[n1];
        const float y1 = y[n1];
        int32_t count = 0;
        for (int64_t n2 = 0; n2 < n; ++n2) {
            const float x12 = x[n2] - x1;
            const float y12 = y[n2] - y1;
            const float distance_square = x12 * x12 + y12 * y12;
            if (distance_square < cutoff_square && n2 != n1) {
                if (count < mn)
                    nl[(int64_t)count * n_idx + k] = (int32_t)n2;
                ++count;
            }
        }
        nn[k] = count;
        for (int32_t q = count; q < mn; ++q)
            nl[(int64_t)q * n_idx + k] = -1;
    }
    return 0;
}
