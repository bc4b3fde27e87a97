/*
 * A C client of the library, using nothing but nbody.h and the CUDA runtime.
 *
 * Two bodies on the x axis, r = 1.5 apart, masses 2 and 0.5, eps2 = 0.01.
 * The softened law ("CUDA N-Body Simulation", §1.2) gives in closed form
 *   a_0 = +m_1 r / (r^2 + eps2)^(3/2) x,   a_1 = -m_0 r / (r^2 + eps2)^(3/2) x.
 * Then one leapfrog step from rest (§1.3: half kick, then drift) with dt = 0.1
 * must give v = dt/2 a_0 and x = x_0 + dt v for each body.
 * Exit status 0 when every check holds; a message and 1 otherwise.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "nbody.h"

static int fail(const char *what) {
  fprintf(stderr, "two_bodies: %s\n", what);
  return 1;
}

/* |got - want| <= tol |want| */
static int close_to(double got, double want, double tol) {
  return fabs(got - want) <= tol * fabs(want);
}

int main(void) {
  const float pm[8] = {0.0f, 0.0f, 0.0f, 2.0f, 1.5f, 0.0f, 0.0f, 0.5f};
  const float eps2 = 0.01f, dt = 0.1f;
  const size_t bytes = sizeof pm;
  float acc[8], vel[8], pos[8];
  float *d_pm = NULL, *d_acc = NULL, *d_vel = NULL;
  int rc;

  if (cudaMalloc((void **)&d_pm, bytes) != cudaSuccess ||
      cudaMalloc((void **)&d_acc, bytes) != cudaSuccess ||
      cudaMalloc((void **)&d_vel, bytes) != cudaSuccess)
    return fail("cudaMalloc failed");
  if (cudaMemcpy(d_pm, pm, bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(d_vel, 0, bytes) != cudaSuccess)
    return fail("upload failed");

  /* accelerations */
  rc = nbody_accel(d_pm, d_acc, 2, eps2);
  if (rc != NBODY_OK) return fail(nbody_strerror(rc));
  rc = nbody_sync(NULL);
  if (rc != NBODY_OK) return fail(nbody_strerror(rc));
  if (cudaMemcpy(acc, d_acc, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail("download failed");
  {
    const double r = 1.5, d = r * r + (double)eps2;
    const double f = r / (d * sqrt(d));
    if (!close_to(acc[0], 0.5 * f, 1e-5) || !close_to(acc[4], -2.0 * f, 1e-5))
      return fail("accelerations differ from the closed form");
    if (acc[1] != 0.0f || acc[2] != 0.0f || acc[5] != 0.0f || acc[6] != 0.0f ||
        acc[3] != 0.0f || acc[7] != 0.0f)
      return fail("y, z or w of an acceleration is not zero");
  }

  /* one leapfrog step from rest, in place on d_pm and d_vel */
  rc = nbody_leapfrog_step(d_pm, d_vel, d_acc, 2, eps2, dt, 1);
  if (rc != NBODY_OK) return fail(nbody_strerror(rc));
  rc = nbody_sync(NULL);
  if (rc != NBODY_OK) return fail(nbody_strerror(rc));
  if (cudaMemcpy(vel, d_vel, bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(pos, d_pm, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail("download failed");
  for (int b = 0; b < 2; ++b) {
    const double v = 0.5 * dt * (double)acc[4 * b];
    if (!close_to(vel[4 * b], v, 1e-6)) return fail("velocity after one step");
    if (!close_to(pos[4 * b], (double)pm[4 * b] + dt * v, 1e-5))
      return fail("position after one step");
    if (pos[4 * b + 3] != pm[4 * b + 3]) return fail("the drift changed a mass");
  }

  /* invalid arguments come back as NBODY_EINVAL, nothing launched */
  if (nbody_accel(d_pm, d_acc, -1, eps2) != NBODY_EINVAL) return fail("n < 0 accepted");
  if (nbody_accel(d_pm, d_acc, 2, 0.0f) != NBODY_EINVAL) return fail("eps2 = 0 accepted");

  nbody_release();
  cudaFree(d_pm);
  cudaFree(d_acc);
  cudaFree(d_vel);
  printf("two_bodies: ok (a_0 = %.9g, a_1 = %.9g)\n", acc[0], acc[4]);
  return 0;
}
