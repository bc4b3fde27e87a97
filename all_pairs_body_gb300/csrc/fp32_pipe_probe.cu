// Calibration of the FP32 (FMA) pipe on this GPU, for reading the force
// kernels' roofline fractions.  One CTA of 256 threads per SM (two warps per
// scheduler, as in the pair-symmetric kernel) runs a fixed instruction mix;
// each CTA times itself with clock64 and the program prints the FP32 lane
// operations retired per SM cycle as a fraction of the nominal 128.
//
//   ffma2, fresh operands  packed FMAs whose three operands all differ from
//                          the previous instruction's
//   ffma2, shared operand  packed FMAs that repeat one operand of the
//                          previous instruction in the same position
//   ffma, fresh operands   scalar FMAs, all operands different
//   pair step             the pair-symmetric kernel's steady state: sources
//                          rotated through the lanes from a duplicated-group
//                          shared-memory tile, loads one step ahead, a scalar
//                          carry per component, 8 packed target pairs, its
//                          interaction (interact2_pair) unchanged
//   pair step, u form     the same loop with the interaction's products
//                          regrouped: u = q^3 r first, then the action m_j u
//                          and the reaction m_i u (17 packed instructions
//                          instead of 16, but the source mass, the target
//                          mass and q^3 each repeat in three consecutive
//                          instructions)
//
// Build and run: python -m all_pairs_body_gb300.build --probe
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "nbody_kernels.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 512;  // sources of the pair-step tile

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) ffma_stream(float* out, long long* cycles, int iters,
                                                          float seed) {
  float2 a[16], b[16], acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    a[k] = make_float2(seed * (k + 1) + threadIdx.x * 1e-6f, seed * (k + 2));
    b[k] = make_float2(0.999f - 1e-4f * k, 0.998f + 1e-5f * k);
    acc[k] = make_float2(0.f, 0.f);
  }
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll 4
    for (int r = 0; r < 8; ++r) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (MODE == 0) {
          acc[k] = __ffma2_rn(a[k], b[k], acc[k]);
        } else if (MODE == 1) {
          acc[k] = __ffma2_rn(a[k], b[0], acc[k]);
        } else {
          acc[k].x = fmaf(a[k].x, b[k].x, acc[k].x);
          acc[k].y = fmaf(a[k].y, b[k].y, acc[k].y);
        }
      }
    }
  }
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) s += acc[k].x + acc[k].y;
  out[blockIdx.x * kThreads + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// interact2_pair with the products regrouped: u = q^3 r, then a += m_j u and
// the reaction b += (-m_i) u.
__device__ __forceinline__ void interact2_pair_u(float2 X, float2 Y, float2 Z, float2 M, float2 nx,
                                                 float2 ny, float2 nz, float2 nm, float2 e2,
                                                 float2& ax, float2& ay, float2& az, float2& bx,
                                                 float2& by, float2& bz) {
  const float2 rx = __fadd2_rn(X, nx);
  const float2 ry = __fadd2_rn(Y, ny);
  const float2 rz = __fadd2_rn(Z, nz);
  float2 d = __ffma2_rn(rx, rx, e2);
  d = __ffma2_rn(ry, ry, d);
  d = __ffma2_rn(rz, rz, d);
  const float2 q = make_float2(nbody::rsqrt_approx(d.x), nbody::rsqrt_approx(d.y));
  const float2 q3 = __fmul2_rn(__fmul2_rn(q, q), q);
  const float2 ux = __fmul2_rn(q3, rx);
  const float2 uy = __fmul2_rn(q3, ry);
  const float2 uz = __fmul2_rn(q3, rz);
  ax = __ffma2_rn(M, ux, ax);
  ay = __ffma2_rn(M, uy, ay);
  az = __ffma2_rn(M, uz, az);
  bx = __ffma2_rn(nm, ux, bx);
  by = __ffma2_rn(nm, uy, by);
  bz = __ffma2_rn(nm, uz, bz);
}

// The steady state of the pair kernel's reaction scheme 3 over one tile,
// repeated `iters` times (no TMA, no barriers, no per-tile work).  FORM 0:
// interact2_pair; FORM 1: interact2_pair_u.
template <int FORM>
__global__ void __launch_bounds__(kThreads, 1) pair_step(const float4* __restrict__ src, float* out,
                                                        long long* cycles, int iters, float eps2) {
  constexpr int P = 8;
  __shared__ __align__(16) float4 tile[4 * kTile];
  for (int b = threadIdx.x; b < kTile; b += kThreads) {
    const float4 x = src[b];
    const int r = 64 * (b >> 5) + (b & 31);
    tile[r] = tile[r + 32] = make_float4(x.x, x.x, x.y, x.y);
    tile[2 * kTile + r] = tile[2 * kTile + r + 32] = make_float4(x.z, x.z, x.w, x.w);
  }
  const int lane = threadIdx.x & 31;
  const float2 e2 = make_float2(eps2, eps2);
  float2 nx[P], ny[P], nz[P], nm[P], tx[P], ty[P], tz[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float f = 0.001f * (threadIdx.x + 37 * p);
    nx[p] = make_float2(-0.3f * f, 0.2f * f);
    ny[p] = make_float2(0.1f * f, -0.5f * f);
    nz[p] = make_float2(0.7f - f, f - 0.2f);
    nm[p] = make_float2(-1e-6f * (p + 1), -2e-6f * (p + 1));
    tx[p] = ty[p] = tz[p] = make_float2(0.f, 0.f);
  }
  float keep = 0.f;
  const int from = (lane + 1) & 31;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    for (int g = 0; g < kTile; g += 32) {
      const float4* lo0 = tile + 2 * g + lane;
      const float4* hi0 = tile + 2 * kTile + 2 * g + lane;
      float4 clo = lo0[0], chi = hi0[0];
      float bxs = 0.f, bys = 0.f, bzs = 0.f;
#pragma unroll 8
      for (int st = 0; st < 32; ++st) {
        const float4 lo = clo, hi = chi;
        if (st + 1 < 32) {
          clo = lo0[st + 1];
          chi = hi0[st + 1];
        }
        bxs = __shfl_sync(0xffffffffu, bxs, from);
        bys = __shfl_sync(0xffffffffu, bys, from);
        bzs = __shfl_sync(0xffffffffu, bzs, from);
        float2 bx = make_float2(bxs, 0.f), by = make_float2(bys, 0.f), bz = make_float2(bzs, 0.f);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          if (FORM == 0)
            nbody::interact2_pair(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                                  make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p],
                                  nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
          else
            interact2_pair_u(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                             make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p],
                             nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
        }
        bxs = bx.x + bx.y;
        bys = by.x + by.y;
        bzs = bz.x + bz.y;
      }
      keep += bxs + bys + bzs;
    }
  }
  const long long t1 = clock64();
  float s = keep;
#pragma unroll
  for (int p = 0; p < P; ++p) s += tx[p].x + tx[p].y + ty[p].x + ty[p].y + tz[p].x + tz[p].y;
  out[blockIdx.x * kThreads + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

double mean_cycles(const long long* d, int n) {
  std::vector<long long> h(n);
  cudaMemcpy(h.data(), d, n * sizeof(long long), cudaMemcpyDeviceToHost);
  double m = 0;
  for (long long v : h) m += static_cast<double>(v);
  return m / n;
}

bool check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return true;
  std::printf("%s: %s\n", what, cudaGetErrorString(e));
  return false;
}

}  // namespace

int main() {
  int sms = 0;
  if (!check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0), "device")) return 1;
  float* out = nullptr;
  long long* cyc = nullptr;
  float4* src = nullptr;
  if (!check(cudaMalloc(&out, static_cast<size_t>(sms) * kThreads * sizeof(float)), "alloc") ||
      !check(cudaMalloc(&cyc, static_cast<size_t>(sms) * sizeof(long long)), "alloc") ||
      !check(cudaMalloc(&src, kTile * sizeof(float4)), "alloc"))
    return 1;
  std::vector<float4> h(kTile);
  for (int b = 0; b < kTile; ++b)
    h[b] = make_float4(std::sin(1.0f * b), std::cos(2.0f * b), std::sin(3.0f * b + 1.f),
                       1e-6f * (1 + b % 7));
  cudaMemcpy(src, h.data(), kTile * sizeof(float4), cudaMemcpyHostToDevice);

  // one CTA per SM: request more shared memory than two CTAs could share
  const int smem = 120 * 1024;
  const int iters = 20000;
  const double ffma_ops = 16.0 * 2 * 8 * iters * kThreads;  // lane-ops per CTA
  struct Run {
    const char* name;
    void (*k)(float*, long long*, int, float);
  } runs[] = {{"ffma2, fresh operands", ffma_stream<0>},
              {"ffma2, shared operand", ffma_stream<1>},
              {"ffma, fresh operands", ffma_stream<2>}};
  std::printf("FP32 lane-ops per SM cycle / 128, %d SMs, %d threads per SM\n", sms, kThreads);
  for (const Run& r : runs) {
    cudaFuncSetAttribute(r.k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    r.k<<<sms, kThreads, smem>>>(out, cyc, 2, 1e-3f);
    r.k<<<sms, kThreads, smem>>>(out, cyc, iters, 1e-3f);
    if (!check(cudaDeviceSynchronize(), r.name)) return 1;
    std::printf("  %-24s %.4f\n", r.name, ffma_ops / (mean_cycles(cyc, sms) * 128.0));
  }
  const int piters = 100;
  // per thread and step: 8 target pairs x 16 packed instructions (32 lane-ops) + 3 adds; the
  // u form does the same work in 17 packed instructions and is counted the same (per pair)
  const double pair_ops = (8.0 * 32 + 3) * kTile * piters * kThreads;
  struct PairRun {
    const char* name;
    void (*k)(const float4*, float*, long long*, int, float);
  } pruns[] = {{"pair step", pair_step<0>}, {"pair step, u form", pair_step<1>}};
  for (const PairRun& r : pruns) {
    cudaFuncSetAttribute(r.k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    r.k<<<sms, kThreads, smem>>>(src, out, cyc, 2, 1e-3f);
    r.k<<<sms, kThreads, smem>>>(src, out, cyc, piters, 1e-3f);
    if (!check(cudaDeviceSynchronize(), r.name)) return 1;
    std::printf("  %-24s %.4f\n", r.name, pair_ops / (mean_cycles(cyc, sms) * 128.0));
  }
  cudaFree(out);
  cudaFree(cyc);
  cudaFree(src);
  return 0;
}
