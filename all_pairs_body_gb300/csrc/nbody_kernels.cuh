// Device code of the all-pairs softened-gravity library (sm_103a).
//
// Computes a_i = sum_j m_j (x_j - x_i) / (|x_j - x_i|^2 + eps2)^(3/2), G = 1
// ("CUDA N-Body Simulation", §1.2), and optionally fuses the leapfrog
// half-kick + drift of §1.3 into the pass that completes each a_i.
//
// Kernels
//   force_tiled<KI,NT,TJ,MINB,UNR,FORM,NLOG>
//                       KI target bodies per thread in registers (KI/2 packed
//                       FP32 pairs); source tiles of TJ bodies brought into a
//                       two-stage shared-memory ring by 1-D TMA bulk copies of
//                       the caller's float4 rows (mbarrier completion), then
//                       expanded by the CTA into two rows (x,x,y,y),(z,z,w0,w1)
//                       per body so each source component is an already
//                       duplicated FP32 pair; packed FFMA2/FADD2/FMUL2 +
//                       MUFU.RSQ inner loop.  Work = (i-block, j-tile) units divided
//                       evenly over the grid; a CTA that covers an i-block's
//                       whole j range finishes it (accel or kick/drift), else
//                       it writes a partial sum for the second pass.
//   finish_streamk      second pass for the tiled kernel: sums the partials
//                       of split i-blocks in CTA (= j) order and finishes.
//   force_pairs<KI,NT,TJ,NB,UNRB,ACC,ROT>
//                       the tiled kernel with each pair of bodies in
//                       different i-blocks evaluated once (Newton's third
//                       law): action on the targets in registers, reaction on
//                       the sources summed over each warp (carried from lane
//                       to lane as the sources rotate through the lanes, or,
//                       in the tuning build, a warp butterfly), then over the
//                       warps in order, into one partial per unit.
//   finish_pairs        its second pass: action + reactions in block order,
//                       then the finish (accel or kick/drift) of every body.
//   accumulate_pairs, finish_accumulated
//                       the same in chunks of i-blocks where the reaction
//                       sums of all units would not fit the scratch.
//   force_warp<KW,NW,U> small-n kernel: a CTA owns KW targets; its NW*32
//                       threads stride over one j slice, loading U sources
//                       ahead; warp shuffles then shared memory (fixed
//                       order) combine the threads.
//   finish_slices       second pass for the warp kernel: sums S slices in order.
//   copy_rows           the positions an odd number of one-kernel drifts left
//                       in the other buffer, into the caller's buffer.
//   Every force and finishing kernel is a programmatic dependent of the
//   kernel before it (allow_dependent_launch / wait_for_prior_grid).
//   render_points       the point shaders of "CUDA N-Body Simulation" §4.3 as a
//                       kernel: normalised device coordinates and mass colour
//                       of every body into a device buffer (no graphics API).
//   neighbors_2d        the 2-D cutoff neighbour list of "CUDA编程（九）原子函数
//                       的合理使用" §3 without atomics: all pairs, packed FP32,
//                       per-target counts and ascending transposed lists.
//
// The pages' tiled kernel ("CUDA N-Body Simulation" §3.1, "Cuda Nbody Notes"
// calculate_forces, The CUDA Handbook ch. 14 shared-memory kernel) keeps one
// target per thread and loads tiles with plain stores plus two barriers;
// the design here keeps that tiling idea and replaces the rest.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "nbody.h"

namespace nbody {

// Index checks of the checked build (compiled with NBODY_BOUNDS_CHECK): each
// computed index into a scratch or output array is tested against the
// capacity the host allocated for that call (passed in the launch's Ctl); a
// failed check records NBODY_EBOUNDS in the calling stream's status word
// (the first error wins) and the access is skipped.  In the release build
// NBODY_IN_BOUNDS is the constant true, so every guarded access compiles
// exactly as unguarded.
enum CapSlot : int {
  kCapRows = 0,   // rows of pos/accel/vel/pos_next/ndc/rgba and of per-body scratch
  kCapPartial,    // float4 rows of `partial`
  kCapReact,      // float4 rows of the pair path's reaction sums
  kCapNeighbors,  // ints of the neighbour list
  kNumCaps
};

// What every launch carries besides its data: the status word of the stream
// it runs on (NBODY_OK until a kernel records a failure; nbody_sync on that
// stream reads and clears it), and in the checked build the capacities of
// the call's arrays.
struct Ctl {
  int* status;
#ifdef NBODY_BOUNDS_CHECK
  long long caps[kNumCaps];
#endif
};

#ifdef NBODY_BOUNDS_CHECK
__device__ __noinline__ bool index_in_bounds(const Ctl& c, long long idx, int slot) {
  if (idx >= 0 && idx < c.caps[slot]) return true;
  atomicCAS(c.status, 0, static_cast<int>(NBODY_EBOUNDS));
  return false;
}
#define NBODY_IN_BOUNDS(ctl, idx, slot) index_in_bounds((ctl), (idx), (slot))
#else
#define NBODY_IN_BOUNDS(ctl, idx, slot) true
#endif

// Phase clocks of the profiling build (compiled with NBODY_PHASE_CLOCKS): the
// pair kernel's warps add the SM cycles they spend in each phase of a tile
// to these counters (lane 0 of every warp, at the end of the launch), read
// and cleared by nbody_phase_read.  The release build has no stamps.
enum PairPhase : int {
  kPhaseWait = 0,   // the tile copy's mbarrier wait and the first CTA barrier
  kPhaseExpand,     // issuing the next copy, the expansion, the second barrier
  kPhaseOwn,        // the arithmetic of a tile of the block itself (one-sided loop)
  kPhaseCross,      // the arithmetic of a tile past the block (rotation, reaction rows)
  kPhaseReduce,     // the third barrier, the warps' reaction sums and the row's store
  kPhaseFold,       // folding the per-tile sums into the running sums
  kPhaseOther,      // the rest: target loads, segment epilogues, set-up
  kNumPhases
};
#ifdef NBODY_PHASE_CLOCKS
__device__ unsigned long long g_phase_cycles[kNumPhases];
#define NBODY_PHASE_DECL long long ph_[kNumPhases] = {}, ph_t_ = clock64()
#define NBODY_PHASE(q)                    \
  do {                                    \
    const long long ph_now_ = clock64();  \
    ph_[(q)] += ph_now_ - ph_t_;          \
    ph_t_ = ph_now_;                      \
  } while (0)
#define NBODY_PHASE_FLUSH()                                                           \
  do {                                                                              \
    NBODY_PHASE(kPhaseOther);                                                       \
    if ((threadIdx.x & 31) == 0)                                                    \
      for (int q_ = 0; q_ < kNumPhases; ++q_)                                       \
        atomicAdd(&g_phase_cycles[q_], static_cast<unsigned long long>(ph_[q_]));   \
  } while (0)
#else
#define NBODY_PHASE_DECL
#define NBODY_PHASE(q)
#define NBODY_PHASE_FLUSH()
#endif

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float rsqrt_approx(float x) {
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` of the mbarrier completes, for at most
// timeout_ns of global time.  Returns false when the limit expired.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 16; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// 1-D TMA bulk copy global -> shared; completion counted on the mbarrier.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// the pair interaction, two target bodies at once
// ---------------------------------------------------------------------------

// One source body (X, Y, Z, M: each component duplicated in both halves)
// against two target bodies whose NEGATED coordinates are (nx, ny, nz):
//   r = x_j - x_i, d = |r|^2 + eps2, q = d^(-1/2), s = m_j q^3, a += s r.
// 12 packed-pair FP32 instructions and 2 MUFU.RSQ for two interactions.
// q^3 is formed as (q q) q and then scaled by the mass, the order the
// pair-symmetric kernel uses, so that both kernels round every term alike.
__device__ __forceinline__ void interact2(float2 X, float2 Y, float2 Z, float2 M, float2 nx,
                                          float2 ny, float2 nz, float2 e2, float2& ax, float2& ay,
                                          float2& az) {
  const float2 rx = __fadd2_rn(X, nx);
  const float2 ry = __fadd2_rn(Y, ny);
  const float2 rz = __fadd2_rn(Z, nz);
  float2 d = __ffma2_rn(rx, rx, e2);
  d = __ffma2_rn(ry, ry, d);
  d = __ffma2_rn(rz, rz, d);
  const float2 q = make_float2(rsqrt_approx(d.x), rsqrt_approx(d.y));
  const float2 q3 = __fmul2_rn(__fmul2_rn(q, q), q);
  const float2 s = __fmul2_rn(M, q3);
  ax = __ffma2_rn(rx, s, ax);
  ay = __ffma2_rn(ry, s, ay);
  az = __ffma2_rn(rz, s, az);
}

// The interaction with a scalar source mass m (both targets see the same
// source): the mass factor costs two scalar multiplies on the FMA pipe, the
// same pipe time as one packed multiply, and needs no duplicated register.
__device__ __forceinline__ void interact2_rsq(float2 X, float2 Y, float2 Z, float m, float2 nx,
                                              float2 ny, float2 nz, float2 e2, float2& ax,
                                              float2& ay, float2& az) {
  const float2 rx = __fadd2_rn(X, nx);
  const float2 ry = __fadd2_rn(Y, ny);
  const float2 rz = __fadd2_rn(Z, nz);
  float2 d = __ffma2_rn(rx, rx, e2);
  d = __ffma2_rn(ry, ry, d);
  d = __ffma2_rn(rz, rz, d);
  const float2 q = make_float2(rsqrt_approx(d.x), rsqrt_approx(d.y));
  const float2 q2 = __fmul2_rn(q, q);
  const float2 s = __fmul2_rn(make_float2(m * q.x, m * q.y), q2);
  ax = __ffma2_rn(rx, s, ax);
  ay = __ffma2_rn(ry, s, ay);
  az = __ffma2_rn(rz, s, az);
}

// The interaction with the mass factor and the inverse 3/2 power taken
// through base-2 logarithms: s = m_j d^(-3/2) = 2^(L_j - 1.5 log2 d), with
// L_j = log2 m_j stored with the source (-inf for m_j = 0, which gives s = +0
// exactly).  Two FP32 operations per interaction fewer than interact2 on the
// FMA pipe, in exchange for one more MUFU; mixing the two forms balances the
// FMA and MUFU pipes.
__device__ __forceinline__ void interact2_lg(float2 X, float2 Y, float2 Z, float L, float2 nx,
                                             float2 ny, float2 nz, float2 e2, float2& ax,
                                             float2& ay, float2& az) {
  const float2 rx = __fadd2_rn(X, nx);
  const float2 ry = __fadd2_rn(Y, ny);
  const float2 rz = __fadd2_rn(Z, nz);
  float2 d = __ffma2_rn(rx, rx, e2);
  d = __ffma2_rn(ry, ry, d);
  d = __ffma2_rn(rz, rz, d);
  const float2 s = make_float2(ex2_approx(fmaf(lg2_approx(d.x), -1.5f, L)),
                               ex2_approx(fmaf(lg2_approx(d.y), -1.5f, L)));
  ax = __ffma2_rn(rx, s, ax);
  ay = __ffma2_rn(ry, s, ay);
  az = __ffma2_rn(rz, s, az);
}

// ---------------------------------------------------------------------------
// finishing a body: write a_i, and for a leapfrog step kick and drift
// ---------------------------------------------------------------------------

// Layouts of the velocity and acceleration arrays (positions are always
// float4 rows): rows of float4 (w of accel 0, w of vel kept), rows of three
// floats, or three blocks x[0..n), y[0..n), z[0..n) ("CUDA N-Body
// Simulation" §3.5 compares the float4 and float3 forms).
enum VecLayout : int { kRows4 = 0, kRows3 = 1, kBlocks3 = 2 };

// Programmatic dependent launch.  Every force and second-pass kernel lets
// the launch of the kernel queued after it (launched with programmatic
// stream serialization) begin once all of its own CTAs are running, so that
// launch overlaps this kernel's tail; and waits, before its first memory
// access, until the kernel before it has completed and its writes are
// visible.  The dependent's CTAs are placed only after every CTA of the
// kernel before it has started, so they never hold back its CTAs.  Both are
// no-ops for kernels launched without the attribute.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void wait_for_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

struct Epilogue {
  const float4* pos;  // start-of-step positions (x, y, z, m)
  float* accel;       // out: accelerations in `layout`
  float* vel;         // step only (nullptr: acceleration only), in `layout`
  float4* pos_next;   // step with a drift: end-of-step positions (nullptr: kick only)
  float kick;         // velocity kick coefficient on a (dt/2 for a half kick)
  float dt;           // drift coefficient on v
  int layout;         // VecLayout of accel and vel
  long long n;        // bodies (block stride of kBlocks3)
  Ctl ctl;
};

__device__ __forceinline__ void store_vec3(float* base, int layout, long long n, long long i, float x,
                                           float y, float z, float w) {
  if (layout == kRows4) {
    reinterpret_cast<float4*>(base)[i] = make_float4(x, y, z, w);
  } else if (layout == kRows3) {
    base[3 * i] = x;
    base[3 * i + 1] = y;
    base[3 * i + 2] = z;
  } else {
    base[i] = x;
    base[n + i] = y;
    base[2 * n + i] = z;
  }
}

__device__ __forceinline__ float4 load_vec3(const float* base, int layout, long long n, long long i) {
  if (layout == kRows4) return reinterpret_cast<const float4*>(base)[i];
  if (layout == kRows3) return make_float4(base[3 * i], base[3 * i + 1], base[3 * i + 2], 0.f);
  return make_float4(base[i], base[n + i], base[2 * n + i], 0.f);
}

// v <- v + kick a ; then, with a drift, x <- x + dt v.
// The pages' step is kick = dt/2 plus the drift ("CUDA N-Body Simulation"
// §1.3); the kick-drift-kick form fuses the closing half kick of one step
// with the opening half kick of the next (kick = dt) and ends with a
// kick-only pass.
// Kept out of line (and taken by value): it runs once per body and segment,
// and inlining it into the force kernel perturbs the register allocation and
// schedule of the inner loop (up to 2.5% in a measured sweep).
// The body's velocity and position as the epilogue needs them (zeros where
// it needs none); the second-pass kernels load them before their sums, so
// that these loads overlap the sums' loads.
struct BodyState {
  float4 v, x;
};

__device__ __forceinline__ BodyState load_body(const Epilogue& e, long long i) {
  BodyState b{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  if (!NBODY_IN_BOUNDS(e.ctl, i, kCapRows)) return b;
  if (e.vel != nullptr) {
    b.v = load_vec3(e.vel, e.layout, e.n, i);
    if (e.pos_next != nullptr) b.x = e.pos[i];
  }
  return b;
}

__device__ __forceinline__ void finish_loaded(const Epilogue& e, long long i, float ax, float ay,
                                              float az, BodyState b) {
  if (!NBODY_IN_BOUNDS(e.ctl, i, kCapRows)) return;
  store_vec3(e.accel, e.layout, e.n, i, ax, ay, az, 0.0f);
  if (e.vel != nullptr) {
    float4 v = b.v;
    v.x = fmaf(e.kick, ax, v.x);
    v.y = fmaf(e.kick, ay, v.y);
    v.z = fmaf(e.kick, az, v.z);
    store_vec3(e.vel, e.layout, e.n, i, v.x, v.y, v.z, v.w);
    if (e.pos_next == nullptr) return;
    float4 x = b.x;
    x.x = fmaf(e.dt, v.x, x.x);
    x.y = fmaf(e.dt, v.y, x.y);
    x.z = fmaf(e.dt, v.z, x.z);
    e.pos_next[i] = x;
  }
}

__device__ __noinline__ void finish_body(const Epilogue e, long long i, float ax, float ay,
                                         float az) {
  finish_loaded(e, i, ax, ay, az, load_body(e, i));
}

// ---------------------------------------------------------------------------
// source tile expansion
// ---------------------------------------------------------------------------

// tile[2b] = (x,x,y,y), tile[2b+1] = (z,z,m,w1) for the staged rows b < tj of
// one tile, zero rows past `live` (zero mass adds exactly nothing); w1 = m
// for form 0, log2 m (-inf for m = 0) for form 1.  Returns whether any live
// mass is negative or NaN.  Out of line: it runs once per tile and, inlined,
// perturbs the register allocation of the inner loop.
__device__ __noinline__ bool expand_tile(const float4* raw, float4* tile, int tj, int nt, int tid,
                                         long long live, int form) {
  bool odd = false;
  for (int b = tid; b < tj; b += nt) {
    const bool ok = b < live;
    const float4 x = ok ? raw[b] : make_float4(0.f, 0.f, 0.f, 0.f);
    float w1 = x.w;
    if (form == 1) {
      odd |= ok && !(x.w >= 0.0f);
      w1 = x.w > 0.0f ? log2f(x.w) : (x.w == 0.0f ? -INFINITY : x.w);
    }
    tile[2 * b] = make_float4(x.x, x.x, x.y, x.y);
    tile[2 * b + 1] = make_float4(x.z, x.z, x.w, w1);
  }
  return odd;
}

// The same expansion with the two halves in separate arrays: tile[b] =
// (x, x, y, y), tile[tj + b] = (z, z, m, m).  Lanes that read consecutive
// sources then read consecutive 16-byte rows (no bank conflicts).
__device__ __noinline__ void expand_tile_split(const float4* raw, float4* tile, int tj, int nt,
                                               int tid, long long live) {
  for (int b = tid; b < tj; b += nt) {
    const float4 x = b < live ? raw[b] : make_float4(0.f, 0.f, 0.f, 0.f);
    tile[b] = make_float4(x.x, x.x, x.y, x.y);
    tile[tj + b] = make_float4(x.z, x.z, x.w, x.w);
  }
}

// The same with every group of 32 sources stored twice in a row, so that a
// lane reading the sources of its group in rotated order, (l + s) mod 32 for
// steps s = 0..31, reads rows l, l + 1, ..., l + 31 of the group's 64 rows:
// constant offsets from one base address, no wrap-around.  Source b of the
// tile sits at rows 64 (b / 32) + (b mod 32) and 32 rows further, first half
// (x, x, y, y) in rows [0, 2 tj), second half (z, z, m, m) in rows
// [2 tj, 4 tj).
__device__ __noinline__ void expand_tile_dup(const float4* raw, float4* tile, int tj, int nt,
                                             int tid, long long live) {
  for (int b = tid; b < tj; b += nt) {
    const float4 x = b < live ? raw[b] : make_float4(0.f, 0.f, 0.f, 0.f);
    const int r = 64 * (b >> 5) + (b & 31);
    const float4 lo = make_float4(x.x, x.x, x.y, x.y);
    const float4 hi = make_float4(x.z, x.z, x.w, x.w);
    tile[r] = lo;
    tile[r + 32] = lo;
    tile[2 * tj + r] = hi;
    tile[2 * tj + r + 32] = hi;
  }
}

// ---------------------------------------------------------------------------
// tiled force kernel with an even (stream-K) division of the work
// ---------------------------------------------------------------------------

struct TiledArgs {
  const float4* pos;  // n rows (x, y, z, m): the targets and the sources
  int n;
  float eps2;
  long long ntiles;  // source tiles over n
  long long units;   // i-blocks * ntiles
  long long grid;    // CTAs launched
  float4* partial;   // [grid][2][KI*NT] partial sums of split i-blocks
  uint64_t timeout_ns;
  long long withhold;  // failure-detection check only: this unit's copy is never issued (-1: none)
};

// First work unit of CTA c when `units` are divided over `grid` CTAs.
__host__ __device__ __forceinline__ long long unit_begin(long long units, long long grid,
                                                         long long c) {
  return units * c / grid;
}

// CTA whose range holds unit u (inverse of unit_begin).
__host__ __device__ __forceinline__ long long unit_owner(long long units, long long grid,
                                                         long long u) {
  return ((u + 1) * grid - 1) / units;
}

template <int KI, int NT, int TJ, int MINB, int UNR, int FORM, int NLOG>
__global__ void __launch_bounds__(NT, MINB) force_tiled(const TiledArgs a, const Epilogue e) {
  static_assert(KI % 2 == 0, "targets are processed in packed pairs");
  constexpr int P = KI / 2;
  constexpr long long B = static_cast<long long>(KI) * NT;

  __shared__ __align__(128) float4 raw[2][TJ];  // TMA targets: the caller's rows
  __shared__ __align__(128) float4 tile[2 * TJ];  // expanded: (x,x,y,y),(z,z,w0,w1)
  __shared__ __align__(8) unsigned long long bar[2];

  const int tid = threadIdx.x;
  allow_dependent_launch();
  wait_for_prior_grid();
  const long long c = blockIdx.x;
  const long long u_lo = unit_begin(a.units, a.grid, c);
  const long long count = unit_begin(a.units, a.grid, c + 1) - u_lo;
  // shared-memory addresses of stage s: base + s * stride
  const uint32_t bar0 = smem_u32(&bar[0]);
  const uint32_t raw0 = smem_u32(&raw[0][0]);
  constexpr uint32_t kRawStride = sizeof(raw[0]);
  auto bar_of = [&](long long k) { return bar0 + static_cast<uint32_t>(k & 1) * 8u; };
  auto raw_of = [&](long long k) { return raw0 + static_cast<uint32_t>(k & 1) * kRawStride; };

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (count <= 0) return;

  // Copy the source rows of local unit k's tile into stage k & 1 (only the
  // rows that exist: the last tile may be short; 16 bytes per row keeps
  // every address and size a multiple of 16).
  auto issue = [&](long long k) {
    const long long j0 = ((u_lo + k) % a.ntiles) * TJ;
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<long long>(TJ), a.n - j0)) * 16u;
    mbar_arrive_expect_tx(bar_of(k), bytes);
    bulk_copy_g2s(raw_of(k), a.pos + j0, bytes, bar_of(k));
  };
  if (tid == 0 && a.withhold != 0) issue(0);

  const float2 e2 = make_float2(a.eps2, a.eps2);
  float2 nx[P], ny[P], nz[P], ax[P], ay[P], az[P];
  long long k = 0;
  bool timed_out = false;

  while (k < count) {
    const long long u = u_lo + k;
    const long long blk = u / a.ntiles;
    const long long tb = u % a.ntiles;
    const long long te = min(a.ntiles, tb + (count - k));
    const bool first_segment = (k == 0);

#pragma unroll
    for (int p = 0; p < P; ++p) {
      const long long i0 = blk * B + (2 * p) * NT + tid;
      const long long i1 = i0 + NT;
      const float4 q0 = a.pos[min(i0, static_cast<long long>(a.n - 1))];
      const float4 q1 = a.pos[min(i1, static_cast<long long>(a.n - 1))];
      nx[p] = make_float2(-q0.x, -q1.x);
      ny[p] = make_float2(-q0.y, -q1.y);
      nz[p] = make_float2(-q0.z, -q1.z);
      ax[p] = ay[p] = az[p] = make_float2(0.f, 0.f);
    }

    for (long long t = tb; t < te; ++t, ++k) {
      const int s = static_cast<int>(k & 1);
      const uint32_t parity = static_cast<uint32_t>((k >> 1) & 1);
      const bool ok = mbar_wait_bounded(bar_of(k), parity, a.timeout_ns);
      // Every thread reaches this barrier in bounded time; it makes the
      // timeout decision uniform and guarantees that all threads are done
      // with the expanded tile (read in the previous iteration) and with
      // stage s^1 of the ring (expanded in the previous iteration) before
      // either is rewritten.
      if (!__syncthreads_and(ok)) {
        timed_out = true;
        break;
      }
      if (tid == 0 && k + 1 < count && k + 1 != a.withhold) issue(k + 1);

      // Expand the tile: rows past n become zero-mass rows, which add exactly
      // nothing.  FORM 1 stores log2 m beside m and runs the whole tile in
      // the rsqrt form when any of its masses is negative or NaN.
      const bool odd_mass =
          expand_tile(raw[s], tile, TJ, NT, tid, static_cast<long long>(a.n) - t * TJ, FORM);
      bool exact = false;
      if (FORM == 1)
        exact = __syncthreads_or(odd_mass) != 0;
      else
        __syncthreads();

      // Per-tile sums, folded into the running sums after the tile: the
      // rounding error grows like sqrt(TJ) + sqrt(n / TJ), not sqrt(n).
      float2 tx[P], ty[P], tz[P];
#pragma unroll
      for (int p = 0; p < P; ++p) tx[p] = ty[p] = tz[p] = make_float2(0.f, 0.f);
      const float4* src = tile;
      if (FORM == 1 && !exact) {
        // mixed form: the first NLOG target pairs take the logarithmic form
#pragma unroll UNR
        for (int j = 0; j < TJ; ++j) {
          const float4 lo = src[2 * j];
          const float4 hi = src[2 * j + 1];
          const float2 X = make_float2(lo.x, lo.y);
          const float2 Y = make_float2(lo.z, lo.w);
          const float2 Z = make_float2(hi.x, hi.y);
#pragma unroll
          for (int p = 0; p < P; ++p) {
            if (p < NLOG)
              interact2_lg(X, Y, Z, hi.w, nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
            else
              interact2_rsq(X, Y, Z, hi.z, nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
          }
        }
      } else if (FORM == 1) {
#pragma unroll UNR
        for (int j = 0; j < TJ; ++j) {
          const float4 lo = src[2 * j];
          const float4 hi = src[2 * j + 1];
          const float2 X = make_float2(lo.x, lo.y);
          const float2 Y = make_float2(lo.z, lo.w);
          const float2 Z = make_float2(hi.x, hi.y);
#pragma unroll
          for (int p = 0; p < P; ++p)
            interact2_rsq(X, Y, Z, hi.z, nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
        }
      } else {
#pragma unroll UNR
        for (int j = 0; j < TJ; ++j) {
          const float4 lo = src[2 * j];
          const float4 hi = src[2 * j + 1];
          const float2 X = make_float2(lo.x, lo.y);
          const float2 Y = make_float2(lo.z, lo.w);
          const float2 Z = make_float2(hi.x, hi.y);
          const float2 M = make_float2(hi.z, hi.w);
#pragma unroll
          for (int p = 0; p < P; ++p)
            interact2(X, Y, Z, M, nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
        }
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        ax[p] = __fadd2_rn(ax[p], tx[p]);
        ay[p] = __fadd2_rn(ay[p], ty[p]);
        az[p] = __fadd2_rn(az[p], tz[p]);
      }
    }
    if (timed_out) break;

    const bool whole = (tb == 0 && te == a.ntiles);
    const long long slot = (c * 2 + (first_segment ? 0 : 1)) * B;
#pragma unroll
    for (int p = 0; p < P; ++p) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long long local = (2 * p + h) * NT + tid;
        const long long i = blk * B + local;
        if (i < a.n) {
          const float fx = h ? ax[p].y : ax[p].x;
          const float fy = h ? ay[p].y : ay[p].x;
          const float fz = h ? az[p].y : az[p].x;
          if (whole)
            finish_body(e, i, fx, fy, fz);
          else if (NBODY_IN_BOUNDS(e.ctl, slot + local, kCapPartial))
            a.partial[slot + local] = make_float4(fx, fy, fz, 0.f);
        }
      }
    }
  }

  if (timed_out && tid == 0) {
    atomicExch(e.ctl.status, static_cast<int>(NBODY_ETIMEOUT));
    // The copy of unit k may still be landing in shared memory: give it a
    // bounded wait before the CTA (and its shared memory) goes away.
    if (k != a.withhold)
      (void)mbar_wait_bounded(bar_of(k), static_cast<uint32_t>((k >> 1) & 1), a.timeout_ns);
  }
}

// Second pass of the tiled kernel: one thread per body; bodies of i-blocks
// that one CTA covered whole were finished already and return at once.
struct StreamkFinishArgs {
  const float4* partial;
  int n;
  long long block;  // target bodies per i-block (KI * NT)
  long long ntiles;
  long long units;
  long long grid;
};

__global__ void finish_streamk(const StreamkFinishArgs a, const Epilogue e) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  const long long blk = i / a.block;
  const long long u0 = blk * a.ntiles;
  const long long c0 = unit_owner(a.units, a.grid, u0);
  const long long c1 = unit_owner(a.units, a.grid, u0 + a.ntiles - 1);
  if (c0 == c1) return;
  const long long local = i - blk * a.block;
  const BodyState b = load_body(e, i);
  float sx = 0.f, sy = 0.f, sz = 0.f;
  // The block's segment is CTA cc's first segment, except for CTA c0 when it
  // started before the block (every later CTA starts inside it).
  const int side0 = unit_begin(a.units, a.grid, c0) >= u0 ? 0 : 1;
  constexpr int D = 8;  // partials loaded eight CTAs at a time, added in CTA order
  for (long long c = c0; c <= c1; c += D) {
    float4 p[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const long long cc = c + d;
      p[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (cc <= c1) {
        const int side = cc == c0 ? side0 : 0;
        const long long at = (cc * 2 + side) * a.block + local;
        if (NBODY_IN_BOUNDS(e.ctl, at, kCapPartial)) p[d] = a.partial[at];
      }
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (c + d <= c1) {
        sx += p[d].x;
        sy += p[d].y;
        sz += p[d].z;
      }
    }
  }
  finish_loaded(e, i, sx, sy, sz, b);
}

// ---------------------------------------------------------------------------
// pair-symmetric tiled force kernel
// ---------------------------------------------------------------------------
//
// Every unordered pair of bodies in different i-blocks is evaluated once: the
// term m_i (x_i - x_j) d^(-3/2) that body i adds to a_j is the negative of what
// the same pair gives a_i with m_j replaced by m_i, bit for bit (the same r,
// d and d^(-3/2) in FP32), so one evaluation serves both bodies (Newton's
// third law).  Pairs inside one i-block are evaluated from both sides, as in
// force_tiled.  Per pair: 3 FADD + 3 FFMA (d) + 1 MUFU.RSQ + 2 FMUL (d^-3/2)
// + 2 FMUL (the two mass factors) + 6 FFMA (action and reaction) = 16 FP32
// lane-ops for two interactions, against 24 for the one-sided form.
//
// Work: block I (B = KI * NT targets) meets the source tiles t of its own
// block and of every later block, tiles [TB*I, ntiles) with TB = B / TJ, in
// that order; the (I, t) units are numbered block by block and divided
// evenly over one wave of CTAs as in force_tiled.  For a tile past block I
// the reaction on its TJ sources is summed over the CTA's B targets (in each
// warp by the lane rotation or the butterfly described at force_pairs, then
// over the NW warps in order through shared memory) and stored as that unit's
// partial; the second pass adds, for each body, its action and the reactions
// from the blocks before its own in block order.

// Units of blocks 0 .. I-1: block I' has ntiles - TB * I' units.
__host__ __device__ __forceinline__ long long pair_units_before(long long I, long long ntiles,
                                                                long long tb) {
  return I * ntiles - tb * (I * (I - 1) / 2);
}

struct PairArgs {
  const float4* pos;  // n rows (x, y, z, m)
  int n;
  float eps2;
  long long ntiles;   // source tiles of TJ bodies over n
  long long nblocks;  // i-blocks of B bodies over n
  long long u_base;   // first unit of this launch (the first unit of its first i-block)
  long long units;    // units of this launch, from u_base
  long long grid;     // CTAs launched
  float4* act;        // [n] action sums of i-blocks one CTA covered whole
  float4* partial;    // [grid][2][B] action sums of split i-blocks
  float4* react;      // [units][TJ] reaction sums of this launch's units (local index)
  uint64_t timeout_ns;
  long long withhold;  // failure-detection check only (see TiledArgs)
  Ctl ctl;
};

// One source (duplicated pairs X, Y, Z, M) against two targets (negated
// coordinates nx, ny, nz and negated masses nm): the action on the targets
// goes to (ax, ay, az), the reaction on the source to (bx, by, bz) per target
// half.
__device__ __forceinline__ void interact2_pair(float2 X, float2 Y, float2 Z, float2 M, float2 nx,
                                               float2 ny, float2 nz, float2 nm, float2 e2,
                                               float2& ax, float2& ay, float2& az, float2& bx,
                                               float2& by, float2& bz) {
  const float2 rx = __fadd2_rn(X, nx);
  const float2 ry = __fadd2_rn(Y, ny);
  const float2 rz = __fadd2_rn(Z, nz);
  float2 d = __ffma2_rn(rx, rx, e2);
  d = __ffma2_rn(ry, ry, d);
  d = __ffma2_rn(rz, rz, d);
  const float2 q = make_float2(rsqrt_approx(d.x), rsqrt_approx(d.y));
  const float2 q3 = __fmul2_rn(__fmul2_rn(q, q), q);
  const float2 si = __fmul2_rn(M, q3);
  const float2 sj = __fmul2_rn(nm, q3);
  ax = __ffma2_rn(rx, si, ax);
  ay = __ffma2_rn(ry, si, ay);
  az = __ffma2_rn(rz, si, az);
  bx = __ffma2_rn(rx, sj, bx);
  by = __ffma2_rn(ry, sj, by);
  bz = __ffma2_rn(rz, sj, bz);
}

// Sum v[0..NB) (one value per source of a batch of NB = 8 or 16) over the 32
// lanes of the warp, leaving source (lane >> (5 - log2 NB))'s total in that
// lane: each butterfly level halves the values a lane keeps (the lanes with
// the level's mask bit keep the upper half), then the remaining levels sum
// the one value left.  3 * (NB - 1 + 5 - log2 NB) shuffles and as many adds.
template <int NB>
__device__ __forceinline__ float3 reduce_scatter(float (&vx)[NB], float (&vy)[NB],
                                                 float (&vz)[NB], int lane) {
  static_assert(NB == 8 || NB == 16, "batches of 8 or 16 sources");
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kLevels = NB == 8 ? 3 : 4;
#pragma unroll
  for (int level = 0; level < kLevels; ++level) {
    const int half = (NB >> level) >> 1;
    const int m = 16 >> level;
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int q = 0; q < half; ++q) {
      const float kx = up ? vx[q + half] : vx[q], sx = up ? vx[q] : vx[q + half];
      const float ky = up ? vy[q + half] : vy[q], sy = up ? vy[q] : vy[q + half];
      const float kz = up ? vz[q + half] : vz[q], sz = up ? vz[q] : vz[q + half];
      vx[q] = kx + __shfl_xor_sync(kAll, sx, m);
      vy[q] = ky + __shfl_xor_sync(kAll, sy, m);
      vz[q] = kz + __shfl_xor_sync(kAll, sz, m);
    }
  }
#pragma unroll
  for (int m = 16 >> kLevels; m >= 1; m >>= 1) {
    vx[0] += __shfl_xor_sync(kAll, vx[0], m);
    vy[0] += __shfl_xor_sync(kAll, vy[0], m);
    vz[0] += __shfl_xor_sync(kAll, vz[0], m);
  }
  return make_float3(vx[0], vy[0], vz[0]);
}

// Dynamic shared memory of force_pairs: with ROT >= 3 first the two-stage
// ring of the caller's source rows (the TMA targets), then the per-warp
// reaction sums of a tile, and with ACC = 1 the targets' running action sums.
__host__ __device__ constexpr size_t pair_reduce_smem(int ki, int nt, int tj, int acc, int rot) {
  // rot 5 (force_pairs_pipe): the ring, two expanded tiles and two sets of reaction rows
  return rot == 5 ? static_cast<size_t>(10) * tj * sizeof(float4) +
                        static_cast<size_t>(2) * (nt / 32) * 3 * tj * sizeof(float)
                  : (rot >= 3 ? static_cast<size_t>(2) * tj * sizeof(float4) : 0) +
                        static_cast<size_t>(nt / 32) * 3 * tj * sizeof(float) +
                        (acc ? static_cast<size_t>(3) * ki * nt * sizeof(float) : 0);
}

// ACC = 0: the running action sums of a segment live in registers beside the
// per-tile sums.  ACC = 1: they live in shared memory ([3][KI/2][NT] float2,
// one column per thread) and are touched once per tile, when the per-tile sums
// are folded in, which leaves 3 KI registers to the inner loop.
//
// ROT = 0: a tile's reactions are reduced over the lanes in batches of NB
// sources (reduce_scatter).  ROT = 1: the sources rotate through the lanes
// instead.  In each group of 32 sources, at step s lane l evaluates source
// (l + s) mod 32 against its targets and adds to that source's reaction sum,
// which it takes from lane l + 1 (the lane that evaluated the source at step
// s - 1); after 32 steps lane l holds the warp's whole sum for source
// (l + 31) mod 32.  That costs 6 shuffles per source and step and no adds or
// selects; UNRB then unrolls the 32 steps.  ROT = 2: two groups of 32 sources
// rotate side by side, each lane carrying two independent sums.
//
// ROT = 3 (the default shapes): the rotation of ROT = 1 with three changes
// that each measured faster in isolation.  (a) The lane passes on one scalar
// per component: its 7 target pairs add to (carried sum, 0) in the packed
// chain and the two halves are added before the shuffle, 3 shuffles and 3
// scalar adds per step instead of 6 shuffles.  (b) The next step's source is
// loaded from shared memory one step ahead into registers.  (c) The tile
// keeps each group of 32 sources twice in a row (expand_tile_dup), so the 32
// steps read 32 consecutive rows from one base address with constant offsets.
// The expanded tile then needs 32 KB, so the TMA ring moves into dynamic
// shared memory.  ROT = 4: the same with two groups side by side.
template <int KI, int NT, int TJ, int NB, int UNRB, int ACC = 0, int ROT = 0>
__global__ void __launch_bounds__(NT, 1) force_pairs(const PairArgs a) {
  static_assert(KI % 2 == 0, "targets are processed in packed pairs");
  static_assert((KI * NT) % TJ == 0 && TJ % NB == 0, "tiles tile an i-block; batches tile a tile");
  constexpr int kGroups = ROT == 2 || ROT == 4 ? 2 : 1;  // rotation groups side by side
  static_assert(ROT == 0 || TJ % (32 * kGroups) == 0, "rotation groups of 32 sources tile a tile");
  constexpr int kShift = NB == 8 ? 2 : 1;  // lane l holds source l >> kShift of a batch
  constexpr int P = KI / 2;
  constexpr int NW = NT / 32;
  constexpr long long B = static_cast<long long>(KI) * NT;
  constexpr long long TB = B / TJ;
  constexpr bool kDup = ROT >= 3;  // duplicated-group tile (expand_tile_dup)

  __shared__ __align__(128) float4 raw_s[kDup ? 1 : 2 * TJ];  // TMA targets (ROT < 3)
  __shared__ __align__(128) float4 tile[kDup ? 4 * TJ : 2 * TJ];  // expanded sources
  __shared__ __align__(8) unsigned long long bar[2];
  extern __shared__ __align__(128) float4 pair_smem[];  // (ring) + [NW][3][TJ] (+ running sums)
  float4* const raw = kDup ? pair_smem : raw_s;  // [2][TJ]: the caller's rows
  float* const react_smem = reinterpret_cast<float*>(kDup ? pair_smem + 2 * TJ : pair_smem);
  auto red = reinterpret_cast<float(*)[3][TJ]>(react_smem);
  float2* const acc_s = reinterpret_cast<float2*>(react_smem + NW * 3 * TJ);  // ACC = 1
  auto acc_at = [&](int c, int p) -> float2& { return acc_s[(c * P + p) * NT + threadIdx.x]; };

  const int tid = threadIdx.x;
  allow_dependent_launch();
  wait_for_prior_grid();
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const long long c = blockIdx.x;
  const long long u_lo = a.u_base + unit_begin(a.units, a.grid, c);  // global unit index
  const long long count = unit_begin(a.units, a.grid, c + 1) - unit_begin(a.units, a.grid, c);
  const uint32_t bar0 = smem_u32(&bar[0]);
  const uint32_t raw0 = smem_u32(raw);
  constexpr uint32_t kRawStride = TJ * sizeof(float4);
  auto bar_of = [&](long long k) { return bar0 + static_cast<uint32_t>(k & 1) * 8u; };
  auto raw_of = [&](long long k) { return raw0 + static_cast<uint32_t>(k & 1) * kRawStride; };

  // block and tile of the CTA's first unit (largest I with units_before(I) <= u_lo)
  long long I0 = 0;
  {
    long long lo = 0, hi = a.nblocks - 1;
    while (lo < hi) {
      const long long mid = (lo + hi + 1) / 2;
      if (pair_units_before(mid, a.ntiles, TB) <= u_lo)
        lo = mid;
      else
        hi = mid - 1;
    }
    I0 = lo;
  }
  const long long t0 = TB * I0 + (u_lo - pair_units_before(I0, a.ntiles, TB));

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (count <= 0) return;

  // Thread 0 issues the copies in unit order with its own (block, tile) cursor.
  long long iss_I = I0, iss_t = t0;
  auto issue_next = [&](long long k) {
    if (k != a.withhold) {
      const long long j0 = iss_t * TJ;
      const uint32_t bytes =
          static_cast<uint32_t>(min(static_cast<long long>(TJ), a.n - j0)) * 16u;
      mbar_arrive_expect_tx(bar_of(k), bytes);
      bulk_copy_g2s(raw_of(k), a.pos + j0, bytes, bar_of(k));
    }
    if (++iss_t == a.ntiles) {
      ++iss_I;
      iss_t = TB * iss_I;
    }
  };
  if (tid == 0) issue_next(0);

  const float2 e2 = make_float2(a.eps2, a.eps2);
  float2 nx[P], ny[P], nz[P], nm[P], ax[P], ay[P], az[P];
  long long k = 0, I = I0, t = t0;
  bool timed_out = false;
  NBODY_PHASE_DECL;

  while (k < count) {
    const long long blk = I;
    const long long tb = t;
    const long long te = min(a.ntiles, tb + (count - k));
    const bool first_segment = (k == 0);

#pragma unroll
    for (int p = 0; p < P; ++p) {
      const long long i0 = blk * B + (2 * p) * NT + tid;
      const long long i1 = i0 + NT;
      const float4 q0 = a.pos[min(i0, static_cast<long long>(a.n - 1))];
      const float4 q1 = a.pos[min(i1, static_cast<long long>(a.n - 1))];
      nx[p] = make_float2(-q0.x, -q1.x);
      ny[p] = make_float2(-q0.y, -q1.y);
      nz[p] = make_float2(-q0.z, -q1.z);
      // targets past n exert no reaction
      nm[p] = make_float2(i0 < a.n ? -q0.w : 0.f, i1 < a.n ? -q1.w : 0.f);
      if constexpr (ACC == 1) {
        acc_at(0, p) = acc_at(1, p) = acc_at(2, p) = make_float2(0.f, 0.f);
      } else {
        ax[p] = ay[p] = az[p] = make_float2(0.f, 0.f);
      }
    }

    for (; t < te; ++t, ++k) {
      const int s = static_cast<int>(k & 1);
      NBODY_PHASE(kPhaseOther);
      const bool ok = mbar_wait_bounded(bar_of(k), static_cast<uint32_t>((k >> 1) & 1), a.timeout_ns);
      // As in force_tiled, and: every thread is done with the previous tile's
      // reaction sums in shared memory before they are rewritten.
      if (!__syncthreads_and(ok)) {
        timed_out = true;
        break;
      }
      NBODY_PHASE(kPhaseWait);
      if (tid == 0 && k + 1 < count) issue_next(k + 1);
      if constexpr (kDup)
        expand_tile_dup(raw + s * TJ, tile, TJ, NT, tid, static_cast<long long>(a.n) - t * TJ);
      else if constexpr (ROT >= 1)
        expand_tile_split(raw + s * TJ, tile, TJ, NT, tid, static_cast<long long>(a.n) - t * TJ);
      else
        (void)expand_tile(raw + s * TJ, tile, TJ, NT, tid, static_cast<long long>(a.n) - t * TJ, 0);
      __syncthreads();
      NBODY_PHASE(kPhaseExpand);

      float2 tx[P], ty[P], tz[P];
#pragma unroll
      for (int p = 0; p < P; ++p) tx[p] = ty[p] = tz[p] = make_float2(0.f, 0.f);
      const float4* src = tile;
      constexpr int kLo = ROT >= 1 ? 1 : 2;   // row of source j's first half: kLo * j
      constexpr int kHi = ROT >= 1 ? TJ : 1;  // its second half: kLo * j + kHi
      if (t < TB * (blk + 1)) {
        // a tile of the block itself: both sides of each pair, as in force_tiled
        if constexpr (kDup) {
          for (int g = 0; g < TJ; g += 32) {
#pragma unroll 2
            for (int j = 0; j < 32; ++j) {
              const float4 lo = src[2 * g + j];
              const float4 hi = src[2 * TJ + 2 * g + j];
#pragma unroll
              for (int p = 0; p < P; ++p)
                interact2(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                          make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p], nz[p],
                          e2, tx[p], ty[p], tz[p]);
            }
          }
        } else {
#pragma unroll 2
          for (int j = 0; j < TJ; ++j) {
            const float4 lo = src[kLo * j];
            const float4 hi = src[kLo * j + kHi];
#pragma unroll
            for (int p = 0; p < P; ++p)
              interact2(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w), make_float2(hi.x, hi.y),
                        make_float2(hi.z, hi.w), nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
          }
        }
        NBODY_PHASE(kPhaseOwn);
      } else {
        if constexpr (ROT == 3 || ROT == 4) {
          constexpr unsigned kAll = 0xffffffffu;
          const int from = (lane + 1) & 31;
          for (int g = 0; g < TJ; g += 32 * kGroups) {
            // rows of this lane's step-0 sources; step st reads st rows further
            const float4* lo0 = src + 2 * g + lane;
            const float4* hi0 = src + 2 * TJ + 2 * g + lane;
            float4 clo[kGroups], chi[kGroups];
            float bxs[kGroups], bys[kGroups], bzs[kGroups];
#pragma unroll
            for (int h = 0; h < kGroups; ++h) {
              clo[h] = lo0[64 * h];
              chi[h] = hi0[64 * h];
              bxs[h] = bys[h] = bzs[h] = 0.f;
            }
#pragma unroll UNRB
            for (int st = 0; st < 32; ++st) {
#pragma unroll
              for (int h = 0; h < kGroups; ++h) {
                const float4 lo = clo[h];
                const float4 hi = chi[h];
                if (st + 1 < 32) {  // the next step's source, one step ahead
                  clo[h] = lo0[64 * h + st + 1];
                  chi[h] = hi0[64 * h + st + 1];
                }
                // this source's sum over the lanes before, from lane + 1
                bxs[h] = __shfl_sync(kAll, bxs[h], from);
                bys[h] = __shfl_sync(kAll, bys[h], from);
                bzs[h] = __shfl_sync(kAll, bzs[h], from);
                float2 bx = make_float2(bxs[h], 0.f), by = make_float2(bys[h], 0.f),
                       bz = make_float2(bzs[h], 0.f);
#pragma unroll
                for (int p = 0; p < P; ++p)
                  interact2_pair(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                                 make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p],
                                 nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
                bxs[h] = bx.x + bx.y;
                bys[h] = by.x + by.y;
                bzs[h] = bz.x + bz.y;
              }
            }
            // lane l now holds the warp's sum for source (l + 31) mod 32 of each group
#pragma unroll
            for (int h = 0; h < kGroups; ++h) {
              const int jj = g + 32 * h + ((lane + 31) & 31);
              red[warp][0][jj] = bxs[h];
              red[warp][1][jj] = bys[h];
              red[warp][2][jj] = bzs[h];
            }
          }
        } else if constexpr (ROT == 1) {
          constexpr unsigned kAll = 0xffffffffu;
          const int from = (lane + 1) & 31;
          for (int g = 0; g < TJ; g += 32) {
            float2 bx = make_float2(0.f, 0.f), by = bx, bz = bx;
#pragma unroll UNRB
            for (int st = 0; st < 32; ++st) {
              const int j = g + ((lane + st) & 31);
              const float4 lo = src[j];
              const float4 hi = src[TJ + j];
              bx.x = __shfl_sync(kAll, bx.x, from);
              bx.y = __shfl_sync(kAll, bx.y, from);
              by.x = __shfl_sync(kAll, by.x, from);
              by.y = __shfl_sync(kAll, by.y, from);
              bz.x = __shfl_sync(kAll, bz.x, from);
              bz.y = __shfl_sync(kAll, bz.y, from);
#pragma unroll
              for (int p = 0; p < P; ++p)
                interact2_pair(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                               make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p],
                               nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
            }
            const int jj = g + ((lane + 31) & 31);
            red[warp][0][jj] = bx.x + bx.y;
            red[warp][1][jj] = by.x + by.y;
            red[warp][2][jj] = bz.x + bz.y;
          }
        } else if constexpr (ROT == 2) {
          // two groups of 32 sources rotate side by side: two independent
          // reaction sums per lane and step
          constexpr unsigned kAll = 0xffffffffu;
          const int from = (lane + 1) & 31;
          for (int g = 0; g < TJ; g += 64) {
            float2 bx0 = make_float2(0.f, 0.f), by0 = bx0, bz0 = bx0;
            float2 bx1 = bx0, by1 = bx0, bz1 = bx0;
#pragma unroll UNRB
            for (int st = 0; st < 32; ++st) {
              const int j = g + ((lane + st) & 31);
              const float4 lo0 = src[j];
              const float4 hi0 = src[TJ + j];
              const float4 lo1 = src[j + 32];
              const float4 hi1 = src[TJ + j + 32];
              bx0.x = __shfl_sync(kAll, bx0.x, from);
              bx0.y = __shfl_sync(kAll, bx0.y, from);
              by0.x = __shfl_sync(kAll, by0.x, from);
              by0.y = __shfl_sync(kAll, by0.y, from);
              bz0.x = __shfl_sync(kAll, bz0.x, from);
              bz0.y = __shfl_sync(kAll, bz0.y, from);
              bx1.x = __shfl_sync(kAll, bx1.x, from);
              bx1.y = __shfl_sync(kAll, bx1.y, from);
              by1.x = __shfl_sync(kAll, by1.x, from);
              by1.y = __shfl_sync(kAll, by1.y, from);
              bz1.x = __shfl_sync(kAll, bz1.x, from);
              bz1.y = __shfl_sync(kAll, bz1.y, from);
#pragma unroll
              for (int p = 0; p < P; ++p) {
                interact2_pair(make_float2(lo0.x, lo0.y), make_float2(lo0.z, lo0.w),
                               make_float2(hi0.x, hi0.y), make_float2(hi0.z, hi0.w), nx[p],
                               ny[p], nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx0, by0, bz0);
                interact2_pair(make_float2(lo1.x, lo1.y), make_float2(lo1.z, lo1.w),
                               make_float2(hi1.x, hi1.y), make_float2(hi1.z, hi1.w), nx[p],
                               ny[p], nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx1, by1, bz1);
              }
            }
            const int jj = g + ((lane + 31) & 31);
            red[warp][0][jj] = bx0.x + bx0.y;
            red[warp][1][jj] = by0.x + by0.y;
            red[warp][2][jj] = bz0.x + bz0.y;
            red[warp][0][jj + 32] = bx1.x + bx1.y;
            red[warp][1][jj + 32] = by1.x + by1.y;
            red[warp][2][jj + 32] = bz1.x + bz1.y;
          }
        } else {
#pragma unroll UNRB
          for (int b0 = 0; b0 < TJ; b0 += NB) {
            float vx[NB], vy[NB], vz[NB];
#pragma unroll
            for (int q = 0; q < NB; ++q) {
              const float4 lo = src[2 * (b0 + q)];
              const float4 hi = src[2 * (b0 + q) + 1];
              float2 bx = make_float2(0.f, 0.f), by = bx, bz = bx;
#pragma unroll
              for (int p = 0; p < P; ++p)
                interact2_pair(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                               make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p],
                               nz[p], nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
              vx[q] = bx.x + bx.y;
              vy[q] = by.x + by.y;
              vz[q] = bz.x + bz.y;
            }
            const float3 r = reduce_scatter<NB>(vx, vy, vz, lane);
            if ((lane & ((1 << kShift) - 1)) == 0) {
              red[warp][0][b0 + (lane >> kShift)] = r.x;
              red[warp][1][b0 + (lane >> kShift)] = r.y;
              red[warp][2][b0 + (lane >> kShift)] = r.z;
            }
          }
        }
        NBODY_PHASE(kPhaseCross);
        __syncthreads();
        // the unit's reaction partial: the NW warps' sums in warp order
        const long long u = u_lo + k;
        for (int j = tid; j < TJ; j += NT) {
          float sx = 0.f, sy = 0.f, sz = 0.f;
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            sx += red[w][0][j];
            sy += red[w][1][j];
            sz += red[w][2][j];
          }
          if (NBODY_IN_BOUNDS(a.ctl, (u - a.u_base) * TJ + j, kCapReact))
            a.react[(u - a.u_base) * TJ + j] = make_float4(sx, sy, sz, 0.f);
        }
        NBODY_PHASE(kPhaseReduce);
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if constexpr (ACC == 1) {
          acc_at(0, p) = __fadd2_rn(acc_at(0, p), tx[p]);
          acc_at(1, p) = __fadd2_rn(acc_at(1, p), ty[p]);
          acc_at(2, p) = __fadd2_rn(acc_at(2, p), tz[p]);
        } else {
          ax[p] = __fadd2_rn(ax[p], tx[p]);
          ay[p] = __fadd2_rn(ay[p], ty[p]);
          az[p] = __fadd2_rn(az[p], tz[p]);
        }
      }
      NBODY_PHASE(kPhaseFold);
    }
    if (timed_out) break;

    const bool whole = (tb == TB * blk && te == a.ntiles);
    const long long slot = (c * 2 + (first_segment ? 0 : 1)) * B;
#pragma unroll
    for (int p = 0; p < P; ++p) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long long local = (2 * p + h) * NT + tid;
        const long long i = blk * B + local;
        if (i < a.n) {
          float2 sx2, sy2, sz2;
          if constexpr (ACC == 1) {
            sx2 = acc_at(0, p);
            sy2 = acc_at(1, p);
            sz2 = acc_at(2, p);
          } else {
            sx2 = ax[p];
            sy2 = ay[p];
            sz2 = az[p];
          }
          const float4 v = make_float4(h ? sx2.y : sx2.x, h ? sy2.y : sy2.x,
                                       h ? sz2.y : sz2.x, 0.f);
          if (whole && NBODY_IN_BOUNDS(a.ctl, i, kCapRows))
            a.act[i] = v;
          else if (!whole && NBODY_IN_BOUNDS(a.ctl, slot + local, kCapPartial))
            a.partial[slot + local] = v;
        }
      }
    }
    if (t == a.ntiles) {  // the segment reached the last tile: next block
      ++I;
      t = TB * I;
    }
  }

  NBODY_PHASE_FLUSH();
  if (timed_out && tid == 0) {
    atomicExch(a.ctl.status, static_cast<int>(NBODY_ETIMEOUT));
    if (k != a.withhold)
      (void)mbar_wait_bounded(bar_of(k), static_cast<uint32_t>((k >> 1) & 1), a.timeout_ns);
  }
}

// The pair kernel with one CTA barrier per tile (reaction scheme 3, running
// sums in registers).  The expanded tile and the warps' reaction rows are
// double-buffered: while the warps rotate tile k's sources over buffer k & 1,
// nothing else touches it; after its rotation each thread, before the tile's
// only barrier, (1) adds the warps' reaction rows of tile k - 1 (buffer
// (k - 1) & 1, complete since the previous barrier) and stores the unit's
// row, and (2) waits for the copy of tile k + 1 and expands it into buffer
// (k + 1) & 1 (last read by tile k - 1's rotation).  The barrier then
// publishes tile k + 1 and frees the rows of tile k - 1; the copy of tile
// k + 3 is issued into the ring stage tile k + 1 has left.  Sums and their
// order are those of force_pairs with the same scheme.
template <int KI, int NT, int TJ, int UNRB>
__global__ void __launch_bounds__(NT, 1) force_pairs_pipe(const PairArgs a) {
  static_assert(KI % 2 == 0, "targets are processed in packed pairs");
  static_assert((KI * NT) % TJ == 0 && TJ % 32 == 0, "tiles tile an i-block; groups tile a tile");
  constexpr int P = KI / 2;
  constexpr int NW = NT / 32;
  constexpr long long B = static_cast<long long>(KI) * NT;
  constexpr long long TB = B / TJ;

  extern __shared__ __align__(128) float4 pipe_smem[];
  float4* const raw = pipe_smem;             // [2][TJ]: the caller's rows (TMA targets)
  float4* const tiles = pipe_smem + 2 * TJ;  // [2][4 TJ]: expanded, duplicated groups
  float* const rows = reinterpret_cast<float*>(pipe_smem + 10 * TJ);  // [2][NW][3][TJ]
  __shared__ __align__(8) unsigned long long bar[2];
  auto red = [&](int buf, int w, int comp) { return rows + ((buf * NW + w) * 3 + comp) * TJ; };

  const int tid = threadIdx.x;
  allow_dependent_launch();
  wait_for_prior_grid();
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const long long c = blockIdx.x;
  const long long u_lo = a.u_base + unit_begin(a.units, a.grid, c);  // global unit index
  const long long count = unit_begin(a.units, a.grid, c + 1) - unit_begin(a.units, a.grid, c);
  const uint32_t bar0 = smem_u32(&bar[0]);
  const uint32_t raw0 = smem_u32(raw);
  constexpr uint32_t kRawStride = TJ * sizeof(float4);
  auto bar_of = [&](long long k) { return bar0 + static_cast<uint32_t>(k & 1) * 8u; };
  auto raw_of = [&](long long k) { return raw0 + static_cast<uint32_t>(k & 1) * kRawStride; };
  auto parity_of = [](long long k) { return static_cast<uint32_t>((k >> 1) & 1); };

  long long I0 = 0;  // block of the CTA's first unit
  {
    long long lo = 0, hi = a.nblocks - 1;
    while (lo < hi) {
      const long long mid = (lo + hi + 1) / 2;
      if (pair_units_before(mid, a.ntiles, TB) <= u_lo)
        lo = mid;
      else
        hi = mid - 1;
    }
    I0 = lo;
  }
  const long long t0 = TB * I0 + (u_lo - pair_units_before(I0, a.ntiles, TB));

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (count <= 0) return;

  // thread 0 issues the copies in unit order with its own cursor
  long long iss_I = I0, iss_t = t0, issued = 0;  // units issued so far
  auto issue_next = [&]() {
    const long long k = issued++;
    if (k != a.withhold) {
      const long long j0 = iss_t * TJ;
      const uint32_t bytes =
          static_cast<uint32_t>(min(static_cast<long long>(TJ), a.n - j0)) * 16u;
      mbar_arrive_expect_tx(bar_of(k), bytes);
      bulk_copy_g2s(raw_of(k), a.pos + j0, bytes, bar_of(k));
    }
    if (++iss_t == a.ntiles) {
      ++iss_I;
      iss_t = TB * iss_I;
    }
  };
  if (tid == 0) {
    issue_next();
    if (count > 1) issue_next();
  }

  const float2 e2 = make_float2(a.eps2, a.eps2);
  float2 nx[P], ny[P], nz[P], nm[P], ax[P], ay[P], az[P];
  bool timed_out = false;
  long long k = 0, I = I0, t = t0;

  // tile 0 into buffer 0
  {
    const bool ok = mbar_wait_bounded(bar_of(0), 0, a.timeout_ns);
    if (!__syncthreads_and(ok)) {
      timed_out = true;
    } else {
      expand_tile_dup(raw, tiles, TJ, NT, tid, static_cast<long long>(a.n) - t0 * TJ);
      __syncthreads();
      if (tid == 0 && count > 2) issue_next();  // into the stage tile 0 has left
    }
  }

  long long blk = -1, seg_tb = 0;  // the current segment's block and first tile
  bool seg_first = true;
  long long pending = -1;          // unit whose reaction rows wait to be added (-1: none)
  while (!timed_out) {
    if (I != blk) {  // a new segment: this block's targets
      blk = I;
      seg_tb = t;
      seg_first = (k == 0);
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const long long i0 = blk * B + (2 * p) * NT + tid;
        const long long i1 = i0 + NT;
        const float4 q0 = a.pos[min(i0, static_cast<long long>(a.n - 1))];
        const float4 q1 = a.pos[min(i1, static_cast<long long>(a.n - 1))];
        nx[p] = make_float2(-q0.x, -q1.x);
        ny[p] = make_float2(-q0.y, -q1.y);
        nz[p] = make_float2(-q0.z, -q1.z);
        nm[p] = make_float2(i0 < a.n ? -q0.w : 0.f, i1 < a.n ? -q1.w : 0.f);
        ax[p] = ay[p] = az[p] = make_float2(0.f, 0.f);
      }
    }
    const int b = static_cast<int>(k & 1);
    const float4* src = tiles + b * 4 * TJ;
    float2 tx[P], ty[P], tz[P];
#pragma unroll
    for (int p = 0; p < P; ++p) tx[p] = ty[p] = tz[p] = make_float2(0.f, 0.f);
    const bool cross = !(t < TB * (blk + 1));
    if (!cross) {
      // a tile of the block itself: both sides of each pair, as in force_tiled
      for (int g = 0; g < TJ; g += 32) {
#pragma unroll 2
        for (int j = 0; j < 32; ++j) {
          const float4 lo = src[2 * g + j];
          const float4 hi = src[2 * TJ + 2 * g + j];
#pragma unroll
          for (int p = 0; p < P; ++p)
            interact2(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w), make_float2(hi.x, hi.y),
                      make_float2(hi.z, hi.w), nx[p], ny[p], nz[p], e2, tx[p], ty[p], tz[p]);
        }
      }
    } else {
      constexpr unsigned kAll = 0xffffffffu;
      const int from = (lane + 1) & 31;
      float* const rx_row = red(b, warp, 0);
      float* const ry_row = red(b, warp, 1);
      float* const rz_row = red(b, warp, 2);
      for (int g = 0; g < TJ; g += 32) {
        const float4* lo0 = src + 2 * g + lane;
        const float4* hi0 = src + 2 * TJ + 2 * g + lane;
        float4 clo = lo0[0], chi = hi0[0];
        float bxs = 0.f, bys = 0.f, bzs = 0.f;
#pragma unroll UNRB
        for (int st = 0; st < 32; ++st) {
          const float4 lo = clo;
          const float4 hi = chi;
          if (st + 1 < 32) {  // the next step's source, one step ahead
            clo = lo0[st + 1];
            chi = hi0[st + 1];
          }
          bxs = __shfl_sync(kAll, bxs, from);
          bys = __shfl_sync(kAll, bys, from);
          bzs = __shfl_sync(kAll, bzs, from);
          float2 bx = make_float2(bxs, 0.f), by = make_float2(bys, 0.f), bz = make_float2(bzs, 0.f);
#pragma unroll
          for (int p = 0; p < P; ++p)
            interact2_pair(make_float2(lo.x, lo.y), make_float2(lo.z, lo.w),
                           make_float2(hi.x, hi.y), make_float2(hi.z, hi.w), nx[p], ny[p], nz[p],
                           nm[p], e2, tx[p], ty[p], tz[p], bx, by, bz);
          bxs = bx.x + bx.y;
          bys = by.x + by.y;
          bzs = bz.x + bz.y;
        }
        const int jj = g + ((lane + 31) & 31);
        rx_row[jj] = bxs;
        ry_row[jj] = bys;
        rz_row[jj] = bzs;
      }
    }
#pragma unroll
    for (int p = 0; p < P; ++p) {
      ax[p] = __fadd2_rn(ax[p], tx[p]);
      ay[p] = __fadd2_rn(ay[p], ty[p]);
      az[p] = __fadd2_rn(az[p], tz[p]);
    }

    // the unit after this one
    long long nI = I, nt = t + 1;
    if (nt == a.ntiles) {
      ++nI;
      nt = TB * nI;
    }
    const bool last = (k + 1 == count);
    if (last || nI != I) {  // the segment ends with this unit: its action sums
      const bool whole = (seg_tb == TB * blk && t + 1 == a.ntiles);
      const long long slot = (c * 2 + (seg_first ? 0 : 1)) * B;
#pragma unroll
      for (int p = 0; p < P; ++p) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const long long local = (2 * p + h) * NT + tid;
          const long long i = blk * B + local;
          if (i < a.n) {
            const float4 v = make_float4(h ? ax[p].y : ax[p].x, h ? ay[p].y : ay[p].x,
                                         h ? az[p].y : az[p].x, 0.f);
            if (whole && NBODY_IN_BOUNDS(a.ctl, i, kCapRows))
              a.act[i] = v;
            else if (!whole && NBODY_IN_BOUNDS(a.ctl, slot + local, kCapPartial))
              a.partial[slot + local] = v;
          }
        }
      }
    }

    // before the barrier: the previous cross tile's reaction row, then tile k + 1
    if (pending >= 0) {
      const int pb = b ^ 1;
      for (int j = tid; j < TJ; j += NT) {
        float sx = 0.f, sy = 0.f, sz = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          sx += red(pb, w, 0)[j];
          sy += red(pb, w, 1)[j];
          sz += red(pb, w, 2)[j];
        }
        if (NBODY_IN_BOUNDS(a.ctl, (pending - a.u_base) * TJ + j, kCapReact))
          a.react[(pending - a.u_base) * TJ + j] = make_float4(sx, sy, sz, 0.f);
      }
    }
    pending = cross ? u_lo + k : -1;
    if (last) break;
    bool ok = mbar_wait_bounded(bar_of(k + 1), parity_of(k + 1), a.timeout_ns);
    if (ok)
      expand_tile_dup(raw + ((k + 1) & 1) * TJ, tiles + ((k + 1) & 1) * 4 * TJ, TJ, NT, tid,
                      static_cast<long long>(a.n) - nt * TJ);
    if (!__syncthreads_and(ok)) {
      timed_out = true;
      ++k;  // the unit whose wait expired
      break;
    }
    if (tid == 0 && issued < count) issue_next();  // tile k + 3, into the stage k + 1 has left
    ++k;
    I = nI;
    t = nt;
  }

  if (!timed_out && pending >= 0) {
    __syncthreads();  // every warp's rows of the last tile are written
    const int pb = static_cast<int>(k & 1);
    for (int j = tid; j < TJ; j += NT) {
      float sx = 0.f, sy = 0.f, sz = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        sx += red(pb, w, 0)[j];
        sy += red(pb, w, 1)[j];
        sz += red(pb, w, 2)[j];
      }
      if (NBODY_IN_BOUNDS(a.ctl, (pending - a.u_base) * TJ + j, kCapReact))
        a.react[(pending - a.u_base) * TJ + j] = make_float4(sx, sy, sz, 0.f);
    }
  }
  if (timed_out && tid == 0) {
    atomicExch(a.ctl.status, static_cast<int>(NBODY_ETIMEOUT));
    // copies issued and not consumed may still be landing: a bounded wait for each
    for (long long q = k; q < issued; ++q)
      if (q != a.withhold) (void)mbar_wait_bounded(bar_of(q), parity_of(q), a.timeout_ns);
  }
}

// Second pass of force_pairs: one thread per body.  a_i = its action (whole
// or the stream-K partials of its block, in CTA order) + the reactions of
// its tile from blocks 0 .. I-1 in block order; then finish_body.
//
// Where the reaction sums of all units would not fit the scratch, the pass
// runs in chunks of consecutive i-blocks [I0, I1) (one force_pairs launch
// each, units numbered from u_base): accumulate_pairs then adds, for every
// body from block I0 on, its action (if its block is in the chunk) and the
// reactions from the chunk's blocks before its own to acc[i] (the first
// chunk stores instead of adding), and finish_accumulated finishes every body
// from acc.  The order of the additions is fixed by the chunking.
struct PairFinishArgs {
  const float4* act;
  const float4* partial;
  const float4* react;
  int n;
  long long block;  // B
  long long tj;
  long long ntiles;
  long long u_base;  // first unit of the launch whose sums are read
  long long units;   // its units
  long long grid;    // its CTAs
  long long I0, I1;  // its i-blocks (all of them for finish_pairs)
  Ctl ctl;
};

// Action sum of body i of block I, whose units all belong to the launch
// described by `a`: the whole-block row, or the partials of the CTAs that
// shared the block, in CTA order.
__device__ __forceinline__ float3 pair_action(const PairFinishArgs& a, long long i, long long I,
                                              long long tb) {
  const long long u0 = pair_units_before(I, a.ntiles, tb) - a.u_base;
  const long long u1 = pair_units_before(I + 1, a.ntiles, tb) - 1 - a.u_base;
  const long long c0 = unit_owner(a.units, a.grid, u0);
  const long long c1 = unit_owner(a.units, a.grid, u1);
  if (c0 == c1) {
    const float4 v = NBODY_IN_BOUNDS(a.ctl, i, kCapRows) ? a.act[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    return make_float3(v.x, v.y, v.z);
  }
  float sx = 0.f, sy = 0.f, sz = 0.f;
  const long long local = i - I * a.block;
  // The block's segment is CTA cc's first segment, except for CTA c0 when it
  // started before the block (every later CTA starts inside it).
  const int side0 = unit_begin(a.units, a.grid, c0) >= u0 ? 0 : 1;
  constexpr int D = 8;  // partials loaded eight CTAs at a time, added in CTA order
  for (long long c = c0; c <= c1; c += D) {
    float4 p[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const long long cc = c + d;
      p[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (cc <= c1) {
        const int side = cc == c0 ? side0 : 0;
        const long long at = (cc * 2 + side) * a.block + local;
        if (NBODY_IN_BOUNDS(a.ctl, at, kCapPartial)) p[d] = a.partial[at];
      }
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (c + d <= c1) {
        sx += p[d].x;
        sy += p[d].y;
        sz += p[d].z;
      }
    }
  }
  return make_float3(sx, sy, sz);
}

// Adds to (sx, sy, sz) the reactions on body i (tile t, row j) from the
// launch's blocks J in [a.I0, J1), in block order.  The rows are loaded
// eight blocks at a time before they are added (in the same order), so that
// a body waits for one memory latency per eight blocks, not per block.
__device__ __forceinline__ void pair_reactions(const PairFinishArgs& a, long long t, long long j,
                                               long long J1, long long tb, float& sx, float& sy,
                                               float& sz) {
  constexpr int D = 8;
  for (long long J0 = a.I0; J0 < J1; J0 += D) {
    float4 r[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const long long J = J0 + d;
      r[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (J < J1) {
        const long long at = (pair_units_before(J, a.ntiles, tb) + t - tb * J - a.u_base) * a.tj + j;
        if (NBODY_IN_BOUNDS(a.ctl, at, kCapReact)) r[d] = a.react[at];
      }
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (J0 + d < J1) {
        sx += r[d].x;
        sy += r[d].y;
        sz += r[d].z;
      }
    }
  }
}

// Body i's block I and tile t, and block / tile (32-bit: n < 2^31).
struct BodyBlock {
  long long I, t, j, tb;
};

__device__ __forceinline__ BodyBlock body_block(const PairFinishArgs& a, long long i) {
  const int ii = static_cast<int>(i);
  const int B = static_cast<int>(a.block), TJ = static_cast<int>(a.tj);
  const int t = ii / TJ;
  return BodyBlock{ii / B, t, ii - t * TJ, B / TJ};
}

__global__ void finish_pairs(const PairFinishArgs a, const Epilogue e) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  const BodyState b = load_body(e, i);
  const BodyBlock k = body_block(a, i);
  float3 s = pair_action(a, i, k.I, k.tb);
  pair_reactions(a, k.t, k.j, k.I, k.tb, s.x, s.y, s.z);
  finish_loaded(e, i, s.x, s.y, s.z, b);
}

__global__ void accumulate_pairs(const PairFinishArgs a, float4* acc, int first) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long i = a.I0 * a.block + static_cast<long long>(blockIdx.x) * blockDim.x +
                      threadIdx.x;
  if (i >= a.n) return;
  const BodyBlock k = body_block(a, i);
  float3 s = make_float3(0.f, 0.f, 0.f);
  if (k.I < a.I1) s = pair_action(a, i, k.I, k.tb);
  pair_reactions(a, k.t, k.j, min(k.I, a.I1), k.tb, s.x, s.y, s.z);
  if (!NBODY_IN_BOUNDS(a.ctl, i, kCapRows)) return;
  if (first) {
    acc[i] = make_float4(s.x, s.y, s.z, 0.f);
  } else {
    const float4 o = acc[i];
    acc[i] = make_float4(o.x + s.x, o.y + s.y, o.z + s.z, 0.f);
  }
}

__global__ void finish_accumulated(const float4* acc, int n, const Epilogue e) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (!NBODY_IN_BOUNDS(e.ctl, i, kCapRows)) return;
  const BodyState b = load_body(e, i);
  const float4 v = acc[i];
  finish_loaded(e, i, v.x, v.y, v.z, b);
}

// ---------------------------------------------------------------------------
// small-n warp-split kernel
// ---------------------------------------------------------------------------

struct WarpArgs {
  const float4* pos;  // n rows (x, y, z, m): targets and sources
  int n;
  float eps2;
  int slices;          // S: j slices (gridDim.y)
  long long slice_len; // sources per slice
  float4* partial;     // [S][n] when S > 1
};

// One level of a reduce-scatter over the 32 lanes of a warp: of the first
// 2H values, the lanes with bit H set keep the upper H, the others the lower
// H, each adding its partner's copy of the half it keeps.  After the levels
// H = 16, 8, 4, 2, 1, lane l holds in w[0] the warp's sum of value l, every
// sum formed in the same fixed order.
template <int H>
__device__ __forceinline__ void reduce_scatter_level(float (&w)[32], int lane) {
  const bool upper = (lane & H) != 0;
#pragma unroll
  for (int k = 0; k < H; ++k) {
    const float send = upper ? w[k] : w[k + H];
    const float keep = upper ? w[k + H] : w[k];
    w[k] = keep + __shfl_xor_sync(0xffffffffu, send, H);
  }
}

// U = 0: the thread's sources are loaded one loop iteration at a time.
// U > 0: in chunks of U, the next chunk's loads issued before the current
// chunk's arithmetic (software pipelining across the L2 latency); the last
// chunk is padded with zero-mass sources at the origin, which add exactly
// nothing.
// RS = 0: the lanes combine their 3 KW sums by a butterfly of shuffles (every
// lane ends with every sum); RS = 1: by a reduce-scatter (31 shuffles for up
// to 32 sums instead of 5 per sum; lane l ends with sum l).
template <int KW, int NW, int U = 0, int RS = 0>
__global__ void __launch_bounds__(NW * 32) force_warp(const WarpArgs a, const Epilogue e) {
  static_assert(KW % 2 == 0, "targets are processed in packed pairs");
  constexpr int P = KW / 2;
  constexpr int NTH = NW * 32;
  __shared__ float red[NW][3 * KW];

  const int tid = threadIdx.x;
  allow_dependent_launch();
  wait_for_prior_grid();
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const long long i_base = static_cast<long long>(blockIdx.x) * KW;
  const long long j_begin = static_cast<long long>(blockIdx.y) * a.slice_len;
  const long long j_end = min(static_cast<long long>(a.n), j_begin + a.slice_len);

  const float2 e2 = make_float2(a.eps2, a.eps2);
  float2 nx[P], ny[P], nz[P], ax[P], ay[P], az[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float4 q0 = a.pos[min(i_base + 2 * p, static_cast<long long>(a.n - 1))];
    const float4 q1 = a.pos[min(i_base + 2 * p + 1, static_cast<long long>(a.n - 1))];
    nx[p] = make_float2(-q0.x, -q1.x);
    ny[p] = make_float2(-q0.y, -q1.y);
    nz[p] = make_float2(-q0.z, -q1.z);
    ax[p] = ay[p] = az[p] = make_float2(0.f, 0.f);
  }
  if constexpr (U == 0) {
#pragma unroll 2
    for (long long j = j_begin + tid; j < j_end; j += NTH) {
      const float4 b = a.pos[j];
      const float2 X = make_float2(b.x, b.x);
      const float2 Y = make_float2(b.y, b.y);
      const float2 Z = make_float2(b.z, b.z);
      const float2 M = make_float2(b.w, b.w);
#pragma unroll
      for (int p = 0; p < P; ++p) interact2(X, Y, Z, M, nx[p], ny[p], nz[p], e2, ax[p], ay[p], az[p]);
    }
  } else {
    // this thread's sources: j_begin + tid + k NTH for k < cnt
    const long long first = j_begin + tid;
    const int cnt = first < j_end ? static_cast<int>((j_end - first + NTH - 1) / NTH) : 0;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 cur[U];
#pragma unroll
    for (int u = 0; u < U; ++u) cur[u] = u < cnt ? a.pos[first + static_cast<long long>(u) * NTH] : zero;
    for (int c = 0; c < cnt; c += U) {
      float4 nxt[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = c + U + u;
        nxt[u] = k < cnt ? a.pos[first + static_cast<long long>(k) * NTH] : zero;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float4 b = cur[u];
        const float2 X = make_float2(b.x, b.x);
        const float2 Y = make_float2(b.y, b.y);
        const float2 Z = make_float2(b.z, b.z);
        const float2 M = make_float2(b.w, b.w);
#pragma unroll
        for (int p = 0; p < P; ++p)
          interact2(X, Y, Z, M, nx[p], ny[p], nz[p], e2, ax[p], ay[p], az[p]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    }
  }

  // Combine the 32 lanes (a butterfly of shuffles, every lane ending with the
  // same bits; or a reduce-scatter), then the warps in ascending order
  // through shared memory.  Sum 3 t + c is component c of target t.
  if constexpr (RS == 0) {
    float v[3 * KW];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      v[6 * p + 0] = ax[p].x;
      v[6 * p + 1] = ay[p].x;
      v[6 * p + 2] = az[p].x;
      v[6 * p + 3] = ax[p].y;
      v[6 * p + 4] = ay[p].y;
      v[6 * p + 5] = az[p].y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int q = 0; q < 3 * KW; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 3 * KW; ++q) red[warp][q] = v[q];
    }
  } else {
    static_assert(3 * KW <= 32, "one sum per lane");
    float w[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) w[q] = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      w[6 * p + 0] = ax[p].x;
      w[6 * p + 1] = ay[p].x;
      w[6 * p + 2] = az[p].x;
      w[6 * p + 3] = ax[p].y;
      w[6 * p + 4] = ay[p].y;
      w[6 * p + 5] = az[p].y;
    }
    reduce_scatter_level<16>(w, lane);
    reduce_scatter_level<8>(w, lane);
    reduce_scatter_level<4>(w, lane);
    reduce_scatter_level<2>(w, lane);
    reduce_scatter_level<1>(w, lane);
    if (lane < 3 * KW) red[warp][lane] = w[0];
  }
  __syncthreads();
  if (tid < KW) {
    float sx = 0.f, sy = 0.f, sz = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      sx += red[w][3 * tid + 0];
      sy += red[w][3 * tid + 1];
      sz += red[w][3 * tid + 2];
    }
    const long long i = i_base + tid;
    if (i < a.n) {
      if (a.slices == 1)
        finish_body(e, i, sx, sy, sz);
      else
        if (NBODY_IN_BOUNDS(e.ctl, static_cast<long long>(blockIdx.y) * a.n + i, kCapPartial))
          a.partial[static_cast<long long>(blockIdx.y) * a.n + i] = make_float4(sx, sy, sz, 0.f);
    }
  }
}

// Second pass of the warp kernel: a_i = sum over slices s = 0..S-1 in order.
__global__ void finish_slices(const float4* __restrict__ partial, int n, int slices,
                              const Epilogue e) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const BodyState b = load_body(e, i);
  float sx = 0.f, sy = 0.f, sz = 0.f;
  constexpr int D = 8;  // slices loaded before they are added, in order
  for (int s0 = 0; s0 < slices; s0 += D) {
    float4 p[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const long long at = static_cast<long long>(s0 + d) * n + i;
      p[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + d < slices && NBODY_IN_BOUNDS(e.ctl, at, kCapPartial)) p[d] = partial[at];
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (s0 + d < slices) {
        sx += p[d].x;
        sy += p[d].y;
        sz += p[d].z;
      }
    }
  }
  finish_loaded(e, i, sx, sy, sz, b);
}

// The end-of-step positions of a pass that drifted into the other buffer of
// the ping-pong pair, copied into the caller's buffer once that pass has
// completed (a one-kernel pass cannot drift in place: another CTA may still
// read a position as a source).  Launched as a programmatic dependent of the
// pass, so the copy starts as soon as it ends.
__global__ void copy_rows(const float4* __restrict__ from, float4* __restrict__ to, long long n,
                          Ctl ctl) {
  wait_for_prior_grid();
  allow_dependent_launch();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    if (NBODY_IN_BOUNDS(ctl, i, kCapRows)) to[i] = from[i];
}

// ---------------------------------------------------------------------------
// point shaders as a kernel
// ---------------------------------------------------------------------------

struct RenderArgs {
  const float4* pos;  // n rows (x, y, z, m)
  float4* ndc;        // out: (x_ndc, y_ndc, z_ndc, 1)
  float4* rgba;       // out: (r, g, b, 1)
  long long n;
  float3 lim;        // (max_x, max_y, max_z)
  float3 scale;      // 2 / (max_c - (-max_c)) per component
  float min_w;
  float inv_range;   // 1 / (max_w - min_w)
  Ctl ctl;           // checked build: rows capacity (not used by the release kernel)
};

// Vertex shader: p_c = 2 (c - (-max_c)) / (max_c - (-max_c)) - 1 and
// weight = (m - min_w) / (max_w - min_w); fragment shader: mix(green, red,
// weight) = (weight, 1 - weight, 0) with alpha 1 ("CUDA N-Body Simulation"
// §4.3).  The per-draw reciprocals are taken once on the host, as a shader
// compiler folds uniforms; no clamping, as in the shaders.  Memory-bound:
// 16 bytes in and 32 bytes out per body; grid-stride over the SMs.
__global__ void render_points(const RenderArgs a) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n;
       i += stride) {
    const float4 b = a.pos[i];
    float4 p;
    p.x = fmaf(b.x + a.lim.x, a.scale.x, -1.0f);
    p.y = fmaf(b.y + a.lim.y, a.scale.y, -1.0f);
    p.z = fmaf(b.z + a.lim.z, a.scale.z, -1.0f);
    p.w = 1.0f;
    const float w = (b.w - a.min_w) * a.inv_range;
    a.ndc[i] = p;
    a.rgba[i] = make_float4(w, 1.0f - w, 0.0f, 1.0f);
  }
}

// ---------------------------------------------------------------------------
// 2-D cutoff neighbour list
// ---------------------------------------------------------------------------

struct NeighborArgs {
  const float* x;  // n source/target x
  const float* y;  // n source/target y
  int n;
  float cutoff_square;  // cutoff * cutoff, rounded to float
  int max_neighbors;    // MN: list slots per target
  int* nn;              // out: neighbours per target
  int* nl;              // out: nl[k * n + i], ascending, -1 past the count
  long long ntiles;
  Ctl ctl;
};

// All pairs in the page's single precision, every operation rounded
// separately (packed round-to-nearest intrinsics are never contracted):
//   x12 = x_j - x_i, y12 = y_j - y_i, d2 = x12 * x12 + y12 * y12,
//   neighbour when d2 < cutoff^2 and j != i.
// KI targets per thread as KI/2 packed pairs; sources staged as (x,x,y,y) in
// a two-buffer shared ring filled by plain loads (one source per thread per
// tile, prefetched into registers during the previous tile).  One CTA covers
// the whole j range of its targets, so every list is appended in ascending j.
// Hits are rare (a few per million pairs): U sources at a time are tested
// into registers, their minimum taken on the ALU pipe (FMNMX), and a single
// branch per group enters the exact per-pair check, which appends in
// ascending j.  Padding sources sit at +inf and padding targets are NaN;
// neither passes the per-pair test (the minimum ignores NaN, the test does
// not).
template <int KI, int NT, int U>
__global__ void __launch_bounds__(NT) neighbors_2d(const NeighborArgs a) {
  static_assert(KI % 2 == 0, "targets are processed in packed pairs");
  constexpr int P = KI / 2;
  constexpr int TJ = NT;
  static_assert(TJ % U == 0, "whole groups per tile");
  __shared__ __align__(16) float4 tile[2][TJ];

  const int tid = threadIdx.x;
  const long long base = static_cast<long long>(blockIdx.x) * KI * NT;
  const float c2 = a.cutoff_square;
  float2 nx[P], ny[P];
  int cnt[KI];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float v[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long i = base + (2 * p + h) * NT + tid;
      v[h][0] = i < a.n ? -a.x[i] : __int_as_float(0x7fc00000);
      v[h][1] = i < a.n ? -a.y[i] : __int_as_float(0x7fc00000);
      cnt[2 * p + h] = 0;
    }
    nx[p] = make_float2(v[0][0], v[1][0]);
    ny[p] = make_float2(v[0][1], v[1][1]);
  }

  long long jl = tid;
  float px = jl < a.n ? a.x[jl] : __int_as_float(0x7f800000);
  float py = jl < a.n ? a.y[jl] : __int_as_float(0x7f800000);
  for (long long t = 0; t < a.ntiles; ++t) {
    const int s = static_cast<int>(t & 1);
    tile[s][tid] = make_float4(px, px, py, py);
    __syncthreads();  // also: every thread is done with tile t-2 (same buffer)
    if (t + 1 < a.ntiles) {
      jl = (t + 1) * TJ + tid;
      px = jl < a.n ? a.x[jl] : __int_as_float(0x7f800000);
      py = jl < a.n ? a.y[jl] : __int_as_float(0x7f800000);
    }
    const long long j0 = t * TJ;
#pragma unroll 1
    for (int jg = 0; jg < TJ; jg += U) {
      float2 d2[U][P];
      float lo = __int_as_float(0x7f800000);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float4 b = tile[s][jg + u];
        const float2 X = make_float2(b.x, b.y);
        const float2 Y = make_float2(b.z, b.w);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const float2 dx = __fadd2_rn(X, nx[p]);
          const float2 dy = __fadd2_rn(Y, ny[p]);
          d2[u][p] = __fadd2_rn(__fmul2_rn(dx, dx), __fmul2_rn(dy, dy));
          lo = fminf(lo, fminf(d2[u][p].x, d2[u][p].y));
        }
      }
      if (lo < c2) {  // rare: some pair of the group is close
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long long j = j0 + jg + u;
#pragma unroll
          for (int p = 0; p < P; ++p) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const long long i = base + (2 * p + h) * NT + tid;
              if ((h ? d2[u][p].y : d2[u][p].x) < c2 && j != i) {
                int& c = cnt[2 * p + h];
                if (c < a.max_neighbors)
                  if (NBODY_IN_BOUNDS(a.ctl, static_cast<long long>(c) * a.n + i, kCapNeighbors))
                    a.nl[static_cast<long long>(c) * a.n + i] = static_cast<int>(j);
                ++c;
              }
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < KI; ++k) {
    const long long i = base + k * NT + tid;
    if (i < a.n) {
      a.nn[i] = cnt[k];
      for (int q = cnt[k]; q < a.max_neighbors; ++q)
        if (NBODY_IN_BOUNDS(a.ctl, static_cast<long long>(q) * a.n + i, kCapNeighbors))
          a.nl[static_cast<long long>(q) * a.n + i] = -1;
    }
  }
}

}  // namespace nbody
