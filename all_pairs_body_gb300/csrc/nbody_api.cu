// Host side of the all-pairs softened-gravity library: argument checks,
// launch plans, cached scratch and the exported C ABI declared in nbody.h.
//
// Nothing here computes physics: every step of the path runs in the kernels
// of nbody_kernels.cuh.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <algorithm>
#include <atomic>
#include <utility>
#include <vector>

#include "nbody.h"
#include "nbody_kernels.cuh"

namespace nbody {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per tile copy: only a fault gets near it
constexpr int kFinishThreads = 256;
// Forced one-sided TILED/SPLIT passes use the smallest tiled blocks up to this
// n, the large shapes above it (latency sweep over n).
constexpr long long kWarpMaxN = 24576;
// AUTO uses the warp kernel (one launch, one j slice) below this n and the
// pair kernel from it on: the pair path's floor is one unit of work per CTA
// (~110 us), which the warp kernel's time passes at about this size
// (measured over n = 6144 ... 24576).
constexpr long long kPairsMinN = 16384;

using TiledKernel = void (*)(const TiledArgs, const Epilogue);

struct TiledConfig {
  int ki, nt, tj;
  int form;  // 0: rsqrt loop; 1: mixed rsqrt/logarithmic loop (rsqrt for flagged tiles)
  TiledKernel kernel;
};

// Target bodies per thread, threads per CTA, sources per tile (kernel
// template: + minimum CTAs per SM for the register cap, + j unroll).  The
// release build holds the rows the plans use; the tuning build
// (NBODY_TUNING_TABLE) appends the other shapes and the mixed
// rsqrt/logarithmic loop, reachable through NBODY_TILED_CONFIG.
const TiledConfig kTiled[] = {
    {10, 256, 512, 0, force_tiled<10, 256, 512, 1, 2, 0, 0>},  // large n, 512-source tiles
    {10, 256, 256, 0, force_tiled<10, 256, 256, 1, 2, 0, 0>},  // large n, 256-source tiles
    {4, 128, 128, 0, force_tiled<4, 128, 128, 2, 4, 0, 0>},  // no-allocation entry point
    {2, 128, 64, 0, force_tiled<2, 128, 64, 4, 4, 0, 0>},  // forced one-sided paths at small n
#ifdef NBODY_TUNING_TABLE
    {8, 256, 256, 0, force_tiled<8, 256, 256, 1, 4, 0, 0>},
    {8, 128, 256, 0, force_tiled<8, 128, 256, 2, 4, 0, 0>},
    {8, 128, 256, 0, force_tiled<8, 128, 256, 3, 4, 0, 0>},
    {6, 256, 256, 0, force_tiled<6, 256, 256, 1, 4, 0, 0>},
    {4, 256, 256, 0, force_tiled<4, 256, 256, 2, 4, 0, 0>},
    {8, 256, 256, 0, force_tiled<8, 256, 256, 1, 2, 0, 0>},
    {8, 256, 256, 0, force_tiled<8, 256, 256, 1, 8, 0, 0>},
    {4, 256, 256, 0, force_tiled<4, 256, 256, 2, 8, 0, 0>},
    {6, 128, 256, 0, force_tiled<6, 128, 256, 3, 4, 0, 0>},
    {4, 128, 256, 0, force_tiled<4, 128, 256, 4, 4, 0, 0>},
    {8, 256, 256, 1, force_tiled<8, 256, 256, 1, 2, 1, 2>},
    {8, 256, 256, 1, force_tiled<8, 256, 256, 1, 2, 1, 3>},
    {8, 256, 256, 1, force_tiled<8, 256, 256, 1, 2, 1, 4>},
    {6, 256, 256, 1, force_tiled<6, 256, 256, 1, 2, 1, 2>},
    {8, 256, 256, 1, force_tiled<8, 256, 256, 1, 4, 1, 2>},
    {4, 256, 256, 1, force_tiled<4, 256, 256, 2, 4, 1, 1>},
    {6, 256, 256, 1, force_tiled<6, 256, 256, 1, 4, 1, 2>},
    {8, 128, 256, 1, force_tiled<8, 128, 256, 3, 2, 1, 2>},
#endif
};
constexpr int kNumTiled = sizeof(kTiled) / sizeof(kTiled[0]);
constexpr int kTiledLarge512 = 0, kTiledLarge256 = 1, kTiledNoAlloc = 2, kTiledSmall = 3;

using PairKernel = void (*)(const PairArgs);

struct PairConfig {
  int ki, nt, tj;
  PairKernel kernel;
  int acc;  // running sums in shared memory (the kernel's ACC)
  int rot;  // the kernel's ROT
  size_t smem() const { return pair_reduce_smem(ki, nt, tj, acc, rot); }  // dynamic shared memory
};

// Shapes of the pair-symmetric kernel (targets per thread, threads, tile;
// template: + reduction batch, batch or step unroll, running sums in shared
// memory, reaction scheme ROT).  The release build holds the plan's
// candidates: the lane rotation with one-step-ahead loads, scalar carries and
// duplicated groups (ROT 3; two groups side by side, ROT 4, for the smaller
// shapes), the first the default.  The tuning build (NBODY_TUNING_TABLE)
// appends the earlier schemes and shapes: batches reduced by a warp butterfly
// (ROT 0) and the plain lane rotation (ROT 1, 2), reachable through
// NBODY_PAIRS_CONFIG.
const PairConfig kPairs[] = {
    {16, 256, 512, force_pairs<16, 256, 512, 32, 8, 1, 3>, 1, 3},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 4, 0, 3>, 0, 3},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 4, 1, 3>, 1, 3},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 2, 1, 4>, 1, 4},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 2, 1, 4>, 1, 4},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 2, 0, 4>, 0, 4},
#ifdef NBODY_TUNING_TABLE
    {14, 256, 512, force_pairs<14, 256, 512, 32, 2, 1, 1>, 1, 1},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 4, 1, 1>, 1, 1},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 2, 1, 2>, 1, 2},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 2, 1, 2>, 1, 2},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 4, 0, 2>, 0, 2},
    {14, 256, 512, force_pairs<14, 256, 512, 16, 1, 1>, 1, 0},
    {12, 256, 512, force_pairs<12, 256, 512, 16, 1>, 0, 0},
    {10, 256, 512, force_pairs<10, 256, 512, 16, 1>, 0, 0},
    {10, 256, 512, force_pairs<10, 256, 512, 8, 1>, 0, 0},
    {8, 256, 512, force_pairs<8, 256, 512, 8, 1>, 0, 0},
    {8, 256, 256, force_pairs<8, 256, 256, 8, 1>, 0, 0},
    {10, 256, 256, force_pairs<10, 256, 256, 8, 1>, 0, 0},
    {8, 256, 128, force_pairs<8, 256, 128, 8, 1>, 0, 0},
    {8, 256, 512, force_pairs<8, 256, 512, 16, 1>, 0, 0},
    {8, 256, 512, force_pairs<8, 256, 512, 8, 2>, 0, 0},
    {6, 256, 512, force_pairs<6, 256, 512, 16, 1>, 0, 0},
    {8, 256, 256, force_pairs<8, 256, 256, 16, 1>, 0, 0},
    {6, 256, 512, force_pairs<6, 256, 512, 8, 2>, 0, 0},
    {10, 256, 640, force_pairs<10, 256, 640, 16, 1>, 0, 0},
    {10, 256, 320, force_pairs<10, 256, 320, 16, 1>, 0, 0},
    {12, 256, 384, force_pairs<12, 256, 384, 16, 1>, 0, 0},
    {14, 256, 512, force_pairs<14, 256, 512, 16, 1>, 0, 0},
    {12, 256, 512, force_pairs<12, 256, 512, 8, 1>, 0, 0},
    {16, 256, 512, force_pairs<16, 256, 512, 16, 1>, 0, 0},
    {12, 256, 256, force_pairs<12, 256, 256, 16, 1>, 0, 0},
    {12, 256, 512, force_pairs<12, 256, 512, 16, 1, 1>, 1, 0},
    {16, 256, 512, force_pairs<16, 256, 512, 16, 1, 1>, 1, 0},
    {10, 256, 512, force_pairs<10, 256, 512, 16, 1, 1>, 1, 0},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 4, 1, 1>, 1, 1},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 4, 0, 1>, 0, 1},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 4, 0, 1>, 0, 1},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 1, 1, 1>, 1, 1},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 4, 1, 1>, 1, 1},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 2, 1, 1>, 1, 1},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 2, 1, 1>, 1, 1},
    {18, 256, 512, force_pairs<18, 256, 512, 32, 2, 1, 1>, 1, 1},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 8, 1, 1>, 1, 1},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 4, 1, 1>, 1, 1},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 1, 1, 1>, 1, 1},
    {14, 256, 256, force_pairs<14, 256, 256, 32, 2, 1, 1>, 1, 1},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 2, 0, 1>, 0, 1},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 2, 0, 1>, 0, 1},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 2, 1, 1>, 1, 1},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 2, 1, 1>, 1, 1},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 2, 1, 1>, 1, 1},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 2, 0, 1>, 0, 1},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 2, 0, 1>, 0, 1},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 1, 1, 2>, 1, 2},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 2, 1, 2>, 1, 2},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 2, 1, 2>, 1, 2},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 4, 1, 2>, 1, 2},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 2, 0, 2>, 0, 2},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 4, 0, 2>, 0, 2},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 2, 0, 2>, 0, 2},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 2, 1, 2>, 1, 2},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 4, 1, 2>, 1, 2},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 4, 1, 2>, 1, 2},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 4, 1, 3>, 1, 3},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 2, 1, 3>, 1, 3},
    {10, 256, 512, force_pairs<10, 256, 512, 32, 4, 1, 3>, 1, 3},
    {8, 256, 512, force_pairs<8, 256, 512, 32, 4, 1, 3>, 1, 3},
    {8, 256, 256, force_pairs<8, 256, 256, 32, 4, 0, 3>, 0, 3},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 8, 1, 3>, 1, 3},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 4, 1, 3>, 1, 3},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 2, 1, 3>, 1, 3},
    {18, 256, 512, force_pairs<18, 256, 512, 32, 4, 1, 3>, 1, 3},
    {18, 256, 512, force_pairs<18, 256, 512, 32, 2, 1, 3>, 1, 3},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 2, 1, 3>, 1, 3},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 8, 1, 3>, 1, 3},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 4, 0, 3>, 0, 3},
    {16, 256, 512, force_pairs<16, 256, 512, 32, 1, 1, 3>, 1, 3},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 1, 1, 3>, 1, 3},
    {20, 256, 512, force_pairs<20, 256, 512, 32, 4, 1, 3>, 1, 3},
    {12, 256, 512, force_pairs<12, 256, 512, 32, 4, 1, 4>, 1, 4},
    {14, 256, 512, force_pairs<14, 256, 512, 32, 4, 1, 4>, 1, 4},
    {14, 256, 512, force_pairs_pipe<14, 256, 512, 4>, 0, 5},
    {14, 256, 512, force_pairs_pipe<14, 256, 512, 8>, 0, 5},
    {16, 256, 512, force_pairs_pipe<16, 256, 512, 4>, 0, 5},
    {16, 256, 512, force_pairs_pipe<16, 256, 512, 8>, 0, 5},
    {12, 256, 512, force_pairs_pipe<12, 256, 512, 4>, 0, 5},
    // 128-thread CTAs, two per SM: one CTA's barriers and reaction sums can
    // overlap the other's rotation loop
    {16, 128, 512, force_pairs<16, 128, 512, 32, 8, 1, 3>, 1, 3},
    {12, 128, 512, force_pairs<12, 128, 512, 32, 4, 1, 3>, 1, 3},
    {14, 128, 256, force_pairs<14, 128, 256, 32, 4, 0, 3>, 0, 3},
    {16, 128, 256, force_pairs<16, 128, 256, 32, 8, 1, 3>, 1, 3},
#endif
};
constexpr int kNumPairs = sizeof(kPairs) / sizeof(kPairs[0]);

using WarpKernel = void (*)(const WarpArgs, const Epilogue);

struct WarpConfig {
  int kw, nw, u;  // targets per CTA, warps per CTA, sources loaded ahead per thread
  WarpKernel kernel;
  int rs = 0;  // lanes combined by a reduce-scatter (1) or a butterfly (0)
};

// Shapes of the small-n warp kernel.  The release rows: 6 targets per CTA,
// 4 warps, 8 sources loaded ahead per thread, which matched or beat the other
// shapes at every n from 1000 to 16384 in a sweep of per-call time (4.7
// against 6.0 us at n = 1000 for the loop without loads ahead); and 8 targets
// per CTA, taken up to kWarpSmallN bodies (6.7 against 7.2 us per call at
// n = 1024, equal at 4097, slower above).  Both combine their lanes' sums by a
// reduce-scatter (1-6% faster per call than the butterfly from n = 1024 to
// 12288).  The tuning build appends the others.
const WarpConfig kWarps[] = {
    {6, 4, 8, force_warp<6, 4, 8, 1>, 1},
    {8, 4, 8, force_warp<8, 4, 8, 1>, 1},
#ifdef NBODY_TUNING_TABLE
    {6, 4, 8, force_warp<6, 4, 8, 0>},
    {4, 4, 0, force_warp<4, 4, 0>},   {4, 4, 4, force_warp<4, 4, 4>},
    {4, 4, 8, force_warp<4, 4, 8>},   {8, 4, 4, force_warp<8, 4, 4>},
    {8, 4, 8, force_warp<8, 4, 8>},   {8, 4, 16, force_warp<8, 4, 16>},
    {16, 4, 8, force_warp<16, 4, 8>}, {8, 8, 8, force_warp<8, 8, 8>},
    {4, 8, 8, force_warp<4, 8, 8>},   {12, 4, 8, force_warp<12, 4, 8>},
    {8, 2, 8, force_warp<8, 2, 8>},
    // lanes combined by a reduce-scatter instead of a butterfly
    {4, 4, 8, force_warp<4, 4, 8, 1>, 1},  {10, 4, 8, force_warp<10, 4, 8, 1>, 1},
#endif
};
constexpr int kNumWarps = sizeof(kWarps) / sizeof(kWarps[0]);


// The pair path keeps one reaction row of TJ float4 per unit; all of them
// come to about 16 N^2 / (2 B) bytes for B targets per i-block (2.5 GB at
// N = 2^20 and B = 3584).  Where they exceed this many bytes the pass runs
// in chunks of consecutive i-blocks whose rows fit, each chunk's reactions
// folded into a per-body accumulator before the next chunk reuses the rows;
// NBODY_PAIRS_MAX_BYTES overrides it.  The chunks cost nothing measurable
// (two more launches each and 32 bytes per body of accumulator traffic).
constexpr long long kPairsMaxBytes = 1LL << 30;

struct DeviceInfo {
  int sms = 0;
  int occupancy[kNumTiled] = {};
  int pair_occupancy[kNumPairs] = {};
};

struct Plan {
  int path = NBODY_PATH_AUTO;
  int cfg = 0;
  int threads = 0;
  long long block = 0;  // targets per CTA
  int tj = 0;           // sources per tile (tiled paths)
  long long ntiles = 0, nblocks = 0, units = 0;
  long long grid = 0;  // CTAs
  bool second_pass = false;
  int slices = 1;  // warp path
  long long slice_len = 0;
  int sms = 0;
  // pair path: chunks of i-blocks, chunk k = [chunk_start[k], chunk_start[k+1])
  std::vector<long long> chunk_start;
  long long grid_max = 0;     // CTAs of a full wave (each chunk: min(its units, this))
  long long chunk_units = 0;  // units of the largest chunk
  int chunks() const { return chunk_start.empty() ? 1 : static_cast<int>(chunk_start.size()) - 1; }
};

struct Buf {
  void* p = nullptr;
  size_t bytes = 0;
};

// Everything the library keeps for one (device, stream): the stream's status
// word, the scratch of its calls, and the plan of the last force pass it
// enqueued there (nbody_last_plan).
struct Scratch {
  Buf status;      // int: NBODY_OK until a kernel on this stream records a failure
  Buf pos_alt;     // end-of-step positions of a one-kernel pass (see step_impl)
  Buf partial;
  Buf act, react;  // pair path: whole-block action sums, per-unit reaction sums
  Buf pair_acc;    // pair path in chunks: per-body running sums
  Buf check[4];    // nbody_selftest_timeout_enqueue: its private problem
  Plan last;       // the last force pass enqueued on this stream
  bool has_last = false;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, uintptr_t>, Scratch> g_scratch;

// measurement hooks (nbody_profile_enable / nbody_profile_read), with a lock
// of their own: calls on several threads may record while another reads
struct Profile {
  std::atomic<bool> enabled{false};
  std::mutex mu;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> force_events;  // guarded by mu
  std::atomic<long long> kernel_launches{0};
};
Profile g_prof;

void count_launches(int k) { g_prof.kernel_launches.fetch_add(k, std::memory_order_relaxed); }

// Record an event on `st` (profiling only); returns nullptr when disabled.
cudaEvent_t prof_event(cudaStream_t st) {
  if (!g_prof.enabled.load(std::memory_order_relaxed)) return nullptr;
  cudaEvent_t ev = nullptr;
  if (cudaEventCreate(&ev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  cudaEventRecord(ev, st);
  return ev;
}

// Keep the events around one force launch for nbody_profile_read; a lone
// event (the other could not be created) is destroyed.
void record_force(cudaEvent_t e0, cudaEvent_t e1) {
  if (e0 != nullptr && e1 != nullptr) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.force_events.emplace_back(e0, e1);
    return;
  }
  if (e0 != nullptr) cudaEventDestroy(e0);
  if (e1 != nullptr) cudaEventDestroy(e1);
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// The control block of one launch: the stream's status word and, in the
// checked build, the capacities for the index checks: rows of the per-body
// arrays, float4 rows of `partial` and of the reaction sums, ints of the
// neighbour list.  They travel as a kernel argument, so calls on different
// streams never see each other's.  NBODY_BOUNDS_SHRINK=<slot> (rows, partial,
// react, neighbors) sets one capacity to 0 so that a test can see the checks
// fire; every access they stop is skipped, none goes out of bounds.
Ctl make_ctl(int* status, long long rows, long long partial, long long react,
             long long neighbors) {
  Ctl c;
  c.status = status;
#ifdef NBODY_BOUNDS_CHECK
  c.caps[kCapRows] = rows;
  c.caps[kCapPartial] = partial;
  c.caps[kCapReact] = react;
  c.caps[kCapNeighbors] = neighbors;
  if (const char* v = std::getenv("NBODY_BOUNDS_SHRINK")) {
    const char* names[kNumCaps] = {"rows", "partial", "react", "neighbors"};
    for (int k = 0; k < kNumCaps; ++k)
      if (std::strcmp(v, names[k]) == 0) c.caps[k] = 0;
  }
#else
  (void)rows, (void)partial, (void)react, (void)neighbors;
#endif
  return c;
}

long long float4_rows(const void* p, size_t bytes) {
  return p == nullptr ? 0 : static_cast<long long>(bytes / sizeof(float4));
}

long long env_int(const char* name, long long dflt) {
  const char* v = std::getenv(name);
  if (v == nullptr || v[0] == '\0') return dflt;
  return std::strtoll(v, nullptr, 10);
}

int device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return NBODY_ECUDA;
    }
    for (int c = 0; c < kNumTiled; ++c) {
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kTiled[c].kernel, kTiled[c].nt, 0) !=
          cudaSuccess) {
        cudaGetLastError();
        return NBODY_ECUDA;
      }
      d.occupancy[c] = occ > 0 ? occ : 1;
    }
    for (int c = 0; c < kNumPairs; ++c) {
      int occ = 0;
      const int smem = static_cast<int>(kPairs[c].smem());
      if (cudaFuncSetAttribute(kPairs[c].kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kPairs[c].kernel, kPairs[c].nt,
                                                        smem) != cudaSuccess) {
        cudaGetLastError();
        return NBODY_ECUDA;
      }
      d.pair_occupancy[c] = occ > 0 ? occ : 1;
    }
    it = g_devices.emplace(dev, d).first;
  }
  *out = it->second;
  return NBODY_OK;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  return NBODY_OK;
}

// --------------------------------------------------------------------------
// launch plans
// --------------------------------------------------------------------------

// The large-n shapes the stream-K plan chooses between, with their speed per
// interaction relative to the first, measured at n = 2^20 (force kernel 379.2
// against 389.8 ms).  The 512-source tiles are faster per interaction; the
// 256-source tiles cut the work into twice as many units, which wins when a
// CTA's share of units is small and its rounding up costs more.
struct LargeShape {
  int cfg;
  double speed;
};
constexpr LargeShape kLargeShapes[] = {{kTiledLarge512, 1.0}, {kTiledLarge256, 0.973}};

long long streamk_grid(long long units, const DeviceInfo& d, int cfg) {
  const long long per_sm = env_int("NBODY_CTAS_PER_SM", d.occupancy[cfg]);
  return std::min(units, static_cast<long long>(d.sms) * std::max(1LL, per_sm));
}

// Time model of a stream-K launch: the slowest CTA runs ceil(units / grid)
// units of tj sources each, at the shape's speed.  It matched the measured
// order of the two shapes at every n from 24577 to 131072.
int choose_large_shape(long long n, const DeviceInfo& d) {
  int best = -1;
  double best_cost = 0.0;
  for (const LargeShape& s : kLargeShapes) {
    const TiledConfig& tc = kTiled[s.cfg];
    const long long units =
        ceil_div(n, static_cast<long long>(tc.ki) * tc.nt) * ceil_div(n, tc.tj);
    const long long grid = streamk_grid(units, d, s.cfg);
    const double cost = static_cast<double>(ceil_div(units, grid)) * tc.tj / s.speed;
    if (best < 0 || cost < best_cost) {  // ties keep the earlier (faster) shape
      best = s.cfg;
      best_cost = cost;
    }
  }
  return best;
}

int auto_tiled_config(long long n, bool streamk, const DeviceInfo& d) {
  const long long forced = env_int("NBODY_TILED_CONFIG", -1);
  if (forced >= 0 && forced < kNumTiled) return static_cast<int>(forced);
  if (n <= kWarpMaxN) return kTiledSmall;  // forced TILED/SPLIT at small n: the smallest blocks
  return streamk ? choose_large_shape(n, d) : kLargeShapes[0].cfg;
}

bool streamk_needs_second_pass(long long units, long long grid, long long ntiles) {
  for (long long c = 1; c < grid; ++c)
    if (unit_begin(units, grid, c) % ntiles != 0) return true;
  return false;
}

void plan_tiled(long long n, int path, int split, const DeviceInfo& d, Plan* p) {
  const bool streamk = !(path == NBODY_PATH_TILED || (path == NBODY_PATH_SPLIT && split > 0));
  p->cfg = auto_tiled_config(n, streamk, d);
  const TiledConfig& tc = kTiled[p->cfg];
  p->threads = tc.nt;
  p->block = static_cast<long long>(tc.ki) * tc.nt;
  p->tj = tc.tj;
  p->ntiles = ceil_div(n, tc.tj);
  p->nblocks = ceil_div(n, p->block);
  p->units = p->nblocks * p->ntiles;
  if (path == NBODY_PATH_TILED) {
    p->grid = p->nblocks;
  } else if (path == NBODY_PATH_SPLIT && split > 0) {
    p->grid = std::min(p->units, p->nblocks * static_cast<long long>(split));
  } else {  // one full wave of CTAs, work divided evenly (stream-K)
    p->grid = streamk_grid(p->units, d, p->cfg);
  }
  p->second_pass = streamk_needs_second_pass(p->units, p->grid, p->ntiles);
}

// Up to this many bodies the warp kernel takes its second release row.
constexpr long long kWarpSmallN = 4096;

// The warp kernel's shape: NBODY_WARP_CONFIG forces a row, else row 1 up to
// kWarpSmallN bodies and row 0 above.
int warp_config(long long n) {
  const long long forced = env_int("NBODY_WARP_CONFIG", -1);
  if (forced >= 0 && forced < kNumWarps) return static_cast<int>(forced);
  return n <= kWarpSmallN ? 1 : 0;
}

void plan_warp(long long n, int split, const DeviceInfo& d, Plan* p) {
  p->cfg = warp_config(n);
  const WarpConfig& wc = kWarps[p->cfg];
  p->threads = wc.nw * 32;
  p->block = wc.kw;
  p->nblocks = ceil_div(n, wc.kw);
  // one slice by default: the single launch beats any split at every n the
  // warp kernel is chosen for (measured); split > 0 forces S slices
  long long s = split > 0 ? split : 1;
  (void)d;
  s = std::min(s, std::min(n, 65535LL));
  p->slice_len = ceil_div(n, s);
  p->slices = static_cast<int>(ceil_div(n, p->slice_len));
  p->grid = p->nblocks * p->slices;
  p->second_pass = p->slices > 1;
}

// Pair shapes the plan chooses between (the release rows), with their speed
// relative to the first: the model's work at n = 2^20 (the slowest CTA's
// ceil(units / grid) units of B x TJ pairs) per measured second, force kernel
// 265.35, 265.78, 272.55, 272.14, 277.52 and 275.72 ms per pass.  More
// targets per CTA are faster per pair; smaller blocks and tiles cut the work
// into more units, which wins when a CTA's share of units is small.
constexpr LargeShape kPairShapes[] = {{0, 1.0},    {1, 0.9977}, {2, 0.9726},
                                      {3, 0.9736}, {4, 0.9539}, {5, 0.9602}};

long long pair_units_of(long long n, const PairConfig& pc) {
  const long long block = static_cast<long long>(pc.ki) * pc.nt;
  return pair_units_before(ceil_div(n, block), ceil_div(n, pc.tj), block / pc.tj);
}

long long pair_grid(long long units, const DeviceInfo& d, int cfg) {
  const long long per_sm = env_int("NBODY_CTAS_PER_SM", d.pair_occupancy[cfg]);
  return std::min(units, static_cast<long long>(d.sms) * std::max(1LL, per_sm));
}

// The stream-K time model of choose_large_shape for the pair kernel: the
// slowest CTA runs ceil(units / grid) units of B x TJ pairs each.
int pair_config(long long n, const DeviceInfo& d) {
  const long long forced = env_int("NBODY_PAIRS_CONFIG", -1);
  if (forced >= 0 && forced < kNumPairs) return static_cast<int>(forced);
  int best = -1;
  double best_cost = 0.0;
  for (const LargeShape& s : kPairShapes) {
    const PairConfig& pc = kPairs[s.cfg];
    const long long units = pair_units_of(n, pc);
    const double cost = static_cast<double>(ceil_div(units, pair_grid(units, d, s.cfg))) *
                        pc.ki * pc.nt * pc.tj / s.speed;
    if (best < 0 || cost < best_cost) {  // ties keep the earlier (faster) shape
      best = s.cfg;
      best_cost = cost;
    }
  }
  return best;
}

void plan_pairs(long long n, const DeviceInfo& d, Plan* p) {
  p->cfg = pair_config(n, d);
  const PairConfig& pc = kPairs[p->cfg];
  p->threads = pc.nt;
  p->block = static_cast<long long>(pc.ki) * pc.nt;
  p->tj = pc.tj;
  p->ntiles = ceil_div(n, pc.tj);
  p->nblocks = ceil_div(n, p->block);
  const long long tb = p->block / pc.tj;
  p->units = pair_units_before(p->nblocks, p->ntiles, tb);
  p->grid_max = pair_grid(LLONG_MAX, d, p->cfg);
  p->grid = std::min(p->units, p->grid_max);
  p->second_pass = true;  // reactions always come from other CTAs
  // Chunks: consecutive i-blocks while their reaction rows fit the cap (one
  // block at least).  Block I has ntiles - TB * I units.
  const long long row = static_cast<long long>(pc.tj) * static_cast<long long>(sizeof(float4));
  const long long cap = std::max(row, env_int("NBODY_PAIRS_MAX_BYTES", kPairsMaxBytes));
  p->chunk_start.assign(1, 0);
  p->chunk_units = 0;
  long long acc = 0;
  for (long long I = 0; I < p->nblocks; ++I) {
    const long long u = p->ntiles - tb * I;
    if (acc > 0 && (acc + u) * row > cap) {
      p->chunk_start.push_back(I);
      p->chunk_units = std::max(p->chunk_units, acc);
      acc = 0;
    }
    acc += u;
  }
  p->chunk_start.push_back(p->nblocks);
  p->chunk_units = std::max(p->chunk_units, acc);
  if (p->chunks() == 1) p->chunk_start.clear();
}

// AUTO: the warp kernel below kPairsMinN, the pair path from it.
int auto_path(long long n) { return n < kPairsMinN ? NBODY_PATH_WARP : NBODY_PATH_PAIRS; }

int make_plan(long long n, int path, int split, int dev, Plan* p) {
  DeviceInfo d;
  const int st = device_info(dev, &d);
  if (st != NBODY_OK) return st;
  *p = Plan();
  p->sms = d.sms;
  int resolved = path;
  if (resolved == NBODY_PATH_AUTO) resolved = auto_path(n);
  p->path = resolved;
  if (resolved == NBODY_PATH_WARP)
    plan_warp(n, split, d, p);
  else if (resolved == NBODY_PATH_PAIRS)
    plan_pairs(n, d, p);
  else
    plan_tiled(n, resolved, path == NBODY_PATH_AUTO ? 0 : split, d, p);
  return NBODY_OK;
}

int launches_accel(const Plan& p) {
  if (p.path == NBODY_PATH_PAIRS && p.chunks() > 1) return 2 * p.chunks() + 1;
  return 1 + (p.second_pass ? 1 : 0);
}

int launches_step1(const Plan& p) { return launches_accel(p); }

// Bytes of reaction rows the pair path keeps (0 for the other paths).
long long react_bytes(const Plan& p) {
  if (p.path != NBODY_PATH_PAIRS) return 0;
  const long long rows = p.chunks() > 1 ? p.chunk_units : p.units;
  return rows * p.tj * static_cast<long long>(sizeof(float4));
}

// The fields nbody_plan and nbody_last_plan report, as far as len allows.
void write_plan(const Plan& p, int64_t* out, int len) {
  const int64_t v[] = {p.path,  p.grid,  p.threads, p.block,
                       p.tj,    p.ntiles, p.units,  p.second_pass ? 1 : 0,
                       launches_accel(p), launches_step1(p), p.sms, react_bytes(p), p.chunks()};
  const int nv = static_cast<int>(sizeof(v) / sizeof(v[0]));
  for (int k = 0; k < len && k < nv; ++k) out[k] = v[k];
}

// --------------------------------------------------------------------------
// scratch
// --------------------------------------------------------------------------

// Grow `b` to at least `bytes` with stream-ordered allocation on `st`: the
// old block is released after the stream's earlier work and the new one is
// ready for its later work, with no host synchronisation.  Host-side fault
// injection: NBODY_FAULT_ALLOC=1 fails every allocation, NBODY_FAULT_ALLOC=
// <kind> only those of that kind ("pairs": the pair path's reaction rows).
int ensure(Buf& b, size_t bytes, cudaStream_t st, const char* kind = "") {
  if (bytes == 0 || b.bytes >= bytes) return NBODY_OK;
  if (const char* v = std::getenv("NBODY_FAULT_ALLOC")) {
    if (std::strcmp(v, "1") == 0 || (kind[0] != '\0' && std::strcmp(v, kind) == 0))
      return NBODY_ENOMEM;
  }
  if (b.p != nullptr) {
    if (cudaFreeAsync(b.p, st) != cudaSuccess) {
      cudaGetLastError();
      return NBODY_ECUDA;
    }
    b.p = nullptr;
    b.bytes = 0;
  }
  if (cudaMallocAsync(&b.p, bytes, st) != cudaSuccess) {
    cudaGetLastError();
    b.p = nullptr;
    return NBODY_ENOMEM;
  }
  b.bytes = bytes;
  return NBODY_OK;
}

// The status word of (dev, st): allocated and zeroed on the stream's first
// use.  Called with g_mu held.
int ensure_status(Scratch& s, cudaStream_t st) {
  if (s.status.p != nullptr) return NBODY_OK;
  if (cudaMallocAsync(&s.status.p, sizeof(int4), st) != cudaSuccess) {
    cudaGetLastError();
    s.status.p = nullptr;
    return NBODY_ENOMEM;
  }
  s.status.bytes = sizeof(int4);
  if (cudaMemsetAsync(s.status.p, 0, sizeof(int4), st) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  return NBODY_OK;
}

Scratch& scratch_of(int dev, cudaStream_t st) {
  return g_scratch[std::make_pair(dev, reinterpret_cast<uintptr_t>(st))];
}

// True when every acceleration of a pass is completed by a later kernel than
// the ones that read the positions (the pair path's finishing passes, the
// warp path's slice sum): that kernel may drift the positions in place.
bool drift_in_place(const Plan& p) {
  return p.path == NBODY_PATH_PAIRS || (p.path == NBODY_PATH_WARP && p.second_pass);
}

int get_scratch(int dev, cudaStream_t st, const Plan& p, long long n, bool leapfrog,
                Scratch** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Scratch& s = scratch_of(dev, st);
  int rc = ensure_status(s, st);
  if (rc != NBODY_OK) return rc;
  if (p.path == NBODY_PATH_PAIRS) {
    const long long rows = p.chunks() > 1 ? p.chunk_units : p.units;
    rc = ensure(s.react, static_cast<size_t>(rows) * p.tj * sizeof(float4), st, "pairs");
    if (rc == NBODY_OK)
      rc = ensure(s.partial, static_cast<size_t>(p.grid) * 2 * p.block * sizeof(float4), st);
    if (rc == NBODY_OK) rc = ensure(s.act, static_cast<size_t>(n) * sizeof(float4), st);
    if (rc == NBODY_OK && p.chunks() > 1)
      rc = ensure(s.pair_acc, static_cast<size_t>(n) * sizeof(float4), st);
  } else if (p.path != NBODY_PATH_WARP) {
    if (p.second_pass)
      rc = ensure(s.partial, static_cast<size_t>(p.grid) * 2 * p.block * sizeof(float4), st);
  } else if (p.second_pass) {
    rc = ensure(s.partial, static_cast<size_t>(p.slices) * n * sizeof(float4), st);
  }
  if (rc == NBODY_OK && leapfrog && !drift_in_place(p))
    rc = ensure(s.pos_alt, static_cast<size_t>(n) * sizeof(float4), st);
  *out = &s;
  return rc;
}

// --------------------------------------------------------------------------
// argument checks
// --------------------------------------------------------------------------

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

bool overlaps_sized(const void* a, size_t abytes, const void* b, size_t bbytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bbytes && y < x + abytes;
}

int check_scalars(int64_t n, float eps2, int path, int split) {
  if (n < 0 || n > static_cast<int64_t>(INT32_MAX)) return NBODY_EINVAL;
  if (!std::isfinite(eps2) || !(eps2 > 0.0f)) return NBODY_EINVAL;
  if (path < NBODY_PATH_AUTO || path > NBODY_PATH_PAIRS) return NBODY_EINVAL;
  if (split < 0) return NBODY_EINVAL;
  return NBODY_OK;
}

int check_device_pointer(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_EINVAL;
  }
  if (at.type == cudaMemoryTypeManaged) return NBODY_OK;
  if (at.type != cudaMemoryTypeDevice || at.device != dev) return NBODY_EINVAL;
  return NBODY_OK;
}

int launch_status() {
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? NBODY_OK : NBODY_ECUDA;
}

// --------------------------------------------------------------------------
// launch sequences
// --------------------------------------------------------------------------

Epilogue make_epilogue(const float4* pos, void* accel, void* vel, float4* pos_next, float kick,
                       float dt, int layout, long long n) {
  Epilogue e;
  e.pos = pos;
  e.accel = static_cast<float*>(accel);
  e.vel = static_cast<float*>(vel);
  e.pos_next = pos_next;
  e.kick = kick;
  e.dt = dt;
  e.layout = layout;
  e.n = n;
  e.ctl = Ctl{};  // set by the launch
  return e;
}

// Bytes and alignment of one velocity/acceleration array in `layout`.
size_t vec_bytes(int layout, long long n) {
  return static_cast<size_t>(n) * (layout == kRows4 ? 16 : 12);
}

bool vec_aligned(const void* p, int layout) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return layout == kRows4 ? (a & 15u) == 0 : (a & 3u) == 0;
}

// The status word of the calling stream, for launches that need no other
// scratch (the point shaders, the neighbour list).
int stream_status(int dev, cudaStream_t st, int** status) {
  std::lock_guard<std::mutex> lk(g_mu);
  Scratch& s = scratch_of(dev, st);
  const int rc = ensure_status(s, st);
  *status = static_cast<int*>(s.status.p);
  return rc;
}

// Plan a force pass and get its scratch.  When the automatic plan chose the
// pair path and its reaction partials cannot be allocated, the one-sided
// stream-K plan (far less scratch) is taken instead; nbody_last_plan reports
// which plan a call used.
int plan_with_scratch(long long n, int path, int split, int dev, cudaStream_t st, bool leapfrog,
                      Plan* p, Scratch** s) {
  int rc = make_plan(n, path, split, dev, p);
  if (rc != NBODY_OK) return rc;
  rc = get_scratch(dev, st, *p, n, leapfrog, s);
  if (rc == NBODY_ENOMEM && path == NBODY_PATH_AUTO && p->path == NBODY_PATH_PAIRS) {
    if ((rc = make_plan(n, NBODY_PATH_SPLIT, 0, dev, p)) != NBODY_OK) return rc;
    rc = get_scratch(dev, st, *p, n, leapfrog, s);
  }
  if (rc == NBODY_OK) {
    std::lock_guard<std::mutex> lk(g_mu);
    (*s)->last = *p;
    (*s)->has_last = true;
  }
  return rc;
}

// Launches a force or second-pass kernel with programmatic stream
// serialization: when the kernel before it on `st` is one of the library's
// (which allow their dependents' launch as they start), this launch overlaps
// that kernel's tail; the kernel itself waits for the one before it to
// complete, with its writes visible, before it touches memory
// (wait_for_prior_grid).  After any other stream work it starts as a plain
// launch would.
template <typename... KArgs, typename... Args>
void launch_dependent(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem,
                      cudaStream_t st, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, args...);  // an error stays for launch_status()
}

// A per-body kernel (the finishing passes, copy_rows): `blocks` CTAs of
// kFinishThreads threads, launched as above.
template <typename... KArgs, typename... Args>
void launch_second_pass(void (*kernel)(KArgs...), long long blocks, cudaStream_t st,
                        Args... args) {
  launch_dependent(kernel, dim3(static_cast<unsigned>(blocks)), kFinishThreads, 0, st, args...);
}

// One force pass (plus its second pass): sources and targets `pos`, finished
// through `epi`, with the stream's status word and the scratch of `s`.
void launch_force(const Plan& p, const float4* pos, long long n, float eps2, const Scratch& s,
                  const Epilogue& epi_in, cudaStream_t st) {
  float4* partial = static_cast<float4*>(s.partial.p);
  const Ctl ctl = make_ctl(static_cast<int*>(s.status.p), n, float4_rows(s.partial.p, s.partial.bytes),
                           float4_rows(s.react.p, s.react.bytes), 0);
  Epilogue epi = epi_in;
  epi.ctl = ctl;
  if (p.path == NBODY_PATH_PAIRS) {
    const PairConfig& pc = kPairs[p.cfg];
    const long long tb = p.block / p.tj;
    float4* act = static_cast<float4*>(s.act.p);
    float4* react = static_cast<float4*>(s.react.p);
    // one launch over the i-blocks [I0, I1)
    auto force_chunk = [&](long long I0, long long I1, long long* u_base, long long* units,
                           long long* grid) {
      *u_base = pair_units_before(I0, p.ntiles, tb);
      *units = pair_units_before(I1, p.ntiles, tb) - *u_base;
      *grid = std::min(*units, p.grid_max);
      PairArgs a{pos,    static_cast<int>(n), eps2,    p.ntiles, p.nblocks,    *u_base,
                 *units, *grid,               act,     partial,  react,        kWaitLimitNs,
                 -1,     ctl};
      cudaEvent_t e0 = prof_event(st);
      launch_dependent(pc.kernel, dim3(static_cast<unsigned>(*grid)), p.threads, pc.smem(), st, a);
      cudaEvent_t e1 = prof_event(st);
      record_force(e0, e1);
    };
    count_launches(launches_accel(p));
    long long u_base = 0, units = 0, grid = 0;
    if (p.chunks() == 1) {
      force_chunk(0, p.nblocks, &u_base, &units, &grid);
      PairFinishArgs f{act,      partial, react, static_cast<int>(n), p.block, p.tj,
                       p.ntiles, u_base,  units, grid,                0,       p.nblocks,
                       ctl};
      launch_second_pass(finish_pairs, ceil_div(n, kFinishThreads), st, f, epi);
      return;
    }
    float4* acc = static_cast<float4*>(s.pair_acc.p);
    for (int k = 0; k < p.chunks(); ++k) {
      const long long I0 = p.chunk_start[k], I1 = p.chunk_start[k + 1];
      force_chunk(I0, I1, &u_base, &units, &grid);
      PairFinishArgs f{act,      partial, react, static_cast<int>(n), p.block, p.tj,
                       p.ntiles, u_base,  units, grid,                I0,      I1,
                       ctl};
      const long long bodies = n - I0 * p.block;
      launch_second_pass(accumulate_pairs, ceil_div(bodies, kFinishThreads), st, f, acc,
                         k == 0 ? 1 : 0);
    }
    launch_second_pass(finish_accumulated, ceil_div(n, kFinishThreads), st,
                       static_cast<const float4*>(acc), static_cast<int>(n), epi);
    return;
  }
  if (p.path == NBODY_PATH_WARP) {
    WarpArgs a{pos, static_cast<int>(n), eps2, p.slices, p.slice_len, partial};
    dim3 grid(static_cast<unsigned>(p.nblocks), static_cast<unsigned>(p.slices));
    cudaEvent_t e0 = prof_event(st);
    launch_dependent(kWarps[p.cfg].kernel, grid, p.threads, 0, st, a, epi);
    cudaEvent_t e1 = prof_event(st);
    record_force(e0, e1);
    count_launches(1 + (p.second_pass ? 1 : 0));
    if (p.second_pass) {
      const long long blocks = ceil_div(n, kFinishThreads);
      launch_second_pass(finish_slices, blocks, st, static_cast<const float4*>(partial),
                         static_cast<int>(n), p.slices, epi);
    }
    return;
  }
  TiledArgs a{pos, static_cast<int>(n), eps2, p.ntiles, p.units, p.grid, partial, kWaitLimitNs, -1};
  cudaEvent_t e0 = prof_event(st);
  launch_dependent(kTiled[p.cfg].kernel, dim3(static_cast<unsigned>(p.grid)), p.threads, 0, st,
                   a, epi);
  cudaEvent_t e1 = prof_event(st);
  record_force(e0, e1);
  count_launches(1 + (p.second_pass ? 1 : 0));
  if (p.second_pass) {
    StreamkFinishArgs f{partial, static_cast<int>(n), p.block, p.ntiles, p.units, p.grid};
    const long long blocks = ceil_div(n, kFinishThreads);
    launch_second_pass(finish_streamk, blocks, st, f, epi);
  }
}

int accel_impl(const float* pos_mass, float* accel, int64_t n, float eps2, int path, int split,
               int layout, cudaStream_t st) {
  int rc = check_scalars(n, eps2, path, split);
  if (rc != NBODY_OK) return rc;
  if (layout < kRows4 || layout > kBlocks3) return NBODY_EINVAL;
  if (n == 0) return NBODY_OK;
  if (pos_mass == nullptr || accel == nullptr) return NBODY_EINVAL;
  if (!aligned16(pos_mass) || !vec_aligned(accel, layout)) return NBODY_EINVAL;
  const size_t bytes = static_cast<size_t>(n) * sizeof(float4);
  const size_t vbytes = vec_bytes(layout, n);
  if (overlaps_sized(pos_mass, bytes, accel, vbytes)) return NBODY_EINVAL;
  int dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(pos_mass, dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(accel, dev)) != NBODY_OK) return rc;
  Plan p;
  Scratch* s = nullptr;
  if ((rc = plan_with_scratch(n, path, split, dev, st, false, &p, &s)) != NBODY_OK) return rc;

  const float4* pos = reinterpret_cast<const float4*>(pos_mass);
  const Epilogue epi = make_epilogue(pos, accel, nullptr, nullptr, 0.f, 0.f, layout, n);
  launch_force(p, pos, n, eps2, *s, epi, st);
  return launch_status();
}

// `steps` steps of either scheme, velocities and accelerations in `layout`.
//   kdk == false: the pages' step, one force pass per step: half kick with
//                 a(x(t)), drift ("CUDA N-Body Simulation" §1.3).
//   kdk == true:  kick-drift-kick, steps + 1 force passes: pass 0 half-kicks
//                 and drifts, passes 1..steps-1 kick by a full dt (closing
//                 half kick of one step fused with the opening half kick of
//                 the next) and drift, the last pass half-kicks only.
// Within a pass every acceleration uses the start-of-pass positions.  Where a
// later kernel than the position readers completes every acceleration (the
// pair path, the warp path with slices) it drifts the caller's positions in
// place.  Otherwise the new positions go to the other buffer of a ping-pong
// pair, and when an odd number of drifts leaves them there, copy_rows copies
// them into the caller's buffer right behind the last drift.
int step_impl(float* pos_mass, float* vel, float* accel, int64_t n, float eps2, float dt,
              int steps, int path, int split, int layout, bool kdk, cudaStream_t st) {
  int rc = check_scalars(n, eps2, path, split);
  if (rc != NBODY_OK) return rc;
  if (!std::isfinite(dt) || steps < 0) return NBODY_EINVAL;
  if (layout < kRows4 || layout > kBlocks3) return NBODY_EINVAL;
  if (n == 0 || steps == 0) return NBODY_OK;
  if (pos_mass == nullptr || vel == nullptr || accel == nullptr) return NBODY_EINVAL;
  if (!aligned16(pos_mass) || !vec_aligned(vel, layout) || !vec_aligned(accel, layout))
    return NBODY_EINVAL;
  const size_t bytes = static_cast<size_t>(n) * sizeof(float4);
  const size_t vbytes = vec_bytes(layout, n);
  if (overlaps_sized(pos_mass, bytes, accel, vbytes) || overlaps_sized(vel, vbytes, accel, vbytes) ||
      overlaps_sized(pos_mass, bytes, vel, vbytes))
    return NBODY_EINVAL;
  int dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(pos_mass, dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(vel, dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(accel, dev)) != NBODY_OK) return rc;
  Plan p;
  Scratch* s = nullptr;
  if ((rc = plan_with_scratch(n, path, split, dev, st, true, &p, &s)) != NBODY_OK) return rc;

  float4* user = reinterpret_cast<float4*>(pos_mass);
  float4* alt = drift_in_place(p) ? user : static_cast<float4*>(s->pos_alt.p);
  float4* cur = user;
  float4* nxt = alt;
  for (int k = 0; k < steps; ++k) {
    const float kick = (kdk && k > 0) ? dt : 0.5f * dt;
    const Epilogue epi = make_epilogue(cur, accel, vel, nxt, kick, dt, layout, n);
    launch_force(p, cur, n, eps2, *s, epi, st);
    std::swap(cur, nxt);
  }
  if (cur != user) {  // an odd number of drifts into the other buffer
    const long long blocks = std::min(ceil_div(n, kFinishThreads), static_cast<long long>(p.sms) * 8);
    count_launches(1);
    launch_second_pass(copy_rows, blocks, st, static_cast<const float4*>(cur), user,
                       static_cast<long long>(n), make_ctl(static_cast<int*>(s->status.p), n, 0, 0, 0));
    cur = user;
  }
  if (kdk) {
    const Epilogue last = make_epilogue(cur, accel, vel, nullptr, 0.5f * dt, dt, layout, n);
    launch_force(p, cur, n, eps2, *s, last, st);
  }
  return launch_status();
}

int render_impl(const float* pos_mass, float* ndc, float* rgba, int64_t n, float max_x,
                float max_y, float max_z, float min_w, float max_w, cudaStream_t st) {
  if (n < 0 || n > static_cast<int64_t>(INT32_MAX)) return NBODY_EINVAL;
  for (float lim : {max_x, max_y, max_z})
    if (!std::isfinite(lim) || !(lim > 0.0f)) return NBODY_EINVAL;
  if (!std::isfinite(min_w) || !std::isfinite(max_w) || !(max_w > min_w)) return NBODY_EINVAL;
  if (n == 0) return NBODY_OK;
  if (pos_mass == nullptr || ndc == nullptr || rgba == nullptr) return NBODY_EINVAL;
  if (!aligned16(pos_mass) || !aligned16(ndc) || !aligned16(rgba)) return NBODY_EINVAL;
  const size_t bytes = static_cast<size_t>(n) * sizeof(float4);
  if (overlaps(pos_mass, ndc, bytes) || overlaps(pos_mass, rgba, bytes) || overlaps(ndc, rgba, bytes))
    return NBODY_EINVAL;
  int rc = NBODY_OK, dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  for (const void* ptr : {static_cast<const void*>(pos_mass), static_cast<const void*>(ndc),
                          static_cast<const void*>(rgba)})
    if ((rc = check_device_pointer(ptr, dev)) != NBODY_OK) return rc;
  DeviceInfo d;
  if ((rc = device_info(dev, &d)) != NBODY_OK) return rc;
  int* status = nullptr;
  if ((rc = stream_status(dev, st, &status)) != NBODY_OK) return rc;
  RenderArgs a;
  a.pos = reinterpret_cast<const float4*>(pos_mass);
  a.ndc = reinterpret_cast<float4*>(ndc);
  a.rgba = reinterpret_cast<float4*>(rgba);
  a.n = n;
  a.lim = make_float3(max_x, max_y, max_z);
  a.scale = make_float3(static_cast<float>(2.0 / (2.0 * max_x)), static_cast<float>(2.0 / (2.0 * max_y)),
                        static_cast<float>(2.0 / (2.0 * max_z)));
  a.min_w = min_w;
  a.inv_range = static_cast<float>(1.0 / (static_cast<double>(max_w) - min_w));
  a.ctl = make_ctl(status, n, 0, 0, 0);
  const long long blocks = std::min(ceil_div(n, 256), static_cast<long long>(d.sms) * 8);
  count_launches(1);
  render_points<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return launch_status();
}

constexpr int kNeighborKI = 8;
constexpr int kNeighborNT = 128;
constexpr int kNeighborU = 4;

int neighbors_impl(const float* x, const float* y, int64_t n, float cutoff, int max_neighbors,
                   int32_t* nn, int32_t* nl, cudaStream_t st) {
  if (n < 0 || n > static_cast<int64_t>(INT32_MAX) || max_neighbors < 0) return NBODY_EINVAL;
  if (!std::isfinite(cutoff) || !(cutoff > 0.0f)) return NBODY_EINVAL;
  const float c2 = cutoff * cutoff;
  if (!(c2 >= 1.17549435e-38f) || !std::isfinite(c2)) return NBODY_EINVAL;  // normal, finite
  if (n == 0) return NBODY_OK;
  if (x == nullptr || y == nullptr || nn == nullptr) return NBODY_EINVAL;
  if (max_neighbors > 0 && nl == nullptr) return NBODY_EINVAL;
  const size_t b4 = static_cast<size_t>(n) * 4;
  const size_t bl = b4 * static_cast<size_t>(max_neighbors);
  for (const void* ptr : {static_cast<const void*>(x), static_cast<const void*>(y),
                          static_cast<const void*>(nn), static_cast<const void*>(nl)})
    if (ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 3u) != 0) return NBODY_EINVAL;
  if (overlaps(nn, x, b4) || overlaps(nn, y, b4)) return NBODY_EINVAL;
  if (max_neighbors > 0) {
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(nl), l1 = l0 + bl;
    for (const void* q : {static_cast<const void*>(x), static_cast<const void*>(y),
                          static_cast<const void*>(nn)}) {
      const uintptr_t q0 = reinterpret_cast<uintptr_t>(q), q1 = q0 + b4;
      if (q0 < l1 && l0 < q1) return NBODY_EINVAL;
    }
  }
  int rc = NBODY_OK, dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  for (const void* ptr : {static_cast<const void*>(x), static_cast<const void*>(y),
                          static_cast<const void*>(nn)})
    if ((rc = check_device_pointer(ptr, dev)) != NBODY_OK) return rc;
  if (max_neighbors > 0 && (rc = check_device_pointer(nl, dev)) != NBODY_OK) return rc;
  int* status = nullptr;
  if ((rc = stream_status(dev, st, &status)) != NBODY_OK) return rc;
  NeighborArgs a{x,  y,  static_cast<int>(n), c2, max_neighbors, nn, nl, ceil_div(n, kNeighborNT),
                 make_ctl(status, n, 0, 0, n * static_cast<long long>(max_neighbors))};
  const long long blocks = ceil_div(n, static_cast<long long>(kNeighborKI) * kNeighborNT);
  count_launches(1);
  neighbors_2d<kNeighborKI, kNeighborNT, kNeighborU>
      <<<static_cast<unsigned>(blocks), kNeighborNT, 0, st>>>(a);
  return launch_status();
}

}  // namespace
}  // namespace nbody

// ============================================================================
// no-allocation variant: scratch in one fixed device array
// ============================================================================

namespace nbody {
namespace {
// force_tiled<4, 128, 128, 2, 4, 0, 0>: 512 targets per i-block, 128-source tiles.
constexpr int kNoAllocCfg = kTiledNoAlloc;
constexpr long long kNoAllocMaxGrid = 384;
constexpr long long kNoAllocRows = kNoAllocMaxGrid * 2 * 512;  // partial sums: 6 MiB of float4
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  float4* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int* status = nullptr;      // device address of g_noalloc_status on this device
  int sms = 0;
  int occupancy = 0;
  bool called = false;        // a call was enqueued since nbody_sync last read the status
  uintptr_t last_stream = 0;  // the stream of the last call
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];  // fixed table: no allocation
}  // namespace
}  // namespace nbody

// Working memory of nbody_accel_noalloc: the partial sums of split i-blocks,
// and the status word its kernels report a failed bounded wait in.
static __device__ __align__(256) float4 g_noalloc_scratch[nbody::kNoAllocRows];
static __device__ int g_noalloc_status;

namespace nbody {
namespace {

// Once per device, with that device current: the device address of the
// array (its name in host code is only a host-side stand-in), SM count and
// the kernel's occupancy.
int noalloc_setup(int dev, NoAllocDevice* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr ||
        cudaGetSymbolAddress(&status, g_noalloc_status) != cudaSuccess || status == nullptr) {
      cudaGetLastError();
      return NBODY_ECUDA;
    }
    int sms = 0, occ = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kTiled[kNoAllocCfg].kernel,
                                                      kTiled[kNoAllocCfg].nt, 0) != cudaSuccess) {
      cudaGetLastError();
      return NBODY_ECUDA;
    }
    d.scratch = static_cast<float4*>(ptr);
    d.status = static_cast<int*>(status);
    d.sms = sms;
    d.occupancy = occ > 0 ? occ : 1;
    d.ready = true;
  }
  *out = d;
  return NBODY_OK;
}

int accel_noalloc_impl(const float* pos_mass, float* accel, int64_t n, float eps2,
                       cudaStream_t st) {
  int rc = check_scalars(n, eps2, NBODY_PATH_AUTO, 0);
  if (rc != NBODY_OK) return rc;
  if (n > NBODY_NOALLOC_MAX_N) return NBODY_EINVAL;
  if (n == 0) return NBODY_OK;
  if (pos_mass == nullptr || accel == nullptr) return NBODY_EINVAL;
  if (!aligned16(pos_mass) || !aligned16(accel)) return NBODY_EINVAL;
  if (overlaps(pos_mass, accel, static_cast<size_t>(n) * sizeof(float4))) return NBODY_EINVAL;
  int dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return NBODY_ECUDA;
  if ((rc = check_device_pointer(pos_mass, dev)) != NBODY_OK) return rc;
  if ((rc = check_device_pointer(accel, dev)) != NBODY_OK) return rc;
  NoAllocDevice d;
  if ((rc = noalloc_setup(dev, &d)) != NBODY_OK) return rc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_noalloc_dev[dev].called = true;
    g_noalloc_dev[dev].last_stream = reinterpret_cast<uintptr_t>(st);
  }

  const TiledConfig& tc = kTiled[kNoAllocCfg];
  const long long block = static_cast<long long>(tc.ki) * tc.nt;
  const long long ntiles = ceil_div(n, tc.tj);
  const long long units = ceil_div(n, block) * ntiles;
  // whole CTAs per SM so that every SM gets the same share, within the array
  const long long per_sm = std::max(1LL, std::min<long long>(d.occupancy, kNoAllocMaxGrid / d.sms));
  const long long grid = std::min(units, std::min(kNoAllocMaxGrid, per_sm * d.sms));
  const bool second = streamk_needs_second_pass(units, grid, ntiles);

  const float4* pos = reinterpret_cast<const float4*>(pos_mass);
  float4* partial = d.scratch;  // every slot a call reads, the same call writes first
  Epilogue epi = make_epilogue(pos, accel, nullptr, nullptr, 0.f, 0.f, kRows4, n);
  epi.ctl = make_ctl(d.status, n, kNoAllocRows, 0, 0);
  TiledArgs a{pos, static_cast<int>(n), eps2, ntiles, units, grid, partial, kWaitLimitNs, -1};
  tc.kernel<<<static_cast<unsigned>(grid), tc.nt, 0, st>>>(a, epi);
  if (second) {
    StreamkFinishArgs f{partial, static_cast<int>(n), block, ntiles, units, grid};
    finish_streamk<<<static_cast<unsigned>(ceil_div(n, kFinishThreads)), kFinishThreads, 0, st>>>(f,
                                                                                               epi);
  }
  return launch_status();
}

// The failure-detection check: one CTA of each tile-copying kernel whose
// first copy is never issued, with a wait limit of timeout_ms: the smallest
// one-sided tiled kernel over one i-block (which & 1), and the default pair
// kernel over two i-blocks (which & 2), on zero bodies (only the wait
// matters).  Its buffers are the stream's scratch; the expired waits go to
// the stream's status word.
int selftest_enqueue(int timeout_ms, cudaStream_t st, int which) {
  if (timeout_ms <= 0) return NBODY_EINVAL;
  int rc = NBODY_OK, dev = 0;
  if ((rc = current_device(&dev)) != NBODY_OK) return rc;
  DeviceInfo d;
  if ((rc = device_info(dev, &d)) != NBODY_OK) return rc;  // sets the kernels' attributes
  const uint64_t limit = static_cast<uint64_t>(timeout_ms) * 1000000ull;
  const TiledConfig& tc = kTiled[kTiledSmall];
  const PairConfig& pc = kPairs[0];
  const long long n1 = static_cast<long long>(tc.ki) * tc.nt;
  const long long pb = static_cast<long long>(pc.ki) * pc.nt;
  const long long n2 = 2 * pb;
  const long long nt2 = ceil_div(n2, pc.tj);
  const long long units2 = pair_units_before(2, nt2, pb / pc.tj);
  const size_t sizes[] = {static_cast<size_t>(n2) * sizeof(float4),  // positions (both)
                          static_cast<size_t>(n2) * sizeof(float4),  // accel / action
                          static_cast<size_t>(2 * pb) * sizeof(float4),
                          static_cast<size_t>(units2 * pc.tj) * sizeof(float4)};
  float4* buf[4] = {};
  int* status = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    Scratch& s = scratch_of(dev, st);
    if ((rc = ensure_status(s, st)) != NBODY_OK) return rc;
    for (int k = 0; k < 4; ++k) {
      if ((rc = ensure(s.check[k], sizes[k], st)) != NBODY_OK) return rc;
      buf[k] = static_cast<float4*>(s.check[k].p);
    }
    status = static_cast<int*>(s.status.p);
  }
  if (cudaMemsetAsync(buf[0], 0, sizes[0], st) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  const Ctl ctl = make_ctl(status, n2, 2 * pb, units2 * pc.tj, 0);
  if (which & 1) {
    TiledArgs a{buf[0], static_cast<int>(n1), 1.0f, ceil_div(n1, tc.tj), ceil_div(n1, tc.tj), 1,
                nullptr, limit, 0};
    Epilogue epi = make_epilogue(buf[0], buf[1], nullptr, nullptr, 0.f, 0.f, kRows4, n1);
    epi.ctl = ctl;
    tc.kernel<<<1, tc.nt, 0, st>>>(a, epi);
    if ((rc = launch_status()) != NBODY_OK) return rc;
  }
  if (which & 2) {
    PairArgs pa{buf[0], static_cast<int>(n2), 1.0f, nt2, 2, 0, units2, 1, buf[1], buf[2], buf[3],
                limit, 0, ctl};
    pc.kernel<<<1, pc.nt, pc.smem(), st>>>(pa);
    if ((rc = launch_status()) != NBODY_OK) return rc;
  }
  return NBODY_OK;
}

}  // namespace
}  // namespace nbody

// ============================================================================
// exported C ABI
// ============================================================================

extern "C" {

int nbody_accel(const float* pos_mass, float* accel, int64_t n, float eps2) {
  return nbody::accel_impl(pos_mass, accel, n, eps2, NBODY_PATH_AUTO, 0, nbody::kRows4, nullptr);
}

int nbody_accel_on_stream(const float* pos_mass, float* accel, int64_t n, float eps2,
                          void* cuda_stream) {
  return nbody::accel_impl(pos_mass, accel, n, eps2, NBODY_PATH_AUTO, 0, nbody::kRows4,
                           static_cast<cudaStream_t>(cuda_stream));
}

int nbody_accel_with(const float* pos_mass, float* accel, int64_t n, float eps2, int path,
                     int split, void* cuda_stream) {
  return nbody::accel_impl(pos_mass, accel, n, eps2, path, split, nbody::kRows4,
                           static_cast<cudaStream_t>(cuda_stream));
}

int nbody_accel_noalloc(const float* pos_mass, float* accel, int64_t n, float eps2,
                        void* cuda_stream) {
  return nbody::accel_noalloc_impl(pos_mass, accel, n, eps2, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_leapfrog_step(float* pos_mass, float* vel, float* accel, int64_t n, float eps2,
                        float dt, int steps) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, NBODY_PATH_AUTO, 0,
                          nbody::kRows4, false, nullptr);
}

int nbody_leapfrog_step_on_stream(float* pos_mass, float* vel, float* accel, int64_t n,
                                  float eps2, float dt, int steps, void* cuda_stream) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, NBODY_PATH_AUTO, 0,
                          nbody::kRows4, false, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_leapfrog_step_with(float* pos_mass, float* vel, float* accel, int64_t n, float eps2,
                             float dt, int steps, int path, int split, void* cuda_stream) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, path, split, nbody::kRows4,
                          false, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_leapfrog_kdk_on_stream(float* pos_mass, float* vel, float* accel, int64_t n, float eps2,
                                 float dt, int steps, void* cuda_stream) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, NBODY_PATH_AUTO, 0,
                          nbody::kRows4, true, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_leapfrog_kdk_with(float* pos_mass, float* vel, float* accel, int64_t n, float eps2,
                            float dt, int steps, int path, int split, void* cuda_stream) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, path, split, nbody::kRows4,
                          true, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_render_points(const float* pos_mass, float* ndc, float* rgba, int64_t n, float max_x,
                        float max_y, float max_z, float min_w, float max_w, void* cuda_stream) {
  return nbody::render_impl(pos_mass, ndc, rgba, n, max_x, max_y, max_z, min_w, max_w,
                            static_cast<cudaStream_t>(cuda_stream));
}

int nbody_neighbors_2d(const float* x, const float* y, int64_t n, float cutoff, int max_neighbors,
                       int32_t* nn, int32_t* nl, void* cuda_stream) {
  return nbody::neighbors_impl(x, y, n, cutoff, max_neighbors, nn, nl,
                               static_cast<cudaStream_t>(cuda_stream));
}

int nbody_accel_layout(const float* pos_mass, float* accel, int64_t n, float eps2, int layout,
                       void* cuda_stream) {
  return nbody::accel_impl(pos_mass, accel, n, eps2, NBODY_PATH_AUTO, 0, layout,
                           static_cast<cudaStream_t>(cuda_stream));
}

int nbody_leapfrog_step_layout(float* pos_mass, float* vel, float* accel, int64_t n, float eps2,
                               float dt, int steps, int layout, void* cuda_stream) {
  return nbody::step_impl(pos_mass, vel, accel, n, eps2, dt, steps, NBODY_PATH_AUTO, 0, layout,
                          false, static_cast<cudaStream_t>(cuda_stream));
}

int nbody_sync(void* cuda_stream) {
  using namespace nbody;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  int dev = 0;
  if (current_device(&dev) != NBODY_OK) return NBODY_ECUDA;
  // the status words this stream's kernels write: the stream's own, and the
  // no-allocation entry point's if its last call ran on this stream
  int* words[2] = {nullptr, nullptr};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_scratch.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(st)));
    if (it != g_scratch.end()) words[0] = static_cast<int*>(it->second.status.p);
    if (dev >= 0 && dev < kNoAllocMaxDevices) {
      NoAllocDevice& d = g_noalloc_dev[dev];
      if (d.ready && d.called && d.last_stream == reinterpret_cast<uintptr_t>(st)) {
        words[1] = d.status;
        d.called = false;
      }
    }
  }
  int status = NBODY_OK;
  for (int* w : words) {
    if (w == nullptr) continue;
    int v = 0;
    if (cudaMemcpyAsync(&v, w, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
      cudaGetLastError();
      return NBODY_ECUDA;
    }
    if (v != NBODY_OK) {
      if (status == NBODY_OK) status = v;
      if (cudaMemsetAsync(w, 0, sizeof(int), st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return NBODY_ECUDA;
      }
    }
  }
  return status;
}

int nbody_last_plan(void* cuda_stream, int64_t* out, int len) {
  using namespace nbody;
  if (out == nullptr && len > 0) return NBODY_EINVAL;
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != NBODY_OK) return rc;
  Plan p;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_scratch.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(cuda_stream)));
    if (it == g_scratch.end() || !it->second.has_last) return NBODY_EINVAL;
    p = it->second.last;
  }
  write_plan(p, out, len);
  return NBODY_OK;
}

int nbody_plan(int64_t n, int path, int split, int64_t* out, int len) {
  int rc = nbody::check_scalars(n, 1.0f, path, split);
  if (rc != NBODY_OK) return rc;
  if (out == nullptr && len > 0) return NBODY_EINVAL;
  int dev = 0;
  if ((rc = nbody::current_device(&dev)) != NBODY_OK) return rc;
  nbody::Plan p;
  if ((rc = nbody::make_plan(n > 0 ? n : 1, path, split, dev, &p)) != NBODY_OK) return rc;
  nbody::write_plan(p, out, len);
  return NBODY_OK;
}

int nbody_table(int which, int row, int64_t* out, int len) {
  using namespace nbody;
  if (out == nullptr && len > 0) return NBODY_EINVAL;
  int64_t v[6] = {};
  if (which == 0) {
    if (row < 0 || row >= kNumTiled) return NBODY_EINVAL;
    const TiledConfig& c = kTiled[row];
    const int64_t w[] = {kNumTiled, c.ki, c.nt, c.tj, c.form, 0};
    std::copy(w, w + 6, v);
  } else if (which == 1) {
    if (row < 0 || row >= kNumPairs) return NBODY_EINVAL;
    const PairConfig& c = kPairs[row];
    const int64_t w[] = {kNumPairs, c.ki, c.nt, c.tj, c.acc, c.rot};
    std::copy(w, w + 6, v);
  } else if (which == 2) {
    if (row < 0 || row >= kNumWarps) return NBODY_EINVAL;
    const WarpConfig& c = kWarps[row];
    const int64_t w[] = {kNumWarps, c.kw, c.nw * 32, c.u, c.rs, 0};
    std::copy(w, w + 6, v);
  } else {
    return NBODY_EINVAL;
  }
  for (int k = 0; k < len && k < 6; ++k) out[k] = v[k];
  return NBODY_OK;
}

int nbody_phase_read(int64_t* out, int len) {
#ifdef NBODY_PHASE_CLOCKS
  if (out == nullptr && len > 0) return NBODY_EINVAL;
  unsigned long long v[nbody::kNumPhases] = {};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(v, nbody::g_phase_cycles, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  const unsigned long long zero[nbody::kNumPhases] = {};
  if (cudaMemcpyToSymbol(nbody::g_phase_cycles, zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return NBODY_ECUDA;
  }
  for (int k = 0; k < len && k < nbody::kNumPhases; ++k) out[k] = static_cast<int64_t>(v[k]);
  return NBODY_OK;
#else
  (void)out, (void)len;
  return NBODY_EINVAL;  // a build without phase clocks
#endif
}

int nbody_profile_enable(int enable) {
  nbody::g_prof.enabled = enable != 0;
  return NBODY_OK;
}

int nbody_profile_read(double* force_ms, int64_t* force_launches, int64_t* kernel_launches) {
  std::lock_guard<std::mutex> lk(nbody::g_prof.mu);
  double total = 0.0;
  int rc = NBODY_OK;
  for (auto& ev : nbody::g_prof.force_events) {
    float ms = 0.f;
    if (cudaEventSynchronize(ev.second) != cudaSuccess ||
        cudaEventElapsedTime(&ms, ev.first, ev.second) != cudaSuccess) {
      cudaGetLastError();
      rc = NBODY_ECUDA;
    }
    total += ms;
    cudaEventDestroy(ev.first);
    cudaEventDestroy(ev.second);
  }
  if (force_ms != nullptr) *force_ms = total;
  if (force_launches != nullptr) *force_launches = static_cast<int64_t>(nbody::g_prof.force_events.size());
  const long long launched = nbody::g_prof.kernel_launches.exchange(0);
  if (kernel_launches != nullptr) *kernel_launches = launched;
  nbody::g_prof.force_events.clear();
  return rc;
}

const char* nbody_strerror(int status) {
  switch (status) {
    case NBODY_OK: return "ok";
    case NBODY_EINVAL: return "invalid argument";
    case NBODY_ENOMEM: return "scratch allocation failed";
    case NBODY_ECUDA: return "CUDA error (no usable device or a failed launch)";
    case NBODY_ETIMEOUT: return "a bounded device-side wait expired";
    case NBODY_EBOUNDS: return "a device-side index check failed (checked build)";
    default: return "unknown status";
  }
}

void nbody_release(void) {
  std::lock_guard<std::mutex> lk(nbody::g_mu);
  int prev = -1;
  const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
  for (auto& kv : nbody::g_scratch) {
    if (cudaSetDevice(kv.first.first) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    cudaDeviceSynchronize();
    nbody::Scratch& s = kv.second;
    for (nbody::Buf* b : {&s.status, &s.pos_alt, &s.partial, &s.act, &s.react, &s.pair_acc,
                          &s.check[0], &s.check[1], &s.check[2], &s.check[3]}) {
      if (b->p != nullptr) cudaFree(b->p);  // stream-ordered blocks; the device is idle
      b->p = nullptr;
      b->bytes = 0;
    }
  }
  nbody::g_scratch.clear();
  if (have_prev) cudaSetDevice(prev);
  cudaGetLastError();
}

int nbody_selftest_timeout_enqueue(int timeout_ms, void* cuda_stream) {
  return nbody::selftest_enqueue(timeout_ms, static_cast<cudaStream_t>(cuda_stream), 3);
}

int nbody_selftest_timeout(int timeout_ms, void* cuda_stream) {
  using namespace nbody;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // each kernel on its own, so that each must report the expired wait
  int rc1 = selftest_enqueue(timeout_ms, st, 1);
  if (rc1 == NBODY_OK) rc1 = nbody_sync(cuda_stream);
  int rc2 = selftest_enqueue(timeout_ms, st, 2);
  if (rc2 == NBODY_OK) rc2 = nbody_sync(cuda_stream);
  if (rc1 != NBODY_ETIMEOUT) return rc1;
  return rc2;
}

}  // extern "C"
