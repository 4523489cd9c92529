// C-ABI of the sharded-Linear library: argument checks, launch plans
// (tensor maps, tile space, chunk order, split-K), launches, the chunk
// scheduler and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/tp_fused.h"
#include "gemm_kernel.cuh"

using namespace tpf;

namespace {

// ------------------------------------------------------------------ constants

constexpr int kMaxP = 8;
constexpr int kPlanSMs = 152;            // SM count the split-K plan assumes (GB300)
constexpr size_t kStatusBytes = 256;     // workspace head: status word, padded
constexpr int kStagesWide = 4;           // 128x256 tiles: 48 KiB per stage
constexpr int kPairKChunks = PAIR_BK / 64;  // 64-wide K chunks per pair k-block (K-major operand maps)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// fp32-output mode: at most this many 64-deep k-blocks (K = 2048) are
// accumulated in one tensor-core accumulator; longer contractions are split
// (deterministic split-K) and the fp32 partials summed in split order.  The
// accumulator's own rounding grows with the number of k-steps it takes, and
// over K = 16384 it alone passes 1e-5 of max|Y|.
constexpr int64_t kPreciseKb = 32;
// An operand that every group of a launch reads through the same maps is
// loaded evict_last when it takes at most this much of the 129 MB L2.
constexpr int64_t kKeepBytes = 64ll << 20;
// Backward dX and dW share one launch whenever that is no slower by the
// makespan model while neither alone takes more than this many waves of CTA
// pairs; longer ones only for a predicted gain of at least 3 %.
constexpr int64_t kFuseWaves = 6;
// Pair launches whose contraction is at least this deep alternate its
// direction wave by wave (GemmParams::k_alternate).  From about 8192 on, the
// ~18 operand panels (256 rows x K) that a wave of 76 tiles reads outgrow
// the L2, so a forward-only wave finds none of the previous wave's panels
// left; running every other wave backwards re-reads the slices that wave
// touched last.  Measured: DRAM reads of the K = 16384 launches of the MLP
// step -8 %, of the sequence-parallel pair (K = 8192, 28672) -16 % and -5 %.
// On shallower contractions the panels a wave shares with the previous one
// stay in L2 either way, and a reversed wave no longer streams in step with
// the previous wave's stragglers (reads +2 to +5 %).
constexpr int64_t kKAlternateDepth = 8192;

// ------------------------------------------------------------------ small helpers

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device wait limit: TP_DEVICE_TIMEOUT_MS from the environment (read once),
// else 2 s; tp_debug_set(TP_DEBUG_TIMEOUT_MS, ...) overrides it.
std::atomic<uint64_t> g_timeout_override_ns{0};
std::atomic<int64_t> g_debug_drop_q{-1};
std::atomic<int64_t> g_debug_tile_mode{0};  // 0 auto, 1 single-CTA tiles only, 2 CTA pairs whenever possible
std::atomic<int64_t> g_debug_no_tail{0};    // 1: no k-slices in the last wave of pair launches
std::atomic<int64_t> g_debug_split_k{0};    // n > 0: split-K factor of launches below one wave
std::atomic<unsigned long long*> g_trace{nullptr};  // timeline trace buffer of the next launches
std::atomic<int64_t> g_trace_cap{0};
std::atomic<unsigned long long> g_launch_epoch{0};  // numbers every launch (slice counters)
std::atomic<int64_t> g_l2_hints{1};         // 1: L2 cache policies on operand loads and output stores
std::atomic<int64_t> g_tma_store{1};        // 1: staged epilogues leave shared memory by TMA store
std::atomic<int64_t> g_debug_no_fuse{0};    // 1: backward dX and dW always as two launches
std::atomic<int64_t> g_k_alternate{1};      // 1: deep contractions alternate their direction by wave

uint64_t device_timeout_ns() {
  const uint64_t o = g_timeout_override_ns.load();
  if (o != 0) return o;
  static uint64_t v = []() -> uint64_t {
    const char* e = std::getenv("TP_DEVICE_TIMEOUT_MS");
    if (e != nullptr) {
      const long long ms = std::atoll(e);
      if (ms > 0) return static_cast<uint64_t>(ms) * 1000000ull;
    }
    return kDefaultTimeoutNs;
  }();
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct DevInfo {
  int sms = 0;
  bool ok = false;
};

// The calling thread's current device, with that device's primary context
// made current on the thread.  A thread that has not yet made a CUDA call of
// its own (an autograd worker thread, a user's thread) may have no current
// context, and tensor-map encoding and launches from it then fail;
// cudaSetDevice binds the primary context.
tp_status bind_device(int* dev) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return TP_ERR_CUDA;
  if (cudaSetDevice(d) != cudaSuccess) return TP_ERR_CUDA;
  *dev = d;
  return TP_OK;
}

tp_status device_info(DevInfo* out) {
  int dev = 0;
  if (bind_device(&dev) != TP_OK) return TP_ERR_CUDA;
  // SM count of each device seen (0: not yet queried; -1: not an sm_103 device)
  static std::atomic<int> sm_count[64] = {};
  if (dev >= 0 && dev < 64) {
    const int c = sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      out->sms = c;
      out->ok = true;
      return TP_OK;
    }
    if (c < 0) return TP_ERR_ARCH;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TP_ERR_CUDA;
  if (major != 10 || minor != 3) {
    if (dev >= 0 && dev < 64) sm_count[dev].store(-1, std::memory_order_relaxed);
    return TP_ERR_ARCH;
  }
  if (dev >= 0 && dev < 64 && sms > 0) sm_count[dev].store(sms, std::memory_order_relaxed);
  out->sms = sms;
  out->ok = true;
  return TP_OK;
}

// bf16 tensor map with 128-byte swizzle over a row-major matrix with
// `inner` contiguous elements per row, `outer` rows and a row pitch of `ld`
// elements.
//   chunks == 0: 2-D map, box = 64 x box_outer;
//   chunks >= 1: 3-D map (64-element chunk, row, chunk index) with the chunk
//     index stepping 128 bytes along the row; box = 64 x box_outer x chunks,
//     which lands in shared memory as `chunks` consecutive 64-wide swizzled
//     sub-tiles -- one copy instead of `chunks`.  Needs inner % 64 == 0.
bool encode_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld,
                int box_outer, int chunks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  if (chunks == 0) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_outer)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (inner % 64 != 0) return false;
  cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(outer), static_cast<cuuint64_t>(inner / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, 128u};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_outer), static_cast<cuuint32_t>(chunks)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map of the TMA-store epilogue: `cols` x `rows` of a row-major
// matrix with a pitch of `ld` elements; boxes of 32 rows x 128 bytes with
// the 128-byte swizzle the staging buffer is written in.
bool encode_out_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld, bool f32) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * (f32 ? 4u : 2u)};
  cuuint32_t box[2] = {f32 ? 32u : 64u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D maps are used for a launch when every operand's contiguous extent is
// a multiple of 64 (K and N here); otherwise 2-D maps with one copy per
// 64-wide sub-tile.
inline bool use_3d(int64_t N, int64_t K) { return N % 64 == 0 && K % 64 == 0; }

// ------------------------------------------------------------------ kernel variants

enum Variant : int {
  V_KN = 0,    // A K-major, B MN-major (X . W forward), 128x256
  V_KK = 1,    // A K-major, B K-major (dY . W^T), 128x256
  V_MM = 2,    // A MN-major, B MN-major (X^T . dY weight gradient), 128x256
  V_SW_MK16,   // swapped: A = W (MN-major), B = tokens (K-major), token tile 16/32/64
  V_SW_MK32,
  V_SW_MK64,
  V_SW_KK16,   // swapped: A = W (K-major), B = tokens (K-major)
  V_SW_KK32,
  V_SW_KK64,
  V_KN2,       // CTA pairs, 256x256 tiles: X . W
  V_KK2,       //                           dY . W^T
  V_MM2,       //                           X^T . dY
};

// cudaFuncSetAttribute(k, MaxDynamicSharedMemorySize, bytes) once per kernel
// and device (`done` is the kernel's own bitmask of devices already set).
template <typename Kernel>
cudaError_t set_smem_once(Kernel k, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <bool A_MN, bool B_MN, bool TAIL>
cudaError_t launch_pair_t(const GemmParams& P, int clusters, cudaStream_t s) {
  using Cfg = PairCfg<A_MN, B_MN, PAIR_BK>;
  auto k = tp_gemm_pair_kernel<A_MN, B_MN, PAIR_BK, TAIL>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = set_smem_once(k, static_cast<int>(Cfg::SMEM_BYTES), smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // no more clusters than can be resident at once (persistent tiles)
  // (per device and instantiation; threads that race to fill it store the same value)
  static std::atomic<int> max_active[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    int m = max_active[dev].load(std::memory_order_relaxed);
    if (m == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0) {
        m = n;
        max_active[dev].store(n, std::memory_order_relaxed);
      }
    }
    if (m > 0 && clusters > m) {
      clusters = m;
      cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
  }
  cudaLaunchAttribute attr2[2] = {attr[0], {}};
  attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr2[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr2;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, k, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Two problems in one CTA-pair launch: dY.W^T (K-major A and B) units first,
// then X^T.dY (MN-major A and B) units.
cudaError_t launch_pair2(const PairLaunch2& L2, int clusters, cudaStream_t s) {
  using Cfg = PairCfg<false, false, PAIR_BK>;
  auto k = tp_gemm_pair2_kernel<false, false, true, true, PAIR_BK>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = set_smem_once(k, static_cast<int>(Cfg::SMEM_BYTES), smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static std::atomic<int> max_active[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    int m = max_active[dev].load(std::memory_order_relaxed);
    if (m == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0) {
        m = n;
        max_active[dev].store(n, std::memory_order_relaxed);
      }
    }
    if (m > 0 && clusters > m) {
      clusters = m;
      cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
  }
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, k, L2);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool A_MN, bool B_MN>
cudaError_t launch_pair(const GemmParams& P, int clusters, cudaStream_t s) {
  return P.tail_split > 1 ? launch_pair_t<A_MN, B_MN, true>(P, clusters, s)
                          : launch_pair_t<A_MN, B_MN, false>(P, clusters, s);
}

template <bool A_MN, bool B_MN, int BN, bool OUT_T, int STAGES>
cudaError_t launch_t(const GemmParams& P, int grid, cudaStream_t s) {
  using Cfg = GemmCfg<A_MN, B_MN, BN, OUT_T, STAGES>;
  auto k = tp_gemm_kernel<A_MN, B_MN, BN, OUT_T, STAGES>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = set_smem_once(k, static_cast<int>(Cfg::SMEM_BYTES), smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

constexpr int stages_for(int bn) { return std::min(12, (220 * 1024) / (128 * 128 + bn * 128)); }

cudaError_t launch_variant(int v, const GemmParams& P, int grid, cudaStream_t s) {
  switch (v) {
    case V_KN2: return launch_pair<false, true>(P, grid, s);
    case V_KK2: return launch_pair<false, false>(P, grid, s);
    case V_MM2: return launch_pair<true, true>(P, grid, s);
    case V_KN: return launch_t<false, true, 256, false, kStagesWide>(P, grid, s);
    case V_KK: return launch_t<false, false, 256, false, kStagesWide>(P, grid, s);
    case V_MM: return launch_t<true, true, 256, false, kStagesWide>(P, grid, s);
    case V_SW_MK16: return launch_t<true, false, 16, true, stages_for(16)>(P, grid, s);
    case V_SW_MK32: return launch_t<true, false, 32, true, stages_for(32)>(P, grid, s);
    case V_SW_MK64: return launch_t<true, false, 64, true, stages_for(64)>(P, grid, s);
    case V_SW_KK16: return launch_t<false, false, 16, true, stages_for(16)>(P, grid, s);
    case V_SW_KK32: return launch_t<false, false, 32, true, stages_for(32)>(P, grid, s);
    case V_SW_KK64: return launch_t<false, false, 64, true, stages_for(64)>(P, grid, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ launch shapes

// Shape of one GEMM launch; everything the split-K and workspace decisions
// need, computed from sizes alone (no pointers).
struct Shape {
  bool swap = false;     // operand-swapped: tokens are the GEMM N axis
  bool pair = false;     // 256x256 tiles on CTA pairs
  bool no_pair = false;  // the launch needs split-K (e.g. the unfused baseline)
  bool precise = false;  // fp32 outputs: cap the k-blocks per accumulator at kPreciseKb
  int bn = 256;          // tile N (token tile when swapped)
  int Gm = 1, Gn = 1, S = 1;
  int64_t rows_g = 0, cols_g = 0, kseg = 0;
  int64_t chunk_tiles = 1;
  int64_t m_tiles = 0, n_tiles = 0, units0 = 0, kb_total = 0;
  int n_split = 1;
  int64_t kb_per_split = 0;
  // CTA pairs: the tiles of a last partial wave run as tail_split k-slices
  int64_t tail_start = 0;
  int tail_split = 1;
  bool empty() const { return rows_g == 0 || cols_g == 0; }
  int64_t tail_tiles() const { return tail_split > 1 ? units0 - tail_start : 0; }
  size_t tail_cnt_bytes() const {
    return static_cast<size_t>((tail_tiles() * 2 * NUM_EPI_WARPS * 8 + 255) / 256 * 256);
  }
  size_t partial_bytes() const {
    if (tail_split > 1)  // counters, then one fp32 256 x 256 tile per slice
      return tail_cnt_bytes() + static_cast<size_t>(tail_tiles()) * tail_split * 256 * 256 * 4u;
    return n_split > 1 ? static_cast<size_t>(n_split) * Gm * Gn * rows_g * cols_g * 4u : 0;
  }
};

// Last partial wave of a CTA-pair launch: W full waves of C = #SM/2
// clusters leave R = units0 % C tiles for the last wave.  Cutting each of
// them into s k-slices makes R*s units that finish in ceil(R*s / C) / s of a
// wave instead of one; take the smallest s (up to 4) with the shortest tail,
// keeping at least 4 k-blocks per slice.
void plan_tail(Shape* s) {
  const int64_t C = kPlanSMs / 2;
  const int64_t R = s->units0 % C;
  const int64_t kb_pair = s->S * cdiv(s->kseg, PAIR_BK);
  if (s->units0 < C || R == 0 || g_debug_no_tail.load() != 0) return;
  double best = 1.0;
  int best_s = 1;
  for (int sp = 2; sp <= 4; ++sp) {
    if (kb_pair / sp < 4) break;
    const double t = static_cast<double>(cdiv(R * sp, C)) / sp;
    if (t < best - 1e-9) {
      best = t;
      best_s = sp;
    }
  }
  // slices cost a partial round trip and a heavier end of the launch; take
  // them where the saving is at least 6 % of the launch (few full waves)
  const double W = static_cast<double>(s->units0 / C);
  if (best_s > 1 && (1.0 - best) / (W + 1.0) >= 0.06) {
    s->tail_split = best_s;
    s->tail_start = s->units0 - R;
  }
}

// Planner option for one call: last-wave slices allowed (the default) or not.
thread_local bool t_plan_tails = true;

void finish_shape(Shape* s) {
  s->m_tiles = cdiv(s->rows_g, BM);
  s->n_tiles = cdiv(s->cols_g, s->bn);
  s->units0 = static_cast<int64_t>(s->Gm) * s->Gn * s->m_tiles * s->n_tiles;
  s->kb_total = s->S * cdiv(s->kseg, BK);
  s->n_split = 1;
  s->kb_per_split = s->kb_total;
  s->pair = false;
  s->tail_start = 0;
  s->tail_split = 1;
  if (s->units0 == 0 || s->kb_total == 0) return;
  // 256x256 tiles on CTA pairs when a group has at least 256 rows and the
  // pair tiles still fill the clusters; otherwise 128x256 tiles (with split-K
  // when there are too few of them).
  const int64_t mode = g_debug_tile_mode.load();
  const bool must_split = s->precise && s->kb_total > kPreciseKb;
  if (!s->swap && !s->no_pair && !must_split && mode != 1) {
    const int64_t pm = cdiv(s->rows_g, 2 * BM);
    const int64_t pu = static_cast<int64_t>(s->Gm) * s->Gn * pm * s->n_tiles;
    if (mode == 2 || (s->rows_g >= 2 * BM && pu >= kPlanSMs / 2)) {
      s->pair = true;
      s->m_tiles = pm;
      s->units0 = pu;
      s->chunk_tiles = cdiv(s->chunk_tiles, 2);
      if (t_plan_tails) plan_tail(s);
      return;
    }
  }
  if (s->units0 < kPlanSMs) {
    // Deterministic split-K, at least 4 k-blocks per split and at most 16
    // splits.  Every split adds an fp32 partial of the whole output to the
    // second stage's reads, and the second stage is a launch of its own: the
    // split is the largest that still runs all units in one wave.  A GEMM too
    // small to repay the second stage is not split.  Where one wave leaves
    // a quarter of the SMs idle on units of 256 k-blocks or more (skinny
    // calls over long contractions, bound by HBM), the split that fills the
    // SMs best over several waves keeps every SM streaming.
    int best = 1;
    for (int ns = 2; ns <= 16; ++ns) {
      if (s->kb_total / ns < 4 || s->units0 * ns > kPlanSMs) break;
      best = ns;
    }
    if (s->units0 * s->kb_total <= 256) {
      best = 1;
    } else if (s->kb_total / best >= 256 && 4 * s->units0 * best < 3 * kPlanSMs) {
      double best_eff = 0.0;
      best = 1;
      for (int ns = 1; ns <= 16; ++ns) {
        if (ns > 1 && s->kb_total / ns < 4) break;
        const int64_t u = s->units0 * ns;
        const double eff = static_cast<double>(u) / (cdiv(u, kPlanSMs) * kPlanSMs);
        if (eff > best_eff + 0.02) {
          best_eff = eff;
          best = ns;
        }
      }
    }
    const int64_t forced = g_debug_split_k.load();
    if (forced > 0) best = static_cast<int>(std::min<int64_t>(forced, s->kb_total));
    if (best > 1) {
      s->kb_per_split = cdiv(s->kb_total, best);
      s->n_split = static_cast<int>(cdiv(s->kb_total, s->kb_per_split));
    }
  }
  if (must_split && s->kb_per_split > kPreciseKb) {
    s->kb_per_split = kPreciseKb;
    s->n_split = static_cast<int>(cdiv(s->kb_total, kPreciseKb));
  }
}

// Chunk used by a call: 0 -> scheduler; clamp to M.
int64_t resolve_chunk(tp_op op, int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m) {
  if (chunk_m == 0) chunk_m = tp_choose_chunk_m(op, p, M, N, K);
  return std::max<int64_t>(1, std::min<int64_t>(chunk_m, std::max<int64_t>(M, 1)));
}

// Token-axis tiling of a chunk: swapped kernel below 128 rows.
void apply_chunk(Shape* s, int64_t chunk) {
  if (chunk < BM) {
    s->swap = true;
    s->bn = chunk <= 16 ? 16 : chunk <= 32 ? 32 : 64;
  } else {
    s->swap = false;
    s->bn = 256;
    s->chunk_tiles = cdiv(chunk, BM);
  }
}

// Shapes of the launches an op makes, in launch order.
std::vector<Shape> op_shapes(tp_op op, int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                             tp_dtype dt) {
  std::vector<Shape> v;
  const int64_t chunk = resolve_chunk(op, p, M, N, K, chunk_m);
  const int64_t Mp = (p > 0) ? M / p : 0;
  const bool precise = dt == TP_FP32;
  Shape s;
  s.precise = precise;
  auto tok = [&](int64_t rows_tok, int64_t other, int gtok, int goth) {
    // tokens along GEMM M (standard) or GEMM N (swapped)
    apply_chunk(&s, chunk);
    if (!s.swap) {
      s.rows_g = rows_tok; s.cols_g = other; s.Gm = gtok; s.Gn = goth;
    } else {
      s.rows_g = other; s.cols_g = rows_tok; s.Gm = goth; s.Gn = gtok;
    }
  };
  switch (op) {
    case TP_OP_ROW_AR:
      s.S = p; s.kseg = K; tok(M, N, 1, 1); break;
    case TP_OP_ROW_AR_UNFUSED:
      s.S = p; s.kseg = K; tok(M, N, 1, 1);
      s.no_pair = true;
      s.precise = false;  // one split per rank, as the per-rank GEMMs it stands for
      finish_shape(&s);
      if (s.units0 > 0 && s.kb_total > 0) {  // one split per rank: fp32 partial per rank
        s.n_split = p;
        s.kb_per_split = cdiv(K, BK);
      }
      v.push_back(s);
      return v;
    case TP_OP_ROW_RS:
      s.S = p; s.kseg = K; tok(Mp, N, p, 1); break;
    case TP_OP_COL_FWD:
      s.S = 1; s.kseg = K; tok(M, N, 1, p); break;
    case TP_OP_AG_MM:
      s.S = 1; s.kseg = K; tok(Mp, N, p, p); break;
    case TP_OP_COL_BWD: {
      s.S = p; s.kseg = N; tok(M, K, 1, 1);
      finish_shape(&s);
      v.push_back(s);
      Shape w;  // dA_k = X^T . dY_k : [K, N] per k, contraction over M
      w.precise = precise;
      w.S = 1; w.kseg = M; w.rows_g = K; w.cols_g = N; w.Gm = 1; w.Gn = p;
      w.chunk_tiles = cdiv(K, BM);
      finish_shape(&w);
      v.push_back(w);
      return v;
    }
    case TP_OP_AG_MM_BWD: {
      s.S = p; s.kseg = N; tok(Mp, K, p, 1);   // dX: ReduceScatter rows of sum_k dY_k A_k^T
      finish_shape(&s);
      v.push_back(s);
      Shape w;  // dA_k = [X_0; ...; X_{p-1}]^T dY_k: segments walk the p token shards
      w.precise = precise;
      w.S = p; w.kseg = Mp; w.rows_g = K; w.cols_g = N; w.Gm = 1; w.Gn = p;
      w.chunk_tiles = cdiv(K, BM);
      finish_shape(&w);
      v.push_back(w);
      return v;
    }
    case TP_OP_ROW_RS_BWD: {
      s.S = 1; s.kseg = N; tok(Mp, K, p, p);   // dX_r: AllGather of dY, group = (source shard, r)
      finish_shape(&s);
      v.push_back(s);
      Shape w;  // dA_r = X_r^T [dY_0; ...; dY_{p-1}]
      w.precise = precise;
      w.S = p; w.kseg = Mp; w.rows_g = K; w.cols_g = N; w.Gm = p; w.Gn = 1;
      w.chunk_tiles = cdiv(K, BM);
      finish_shape(&w);
      v.push_back(w);
      return v;
    }
    case TP_OP_ROW_BWD: {
      s.S = 1; s.kseg = N; tok(M, K, 1, p);
      finish_shape(&s);
      v.push_back(s);
      Shape w;  // dA_k = X_k^T . dY : [K, N] per k
      w.precise = precise;
      w.S = 1; w.kseg = M; w.rows_g = K; w.cols_g = N; w.Gm = p; w.Gn = 1;
      w.chunk_tiles = cdiv(K, BM);
      finish_shape(&w);
      v.push_back(w);
      return v;
    }
  }
  finish_shape(&s);
  v.push_back(s);
  return v;
}

size_t workspace_for(const std::vector<Shape>& shapes) {
  size_t need = 0;
  for (const Shape& s : shapes) need = std::max(need, s.partial_bytes());
  return kStatusBytes + need;
}

// The launches of a call for a workspace of ws_bytes: the fastest plan, or,
// when the workspace is too small for its last-wave slices, the same plan
// without them (which then needs no more than the smaller workspace, or the
// call fails the workspace check).
std::vector<Shape> plan_call(tp_op op, int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m, tp_dtype dt,
                             size_t ws_bytes) {
  std::vector<Shape> v = op_shapes(op, p, M, N, K, chunk_m, dt);
  if (workspace_for(v) <= ws_bytes) return v;
  t_plan_tails = false;
  std::vector<Shape> w = op_shapes(op, p, M, N, K, chunk_m, dt);
  t_plan_tails = true;
  return workspace_for(w) <= ws_bytes ? w : v;
}

// ------------------------------------------------------------------ launching a plan

struct Launch {
  Shape shape;
  GemmParams P;
  int variant = V_KN;
  bool bf16_chain = false;  // split-K second stage sums as a bf16 collective would
};

void init_params(GemmParams* P) { std::memset(P, 0, sizeof(*P)); }

void fill_common(GemmParams* P, const Shape& s) {
  P->Gm = s.Gm;
  P->Gn = s.Gn;
  P->m_tiles = static_cast<int32_t>(s.m_tiles);
  P->n_tiles = static_cast<int32_t>(s.n_tiles);
  P->chunk_tiles = static_cast<int32_t>(s.swap ? 1 : std::min<int64_t>(s.chunk_tiles, s.Gm * s.m_tiles));
  P->chunk_on_n = s.swap ? 1 : 0;
  // raster band: 8 N-tiles for 128x256 tiles (about 19 m-tiles x 8 n-tiles
  // in flight on 152 SMs, which minimises A+B bytes per wave); the swapped
  // kernels stream distinct weight tiles anyway.
  const int64_t TO = s.swap ? s.Gm * s.m_tiles : s.Gn * s.n_tiles;
  P->band = static_cast<int32_t>(std::max<int64_t>(1, s.swap ? TO : std::min<int64_t>(8, TO)));
  P->S = s.S;
  P->kb_per_seg = static_cast<int32_t>(cdiv(s.kseg, s.pair ? PAIR_BK : BK));
  P->n_split = s.n_split;
  P->kb_per_split = static_cast<int32_t>(s.pair ? s.S * P->kb_per_seg : s.kb_per_split);
  P->num_units = static_cast<int32_t>(s.units0 * s.n_split + s.tail_tiles() * (s.tail_split - 1));
  P->tail_start = static_cast<int32_t>(s.tail_start);
  P->tail_split = s.tail_split;
  P->rows_g = static_cast<int32_t>(s.rows_g);
  P->cols_g = static_cast<int32_t>(s.cols_g);
  P->n_rep = 1;
  P->timeout_ns = device_timeout_ns();
  P->debug_drop_q = static_cast<int32_t>(g_debug_drop_q.load());
  P->trace = g_trace.load();
  P->trace_cap = static_cast<int32_t>(std::min<int64_t>(g_trace_cap.load(), INT32_MAX));
}

size_t esize(tp_dtype d) { return d == TP_FP32 ? 4 : 2; }

// Output maps of the TMA-store epilogue for the group outputs `ptrs` (pitch
// `ld`): one map per group output (and replica) when there are at most
// MAX_MAPS of them, each clipped to the group's rows and columns; otherwise,
// when the groups are row blocks gm of p column buffers gn (the AllGather
// layouts: ptrs[gm * Gn + gn] = ptrs[gn] + gm * rows_g rows) and rows_g is a
// multiple of the 32-row box, one map per buffer with row offsets.  False
// when neither applies (the epilogue then stores with plain instructions).
bool plan_out_maps(const Shape& s, void* const* ptrs, int n_rep, int64_t ld, bool f32, CUtensorMap* maps,
                   int32_t* mapidx, int32_t* row0) {
  const int G = s.Gm * s.Gn;
  if (G * n_rep <= MAX_MAPS) {
    for (int g = 0; g < G; ++g) {
      mapidx[g] = g * n_rep;
      row0[g] = 0;
      for (int r = 0; r < n_rep; ++r)
        if (!encode_out_map(&maps[g * n_rep + r], ptrs[g + r], s.cols_g, s.rows_g, ld, f32)) return false;
    }
    return true;
  }
  if (n_rep != 1 || s.Gn > MAX_MAPS || s.rows_g % 32 != 0) return false;
  const size_t es = f32 ? 4 : 2;
  for (int gm = 0; gm < s.Gm; ++gm)
    for (int gn = 0; gn < s.Gn; ++gn)
      if (static_cast<const uint8_t*>(ptrs[gm * s.Gn + gn]) !=
          static_cast<const uint8_t*>(ptrs[gn]) + static_cast<size_t>(gm) * s.rows_g * ld * es)
        return false;
  for (int gn = 0; gn < s.Gn; ++gn)
    if (!encode_out_map(&maps[gn], ptrs[gn], s.cols_g, s.Gm * s.rows_g, ld, f32)) return false;
  for (int gm = 0; gm < s.Gm; ++gm)
    for (int gn = 0; gn < s.Gn; ++gn) {
      mapidx[gm * s.Gn + gn] = gn;
      row0[gm * s.Gn + gn] = static_cast<int32_t>(gm * s.rows_g);
    }
  return true;
}

tp_status run_launch_phases(Launch& L, tp_dtype out_dtype, void* ws, cudaStream_t stream,
                            const DevInfo& di, int phases);
void prepare_gemm(Launch& L, tp_dtype out_dtype, void* ws);

// Second stage over the launch's groups: out = epilogue(bias + sum of the
// n_split fp32 partials in split order); n_split == 0 sums nothing.
tp_status launch_reduce(const Launch& L, const Shape& s, int n_split, cudaStream_t stream,
                        const DevInfo& di) {
  const GemmParams& P = L.P;
  ReduceParams R;
  std::memset(&R, 0, sizeof(R));
  for (int g = 0; g < MAX_GROUPS; ++g) {
    R.out[g] = P.out[g];
    R.aux[g] = P.aux[g];
    R.bias[g] = P.bias[g];
  }
  R.partial = P.partial;
  R.G = s.Gm * s.Gn;
  R.A = static_cast<int32_t>(s.swap ? s.cols_g : s.rows_g);
  R.B = static_cast<int32_t>(s.swap ? s.rows_g : s.cols_g);
  R.ld_out = P.ld_out;
  R.ld_aux = P.ld_aux;
  R.out_f32 = P.out_f32;
  R.epi = P.epi;
  R.n_split = n_split;
  R.n_rep = P.n_rep;
  R.bf16_chain = L.bf16_chain ? 1 : 0;
  const int64_t total4 = static_cast<int64_t>(R.G) * R.A * R.B / 4;
  const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(total4, 256), di.sms * 8)));
  tp_splitk_reduce_kernel<<<rgrid, 256, 0, stream>>>(R);
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// db[o] = sum over rows (and, in order, over the src_per_out sources of o)
// of the bf16 [rows, N] sources; n_src / src_per_out outputs.
tp_status bias_grad(const void* const* src, int n_src, int src_per_out, void* const* out, int64_t rows,
                    int64_t N, tp_dtype dt, cudaStream_t stream) {
  if (N == 0) return TP_OK;
  BiasGradParams B;
  std::memset(&B, 0, sizeof(B));
  for (int i = 0; i < n_src; ++i) B.src[i] = src[i];
  const int n_out = n_src / src_per_out;
  for (int o = 0; o < n_out; ++o) B.out[o] = out[o];
  B.src_per_out = src_per_out;
  B.N = static_cast<int32_t>(N);
  B.rows = rows;
  B.out_f32 = dt == TP_FP32 ? 1 : 0;
  const dim3 grid(static_cast<unsigned>(cdiv(N, BG_COLS)), static_cast<unsigned>(n_out));
  tp_bias_grad_kernel<<<grid, BG_COLS / 8 * BG_LANES, 0, stream>>>(B);
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status run_launch(Launch& L, tp_dtype out_dtype, void* ws, cudaStream_t stream,
                     const DevInfo& di) {
  return run_launch_phases(L, out_dtype, ws, stream, di, 3);
}

// Longest per-cluster run, in k-blocks, of a pair launch's units under the
// kernel's static assignment (unit t on cluster t mod C): n0 units of kb0
// k-blocks, then n1 units of kb1 (n1 = 0: one problem, whose last partial
// wave may run as `tail` k-slices of each of its last tiles).
int64_t pair_makespan(int64_t n0, int64_t kb0, int64_t n1, int64_t kb1, int64_t C, int tail) {
  if (tail > 1 && n1 == 0) {
    const int64_t R = n0 % C;
    return (n0 / C) * kb0 + cdiv(cdiv(R * tail, C) * kb0, tail);
  }
  int64_t worst = 0;
  for (int64_t c = 0; c < std::min<int64_t>(C, n0 + n1); ++c) {
    const int64_t a = n0 > c ? (n0 - c + C - 1) / C : 0;
    const int64_t all = (n0 + n1 - c + C - 1) / C;
    worst = std::max(worst, a * kb0 + (all - a) * kb1);
  }
  return worst;
}

// The dX (dY.W^T) and dW (X^T.dY) launches of one backward call: one CTA-pair
// launch for both when both are plain pair launches (no split-K) and the
// combined static assignment finishes no later than the two launches one
// after the other -- for launches of more than kFuseWaves waves only when it
// finishes at least 3 % sooner; otherwise the two launches.  The two GEMMs
// are independent: neither reads what the other writes.  Short launches gain
// most (one fill, drain and partial last wave instead of two).  On long ones
// the saving is at most one wave, and where that is small the fused launch
// measured slower (sequence-parallel backward, 47 waves each: 1.5-3 %); the
// MLP block's row backward (2 x 13.5 waves: 27 fused against 28) gained.
tp_status run_bwd_pair(Launch& LX, bool do_x, Launch& LW, bool do_w, tp_dtype out_dtype, void* ws,
                       cudaStream_t stream, const DevInfo& di) {
  const Shape& a = LX.shape;
  const Shape& b = LW.shape;
  const bool both = do_x && do_w && !a.empty() && !b.empty() && a.kb_total > 0 && b.kb_total > 0 &&
                    a.pair && b.pair && !a.swap && LX.variant == V_KK && LW.variant == V_MM &&
                    g_debug_no_fuse.load() == 0;
  if (both) {
    const int64_t C = di.sms / 2;
    const int64_t kba = a.S * cdiv(a.kseg, PAIR_BK), kbb = b.S * cdiv(b.kseg, PAIR_BK);
    const int64_t sep = pair_makespan(a.units0, kba, 0, 0, C, a.tail_split) +
                        pair_makespan(b.units0, kbb, 0, 0, C, b.tail_split);
    const int64_t fused = pair_makespan(a.units0, kba, b.units0, kbb, C, 1);
    const bool short_launches = std::max(a.units0, b.units0) <= kFuseWaves * C;
    if (fused <= sep && (short_launches || fused * 100 <= sep * 97)) {
      // whole tiles only: the fused launch has a single partial last wave
      Shape sa = a, sb = b;
      sa.tail_split = sb.tail_split = 1;
      sa.tail_start = sb.tail_start = 0;
      fill_common(&LX.P, sa);
      fill_common(&LW.P, sb);
      LX.shape = sa;
      LW.shape = sb;
      prepare_gemm(LX, out_dtype, ws);
      prepare_gemm(LW, out_dtype, ws);
      LW.P.epoch = LX.P.epoch;
      static thread_local PairLaunch2 L2;   // 14 KB: kept off the stack
      L2.P[0] = LX.P;
      L2.P[1] = LW.P;
      L2.split = LX.P.num_units;
      L2.total = LX.P.num_units + LW.P.num_units;
      const int clusters = static_cast<int>(std::min<int64_t>(L2.total, di.sms / 2));
      return launch_pair2(L2, clusters, stream) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
    }
  }
  if (do_x) {
    const tp_status st = run_launch(LX, out_dtype, ws, stream, di);
    if (st != TP_OK) return st;
  }
  return do_w ? run_launch(LW, out_dtype, ws, stream, di) : TP_OK;
}

// phases: bit 0 = the GEMM launch (or the K == 0 fill), bit 1 = the split-K
// second stage.
tp_status run_launch_phases(Launch& L, tp_dtype out_dtype, void* ws, cudaStream_t stream,
                            const DevInfo& di, int phases) {
  const Shape& s = L.shape;
  if (s.empty()) return TP_OK;
  if (s.pair) L.variant = L.variant == V_KN ? V_KN2 : L.variant == V_KK ? V_KK2 : V_MM2;
  GemmParams& P = L.P;
  P.status = static_cast<uint32_t*>(ws);
  P.out_f32 = out_dtype == TP_FP32 ? 1 : 0;
  const int G = s.Gm * s.Gn;
  bool any_bias = false;
  for (int g = 0; g < G; ++g) any_bias = any_bias || P.bias[g] != nullptr;
  if (s.kb_total == 0 && any_bias) {
    // K == 0 with a bias: out = epilogue(bias), from the second-stage kernel
    // summing zero partials.
    if (!(phases & 1)) return TP_OK;
    return launch_reduce(L, s, 0, stream, di);
  }
  if (s.kb_total == 0) {
    if (!(phases & 1)) return TP_OK;
    // K == 0: the product is zero; GeLU(0) = 0 and G * GeLU'(.) = 0 too.
    const int64_t A = s.swap ? s.cols_g : s.rows_g;
    const int64_t B = s.swap ? s.rows_g : s.cols_g;
    for (int g = 0; g < G; ++g) {
      for (int r = 0; r < (g == 0 ? P.n_rep : 1); ++r) {
        if (cudaMemset2DAsync(P.out[g + r], P.ld_out * esize(out_dtype), 0, B * esize(out_dtype), A,
                              stream) != cudaSuccess)
          return TP_ERR_CUDA;
      }
      if (P.epi == EPI_GELU && P.aux[g] != nullptr) {
        if (cudaMemset2DAsync(P.aux[g], P.ld_aux * esize(out_dtype), 0, B * esize(out_dtype), A,
                              stream) != cudaSuccess)
          return TP_ERR_CUDA;
      }
    }
    return TP_OK;
  }
  prepare_gemm(L, out_dtype, ws);
  const int grid = s.pair ? static_cast<int>(std::min<int64_t>(P.num_units, di.sms / 2))
                         : static_cast<int>(std::min<int64_t>(P.num_units, di.sms));
  if ((phases & 1) && launch_variant(L.variant, P, grid, stream) != cudaSuccess) return TP_ERR_CUDA;
  if (s.n_split > 1 && (phases & 2)) return launch_reduce(L, s, s.n_split, stream, di);
  return TP_OK;
}

// The launch-time fields of a GEMM launch with work to do (K > 0): workspace
// regions, the launch number, L2 policies and the TMA-store output maps.
void prepare_gemm(Launch& L, tp_dtype out_dtype, void* ws) {
  const Shape& s = L.shape;
  GemmParams& P = L.P;
  P.status = static_cast<uint32_t*>(ws);
  P.out_f32 = out_dtype == TP_FP32 ? 1 : 0;
  if (s.n_split > 1) P.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  // slice counters tagged with another launch's number read as zero
  P.epoch = g_launch_epoch.fetch_add(1) + 1;
  if (s.tail_split > 1) {
    uint8_t* base = static_cast<uint8_t*>(ws) + kStatusBytes;
    P.tail_cnt = reinterpret_cast<unsigned long long*>(base);
    P.tail_part = reinterpret_cast<float*>(base + s.tail_cnt_bytes());
  }
  // L2 policies: an operand shared by every group (one set of maps for all
  // of them, re-read by every group's tiles) is kept while the other
  // streams past it, if it fits in half the L2; final outputs, which nothing
  // in the launch reads back, are written evict_first (plain and TMA
  // stores), and the GeLU' epilogue reads the saved H, used once, the same way.
  // Bytes of each operand over the whole launch: distinct maps x the panel
  // rows or columns x the contraction each map covers (every segment's, when
  // the segments walk one map at K offsets).
  const int64_t a_bytes = (P.a_idx_gm ? s.Gm : 1) * (P.a_idx_gn ? s.Gn : 1) * (P.a_idx_s ? s.S : 1) * s.rows_g *
                          s.kseg * (P.a_koff_s && !P.a_idx_s ? s.S : 1) * 2;
  const int64_t b_bytes = (P.b_idx_gm ? s.Gm : 1) * (P.b_idx_gn ? s.Gn : 1) * (P.b_idx_s ? s.S : 1) * s.cols_g *
                          s.kseg * (P.b_koff_s && !P.b_idx_s ? s.S : 1) * 2;
  // Raster band: when the whole B operand fits in the L2 budget and A does
  // not, one band spans every N-tile, so that A streams through exactly once
  // while B stays resident (e.g. dW = X_r^T . dY with dY shared by the p
  // groups: 8-tile bands read the p X_r shards from DRAM once per band).
  // Where both fit, the 8-tile band is kept (one band measured 2 % slower
  // on the MHA W_O backward, with the same DRAM bytes).
  if (s.pair && b_bytes <= kKeepBytes && a_bytes > kKeepBytes) P.band = static_cast<int32_t>(s.Gn * s.n_tiles);
  // groups along M that offset their rows within the same A maps (the
  // ReduceScatter layouts) read different data, as do groups along N that
  // offset their columns within the same B maps
  const bool a_shared = (P.a_idx_gm == 0 && P.a_row_gm == 0 && s.Gm > 1) || (P.a_idx_gn == 0 && s.Gn > 1);
  const bool b_shared = (P.b_idx_gm == 0 && s.Gm > 1) || (P.b_idx_gn == 0 && P.b_col_gn == 0 && s.Gn > 1);
  // Where A stays in L2 (shared by every group and within the budget), a
  // band only needs to keep its B panels.  When an 8-tile band would spread
  // each B panel's uses over more than a wave, the band is narrowed to half
  // the width whose tiles fill one wave: the MLP column forward (16 row
  // tiles) runs bands of 2 N-tiles, which cut its DRAM reads from 324 to
  // 234 MB and its time by 3.5 %.  Bands of 4 and of 1 measured slower.
  if (s.pair && a_shared && a_bytes <= kKeepBytes && P.band == 8) {
    const int64_t fit = (kPlanSMs / 2) / std::max<int32_t>(1, P.chunk_tiles);   // one wave of tiles
    if (fit < 8) P.band = static_cast<int32_t>(std::max<int64_t>(1, fit / 2));
  }
  P.a_hint = P.b_hint = P.out_hint = 0;
  if (g_l2_hints.load() != 0) {
    P.a_hint = a_shared && a_bytes <= kKeepBytes ? 1 : 0;
    P.b_hint = b_shared && b_bytes <= kKeepBytes ? 1 : 0;
    P.out_hint = 2;
  }
  P.k_alternate = g_k_alternate.load() != 0 && s.pair && s.S * s.kseg >= kKAlternateDepth ? 1 : 0;
  // staged epilogues (non-swapped tiles, no split-K partials) store through TMA
  P.out_tma = 0;
  if (g_tma_store.load() != 0 && !s.swap && s.n_split == 1) {
    const bool f32 = out_dtype == TP_FP32;
    bool ok = plan_out_maps(s, P.out, P.n_rep, P.ld_out, f32, P.tmO, P.omap, P.orow);
    if (ok && P.epi == EPI_GELU && P.aux[0] != nullptr)
      ok = plan_out_maps(s, P.aux, 1, P.ld_aux, f32, P.tmH, P.hmap, P.hrow);
    P.out_tma = ok ? 1 : 0;
  }
}

// ------------------------------------------------------------------ validation

struct Range {
  const void* p;
  size_t bytes;
};

bool overlap(const Range& a, const Range& b) {
  if (a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool any_overlap(const std::vector<Range>& outs, const std::vector<Range>& ins) {
  for (size_t i = 0; i < outs.size(); ++i) {
    for (const Range& r : ins)
      if (overlap(outs[i], r)) return true;
    for (size_t j = i + 1; j < outs.size(); ++j)
      if (overlap(outs[i], outs[j])) return true;
  }
  return false;
}

tp_status check_sizes(int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m, tp_dtype dt) {
  if (p < 1 || p > kMaxP) return TP_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || chunk_m < 0) return TP_ERR_INVALID_ARG;
  if (dt != TP_BF16 && dt != TP_FP32) return TP_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim || K > lim || static_cast<int64_t>(p) * K > lim) return TP_ERR_UNSUPPORTED_SHAPE;
  if (N % 8 != 0 || K % 8 != 0) return TP_ERR_ALIGNMENT;
  return TP_OK;
}

tp_status check_ptrs(const void* const* a, int n, bool need) {
  if (!need) return TP_OK;
  if (a == nullptr) return TP_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (a[i] == nullptr) return TP_ERR_INVALID_ARG;
    if (!aligned16(a[i])) return TP_ERR_ALIGNMENT;
  }
  return TP_OK;
}

tp_status check_ptr(const void* a, bool need) {
  if (!need) return TP_OK;
  if (a == nullptr) return TP_ERR_INVALID_ARG;
  return aligned16(a) ? TP_OK : TP_ERR_ALIGNMENT;
}

tp_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return TP_ERR_INVALID_ARG;
  if (!aligned16(ws)) return TP_ERR_ALIGNMENT;
  if (ws_bytes < need) return TP_ERR_WORKSPACE_TOO_SMALL;
  return TP_OK;
}

#define TP_TRY(expr)                     \
  do {                                   \
    tp_status _st = (expr);              \
    if (_st != TP_OK) return _st;        \
  } while (0)

void add_ranges(std::vector<Range>* v, const void* const* a, int n, size_t bytes) {
  if (a == nullptr) return;
  for (int i = 0; i < n; ++i)
    if (a[i] != nullptr) v->push_back({a[i], bytes});
}

int sw_variant_mk(int bn) { return bn == 16 ? V_SW_MK16 : bn == 32 ? V_SW_MK32 : V_SW_MK64; }
int sw_variant_kk(int bn) { return bn == 16 ? V_SW_KK16 : bn == 32 ? V_SW_KK32 : V_SW_KK64; }

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_INVALID_ARG: return "invalid argument (p, size, null pointer, aliasing or enum)";
    case TP_ERR_ALIGNMENT: return "pointer or row pitch not 16-byte aligned (K and N must be multiples of 8)";
    case TP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (M must be divisible by p for ReduceScatter/AllGather; sizes < 2^31)";
    case TP_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than tp_workspace_size()";
    case TP_ERR_ARCH: return "device is not sm_103 (GB300)";
    case TP_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case TP_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out (latched in the workspace)";
  }
  return "unknown status";
}

tp_status tp_debug_set(tp_debug_key key, int64_t value) {
  switch (key) {
    case TP_DEBUG_TIMEOUT_MS:
      if (value < 0) return TP_ERR_INVALID_ARG;
      g_timeout_override_ns.store(static_cast<uint64_t>(value) * 1000000ull);
      return TP_OK;
    case TP_DEBUG_DROP_LOAD:
      if (value < -1 || value > INT32_MAX) return TP_ERR_INVALID_ARG;
      g_debug_drop_q.store(value);
      return TP_OK;
    case TP_DEBUG_TILE_MODE:
      if (value < 0 || value > 2) return TP_ERR_INVALID_ARG;
      g_debug_tile_mode.store(value);
      return TP_OK;
    case TP_DEBUG_NO_TAIL_SLICES:
      if (value < 0 || value > 1) return TP_ERR_INVALID_ARG;
      g_debug_no_tail.store(value);
      return TP_OK;
    case TP_DEBUG_SPLIT_K:
      if (value < 0 || value > 16) return TP_ERR_INVALID_ARG;
      g_debug_split_k.store(value);
      return TP_OK;
    case TP_DEBUG_L2_HINTS:
      if (value < 0 || value > 1) return TP_ERR_INVALID_ARG;
      g_l2_hints.store(value);
      return TP_OK;
    case TP_DEBUG_TMA_STORE:
      if (value < 0 || value > 1) return TP_ERR_INVALID_ARG;
      g_tma_store.store(value);
      return TP_OK;
    case TP_DEBUG_NO_BWD_FUSION:
      if (value < 0 || value > 1) return TP_ERR_INVALID_ARG;
      g_debug_no_fuse.store(value);
      return TP_OK;
    case TP_DEBUG_K_ALTERNATE:
      if (value < 0 || value > 1) return TP_ERR_INVALID_ARG;
      g_k_alternate.store(value);
      return TP_OK;
  }
  return TP_ERR_INVALID_ARG;
}

tp_status tp_trace_set(void* buf, int64_t cap_units) {
  if (cap_units < 0 || (buf == nullptr) != (cap_units == 0)) return TP_ERR_INVALID_ARG;
  if (buf != nullptr && !aligned16(buf)) return TP_ERR_ALIGNMENT;
  g_trace.store(static_cast<unsigned long long*>(buf));
  g_trace_cap.store(cap_units);
  return TP_OK;
}

double tp_pipeline_time(double c, double m, int64_t n_chunks) {
  if (n_chunks <= 0) return 0.0;
  return c + static_cast<double>(n_chunks - 1) * std::max(c, m) + m;
}

int64_t tp_num_chunks(int64_t M, int64_t chunk_m) {
  if (M <= 0) return 0;
  if (chunk_m <= 0) chunk_m = M;
  const int64_t c = std::min(chunk_m, M);
  return cdiv(M, c);
}

int64_t tp_choose_chunk_m(tp_op op, int p, int64_t M, int64_t N, int64_t K) {
  if (M <= 0) return 0;
  if (p < 1) p = 1;
  // Model constants: dense bf16 tensor rate and HBM copy rate of a GB300,
  // and the weight-set size below which the weights stay in L2 from one
  // chunk to the next: half of the 129 MB L2, since the activations, the
  // outputs and the other half of each wave's operands share it (a 100 MB
  // weight set re-read per 512-row chunk cost the QKV projection 8 %).
  const double peak = 1.9e15, bw = 6.7e12, l2 = 48.0 * (1 << 20);
  double flops = 0, wbytes = 0, in_row = 0, out_row = 0;
  switch (op) {
    case TP_OP_ROW_AR: case TP_OP_ROW_RS:
      flops = 2.0 * M * N * K * p; wbytes = 2.0 * K * N * p; in_row = 2.0 * K * p; out_row = 2.0 * N; break;
    case TP_OP_COL_FWD: case TP_OP_AG_MM:
      flops = 2.0 * M * N * K * p; wbytes = 2.0 * K * N * p; in_row = 2.0 * K; out_row = 2.0 * N * p; break;
    case TP_OP_COL_BWD:
      flops = 2.0 * M * N * K * p; wbytes = 2.0 * K * N * p; in_row = 2.0 * N * p; out_row = 2.0 * K; break;
    case TP_OP_ROW_BWD:
      flops = 2.0 * M * N * K * p; wbytes = 2.0 * K * N * p; in_row = 2.0 * N; out_row = 2.0 * K * p; break;
  }
  // Candidates from one chunk (M rows) down to 16 rows.  A chunk's compute
  // time c is its MMA time at the tile's MMA-width efficiency or its
  // compulsory streaming time, whichever is larger, plus the time to stream
  // the weights again when they do not stay in L2 across chunks (the
  // pipeline stalls on those re-reads).  Its reduce time m is the write-out
  // of its rows.  A smaller chunk must beat the best so far by more than 2 %
  // to be chosen: fewer chunks keep more operand reuse in flight.
  std::vector<int64_t> cand;
  cand.push_back(M);
  int64_t top = 16;
  while (top * 2 < M) top *= 2;
  for (int64_t c = top; c >= 16; c /= 2)
    if (c < M) cand.push_back(c);
  int64_t best = M;
  double best_t = 1e300;
  for (int64_t c : cand) {
    const int64_t rows = std::min(c, M);
    const int64_t n = cdiv(M, rows);
    const double eff = rows >= BM ? 1.0 : static_cast<double>(cdiv(rows, 16) * 16) / BM;
    const double first = wbytes / n + rows * (in_row + out_row);
    const double again = (wbytes > l2 && n > 1) ? wbytes * (n - 1) / n : 0.0;
    const double cc = std::max(flops * rows / M / (peak * eff), first / bw) + again / bw;
    const double mm = rows * out_row / bw;
    const double t = tp_pipeline_time(cc, mm, n);
    if (t < best_t * 0.98) {
      best_t = t;
      best = c;
    }
  }
  return std::min(best, M);
}

int64_t tp_choose_chunk_m_measured(int64_t M, const int64_t* chunk, const double* c, const double* m,
                                   int n) {
  if (n <= 0 || M <= 0 || chunk == nullptr || c == nullptr || m == nullptr) return 0;
  int64_t best = 0;
  double best_t = 0.0;
  for (int i = 0; i < n; ++i) {
    if (chunk[i] <= 0) continue;
    const double t = tp_pipeline_time(c[i], m[i], tp_num_chunks(M, chunk[i]));
    if (best == 0 || t < best_t) {
      best = chunk[i];
      best_t = t;
    }
  }
  return best;
}

size_t tp_workspace_size(tp_op op, int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                         tp_dtype out_dtype) {
  if (p < 1 || p > kMaxP || M < 0 || N < 0 || K < 0 || chunk_m < 0) return kStatusBytes;
  if ((op == TP_OP_ROW_RS || op == TP_OP_AG_MM) && M % p != 0) return kStatusBytes;
  return workspace_for(op_shapes(op, p, M, N, K, chunk_m, out_dtype));
}

tp_status tp_get_device_status(void* ws, cudaStream_t stream) {
  if (ws == nullptr) return TP_ERR_INVALID_ARG;
  int dev = 0;
  if (bind_device(&dev) != TP_OK) return TP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TP_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return TP_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return TP_ERR_CUDA;
    return TP_ERR_DEVICE_TIMEOUT;
  }
  return TP_OK;
}

// ---------------------------------------------------------------- row parallel

static tp_status row_fwd_impl(bool rs, const void* const* x, const void* const* w, const void* bias,
                              void* const* y, int n_out, int p, int64_t M, int64_t N, int64_t K,
                              int64_t chunk_m, tp_dtype dt, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, dt));
  if (rs) {
    if (M % p != 0) return TP_ERR_UNSUPPORTED_SHAPE;
    n_out = p;
  } else if (n_out != 1 && n_out != p) {
    return TP_ERR_INVALID_ARG;
  }
  const bool work = M > 0 && N > 0;
  TP_TRY(check_ptrs(x, p, work && K > 0));
  TP_TRY(check_ptrs(w, p, work && K > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(y), n_out, work));
  TP_TRY(check_ptr(bias, work && bias != nullptr));
  const tp_op op = rs ? TP_OP_ROW_RS : TP_OP_ROW_AR;
  std::vector<Shape> shapes = plan_call(op, p, M, N, K, chunk_m, dt, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  if (!work) return TP_OK;
  const int64_t Mp = M / p;
  {
    std::vector<Range> ins, outs;
    add_ranges(&ins, x, p, M * K * 2);
    add_ranges(&ins, w, p, K * N * 2);
    if (bias != nullptr) ins.push_back({bias, static_cast<size_t>(N * 2)});
    add_ranges(&outs, const_cast<const void* const*>(y), n_out, (rs ? Mp : M) * N * esize(dt));
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  DevInfo di;
  TP_TRY(device_info(&di));
  Launch L;
  L.shape = shapes[0];
  init_params(&L.P);
  fill_common(&L.P, L.shape);
  GemmParams& P = L.P;
  const Shape& s = L.shape;
  const bool m3 = use_3d(N, K);
  P.map3d = m3 ? 1 : 0;
  if (K > 0) {
    for (int r = 0; r < p; ++r) {
      if (!s.swap) {
        if (!encode_map(&P.tmA[r], x[r], K, M, K, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0) ||
            !encode_map(&P.tmB[r], w[r], N, K, N, s.pair ? PAIR_BK : 64, m3 ? (s.pair ? 2 : 4) : 0))
          return TP_ERR_CUDA;
      } else {
        if (!encode_map(&P.tmA[r], w[r], N, K, N, 64, m3 ? 2 : 0) ||
            !encode_map(&P.tmB[r], x[r], K, M, K, s.bn, m3 ? 1 : 0))
          return TP_ERR_CUDA;
      }
    }
  }
  P.a_idx_s = 1;
  P.b_idx_s = 1;
  P.ld_out = N;
  P.epi = EPI_NONE;
  if (!rs) {
    for (int i = 0; i < n_out; ++i) P.out[i] = y[i];
    P.n_rep = n_out;
    P.bias[0] = bias;  // once, after the reduction; replicas share it
  } else {
    for (int j = 0; j < p; ++j) {
      P.out[j] = y[j];
      P.bias[j] = bias;
    }
    if (!s.swap) P.a_row_gm = static_cast<int32_t>(Mp);
    else P.b_col_gn = static_cast<int32_t>(Mp);
  }
  L.variant = s.swap ? sw_variant_mk(s.bn) : V_KN;
  return run_launch(L, dt, ws, stream, di);
}

tp_status tp_row_linear_fwd_allreduce(const void* const* x, const void* const* w, const void* bias,
                                      void* const* y, int n_out, int p, int64_t M, int64_t N,
                                      int64_t K, int64_t chunk_m, tp_dtype out_dtype, void* ws,
                                      size_t ws_bytes, cudaStream_t stream) {
  return row_fwd_impl(false, x, w, bias, y, n_out, p, M, N, K, chunk_m, out_dtype, ws, ws_bytes,
                      stream);
}

tp_status tp_row_linear_fwd_reducescatter(const void* const* x, const void* const* w,
                                          const void* bias, void* const* y, int p, int64_t M,
                                          int64_t N, int64_t K, int64_t chunk_m, tp_dtype out_dtype,
                                          void* ws, size_t ws_bytes, cudaStream_t stream) {
  return row_fwd_impl(true, x, w, bias, y, p, p, M, N, K, chunk_m, out_dtype, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- column parallel

static tp_status col_like_fwd(bool ag, const void* const* xs, const void* x1, const void* const* w,
                              const void* const* bias, void* const* y, void* const* preact,
                              tp_epilogue epi, int p,
                              int64_t M, int64_t N, int64_t K, int64_t chunk_m, tp_dtype dt,
                              void* ws, size_t ws_bytes, cudaStream_t stream, void* x_gathered) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, dt));
  if (epi != TP_EPI_NONE && epi != TP_EPI_GELU) return TP_ERR_INVALID_ARG;
  if (ag && M % p != 0) return TP_ERR_UNSUPPORTED_SHAPE;
  const bool work = M > 0 && N > 0;
  if (ag) TP_TRY(check_ptrs(xs, p, M > 0 && (K > 0) && (work || x_gathered != nullptr)));
  else TP_TRY(check_ptr(x1, work && K > 0));
  TP_TRY(check_ptrs(w, p, work && K > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(y), p, work));
  const bool want_h = epi == TP_EPI_GELU && preact != nullptr;
  TP_TRY(check_ptrs(const_cast<const void* const*>(preact), p, work && want_h));
  TP_TRY(check_ptr(x_gathered, x_gathered != nullptr));
  TP_TRY(check_ptrs(bias, p, work && bias != nullptr));
  const tp_op op = ag ? TP_OP_AG_MM : TP_OP_COL_FWD;
  std::vector<Shape> shapes = plan_call(op, p, M, N, K, chunk_m, dt, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  const int64_t Mp = M / p;
  {
    std::vector<Range> ins, outs;
    if (ag) add_ranges(&ins, xs, p, Mp * K * 2);
    else if (x1 != nullptr) ins.push_back({x1, static_cast<size_t>(M * K * 2)});
    add_ranges(&ins, w, p, K * N * 2);
    if (work) add_ranges(&ins, bias, p, N * 2);
    add_ranges(&outs, const_cast<const void* const*>(y), p, M * N * esize(dt));
    if (want_h) add_ranges(&outs, const_cast<const void* const*>(preact), p, M * N * esize(dt));
    if (x_gathered != nullptr) outs.push_back({x_gathered, static_cast<size_t>(M * K * 2)});
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  if (!work && x_gathered == nullptr) return TP_OK;
  DevInfo di;
  TP_TRY(device_info(&di));
  if (ag && x_gathered != nullptr && M > 0 && K > 0) {
    for (int s = 0; s < p; ++s)
      if (cudaMemcpyAsync(static_cast<uint8_t*>(x_gathered) + s * Mp * K * 2, xs[s], Mp * K * 2,
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return TP_ERR_CUDA;
  }
  if (!work) return TP_OK;
  Launch L;
  L.shape = shapes[0];
  init_params(&L.P);
  fill_common(&L.P, L.shape);
  GemmParams& P = L.P;
  const Shape& s = L.shape;
  const bool m3 = use_3d(N, K);
  P.map3d = m3 ? 1 : 0;
  const size_t es = esize(dt);
  if (K > 0) {
    for (int k = 0; k < p; ++k) {
      // weights: MN-major in both orientations ([K, N] row-major)
      CUtensorMap* wm = s.swap ? &P.tmA[k] : &P.tmB[k];
      if (!encode_map(wm, w[k], N, K, N, s.pair ? PAIR_BK : 64, m3 ? (s.swap ? 2 : s.pair ? 2 : 4) : 0))
        return TP_ERR_CUDA;
    }
    const int tok_box = s.swap ? s.bn : BM;
    if (!ag) {
      CUtensorMap* xm = s.swap ? &P.tmB[0] : &P.tmA[0];
      if (!encode_map(xm, x1, K, M, K, tok_box, m3 ? (s.pair ? kPairKChunks : 1) : 0)) return TP_ERR_CUDA;
    } else {
      for (int t = 0; t < p; ++t) {
        CUtensorMap* xm = s.swap ? &P.tmB[t] : &P.tmA[t];
        if (!encode_map(xm, xs[t], K, Mp, K, tok_box, m3 ? (s.pair ? kPairKChunks : 1) : 0)) return TP_ERR_CUDA;
      }
    }
  }
  P.ld_out = N;
  P.ld_aux = N;
  P.epi = epi == TP_EPI_GELU ? EPI_GELU : EPI_NONE;
  if (!ag) {
    if (!s.swap) P.b_idx_gn = 1;   // groups along N are the shards k
    else P.a_idx_gm = 1;           // groups along M are the shards k
    for (int k = 0; k < p; ++k) {
      P.out[k] = y[k];
      P.aux[k] = want_h ? preact[k] : nullptr;
      P.bias[k] = bias ? bias[k] : nullptr;
    }
  } else {
    // group (gm, gn): standard gm = source shard s, gn = shard k;
    //                 swapped  gm = shard k,        gn = source shard s.
    if (!s.swap) { P.a_idx_gm = 1; P.b_idx_gn = 1; }
    else { P.a_idx_gm = 1; P.b_idx_gn = 1; }
    for (int gm = 0; gm < p; ++gm) {
      for (int gn = 0; gn < p; ++gn) {
        const int k = s.swap ? gm : gn;
        const int src = s.swap ? gn : gm;
        const int64_t off = static_cast<int64_t>(src) * Mp * N * es;
        P.out[gm * p + gn] = static_cast<uint8_t*>(y[k]) + off;
        P.aux[gm * p + gn] = want_h ? static_cast<uint8_t*>(preact[k]) + off : nullptr;
        P.bias[gm * p + gn] = bias ? bias[k] : nullptr;
      }
    }
  }
  L.variant = s.swap ? sw_variant_mk(s.bn) : V_KN;
  return run_launch(L, dt, ws, stream, di);
}

tp_status tp_col_linear_fwd(const void* x, const void* const* w, const void* const* bias,
                            void* const* y, void* const* preact, tp_epilogue epi, int p, int64_t M,
                            int64_t N, int64_t K, int64_t chunk_m, tp_dtype out_dtype, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  return col_like_fwd(false, nullptr, x, w, bias, y, preact, epi, p, M, N, K, chunk_m, out_dtype, ws,
                      ws_bytes, stream, nullptr);
}

tp_status tp_ag_matmul(const void* const* x, const void* const* w, const void* const* bias,
                       void* const* y, void* x_gathered, tp_epilogue epi, void* const* preact, int p,
                       int64_t M, int64_t N, int64_t K, int64_t chunk_m, tp_dtype out_dtype,
                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  return col_like_fwd(true, x, nullptr, w, bias, y, preact, epi, p, M, N, K, chunk_m, out_dtype, ws,
                      ws_bytes, stream, x_gathered);
}

// ---------------------------------------------------------------- backward

// Weight gradient dA_g = Xsrc_g^T . dYsrc_g for g = 0..p-1 ([K, N] each,
// contraction over the M tokens); both operands MN-major.  Fills L for
// run_bwd_pair.
static tp_status weight_grad(Launch& L, const Shape& s, const void* const* xk, const void* x1,
                             const void* const* dyk, const void* dy1, void* const* dw, int p,
                             int64_t M, int64_t N, int64_t K) {
  L.shape = s;
  init_params(&L.P);
  fill_common(&L.P, s);
  GemmParams& P = L.P;
  const bool m3 = use_3d(N, K);
  P.map3d = m3 ? 1 : 0;
  if (M > 0) {
    for (int k = 0; k < (xk ? p : 1); ++k)
      if (!encode_map(&P.tmA[k], xk ? xk[k] : x1, K, M, K, s.pair ? PAIR_BK : 64, m3 ? 2 : 0)) return TP_ERR_CUDA;
    for (int k = 0; k < (dyk ? p : 1); ++k)
      if (!encode_map(&P.tmB[k], dyk ? dyk[k] : dy1, N, M, N, s.pair ? PAIR_BK : 64, m3 ? (s.pair ? 2 : 4) : 0))
        return TP_ERR_CUDA;
  }
  // the p problems are the groups (along N for the column case, along M for the row case)
  if (s.Gn == p && s.Gm == 1) {
    P.a_idx_gn = xk ? 1 : 0;
    P.b_idx_gn = dyk ? 1 : 0;
  } else {
    P.a_idx_gm = xk ? 1 : 0;
    P.b_idx_gm = dyk ? 1 : 0;
  }
  for (int k = 0; k < p; ++k) P.out[k] = dw[k];
  P.ld_out = N;
  P.epi = EPI_NONE;
  L.variant = V_MM;
  return TP_OK;
}

tp_status tp_col_linear_bwd(const void* x, const void* const* w, const void* const* dy, void* dx,
                            void* const* dw, void* const* db, int p, int64_t M, int64_t N, int64_t K,
                            int64_t chunk_m, tp_dtype out_dtype, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  if (dx == nullptr && dw == nullptr && db == nullptr) return TP_ERR_INVALID_ARG;
  const bool dx_work = dx != nullptr && M > 0 && K > 0;
  const bool dw_work = dw != nullptr && K > 0 && N > 0;
  const bool db_work = db != nullptr && N > 0;
  TP_TRY(check_ptr(dx, dx_work));
  TP_TRY(check_ptrs(w, p, dx_work && N > 0));
  TP_TRY(check_ptrs(dy, p, (dx_work && N > 0) || ((dw_work || db_work) && M > 0)));
  TP_TRY(check_ptrs(const_cast<const void* const*>(db), p, db_work));
  TP_TRY(check_ptr(x, dw_work && M > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(dw), p, dw_work));
  std::vector<Shape> shapes = plan_call(TP_OP_COL_BWD, p, M, N, K, chunk_m, out_dtype, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  {
    std::vector<Range> ins, outs;
    if (x) ins.push_back({x, static_cast<size_t>(M * K * 2)});
    add_ranges(&ins, w, p, K * N * 2);
    add_ranges(&ins, dy, p, M * N * 2);
    if (dx) outs.push_back({dx, static_cast<size_t>(M * K * esize(out_dtype))});
    if (dw) add_ranges(&outs, const_cast<const void* const*>(dw), p, K * N * esize(out_dtype));
    if (db) add_ranges(&outs, const_cast<const void* const*>(db), p, N * esize(out_dtype));
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  if (!dx_work && !dw_work && !db_work) return TP_OK;
  DevInfo di;
  TP_TRY(device_info(&di));
  Launch LX, LW;
  if (dx_work) {
    Launch& L = LX;
    L.shape = shapes[0];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (N > 0) {
      for (int k = 0; k < p; ++k) {
        if (!s.swap) {
          if (!encode_map(&P.tmA[k], dy[k], N, M, N, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0) ||
              !encode_map(&P.tmB[k], w[k], N, K, N, s.pair ? 128 : 256, m3 ? (s.pair ? kPairKChunks : 1) : 0))
            return TP_ERR_CUDA;
        } else {
          if (!encode_map(&P.tmA[k], w[k], N, K, N, BM, m3 ? 1 : 0) ||
              !encode_map(&P.tmB[k], dy[k], N, M, N, s.bn, m3 ? 1 : 0))
            return TP_ERR_CUDA;
        }
      }
    }
    P.a_idx_s = 1;
    P.b_idx_s = 1;
    P.out[0] = dx;
    P.ld_out = K;
    P.epi = EPI_NONE;
    L.variant = s.swap ? sw_variant_kk(s.bn) : V_KK;
  }
  if (dw_work) TP_TRY(weight_grad(LW, shapes[1], nullptr, x, dy, nullptr, dw, p, M, N, K));
  TP_TRY(run_bwd_pair(LX, dx_work, LW, dw_work, out_dtype, ws, stream, di));
  if (db_work) TP_TRY(bias_grad(dy, p, 1, db, M, N, out_dtype, stream));   // db_k = sum of dY_k's rows
  return TP_OK;
}

tp_status tp_row_linear_bwd(const void* const* x, const void* const* w, const void* dy,
                            void* const* dx, void* const* dw, void* db, const void* const* preact,
                            int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                            tp_dtype out_dtype, void* ws, size_t ws_bytes, cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  const bool dx_work = dx != nullptr && M > 0 && K > 0;
  const bool dw_work = dw != nullptr && K > 0 && N > 0;
  const bool db_work = db != nullptr && N > 0;
  if (dx == nullptr && dw == nullptr && db == nullptr) return TP_ERR_INVALID_ARG;
  TP_TRY(check_ptrs(const_cast<const void* const*>(dx), p, dx_work));
  TP_TRY(check_ptrs(w, p, dx_work && N > 0));
  TP_TRY(check_ptr(dy, (dx_work && N > 0) || ((dw_work || db_work) && M > 0)));
  TP_TRY(check_ptr(db, db_work));
  TP_TRY(check_ptrs(x, p, dw_work && M > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(dw), p, dw_work));
  TP_TRY(check_ptrs(preact, p, dx_work && preact != nullptr));
  std::vector<Shape> shapes = plan_call(TP_OP_ROW_BWD, p, M, N, K, chunk_m, out_dtype, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  {
    std::vector<Range> ins, outs;
    add_ranges(&ins, x, p, M * K * 2);
    add_ranges(&ins, w, p, K * N * 2);
    if (dy) ins.push_back({dy, static_cast<size_t>(M * N * 2)});
    add_ranges(&ins, preact, p, M * K * 2);
    if (dx) add_ranges(&outs, const_cast<const void* const*>(dx), p, M * K * esize(out_dtype));
    if (dw) add_ranges(&outs, const_cast<const void* const*>(dw), p, K * N * esize(out_dtype));
    if (db) outs.push_back({db, static_cast<size_t>(N * esize(out_dtype))});
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  if (!dx_work && !dw_work && !db_work) return TP_OK;
  DevInfo di;
  TP_TRY(device_info(&di));
  Launch LX, LW;
  if (dx_work) {
    Launch& L = LX;
    L.shape = shapes[0];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (N > 0) {
      for (int k = 0; k < p; ++k) {
        if (!s.swap) {
          if (!encode_map(&P.tmB[k], w[k], N, K, N, s.pair ? 128 : 256, m3 ? (s.pair ? kPairKChunks : 1) : 0)) return TP_ERR_CUDA;
        } else {
          if (!encode_map(&P.tmA[k], w[k], N, K, N, BM, m3 ? 1 : 0)) return TP_ERR_CUDA;
        }
      }
      if (!s.swap) {
        if (!encode_map(&P.tmA[0], dy, N, M, N, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0)) return TP_ERR_CUDA;
      } else {
        if (!encode_map(&P.tmB[0], dy, N, M, N, s.bn, m3 ? 1 : 0)) return TP_ERR_CUDA;
      }
    }
    if (!s.swap) P.b_idx_gn = 1;
    else P.a_idx_gm = 1;
    for (int k = 0; k < p; ++k) {
      P.out[k] = dx[k];
      P.aux[k] = preact ? const_cast<void*>(preact[k]) : nullptr;
    }
    P.ld_out = K;
    P.ld_aux = K;
    P.epi = preact ? EPI_DGELU : EPI_NONE;
    L.variant = s.swap ? sw_variant_kk(s.bn) : V_KK;
  }
  if (dw_work) TP_TRY(weight_grad(LW, shapes[1], x, nullptr, nullptr, dy, dw, p, M, N, K));
  TP_TRY(run_bwd_pair(LX, dx_work, LW, dw_work, out_dtype, ws, stream, di));
  if (db_work) TP_TRY(bias_grad(&dy, 1, 1, &db, M, N, out_dtype, stream));   // db = sum of dY's rows
  return TP_OK;
}

}  // extern "C"


// ---------------------------------------------------------------- sequence-parallel backward

extern "C" tp_status tp_ag_matmul_bwd(const void* const* x, const void* const* w, const void* const* dy,
                                      void* const* dx, void* const* dw, void* const* db, int p,
                                      int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                                      tp_dtype out_dtype, void* ws, size_t ws_bytes,
                                      cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  if (M % p != 0) return TP_ERR_UNSUPPORTED_SHAPE;
  if (dx == nullptr && dw == nullptr && db == nullptr) return TP_ERR_INVALID_ARG;
  const int64_t Mp = M / p;
  const bool dx_work = dx != nullptr && M > 0 && K > 0;
  const bool dw_work = dw != nullptr && K > 0 && N > 0;
  const bool db_work = db != nullptr && N > 0;
  TP_TRY(check_ptrs(const_cast<const void* const*>(dx), p, dx_work));
  TP_TRY(check_ptrs(w, p, dx_work && N > 0));
  TP_TRY(check_ptrs(dy, p, (dx_work && N > 0) || ((dw_work || db_work) && M > 0)));
  TP_TRY(check_ptrs(const_cast<const void* const*>(db), p, db_work));
  TP_TRY(check_ptrs(x, p, dw_work && M > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(dw), p, dw_work));
  std::vector<Shape> shapes = plan_call(TP_OP_AG_MM_BWD, p, M, N, K, chunk_m, out_dtype, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  {
    std::vector<Range> ins, outs;
    add_ranges(&ins, x, p, Mp * K * 2);
    add_ranges(&ins, w, p, K * N * 2);
    add_ranges(&ins, dy, p, M * N * 2);
    if (dx) add_ranges(&outs, const_cast<const void* const*>(dx), p, Mp * K * esize(out_dtype));
    if (dw) add_ranges(&outs, const_cast<const void* const*>(dw), p, K * N * esize(out_dtype));
    if (db) add_ranges(&outs, const_cast<const void* const*>(db), p, N * esize(out_dtype));
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  if (!dx_work && !dw_work && !db_work) return TP_OK;
  DevInfo di;
  TP_TRY(device_info(&di));
  Launch LX, LW;
  if (dx_work) {
    Launch& L = LX;
    L.shape = shapes[0];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (N > 0) {
      for (int k = 0; k < p; ++k) {
        if (!s.swap) {
          if (!encode_map(&P.tmA[k], dy[k], N, M, N, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0) ||
              !encode_map(&P.tmB[k], w[k], N, K, N, s.pair ? 128 : 256, m3 ? (s.pair ? kPairKChunks : 1) : 0))
            return TP_ERR_CUDA;
        } else {
          if (!encode_map(&P.tmA[k], w[k], N, K, N, BM, m3 ? 1 : 0) ||
              !encode_map(&P.tmB[k], dy[k], N, M, N, s.bn, m3 ? 1 : 0))
            return TP_ERR_CUDA;
        }
      }
    }
    P.a_idx_s = 1;
    P.b_idx_s = 1;
    if (!s.swap) P.a_row_gm = static_cast<int32_t>(Mp);  // groups along M pick their rows of dY_k
    else P.b_col_gn = static_cast<int32_t>(Mp);
    for (int j = 0; j < p; ++j) P.out[j] = dx[j];
    P.ld_out = K;
    P.epi = EPI_NONE;
    L.variant = s.swap ? sw_variant_kk(s.bn) : V_KK;
  }
  if (dw_work) {
    Launch& L = LW;
    L.shape = shapes[1];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (M > 0) {
      for (int t = 0; t < p; ++t) {
        if (!encode_map(&P.tmA[t], x[t], K, Mp, K, s.pair ? PAIR_BK : 64, m3 ? 2 : 0) ||
            !encode_map(&P.tmB[t], dy[t], N, M, N, s.pair ? PAIR_BK : 64, m3 ? (s.pair ? 2 : 4) : 0))
          return TP_ERR_CUDA;
      }
    }
    P.a_idx_s = 1;                                 // segment s reads token shard X_s from row 0
    P.b_idx_gn = 1;                                // group k reads dY_k ...
    P.b_koff_s = static_cast<int32_t>(Mp);         // ... at rows s*M/p of segment s
    for (int k = 0; k < p; ++k) P.out[k] = dw[k];
    P.ld_out = N;
    P.epi = EPI_NONE;
    L.variant = V_MM;
  }
  TP_TRY(run_bwd_pair(LX, dx_work, LW, dw_work, out_dtype, ws, stream, di));
  if (db_work) TP_TRY(bias_grad(dy, p, 1, db, M, N, out_dtype, stream));   // db_k = sum of dY_k's M rows
  return TP_OK;
}

extern "C" tp_status tp_row_linear_bwd_reducescatter(const void* const* x, const void* const* w,
                                                     const void* const* dy, void* const* dx,
                                                     void* const* dw, void* db,
                                                     const void* const* preact, int p, int64_t M,
                                                     int64_t N, int64_t K, int64_t chunk_m,
                                                     tp_dtype out_dtype, void* ws, size_t ws_bytes,
                                                     cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  if (M % p != 0) return TP_ERR_UNSUPPORTED_SHAPE;
  if (dx == nullptr && dw == nullptr && db == nullptr) return TP_ERR_INVALID_ARG;
  const int64_t Mp = M / p;
  const bool dx_work = dx != nullptr && M > 0 && K > 0;
  const bool dw_work = dw != nullptr && K > 0 && N > 0;
  const bool db_work = db != nullptr && N > 0;
  TP_TRY(check_ptrs(const_cast<const void* const*>(dx), p, dx_work));
  TP_TRY(check_ptrs(w, p, dx_work && N > 0));
  TP_TRY(check_ptrs(dy, p, (dx_work && N > 0) || ((dw_work || db_work) && M > 0)));
  TP_TRY(check_ptr(db, db_work));
  TP_TRY(check_ptrs(x, p, dw_work && M > 0));
  TP_TRY(check_ptrs(const_cast<const void* const*>(dw), p, dw_work));
  TP_TRY(check_ptrs(preact, p, dx_work && preact != nullptr));
  std::vector<Shape> shapes = plan_call(TP_OP_ROW_RS_BWD, p, M, N, K, chunk_m, out_dtype, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  {
    std::vector<Range> ins, outs;
    add_ranges(&ins, x, p, M * K * 2);
    add_ranges(&ins, w, p, K * N * 2);
    add_ranges(&ins, dy, p, Mp * N * 2);
    add_ranges(&ins, preact, p, M * K * 2);
    if (dx) add_ranges(&outs, const_cast<const void* const*>(dx), p, M * K * esize(out_dtype));
    if (dw) add_ranges(&outs, const_cast<const void* const*>(dw), p, K * N * esize(out_dtype));
    if (db) outs.push_back({db, static_cast<size_t>(N * esize(out_dtype))});
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  if (!dx_work && !dw_work && !db_work) return TP_OK;
  DevInfo di;
  TP_TRY(device_info(&di));
  const size_t es = esize(out_dtype);
  Launch LX, LW;
  if (dx_work) {
    Launch& L = LX;
    L.shape = shapes[0];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (N > 0) {
      for (int t = 0; t < p; ++t) {
        // shard t of dY (source rows) and weight A_t (output r = t)
        if (!s.swap) {
          if (!encode_map(&P.tmA[t], dy[t], N, Mp, N, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0) ||
              !encode_map(&P.tmB[t], w[t], N, K, N, s.pair ? 128 : 256, m3 ? (s.pair ? kPairKChunks : 1) : 0))
            return TP_ERR_CUDA;
        } else {
          if (!encode_map(&P.tmA[t], w[t], N, K, N, BM, m3 ? 1 : 0) ||
              !encode_map(&P.tmB[t], dy[t], N, Mp, N, s.bn, m3 ? 1 : 0))
            return TP_ERR_CUDA;
        }
      }
    }
    // standard: gm = source shard of dY, gn = output r; swapped: gm = r, gn = source shard
    P.a_idx_gm = 1;
    P.b_idx_gn = 1;
    for (int gm = 0; gm < p; ++gm) {
      for (int gn = 0; gn < p; ++gn) {
        const int r = s.swap ? gm : gn;
        const int src = s.swap ? gn : gm;
        const int64_t off_o = static_cast<int64_t>(src) * Mp * K * es;
        const int64_t off_a = static_cast<int64_t>(src) * Mp * K * 2;
        P.out[gm * p + gn] = static_cast<uint8_t*>(dx[r]) + off_o;
        P.aux[gm * p + gn] = preact ? static_cast<uint8_t*>(const_cast<void*>(preact[r])) + off_a : nullptr;
      }
    }
    P.ld_out = K;
    P.ld_aux = K;
    P.epi = preact ? EPI_DGELU : EPI_NONE;
    L.variant = s.swap ? sw_variant_kk(s.bn) : V_KK;
  }
  if (dw_work) {
    Launch& L = LW;
    L.shape = shapes[1];
    init_params(&L.P);
    fill_common(&L.P, L.shape);
    GemmParams& P = L.P;
    const Shape& s = L.shape;
    const bool m3 = use_3d(N, K);
    P.map3d = m3 ? 1 : 0;
    if (M > 0) {
      for (int t = 0; t < p; ++t) {
        if (!encode_map(&P.tmA[t], x[t], K, M, K, s.pair ? PAIR_BK : 64, m3 ? 2 : 0) ||
            !encode_map(&P.tmB[t], dy[t], N, Mp, N, s.pair ? PAIR_BK : 64, m3 ? (s.pair ? 2 : 4) : 0))
          return TP_ERR_CUDA;
      }
    }
    if (s.Gm == p) P.a_idx_gm = 1;              // group r reads X_r ...
    else P.a_idx_gn = 1;
    P.a_koff_s = static_cast<int32_t>(Mp);      // ... at token rows s*M/p in segment s
    P.b_idx_s = 1;                              // segment s reads dY shard s from row 0
    for (int r = 0; r < p; ++r) P.out[r] = dw[r];
    P.ld_out = N;
    P.epi = EPI_NONE;
    L.variant = V_MM;
  }
  TP_TRY(run_bwd_pair(LX, dx_work, LW, dw_work, out_dtype, ws, stream, di));
  // db = sum over the p token shards of dY, in shard order, of their rows
  if (db_work) TP_TRY(bias_grad(dy, p, p, &db, Mp, N, out_dtype, stream));
  return TP_OK;
}

// ====================================================================== unfused baseline

extern "C" tp_status tp_row_linear_fwd_unfused(const void* const* x, const void* const* w, void* y,
                                               int p, int64_t M, int64_t N, int64_t K,
                                               int64_t chunk_m, tp_dtype out_dtype, int phases,
                                               int flags, void* ws, size_t ws_bytes,
                                               cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  if (phases < 1 || phases > 3) return TP_ERR_INVALID_ARG;
  if ((flags & ~TP_UNFUSED_BF16_COLLECTIVE) != 0) return TP_ERR_INVALID_ARG;
  const bool work = M > 0 && N > 0;
  TP_TRY(check_ptrs(x, p, work && K > 0));
  TP_TRY(check_ptrs(w, p, work && K > 0));
  TP_TRY(check_ptr(y, work));
  std::vector<Shape> shapes = plan_call(TP_OP_ROW_AR_UNFUSED, p, M, N, K, chunk_m, out_dtype, ws_bytes);
  TP_TRY(check_ws(ws, ws_bytes, workspace_for(shapes)));
  if (!work) return TP_OK;
  {
    std::vector<Range> ins, outs;
    add_ranges(&ins, x, p, M * K * 2);
    add_ranges(&ins, w, p, K * N * 2);
    outs.push_back({y, static_cast<size_t>(M * N * esize(out_dtype))});
    if (any_overlap(outs, ins)) return TP_ERR_INVALID_ARG;
  }
  DevInfo di;
  TP_TRY(device_info(&di));
  Launch L;
  L.shape = shapes[0];
  init_params(&L.P);
  fill_common(&L.P, L.shape);
  GemmParams& P = L.P;
  const Shape& s = L.shape;
  const bool m3 = use_3d(N, K);
  P.map3d = m3 ? 1 : 0;
  if (K > 0) {
    for (int r = 0; r < p; ++r) {
      if (!s.swap) {
        if (!encode_map(&P.tmA[r], x[r], K, M, K, BM, m3 ? (s.pair ? kPairKChunks : 1) : 0) ||
            !encode_map(&P.tmB[r], w[r], N, K, N, s.pair ? PAIR_BK : 64, m3 ? (s.pair ? 2 : 4) : 0))
          return TP_ERR_CUDA;
      } else {
        if (!encode_map(&P.tmA[r], w[r], N, K, N, 64, m3 ? 2 : 0) ||
            !encode_map(&P.tmB[r], x[r], K, M, K, s.bn, m3 ? 1 : 0))
          return TP_ERR_CUDA;
      }
    }
  }
  P.a_idx_s = 1;
  P.b_idx_s = 1;
  P.ld_out = N;
  P.epi = EPI_NONE;
  P.out[0] = y;
  L.variant = s.swap ? sw_variant_mk(s.bn) : V_KN;
  L.bf16_chain = (flags & TP_UNFUSED_BF16_COLLECTIVE) != 0;
  return run_launch_phases(L, out_dtype, ws, stream, di, phases);
}

// ====================================================================== no-allocation entry point
//
// Scratch of tp_row_linear_fwd_allreduce_noalloc: a static device array, so
// that callers which cannot allocate device memory still get the split-K
// path.  Host code must not pass `g_noalloc_scratch` itself to a kernel --
// on the host that name is only a stand-in for the device symbol -- but the
// device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// The current context's driver-assigned ID (unique over the process's
// lifetime, unlike the context handle, which may be reused), or 0.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(a);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(b);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current device's primary
// context.  Looked up with that device current on the first call, and again
// whenever the context has changed since (after a cudaDeviceReset the module
// is loaded anew and the array may sit elsewhere).
tp_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  if (bind_device(&dev) != TP_OK) return TP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return TP_ERR_CUDA;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return TP_OK;
}

}  // namespace

extern "C" tp_status tp_row_linear_fwd_allreduce_noalloc(const void* const* x, const void* const* w,
                                                         void* const* y, int n_out, int p,
                                                         int64_t M, int64_t N, int64_t K,
                                                         int64_t chunk_m, tp_dtype out_dtype,
                                                         cudaStream_t stream) {
  TP_TRY(check_sizes(p, M, N, K, chunk_m, out_dtype));
  if (workspace_for(plan_call(TP_OP_ROW_AR, p, M, N, K, chunk_m, out_dtype, TP_NOALLOC_SCRATCH_BYTES)) >
      TP_NOALLOC_SCRATCH_BYTES)
    return TP_ERR_WORKSPACE_TOO_SMALL;
  if (M == 0 || N == 0) return TP_OK;
  void* scratch = nullptr;
  TP_TRY(noalloc_scratch(&scratch));
  return row_fwd_impl(false, x, w, nullptr, y, n_out, p, M, N, K, chunk_m, out_dtype, scratch,
                      TP_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" tp_status tp_noalloc_device_status(cudaStream_t stream) {
  void* scratch = nullptr;
  TP_TRY(noalloc_scratch(&scratch));
  return tp_get_device_status(scratch, stream);
}
