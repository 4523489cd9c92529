// Persistent, warp-specialised tcgen05 GEMM for the sharded Linear.
//
// One launch covers a whole sharded-Linear call.  Its tile space is
//   groups along M (Gm) x groups along N (Gn) x m-tiles x n-tiles x splits,
// and its K loop walks S "segments" -- one per rank whose partial product is
// being reduced -- in rank order, each segment being K/64 k-blocks (the
// pair kernel's whole tiles on a deep contraction walk every other wave in
// reverse order; see GemmParams::k_alternate).  All segments of a tile
// accumulate into the same fp32 tensor-memory accumulator, so the
// cross-rank reduction happens in TMEM and the reduced tile is written once.
//
// Roles (320 threads):
//   warp 0     one thread issues TMA loads of A and B k-blocks into a
//              STAGES-deep shared-memory ring (full/empty mbarriers);
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma into
//              one of two TMEM accumulators and commits to the ring's
//              empty barriers and to the accumulator-full barrier;
//   warps 2-9  epilogue: tcgen05.ld the finished accumulator (warp w reads
//              TMEM lanes 32*(w%4)..+31; warps 2-5 take the left half of the
//              columns, warps 6-9 the right half), apply bias / GeLU / GeLU'
//              / cast, stage 128-byte rows in shared memory and store whole
//              lines, then release the accumulator -- overlapping the next
//              tile's MMAs on the other accumulator.
//
// Tiles are visited chunk-major: all tiles of rows chunk c (over every
// N-tile) precede those of chunk c+1, in bands of N-tiles within a chunk,
// so a chunk's write-out overlaps the next chunk's MMAs ("ai-infra-kb
// M027", §02-§03).  Two kernels share this structure: tp_gemm_kernel (one
// CTA per 128 x BN tile, optionally operand-swapped for token tiles below
// 128, with split-K and a second-stage kernel) and tp_gemm_pair_kernel
// (CTA pairs, 256 x 256 tiles via tcgen05.mma.cta_group::2, whose last
// partial wave may run as k-slices that the last-finishing warp sums).
//
// Every mbarrier wait is bounded in time: on expiry the kernel latches an
// error bit in the status word, tells the other roles to stop, waits (again
// bounded) for its own TMA loads and MMAs in flight, frees TMEM and returns.
// An optional trace records per-unit %globaltimer stamps (see
// GemmParams::trace).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace tpf {

constexpr int BM = 128;           // tile rows (UMMA M)
constexpr int BK = 64;            // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int MAX_MAPS = 8;
constexpr int MAX_GROUPS = 64;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;

enum Epi : int32_t { EPI_NONE = 0, EPI_GELU = 1, EPI_DGELU = 2 };

// Status word bits (workspace word 0).
constexpr uint32_t ST_TIMEOUT = 1u;

struct GemmParams {
  CUtensorMap tmA[MAX_MAPS];
  CUtensorMap tmB[MAX_MAPS];
  void* out[MAX_GROUPS];  // per-group output base (group g = gm * Gn + gn)
  void* aux[MAX_GROUPS];  // GELU: H out (nullable); DGELU: H in (bf16)
  const void* bias[MAX_GROUPS];  // per-group bias over the output's columns (bf16, nullable),
                                 // added to the accumulator before the activation
  int32_t Gm, Gn;
  int32_t m_tiles, n_tiles;  // per group
  int32_t chunk_tiles;       // tiles per chunk along the chunked axis
  int32_t chunk_on_n;        // chunks run along GEMM N (operand-swapped kernels)
  int32_t band;              // other-axis tiles per raster band inside a chunk
  int32_t map3d;             // operand maps are 3-D (64-element chunks as the third axis):
                             // one copy per operand per stage
  int32_t num_units;         // Gm*Gn*m_tiles*n_tiles*n_split
  int32_t S;                 // K segments (ranks reduced)
  int32_t kb_per_seg;        // k-blocks per segment
  int32_t n_split;           // split-K factor
  int32_t kb_per_split;      // k-blocks per split over the S*kb_per_seg space
  int32_t a_idx_gm, a_idx_gn, a_idx_s;
  int32_t b_idx_gm, b_idx_gn, b_idx_s;
  int32_t a_row_gm;          // GEMM-M coordinate offset of group gm in its A map
  int32_t b_col_gn;          // GEMM-N coordinate offset of group gn in its B map
  int32_t a_koff_s, b_koff_s;  // K coordinate offset of segment s in the A / B map (a
                               // contraction over tokens that walks the p row shards)
  int32_t rows_g, cols_g;    // valid GEMM rows / cols of one group
  int64_t ld_out, ld_aux;    // row pitch (elements) of out / aux
  int32_t out_f32;           // output is fp32 (else bf16)
  int32_t epi;
  int32_t n_rep;             // replicas of a single-group output (out[0..n_rep))
  float* partial;            // split-K fp32 partials, dense, output orientation
  uint32_t* status;
  uint64_t timeout_ns;
  int32_t debug_drop_q;      // test hook: CTA 0's producer never arms its k-block number
                             // debug_drop_q (-1: off), so a wait runs out of time
  // CTA-pair kernel, last partial wave: units t >= tail_start are k-slices,
  // tail_split per tile, of the tiles tail_start, tail_start + 1, ...
  int32_t tail_start;
  int32_t tail_split;        // 1: no slicing
  float* tail_part;          // fp32 partials of the slices, per (tile, slice, CTA, warp)
  unsigned long long* tail_cnt;  // per (tile, CTA, epilogue warp): slices finished (see finish_slice)
  // optional timeline trace (nullptr: off): per unit t < trace_cap, four
  // words: first MMA issued, accumulator seen full, last warp drained (ns
  // of %globaltimer), and (chunk << 32 | CTA or cluster index)
  unsigned long long* trace;
  int32_t trace_cap;
  // this launch's number (never 0): slice counters left by an earlier launch,
  // finished or stopped, read as zero
  unsigned long long epoch;
  // L2 policies (see l2_policy): of the A and B operand loads (3-D maps), and
  // of the final output stores and the GeLU' epilogue's loads of H
  int32_t a_hint, b_hint, out_hint;
  // CTA-pair kernel: whole tiles of odd waves (a cluster's 2nd, 4th, ...
  // unit of this problem) walk their k-blocks from last to first, so a wave
  // starts on the operand slices the previous wave read last, which are
  // still in L2 where the two waves share panels.
  int32_t k_alternate;
  // Staged epilogue by TMA store (out_tma = 1): group g (replica r) writes
  // its 32-row x 128-byte chunks through tmO[omap[g] + r] at row orow[g] + i,
  // and its GeLU pre-activation through tmH[hmap[g]] at row hrow[g] + i.
  // Boxes are 32 rows x 128 bytes with the staging buffer's 128-byte swizzle.
  int32_t out_tma;
  CUtensorMap tmO[MAX_MAPS];
  CUtensorMap tmH[MAX_MAPS];
  int32_t omap[MAX_GROUPS], orow[MAX_GROUPS];
  int32_t hmap[MAX_GROUPS], hrow[MAX_GROUPS];
};

struct Unit {
  int32_t gm, gn, mt, nt, q0, q1;
  int32_t ch;  // chunk of the chunked axis this tile belongs to
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& P, int32_t t) {
  Unit u;
  const int32_t sp = t % P.n_split;
  const int32_t v = t / P.n_split;
  const int32_t TM = P.Gm * P.m_tiles;
  const int32_t TN = P.Gn * P.n_tiles;
  // Chunked axis C (token rows), other axis O.  Inside a chunk the tiles
  // are rastered in bands of `band` O-tiles: band by band, C then O within
  // the band, so the ~#SM tiles in flight form a (#SM/band) x band block
  // that shares both its A rows and its B columns through L2.
  const int32_t TC = P.chunk_on_n ? TN : TM;
  const int32_t TO = P.chunk_on_n ? TM : TN;
  const int32_t per_chunk = P.chunk_tiles * TO;
  const int32_t c = v / per_chunk;
  const int32_t r = v % per_chunk;
  const int32_t lo = c * P.chunk_tiles;
  const int32_t cnt = min(P.chunk_tiles, TC - lo);
  const int32_t nb = r / (cnt * P.band);
  const int32_t rem = r % (cnt * P.band);
  const int32_t width = min(P.band, TO - nb * P.band);
  const int32_t O = nb * P.band + rem % width;
  const int32_t C = lo + rem / width;
  const int32_t GM = P.chunk_on_n ? O : C;
  const int32_t GN = P.chunk_on_n ? C : O;
  u.gm = GM / P.m_tiles;
  u.mt = GM % P.m_tiles;
  u.gn = GN / P.n_tiles;
  u.nt = GN % P.n_tiles;
  u.ch = c;
  const int32_t kb_total = P.S * P.kb_per_seg;
  u.q0 = sp * P.kb_per_split;
  u.q1 = min(kb_total, u.q0 + P.kb_per_split);
  return u;
}

// Timeline trace (see GemmParams::trace).
__device__ __forceinline__ void trace_mma_start(const GemmParams& P, int32_t t, int32_t ch, uint32_t who) {
  if (P.trace != nullptr && t < P.trace_cap) {
    P.trace[4 * static_cast<size_t>(t)] = globaltimer_ns();
    P.trace[4 * static_cast<size_t>(t) + 3] = (static_cast<unsigned long long>(ch) << 32) | who;
  }
}
__device__ __forceinline__ void trace_acc_full(const GemmParams& P, int32_t t) {
  if (P.trace != nullptr && t < P.trace_cap) P.trace[4 * static_cast<size_t>(t) + 1] = globaltimer_ns();
}
__device__ __forceinline__ void trace_drained(const GemmParams& P, int32_t t) {
  if (P.trace != nullptr && t < P.trace_cap)
    atomicMax(&P.trace[4 * static_cast<size_t>(t) + 2], static_cast<unsigned long long>(globaltimer_ns()));
}

// Pair-kernel unit t: a whole tile, or (t >= tail_start) k-slice tk of tail
// tile tj (tj = -1 for a whole tile).  The slices of a tile split its
// k-blocks into tail_split contiguous ranges.
__device__ __forceinline__ Unit decode_pair_unit(const GemmParams& P, int32_t t, int32_t& tj, int32_t& tk) {
  if (P.tail_split > 1 && t >= P.tail_start) {
    const int32_t i = t - P.tail_start;
    tj = i / P.tail_split;
    tk = i % P.tail_split;
    Unit u = decode_unit(P, P.tail_start + tj);
    const int32_t q0 = u.q0, n = u.q1 - u.q0;
    u.q0 = q0 + tk * n / P.tail_split;
    u.q1 = q0 + (tk + 1) * n / P.tail_split;
    return u;
  }
  tj = -1;
  tk = 0;
  return decode_unit(P, t);
}

// Bounded wait; false on timeout (latched) or when another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const GemmParams& P,
                                         volatile int32_t* abort_flag, uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 127u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > P.timeout_ns) {
        *abort_flag = 1;
        atomicOr(P.status, ST_TIMEOUT | (role << 4));
        return false;
      }
    }
  }
}

// Bounded wait used while shutting down: never latches, never aborts others.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Normal tail Phi(-|h|) and the Gaussian factor e = exp(-h^2 / 2), from
// Abramowitz & Stegun, Handbook of Mathematical Functions (1964), formula
// 7.1.26: for z >= 0, erfc(z) = (a1 t + a2 t^2 + ... + a5 t^5) exp(-z^2) with
// t = 1 / (1 + p z) and an absolute error of at most 1.5e-7.  With
// z = |h| / sqrt(2) the tail is erfc(z) / 2, and exp(-z^2) is e, which the
// GeLU derivative's density term reuses.  The halves of a1..a5 (exact in
// fp32) fold the division by 2 into the polynomial.
constexpr float kTailP = 0.3275911f * 0.70710678118654752f;  // p / sqrt(2): t from |h| directly
constexpr float kTailA1 = 0.5f * 0.254829592f, kTailA2 = 0.5f * -0.284496736f, kTailA3 = 0.5f * 1.421413741f,
                kTailA4 = 0.5f * -1.453152027f, kTailA5 = 0.5f * 1.061405429f;
constexpr float kTailE = -0.72134752044448170f;  // exp(-h^2/2) = 2^(-h^2 log2(e) / 2)
constexpr float kPdf = 0.39894228040143268f;     // 1 / sqrt(2 pi)

__device__ __forceinline__ float normal_tail(float h, float& e) {
  const float t = rcp_approx(fmaf(kTailP, fabsf(h), 1.0f));
  const float q = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kTailA5, kTailA4), kTailA3), kTailA2), kTailA1);
  e = ex2_approx(h * h * kTailE);
  return q * e;
}

// GeLU(h) = h Phi(h) ([TP] §7.1, exact erf form; Phi from the tail above,
// within 3e-7 of the exact value in fp32).
__device__ __forceinline__ float gelu_f(float h) {
  float e;
  const float c = normal_tail(h, e);
  return h * (h >= 0.0f ? fmaf(c, -1.0f, 1.0f) : c);
}

// GeLU'(h) = Phi(h) + h phi(h), phi(h) = e / sqrt(2 pi).
__device__ __forceinline__ float gelu_prime_f(float h) {
  float e;
  const float c = normal_tail(h, e);
  return fmaf(h * e, kPdf, h >= 0.0f ? fmaf(c, -1.0f, 1.0f) : c);
}

// The same for two values at once, in packed fp32 arithmetic: every lane
// performs exactly the operations of the scalar functions above, so the
// results are bit for bit those of gelu_f / gelu_prime_f.
__device__ __forceinline__ void normal_tail2(float h0, float h1, uint64_t& hv, uint64_t& c, uint64_t& e) {
  hv = pk2(h0, h1);
  uint64_t d = fma2(pk2(kTailP, kTailP), pk2(fabsf(h0), fabsf(h1)), pk2(1.0f, 1.0f));
  float d0, d1;
  upk2(d, d0, d1);
  const uint64_t t = pk2(rcp_approx(d0), rcp_approx(d1));
  uint64_t q = fma2(t, pk2(kTailA5, kTailA5), pk2(kTailA4, kTailA4));
  q = fma2(t, q, pk2(kTailA3, kTailA3));
  q = fma2(t, q, pk2(kTailA2, kTailA2));
  q = fma2(t, q, pk2(kTailA1, kTailA1));
  q = mul2(t, q);
  float g0, g1;
  upk2(mul2(mul2(hv, hv), pk2(kTailE, kTailE)), g0, g1);
  e = pk2(ex2_approx(g0), ex2_approx(g1));
  c = mul2(q, e);
}

// Phi of the two values from their tails c (packed): 1 - c where h >= 0.
__device__ __forceinline__ uint64_t phi2(float h0, float h1, uint64_t c) {
  float c0, c1, o0, o1;
  upk2(c, c0, c1);
  upk2(fma2(c, pk2(-1.0f, -1.0f), pk2(1.0f, 1.0f)), o0, o1);
  return pk2(h0 >= 0.0f ? o0 : c0, h1 >= 0.0f ? o1 : c1);
}

__device__ __forceinline__ void gelu2(float& x0, float& x1) {
  uint64_t hv, c, e;
  normal_tail2(x0, x1, hv, c, e);
  upk2(mul2(hv, phi2(x0, x1, c)), x0, x1);
}

// v0, v1 times GeLU'(h0), GeLU'(h1)
__device__ __forceinline__ void times_gelu_prime2(float& v0, float& v1, float h0, float h1) {
  uint64_t hv, c, e;
  normal_tail2(h0, h1, hv, c, e);
  const uint64_t gp = fma2(mul2(hv, e), pk2(kPdf, kPdf), phi2(h0, h1, c));
  upk2(mul2(pk2(v0, v1), gp), v0, v1);
}

__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}




// Scalar epilogue for the transposed (operand-swapped) orientation.
__device__ __forceinline__ void epi_store1(const GemmParams& P, float v, void* out, void* aux,
                                           int64_t off_out, int64_t off_aux) {
  if (P.epi == EPI_GELU) {
    if (aux != nullptr) {
      if (P.out_f32) reinterpret_cast<float*>(aux)[off_aux] = v;
      else reinterpret_cast<__nv_bfloat16*>(aux)[off_aux] = __float2bfloat16_rn(v);
    }
    v = gelu_f(v);
  } else if (P.epi == EPI_DGELU) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(aux)[off_aux];
    v *= gelu_prime_f(bf16_bits_to_f(h));
  }
  if (P.out_f32) reinterpret_cast<float*>(out)[off_out] = v;
  else reinterpret_cast<__nv_bfloat16*>(out)[off_out] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- staged epilogue
//
// Each epilogue warp owns 32 accumulator rows (one per lane) and stages one
// chunk of them at a time in a 4 KiB shared-memory buffer of 32 rows x 128
// bytes, so that global stores (and the loads of H for GeLU') move whole
// 128-byte lines: lane l handles 16-byte unit l % U of row l / U (U units
// per row), instead of one 16-byte piece of each of 32 rows.  Unit u of row r
// sits at r * 128 + 16 * (u ^ (r % 8)): writing a row per lane and reading a
// line per 8 lanes are both free of bank conflicts.

constexpr uint32_t STAGE_BYTES_PER_WARP = 32 * 128;

__device__ __forceinline__ uint32_t stg_off(int r, int u) {
  return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

// rows [0, rows_valid) x units [0, units_valid) of the staged chunk -> global
template <int U>
__device__ __forceinline__ void stage_store(const uint8_t* stg, uint8_t* dst, int64_t ld_bytes,
                                            int rows_valid, int units_valid, int lane, uint64_t policy) {
  constexpr int RPI = 32 / U;  // rows per instruction
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int r = k * RPI + lane / U;
    const int u = lane % U;
    if (r < rows_valid && u < units_valid)
      st_global_v4_hint(dst + r * ld_bytes + u * 16, *reinterpret_cast<const uint4*>(stg + stg_off(r, u)), policy);
  }
}

// global -> staged chunk (the same footprint); rows or units outside the
// valid range are left unwritten
template <int U>
__device__ __forceinline__ void stage_load(uint8_t* stg, const uint8_t* src, int64_t ld_bytes,
                                           int rows_valid, int units_valid, int lane, uint64_t policy) {
  constexpr int RPI = 32 / U;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int r = k * RPI + lane / U;
    const int u = lane % U;
    if (r < rows_valid && u < units_valid)
      *reinterpret_cast<uint4*>(stg + stg_off(r, u)) = ld_global_v4_hint(src + r * ld_bytes + u * 16, policy);
  }
}

// This lane's row of a chunk: 8 units of packed values (bf16: 8 per unit,
// fp32: 4 per unit) into the staging buffer.
template <bool F32, int NV>
__device__ __forceinline__ void stage_row(uint8_t* stg, int lane, const float (&v)[NV]) {
  static_assert(NV == (F32 ? 32 : 64), "one 128-byte row");
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    uint4 q;
    if (F32) {
      q = make_uint4(__float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]), __float_as_uint(v[4 * u + 2]),
                     __float_as_uint(v[4 * u + 3]));
    } else {
      q = make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                     pack_bf16x2(v[8 * u + 4], v[8 * u + 5]), pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
    }
    *reinterpret_cast<uint4*>(stg + stg_off(lane, u)) = q;
  }
}

// NV accumulator columns of this lane's TMEM row starting at taddr.
template <int NV>
__device__ __forceinline__ void load_chunk_tmem(uint32_t taddr, float (&v)[NV]) {
  uint32_t r0[32];
  tmem_ld_32x32b_x32(taddr, r0);
  if constexpr (NV == 64) {
    uint32_t r1[32];
    tmem_ld_32x32b_x32(taddr + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = __uint_as_float(r0[i]);
      v[32 + i] = __uint_as_float(r1[i]);
    }
  } else {
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r0[i]);
  }
}

// One chunk of NV columns (128 bytes of output per row) of the warp's 32
// rows, starting at group column gj0, values v (this lane's row): bias ->
// (H out) -> GeLU / GeLU' -> staged stores.
// The staging buffer may be rewritten: the bulk stores of it this warp
// issued (lane 0) have read it.
__device__ __forceinline__ void stage_free(const GemmParams& P, int lane) {
  if (P.out_tma) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }
}

// The staged chunk (rows gi0.., columns gj0.. of the group) -> global through
// one bulk tensor store issued by lane 0.
__device__ __forceinline__ void stage_store_tma(const CUtensorMap* m, const uint8_t* stg, int32_t x, int32_t y,
                                                bool valid, int lane, uint64_t policy) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && valid) {
    tma_store_2d(m, smem_u32(stg), x, y, policy);
    bulk_commit();
  }
}

template <bool F32>
__device__ __forceinline__ void finish_chunk_staged(const GemmParams& P, int32_t g, int32_t gi0, int32_t gj0,
                                                    float (&v)[F32 ? 32 : 64], uint8_t* stg, int lane) {
  constexpr int NV = F32 ? 32 : 64;
  constexpr int ESZ = F32 ? 4 : 2;
  const int rows_valid = min(32, P.rows_g - gi0);
  const int cols_valid = min(NV, P.cols_g - gj0);     // a multiple of 8 (or <= 0)
  const int units_valid = cols_valid * ESZ / 16;
  const bool any = rows_valid > 0 && cols_valid > 0;
  if (P.bias[g] != nullptr) {
    const uint16_t* b = static_cast<const uint16_t*>(P.bias[g]) + gj0;
#pragma unroll
    for (int i = 0; i < NV; i += 8) {
      if (i < cols_valid) {
        const uint4 q = *reinterpret_cast<const uint4*>(b + i);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[i + 2 * k] += bf16_bits_to_f(static_cast<uint16_t>(w[k] & 0xFFFFu));
          v[i + 2 * k + 1] += bf16_bits_to_f(static_cast<uint16_t>(w[k] >> 16));
        }
      }
    }
  }
  if (P.epi == EPI_GELU) {
    if (P.aux[g] != nullptr) {
      stage_free(P, lane);
      stage_row<F32>(stg, lane, v);
      if (P.out_tma) {
        stage_store_tma(&P.tmH[P.hmap[g]], stg, gj0, P.hrow[g] + gi0, any, lane, l2_policy(P.out_hint));
      } else {
        __syncwarp();
        uint8_t* dst = static_cast<uint8_t*>(P.aux[g]) + (static_cast<int64_t>(gi0) * P.ld_aux + gj0) * ESZ;
        stage_store<8>(stg, dst, P.ld_aux * ESZ, rows_valid, units_valid, lane, l2_policy(P.out_hint));
        __syncwarp();
      }
    }
#pragma unroll
    for (int i = 0; i < NV; i += 2) gelu2(v[i], v[i + 1]);
  } else if (P.epi == EPI_DGELU) {
    // H is bf16: NV * 2 bytes per row
    constexpr int UH = NV * 2 / 16;
    const uint8_t* src = static_cast<const uint8_t*>(P.aux[g]) + (static_cast<int64_t>(gi0) * P.ld_aux + gj0) * 2;
    stage_free(P, lane);
    stage_load<UH>(stg, src, P.ld_aux * 2, rows_valid, cols_valid * 2 / 16, lane, l2_policy(P.out_hint));
    __syncwarp();
#pragma unroll
    for (int u = 0; u < UH; ++u) {
      const uint4 h = *reinterpret_cast<const uint4*>(stg + stg_off(lane, u));
      const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        times_gelu_prime2(v[8 * u + 2 * k], v[8 * u + 2 * k + 1], bf16_bits_to_f(static_cast<uint16_t>(w[k] & 0xFFFFu)),
                          bf16_bits_to_f(static_cast<uint16_t>(w[k] >> 16)));
    }
    __syncwarp();
  }
  stage_free(P, lane);
  stage_row<F32>(stg, lane, v);
  if (P.out_tma) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && any) {
      const uint64_t pol = l2_policy(P.out_hint);
      for (int rep = 0; rep < P.n_rep; ++rep)
        tma_store_2d(&P.tmO[P.omap[g] + rep], smem_u32(stg), gj0, P.orow[g] + gi0, pol);
      bulk_commit();
    }
    return;
  }
  __syncwarp();
  for (int rep = 0; rep < P.n_rep; ++rep) {
    uint8_t* dst = static_cast<uint8_t*>(P.out[g + rep]) + (static_cast<int64_t>(gi0) * P.ld_out + gj0) * ESZ;
    stage_store<8>(stg, dst, P.ld_out * ESZ, rows_valid, units_valid, lane, l2_policy(P.out_hint));
  }
  __syncwarp();
}

// Sum, in slice order k = 0, 1, ..., of the partials of this lane's row for
// NV columns starting at 32-column chunk c32 of the warp's region; slice k's
// region starts at base + k * kstride (float4 units).
template <int NV>
__device__ __forceinline__ void load_chunk_parts(const float4* base, size_t kstride, int nparts, int c32, int lane,
                                                 float (&v)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = 0.f;
  for (int k = 0; k < nparts; ++k) {
#pragma unroll
    for (int h = 0; h < NV / 32; ++h) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float4 q = __ldcg(base + k * kstride + ((c32 + h) * 8 + m) * 32 + lane);
        float* d = &v[32 * h + 4 * m];
        if (k == 0) {
          d[0] = q.x; d[1] = q.y; d[2] = q.z; d[3] = q.w;
        } else {
          d[0] += q.x; d[1] += q.y; d[2] += q.z; d[3] += q.w;
        }
      }
    }
  }
}

// The warp's 128-column half of a tail tile through the staged epilogue,
// values summed from the tail partials.
__device__ __forceinline__ void drain_half_from_parts(const GemmParams& P, int32_t g, int32_t gi0, int32_t gj_half,
                                                      uint8_t* stg, const float4* base, size_t kstride, int nparts) {
  const int lane = threadIdx.x & 31;
  if (P.out_f32) {
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      float v[32];
      load_chunk_parts<32>(base, kstride, nparts, c / 32, lane, v);
      finish_chunk_staged<true>(P, g, gi0, gj_half + c, v, stg, lane);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
      float v[64];
      load_chunk_parts<64>(base, kstride, nparts, c / 32, lane, v);
      finish_chunk_staged<false>(P, g, gi0, gj_half + c, v, stg, lane);
    }
  }
}

// Counts this warp's slice of a (tile, warp) region as finished; true for
// the warp whose slice is the last of n.  A counter holds (launch epoch <<
// 16 | slices finished); one left by another launch counts as zero, so a
// launch stopped part-way (a device timeout) leaves nothing the next launch
// could miscount.  The last warp also sets the counter back to zero, so
// that a launch replayed with the same number (a CUDA graph) starts from
// zero too.  Each compare-and-swap that fails means another of the region's
// n warps succeeded, so at most n attempts are needed; past that bound the
// status word latches an error.
__device__ __forceinline__ bool finish_slice(const GemmParams& P, unsigned long long* cnt, int n) {
  __threadfence();
  __syncwarp();
  uint32_t last = 0;
  if ((threadIdx.x & 31) == 0) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(cnt);
    unsigned long long next = 0;
    bool done = false;
    for (int i = 0; i <= n + 4 && !done; ++i) {
      next = (cur >> 16) == P.epoch ? cur + 1 : ((P.epoch << 16) | 1ull);
      const unsigned long long prev = atomicCAS(cnt, cur, next);
      done = prev == cur;
      cur = prev;
    }
    if (!done) atomicOr(P.status, ST_TIMEOUT | (5u << 4));
    last = done && (next & 0xFFFFull) == static_cast<unsigned long long>(n);
    if (last) atomicExch(cnt, 0ull);  // every slice of the region has arrived: no other writer is left
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// One k-slice of a 256-column accumulator, for one epilogue warp (32 rows x
// 128 columns, half `half`): the slice's fp32 accumulator goes to its
// partial, lane-major (float4 m of 32-column chunk c of lane l at
// ((c * 8 + m) * 32 + l): every warp store and load moves 512 contiguous
// bytes); the warp that finishes its region's last slice sums the n slices
// in slice order 0, 1, ... (the same order whichever warp is last, so the
// result is deterministic) and runs the staged epilogue.  No warp waits for
// another.  Regions: ((tile * n + k) * ncta + cta) * NUM_EPI_WARPS + warp.
__device__ __forceinline__ void drain_slice_wide(const GemmParams& P, const Unit& u, float* part,
                                                 unsigned long long* cnt,
                                                 int32_t tile, int32_t k, int32_t n, int ncta, uint32_t cta,
                                                 int32_t g, int32_t gi, uint32_t t_row, int half, int wslot,
                                                 uint8_t* stg) {
  const int lane = threadIdx.x & 31;
  constexpr size_t region = 32 * 32;  // float4 per warp region (32 rows x 128 columns)
  const size_t kstride = static_cast<size_t>(ncta) * NUM_EPI_WARPS * region;
  const float4* base = reinterpret_cast<const float4*>(part) + static_cast<size_t>(tile) * n * kstride +
                       (static_cast<size_t>(cta) * NUM_EPI_WARPS + wslot) * region;
  float4* mine = const_cast<float4*>(base) + k * kstride;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    load_chunk_tmem<32>(t_row + half * 128 + c * 32, v);
#pragma unroll
    for (int m = 0; m < 8; ++m)
      mine[(c * 8 + m) * 32 + lane] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
  }
  if (!finish_slice(P, cnt + (static_cast<size_t>(tile) * ncta + cta) * NUM_EPI_WARPS + wslot, n)) return;
  drain_half_from_parts(P, g, gi - lane, u.nt * 256 + half * 128, stg, base, kstride, n);
}

// Epilogue of one accumulator for one epilogue warp: columns
// [half*BN/2, (half+1)*BN/2) of TMEM row `t_row` (this thread's lane), i.e.
// GEMM row `gi` of group `g`; raw fp32 partials when the launch splits K.
// With a staging buffer (non-transposed orientation, no split) the output
// goes through drain_chunk_staged in 128-byte-per-row chunks.
template <int BN, bool OUT_T>
__device__ __forceinline__ void drain_tile(const GemmParams& P, const Unit& u, int32_t sp, int32_t g,
                                           int32_t gi, bool row_ok, uint32_t t_row, int half,
                                           uint8_t* stg) {
  constexpr int HALF = BN / 2;
  constexpr int CW = HALF < 32 ? HALF : 32;
  // non-swapped tiles are 256 wide and always drain through the staging
  // buffer (or, with split-K, into the dense partials below)
  static_assert(OUT_T || HALF == 128, "non-swapped tiles are 128 x 256");
  if constexpr (!OUT_T) {
    if (P.n_split == 1) {
      const int lane = threadIdx.x & 31;
      const int32_t gi0 = gi - lane;
      if (P.out_f32) {
#pragma unroll 1
        for (int c0 = half * HALF; c0 < (half + 1) * HALF; c0 += 32) {
          float v[32];
          load_chunk_tmem<32>(t_row + c0, v);
          finish_chunk_staged<true>(P, g, gi0, u.nt * BN + c0, v, stg, lane);
        }
      } else {
#pragma unroll 1
        for (int c0 = half * HALF; c0 < (half + 1) * HALF; c0 += 64) {
          float v[64];
          load_chunk_tmem<64>(t_row + c0, v);
          finish_chunk_staged<false>(P, g, gi0, u.nt * BN + c0, v, stg, lane);
        }
      }
      return;
    }
  }
#pragma unroll 1
  for (int c0 = half * HALF; c0 < (half + 1) * HALF; c0 += CW) {
    uint32_t r[32];
    if constexpr (CW == 32) {
      tmem_ld_32x32b_x32(t_row + c0, r);
    } else if constexpr (CW == 16) {
      tmem_ld_32x32b_x16(t_row + c0, r);
    } else {
      tmem_ld_32x32b_x8(t_row + c0, r);
    }
    tmem_wait_ld();
    if (!row_ok) continue;
    const int32_t gj0 = u.nt * BN + c0;
    if (P.n_split > 1) {
      // raw fp32 partial, dense, in output orientation
      float* part = P.partial + static_cast<int64_t>(sp * P.Gm * P.Gn + g) *
                                    static_cast<int64_t>(P.rows_g) * P.cols_g;
      if (OUT_T) {
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const int32_t gj = gj0 + i;
          if (gj < P.cols_g) part[static_cast<int64_t>(gj) * P.rows_g + gi] = __uint_as_float(r[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < CW; i += 4) {
          const int32_t gj = gj0 + i;
          if (gj < P.cols_g)
            *reinterpret_cast<float4*>(part + static_cast<int64_t>(gi) * P.cols_g + gj) =
                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                            __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
        }
      }
      continue;
    }
    if constexpr (OUT_T) {
      // operand-swapped: GEMM row gi is the output column, so one bias value
      const float bsc = P.bias[g] != nullptr
                            ? bf16_bits_to_f(static_cast<const uint16_t*>(P.bias[g])[gi])
                            : 0.0f;
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const int32_t gj = gj0 + i;
        if (gj < P.cols_g) {
          const int64_t off_o = static_cast<int64_t>(gj) * P.ld_out + gi;
          const int64_t off_a = static_cast<int64_t>(gj) * P.ld_aux + gi;
          for (int rep = 0; rep < P.n_rep; ++rep)
            epi_store1(P, __uint_as_float(r[i]) + bsc, P.out[g + rep], P.aux[g], off_o, off_a);
        }
      }
    }
  }
}

template <bool A_MN, bool B_MN, int BN, bool OUT_T, int STAGES>
struct GemmCfg {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B is loaded in 64-wide boxes");
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                      : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 5;
  static_assert(NUM_BARS * 8 + 16 <= 256, "barriers and the TMEM slot fit in 256 bytes");
  // epilogue staging (non-transposed outputs): 4 KiB per epilogue warp
  // 1024-byte aligned: the staging buffers are 128-byte-swizzled TMA store sources
  static constexpr uint32_t STG_OFF = (STAGES * STAGE_BYTES + 256 + 1023) / 1024 * 1024;
  static constexpr uint32_t STG_BYTES = OUT_T ? 0u : NUM_EPI_WARPS * STAGE_BYTES_PER_WARP;
  // +1024 so the ring can be aligned to 1024 bytes inside dynamic smem
  static constexpr uint32_t SMEM_BYTES = 1024 + STG_OFF + STG_BYTES;
  static_assert(SMEM_BYTES <= 232448, "227 KiB of dynamic shared memory per CTA");
  static constexpr int HALF = BN / 2;                 // columns per epilogue warp
  static constexpr int CW = HALF < 32 ? HALF : 32;  // epilogue columns per TMEM load
};

template <bool A_MN, bool B_MN, int BN, bool OUT_T, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tp_gemm_kernel(const __grid_constant__ GemmParams P) {
  using Cfg = GemmCfg<A_MN, B_MN, BN, OUT_T, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);

  const uint32_t sA0 = base;
  const uint32_t sB0 = base + STAGES * Cfg::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * Cfg::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up above touches no global memory: it overlaps the previous kernel
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      int32_t n_issued = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(P.a_hint);
      const uint64_t pol_b = l2_policy(P.b_hint);
      for (int32_t t = blockIdx.x; t < P.num_units && ok; t += gridDim.x) {
        const Unit u = decode_unit(P, t);
        const int32_t arow = P.a_row_gm * u.gm + u.mt * BM;
        const int32_t bcol = P.b_col_gn * u.gn + u.nt * BN;
        for (int32_t q = u.q0; q < u.q1; ++q) {
          const int32_t s = q / P.kb_per_seg;
          const int32_t kc = (q % P.kb_per_seg) * BK;
          const int32_t kca = kc + s * P.a_koff_s;
          const int32_t kcb = kc + s * P.b_koff_s;
          if (!wait_bar(empty_bar(stage), phase ^ 1u, P, abort_flag, 1u)) {
            ok = false;
            break;
          }
          if (blockIdx.x == 0 && n_issued++ == P.debug_drop_q) {
            // test hook: leave this stage unarmed; its consumer's wait runs out
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const CUtensorMap* am = &P.tmA[P.a_idx_gm * u.gm + P.a_idx_gn * u.gn + P.a_idx_s * s];
          const CUtensorMap* bm = &P.tmB[P.b_idx_gm * u.gm + P.b_idx_gn * u.gn + P.b_idx_s * s];
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
          const uint32_t sa = sA0 + stage * Cfg::A_BYTES;
          const uint32_t sb = sB0 + stage * Cfg::B_BYTES;
          if (P.map3d) {
            if (A_MN) tma_load_3d(sa, am, fb, 0, kca, arow / 64, pol_a);
            else tma_load_3d(sa, am, fb, 0, arow, kca / 64, pol_a);
            if (B_MN) tma_load_3d(sb, bm, fb, 0, kcb, bcol / 64, pol_b);
            else tma_load_3d(sb, bm, fb, 0, bcol, kcb / 64, pol_b);
          } else {
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j) tma_load_2d(sa + j * (64 * BK * 2), am, fb, arow + 64 * j, kca);
            } else {
              tma_load_2d(sa, am, fb, kca, arow);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * (64 * BK * 2), bm, fb, bcol + 64 * j, kcb);
            } else {
              tma_load_2d(sb, bm, fb, kcb, bcol);
            }
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every armed stage's last phase completes once its bytes have landed.
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) drain_wait(full_bar(s), (armed_parity >> s) & 1u, P.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int32_t t = blockIdx.x; t < P.num_units && ok; t += gridDim.x) {
        const Unit u = decode_unit(P, t);
        if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, P, abort_flag, 2u)) break;
        tc_fence_after();
        trace_mma_start(P, t, u.ch, blockIdx.x);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int32_t q = u.q0; q < u.q1; ++q) {
          if (!wait_bar(full_bar(stage), phase, P, abort_flag, 3u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sA0 + stage * Cfg::A_BYTES;
          const uint32_t sb = sB0 + stage * Cfg::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t ad = A_MN ? make_sw128_desc(sa + kk * (UMMA_K * 128), 64 * BK * 2, 1024)
                                     : make_sw128_desc(sa + kk * (UMMA_K * 2), 16, 1024);
            const uint64_t bd = B_MN ? make_sw128_desc(sb + kk * (UMMA_K * 128), 64 * BK * 2, 1024)
                                     : make_sw128_desc(sb + kk * (UMMA_K * 2), 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (q > u.q0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread complete before TMEM is freed.
      umma_commit(drain_bar);
      drain_wait(drain_bar, 0, P.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;
    const int row_in_tile = 32 * q + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int32_t t = blockIdx.x; t < P.num_units; t += gridDim.x) {
      const Unit u = decode_unit(P, t);
      bool ok = wait_bar(tfull_bar(acc), acc_phase, P, abort_flag, 4u);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();

      const int32_t g = u.gm * P.Gn + u.gn;
      const int32_t gi = u.mt * BM + row_in_tile;  // GEMM row within the group
      const bool row_ok = gi < P.rows_g;
      const int32_t sp = t % P.n_split;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * BN);
      uint8_t* stg = OUT_T ? nullptr
                           : base_ptr + Cfg::STG_OFF + (warp - 2) * STAGE_BYTES_PER_WARP;
      if (warp == 2 && lane == 0) trace_acc_full(P, t);
      drain_tile<BN, OUT_T>(P, u, sp, g, gi, row_ok, t_row, half, stg);
      if (lane == 0) trace_drained(P, t);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // this warp's bulk stores complete before the CTA exits
    if (P.out_tma && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------- CTA-pair kernel
//
// The same tile space with 256 x 256 tiles, each computed by a cluster of
// two CTAs on two SMs: tcgen05.mma.cta_group::2 (M = 256, N = 256) reads CTA
// r's 128 rows of A and 128 columns of B from CTA r's shared memory and
// writes CTA r's 128 rows of the accumulator into CTA r's tensor memory, so
// each SM stages 32 KiB per k-block instead of the 48 KiB of a 128 x 256
// tile; k-blocks are PAIR_BK = 128 deep (3 stages of 64 KiB per CTA), which
// halves the barrier round trips and copies per byte.  Protocol:
//   - both producers wait on their own empty barrier, then load their
//     halves; every load counts its bytes on the full barrier of CTA 0,
//     whose producer arms it for both halves;
//   - one thread of CTA 0 issues the pair MMAs and commits to the empty
//     and accumulator-full barriers of both CTAs (multicast);
//   - each CTA's epilogue warps drain its own tensor memory and release the
//     accumulator on CTA 0's accumulator-empty barrier;
//   - both CTAs meet at a cluster barrier before tensor memory is freed.

constexpr int PAIR_BK = 128;  // k-block depth of the pair kernel: 64 KiB stages, fewer round trips

template <bool A_MN, bool B_MN, int BKP>
struct PairCfg {
  static constexpr int BN = 256;                       // pair tile N
  static constexpr int BNH = 128;                      // B columns held by each CTA
  static constexpr uint32_t A_BYTES = BM * BKP * 2;    // 32 KiB at BKP = 128
  static constexpr uint32_t B_BYTES = BNH * BKP * 2;   // 32 KiB
  static constexpr int STAGES = (192 * 1024) / (A_BYTES + B_BYTES);
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 5;
  static_assert(NUM_BARS * 8 + 16 <= 256, "barriers and the TMEM slot fit in 256 bytes");
  static constexpr uint32_t STG_OFF = (STAGES * STAGE_BYTES + 256 + 1023) / 1024 * 1024;
  static constexpr uint32_t SMEM_BYTES = 1024 + STG_OFF + NUM_EPI_WARPS * STAGE_BYTES_PER_WARP;
  static_assert(SMEM_BYTES <= 232448, "227 KiB of dynamic shared memory per CTA");
};

// One launch of the pair kernel may carry two independent GEMM problems
// (the dX and dW products of one backward call): units [0, split) are problem
// 0's, units [split, total) problem 1's, on the same clusters, so the two
// share one fill, one drain and one partial last wave.
struct PairLaunch2 {
  GemmParams P[2];
  int32_t split;  // units of problem 0
  int32_t total;  // units of both problems
};

// Body of the CTA-pair kernel over NPROB problems (1 or 2): problem i has
// operand majors (A_i, B_i).  Launch-wide state -- the status word, the
// device wait limit, the trace and the test hook -- comes from problem 0.
template <bool A0, bool B0, bool A1, bool B1, int BKP, bool TAIL, int NPROB>
__device__ __forceinline__ void pair_body(const GemmParams* Ps, int32_t split, int32_t total) {
  using Cfg = PairCfg<A0, B0, BKP>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int KC = BKP / 64;  // 64-wide K chunks per k-block
  static_assert(NPROB == 1 || !TAIL, "last-wave slices only in single-problem launches");
  const GemmParams& P = Ps[0];
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);

  const uint32_t sA0 = base;
  const uint32_t sB0 = base + STAGES * Cfg::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * Cfg::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int32_t first = static_cast<int32_t>(blockIdx.x >> 1);
  const int32_t stride = static_cast<int32_t>(gridDim.x >> 1);
  // problem of unit t, and t's index within it
  auto prob_of = [&](int32_t t) -> int { return (NPROB == 2 && t >= split) ? 1 : 0; };
  auto local = [&](int32_t t, int pi) -> int32_t { return pi ? t - split : t; };
  // whole tiles of a cluster's odd units (within their problem) reverse K
  auto k_reversed = [&](const GemmParams& Q, int32_t t, int pi, int32_t tj) -> bool {
    return Q.k_alternate != 0 && tj < 0 && ((local(t, pi) / stride) & 1) != 0;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up above touches no global memory: it overlaps the previous kernel
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producers (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      int32_t n_issued = 0;
      bool ok = true;
      uint64_t pol_a[NPROB], pol_b[NPROB];
#pragma unroll
      for (int i = 0; i < NPROB; ++i) {
        pol_a[i] = l2_policy(Ps[i].a_hint);
        pol_b[i] = l2_policy(Ps[i].b_hint);
      }
      for (int32_t t = first; t < total && ok; t += stride) {
        const int pi = prob_of(t);
        const GemmParams& Q = Ps[pi];
        const bool a_mn = pi ? A1 : A0;
        const bool b_mn = pi ? B1 : B0;
        int32_t tj = -1, tk = 0;
        const Unit u = TAIL ? decode_pair_unit(Q, t, tj, tk) : decode_unit(Q, local(t, pi));
        const int32_t arow = Q.a_row_gm * u.gm + u.mt * (2 * BM) + static_cast<int32_t>(crank) * BM;
        const int32_t bcol = Q.b_col_gn * u.gn + u.nt * Cfg::BN + static_cast<int32_t>(crank) * Cfg::BNH;
        const bool rev = k_reversed(Q, t, pi, tj);
        for (int32_t i = u.q0; i < u.q1; ++i) {
          const int32_t q = rev ? u.q0 + u.q1 - 1 - i : i;
          const int32_t s = q / Q.kb_per_seg;
          const int32_t kc = (q % Q.kb_per_seg) * BKP;
          const int32_t kca = kc + s * Q.a_koff_s;
          const int32_t kcb = kc + s * Q.b_koff_s;
          if (!wait_bar(empty_bar(stage), phase ^ 1u, P, abort_flag, 1u)) {
            ok = false;
            break;
          }
          if (blockIdx.x == 0 && n_issued++ == P.debug_drop_q) {
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const CUtensorMap* am = &Q.tmA[Q.a_idx_gm * u.gm + Q.a_idx_gn * u.gn + Q.a_idx_s * s];
          const CUtensorMap* bm = &Q.tmB[Q.b_idx_gm * u.gm + Q.b_idx_gn * u.gn + Q.b_idx_s * s];
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * Cfg::STAGE_BYTES);
          const uint32_t sa = sA0 + stage * Cfg::A_BYTES;
          const uint32_t sb = sB0 + stage * Cfg::B_BYTES;
          // Shared-memory tiles: K-major operands as KC consecutive [rows][64]
          // sub-tiles (one per 64-wide K chunk), MN-major operands as
          // consecutive [BKP K-rows][64] sub-tiles (one per 64-wide MN block).
          if (Q.map3d) {
            if (a_mn) tma_load_3d_pair(sa, am, fb, 0, kca, arow / 64, pol_a[pi]);
            else tma_load_3d_pair(sa, am, fb, 0, arow, kca / 64, pol_a[pi]);
            if (b_mn) tma_load_3d_pair(sb, bm, fb, 0, kcb, bcol / 64, pol_b[pi]);
            else tma_load_3d_pair(sb, bm, fb, 0, bcol, kcb / 64, pol_b[pi]);
          } else {
            if (a_mn) {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j)
                tma_load_2d_pair(sa + j * (64 * BKP * 2), am, fb, arow + 64 * j, kca);
            } else {
#pragma unroll
              for (int h = 0; h < KC; ++h) tma_load_2d_pair(sa + h * (BM * 128), am, fb, kca + 64 * h, arow);
            }
            if (b_mn) {
#pragma unroll
              for (int j = 0; j < Cfg::BNH / 64; ++j)
                tma_load_2d_pair(sb + j * (64 * BKP * 2), bm, fb, bcol + 64 * j, kcb);
            } else {
#pragma unroll
              for (int h = 0; h < KC; ++h)
                tma_load_2d_pair(sb + h * (Cfg::BNH * 128), bm, fb, kcb + 64 * h, bcol);
            }
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // CTA 0's full barriers count both CTAs' bytes: once its armed stages
      // complete, every load of the pair for them has landed.
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) drain_wait(full_bar(s), (armed_parity >> s) & 1u, P.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ pair MMA issuer (CTA 0)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int32_t t = first; t < total && ok; t += stride) {
        const int pi = prob_of(t);
        const GemmParams& Q = Ps[pi];
        const bool a_mn = pi ? A1 : A0;
        const bool b_mn = pi ? B1 : B0;
        const uint32_t idesc = pi ? make_idesc_bf16(2 * BM, Cfg::BN, A1, B1) : make_idesc_bf16(2 * BM, Cfg::BN, A0, B0);
        int32_t tj = -1, tk = 0;
        const Unit u = TAIL ? decode_pair_unit(Q, t, tj, tk) : decode_unit(Q, local(t, pi));
        if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, P, abort_flag, 2u)) break;
        tc_fence_after();
        trace_mma_start(P, t, u.ch, blockIdx.x >> 1);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::BN);
        // the k-blocks arrive in the producer's order (forward or reversed);
        // only the first one of the unit overwrites the accumulator
        for (int32_t q = u.q0; q < u.q1; ++q) {
          if (!wait_bar(full_bar(stage), phase, P, abort_flag, 3u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sA0 + stage * Cfg::A_BYTES;
          const uint32_t sb = sB0 + stage * Cfg::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BKP / UMMA_K; ++kk) {
            // K-major: chunk kk/4, 32-byte step (kk%4) inside the swizzled row;
            // MN-major: 16 K-rows of 128 bytes per step.
            const uint32_t ka = (kk / 4) * (BM * 128) + (kk % 4) * (UMMA_K * 2);
            const uint32_t kb = (kk / 4) * (Cfg::BNH * 128) + (kk % 4) * (UMMA_K * 2);
            const uint64_t ad = a_mn ? make_sw128_desc(sa + kk * (UMMA_K * 128), 64 * BKP * 2, 1024)
                                     : make_sw128_desc(sa + ka, 16, 1024);
            const uint64_t bd = b_mn ? make_sw128_desc(sb + kk * (UMMA_K * 128), 64 * BKP * 2, 1024)
                                     : make_sw128_desc(sb + kb, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (q > u.q0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(empty_bar(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(tfull_bar(acc), 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit_pair(drain_bar, 0x1);
      drain_wait(drain_bar, 0, P.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) / 4;
    const int row_in_tile = 32 * q + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int32_t t = first; t < total; t += stride) {
      const int pi = prob_of(t);
      const GemmParams& Q = Ps[pi];
      int32_t tj = -1, tk = 0;
      const Unit u = TAIL ? decode_pair_unit(Q, t, tj, tk) : decode_unit(Q, local(t, pi));
      bool ok = wait_bar(tfull_bar(acc), acc_phase, P, abort_flag, 4u);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      const int32_t g = u.gm * Q.Gn + u.gn;
      const int32_t gi = u.mt * (2 * BM) + static_cast<int32_t>(crank) * BM + row_in_tile;
      const bool row_ok = gi < Q.rows_g;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * Cfg::BN);
      uint8_t* stg = base_ptr + Cfg::STG_OFF + (warp - 2) * STAGE_BYTES_PER_WARP;
      if (leader && warp == 2 && lane == 0) trace_acc_full(P, t);
      if (TAIL && tj >= 0)
        drain_slice_wide(Q, u, Q.tail_part, Q.tail_cnt, tj, tk, Q.tail_split, 2, crank, g, gi, t_row, half,
                         warp - 2, stg);
      else drain_tile<Cfg::BN, false>(Q, u, 0, g, gi, row_ok, t_row, half, stg);
      if (lane == 0) trace_drained(P, t);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // this warp's bulk stores complete before the CTA exits
    bool any_tma = P.out_tma != 0;
    if (NPROB == 2) any_tma = any_tma || Ps[NPROB - 1].out_tma != 0;
    if (any_tma && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (*abort_flag) {
    // after a timeout, give the peer's copies into this CTA time to land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  __syncwarp();
  cluster_sync_all();  // no CTA frees tensor memory or exits while its peer may use it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// TAIL: the launch runs its last partial wave as k-slices (P.tail_split >
// 1).  A separate instantiation, so that launches without slices carry none
// of that code.
template <bool A_MN, bool B_MN, int BKP, bool TAIL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tp_gemm_pair_kernel(const __grid_constant__ GemmParams P) {
  pair_body<A_MN, B_MN, A_MN, B_MN, BKP, TAIL, 1>(&P, P.num_units, P.num_units);
}

// Two problems in one launch (PairLaunch2), majors (A0, B0) then (A1, B1).
template <bool A0, bool B0, bool A1, bool B1, int BKP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tp_gemm_pair2_kernel(const __grid_constant__ PairLaunch2 L) {
  pair_body<A0, B0, A1, B1, BKP, false, 2>(L.P, L.split, L.total);
}

// ------------------------------------------------------------- split-K stage 2

struct ReduceParams {
  void* out[MAX_GROUPS];
  void* aux[MAX_GROUPS];
  const void* bias[MAX_GROUPS];  // as GemmParams::bias, indexed by the output column b
  const float* partial;
  int32_t G;          // groups
  int32_t A, B;       // output-orientation extents of one group (B contiguous)
  int64_t ld_out, ld_aux;
  int32_t out_f32, epi, n_split, n_rep;
  int32_t bf16_chain;  // 1: round every partial and every running sum to bf16
};

__device__ __forceinline__ float bf16_round_f(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// out[g][a, b] = epilogue( sum_{s=0}^{n_split-1} partial[s][g][a][b] ), the
// partials summed in split order; 4 consecutive b per thread.  With
// bf16_chain the sum is the one a bf16 collective forms from bf16 partials:
// acc = bf16(P_0), then acc = bf16(acc + bf16(P_s)) for s = 1, 2, ...
// n_split == 0 (a contraction of length zero) sums nothing: out = epilogue(bias).
__global__ void tp_splitk_reduce_kernel(const __grid_constant__ ReduceParams R) {
  const int64_t per_group = static_cast<int64_t>(R.A) * R.B;
  const int64_t total4 = static_cast<int64_t>(R.G) * per_group / 4;
  const int64_t split_stride = static_cast<int64_t>(R.G) * per_group;
  for (int64_t i4 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i4 < total4;
       i4 += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i4 * 4;
    float4 acc = R.n_split > 0 ? *reinterpret_cast<const float4*>(R.partial + e)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    if (R.bf16_chain) {
      acc = make_float4(bf16_round_f(acc.x), bf16_round_f(acc.y), bf16_round_f(acc.z),
                        bf16_round_f(acc.w));
      for (int s = 1; s < R.n_split; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(R.partial + s * split_stride + e);
        acc.x = bf16_round_f(acc.x + bf16_round_f(v.x));
        acc.y = bf16_round_f(acc.y + bf16_round_f(v.y));
        acc.z = bf16_round_f(acc.z + bf16_round_f(v.z));
        acc.w = bf16_round_f(acc.w + bf16_round_f(v.w));
      }
    } else {
      // four splits' loads in flight at a time; the additions stay in split order
      int s = 1;
      for (; s + 3 < R.n_split; s += 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const float4*>(R.partial + (s + j) * split_stride + e);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc.x += v[j].x;
          acc.y += v[j].y;
          acc.z += v[j].z;
          acc.w += v[j].w;
        }
      }
      for (; s < R.n_split; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(R.partial + s * split_stride + e);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
    const int32_t g = static_cast<int32_t>(e / per_group);
    const int64_t rem = e % per_group;
    const int64_t a = rem / R.B;
    const int64_t b = rem % R.B;
    if (R.bias[g] != nullptr) {
      const uint2 q = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(R.bias[g]) + b);
      acc.x += bf16_bits_to_f(static_cast<uint16_t>(q.x & 0xFFFFu));
      acc.y += bf16_bits_to_f(static_cast<uint16_t>(q.x >> 16));
      acc.z += bf16_bits_to_f(static_cast<uint16_t>(q.y & 0xFFFFu));
      acc.w += bf16_bits_to_f(static_cast<uint16_t>(q.y >> 16));
    }
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    if (R.epi == EPI_GELU) {
      if (R.aux[g] != nullptr) {
        if (R.out_f32) {
          *reinterpret_cast<float4*>(static_cast<float*>(R.aux[g]) + a * R.ld_aux + b) = acc;
        } else {
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(R.aux[g]) + a * R.ld_aux + b) =
              make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = gelu_f(v[i]);
    } else if (R.epi == EPI_DGELU) {
      const uint2 h = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(R.aux[g]) +
                                                      a * R.ld_aux + b);
      v[0] *= gelu_prime_f(bf16_bits_to_f(static_cast<uint16_t>(h.x & 0xFFFFu)));
      v[1] *= gelu_prime_f(bf16_bits_to_f(static_cast<uint16_t>(h.x >> 16)));
      v[2] *= gelu_prime_f(bf16_bits_to_f(static_cast<uint16_t>(h.y & 0xFFFFu)));
      v[3] *= gelu_prime_f(bf16_bits_to_f(static_cast<uint16_t>(h.y >> 16)));
    }
    for (int rep = 0; rep < R.n_rep; ++rep) {
      if (R.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(R.out[g + rep]) + a * R.ld_out + b) =
            make_float4(v[0], v[1], v[2], v[3]);
      } else {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(R.out[g + rep]) + a * R.ld_out + b) =
            make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
      }
    }
  }
}

// ---------------------------------------------------------------- bias gradient

struct BiasGradParams {
  const void* src[MAX_MAPS];  // bf16 [rows, N] row-major sources
  void* out[MAX_MAPS];        // [N] outputs
  int32_t src_per_out;        // output o sums sources o*src_per_out .. (o+1)*src_per_out-1, in order
  int32_t N;
  int64_t rows;               // rows of every source
  int32_t out_f32;
};

constexpr int BG_COLS = 64;   // columns per CTA: 8 threads x 8 bf16 (one 16-byte load each)
constexpr int BG_LANES = 32;  // row lanes per CTA

// out[o][j] = sum over the sources of o, in order, and over their rows of
// src[i, j].  CTA (blockIdx.x, blockIdx.y = o) owns 64 columns; thread
// (lane, cg) sums rows lane, lane + 32, ... of 8 columns with 16-byte loads
// (a warp reads four 128-byte row segments), then the 32 lanes are summed in
// lane order through shared memory: the result does not depend on timing.
__global__ void __launch_bounds__(BG_COLS / 8 * BG_LANES)
    tp_bias_grad_kernel(const __grid_constant__ BiasGradParams B) {
  __shared__ float red[BG_LANES][BG_COLS + 1];
  const int cg = threadIdx.x % (BG_COLS / 8);
  const int lane = threadIdx.x / (BG_COLS / 8);
  const int o = blockIdx.y;
  const int32_t c0 = blockIdx.x * BG_COLS + cg * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c0 < B.N && B.rows > 0) {
    for (int s = 0; s < B.src_per_out; ++s) {
      const uint16_t* src = static_cast<const uint16_t*>(B.src[o * B.src_per_out + s]) + c0;
#pragma unroll 4
      for (int64_t i = lane; i < B.rows; i += BG_LANES) {
        const uint4 q = *reinterpret_cast<const uint4*>(src + i * B.N);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] += bf16_bits_to_f(static_cast<uint16_t>(w[k] & 0xFFFFu));
          acc[2 * k + 1] += bf16_bits_to_f(static_cast<uint16_t>(w[k] >> 16));
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[lane][cg * 8 + k] = acc[k];
  __syncthreads();
  if (threadIdx.x < BG_COLS) {
    const int32_t col = blockIdx.x * BG_COLS + threadIdx.x;
    float sum = 0.f;
    for (int l = 0; l < BG_LANES; ++l) sum += red[l][threadIdx.x];
    if (col < B.N) {
      if (B.out_f32) static_cast<float*>(B.out[o])[col] = sum;
      else static_cast<__nv_bfloat16*>(B.out[o])[col] = __float2bfloat16_rn(sum);
    }
  }
}

}  // namespace tpf
