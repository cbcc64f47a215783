// bwd_tcgen05.cu -- attention backward (dQ, dK, dV) for sm_103a.
//
// Gradients of O = softmax(S) V with S = scale * Q K^T [causal], from
// "GPU Engineering: Correctness, Throughput, and Attention" (sections 22.5
// and 22.7): dV = P^T dO, dP = dO V^T, dS = P * (dP - Delta) with the row
// correction Delta = rowsum(dO * O) (the section 22.7 identity), dQ =
// scale * dS K, dK = scale * dS^T Q; P is recomputed tile by tile from the
// forward's log-sum-exp (P = exp(S - LSE)), never stored whole.
//
// Three launches, no atomics (the two gradient kernels each own their
// output rows, so the result is deterministic):
//   bwd_delta_kernel   Delta_i = sum_c dO_ic O_ic, one warp per query row.
//   bwd_dkdv_kernel    one CTA per (b, K/V head, 128-key tile), K and V
//                      resident in shared memory, streaming (Q, dO) tiles of
//                      every query head of the group:
//                        S^T  = K Q^T,  dP^T = V dO^T      (SS MMA -> TMEM)
//                        P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//                        dS^T = P^T * (dP^T - Delta)       (elementwise warps)
//                        dV  += P^T dO,  dK += dS^T Q       (TS MMA, A = TMEM)
//                      TMEM: S^T [0,128) dP^T [128,256) dV [256,384) dK [384,512);
//                      P^T and dS^T overwrite S^T and dP^T as bf16.
//   bwd_dq_kernel      one CTA per (b, h, 128-query tile), Q and dO resident,
//                      streaming (K, V) tiles: S = Q K^T, dP = dO V^T,
//                      dS = P * (dP - Delta), dQ += dS K.
//                      TMEM: S [0,128) dP [128,256) dQ [256,384).
// Warp roles in both: warps 0-7 elementwise (warp w owns TMEM lane quarter
// w % 4 = 32 rows and column half w / 4 = 64 columns), warp 8 single-thread
// MMA issuer, warp 9 TMA producer.  The elementwise work of a tile runs in
// two phases so that it overlaps the tensor core: phase A turns S into P
// while dP is computed, phase B turns dP into dS while the MMA that needs
// only P (dV, or the next tile's S) runs.  Every mbarrier wait is bounded; a
// timeout sets the status word and the CTA leaves cleanly.
// The head dims are compile-time constants of this translation unit: d of
// Q, K (and dQ, dK) and dv of V, O, dO (and dV).  Compiled alone both are
// 128; the bwd_tcgen05_d*.cu files define ATTN_BWD_HEAD_DIM and
// ATTN_BWD_VALUE_DIM and include this file.  Each build exports
// launch_bwd<d, dv>.
#ifndef ATTN_BWD_HEAD_DIM
#define ATTN_BWD_HEAD_DIM 128
#endif
#ifndef ATTN_BWD_VALUE_DIM
#define ATTN_BWD_VALUE_DIM ATTN_BWD_HEAD_DIM
#endif

#include <algorithm>
#include <cuda_bf16.h>

#include "attn.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int D = ATTN_BWD_HEAD_DIM;       // head dim of Q and K
constexpr int DV = ATTN_BWD_VALUE_DIM;     // head dim of V, O and dO
static_assert(((D == 64 || D == 128) && (DV == 64 || DV == 128)) || (D == 96 && DV == 96),
              "head dims 64 and 128 (any pair), or 96 with 96");
constexpr int T = 128;                    // rows per query tile and per key tile
constexpr int kEwWarps = 8;
constexpr int kEwThreads = kEwWarps * 32;
constexpr int kThreads = kEwThreads + 64;
constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
constexpr uint32_t kAtomBytes = 128u * 128u;  // [128 rows][64 bf16] swizzled box
// One [128][d] bf16 tile (Q, K) takes ceil(d / 64) atoms, one [128][dv] tile
// (V, dO) ceil(dv / 64); at 96 the second atom's columns 96-127 are the
// tensor map's zero fill, never read by an MMA.
constexpr int kDAtoms = (D + 63) / 64, kDVAtoms = (DV + 63) / 64;
constexpr uint32_t kQKTileBytes = kDAtoms * kAtomBytes;
constexpr uint32_t kVTileBytes = kDVAtoms * kAtomBytes;
constexpr int kStagesA = 3;  // ring A (Q tiles in the dK/dV kernel, K tiles in the dQ kernel)
constexpr int kStagesB = 2;  // ring B (dO tiles, respectively V tiles)
constexpr uint32_t kIdescSS = idesc_bf16_f32(T, T, 0);  // both operands K-major
constexpr uint32_t kIdescTS = idesc_bf16_f32(T, D, 1);   // B (N = d) MN-major: dK, dQ
constexpr uint32_t kIdescTSV = idesc_bf16_f32(T, DV, 1); // B (N = dv) MN-major: dV
constexpr float kLog2e = 1.4426950408889634074f;

// Shared memory: 2 resident tiles, then ring A (kStagesA tiles: the operand
// the next S needs, so it is prefetched deepest) and ring B (kStagesB tiles),
// then the per-tile row statistics, barriers and bookkeeping.  The rings
// have their own barriers, so a slot is refilled as soon as the last MMA
// that reads it is done.  The dynamic shared memory is declared 1024-byte
// aligned (the 128-byte swizzle needs it) and the kernels check that it is,
// which leaves no room for an alignment slack: 231,592 of 232,448 bytes.
// Resident: a d-wide tile (K, respectively Q) then a dv-wide one (V, dO);
// ring A holds d-wide tiles (Q, respectively K), ring B dv-wide ones (dO, V).
constexpr uint32_t kOffRes = 0;
constexpr uint32_t kOffRes2 = kQKTileBytes;
constexpr uint32_t kOffRingA = kQKTileBytes + kVTileBytes;
constexpr uint32_t kOffRingB = kOffRingA + kStagesA * kQKTileBytes;
constexpr uint32_t kOffStat = kOffRingB + kStagesB * kVTileBytes;  // 2 x [2][128] floats
constexpr uint32_t kOffBar = kOffStat + 2 * 2 * T * 4;
// barriers: res_full, full_a[3], full_b[2], empty_a[3], empty_b[2], s_full,
// dp_full, p (dK/dV kernel: P stored; dQ kernel: S read, its columns free),
// ds (dS stored), acc_full, drain, stats_ready[2] (dK/dV kernel: per-tile row
// statistics written by the elementwise threads, one arrival each)
constexpr int kBarRes = 0, kBarFullA = 1, kBarFullB = kBarFullA + kStagesA,
              kBarEmptyA = kBarFullB + kStagesB, kBarEmptyB = kBarEmptyA + kStagesA,
              kBarS = kBarEmptyB + kStagesB, kBarDP = kBarS + 1, kBarP = kBarDP + 1,
              kBarDS = kBarP + 1, kBarAcc = kBarDS + 1, kBarDrain = kBarAcc + 1,
              kBarStat = kBarDrain + 1, kNumBars = kBarStat + 2;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448 && kSmemBytes > 232448 / 2, "one CTA per SM");
// TMEM columns of the dK/dV kernel's accumulators (after S^T and dP^T).
constexpr uint32_t kColDV = 256, kColDK = 256 + DV;
static_assert(kColDK + D <= 512, "tensor memory budget");
// Status word bit set (and the kernel skipped) if the dynamic shared memory
// were ever not 1024-byte aligned.
constexpr int kStatusMisaligned = 2;

// Packed bf16 operands (P or dS, two values per 32-bit column) are stored
// by column half: half h of a 128-wide row packs its 64 values into the
// first 32 columns of its own 64-column range, so K step kk (16 values)
// sits at column 64 (kk / 4) + 8 (kk % 4).

struct BwdParams {
  const __nv_bfloat16 *o, *dout;
  const float* lse;
  float* delta;
  __nv_bfloat16 *dq, *dk, *dv;
  int* status;
  int64_t B, H, Hkv, Nq, Nk, qoff;
  int64_t kv_per_group;  // dK/dV kernel: K/V heads per scheduling group
  int64_t q_per_group;   // dQ kernel: query heads per scheduling group
  int causal;
  float scale;
  float sc_log2;  // scale * log2(e)
  uint64_t timeout_ns;
};

struct Waiter {
  volatile int* abort_flag;
  int* status;
  uint64_t timeout_ns;
  __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((spin & 31u) == 0) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
          *abort_flag = 1;
          atomicOr(status, 1);
          return false;
        }
      }
    }
  }
};

// K-major SW128 operand (rows = M or N, 128 x 128 bf16 tile): K step kk.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  return sdesc_sw128(tile + (kk >> 2) * kAtomBytes + (kk & 3) * 32, 16, 1024);
}
// MN-major SW128 operand (rows = K, N = d contiguous): K step kk (16 rows).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
  return sdesc_sw128(tile + kk * 16 * 128, kAtomBytes, 1024);
}

// D = A B^T over the W columns of two K-major [128][W] tiles: W / 16 MMAs
// from one elect.sync.
template <int W>
__device__ __forceinline__ void mma_ss_tiles_w(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile) {
  static_assert(W == 64 || W == 96 || W == 128, "tile widths 64, 96 and 128");
  if constexpr (W == 128)
    mma_ss_run8_w(d_tmem, desc_kmajor(a_tile, 0), desc_kmajor(b_tile, 0), kIdescSS, 0u);
  else if constexpr (W == 96)
    mma_ss_run6_w(d_tmem, desc_kmajor(a_tile, 0), desc_kmajor(b_tile, 0), kIdescSS, 0u);
  else
    mma_ss_run4_w(d_tmem, desc_kmajor(a_tile, 0), desc_kmajor(b_tile, 0), kIdescSS, 0u);
}
// D (+)= A B over 128 K rows: A is a packed bf16 operand in tensor memory
// (by column half, as above), B an MN-major [128][N] tile (N = d or dv, as
// `idesc` says); eight MMAs from one elect.sync.
__device__ __forceinline__ void mma_ts_tile_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_tile,
                                              uint32_t idesc, bool accumulate) {
  static_assert(T == 128, "eight K steps of 16");
  mma_ts_run8_halves_w(d_tmem, a_tmem, desc_mnmajor(b_tile, 0), idesc, accumulate ? 1u : 0u);
}

// One [128][W] bf16 tile (ceil(W / 64) swizzle atoms).
template <int W>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int row, int64_t z) {
  for (int a = 0; a < (W + 63) / 64; ++a)
    tma_load_3d(dst + a * kAtomBytes, map, bar, a * 64, row, static_cast<int>(z));
}

// Shared prologue: barriers, TMEM (512 columns), abort flag.
struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  volatile int* abort_flag;
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + kOffBar + 8u * i; }
};

// Callers have checked that smem_raw is 1024-byte aligned.
__device__ __forceinline__ Ctx prologue(uint8_t* smem_raw, int warp) {
  Ctx c;
  c.smem = smem_raw;
  c.sbase = smem_u32(smem_raw);
  c.abort_flag = reinterpret_cast<volatile int*>(c.smem + kOffMisc + 4);
  if (threadIdx.x == 0) {
    mbar_init(c.bar(kBarRes), 1);
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(c.bar(kBarFullA + s), 1);
      mbar_init(c.bar(kBarEmptyA + s), 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(c.bar(kBarFullB + s), 1);
      mbar_init(c.bar(kBarEmptyB + s), 1);
    }
    mbar_init(c.bar(kBarS), 1);
    mbar_init(c.bar(kBarDP), 1);
    mbar_init(c.bar(kBarP), kEwWarps);
    mbar_init(c.bar(kBarDS), kEwWarps);
    mbar_init(c.bar(kBarAcc), 1);
    mbar_init(c.bar(kBarDrain), 1);
    mbar_init(c.bar(kBarStat + 0), kEwThreads);
    mbar_init(c.bar(kBarStat + 1), kEwThreads);
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  uint32_t* slot = reinterpret_cast<uint32_t*>(c.smem + kOffMisc);
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *slot;
  return c;
}

__device__ __forceinline__ void epilogue_sync(const Ctx& c, int warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(c.tmem, 512);
  }
}

// Row statistics of one 128-query tile as the exponent offsets the
// elementwise warps use: nl2[i] = -LSE_i*log2(e) (-inf where the row has no
// admissible key or lies past Nq, so P = 0 there) and nd[i] = -Delta_i.
// Elementwise thread t < 128 supplies nl2[t], thread 128 + t supplies nd[t].
// fetch_stat only loads the raw LSE or Delta (an in-bounds row: past Nq it
// reads row Nq - 1), so nothing waits for the load until put_stat turns the
// value into the offset and stores it into the tile's buffer [nl2 | nd].
__device__ __forceinline__ float fetch_stat(const BwdParams& p, int64_t row_base, int64_t q0,
                                            int t) {
  const int64_t i = min(q0 + (t & (T - 1)), p.Nq - 1);
  return (t < T ? p.lse : p.delta)[row_base + i];
}
__device__ __forceinline__ void put_stat(const BwdParams& p, float* stats, int64_t q0, int t,
                                         float raw) {
  const bool live = q0 + (t & (T - 1)) < p.Nq;
  float v;
  if (t < T)
    v = (!live || raw == -INFINITY) ? -INFINITY : -raw * kLog2e;
  else
    v = live ? -raw : 0.0f;
  stats[(t < T ? 0 : T) + (t & (T - 1))] = v;
}

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                               float mul, bool zero) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * mul, __uint_as_float(v[8 * q + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * mul, __uint_as_float(v[8 * q + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * mul, __uint_as_float(v[8 * q + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * mul, __uint_as_float(v[8 * q + 7]) * mul);
    if (zero) w = make_uint4(0u, 0u, 0u, 0u);
    d4[q] = w;
  }
}

// ======================================================================= Delta
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, int64_t rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto hi = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
  float acc;  // O and dO rows are dv wide
  if constexpr (DV == 128) {  // four elements per lane
    const uint2 a = *reinterpret_cast<const uint2*>(o + row * DV + 4 * lane);
    const uint2 b = *reinterpret_cast<const uint2*>(dout + row * DV + 4 * lane);
    acc = lo(a.x) * lo(b.x) + hi(a.x) * hi(b.x) + lo(a.y) * lo(b.y) + hi(a.y) * hi(b.y);
  } else if constexpr (DV == 96) {  // three elements per lane, 32 apart
    acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 3; ++e)
      acc += __bfloat162float(o[row * DV + 32 * e + lane]) *
             __bfloat162float(dout[row * DV + 32 * e + lane]);
  } else {  // two elements per lane
    const uint32_t a = *reinterpret_cast<const uint32_t*>(o + row * DV + 2 * lane);
    const uint32_t b = *reinterpret_cast<const uint32_t*>(dout + row * DV + 2 * lane);
    acc = lo(a) * lo(b) + hi(a) * hi(b);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// Loader of the two rings: tile n of ring A, then tile n of ring B, each
// into its slot once the slot's previous tile is released.  Before returning
// it waits for every copy it issued (the CTA must not exit with copies in
// flight): per slot only the latest load's phase, which no later load can
// have advanced.
template <typename LoadA, typename LoadB>
__device__ __forceinline__ void run_loader(const Ctx& c, const Waiter& wait, const BwdParams& p,
                                           int n_items, LoadA load_a, LoadB load_b) {
  int last_a = -1, last_b = -1;
  for (int n = 0; n < n_items; ++n) {
    const int sa = static_cast<int>(n % kStagesA), sb = static_cast<int>(n % kStagesB);
    if (n >= kStagesA &&
        !wait(c.bar(kBarEmptyA + sa), static_cast<uint32_t>(((n / kStagesA) - 1) & 1)))
      break;
    mbar_arrive_expect_tx(c.bar(kBarFullA + sa), kQKTileBytes);
    load_a(n, c.bar(kBarFullA + sa));
    last_a = n;
    if (n >= kStagesB &&
        !wait(c.bar(kBarEmptyB + sb), static_cast<uint32_t>(((n / kStagesB) - 1) & 1)))
      break;
    mbar_arrive_expect_tx(c.bar(kBarFullB + sb), kVTileBytes);
    load_b(n, c.bar(kBarFullB + sb));
    last_b = n;
  }
  volatile int no_abort = 0;
  const Waiter own{&no_abort, p.status, p.timeout_ns};
  own(c.bar(kBarRes), 0);
  for (int n = last_a - kStagesA + 1; n <= last_a; ++n)
    if (n >= 0) own(c.bar(kBarFullA + n % kStagesA), static_cast<uint32_t>((n / kStagesA) & 1));
  for (int n = last_b - kStagesB + 1; n <= last_b; ++n)
    if (n >= 0) own(c.bar(kBarFullB + n % kStagesB), static_cast<uint32_t>((n / kStagesB) & 1));
}

// ======================================================================= dK, dV
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem_raw) & 1023u) {  // same for every thread: the whole CTA leaves
    if (threadIdx.x == 0) atomicOr(p.status, kStatusMisaligned);
    return;
  }
  const Ctx c = prologue(smem_raw, warp);
  const Waiter wait{c.abort_flag, p.status, p.timeout_ns};

  // CTA -> (b, K/V head, key tile).  Groups of consecutive K/V heads whose
  // streamed Q and dO fit in L2 together; inside a group key tiles go in
  // ascending order (under a causal mask the first key tiles see the most
  // query tiles), so the CTAs dispatched last are the shortest.
  // Item and head indices are below 2^31 (checked on the host): the
  // divisions run in 32 bits (64-bit ones are slow software routines).
  const int64_t n_kt = (p.Nk + T - 1) / T;
  int64_t bkv, k0;
  {
    const uint32_t kvg = static_cast<uint32_t>(p.kv_per_group);
    const uint32_t per_group = kvg * static_cast<uint32_t>(n_kt);
    const uint32_t u0 = (blockIdx.x / per_group) * kvg;
    const uint32_t r = blockIdx.x % per_group;
    const uint32_t gu = min(kvg, static_cast<uint32_t>(p.B * p.Hkv) - u0);
    bkv = u0 + r % gu;
    k0 = static_cast<int64_t>(r / gu) * T;
  }
  const uint32_t Hkv32 = static_cast<uint32_t>(p.Hkv);
  const int64_t b = static_cast<uint32_t>(bkv) / Hkv32, hk = static_cast<uint32_t>(bkv) % Hkv32;
  const int64_t G = static_cast<uint32_t>(p.H) / Hkv32;
  const int64_t n_qt = (p.Nq + T - 1) / T;
  // First query tile whose rows can see a key of this tile (causal).
  int64_t qt_first = 0;
  if (p.causal) {
    const int64_t need = k0 - p.qoff - (T - 1);  // smallest q0 with q0 + T - 1 + off >= k0
    qt_first = need <= 0 ? 0 : (need + T - 1) / T;
  }
  const int64_t per_head = qt_first < n_qt ? n_qt - qt_first : 0;
  const int n_items = static_cast<int>(G * per_head);  // < 2^31 (host check)
  const uint32_t per_head32 = per_head > 0 ? static_cast<uint32_t>(per_head) : 1u;
  auto item_rows = [&](int n, int64_t& bh, int64_t& q0) {
    const uint32_t g = static_cast<uint32_t>(n) / per_head32;
    bh = b * p.H + hk * G + g;
    q0 = (qt_first + static_cast<uint32_t>(n) % per_head32) * T;
  };

  const uint32_t sK = c.sbase + kOffRes, sV = c.sbase + kOffRes2;
  auto sQ = [&](int n) { return c.sbase + kOffRingA + static_cast<uint32_t>(n % kStagesA) * kQKTileBytes; };
  auto sdO = [&](int n) { return c.sbase + kOffRingB + static_cast<uint32_t>(n % kStagesB) * kVTileBytes; };
  auto slot_a = [](int n) { return n % kStagesA; };
  auto slot_b = [](int n) { return n % kStagesB; };
  auto par_a = [](int n) { return static_cast<uint32_t>((n / kStagesA) & 1); };
  auto par_b = [](int n) { return static_cast<uint32_t>((n / kStagesB) & 1); };
  const uint32_t tS = c.tmem + 0, tdP = c.tmem + 128, tdV = c.tmem + kColDV,
                 tdK = c.tmem + kColDK;

  if (warp == kWarpLoad) {
    if (lane == 0) {
      mbar_arrive_expect_tx(c.bar(kBarRes), kQKTileBytes + kVTileBytes);
      load_tile<D>(sK, &tk, c.bar(kBarRes), static_cast<int>(k0), bkv);
      load_tile<DV>(sV, &tv, c.bar(kBarRes), static_cast<int>(k0), bkv);
      run_loader(
          c, wait, p, n_items,
          [&](int n, uint32_t bar) {
            int64_t bh, q0;
            item_rows(n, bh, q0);
            load_tile<D>(sQ(n), &tq, bar, static_cast<int>(q0), bh);
          },
          [&](int n, uint32_t bar) {
            int64_t bh, q0;
            item_rows(n, bh, q0);
            load_tile<DV>(sdO(n), &tdo, bar, static_cast<int>(q0), bh);
          });
    }
  } else if (warp == kWarpMma) {
    // Issue order per tile n: ... dV(n), S(n+1), dK(n), dP(n+1), ...; the
    // tensor pipe executes in issue order, so S(n+1) overwrites P(n) only
    // after dV(n) read it, and dP(n+1) overwrites dS(n) only after dK(n).
    // dO(n) is released after dV(n), Q(n) after dK(n).
    // The whole warp runs this loop (waits made warp-uniform); the MMA and
    // commit calls elect one lane to issue.
    auto wait_w = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait(b, parity));
    };
    if (n_items > 0) {
      auto issue_s = [&](int n) {  // S^T = K Q^T
        mma_ss_tiles_w<D>(tS, sK, sQ(n));
        mma_commit_w(c.bar(kBarS));
      };
      auto issue_dp = [&](int n) {  // dP^T = V dO^T
        mma_ss_tiles_w<DV>(tdP, sV, sdO(n));
        mma_commit_w(c.bar(kBarDP));
      };
      bool ok = wait_w(c.bar(kBarRes), 0) && wait_w(c.bar(kBarFullA), 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = wait_w(c.bar(kBarFullB), 0);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
      }
      for (int n = 0; n < n_items && ok; ++n) {
        ok = wait_w(c.bar(kBarP), n & 1);
        if (!ok) break;
        tc_fence_after();
        mma_ts_tile_w(tdV, tS, sdO(n), kIdescTSV, n > 0);
        mma_commit_w(c.bar(kBarEmptyB + slot_b(n)));
        const bool more = n + 1 < n_items;
        if (more) {
          ok = wait_w(c.bar(kBarFullA + slot_a(n + 1)), par_a(n + 1));
          if (!ok) break;
          tc_fence_after();
          issue_s(n + 1);
        }
        ok = wait_w(c.bar(kBarDS), n & 1);
        if (!ok) break;
        tc_fence_after();
        mma_ts_tile_w(tdK, tdP, sQ(n), kIdescTS, n > 0);
        mma_commit_w(c.bar(kBarEmptyA + slot_a(n)));
        if (more) {
          ok = wait_w(c.bar(kBarFullB + slot_b(n + 1)), par_b(n + 1));
          if (!ok) break;
          tc_fence_after();
          issue_dp(n + 1);
        }
      }
      if (ok) mma_commit_w(c.bar(kBarAcc));
      mma_commit_w(c.bar(kBarDrain));
      volatile int no_abort = 0;
      const Waiter own{&no_abort, p.status, p.timeout_ns};
      own(c.bar(kBarDrain), 0);
    }
  } else {
    // ---------------------------------------------------------- elementwise
    const int quarter = warp & 3, half = warp >> 2;
    const int jl = (quarter << 5) + lane;  // key row in the tile = TMEM lane
    const int64_t j = k0 + jl;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int col0 = 64 * half;
    float* stat_buf = reinterpret_cast<float*>(c.smem + kOffStat);  // [2][2][128]
    const uint64_t c2 = f2_pack(p.sc_log2, p.sc_log2);
    const bool row_live = j < p.Nk;
    bool ok = true;
    // Each thread supplies one statistic per tile; the eight warps meet on
    // a (bounded) mbarrier per tile, double-buffered by tile parity.  The
    // statistic of tile n + 1 is read from global memory at the start of
    // tile n and stored after tile n's phase B, so its latency hides behind
    // the tile's work.  Slot (n + 1) % 2 last served tile n - 1, whose every
    // reader arrived for tile n (after its phase B of n - 1) before this
    // thread got past tile n's wait.
    if (n_items > 0) {
      int64_t bh, q0;
      item_rows(0, bh, q0);
      put_stat(p, stat_buf, q0, threadIdx.x, fetch_stat(p, bh * p.Nq, q0, threadIdx.x));
      mbar_arrive(c.bar(kBarStat));  // release: this thread's statistic is written
    }
    for (int n = 0; n < n_items; ++n) {
      int64_t bh, q0;
      item_rows(n, bh, q0);
      float* nl2 = stat_buf + (n & 1) * 2 * T;
      float* nd = nl2 + T;
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarStat + (n & 1)), (n >> 1) & 1));
      if (!ok) break;
      float stat_next = 0.0f;
      int64_t q_next = 0;
      if (n + 1 < n_items) {
        int64_t bh1;
        item_rows(n + 1, bh1, q_next);
        stat_next = fetch_stat(p, bh1 * p.Nq, q_next, threadIdx.x);
      }
      // Key j is visible to query i = q0 + col iff j < Nk and (not causal or
      // j <= i + off), i.e. col >= thr.  Tiles where no lane masks any of
      // its columns take the unmasked path.
      const int64_t thr64 = p.causal ? j - q0 - p.qoff : -1;
      const int thr = row_live ? static_cast<int>(thr64 < -1 ? -1 : (thr64 > T ? T : thr64)) : T;
      const bool masked = __any_sync(0xffffffffu, thr > col0);

      // Phase A: P^T = exp2(S^T c - LSE log2e), stored as bf16 over S^T.
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarS), n & 1));
      if (!ok) break;
      tc_fence_after();
      float pf[64];
      {
        uint32_t sr[64];
        tmem_ld_x64(tS + lane_off + col0, sr);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = col0 + 4 * e;
          const float4 l4 = *reinterpret_cast<const float4*>(nl2 + col);
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * e]), __uint_as_float(sr[4 * e + 1])),
                           c2, f2_pack(l4.x, l4.y)),
                    x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * e + 2]), __uint_as_float(sr[4 * e + 3])),
                           c2, f2_pack(l4.z, l4.w)),
                    x2, x3);
          if (masked) {
            if (col < thr) x0 = -INFINITY;
            if (col + 1 < thr) x1 = -INFINITY;
            if (col + 2 < thr) x2 = -INFINITY;
            if (col + 3 < thr) x3 = -INFINITY;
          }
          pf[4 * e] = ex2_approx(x0);
          pf[4 * e + 1] = ex2_approx(x1);
          pf[4 * e + 2] = ex2_approx(x2);
          pf[4 * e + 3] = ex2_approx(x3);
        }
      }
      {
        uint32_t pp[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pp[e] = pack_bf16x2(pf[2 * e], pf[2 * e + 1]);
        tmem_st_x32(tS + lane_off + col0, pp);  // columns this thread has already read
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarP));

      // Phase B: dS^T = P^T (dP^T - Delta), stored as bf16 over dP^T.
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarDP), n & 1));
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t dr[64], pd[32];
        tmem_ld_x64(tdP + lane_off + col0, dr);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = col0 + 4 * e;
          const float4 d4 = *reinterpret_cast<const float4*>(nd + col);
          float t0, t1, t2, t3;
          f2_unpack(f2_mul(f2_pack(pf[4 * e], pf[4 * e + 1]),
                           f2_add(f2_pack(__uint_as_float(dr[4 * e]), __uint_as_float(dr[4 * e + 1])),
                                  f2_pack(d4.x, d4.y))),
                    t0, t1);
          f2_unpack(f2_mul(f2_pack(pf[4 * e + 2], pf[4 * e + 3]),
                           f2_add(f2_pack(__uint_as_float(dr[4 * e + 2]), __uint_as_float(dr[4 * e + 3])),
                                  f2_pack(d4.z, d4.w))),
                    t2, t3);
          pd[2 * e] = pack_bf16x2(t0, t1);
          pd[2 * e + 1] = pack_bf16x2(t2, t3);
        }
        tmem_st_x32(tdP + lane_off + col0, pd);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarDS));
      if (n + 1 < n_items) {
        put_stat(p, stat_buf + ((n + 1) & 1) * 2 * T, q_next, threadIdx.x, stat_next);
        mbar_arrive(c.bar(kBarStat + ((n + 1) & 1)));
      }
    }
    if (ok && n_items > 0) {
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarAcc), 0));
      if (ok) tc_fence_after();
    }
    if (ok) {
      // Each thread stores half of its row's 32-column chunks of dK (chunk
      // cc with cc % 2 = half) and half of those of dV.
      const int64_t kv_row = bkv * p.Nk + j;
#pragma unroll 1
      for (int cc = half; cc < D / 32; cc += 2) {
        const uint32_t col = static_cast<uint32_t>(32 * cc);
        uint32_t kd[32] = {};
        if (n_items > 0) tmem_ld_x32(tdK + lane_off + col, kd);
        if (row_live) store_row_bf16(p.dk + kv_row * D + col, kd, p.scale, n_items == 0);
      }
#pragma unroll 1
      for (int cc = half; cc < DV / 32; cc += 2) {
        const uint32_t col = static_cast<uint32_t>(32 * cc);
        uint32_t vd[32] = {};
        if (n_items > 0) tmem_ld_x32(tdV + lane_off + col, vd);
        if (row_live) store_row_bf16(p.dv + kv_row * DV + col, vd, 1.0f, n_items == 0);
      }
    }
  }
  epilogue_sync(c, warp);
}

// ======================================================================= dQ
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem_raw) & 1023u) {  // same for every thread: the whole CTA leaves
    if (threadIdx.x == 0) atomicOr(p.status, kStatusMisaligned);
    return;
  }
  const Ctx c = prologue(smem_raw, warp);
  const Waiter wait{c.abort_flag, p.status, p.timeout_ns};

  // CTA -> (b, h, query tile).  Groups of consecutive query heads whose K
  // and V fit in L2 together; inside a group query tiles go last first
  // (under a causal mask the last query tiles see the most key tiles).
  // Item and head indices are below 2^31 (checked on the host): 32-bit
  // divisions.
  const int64_t n_qt = (p.Nq + T - 1) / T;
  int64_t bh, q0;
  {
    const uint32_t qg = static_cast<uint32_t>(p.q_per_group);
    const uint32_t per_group = qg * static_cast<uint32_t>(n_qt);
    const uint32_t u0 = (blockIdx.x / per_group) * qg;
    const uint32_t r = blockIdx.x % per_group;
    const uint32_t gu = min(qg, static_cast<uint32_t>(p.B * p.H) - u0);
    bh = u0 + r % gu;
    q0 = (n_qt - 1 - static_cast<int64_t>(r / gu)) * T;
  }
  const uint32_t H32 = static_cast<uint32_t>(p.H), Hkv32 = static_cast<uint32_t>(p.Hkv);
  const int64_t b = static_cast<uint32_t>(bh) / H32, h = static_cast<uint32_t>(bh) % H32;
  const int64_t bkv = b * p.Hkv + static_cast<uint32_t>(h) / (H32 / Hkv32);
  int n_kt = static_cast<int>((p.Nk + T - 1) / T);
  if (p.causal) {
    const int64_t last_key = min(q0 + T - 1, p.Nq - 1) + p.qoff;
    n_kt = last_key < 0 ? 0 : static_cast<int>(min(static_cast<int64_t>(n_kt), last_key / T + 1));
  }

  const uint32_t sQ = c.sbase + kOffRes, sdO = c.sbase + kOffRes2;
  auto sK = [&](int n) { return c.sbase + kOffRingA + static_cast<uint32_t>(n % kStagesA) * kQKTileBytes; };
  auto sV = [&](int n) { return c.sbase + kOffRingB + static_cast<uint32_t>(n % kStagesB) * kVTileBytes; };
  auto slot_a = [](int n) { return n % kStagesA; };
  auto slot_b = [](int n) { return n % kStagesB; };
  auto par_a = [](int n) { return static_cast<uint32_t>((n / kStagesA) & 1); };
  auto par_b = [](int n) { return static_cast<uint32_t>((n / kStagesB) & 1); };
  const uint32_t tS = c.tmem + 0, tdP = c.tmem + 128, tdQ = c.tmem + 256;

  if (warp == kWarpLoad) {
    if (lane == 0 && n_kt > 0) {
      mbar_arrive_expect_tx(c.bar(kBarRes), kQKTileBytes + kVTileBytes);
      load_tile<D>(sQ, &tq, c.bar(kBarRes), static_cast<int>(q0), bh);
      load_tile<DV>(sdO, &tdo, c.bar(kBarRes), static_cast<int>(q0), bh);
      run_loader(
          c, wait, p, n_kt,
          [&](int n, uint32_t bar) { load_tile<D>(sK(n), &tk, bar, n * T, bkv); },
          [&](int n, uint32_t bar) { load_tile<DV>(sV(n), &tv, bar, n * T, bkv); });
    }
  } else if (warp == kWarpMma) {
    // Issue order per tile n: ... S(n+1) (once tile n's S is read), dQ(n),
    // dP(n+1), ...; dP(n+1) overwrites dS(n) only after dQ(n) read it.  V(n)
    // is released after dP(n), K(n) after dQ(n).
    // The whole warp runs this loop (waits made warp-uniform); the MMA and
    // commit calls elect one lane to issue.
    auto wait_w = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait(b, parity));
    };
    if (n_kt > 0) {
      auto issue_s = [&](int n) {  // S = Q K^T
        mma_ss_tiles_w<D>(tS, sQ, sK(n));
        mma_commit_w(c.bar(kBarS));
      };
      auto issue_dp = [&](int n) {  // dP = dO V^T
        mma_ss_tiles_w<DV>(tdP, sdO, sV(n));
        mma_commit_w(c.bar(kBarDP));
        mma_commit_w(c.bar(kBarEmptyB + slot_b(n)));
      };
      bool ok = wait_w(c.bar(kBarRes), 0) && wait_w(c.bar(kBarFullA), 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = wait_w(c.bar(kBarFullB), 0);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
      }
      for (int n = 0; n < n_kt && ok; ++n) {
        const bool more = n + 1 < n_kt;
        if (more) {
          ok = wait_w(c.bar(kBarFullA + slot_a(n + 1)), par_a(n + 1)) &&
               wait_w(c.bar(kBarP), n & 1);  // S(n) read: its columns are free
          if (!ok) break;
          tc_fence_after();
          issue_s(n + 1);
        }
        ok = wait_w(c.bar(kBarDS), n & 1);
        if (!ok) break;
        tc_fence_after();
        mma_ts_tile_w(tdQ, tdP, sK(n), kIdescTS, n > 0);
        mma_commit_w(c.bar(kBarEmptyA + slot_a(n)));
        if (more) {
          ok = wait_w(c.bar(kBarFullB + slot_b(n + 1)), par_b(n + 1));
          if (!ok) break;
          tc_fence_after();
          issue_dp(n + 1);
        }
      }
      if (ok) mma_commit_w(c.bar(kBarAcc));
      mma_commit_w(c.bar(kBarDrain));
      volatile int no_abort = 0;
      const Waiter own{&no_abort, p.status, p.timeout_ns};
      own(c.bar(kBarDrain), 0);
    }
  } else {
    // ---------------------------------------------------------- elementwise
    const int quarter = warp & 3, half = warp >> 2;
    const int il = (quarter << 5) + lane;  // query row in the tile = TMEM lane
    const int64_t i = q0 + il;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int col0 = 64 * half;
    float nl2 = -INFINITY, nd = 0.0f;
    if (i < p.Nq) {
      const float lse = p.lse[bh * p.Nq + i];
      nl2 = (lse == -INFINITY) ? -INFINITY : -lse * kLog2e;
      nd = -p.delta[bh * p.Nq + i];
    }
    const uint64_t c2 = f2_pack(p.sc_log2, p.sc_log2);
    const uint64_t l22 = f2_pack(nl2, nl2);
    const uint64_t nd2 = f2_pack(nd, nd);
    // Last admissible key of this row.
    const int64_t lim = p.causal ? min(p.Nk - 1, i + p.qoff) : p.Nk - 1;
    bool ok = true;
    for (int n = 0; n < n_kt; ++n) {
      const int64_t k0 = static_cast<int64_t>(n) * T;
      const int64_t rel64 = lim - k0;
      const int rel = static_cast<int>(rel64 < -1 ? -1 : (rel64 > T ? T : rel64));
      const bool masked = __any_sync(0xffffffffu, rel < col0 + 63);

      // Phase A: P = exp2(S c - LSE log2e) into registers; S's columns free.
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarS), n & 1));
      if (!ok) break;
      tc_fence_after();
      float pf[64];
      {
        uint32_t sr[64];
        tmem_ld_x64(tS + lane_off + col0, sr);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = col0 + 2 * e;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                           c2, l22),
                    x0, x1);
          if (masked) {
            if (col > rel) x0 = -INFINITY;
            if (col + 1 > rel) x1 = -INFINITY;
          }
          pf[2 * e] = ex2_approx(x0);
          pf[2 * e + 1] = ex2_approx(x1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarP));

      // Phase B: dS = P (dP - Delta), stored as bf16 over dP.
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarDP), n & 1));
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t dr[64], pd[32];
        tmem_ld_x64(tdP + lane_off + col0, dr);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float t0, t1;
          f2_unpack(f2_mul(f2_pack(pf[2 * e], pf[2 * e + 1]),
                           f2_add(f2_pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])),
                                  nd2)),
                    t0, t1);
          pd[e] = pack_bf16x2(t0, t1);
        }
        tmem_st_x32(tdP + lane_off + col0, pd);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarDS));
    }
    if (ok && n_kt > 0) {
      ok = __all_sync(0xffffffffu, wait(c.bar(kBarAcc), 0));
      if (ok) tc_fence_after();
    }
    if (ok) {
      // Each thread stores half of its row's 32-column chunks (chunk cc with
      // cc % 2 = half).
      const bool valid = i < p.Nq;
#pragma unroll 1
      for (int cc = half; cc < D / 32; cc += 2) {
        const uint32_t col = static_cast<uint32_t>(32 * cc);
        uint32_t qd[32] = {};
        if (n_kt > 0) tmem_ld_x32(tdQ + lane_off + col, qd);
        // A row with no admissible key stores +0 exactly (its dS is +-0).
        if (valid)
          store_row_bf16(p.dq + (bh * p.Nq + i) * D + col, qd, p.scale,
                         n_kt == 0 || nl2 == -INFINITY);
      }
    }
  }
  epilogue_sync(c, warp);
}

}  // namespace

template <>
cudaError_t launch_bwd<D, DV>(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t stream) {
  BwdParams p;
  p.o = static_cast<const __nv_bfloat16*>(a.o);
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.status = a.status;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.qoff = a.query_offset;
  p.causal = a.causal;
  p.scale = a.scale;
  p.sc_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.timeout_ns = a.timeout_ns;
  // Scheduling groups sized so that the tiles one group streams (Q and dO of
  // its query heads for the dK/dV kernel, K and V for the dQ kernel) take
  // about 48 MB of L2.
  const int64_t G = a.H / a.Hkv;
  const double q_head_bytes = static_cast<double>(a.Nq) * (D + DV) * 2.0;
  const double kv_head_bytes = static_cast<double>(a.Nk) * (D + DV) * 2.0;
  p.kv_per_group = std::min<int64_t>(
      a.B * a.Hkv, std::max<int64_t>(1, static_cast<int64_t>(48.0e6 / (q_head_bytes * G))));
  p.q_per_group = std::min<int64_t>(
      a.B * a.H, std::max<int64_t>(1, static_cast<int64_t>(48.0e6 / kv_head_bytes)));

  const int64_t rows = a.B * a.H * a.Nq;
  bwd_delta_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p.o, p.dout,
                                                                               a.delta, rows);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  const int64_t n_kt = (a.Nk + T - 1) / T, n_qt = (a.Nq + T - 1) / T;
  bwd_dkdv_kernel<<<static_cast<unsigned>(a.B * a.Hkv * n_kt), kThreads, kSmemBytes, stream>>>(
      tq, tk, tv, tdo, p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  bwd_dq_kernel<<<static_cast<unsigned>(a.B * a.H * n_qt), kThreads, kSmemBytes, stream>>>(
      tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace attn
