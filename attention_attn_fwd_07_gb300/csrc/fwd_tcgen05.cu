// fwd_tcgen05.cu -- fused attention forward (prefill) for sm_103a.
//
// Computes, per (batch*head, query row), O = softmax(scale * Q K^T [causal]) V
// and LSE = ln sum exp(scores), by the online-softmax recurrence of
// "GPU Engineering: Correctness, Throughput, and Attention" (section 22.5:
// running maximum m, normaliser l, unnormalised accumulator o; old state is
// rescaled by exp(m - m_new) when the maximum grows; output o / l), with the
// section 22.7 lab's conventions (causal rule j > i + query_offset applied
// before maxima and sums, "safe" exponent reference 0 for a row that is still
// fully masked, output 0 and LSE -inf for a row with no admissible key,
// LSE = m + ln l).  The score tile lives only in tensor memory; nothing of
// size Nq x Nk touches device memory.
//
// Two kernels share the roles below.  attn_fwd_tcgen05_kernel: one CTA per
// work item of 256 query rows of one (b,h) as two 128-row tiles A and B that
// share every K/V tile, read from the query head's K/V head when K/V heads
// are grouped (prior art: the producer/consumer, TMA-fed, on-chip
// accumulator pipeline described for FlashAttention-3 on H100; here rebuilt
// on tcgen05 with TMEM accumulators):
//   warp 9      TMA producer: Q_A, Q_B once, then K0 V0 K1 V1 ... through an
//               NS-stage shared-memory ring (full/empty mbarriers).
//   warp 8      MMA issuer: S_X = Q_X K^T into TMEM (SS MMA), and
//               O_X += P_X V (TS MMA, P read from TMEM) for X in {A, B}
//               (with FP8 Q and K, S comes from kind::f8f6f4 MMAs instead),
//               ordered so that the tensor core works on one tile while the
//               other tile's softmax runs (ping-pong).
//   warps 0-3   softmax of tile A; warps 4-7 softmax of tile B.  One thread
//               per query row (TMEM lane = row): tcgen05.ld of the 128-score
//               row (its max-reducing form, which also returns the row max of
//               an unmasked tile), mask and row max on diagonal and edge tiles,
//               exp2, row sum, bf16 P written back into the
//               S columns with tcgen05.st in two halves of 64 keys, each
//               announced on its own barrier so that O += P V starts on the
//               first half while the second is computed; O rescaled in TMEM
//               only when the row maximum grew by more than 2^8 (otherwise
//               the stale reference is kept; o and l share it, so o / l is
//               unchanged).  Epilogue: O / l -> bf16 global, LSE -> f32 global.
// TMEM (512 columns): S_A [0,128) S_B [128,256) O_A [256,256+d) O_B [256+d', ...).
// Head dims 64, 96 and 128 (96: Q/K rows of one and a half 128-byte swizzle
// atoms, the rest zero-filled by the tensor map, six MMA K steps).
//
// attn_fwd_persistent_kernel: one query tile of 128 rows per work item
// (warps 0-3 softmax, warp 4 MMA, warp 5 TMA), one CTA per SM (d = 256) or
// two (d = 64), each walking its share of the items.  The next tile's
// S = Q K^T runs while the softmax works on the current one: with two score
// buffers at d = 256 (S0, S1 and a 256-column O fill the 512 columns), with
// P in columns of its own at d = 64 (S 128, P 64, O 64: 256 columns, two CTAs
// per SM); the K/V ring is filled in that consumption order.
//
// Every mbarrier wait is bounded (globaltimer budget); on expiry the CTA
// records a timeout in the status word, all roles leave their loops, pending
// TMA loads and MMAs are awaited (bounded), TMEM is freed and the CTA exits.
#include <algorithm>
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "attn.h"

namespace attn {
namespace {

constexpr int BM = 128;            // query rows per tile (= TMEM lanes)
constexpr int BN = 128;            // keys per K/V tile
// NT query tiles per CTA: 4 NT softmax warps, then the MMA and TMA warps.
__host__ __device__ constexpr int threads_for(int NT) { return 128 * NT + 64; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when m grows by > 2^8

// D: head dim of Q and K; DV: head dim of V and O (the value dim may differ);
// NT: query tiles per CTA.  Two tiles share every K/V tile and ping-pong on
// the tensor core inside one CTA (one CTA per SM: 512 TMEM columns); one
// tile takes 128 + DV columns (a 256-column allocation) and a ring small
// enough that two CTAs share an SM, their pipelines covering each other's
// start, drain and softmax latency -- the better trade when CTAs are short.
// SB: score buffers per query tile (one-tile CTAs only).  With two, the
// next tile's S = Q K^T runs while the softmax works on the current one,
// and P V of a tile runs while the softmax works on the next.
// PS: P in tensor-memory columns of its own (one-tile CTAs, value dims up
// to 64) instead of over S: S is free for the next Q K^T as soon as the
// softmax has loaded it, so the same overlap as two score buffers fits in
// 256 columns (S 128, P 64, O 64) and two CTAs still share an SM.
template <int D, int DV, bool FP8, int NT = 2, int SB = 1, bool PS = false>
struct Cfg {
  static_assert(NT == 1 || NT == 2, "one or two query tiles per CTA");
  static_assert(SB == 1 || (SB == 2 && NT == 1), "two score buffers for one-tile CTAs");
  static_assert(!PS || (NT == 1 && SB == 1 && DV <= 64), "separate P: one tile, one S buffer");
  static constexpr bool kOverlap = SB == 2 || PS;  // next S computed during this softmax
  static constexpr int kSBufs = NT * SB;                    // S slots of 128 columns
  static constexpr int kQKElem = FP8 ? 1 : 2;               // bytes per Q/K element
  static constexpr int kQKRowBytes = D * kQKElem;
  // 128-byte swizzle atoms per Q/K row; a partial last atom (d = 96: 192
  // bytes per row) is zero-filled past the row by the tensor map's bounds.
  static constexpr int kQKAtoms = (kQKRowBytes + 127) / 128;
  static constexpr int kQKSteps = kQKRowBytes / 32;         // MMA K steps (32 bytes each)
  static constexpr int kVAtoms = (DV + 63) / 64;            // ... per V row (bf16)
  static constexpr uint32_t kAtomBytes = 128u * 128u;       // one [128 rows][128 B] box
  static constexpr uint32_t kQBytes = kQKAtoms * kAtomBytes;  // one Q tile (BM rows)
  static constexpr uint32_t kKBytes = kQKAtoms * kAtomBytes;  // one K tile (BN rows)
  static constexpr uint32_t kVBytes = kVAtoms * kAtomBytes;   // one V tile
  static constexpr uint32_t kKVBytes = kKBytes > kVBytes ? kKBytes : kVBytes;  // one ring stage
  static constexpr int kStages =
      NT == 2 ? ((kKVBytes >= 32768u) ? 4 : 8)
              : ((kKVBytes >= 32768u) ? 2 : (SB == 2 ? 8 : 5));
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = NT * kQBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kKVBytes;
  // barriers: full[S], empty[S], q_full, s_full[2], p_ready[2] (keys 0-63 of
  // P stored), p2_ready[2] (keys 64-127), o_full[2], drain, o_step (P V of
  // one tile done; two score buffers only), q_free (the work item's last
  // Q K^T done: the next item's Q may load).  s_full / p_ready / p2_ready are
  // per query tile with two tiles, per score buffer with two buffers.
  static constexpr int kBarFull = 0;
  static constexpr int kBarEmpty = kStages;
  static constexpr int kBarQ = 2 * kStages;
  static constexpr int kBarS = kBarQ + 1;
  static constexpr int kBarP = kBarS + 2;
  static constexpr int kBarP2 = kBarP + 2;
  static constexpr int kBarO = kBarP2 + 2;
  static constexpr int kBarDrain = kBarO + 2;
  static constexpr int kBarOStep = kBarDrain + 1;
  static constexpr int kBarQFree = kBarOStep + 1;  // an item's last Q K^T completed
  static constexpr int kBarSFree = kBarQFree + 1;  // separate P: S loaded by the softmax
  static constexpr int kNumBars = kBarSFree + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + 1 KiB alignment slack
  static constexpr uint32_t kColS = 0;              // + 128 * (tile or score buffer)
  static constexpr uint32_t kColP = 128 * kSBufs;   // separate P (64 columns)
  static constexpr uint32_t kColO = kColP + (PS ? 64 : 0);  // + kOStride * tile
  static constexpr uint32_t kOStride = (DV + 63) / 64 * 64;  // O columns per tile, 64-aligned
  static constexpr uint32_t kTmemCols = (kColO + NT * kOStride) <= 256 ? 256 : 512;
  static constexpr int kThreads = threads_for(NT);
  static constexpr int kWarpMma = 4 * NT;
  static constexpr int kWarpLoad = 4 * NT + 1;
  static constexpr uint32_t kIdescQK = FP8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, DV, 1);
  static_assert(kQKSteps == 4 || kQKSteps == 6 || kQKSteps == 8 || kQKSteps == 16,
                "Q/K rows of 64, 96, 128 or 256 bf16 (128 e4m3)");
  static_assert(DV % 32 == 0 && DV <= 256, "value rows of 32-column multiples up to 256");
  static_assert(kColO + NT * kOStride <= 512, "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // A CTA that takes all 512 TMEM columns must be alone on its SM (its
  // shared memory keeps a second one out); 256-column CTAs pair up.
  static_assert(kTmemCols == 256 || kSmemBytes > 232448 / 2,
                "a 512-column CTA keeps the SM's tensor memory to itself");
  static_assert(NT == 2 || kTmemCols == 512 || 2 * (kSmemBytes + 1024) <= 232448,
                "two one-tile CTAs per SM (256 TMEM columns each)");
};

// Division by a divisor fixed for the launch, for dividends below 2^31:
// q = (n m) >> s with s = 31 + ceil(log2 d) and m = ceil(2^s / d).  The
// rounding error n (m - 2^s / d) / 2^s stays below 2^31 / 2^s <= 1 / d, so
// q is exact (division by invariant integers with a multiply and a shift,
// as in Granlund and Montgomery, 1994); it replaces the ~20-instruction
// division sequence on the item decode's dependency chain.
struct FastDiv {
  uint64_t m;
  uint32_t s, d;
};
inline FastDiv make_fastdiv(uint32_t d) {
  if (d == 0) d = 1;  // (empty launches: never used)
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  const uint32_t s = 31 + l;
  return FastDiv{((uint64_t{1} << s) + d - 1) / d, s, d};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> f.s);
}

struct KParams {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int64_t Nq, Nk, qoff;
  int64_t H, group;  // query heads per batch; query heads per K/V head
  int64_t n_bh;       // batch x query heads
  int64_t chunk;      // items per causal scheduling chunk (whole rounds of the grid)
  int64_t heads_per_group;  // (b, h) slices per causal group (one CTA per item)
  int n_qblk;
  int causal;
  float sc_log2;  // scale * log2(e)
  uint32_t flags;
  uint64_t timeout_ns;
  // Divisors of the persistent kernel's item decode: query blocks per
  // (b, h), items per causal chunk, query heads per batch, query heads per
  // K/V head; K/V heads per batch.
  FastDiv fd_nq, fd_chunk, fd_h, fd_group;
  uint32_t kv_per_batch;
};

struct Waiter {
  volatile int* abort_flag;
  int* status;
  uint64_t timeout_ns;

  // Bounded wait for the phase of `bar` with parity `parity`.  Returns false
  // when the CTA is aborting (another role timed out) or this wait timed out.
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

// Ring order of the K and V tiles with two score buffers: the order the MMA
// warp consumes them (S(0), S(1), P(0) V, S(2), P(1) V, S(3), ...), i.e.
// K0 K1 V0 K2 V1 K3 V2 ... K(n-1) V(n-2) V(n-1), so that every load waits
// only for the release of the tile two positions before it.  These give the
// ring position of K(j) and V(j) for n tiles, and what position t holds.
__device__ __forceinline__ int kpos2(int j) { return j <= 1 ? j : 2 * j - 1; }
__device__ __forceinline__ int vpos2(int j, int n) { return j <= n - 2 ? 2 + 2 * j : 2 * n - 1; }
__device__ __forceinline__ void item2(int t, int n, bool& is_v, int& j) {
  if (n == 1) { is_v = t == 1; j = 0; return; }
  if (t <= 1) { is_v = false; j = t; return; }
  if (t >= 2 * n - 2) { is_v = true; j = t - n; return; }
  const int m = (t - 2) >> 1;
  is_v = ((t - 2) & 1) == 0;
  j = is_v ? m : m + 2;
}

// Number of K/V tiles query tile `row0` (128 rows) must visit; 0 if the tile
// is past Nq or (negative offsets only) no row of it sees any key.
__device__ __forceinline__ int tiles_for(int64_t row0, const KParams& p) {
  if (row0 >= p.Nq) return 0;
  const int64_t n_all = (p.Nk + BN - 1) / BN;
  if (!p.causal) return static_cast<int>(n_all);
  const int64_t last_row = min(row0 + BM - 1, p.Nq - 1);
  const int64_t last_key = last_row + p.qoff;
  if (last_key < 0) return 0;
  return static_cast<int>(min(n_all, last_key / BN + 1));
}

// One work item: 128 * NT query rows of one (b, h).  Items are numbered in
// the launch's scheduling order.  Causal problems take consecutive chunks of
// the (b, h)-major item list, each chunk sized to whole rounds of the grid
// and to K/V that fit in L2 together, and order every chunk heaviest first
// (last query block first, then by head): dealt out in the alternating
// rounds of item_of(), a chunk's heavy and light items pair up on each CTA,
// and K/V are read from DRAM about once.
struct Item {
  int64_t bh, bkv, q0;
  int ntile[2];
  int n_kv;
};

template <int NT>
__device__ __forceinline__ Item decode_item(int64_t idx, const KParams& p) {
  Item it;
  int64_t qb;
  const int64_t nq = p.n_qblk;
  // Item indices and counts are below 2^31 (checked on the host): 32-bit
  // divisions (64-bit ones are slow software routines).
  const uint32_t nq32 = static_cast<uint32_t>(nq);
  const uint32_t idx32 = static_cast<uint32_t>(idx);
  if (p.causal) {
    const uint32_t chunk = p.fd_chunk.d;
    const uint32_t n_items = static_cast<uint32_t>(p.n_bh) * nq32;
    const uint32_t a = fdiv(idx32, p.fd_chunk) * chunk;  // chunk [a, e) of the (b, h)-major list
    const uint32_t e = min(a + chunk, n_items);
    const uint32_t h_first = fdiv(a, p.fd_nq), h_last = fdiv(e - 1, p.fd_nq);
    // first block of h_first, last of h_last
    const uint32_t a0 = a - h_first * nq32, e0 = (e - 1) - h_last * nq32;
    // Rank r inside the chunk: query blocks from the last down, the chunk's
    // heads holding that block in (b, h) order.  Block qb is held by the
    // chunk's hc heads except h_first (when qb < a0) and h_last (when
    // qb > e0), so the heads per block are constant on three ranges of
    // blocks, from the top: [u1, nq) with hc - 1, [u2, u1) with c2 (all hc
    // on [a0, e0], or hc - 2 between e0 and a0), [0, u2) with hc - 1.  (A
    // chunk inside one head has only the middle range.)
    const uint32_t hc = h_last - h_first + 1;
    const uint32_t u1 = max(a0, e0 + 1);
    const bool inner = a0 <= e0;
    const uint32_t u2 = inner ? a0 : e0 + 1;
    const uint32_t c2 = inner ? hc : hc - 2;
    const uint32_t lo2 = inner ? h_first : h_first + 1;
    const uint32_t c1 = hc - 1;
    const uint32_t n1 = (nq32 - u1) * c1, n2 = (u1 - u2) * c2;
    uint32_t r = idx32 - a, h, q;
    if (r < n1) {
      h = h_first + r % c1;
      q = nq32 - 1 - r / c1;
    } else if ((r -= n1) < n2) {
      h = lo2 + r % c2;
      q = u1 - 1 - r / c2;
    } else {
      r -= n2;
      h = h_first + 1 + r % c1;
      q = u2 - 1 - r / c1;
    }
    it.bh = h;
    qb = q;
  } else {
    const uint32_t bh = fdiv(idx32, p.fd_nq);
    it.bh = bh;
    qb = idx32 - bh * nq32;
  }
  it.q0 = qb * (NT * BM);
  // K/V head of this query head (grouped K/V heads: H / group per batch).
  const uint32_t bh32 = static_cast<uint32_t>(it.bh);
  const uint32_t b32 = fdiv(bh32, p.fd_h);
  it.bkv = b32 * p.kv_per_batch + fdiv(bh32 - b32 * p.fd_h.d, p.fd_group);
  it.ntile[0] = tiles_for(it.q0, p);
  it.ntile[1] = NT == 2 ? tiles_for(it.q0 + BM, p) : 0;
  it.n_kv = max(it.ntile[0], it.ntile[1]);
  return it;
}

// The k-th work item of CTA c out of G: rounds of G items, alternately in
// and against CTA order (so a CTA that drew a heavy item in one round draws
// a light one in the next); -1 once the rounds pass the last item.
__device__ __forceinline__ int64_t item_of(int64_t k, int64_t c, int64_t G, int64_t n_items) {
  const int64_t idx = k * G + ((k & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

// One CTA per work item (NT query tiles of one (b, h)), dispatched in index
// order by the hardware.
template <int D, int DV, bool FP8, int NT>
__global__ void __launch_bounds__(threads_for(NT), 3 - NT)
    attn_fwd_tcgen05_kernel(const __grid_constant__ CUtensorMap tq,
                            const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv, const KParams p) {
  using C = Cfg<D, DV, FP8, NT>;
  constexpr int kWarpMma = C::kWarpMma;
  constexpr int kWarpLoad = C::kWarpLoad;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA -> (bh, query block).  Causal grids run in groups of consecutive
  // (b, h) slices whose K and V fit in L2 together; inside a group the CTAs
  // go longest-first (last query block first, then by head), so the CTAs
  // dispatched last are short and K/V are read from DRAM about once.
  // Item indices, head counts and block counts are below 2^31 (checked on
  // the host), so the divisions run in 32 bits: 64-bit ones are software
  // routines that held every CTA's start back by ~1800 cycles.
  int64_t bh;
  int qb;
  {
    const uint32_t idx = blockIdx.x;
    const uint32_t nq = static_cast<uint32_t>(p.n_qblk);
    uint32_t h32, q32;
    if (p.causal) {
      const uint32_t hpg = static_cast<uint32_t>(p.heads_per_group);
      const uint32_t per_group = hpg * nq;
      const uint32_t h0 = (idx / per_group) * hpg;
      const uint32_t r = idx % per_group;
      const uint32_t gh = min(hpg, static_cast<uint32_t>(p.n_bh) - h0);  // the last group may be smaller
      h32 = h0 + r % gh;
      q32 = nq - 1 - r / gh;
    } else {
      h32 = idx / nq;
      q32 = idx % nq;
    }
    bh = h32;
    qb = static_cast<int>(q32);
  }
  const int64_t q0 = static_cast<int64_t>(qb) * (NT * BM);
  // K/V head of this query head (grouped K/V heads: H / group per batch).
  const uint32_t H32 = static_cast<uint32_t>(p.H), G32 = static_cast<uint32_t>(p.group);
  const int64_t bkv = (static_cast<uint32_t>(bh) / H32) * (H32 / G32) +
                      (static_cast<uint32_t>(bh) % H32) / G32;
  int ntile[2];
  ntile[0] = tiles_for(q0, p);
  ntile[1] = NT == 2 ? tiles_for(q0 + BM, p) : 0;
  const int n_kv = max(ntile[0], ntile[1]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarQ), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::kBarS + x), 1);
      mbar_init(bar(C::kBarP + x), 4);  // one arrival per softmax warp
      mbar_init(bar(C::kBarP2 + x), 4);
      mbar_init(bar(C::kBarO + x), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    mbar_init(bar(C::kBarOStep), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter wait{abort_flag, p.status, p.timeout_ns};

  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sKV = sbase + C::kOffKV;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      uint32_t qbytes = 0;
      for (int x = 0; x < NT; ++x) qbytes += ntile[x] > 0 ? C::kQBytes : 0u;
      mbar_arrive_expect_tx(bar(C::kBarQ), qbytes);
      for (int x = 0; x < NT; ++x) {
        if (ntile[x] == 0) continue;
        for (int a = 0; a < C::kQKAtoms; ++a)
          tma_load_3d(sQ + x * C::kQBytes + a * C::kAtomBytes, &tq, bar(C::kBarQ),
                      a * (128 / C::kQKElem), static_cast<int>(q0 + x * BM),
                      static_cast<int>(bh));
      }
      // Ring position t: K(t/2) for even t, V(t/2) for odd t (one score
      // buffer per tile); the consumption order of item2() with two.
      int last_t[C::kStages];
      for (int s = 0; s < C::kStages; ++s) last_t[s] = -1;
      int skipped = -1;
      bool ok = true;
      for (int t = 0; t < 2 * n_kv && ok; ++t) {
        const int s = t % C::kStages;
        if (t >= C::kStages) ok = wait(bar(C::kBarEmpty + s), ((t / C::kStages) - 1) & 1);
        if (!ok) break;
        last_t[s] = t;
        if ((p.flags & ATTN_FLAG_TEST_SKIP_LOAD) && t == 1) {  // fault injection
          skipped = t;
          continue;
        }
        bool is_v = (t & 1) != 0;
        int tile = t >> 1;
        mbar_arrive_expect_tx(bar(C::kBarFull + s), is_v ? C::kVBytes : C::kKBytes);
        const int key0 = tile * BN;
        const int atoms = is_v ? C::kVAtoms : C::kQKAtoms;
        const int per_atom = is_v ? 64 : 128 / C::kQKElem;  // elements per 128-byte row
        for (int a = 0; a < atoms; ++a)
          tma_load_3d(sKV + s * C::kKVBytes + a * C::kAtomBytes, is_v ? &tv : &tk,
                      bar(C::kBarFull + s), a * per_atom, key0, static_cast<int>(bkv));
      }
      // Every issued load must land before the CTA can exit.  Only this
      // thread arrives on the full barriers, so the phase of the last load
      // into a stage stays complete once it lands.  These waits ignore the
      // abort flag (they cover copies in flight) but are still bounded.
      volatile int no_abort = 0;
      const Waiter own{&no_abort, p.status, p.timeout_ns};
      own(bar(C::kBarQ), 0);
      for (int s = 0; s < C::kStages; ++s)
        if (last_t[s] >= 0 && last_t[s] != skipped)
          own(bar(C::kBarFull + s), (last_t[s] / C::kStages) & 1);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits made warp-uniform); each run of
    // MMAs and each commit elects one lane to issue.
    auto wait_w = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait(b, parity));
    };
    auto commit = [&](uint32_t b) { mma_commit_w(b); };
    if (n_kv > 0) {
      // S = Q_x K^T into score slot `slot` (the tile's own with two tiles,
      // the alternating buffer with two score buffers).
      auto qk = [&](int x, int stage, int slot) {
        const uint32_t d_tmem = tmem + C::kColS + 128 * slot;
        const uint64_t a = sdesc_sw128(sQ + x * C::kQBytes, 16, 1024);
        const uint64_t b = sdesc_sw128(sKV + stage * C::kKVBytes, 16, 1024);
        // One MMA consumes 32 bytes of each Q/K row (16 bf16 or 32 e4m3).
        if constexpr (FP8) {
          mma_ss_f8_run4_w(d_tmem, a, b, C::kIdescQK, 0u);
        } else if constexpr (C::kQKSteps == 16) {
          // Two runs of eight steps; the second starts two atoms (32 KB =
          // 2048 descriptor units) further and accumulates.
          mma_ss_run8_w(d_tmem, a, b, C::kIdescQK, 0u);
          mma_ss_run8_w(d_tmem, a + 2048, b + 2048, C::kIdescQK, 1u);
        } else if constexpr (C::kQKSteps == 8) {
          mma_ss_run8_w(d_tmem, a, b, C::kIdescQK, 0u);
        } else if constexpr (C::kQKSteps == 6) {
          mma_ss_run6_w(d_tmem, a, b, C::kIdescQK, 0u);
        } else {
          mma_ss_run4_w(d_tmem, a, b, C::kIdescQK, 0u);
        }
      };
      // O_X += P_X V over keys 64 h .. 64 h + 63 (four K steps of 16 keys;
      // P's bf16 pairs for those keys sit in columns 32 h .. 32 h + 31).
      auto pv_half = [&](int x, int stage, int h, bool acc, int slot) {
        const uint32_t d_tmem = tmem + C::kColO + C::kOStride * x;
        const uint32_t p_tmem = tmem + C::kColS + 128 * slot + 32 * h;
        const uint64_t b =
            sdesc_sw128(sKV + stage * C::kKVBytes + h * 64 * 128, C::kAtomBytes, 1024);
        static_assert(BN == 128, "two halves of four K steps of 16 keys");
        mma_ts_run4_w(d_tmem, p_tmem, b, C::kIdescPV, acc ? 1u : 0u);
      };
      bool ok = wait_w(bar(C::kBarQ), 0);
      if (ok) ok = wait_w(bar(C::kBarFull + 0), 0);
      if (ok) {
        tc_fence_after();
        for (int x = 0; x < NT; ++x) {
          if (ntile[x] > 0) {
            qk(x, 0, x);
            commit(bar(C::kBarS + x));
          }
        }
        commit(bar(C::kBarEmpty + 0));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int tV = 2 * j + 1, sV = tV % C::kStages;
        const int tK = 2 * j + 2, sK = tK % C::kStages;
        const bool next = j + 1 < n_kv;
        bool k_ready = false;
        ok = wait_w(bar(C::kBarFull + sV), (tV / C::kStages) & 1);
        if (!ok) break;
        for (int x = 0; x < NT && ok; ++x) {
          if (j >= ntile[x]) continue;
          ok = wait_w(bar(C::kBarP + x), j & 1);
          if (!ok) break;
          tc_fence_after();
          pv_half(x, sV, 0, j > 0, x);
          ok = wait_w(bar(C::kBarP2 + x), j & 1);
          if (!ok) break;
          tc_fence_after();
          pv_half(x, sV, 1, true, x);
          if (j == ntile[x] - 1) commit(bar(C::kBarO + x));
          if (j + 1 < ntile[x]) {
            if (!k_ready) {
              ok = wait_w(bar(C::kBarFull + sK), (tK / C::kStages) & 1);
              if (!ok) break;
              tc_fence_after();
              k_ready = true;
            }
            qk(x, sK, x);
            commit(bar(C::kBarS + x));
          }
        }
        if (!ok) break;
        commit(bar(C::kBarEmpty + sV));
        if (next) {
          if (!k_ready) {  // K(j+1) is used by no tile: still consume it in order
            ok = wait_w(bar(C::kBarFull + sK), (tK / C::kStages) & 1);
            if (!ok) break;
          }
          commit(bar(C::kBarEmpty + sK));
        }
      }
      // All issued MMAs must complete before TMEM is released (bounded wait
      // that ignores the abort flag).
      commit(bar(C::kBarDrain));
      volatile int no_abort = 0;
      const Waiter own{&no_abort, p.status, p.timeout_ns};
      own(bar(C::kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;  // query tile
    const int row_in_tile = ((warp & 3) << 5) + lane;
    const int64_t row0 = q0 + x * BM;
    const int64_t row = row0 + row_in_tile;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS0 = tmem + lane_off + C::kColS + 128 * x;  // (first) score buffer
    const uint32_t tO = tmem + lane_off + C::kColO + C::kOStride * x;
    const int n = ntile[x];
    // Last admissible key of this row and of the tile's first row.
    const int64_t lim = p.causal ? min(p.Nk - 1, row + p.qoff) : p.Nk - 1;
    const int64_t lim_tile = p.causal ? min(p.Nk - 1, row0 + p.qoff) : p.Nk - 1;

    float m_run = -INFINITY;  // running maximum of scaled scores (log2 units)
    float m_ref = -INFINITY;  // exponent reference shared by o and l
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int slot = x;
      const uint32_t ph = static_cast<uint32_t>(j & 1);
      const uint32_t tS = tS0;
      // tcgen05.ld/st below are warp-collective: the warp leaves together.
      ok = __all_sync(0xffffffffu, wait(bar(C::kBarS + slot), ph));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[128];
      // The load returns the row maximum of the unmasked tile.
      float tmax = tmem_ld_max_x128(tS, sr);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      const int64_t k0 = static_cast<int64_t>(j) * BN;
      if (k0 + BN - 1 > lim_tile) {  // edge or diagonal tile (uniform per tile)
        const int64_t rel64 = lim - k0;
        const int rel = static_cast<int>(rel64 < -1 ? -1 : (rel64 > BN ? BN : rel64));
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c > rel) ? -INFINITY : s[c];
        // Masking invalidates the load's maximum: eight independent
        // 16-element chains of 3-input maxima over the masked row.
        float mx[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          mx[g] = fmaxf(s[16 * g], s[16 * g + 1]);
#pragma unroll
          for (int c = 2; c < 16; c += 2) mx[g] = fmax3f(mx[g], s[16 * g + c], s[16 * g + c + 1]);
        }
        tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                      fmaxf(mx[6], mx[7]));
      }
      const float m_new = fmaxf(m_run, tmax * p.sc_log2);
      m_run = m_new;
      float alpha = 1.0f;
      bool rescale = false;
      if (m_new > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
        rescale = (m_ref != -INFINITY);
        l *= alpha;
        m_ref = m_new;
      }
      const float neg_ref = (m_ref == -INFINITY) ? 0.0f : -m_ref;
      // p = 2^(s * scale * log2 e - m_ref), two lanes per instruction; the
      // row sum uses four independent packed accumulators.  P goes back to
      // tensor memory in two halves (keys 0-63, then 64-127), each announced
      // on its own barrier, so the first half of P V starts while the second
      // half is exponentiated.  The rare O rescale lands before the first
      // announcement.
      const uint64_t scale2 = f2_pack(p.sc_log2, p.sc_log2);
      const uint64_t bias2 = f2_pack(neg_ref, neg_ref);
      uint64_t acc2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[i] = 0ull;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int cc = 32 * h + c;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[2 * cc], s[2 * cc + 1]), scale2, bias2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          acc2[c & 3] = f2_add(acc2[c & 3], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st_x32(tS + 32 * h, pk);
        if (h == 0 && __any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t o[32];
            tmem_ld_x32(tO + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_x32(tO + cc * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar((h == 0 ? C::kBarP : C::kBarP2) + slot));
      }
      float sum_lo, sum_hi;
      f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), sum_lo, sum_hi);
      l += sum_lo + sum_hi;
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, wait(bar(C::kBarO + x), 0));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool valid = row < p.Nq;
      const bool empty = (n == 0) || !(l > 0.0f);
      if (n > 0) {
        const float inv = empty ? 0.0f : 1.0f / l;
        uint4* dst = reinterpret_cast<uint4*>(p.o + (bh * p.Nq + row) * DV);
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(tO + cc * 32, o);
          if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
              if (empty) w = make_uint4(0u, 0u, 0u, 0u);
              dst[cc * 4 + v4] = w;
            }
          }
        }
      } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + (bh * p.Nq + row) * DV);
        for (int i = 0; i < DV / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (valid)
        p.lse[bh * p.Nq + row] =
            empty ? -INFINITY : (m_ref + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Persistent form for one-tile CTAs whose next S overlaps the softmax (two
// score buffers, or P apart from S): one or two CTAs per SM, each walking
// its share of the work items; barrier phases are counted across items and
// the next item's Q loads once the last Q K^T of the current one completed,
// so CTA start-up, the first loads and the epilogue of one item overlap the
// work of the next.
template <int D, int DV, int SB, bool PS>
__global__ void __launch_bounds__(threads_for(1), 2)
    attn_fwd_persistent_kernel(const __grid_constant__ CUtensorMap tq,
                               const __grid_constant__ CUtensorMap tk,
                               const __grid_constant__ CUtensorMap tv, const KParams p) {
  constexpr int NT = 1;
  constexpr bool FP8 = false;
  using C = Cfg<D, DV, FP8, NT, SB, PS>;
  static_assert(C::kOverlap, "two score buffers or P apart from S");
  constexpr int kWarpMma = C::kWarpMma;
  constexpr int kWarpLoad = C::kWarpLoad;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // This CTA walks work items item_of(0), item_of(1), ... (one item per CTA
  // when the grid has one CTA per item).  Every role walks the same list and
  // counts barrier phases across items.
  const int64_t n_items = p.n_bh * p.n_qblk;
  const int64_t G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarQ), 1);
    mbar_init(bar(C::kBarQFree), 1);
    mbar_init(bar(C::kBarSFree), 4);  // one arrival per softmax warp
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::kBarS + x), 1);
      mbar_init(bar(C::kBarP + x), 4);  // one arrival per softmax warp
      mbar_init(bar(C::kBarP2 + x), 4);
      mbar_init(bar(C::kBarO + x), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    mbar_init(bar(C::kBarOStep), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter wait{abort_flag, p.status, p.timeout_ns};

  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sKV = sbase + C::kOffKV;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Ring position T runs on across items: within an item, position t is
      // K(t/2) for even t, V(t/2) for odd t (one score buffer per tile), or
      // the consumption order of item2() (two).
      int64_t last_T[C::kStages];
      for (int s = 0; s < C::kStages; ++s) last_T[s] = -1;
      int64_t T = 0, skipped = -1;
      int q_loads = 0;
      bool ok = true;
      for (int64_t k = 0; ok; ++k) {
        const int64_t idx = item_of(k, cta, G, n_items);
        if (idx < 0) break;
        const Item it = decode_item<NT>(idx, p);
        if (it.n_kv == 0) continue;
        // The Q tiles are overwritten once the previous item's last Q K^T
        // has completed.
        if (q_loads > 0) ok = wait(bar(C::kBarQFree), (q_loads - 1) & 1);
        if (!ok) break;
        uint32_t qbytes = 0;
        for (int x = 0; x < NT; ++x) qbytes += it.ntile[x] > 0 ? C::kQBytes : 0u;
        mbar_arrive_expect_tx(bar(C::kBarQ), qbytes);
        for (int x = 0; x < NT; ++x) {
          if (it.ntile[x] == 0) continue;
          for (int a = 0; a < C::kQKAtoms; ++a)
            tma_load_3d(sQ + x * C::kQBytes + a * C::kAtomBytes, &tq, bar(C::kBarQ),
                        a * (128 / C::kQKElem), static_cast<int>(it.q0 + x * BM),
                        static_cast<int>(it.bh));
        }
        ++q_loads;
        for (int t = 0; t < 2 * it.n_kv && ok; ++t) {
          const int64_t TT = T + t;
          const int s = static_cast<int>(TT % C::kStages);
          if (TT >= C::kStages) ok = wait(bar(C::kBarEmpty + s), ((TT / C::kStages) - 1) & 1);
          if (!ok) break;
          last_T[s] = TT;
          if ((p.flags & ATTN_FLAG_TEST_SKIP_LOAD) && TT == 1) {  // fault injection
            skipped = TT;
            continue;
          }
          bool is_v = (t & 1) != 0;
          int tile = t >> 1;
          if constexpr (C::kOverlap) item2(t, it.n_kv, is_v, tile);
          mbar_arrive_expect_tx(bar(C::kBarFull + s), is_v ? C::kVBytes : C::kKBytes);
          const int key0 = tile * BN;
          const int atoms = is_v ? C::kVAtoms : C::kQKAtoms;
          const int per_atom = is_v ? 64 : 128 / C::kQKElem;  // elements per 128-byte row
          for (int a = 0; a < atoms; ++a)
            tma_load_3d(sKV + s * C::kKVBytes + a * C::kAtomBytes, is_v ? &tv : &tk,
                        bar(C::kBarFull + s), a * per_atom, key0, static_cast<int>(it.bkv));
        }
        T += 2 * it.n_kv;
      }
      // Every issued load must land before the CTA can exit.  Only this
      // thread arrives on the full and Q barriers, so the phase of the last
      // load into each stays complete once it lands.  These waits ignore the
      // abort flag (they cover copies in flight) but are still bounded.
      volatile int no_abort = 0;
      const Waiter own{&no_abort, p.status, p.timeout_ns};
      if (q_loads > 0) own(bar(C::kBarQ), (q_loads - 1) & 1);
      for (int s = 0; s < C::kStages; ++s)
        if (last_T[s] >= 0 && last_T[s] != skipped)
          own(bar(C::kBarFull + s), (last_T[s] / C::kStages) & 1);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits made warp-uniform); each run of
    // MMAs and each commit elects one lane to issue.
    auto wait_w = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait(b, parity));
    };
    auto commit = [&](uint32_t b) { mma_commit_w(b); };
    // Ring stage and phase of position T + o, o >= 0 a small offset inside
    // the current item: 32-bit arithmetic from the item's base (the MMA
    // warp's issue slots are on the softmax's critical path).
    uint32_t base_s = 0, base_ph = 0;
    auto stage_of = [&](int o) { return static_cast<int>((base_s + static_cast<uint32_t>(o)) % C::kStages); };
    auto phase_of = [&](int o) {
      return base_ph ^ (((base_s + static_cast<uint32_t>(o)) / C::kStages) & 1u);
    };
    // S = Q_x K^T into score slot `slot` (the tile's own with two tiles,
    // the alternating buffer with two score buffers).
    auto qk = [&](int x, int stage, int slot) {
      const uint32_t d_tmem = tmem + C::kColS + 128 * slot;
      const uint64_t a = sdesc_sw128(sQ + x * C::kQBytes, 16, 1024);
      const uint64_t b = sdesc_sw128(sKV + stage * C::kKVBytes, 16, 1024);
      // One MMA consumes 32 bytes of each Q/K row (16 bf16 or 32 e4m3).
      if constexpr (FP8) {
        mma_ss_f8_run4_w(d_tmem, a, b, C::kIdescQK, 0u);
      } else if constexpr (C::kQKSteps == 16) {
        // Two runs of eight steps; the second starts two atoms (32 KB =
        // 2048 descriptor units) further and accumulates.
        mma_ss_run8_w(d_tmem, a, b, C::kIdescQK, 0u);
        mma_ss_run8_w(d_tmem, a + 2048, b + 2048, C::kIdescQK, 1u);
      } else if constexpr (C::kQKSteps == 8) {
        mma_ss_run8_w(d_tmem, a, b, C::kIdescQK, 0u);
      } else if constexpr (C::kQKSteps == 6) {
        mma_ss_run6_w(d_tmem, a, b, C::kIdescQK, 0u);
      } else {
        mma_ss_run4_w(d_tmem, a, b, C::kIdescQK, 0u);
      }
    };
    // O_X += P_X V over keys 64 h .. 64 h + 63 (four K steps of 16 keys;
    // P's bf16 pairs for those keys sit in columns 32 h .. 32 h + 31).  The
    // first half of an item's first tile overwrites O: the softmax warps read
    // the previous item's O before they announced this item's first P.
    auto pv_half = [&](int x, int stage, int h, bool acc, int slot) {
      const uint32_t d_tmem = tmem + C::kColO + C::kOStride * x;
      const uint32_t p_tmem =
          tmem + (PS ? C::kColP : C::kColS + 128 * slot) + 32 * h;
      const uint64_t b =
          sdesc_sw128(sKV + stage * C::kKVBytes + h * 64 * 128, C::kAtomBytes, 1024);
      static_assert(BN == 128, "two halves of four K steps of 16 keys");
      mma_ts_run4_w(d_tmem, p_tmem, b, C::kIdescPV, acc ? 1u : 0u);
    };
    int64_t T = 0;     // ring position of the item's first tile
    int q_uses = 0;    // items with work so far (Q barrier phases)
    int64_t sc[2] = {0, 0};  // score tiles handled so far, per query tile
    bool ok = true;
    for (int64_t k = 0; ok; ++k) {
      const int64_t idx = item_of(k, cta, G, n_items);
      if (idx < 0) break;
      const Item it = decode_item<NT>(idx, p);
      if (it.n_kv == 0) continue;
      base_s = static_cast<uint32_t>(T % C::kStages);
      base_ph = static_cast<uint32_t>((T / C::kStages) & 1);
      ok = wait_w(bar(C::kBarQ), q_uses & 1);
      if (ok) ok = wait_w(bar(C::kBarFull + stage_of(0)), phase_of(0));
      if (!ok) break;
      if constexpr (PS) {
        // One tile, P apart from S.  Issue order: S(0), then for each j:
        // S(j+1) as soon as the softmax has loaded S(j), P(j) V (two
        // halves, as P arrives).  A commit after every P V tells the
        // softmax that P's columns may be rewritten and O rescaled.
        const int n = it.ntile[0];
        const int64_t g0 = sc[0];  // score tiles before this item
        tc_fence_after();
        qk(0, stage_of(0), 0);
        commit(bar(C::kBarS + 0));
        commit(bar(C::kBarEmpty + stage_of(0)));
        if (n == 1) commit(bar(C::kBarQFree));  // the item's only Q K^T
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t ph = static_cast<uint32_t>((g0 + j) & 1);
          if (j + 1 < n) {
            const int tK = kpos2(j + 1);
            ok = wait_w(bar(C::kBarSFree), ph);
            if (ok) ok = wait_w(bar(C::kBarFull + stage_of(tK)), phase_of(tK));
            if (!ok) break;
            tc_fence_after();
            qk(0, stage_of(tK), 0);
            commit(bar(C::kBarS + 0));
            commit(bar(C::kBarEmpty + stage_of(tK)));
            if (j + 2 == n) commit(bar(C::kBarQFree));  // the item's last Q K^T
          }
          const int tV = vpos2(j, n);
          ok = wait_w(bar(C::kBarFull + stage_of(tV)), phase_of(tV));
          if (!ok) break;
          ok = wait_w(bar(C::kBarP + 0), ph);
          if (!ok) break;
          tc_fence_after();
          pv_half(0, stage_of(tV), 0, j > 0, 0);
          ok = wait_w(bar(C::kBarP2 + 0), ph);
          if (!ok) break;
          tc_fence_after();
          pv_half(0, stage_of(tV), 1, true, 0);
          commit(bar(C::kBarOStep));
          if (j == n - 1) commit(bar(C::kBarO + 0));
          commit(bar(C::kBarEmpty + stage_of(tV)));
        }
      } else if constexpr (SB == 2) {
        // One tile, two score buffers.  Issue order: S(0), S(1), then for
        // each j: P(j) V (two halves, as P arrives), S(j+2) into P(j)'s
        // buffer (in order after the P V that reads it).  A commit after
        // every P V tells the softmax when O may be rescaled.
        const int n = it.ntile[0];
        const int64_t g0 = sc[0];  // score tiles before this item
        tc_fence_after();
        qk(0, stage_of(0), static_cast<int>(g0 & 1));
        commit(bar(C::kBarS + static_cast<int>(g0 & 1)));
        commit(bar(C::kBarEmpty + stage_of(0)));
        if (n > 1) {
          const int tK = kpos2(1);
          ok = wait_w(bar(C::kBarFull + stage_of(tK)), phase_of(tK));
          if (!ok) break;
          tc_fence_after();
          qk(0, stage_of(tK), static_cast<int>((g0 + 1) & 1));
          commit(bar(C::kBarS + static_cast<int>((g0 + 1) & 1)));
          commit(bar(C::kBarEmpty + stage_of(tK)));
        }
        if (n <= 2) commit(bar(C::kBarQFree));  // the item's last Q K^T is issued
        for (int j = 0; j < n && ok; ++j) {
          const int64_t g = g0 + j;
          const int b = static_cast<int>(g & 1);
          const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
          const int tV = vpos2(j, n);
          ok = wait_w(bar(C::kBarFull + stage_of(tV)), phase_of(tV));
          if (!ok) break;
          ok = wait_w(bar(C::kBarP + b), ph);
          if (!ok) break;
          tc_fence_after();
          pv_half(0, stage_of(tV), 0, j > 0, b);
          ok = wait_w(bar(C::kBarP2 + b), ph);
          if (!ok) break;
          tc_fence_after();
          pv_half(0, stage_of(tV), 1, true, b);
          commit(bar(C::kBarOStep));
          if (j == n - 1) commit(bar(C::kBarO + 0));
          commit(bar(C::kBarEmpty + stage_of(tV)));
          if (j + 2 < n) {
            const int tK = kpos2(j + 2);
            ok = wait_w(bar(C::kBarFull + stage_of(tK)), phase_of(tK));
            if (!ok) break;
            tc_fence_after();
            qk(0, stage_of(tK), b);
            commit(bar(C::kBarS + b));
            commit(bar(C::kBarEmpty + stage_of(tK)));
            if (j + 3 == n) commit(bar(C::kBarQFree));
          }
        }
      }
      T += 2 * it.n_kv;
      for (int x = 0; x < NT; ++x) sc[x] += it.ntile[x];
      ++q_uses;
    }
    // All issued MMAs must complete before TMEM is released (bounded wait
    // that ignores the abort flag).
    commit(bar(C::kBarDrain));
    volatile int no_abort = 0;
    const Waiter own{&no_abort, p.status, p.timeout_ns};
    own(bar(C::kBarDrain), 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;  // query tile
    const int row_in_tile = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS0 = tmem + lane_off + C::kColS + 128 * x;  // (first) score buffer
    const uint32_t tO = tmem + lane_off + C::kColO + C::kOStride * x;
    const uint32_t tP = tmem + lane_off + C::kColP;  // separate P (PS only)
    int64_t sc = 0;  // score tiles of this query tile handled so far
    int o_uses = 0;  // items in which this query tile had keys (O barrier phases)
    bool ok = true;
    // The next item is decoded while the last P V of the current one runs
    // (its integer divisions are otherwise on the softmax's critical path).
    int64_t idx = item_of(0, cta, G, n_items);
    Item it = {};
    if (idx >= 0) it = decode_item<NT>(idx, p);
    for (int64_t k = 0; ok && idx >= 0; ++k) {
      const int64_t row0 = it.q0 + x * BM;
      const int64_t row = row0 + row_in_tile;
      const int n = it.ntile[x];
      // Last admissible key of this row and of the tile's first row.
      const int64_t lim = p.causal ? min(p.Nk - 1, row + p.qoff) : p.Nk - 1;
      const int64_t lim_tile = p.causal ? min(p.Nk - 1, row0 + p.qoff) : p.Nk - 1;

      float m_run = -INFINITY;  // running maximum of scaled scores (log2 units)
      float m_ref = -INFINITY;  // exponent reference shared by o and l
      float l = 0.0f;
      for (int j = 0; j < n; ++j) {
        // Score slot and barrier phase of this tile: the tile's own slot with
        // one buffer, alternating buffers (each used every other tile) with
        // two.
        const int64_t g = sc + j;
        const int slot = SB == 2 ? static_cast<int>(g & 1) : x;
        const uint32_t ph = static_cast<uint32_t>(SB == 2 ? ((g >> 1) & 1) : (g & 1));
        const uint32_t tS = tS0 + 128 * (SB == 2 ? static_cast<uint32_t>(g & 1) : 0u);
        // tcgen05.ld/st below are warp-collective: the warp leaves together.
        ok = __all_sync(0xffffffffu, wait(bar(C::kBarS + slot), ph));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        // The load returns the row maximum of the unmasked tile.
        float tmax = tmem_ld_max_x128(tS, sr);
        if constexpr (PS) {
          // S is in registers: its columns may take the next Q K^T.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kBarSFree));
        }
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        const int64_t k0 = static_cast<int64_t>(j) * BN;
        if (k0 + BN - 1 > lim_tile) {  // edge or diagonal tile (uniform per tile)
          const int64_t rel64 = lim - k0;
          const int rel = static_cast<int>(rel64 < -1 ? -1 : (rel64 > BN ? BN : rel64));
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c > rel) ? -INFINITY : s[c];
          // Masking invalidates the load's maximum: eight independent
          // 16-element chains of 3-input maxima over the masked row.
          float mx[8];
#pragma unroll
          for (int gg = 0; gg < 8; ++gg) {
            mx[gg] = fmaxf(s[16 * gg], s[16 * gg + 1]);
#pragma unroll
            for (int c = 2; c < 16; c += 2)
              mx[gg] = fmax3f(mx[gg], s[16 * gg + c], s[16 * gg + c + 1]);
          }
          tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                        fmaxf(mx[6], mx[7]));
        }
        const float m_new = fmaxf(m_run, tmax * p.sc_log2);
        m_run = m_new;
        float alpha = 1.0f;
        bool rescale = false;
        if (m_new > m_ref + kRescaleThreshold) {
          alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
          rescale = (m_ref != -INFINITY);
          l *= alpha;
          m_ref = m_new;
        }
        if constexpr (SB == 2) {
          // With two score buffers P V of the previous tile may still be
          // running: an O rescale waits for it first (rare: the threshold).
          if (j > 0 && __any_sync(0xffffffffu, rescale)) {
            ok = __all_sync(0xffffffffu, wait(bar(C::kBarOStep), static_cast<uint32_t>((g - 1) & 1)));
            if (!ok) break;
            tc_fence_after();
          }
        }
        const float neg_ref = (m_ref == -INFINITY) ? 0.0f : -m_ref;
        // p = 2^(s * scale * log2 e - m_ref), two lanes per instruction; the
        // row sum uses four independent packed accumulators.  P goes back to
        // tensor memory in two halves (keys 0-63, then 64-127), each announced
        // on its own barrier, so the first half of P V starts while the second
        // half is exponentiated.  The rare O rescale lands before the first
        // announcement.
        const uint64_t scale2 = f2_pack(p.sc_log2, p.sc_log2);
        const uint64_t bias2 = f2_pack(neg_ref, neg_ref);
        uint64_t acc2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc2[i] = 0ull;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int cc = 32 * h + c;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[2 * cc], s[2 * cc + 1]), scale2, bias2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc2[c & 3] = f2_add(acc2[c & 3], f2_pack(p0, p1));
            pk[c] = pack_bf16x2(p0, p1);
          }
          if constexpr (PS) {
            // P V of the previous tile must have read P's columns before
            // they are rewritten (and O before it is rescaled); the wait
            // comes after the first half's exponentials, which hide it.
            if (h == 0 && j > 0) {
              ok = __all_sync(0xffffffffu,
                              wait(bar(C::kBarOStep), static_cast<uint32_t>((g - 1) & 1)));
              if (!ok) break;
              tc_fence_after();
            }
          }
          tmem_st_x32((PS ? tP : tS) + 32 * h, pk);
          if (h == 0 && __any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll 1
            for (int cc = 0; cc < DV / 32; ++cc) {
              uint32_t o[32];
              tmem_ld_x32(tO + cc * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st_x32(tO + cc * 32, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar((h == 0 ? C::kBarP : C::kBarP2) + slot));
        }
        if (!ok) break;
        float sum_lo, sum_hi;
        f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), sum_lo, sum_hi);
        l += sum_lo + sum_hi;
      }
      if (!ok) break;
      const int64_t next_idx = item_of(k + 1, cta, G, n_items);
      Item next = {};
      if (next_idx >= 0) next = decode_item<NT>(next_idx, p);
      if (n > 0) {
        ok = __all_sync(0xffffffffu, wait(bar(C::kBarO + x), static_cast<uint32_t>(o_uses & 1)));
        if (!ok) break;
        tc_fence_after();
      }
      const bool valid = row < p.Nq;
      const bool empty = (n == 0) || !(l > 0.0f);
      uint4* dst = reinterpret_cast<uint4*>(p.o + (it.bh * p.Nq + row) * DV);
      if (n > 0) {
        const float inv = empty ? 0.0f : 1.0f / l;
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(tO + cc * 32, o);
          if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
              if (empty) w = make_uint4(0u, 0u, 0u, 0u);
              dst[cc * 4 + v4] = w;
            }
          }
        }
      } else if (valid) {
        for (int i = 0; i < DV / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (valid)
        p.lse[it.bh * p.Nq + row] =
            empty ? -INFINITY : (m_ref + log2f(l)) * 0.69314718055994530942f;
      sc += n;
      o_uses += n > 0 ? 1 : 0;
      idx = next_idx;
      it = next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Fields of KParams shared by both kernels.
template <int NT>
KParams make_params(const FwdArgs& a) {
  KParams p = {};
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.status = a.status;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.qoff = a.query_offset;
  p.H = a.H;
  p.group = a.group;
  p.n_qblk = static_cast<int>((a.Nq + NT * BM - 1) / (NT * BM));
  p.n_bh = a.BH;
  p.causal = a.causal;
  p.sc_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.flags = a.flags;
  p.timeout_ns = a.timeout_ns;
  p.fd_nq = make_fastdiv(static_cast<uint32_t>(p.n_qblk));
  p.fd_chunk = make_fastdiv(1);
  p.fd_h = make_fastdiv(static_cast<uint32_t>(a.H));
  p.fd_group = make_fastdiv(static_cast<uint32_t>(a.group));
  p.kv_per_batch = static_cast<uint32_t>(a.H / a.group);
  return p;
}

// K and V bytes of one K/V head.
inline double kv_head_bytes(const FwdArgs& a, int d, int dv, bool fp8) {
  return static_cast<double>(a.Nk) * (d * (fp8 ? 1.0 : 2.0) + dv * 2.0);
}

// One CTA per work item.  Causal grids run in groups of whole K/V heads
// whose K and V take about 48 MB of L2.
template <int D, int DV, bool FP8, int NT = 2>
cudaError_t launch(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                   const CUtensorMap& tv, cudaStream_t stream) {
  using C = Cfg<D, DV, FP8, NT>;
  static_assert(C::kSmemBytes < (1u << 20), "");
  cudaError_t err = cudaFuncSetAttribute(attn_fwd_tcgen05_kernel<D, DV, FP8, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
  if (err != cudaSuccess) return err;
  KParams p = make_params<NT>(a);
  const int64_t kv_fit =
      std::max<int64_t>(1, static_cast<int64_t>(48.0e6 / kv_head_bytes(a, D, DV, FP8)));
  p.heads_per_group = std::min<int64_t>(a.BH, kv_fit * a.group);
  const int64_t blocks = a.BH * p.n_qblk;
  attn_fwd_tcgen05_kernel<D, DV, FP8, NT><<<dim3(static_cast<unsigned>(blocks)), dim3(C::kThreads),
                                            C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// Persistent launch: as many CTAs as fit on the GPU at once (one per SM for
// 512 TMEM columns, two for 256).
template <int D, int DV, int SB, bool PS>
cudaError_t launch_persistent(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream) {
  using C = Cfg<D, DV, false, 1, SB, PS>;
  cudaError_t err = cudaFuncSetAttribute(attn_fwd_persistent_kernel<D, DV, SB, PS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
  if (err != cudaSuccess) return err;
  KParams p = make_params<1>(a);
  int dev = 0, sms = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int64_t per_sm = C::kTmemCols == 512 ? 1 : 2;
  const int64_t n_items = a.BH * p.n_qblk;
  const int64_t blocks = std::min<int64_t>(n_items, std::max(sms, 1) * per_sm);
  // Causal scheduling chunks: pairs of rounds of the grid (a heavy and a
  // light item per CTA), as many pairs as keep the chunk's K and V within
  // about 48 MB of L2 (query heads sharing a K/V head count once).
  const double pair_kv_bytes = static_cast<double>(2 * blocks) / p.n_qblk /
                               static_cast<double>(a.group) * kv_head_bytes(a, D, DV, false);
  const int64_t pairs = std::max<int64_t>(1, static_cast<int64_t>(48.0e6 / pair_kv_bytes));
  p.chunk = std::min<int64_t>(n_items, 2 * blocks * pairs);
  p.fd_chunk = make_fastdiv(static_cast<uint32_t>(p.chunk));
  attn_fwd_persistent_kernel<D, DV, SB, PS><<<dim3(static_cast<unsigned>(blocks)),
                                              dim3(C::kThreads), C::kSmemBytes, stream>>>(
      tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tcgen05(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, cudaStream_t stream) {
  // Head dims 96 and 256 (value dim equal): 96 runs the two-tile layout of
  // 128 (Q/K rows padded to two atoms by the tensor map's zero fill, six K
  // steps); 256 takes one query tile per CTA with S and a 256-column O in
  // all 512 TMEM columns and a two-stage ring of 64 KB tiles.
  if (a.d == 96) return launch<96, 96, false>(a, tq, tk, tv, stream);
  if (a.d == 256) return launch_persistent<256, 256, 2, false>(a, tq, tk, tv, stream);
  if (a.fp8_qk)
    return a.dv == 64 ? launch<128, 64, true>(a, tq, tk, tv, stream)
                      : launch<128, 128, true>(a, tq, tk, tv, stream);
  if (a.d == 64) {
    if (a.dv == 128) return launch<64, 128, false>(a, tq, tk, tv, stream);
    return launch_persistent<64, 64, 1, true>(a, tq, tk, tv, stream);
  }
  if (a.dv == 64) return launch<128, 64, false>(a, tq, tk, tv, stream);
  return launch<128, 128, false>(a, tq, tk, tv, stream);
}

}  // namespace attn
