// splitkv.cu -- memory-bound split-KV attention for short queries (decode)
// and the log-sum-exp combine.
//
// Partial kernel: one CTA per (batch * K/V head, block of QB query rows, key
// split s).  The query rows of a K/V head are those of every query head in
// its group (grouped-query / multi-query attention) at every query position,
// so a split's K/V slice is read from memory once for the whole group.  The split's keys [s*L, min((s+1)*L, Nk)) are streamed once from device
// memory with 16-byte read-only loads: a key row of d bf16 is read by d/8
// adjacent lanes, so a warp reads 32/(d/8) whole rows per instruction and the
// CTA's 8 warps read consecutive rows.  Each lane group keeps the online
// softmax state of section 22.5 of "GPU Engineering: Correctness, Throughput,
// and Attention" (running maximum m, normaliser l, unnormalised o, rescale
// by exp2(m - m_new)) for its keys, in log2 units (q is pre-multiplied by
// scale * log2(e)); group, warp and CTA states are merged by the same
// rescaling.  Output per (row, split): the normalised o (f32) and its
// natural-log LSE; an empty or fully masked split gives o = 0, lse = -inf.
//
// Pipelined variant (several query rows per K/V head: GQA groups or Nq > 1):
// a producer warp streams the split's contiguous K and V slices into a
// 4-stage shared-memory ring with 1-D bulk copies, so the bytes in flight do
// not depend on registers; the consumer warps run the same online-softmax
// arithmetic from shared memory.  It is persistent: one CTA per SM walks
// the (K/V head, row block, split) items, and the ring runs on from one
// item to the next, so no CTA start or pipeline refill separates them.  Its
// waits are bounded like the prefill kernel's (timeout -> status word,
// clean exit).
//
// Combine kernel: one warp per (batch*head, query row) merges the splits:
// M = max lse_s, w_s = exp(lse_s - M), O = sum w_s o_s / sum w_s (-> bf16),
// LSE = M + ln sum w_s; M = -inf gives O = +0.0, LSE = -inf (the section 22.7
// lab's policy for a row with no admissible key).
#include <algorithm>
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kLog2e = 1.4426950408889634074f;
constexpr float kLn2 = 0.69314718055994530942f;

struct PartialParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  float* o_part;
  float* lse_part;
  int64_t Nq, Nk, qoff, L;
  int64_t H, Hkv, G, R;  // query heads, K/V heads, group size, rows per K/V head
  int S, n_qb, causal;
  int64_t n_items;  // pipelined kernel: (K/V head, row block, split) work items
  float sc_log2;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint4 ld_stream(const uint16_t* ptr) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr));
  return r;
}

// 8-byte form, for value rows narrower than the key rows.
__device__ __forceinline__ uint2 ld_stream8(const uint16_t* ptr) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
      : "=r"(r.x), "=r"(r.y)
      : "l"(ptr));
  return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& r, float (&f)[8]) {
  f[0] = bf_lo(r.x); f[1] = bf_hi(r.x);
  f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
  f[4] = bf_lo(r.z); f[5] = bf_hi(r.z);
  f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
}

// Merge state (m2, l2, o2) into (m, l, o); all in log2 units.
template <int E>
__device__ __forceinline__ void merge_state(float& m, float& l, float (&o)[E], float m2, float l2,
                                            const float (&o2)[E]) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  const float a = ex2_approx(m - mn);
  const float b = ex2_approx(m2 - mn);
  l = l * a + l2 * b;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = o[e] * a + o2[e] * b;
  m = mn;
}

// The VE values of a value row this lane owns (VE = 4, 8 or 16 bf16), as
// bf16 pairs, and their f32 widening.
template <int VE>
struct VSlice {
  uint32_t w[VE / 2];
  __device__ __forceinline__ void load(const uint16_t* ptr) {
    if constexpr (VE == 4) {
      const uint2 r = ld_stream8(ptr);
      w[0] = r.x; w[1] = r.y;
    } else {
#pragma unroll
      for (int c = 0; c < VE / 8; ++c) {
        const uint4 r = ld_stream(ptr + 8 * c);
        w[4 * c] = r.x; w[4 * c + 1] = r.y; w[4 * c + 2] = r.z; w[4 * c + 3] = r.w;
      }
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < VE / 2; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ void widen(float (&f)[VE]) const {
#pragma unroll
    for (int i = 0; i < VE / 2; ++i) {
      f[2 * i] = bf_lo(w[i]);
      f[2 * i + 1] = bf_hi(w[i]);
    }
  }
};

// D: key head dim; DV: value head dim (the lanes of a key row also own the
// value row, DV / (D / 8) values each).
template <int D, int DV, int QB, int U, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) splitkv_partial_kernel(const PartialParams p) {
  constexpr int LPR = D / 8;      // lanes per key row (16 B each)
  constexpr int G = 32 / LPR;     // key rows per warp instruction
  constexpr int STEP = kWarps * G * U;
  constexpr int VE = DV / LPR;    // values of a value row per lane
  static_assert(VE == 4 || VE == 8 || VE == 16, "value dims 64 and 128");

  __shared__ float sm_m[kWarps][QB];
  __shared__ float sm_l[kWarps][QB];
  __shared__ __align__(16) float sm_o[kWarps][QB][DV];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int64_t lin = blockIdx.x;
  // lin = (bkv * S + s) * n_qb + qb: the row blocks of one K/V slice are
  // neighbours, so they run together and read the slice once from memory.
  const int qb = static_cast<int>(lin % p.n_qb);
  const int64_t rest = lin / p.n_qb;
  const int s = static_cast<int>(rest % p.S);
  const int64_t bkv = rest / p.S;  // batch * Hkv + K/V head
  const int64_t r0 = static_cast<int64_t>(qb) * QB;
  // Row r of this K/V head: query head (group member r / Nq), position r % Nq.
  int64_t qrow[QB], pos[QB];
#pragma unroll
  for (int qi = 0; qi < QB; ++qi) {
    const int64_t r = min(r0 + qi, p.R - 1);
    const int64_t g = r / p.Nq;
    pos[qi] = r % p.Nq;
    const int64_t h = (bkv % p.Hkv) * p.G + g;
    qrow[qi] = ((bkv / p.Hkv) * p.H + h) * p.Nq + pos[qi];
  }

  const int64_t k_lo = static_cast<int64_t>(s) * p.L;
  int64_t k_hi = min(k_lo + p.L, p.Nk);
  int64_t lim[QB];  // last admissible key per query row
#pragma unroll
  for (int qi = 0; qi < QB; ++qi) lim[qi] = p.causal ? min(p.Nk - 1, pos[qi] + p.qoff) : p.Nk - 1;
  if (p.causal) {
    int64_t top = lim[0];
#pragma unroll
    for (int qi = 1; qi < QB; ++qi) top = max(top, lim[qi]);
    k_hi = min(k_hi, top + 1);
  }

  float qf[QB][8];
#pragma unroll
  for (int qi = 0; qi < QB; ++qi) {
    const uint4 r = ld_stream(p.q + qrow[qi] * D + 8 * sub);
    unpack8(r, qf[qi]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[qi][e] *= p.sc_log2;
  }

  float m[QB], l[QB], o[QB][VE];
#pragma unroll
  for (int qi = 0; qi < QB; ++qi) {
    m[qi] = -INFINITY;
    l[qi] = 0.0f;
#pragma unroll
    for (int e = 0; e < VE; ++e) o[qi][e] = 0.0f;
  }

  const uint16_t* kbase = p.k + bkv * p.Nk * D + 8 * sub;
  const uint16_t* vbase = p.v + bkv * p.Nk * DV + VE * sub;
  for (int64_t base = k_lo; base < k_hi; base += STEP) {
    uint4 kr[U];
    VSlice<VE> vr[U];
    int64_t key[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      key[u] = base + u * (kWarps * G) + warp * G + grp;
      if (key[u] < k_hi) {
        kr[u] = ld_stream(kbase + key[u] * D);
        vr[u].load(vbase + key[u] * DV);
      } else {
        kr[u] = make_uint4(0u, 0u, 0u, 0u);
        vr[u].zero();
      }
    }
    float sc[QB][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      unpack8(kr[u], kf);
#pragma unroll
      for (int qi = 0; qi < QB; ++qi) {
        float dot = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(qf[qi][e], kf[e], dot);
#pragma unroll
        for (int off = 1; off < LPR; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const bool live = key[u] < k_hi && key[u] <= lim[qi];
        sc[qi][u] = live ? dot : -INFINITY;
      }
    }
#pragma unroll
    for (int qi = 0; qi < QB; ++qi) {
      float mx = sc[qi][0];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[qi][u]);
      const float m_new = fmaxf(m[qi], mx);
      if (m_new == -INFINITY) continue;  // nothing admissible yet
      const float alpha = ex2_approx(m[qi] - m_new);
      l[qi] *= alpha;
#pragma unroll
      for (int e = 0; e < VE; ++e) o[qi][e] *= alpha;
      m[qi] = m_new;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float pu = ex2_approx(sc[qi][u] - m_new);
        l[qi] += pu;
        float vf[VE];
        vr[u].widen(vf);
#pragma unroll
        for (int e = 0; e < VE; ++e) o[qi][e] = fmaf(pu, vf[e], o[qi][e]);
      }
    }
  }

  // Merge the lane groups of this warp (groups differ in lane / LPR).
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int qi = 0; qi < QB; ++qi) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[qi], off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[qi], off);
      float o2[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, o[qi][e], off);
      merge_state<VE>(m[qi], l[qi], o[qi], m2, l2, o2);
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int qi = 0; qi < QB; ++qi) {
#pragma unroll
      for (int e = 0; e < VE; ++e) sm_o[warp][qi][VE * sub + e] = o[qi][e];
      if (sub == 0) {
        sm_m[warp][qi] = m[qi];
        sm_l[warp][qi] = l[qi];
      }
    }
  }
  __syncthreads();

  // Merge the warps and write the split's normalised output and LSE.
  for (int idx = threadIdx.x; idx < QB * DV; idx += kThreads) {
    const int qi = idx / DV, e = idx % DV;
    if (r0 + qi >= p.R) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][qi]);
    float L = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2_approx(sm_m[w][qi] - M);
        L = fmaf(sm_l[w][qi], f, L);
        acc = fmaf(sm_o[w][qi][e], f, acc);
      }
    }
    const bool empty = !(L > 0.0f);
    // partial slot of (batch * H + query head, split s, position)
    const int64_t bh = qrow[qi] / p.Nq;
    const int64_t slot = (bh * p.S + s) * p.Nq + pos[qi];
    p.o_part[slot * DV + e] = empty ? 0.0f : acc / L;
    if (e == 0) p.lse_part[slot] = empty ? -INFINITY : (M + log2f(L)) * kLn2;
  }
}

// Barrier 1 among the first `nthreads` threads (the consumer warps; the
// producer warp, numbered after them, never takes part).
__device__ __forceinline__ void consumers_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
// Same barrier, returning the OR of `pred` over the participants (so every
// consumer takes the same branch after it).
__device__ __forceinline__ bool consumers_sync_or(bool pred, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Consumer warps: twelve for a block of four rows (more warps hide the
// latency of the per-stage shuffle / exponential chain).
__host__ __device__ constexpr int bulk_warps(int QB) { return QB == 4 ? 12 : 0; }
__host__ __device__ constexpr int bulk_threads(int QB) { return (bulk_warps(QB) + 1) * 32; }  // + one producer warp
constexpr int kKeysPerWarp = 8;                       // keys per consumer warp per stage
__host__ __device__ constexpr int bulk_chunk(int QB) { return bulk_warps(QB) * kKeysPerWarp; }  // keys per stage
constexpr int kBulkStages = 4;

template <int D, int QB>
constexpr uint32_t bulk_smem_bytes() {
  return kBulkStages * 2u * bulk_chunk(QB) * D * 2u + 2u * kBulkStages * 8u + 16u;
}

template <int D, int QB>
__global__ void __launch_bounds__(bulk_threads(QB), 1)
    splitkv_partial_bulk_kernel(const PartialParams p) {
  constexpr int kBulkWarps = bulk_warps(QB);
  constexpr int kConsumerThreads = kBulkWarps * 32;
  constexpr int kChunk = bulk_chunk(QB);
  constexpr int LPR = D / 8;            // lanes per key row (16 B each)
  constexpr int G = 32 / LPR;           // key rows per warp instruction
  constexpr int KPW = kChunk / kBulkWarps;  // keys per warp per stage
  constexpr int U = KPW / G;            // key rows per lane group per stage
  constexpr int UB = U;  // key rows per online-softmax step
  constexpr uint32_t kChunkBytes = kChunk * D * 2;
  static_assert(U >= 1 && KPW % G == 0, "stage split");

  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ float sm_m[kBulkWarps][QB];
  __shared__ float sm_l[kBulkWarps][QB];
  __shared__ __align__(16) float sm_o[kBulkWarps][QB][D];
  const uint32_t sbase = smem_u32(dyn);
  const uint32_t bar_base = sbase + kBulkStages * 2u * kChunkBytes;
  auto full = [&](int st) { return bar_base + 8u * st; };
  auto empty = [&](int st) { return bar_base + 8u * (kBulkStages + st); };
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(dyn + kBulkStages * 2u * kChunkBytes + 16u * kBulkStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  // Work item lin = (K/V head bkv, block qb of QB rows, split s); this CTA
  // takes items blockIdx.x, blockIdx.x + gridDim.x, ...  The producer's ring
  // position and the consumers' run on across items, so the next item's
  // K/V stream in while the consumers finish the current one.
  int s = 0;
  int64_t bkv = 0, r0 = 0, k_lo = 0, k_hi = 0;
  int n_chunks = 0;
  int lim_rel[QB];  // last admissible key of each row, relative to k_lo (clamped)
  // Row qi of the current item: query row index (batch*H + head)*Nq + position.
  auto row_of = [&](int qi, int64_t& position) -> int64_t {
    const int64_t r = min(r0 + qi, p.R - 1);
    position = r % p.Nq;
    const int64_t h = (bkv % p.Hkv) * p.G + r / p.Nq;
    return ((bkv / p.Hkv) * p.H + h) * p.Nq + position;
  };
  auto set_item = [&](int64_t lin) {
    r0 = (lin % p.n_qb) * QB;  // same item order as the register-streaming kernel
    const int64_t rest = lin / p.n_qb;
    s = static_cast<int>(rest % p.S);
    bkv = rest / p.S;
    k_lo = static_cast<int64_t>(s) * p.L;
    k_hi = min(k_lo + p.L, p.Nk);
    int64_t top = -1;
#pragma unroll
    for (int qi = 0; qi < QB; ++qi) {
      int64_t position;
      row_of(qi, position);
      const int64_t lim = p.causal ? min(p.Nk - 1, position + p.qoff) : p.Nk - 1;
      top = max(top, lim);
      const int64_t rel = lim - k_lo;
      lim_rel[qi] = static_cast<int>(rel < -1 ? -1 : (rel > (1 << 30) ? (1 << 30) : rel));
    }
    k_hi = min(k_hi, top + 1);
    n_chunks = k_hi > k_lo ? static_cast<int>((k_hi - k_lo + kChunk - 1) / kChunk) : 0;
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < kBulkStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kBulkWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Bounded wait; false when this CTA is aborting or the wait timed out.
  auto wait = [&](uint32_t bar, uint32_t parity, bool honour_abort) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((spin & 31u) == 0) {
        if (honour_abort && *abort_flag) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
          *abort_flag = 1;
          atomicOr(p.status, 1);
          return false;
        }
      }
    }
  };

  if (warp == kBulkWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t last[kBulkStages];
      for (int st = 0; st < kBulkStages; ++st) last[st] = -1;
      int64_t gc = 0;  // ring position over all items
      bool ok = true;
      for (int64_t lin = blockIdx.x; lin < p.n_items && ok; lin += gridDim.x) {
        set_item(lin);
        const uint16_t* kg = p.k + bkv * p.Nk * D;
        const uint16_t* vg = p.v + bkv * p.Nk * D;
        for (int c = 0; c < n_chunks; ++c, ++gc) {
          const int st = static_cast<int>(gc % kBulkStages);
          if (gc >= kBulkStages &&
              !wait(empty(st), static_cast<uint32_t>(((gc / kBulkStages) - 1) & 1), true)) {
            ok = false;
            break;
          }
          const int64_t key0 = k_lo + static_cast<int64_t>(c) * kChunk;
          const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kChunk), k_hi - key0)) * D * 2;
          mbar_arrive_expect_tx(full(st), 2 * bytes);
          bulk_load(sbase + st * 2u * kChunkBytes, kg + key0 * D, bytes, full(st));
          bulk_load(sbase + st * 2u * kChunkBytes + kChunkBytes, vg + key0 * D, bytes, full(st));
          last[st] = gc;
        }
      }
      // Copies in flight must land before the CTA exits (bounded, ignores abort).
      for (int st = 0; st < kBulkStages; ++st)
        if (last[st] >= 0) wait(full(st), static_cast<uint32_t>((last[st] / kBulkStages) & 1), false);
    }
  } else {
    // ------------------------------------------------------------ consumers
    int64_t gc = 0;  // ring position of the current item's first chunk
    for (int64_t lin = blockIdx.x; lin < p.n_items; lin += gridDim.x) {
      set_item(lin);
      bool ok = true;
      float m[QB], l[QB], o[QB][8];
      static_assert(QB * UB == LPR && UB == U, "four rows of a K/V head per item");
      // One score per lane (the UB = U keys of a stage at once): after packed
      // partial dot products, a
      // reduce-scatter over the LPR lanes of a key row leaves lane `sub` the
      // full score of (row sub / UB, key sub % UB) of the current UB keys, so
      // each exponential is computed once, the row max and sum take
      // log2(UB) shuffles, and the P V update broadcasts p and alpha.
      uint64_t q2[QB][4];
#pragma unroll
      for (int qi = 0; qi < QB; ++qi) {
        int64_t position;
        const uint4 r = ld_stream(p.q + row_of(qi, position) * D + 8 * sub);
        float qf[8];
        unpack8(r, qf);
#pragma unroll
        for (int e = 0; e < 4; ++e) q2[qi][e] = f2_pack(qf[2 * e] * p.sc_log2, qf[2 * e + 1] * p.sc_log2);
      }
      const int own_row = sub / UB, own_u = sub % UB;
      int lim_own = lim_rel[0];
#pragma unroll
      for (int qi = 1; qi < QB; ++qi) lim_own = (own_row == qi) ? lim_rel[qi] : lim_own;
      float m_row = -INFINITY, l_row = 0.0f;  // state of row own_row (same in its UB lanes)
      uint64_t o2[QB][4];
#pragma unroll
      for (int qi = 0; qi < QB; ++qi)
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[qi][e] = 0ull;
      for (int c = 0; c < n_chunks; ++c) {
        const int st = static_cast<int>((gc + c) % kBulkStages);
        if (!__all_sync(0xffffffffu,
                        wait(full(st), static_cast<uint32_t>(((gc + c) / kBulkStages) & 1), true))) {
          ok = false;
          break;
        }
        const int64_t key0 = k_lo + static_cast<int64_t>(c) * kChunk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(kChunk), k_hi - key0));
        const uint16_t* ks = reinterpret_cast<const uint16_t*>(dyn + st * 2u * kChunkBytes);
        const uint16_t* vs = ks + kChunk * D;
        uint4 kr[UB], vr[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
          const int kk = warp * KPW + u * G + grp;
          if (kk < nk) {
            kr[u] = *reinterpret_cast<const uint4*>(ks + kk * D + 8 * sub);
            vr[u] = *reinterpret_cast<const uint4*>(vs + kk * D + 8 * sub);
          } else {
            kr[u] = make_uint4(0u, 0u, 0u, 0u);
            vr[u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(st));  // release orders this warp's reads
        float part[QB * UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
          float kf[8];
          unpack8(kr[u], kf);
#pragma unroll
          for (int qi = 0; qi < QB; ++qi) {
            uint64_t d2 = f2_mul(q2[qi][0], f2_pack(kf[0], kf[1]));
            d2 = f2_fma(q2[qi][1], f2_pack(kf[2], kf[3]), d2);
            d2 = f2_fma(q2[qi][2], f2_pack(kf[4], kf[5]), d2);
            d2 = f2_fma(q2[qi][3], f2_pack(kf[6], kf[7]), d2);
            float x0, x1;
            f2_unpack(d2, x0, x1);
            part[qi * UB + u] = x0 + x1;
          }
        }
        // Reduce-scatter: at mask m the lane keeps the half of its values
        // selected by bit m of sub and adds its partner's copy of that half.
#pragma unroll
        for (int m = LPR / 2, n = QB * UB; m >= 1; m >>= 1, n >>= 1) {
          const bool upper = (sub & m) != 0;
#pragma unroll
          for (int i = 0; i < n / 2; ++i) {
            const float keep = upper ? part[i + n / 2] : part[i];
            const float send = upper ? part[i] : part[i + n / 2];
            part[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        const int kk_own = warp * KPW + own_u * G + grp;
        const int key_rel = static_cast<int>(key0 - k_lo) + kk_own;
        const float s_own = (kk_own < nk && key_rel <= lim_own) ? part[0] : -INFINITY;
        float mx = s_own;
#pragma unroll
        for (int m = 1; m < UB; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        const float m_new = fmaxf(m_row, mx);
        const bool live = m_new != -INFINITY;
        const float alpha_own = live ? ex2_approx(m_row - m_new) : 1.0f;  // 0 when m_row = -inf
        const float p_own = live ? ex2_approx(s_own - m_new) : 0.0f;
        float ps = p_own;
#pragma unroll
        for (int m = 1; m < UB; m <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, m);
        l_row = l_row * alpha_own + ps;
        if (live) m_row = m_new;
        // P V: every lane updates its 8 d-columns of every row.
        const int base = grp * LPR;
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
          const float al = __shfl_sync(0xffffffffu, alpha_own, base + qi * UB);
          const uint64_t al2 = f2_pack(al, al);
#pragma unroll
          for (int e = 0; e < 4; ++e) o2[qi][e] = f2_mul(o2[qi][e], al2);
        }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
          float vf[8];
          unpack8(vr[u], vf);
#pragma unroll
          for (int qi = 0; qi < QB; ++qi) {
            const float pu = __shfl_sync(0xffffffffu, p_own, base + qi * UB + u);
            const uint64_t p2 = f2_pack(pu, pu);
#pragma unroll
            for (int e = 0; e < 4; ++e) o2[qi][e] = f2_fma(p2, f2_pack(vf[2 * e], vf[2 * e + 1]), o2[qi][e]);
          }
        }
      }
      // Per-row state of every row in every lane, for the merges below.
#pragma unroll
      for (int qi = 0; qi < QB; ++qi) {
        m[qi] = __shfl_sync(0xffffffffu, m_row, grp * LPR + qi * UB);
        l[qi] = __shfl_sync(0xffffffffu, l_row, grp * LPR + qi * UB);
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(o2[qi][e], o[qi][2 * e], o[qi][2 * e + 1]);
      }
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m[qi], off);
          const float l2 = __shfl_xor_sync(0xffffffffu, l[qi], off);
          float o2[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, o[qi][e], off);
          merge_state(m[qi], l[qi], o[qi], m2, l2, o2);
        }
      }
      gc += n_chunks;
      if (grp == 0) {
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
#pragma unroll
          for (int e = 0; e < 8; ++e) sm_o[warp][qi][8 * sub + e] = o[qi][e];
          if (sub == 0) {
            sm_m[warp][qi] = m[qi];
            sm_l[warp][qi] = l[qi];
          }
        }
      }
      consumers_sync(kConsumerThreads);

      for (int idx = threadIdx.x; idx < QB * D; idx += kConsumerThreads) {
        const int qi = idx / D, e = idx % D;
        if (r0 + qi >= p.R) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kBulkWarps; ++w) M = fmaxf(M, sm_m[w][qi]);
        float L = 0.0f, acc = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kBulkWarps; ++w) {
            const float f = ex2_approx(sm_m[w][qi] - M);
            L = fmaf(sm_l[w][qi], f, L);
            acc = fmaf(sm_o[w][qi][e], f, acc);
          }
        }
        const bool empty_row = !(L > 0.0f);
        int64_t ps;
        const int64_t qr = row_of(qi, ps);
        const int64_t slot = ((qr / p.Nq) * p.S + s) * p.Nq + ps;
        p.o_part[slot * D + e] = empty_row ? 0.0f : acc / L;
        if (e == 0) p.lse_part[slot] = empty_row ? -INFINITY : (M + log2f(L)) * kLn2;
      }
      // Second meeting: the shared state may be overwritten by the next
      // item, and the consumers leave together if any of them gave up a wait.
      if (consumers_sync_or(!ok, kConsumerThreads)) break;
    }  // items
  }
}

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part,
                                                      uint16_t* __restrict__ o,
                                                      float* __restrict__ lse, int64_t rows,
                                                      int64_t Nq, int S) {
  constexpr int E = D / 32;  // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  const int64_t bh = row / Nq, i = row % Nq;
  const float* lp = lse_part + bh * S * Nq + i;  // split s at lp[s * Nq]

  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lp[static_cast<int64_t>(s) * Nq]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  static_assert(E == 2 || E == 3 || E == 4 || E == 8, "head dims 64, 96, 128, 256");
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float W = 0.0f;
  if (M != -INFINITY) {
    // Lane j computes the weight of split s0 + j; the splits' partial rows
    // are then read eight at a time (independent loads in flight) with the
    // weight broadcast from its lane.
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int n = min(32, S - s0);
      const float w_lane =
          lane < n ? ex2_approx((lp[static_cast<int64_t>(s0 + lane) * Nq] - M) * kLog2e) : 0.0f;
      W += w_lane;
      const float* op = o_part + ((bh * S + s0) * Nq + i) * D + lane * E;
      const int64_t stride = Nq * D;  // one split further
#pragma unroll 8
      for (int j = 0; j < n; ++j) {
        const float w = __shfl_sync(0xffffffffu, w_lane, j);
        if constexpr (E == 4 || E == 8) {
#pragma unroll
          for (int c = 0; c < E / 4; ++c) {
            const float4 x = *reinterpret_cast<const float4*>(op + j * stride + 4 * c);
            acc[4 * c + 0] = fmaf(w, x.x, acc[4 * c + 0]);
            acc[4 * c + 1] = fmaf(w, x.y, acc[4 * c + 1]);
            acc[4 * c + 2] = fmaf(w, x.z, acc[4 * c + 2]);
            acc[4 * c + 3] = fmaf(w, x.w, acc[4 * c + 3]);
          }
        } else if constexpr (E == 3) {
#pragma unroll
          for (int c = 0; c < 3; ++c) acc[c] = fmaf(w, op[j * stride + c], acc[c]);
        } else {
          const float2 x = *reinterpret_cast<const float2*>(op + j * stride);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  }
  const bool empty = !(W > 0.0f);
  const float inv = empty ? 0.0f : 1.0f / W;
  uint16_t* dst = o + row * D + lane * E;
  if constexpr (E == 8) {
    uint4 pk;
    pk.x = empty ? 0u : pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = empty ? 0u : pack_bf16x2(acc[2] * inv, acc[3] * inv);
    pk.z = empty ? 0u : pack_bf16x2(acc[4] * inv, acc[5] * inv);
    pk.w = empty ? 0u : pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(dst) = pk;
  } else if constexpr (E == 4) {
    uint2 pk;
    pk.x = empty ? 0u : pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = empty ? 0u : pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else if constexpr (E == 3) {
    // Three values per lane (d = 96): 6-byte rows slices, 2-byte stores.
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const uint32_t b = empty ? 0u : pack_bf16x2(acc[c] * inv, 0.0f);
      dst[c] = static_cast<uint16_t>(b & 0xFFFFu);
    }
  } else {
    *reinterpret_cast<uint32_t*>(dst) = empty ? 0u : pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) lse[row] = empty ? -INFINITY : M + logf(W);
}

template <int D, int DV, int QB, int U, int MINB>
cudaError_t launch_partial(const SplitArgs& a, cudaStream_t stream) {
  PartialParams p = {};
  p.q = static_cast<const uint16_t*>(a.q);
  p.k = static_cast<const uint16_t*>(a.k);
  p.v = static_cast<const uint16_t*>(a.v);
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.qoff = a.query_offset;
  p.L = a.keys_per_split;
  p.S = a.splits;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.R = p.G * a.Nq;
  p.n_qb = static_cast<int>((p.R + QB - 1) / QB);
  p.causal = a.causal;
  p.sc_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  const int64_t blocks = (a.BH / p.G) * p.n_qb * a.splits;
  splitkv_partial_kernel<D, DV, QB, U, MINB>
      <<<dim3(static_cast<unsigned>(blocks)), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int QB>
cudaError_t launch_partial_bulk(const SplitArgs& a, cudaStream_t stream) {
  PartialParams p = {};
  p.q = static_cast<const uint16_t*>(a.q);
  p.k = static_cast<const uint16_t*>(a.k);
  p.v = static_cast<const uint16_t*>(a.v);
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.qoff = a.query_offset;
  p.L = a.keys_per_split;
  p.S = a.splits;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.R = p.G * a.Nq;
  p.n_qb = static_cast<int>((p.R + QB - 1) / QB);
  p.causal = a.causal;
  p.sc_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  constexpr uint32_t smem = bulk_smem_bytes<D, QB>();
  cudaError_t err = cudaFuncSetAttribute(splitkv_partial_bulk_kernel<D, QB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  p.n_items = (a.BH / p.G) * p.n_qb * a.splits;
  // Persistent: one CTA per SM (the ring takes most of an SM's shared
  // memory), each walking every gridDim.x-th item.
  int dev = 0, sms = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int64_t blocks = std::min<int64_t>(p.n_items, std::max(sms, 1));
  splitkv_partial_bulk_kernel<D, QB>
      <<<dim3(static_cast<unsigned>(blocks)), bulk_threads(QB), smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitkv_partial(const SplitArgs& a, cudaStream_t stream) {
  // One row per K/V head: register streaming.  Several rows (GQA groups,
  // Nq > 1): the bulk-copy pipeline, which reads each K/V byte once per CTA.
  // A value dim different from the key dim: register streaming, one row per
  // CTA (the caller sized the grid for that).
  if (a.dv > 0 && a.dv != a.d)
    return a.d == 64 ? launch_partial<64, 128, 1, 4, 2>(a, stream)
                     : launch_partial<128, 64, 1, 4, 2>(a, stream);
  const int64_t qb = splitkv_rows_per_cta((a.H / a.Hkv) * a.Nq);
  if (a.d == 64)
    return qb == 1 ? launch_partial<64, 64, 1, 4, 2>(a, stream)
                   : launch_partial_bulk<64, 4>(a, stream);
  return qb == 1 ? launch_partial<128, 128, 1, 4, 2>(a, stream)
                 : launch_partial_bulk<128, 4>(a, stream);
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                           int64_t BH, int64_t Nq, int d, int splits, cudaStream_t stream) {
  const int64_t rows = BH * Nq;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  uint16_t* out = static_cast<uint16_t*>(o);
  switch (d) {
    case 64: combine_kernel<64><<<blocks, 256, 0, stream>>>(o_part, lse_part, out, lse, rows, Nq, splits); break;
    case 96: combine_kernel<96><<<blocks, 256, 0, stream>>>(o_part, lse_part, out, lse, rows, Nq, splits); break;
    case 256: combine_kernel<256><<<blocks, 256, 0, stream>>>(o_part, lse_part, out, lse, rows, Nq, splits); break;
    default: combine_kernel<128><<<blocks, 256, 0, stream>>>(o_part, lse_part, out, lse, rows, Nq, splits); break;
  }
  return cudaGetLastError();
}

}  // namespace attn
