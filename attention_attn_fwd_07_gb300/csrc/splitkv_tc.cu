// splitkv_tc.cu -- split-KV partial on the tensor cores, for the query rows
// that share one K/V head (grouped-query heads, several query positions).
//
// The rows of one K/V head are G query heads x Nq positions, and in the
// [B][H][Nq][d] layout they are G*Nq consecutive rows, so one 128-row TMA box
// loads a block of them.  One CTA per (b, K/V head, key split, block of up to
// 128 rows) runs the prefill kernel's pipeline over the split's keys
// [s*L, min((s+1)*L, Nk)) (online softmax of "GPU Engineering: Correctness,
// Throughput, and Attention", section 22.5, with the section 22.7 lab's mask
// j > i + query_offset, i the row's position):
//   warp 5      TMA producer: the Q block once, then K0 V0 K1 V1 ... through
//               an NS-stage shared-memory ring (full/empty mbarriers);
//   warp 4      MMA issuer: S = Q K^T (SS MMA into TMEM), O += P V (TS MMA,
//               P read from TMEM), the next S after P V;
//   warps 0-3   softmax, one thread per row (TMEM lane = row): the row
//               maximum comes with the TMEM load on tiles that need no mask;
//               rows past the block are never written out, so they are left
//               unmasked, and a warp with no row in the block only keeps pace
//               with the barriers; P goes back into the S columns in two
//               halves of 64 keys, each announced on its own barrier; O is
//               rescaled in TMEM only when the row maximum grew by more than
//               2^8.  Epilogue: the normalised o (f32) and the natural-log
//               LSE of the split, o = 0 and lse = -inf for a row with no
//               admissible key in the split.
// TMEM: S [0,128), O [128,128+d), 256 columns, and a 2-stage ring (4 at
// d = 64) so that two CTAs share an SM: their independent S -> softmax ->
// P V chains cover each other's latency (d = 256: 512 columns and 192 KB of
// shared memory, one CTA per SM).  The tensor core is far from busy
// (a few real rows per MMA); the point is to keep the CUDA cores out of the
// dot products, so that any number of rows per K/V head streams K and V at
// memory speed.  Every mbarrier wait is bounded (status word, clean exit).
#include <algorithm>
#include <cuda_bf16.h>

#include "attn.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // rows per block (= TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int kThreads = 192;
constexpr int kWarpMma = 4;
constexpr int kWarpLoad = 5;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct TcCfg {
  // 128-byte swizzle atoms per row; d = 96 leaves half of its second atom to
  // the tensor map's zero fill.
  static constexpr int kAtoms = (D + 63) / 64;
  static constexpr int kQKSteps = D / 16;                  // MMA K steps of 16 bf16
  static constexpr uint32_t kAtomBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kAtoms * kAtomBytes;  // Q block, K tile, V tile
  // Two CTAs per SM (256 TMEM columns each) up to d = 128; d = 256 needs
  // 384 columns and 192 KB of shared memory, one CTA per SM.
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = kTileBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kTileBytes;
  // barriers: full[S], empty[S], q_full, s_full, p_ready (keys 0-63 of P),
  // p2_ready (keys 64-127), o_full, drain
  static constexpr int kBarFull = 0;
  static constexpr int kBarEmpty = kStages;
  static constexpr int kBarQ = 2 * kStages;
  static constexpr int kBarS = kBarQ + 1;
  static constexpr int kBarP = kBarS + 1;
  static constexpr int kBarP2 = kBarP + 1;
  static constexpr int kBarO = kBarP2 + 1;
  static constexpr int kBarDrain = kBarO + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0, kColO = 128;
  static constexpr uint32_t kTmemCols = 128 + D <= 256 ? 256 : 512;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, 1);
  static_assert(D == 64 || D == 96 || D == 128 || D == 256, "head dims 64, 96, 128, 256");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kTmemCols == 256 || kSmemBytes > 232448 / 2,
                "a 512-column CTA keeps the SM's tensor memory to itself");
  static_assert(kTmemCols == 512 || 2 * (kSmemBytes + 1024) <= 232448, "two CTAs per SM");
};

struct TcParams {
  float* o_part;    // f32 [B*H][S][Nq][d]
  float* lse_part;  // f32 [B*H][S][Nq]
  int* status;
  int64_t Nq, Nk, qoff, L;
  int64_t H, Hkv, G, R;  // query heads, K/V heads, group size, rows per K/V head
  int S, n_rb, causal;
  float sc_log2;
  uint64_t timeout_ns;
};

struct TcWaiter {
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

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    splitkv_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcParams p) {
  using C = TcCfg<D>;
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

  // CTA -> (K/V head bkv, split s, row block rb); the row blocks of one K/V
  // slice are neighbours, so they run together and share the slice in L2.
  const int64_t lin = blockIdx.x;
  const int rb = static_cast<int>(lin % p.n_rb);
  const int64_t rest = lin / p.n_rb;
  const int s = static_cast<int>(rest % p.S);
  const int64_t bkv = rest / p.S;  // batch * Hkv + K/V head
  const int64_t r0 = static_cast<int64_t>(rb) * BM;   // first row of the block in the group
  const int rows = static_cast<int>(min(static_cast<int64_t>(BM), p.R - r0));
  const int64_t b = bkv / p.Hkv, hk = bkv % p.Hkv;
  const int64_t q_row0 = (b * p.H + hk * p.G) * p.Nq + r0;  // flattened [B*H*Nq] row
  const int64_t k_lo = static_cast<int64_t>(s) * p.L;
  int64_t k_hi = min(k_lo + p.L, p.Nk);
  if (p.causal) {
    // Largest position among the block's rows (consecutive modulo Nq).
    const int64_t pos0 = r0 % p.Nq;
    const int64_t max_pos = (pos0 + rows - 1 >= p.Nq) ? p.Nq - 1 : pos0 + rows - 1;
    k_hi = min(k_hi, max_pos + p.qoff + 1);
  }
  const int n_blk = k_hi > k_lo ? static_cast<int>((k_hi - k_lo + BN - 1) / BN) : 0;

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(bar(C::kBarFull + st), 1);
      mbar_init(bar(C::kBarEmpty + st), 1);
    }
    mbar_init(bar(C::kBarQ), 1);
    mbar_init(bar(C::kBarS), 1);
    mbar_init(bar(C::kBarP), 4);  // one arrival per softmax warp
    mbar_init(bar(C::kBarP2), 4);
    mbar_init(bar(C::kBarO), 1);
    mbar_init(bar(C::kBarDrain), 1);
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
  const TcWaiter wait{abort_flag, p.status, p.timeout_ns};
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sKV = sbase + C::kOffKV;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_blk > 0) {
      mbar_arrive_expect_tx(bar(C::kBarQ), C::kTileBytes);
      for (int a = 0; a < C::kAtoms; ++a)
        tma_load_3d(sQ + a * C::kAtomBytes, &tq, bar(C::kBarQ), a * 64, static_cast<int>(q_row0), 0);
      // Ring position t: K(t/2) for even t, V(t/2) for odd t.
      int last_t[C::kStages];
      for (int st = 0; st < C::kStages; ++st) last_t[st] = -1;
      bool ok = true;
      for (int t = 0; t < 2 * n_blk && ok; ++t) {
        const int st = t % C::kStages;
        if (t >= C::kStages) ok = wait(bar(C::kBarEmpty + st), ((t / C::kStages) - 1) & 1);
        if (!ok) break;
        last_t[st] = t;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), C::kTileBytes);
        const int key0 = static_cast<int>(k_lo) + (t >> 1) * BN;
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d(sKV + st * C::kTileBytes + a * C::kAtomBytes, (t & 1) ? &tv : &tk,
                      bar(C::kBarFull + st), a * 64, key0, static_cast<int>(bkv));
      }
      // Every issued copy must land before the CTA exits (bounded, ignores
      // the abort flag: these cover copies in flight).
      volatile int no_abort = 0;
      const TcWaiter own{&no_abort, p.status, p.timeout_ns};
      own(bar(C::kBarQ), 0);
      for (int st = 0; st < C::kStages; ++st)
        if (last_t[st] >= 0) own(bar(C::kBarFull + st), (last_t[st] / C::kStages) & 1);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits made warp-uniform); each run of
    // MMAs and each commit elects one lane to issue.
    auto wait_w = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait(b, parity));
    };
    if (n_blk > 0) {
      auto qk = [&](int stage) {
        const uint64_t a = sdesc_sw128(sQ, 16, 1024);
        const uint64_t bd = sdesc_sw128(sKV + stage * C::kTileBytes, 16, 1024);
        if constexpr (C::kQKSteps == 16) {
          mma_ss_run8_w(tmem + C::kColS, a, bd, C::kIdescQK, 0u);
          mma_ss_run8_w(tmem + C::kColS, a + 2048, bd + 2048, C::kIdescQK, 1u);  // atoms 2, 3
        } else if constexpr (C::kQKSteps == 8) {
          mma_ss_run8_w(tmem + C::kColS, a, bd, C::kIdescQK, 0u);
        } else if constexpr (C::kQKSteps == 6) {
          mma_ss_run6_w(tmem + C::kColS, a, bd, C::kIdescQK, 0u);
        } else {
          mma_ss_run4_w(tmem + C::kColS, a, bd, C::kIdescQK, 0u);
        }
        mma_commit_w(bar(C::kBarS));
      };
      // O += P V over keys 64 h .. 64 h + 63 (P's bf16 pairs in columns 32 h ..).
      auto pv_half = [&](int stage, int h, bool acc) {
        const uint64_t bd = sdesc_sw128(sKV + stage * C::kTileBytes + h * 64 * 128, C::kAtomBytes, 1024);
        mma_ts_run4_w(tmem + C::kColO, tmem + C::kColS + 32 * h, bd, C::kIdescPV, acc ? 1u : 0u);
      };
      bool ok = wait_w(bar(C::kBarQ), 0) && wait_w(bar(C::kBarFull + 0), 0);
      if (ok) {
        tc_fence_after();
        qk(0);
        mma_commit_w(bar(C::kBarEmpty + 0));
      }
      for (int j = 0; j < n_blk && ok; ++j) {
        const int tV = 2 * j + 1, sV = tV % C::kStages;
        const int tK = 2 * j + 2, sK = tK % C::kStages;
        ok = wait_w(bar(C::kBarFull + sV), (tV / C::kStages) & 1) && wait_w(bar(C::kBarP), j & 1);
        if (!ok) break;
        tc_fence_after();
        pv_half(sV, 0, j > 0);
        ok = wait_w(bar(C::kBarP2), j & 1);
        if (!ok) break;
        tc_fence_after();
        pv_half(sV, 1, true);
        mma_commit_w(bar(C::kBarEmpty + sV));
        if (j + 1 < n_blk) {
          ok = wait_w(bar(C::kBarFull + sK), (tK / C::kStages) & 1);
          if (!ok) break;
          tc_fence_after();
          qk(sK);
          mma_commit_w(bar(C::kBarEmpty + sK));
        }
      }
      if (ok) mma_commit_w(bar(C::kBarO));
      // All issued MMAs complete before TMEM is released (bounded, ignores abort).
      mma_commit_w(bar(C::kBarDrain));
      volatile int no_abort = 0;
      const TcWaiter own{&no_abort, p.status, p.timeout_ns};
      own(bar(C::kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = (warp << 5) + lane;  // row of the block = TMEM lane
    const bool valid = row < rows;
    const int64_t r = r0 + row;          // row within the K/V head's group
    const int64_t pos = valid ? r % p.Nq : 0;
    // Last admissible key (absolute).  Rows past the block are left unmasked:
    // their rows of P and O are never read back, and a warp with nothing to
    // mask takes the row maximum from the TMEM load.
    int64_t lim = k_hi - 1;
    if (valid && p.causal) lim = min(lim, pos + p.qoff);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS;
    const uint32_t tO = tmem + lane_off + C::kColO;
    // A warp none of whose rows is in the block only keeps pace with the
    // barriers: its rows of P and O are never read back (each row of P V
    // depends on that row of P alone), so it skips the softmax and the
    // epilogue, leaving the issue slots of its SMSP to the live rows.
    const bool idle = __all_sync(0xffffffffu, !valid);
    float m_run = -INFINITY, m_ref = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; idle && j < n_blk; ++j) {
      ok = __all_sync(0xffffffffu, wait(bar(C::kBarS), j & 1));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive(bar(C::kBarP));
        mbar_arrive(bar(C::kBarP2));
      }
    }
    for (int j = 0; !idle && j < n_blk; ++j) {
      ok = __all_sync(0xffffffffu, wait(bar(C::kBarS), j & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[128];
      // The load returns the row maximum of the unmasked tile.
      float tmax = tmem_ld_max_x128(tS, sr);
      float sv[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(sr[c]);
      const int64_t k0 = k_lo + static_cast<int64_t>(j) * BN;
      {
        const int64_t rel64 = lim - k0;
        const int rel = static_cast<int>(rel64 < -1 ? -1 : (rel64 > BN ? BN : rel64));
        if (__any_sync(0xffffffffu, rel < BN - 1)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c > rel) ? -INFINITY : sv[c];
          // Masking invalidates the load's maximum.
          float mx[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            mx[g] = fmaxf(sv[16 * g], sv[16 * g + 1]);
#pragma unroll
            for (int c = 2; c < 16; c += 2) mx[g] = fmax3f(mx[g], sv[16 * g + c], sv[16 * g + c + 1]);
          }
          tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                        fmaxf(mx[6], mx[7]));
        }
      }
      const float m_new = fmaxf(m_run, tmax * p.sc_log2);
      m_run = m_new;
      float alpha = 1.0f;
      bool rescale = false;
      if (m_new > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
        rescale = valid && (m_ref != -INFINITY);  // rows past the block: no O to keep
        l *= alpha;
        m_ref = m_new;
      }
      const float neg_ref = (m_ref == -INFINITY) ? 0.0f : -m_ref;
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
          f2_unpack(f2_fma(f2_pack(sv[2 * cc], sv[2 * cc + 1]), scale2, bias2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          acc2[c & 3] = f2_add(acc2[c & 3], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st_x32(tS + 32 * h, pk);
        if (h == 0 && __any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
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
        if (lane == 0) mbar_arrive(bar(h == 0 ? C::kBarP : C::kBarP2));
      }
      float sum_lo, sum_hi;
      f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), sum_lo, sum_hi);
      l += sum_lo + sum_hi;
    }
    if (ok && n_blk > 0 && !idle) {
      ok = __all_sync(0xffffffffu, wait(bar(C::kBarO), 0));
      if (ok) tc_fence_after();
    }
    if (ok && !idle) {
      // Partial slot of (batch*H + query head, split s, position).
      const int64_t bh = b * p.H + hk * p.G + (valid ? r / p.Nq : 0);
      const int64_t slot = (bh * p.S + s) * p.Nq + pos;
      const bool empty = (n_blk == 0) || !(l > 0.0f);
      const float inv = empty ? 0.0f : 1.0f / l;
      float4* dst = reinterpret_cast<float4*>(p.o_part + slot * D);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32] = {};
        if (n_blk > 0) tmem_ld_x32(tO + cc * 32, o);  // warp-collective: every lane
        if (valid) {
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            float4 w = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (!empty)
              w = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                              __uint_as_float(o[4 * v4 + 2]) * inv,
                              __uint_as_float(o[4 * v4 + 3]) * inv);
            dst[cc * 8 + v4] = w;
          }
        }
      }
      if (valid) p.lse_part[slot] = empty ? -INFINITY : (m_ref + log2f(l)) * kLn2;
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

template <int D>
cudaError_t launch_tc(const SplitArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, cudaStream_t stream) {
  using C = TcCfg<D>;
  cudaError_t err = cudaFuncSetAttribute(splitkv_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
  if (err != cudaSuccess) return err;
  TcParams p = {};
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.status = a.status;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.qoff = a.query_offset;
  p.L = a.keys_per_split;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.R = p.G * a.Nq;
  p.S = a.splits;
  p.n_rb = static_cast<int>((p.R + BM - 1) / BM);
  p.causal = a.causal;
  p.sc_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.timeout_ns = a.timeout_ns;
  const int64_t blocks = (a.BH / p.G) * p.n_rb * a.splits;
  splitkv_tc_kernel<D><<<dim3(static_cast<unsigned>(blocks)), dim3(kThreads), C::kSmemBytes,
                         stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitkv_partial_tc(const SplitArgs& a, const CUtensorMap& tq,
                                      const CUtensorMap& tk, const CUtensorMap& tv,
                                      cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_tc<64>(a, tq, tk, tv, stream);
    case 96: return launch_tc<96>(a, tq, tk, tv, stream);
    case 256: return launch_tc<256>(a, tq, tk, tv, stream);
    default: return launch_tc<128>(a, tq, tk, tv, stream);
  }
}

}  // namespace attn
