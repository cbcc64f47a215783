// internal.cuh -- launch interfaces between the C-ABI layer (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "attn.h"

namespace attn {

// Argument checks shared by the forward entry points (api.cu): null
// pointers, sizes, scale, offsets, head dims, size limits and alignment.
// Returns ATTN_OK or the attn_status to report; makes no CUDA call.
int validate(const attn_params* p);

// Head dims the forward entry points take: 64, 96, 128 and 256.
bool head_dim_supported(int64_t d);

// Keys per split-KV range: ceil(Nk / splits) rounded up to a multiple of 128.
int64_t keys_per_split(int64_t Nk, int splits);

// x rounded up to a multiple of 256 (workspace sub-buffer alignment).
size_t align256(size_t x);

// Arguments of one prefill (tcgen05) launch, already validated.
struct FwdArgs {
  void* o;             // bf16 [B][H][Nq][d]
  float* lse;          // f32  [B][H][Nq]
  int* status;         // device status word (bit 0 = wait timeout)
  int64_t BH, Nq, Nk, query_offset;
  int64_t H, group;    // query heads per batch; query heads per K/V head
  int fp8_qk;          // Q and K are e4m3 (scale already includes the descales)
  int d;               // head dim of Q and K
  int dv;              // head dim of V and O
  int causal;
  float scale;
  uint32_t flags;
  uint64_t timeout_ns;
};

// Arguments of one split-KV decode launch pair, already validated.
struct SplitArgs {
  const void *q, *k, *v;  // bf16 q [B][H][Nq][d], k [B][Hkv][Nk][d], v [B][Hkv][Nk][dv]
  float* o_part;          // f32 [BH][S][Nq][dv]
  float* lse_part;        // f32 [BH][S][Nq]
  int64_t BH, Nq, Nk, query_offset;  // BH: batch x query heads
  int64_t H, Hkv;                     // query heads and K/V heads per batch
  int64_t keys_per_split;
  int d;
  int dv = 0;  // value head dim (0 = d); dv != d runs one query row per partial CTA
  int splits;
  int causal;
  float scale;
  int* status;          // device status word (bit 0 = wait timeout)
  uint64_t timeout_ns;  // per-wait limit of the pipelined partial kernel
};

// Fewest query rows per CTA of the prefill kernel (one 128-row tile; two-tile
// configurations take 256), for grid-size checks.
constexpr int kFwdRowsPerCta = 128;

// Query rows one split-KV partial work item serves, out of the rows that
// share one K/V head (query heads of the group x query positions): one, or
// blocks of four (the pipelined kernel's reduce-scatter layout; larger
// groups take several blocks, which read the same K/V slice back to back).
inline int64_t splitkv_rows_per_cta(int64_t rows_per_kv_head) {
  return rows_per_kv_head == 1 ? 1 : 4;
}

// Arguments of one backward pass, already validated.
struct BwdArgs {
  const void *o, *dout;  // bf16 [B][H][Nq][dv]
  const float* lse;      // f32 [B][H][Nq] from the forward pass
  float* delta;          // workspace f32 [B][H][Nq]: rowsum(dO * O)
  void *dq, *dk, *dv;    // bf16 outputs, [B][H][Nq][d], [B][Hkv][Nk][d], [B][Hkv][Nk][dv]
  int* status;
  int64_t B, H, Hkv, Nq, Nk, query_offset;
  int causal;
  float scale;
  uint64_t timeout_ns;
};

// Backward launches for key head dim D and value head dim DV, one
// translation unit each (bwd_tcgen05.cu: 128/128, bwd_tcgen05_d64.cu: 64/64,
// bwd_tcgen05_d64_v128.cu, bwd_tcgen05_d128_v64.cu, bwd_tcgen05_d96.cu: 96/96).
template <int D, int DV>
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t stream);
#define ATTN_DECLARE_BWD(D_, DV_)                                                        \
  template <>                                                                            \
  cudaError_t launch_bwd<D_, DV_>(const BwdArgs&, const CUtensorMap&, const CUtensorMap&, \
                                  const CUtensorMap&, const CUtensorMap&, cudaStream_t);
ATTN_DECLARE_BWD(64, 64)
ATTN_DECLARE_BWD(128, 128)
ATTN_DECLARE_BWD(64, 128)
ATTN_DECLARE_BWD(128, 64)
ATTN_DECLARE_BWD(96, 96)
#undef ATTN_DECLARE_BWD

// Split-KV partial on the tensor cores for rows that share K/V heads
// (splitkv_tc.cu): tq maps Q as [B*H*Nq rows][d] (z extent 1), tk and tv as
// the prefill's [B*Hkv][Nk][d] maps.  dv must equal d.
cudaError_t launch_splitkv_partial_tc(const SplitArgs& a, const CUtensorMap& tq,
                                      const CUtensorMap& tk, const CUtensorMap& tv,
                                      cudaStream_t stream);

// Smallest number of query rows per K/V head that the split-KV path serves
// with the tensor-core partial kernel, per head dim; fewer go to the
// CUDA-core kernels.  Measured, B16 H32 Nk 32768 (tensor cores vs CUDA
// cores): d = 128, two rows 0.605 vs 0.636 ms, four 0.320 vs 0.344, eight
// 0.170 vs 0.336; d = 64, four rows 0.246 vs 0.233.
#ifndef ATTN_SPLITKV_TC_MIN_ROWS_D128
#define ATTN_SPLITKV_TC_MIN_ROWS_D128 2
#endif
#ifndef ATTN_SPLITKV_TC_MIN_ROWS_D64
#define ATTN_SPLITKV_TC_MIN_ROWS_D64 5
#endif

cudaError_t launch_fwd_tcgen05(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, cudaStream_t stream);

cudaError_t launch_splitkv_partial(const SplitArgs& a, cudaStream_t stream);

cudaError_t launch_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                           int64_t BH, int64_t Nq, int d, int splits, cudaStream_t stream);

// Address of the library's own device status word on the current device.
cudaError_t default_status_word(int** ptr);

}  // namespace attn
