// noalloc.cu -- attn_fwd_splitkv_noalloc: the split-KV forward with its
// scratch (the per-split partial outputs and log-sum-exps) in a fixed
// device array owned by this library, for callers that cannot allocate
// device memory themselves.
//
// Who needs this: a caller whose device memory is entirely planned and
// owned by an outer arena (for example a serving process that reserves all
// memory at start-up and forbids any further cudaMalloc), a plug-in running
// inside a host program that exposes no allocator, or a latency-critical
// loop where cudaMalloc/cudaFree may synchronise the device.  Such callers
// still pass their own q, k, v, o and lse; only the scratch moves here.
//
// The array below is ATTN_NOALLOC_SCRATCH_BYTES (32 MiB) on every GPU that
// loads this library, held until the process exits.  Every call shares it
// and it keeps the previous call's contents.  Nothing in it needs clearing:
// the partial kernel writes every slot the combine kernel reads in the same
// call (an empty split writes o = 0, lse = -inf).  Calls that overlap on the
// GPU (different streams, or different host threads on one device) race on
// the array and give undefined results; serialise them.
#include <cstdint>

#include "attn.h"
#include "internal.cuh"

namespace attn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// With the caller's device current: translate the array's host-side name
// into its device address on that device.  The name itself is only a host
// stand-in and must never be passed to a kernel.  The lookup is repeated on
// every call (a host-side table lookup, no device work), so an address from
// a context that was since torn down (cudaDeviceReset) is never reused.
int scratch_address(void** out) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
    return ATTN_ERR_CUDA;
  *out = ptr;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                                        int64_t d, int causal, float scale, int num_splits,
                                        cudaStream_t stream) {
  // The argument rules of attn_fwd_splitkv: the same checks, from the same
  // function.
  attn_params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.causal = causal;
  p.scale = scale;
  const int rc0 = validate(&p);
  if (rc0 != ATTN_OK) return rc0;
  // The CUDA-core partial kernels cover head dims 64 and 128.
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (num_splits < 1 || num_splits > 256) return ATTN_ERR_INVALID;
  // Sizes beyond the fixed array are refused before anything is launched.
  const size_t need = attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (need == 0) return ATTN_ERR_UNSUPPORTED;
  if (need > static_cast<size_t>(ATTN_NOALLOC_SCRATCH_BYTES)) return ATTN_ERR_WORKSPACE;
  const int64_t kMaxDim = (int64_t{1} << 31) - 1;  // grid size limit
  const int64_t BH = B * H;
  const int64_t qb = splitkv_rows_per_cta(Nq);
  if (BH * ((Nq + qb - 1) / qb) * num_splits > kMaxDim) return ATTN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;

  const size_t rows = static_cast<size_t>(BH) * num_splits * static_cast<size_t>(Nq);
  SplitArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_part = static_cast<float*>(scratch);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                        align256(rows * static_cast<size_t>(d) * 4));
  a.BH = BH;
  a.H = H;
  a.Hkv = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.query_offset = 0;
  a.keys_per_split = keys_per_split(Nk, num_splits);
  a.d = static_cast<int>(d);
  a.dv = a.d;
  a.splits = num_splits;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  if (default_status_word(&a.status) != cudaSuccess) return ATTN_ERR_CUDA;
  a.timeout_ns = 1000000000ull;
  // Always the CUDA-core partial kernels (they need no tensor maps), also
  // for shapes where attn_fwd_splitkv picks the tensor-core partial kernel.
  if (launch_splitkv_partial(a, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  if (launch_combine(a.o_part, a.lse_part, o, lse, BH, Nq, a.d, num_splits, stream) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}
