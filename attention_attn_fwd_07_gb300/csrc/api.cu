// api.cu -- the C ABI declared in include/attn.h: argument validation,
// TMA descriptor encoding, workspace layout and kernel launches.  No device
// memory is allocated here and no work runs anywhere but in this library's
// kernels.  Validation happens before any CUDA call, so argument errors are
// reported identically with or without a GPU.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "internal.cuh"

namespace attn {

// The library's own status word, one per device (used when the caller does
// not pass attn_params.dev_status).  Bit 0: some kernel gave up a wait.
__device__ int g_status_word;

cudaError_t default_status_word(int** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_status_word);
}

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;  // TMA coordinates and grid size
constexpr int64_t kMaxOffset = int64_t{1} << 40;
constexpr int kMaxSplits = 256;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [BH][N][d] viewed as a 3-D tensor (d fastest) of 2-byte (bf16) or 1-byte
// (e4m3) elements; boxes of 128 bytes x 128 rows x 1 with the 128-byte
// swizzle the MMA descriptors expect; out-of-range rows read 0.
bool encode_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* ptr,
                int64_t N, int64_t BH, int64_t d, int elem_bytes = 2) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * elem_bytes),
                           static_cast<cuuint64_t>(N * d * elem_bytes)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                   3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

bool head_dim_supported(int64_t d) { return d == 64 || d == 96 || d == 128 || d == 256; }

// Checks shared by the forward entry points (attn_fwd_ex, attn_fwd_splitkv_ex
// and attn_fwd_splitkv_noalloc).
int validate(const attn_params* p) {
  if (p == nullptr) return ATTN_ERR_INVALID;
  if (!p->q || !p->k || !p->v || !p->o || !p->lse) return ATTN_ERR_INVALID;
  if (p->B < 1 || p->H < 1 || p->Nq < 1 || p->Nk < 1) return ATTN_ERR_INVALID;
  if (!std::isfinite(p->scale) || !(p->scale > 0.0f)) return ATTN_ERR_INVALID;
  if (p->query_offset < -kMaxOffset || p->query_offset > kMaxOffset) return ATTN_ERR_INVALID;
  if (p->query_offset < 0 && !(p->flags & ATTN_FLAG_ALLOW_NEG_OFFSET)) return ATTN_ERR_INVALID;
  if (p->Hkv < 0 || p->Hkv > p->H || (p->Hkv > 0 && p->H % p->Hkv != 0)) return ATTN_ERR_INVALID;
  if (!head_dim_supported(p->d)) return ATTN_ERR_UNSUPPORTED;
  if (p->dv < 0) return ATTN_ERR_INVALID;
  // A value dim of its own: 64 or 128 with a key dim of 64 or 128; head
  // dims 96 and 256 take dv = d.
  if (p->dv != 0 && p->dv != p->d &&
      ((p->dv != 64 && p->dv != 128) || (p->d != 64 && p->d != 128)))
    return ATTN_ERR_UNSUPPORTED;
  if (p->B > kMaxDim || p->H > kMaxDim || p->B * p->H > kMaxDim || p->Nq > kMaxDim ||
      p->Nk > kMaxDim)
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->v, 16) || !aligned(p->o, 16) ||
      !aligned(p->lse, 4))
    return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

int64_t keys_per_split(int64_t Nk, int splits) {
  const int64_t per = (Nk + splits - 1) / splits;
  return (per + 127) / 128 * 128;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_ex(const attn_params* p, cudaStream_t stream) {
  int rc = validate(p);
  if (rc != ATTN_OK) return rc;
  const int64_t BH = p->B * p->H;
  const int64_t blocks = BH * ((p->Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta);
  if (blocks > kMaxDim) return ATTN_ERR_UNSUPPORTED;
  const bool fp8 = p->qk_dtype == ATTN_QK_E4M3;
  if (p->qk_dtype != ATTN_QK_BF16 && !fp8) return ATTN_ERR_INVALID;
  if (fp8) {
    if (!std::isfinite(p->q_descale) || !(p->q_descale > 0.0f) ||
        !std::isfinite(p->k_descale) || !(p->k_descale > 0.0f))
      return ATTN_ERR_INVALID;
    if (p->d != 128) return ATTN_ERR_UNSUPPORTED;
  }
  const int64_t dv = p->dv > 0 ? p->dv : p->d;

  int* status = p->dev_status;
  if (status == nullptr && default_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  const int64_t Hkv = p->Hkv > 0 ? p->Hkv : p->H;
  const int64_t BHkv = p->B * Hkv;
  CUtensorMap tq, tk, tv;
  const int qk_bytes = fp8 ? 1 : 2;
  if (!encode_map(enc, &tq, p->q, p->Nq, BH, p->d, qk_bytes) ||
      !encode_map(enc, &tk, p->k, p->Nk, BHkv, p->d, qk_bytes) ||
      !encode_map(enc, &tv, p->v, p->Nk, BHkv, dv))
    return ATTN_ERR_CUDA;

  FwdArgs a;
  a.o = p->o;
  a.lse = p->lse;
  a.status = status;
  a.BH = BH;
  a.Nq = p->Nq;
  a.Nk = p->Nk;
  a.query_offset = p->query_offset;
  a.H = p->H;
  a.group = p->H / Hkv;
  a.d = static_cast<int>(p->d);
  a.dv = static_cast<int>(dv);
  a.causal = p->causal ? 1 : 0;
  a.fp8_qk = fp8 ? 1 : 0;
  a.scale = fp8 ? static_cast<float>(static_cast<double>(p->scale) * p->q_descale * p->k_descale)
                : p->scale;
  a.flags = p->flags;
  a.timeout_ns = 1000ull * (p->wait_timeout_us ? p->wait_timeout_us : 1000000u);
  return launch_fwd_tcgen05(a, tq, tk, tv, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                        float scale, cudaStream_t stream) {
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
  return attn_fwd_ex(&p, stream);
}

namespace {

// One event per use, created without timing; destroying a recorded event
// before it completes is allowed (its resources are released afterwards).
cudaError_t record_new_event(cudaEvent_t* ev, cudaStream_t s) {
  cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  return cudaEventRecord(*ev, s);
}

}  // namespace

extern "C" int attn_fwd_from_host(const attn_params* p, const void* q_host, const void* k_host,
                                  const void* v_host, void* o_host, float* lse_host,
                                  int chunk_heads, cudaStream_t stream,
                                  cudaStream_t upload_stream, cudaStream_t download_stream) {
  int rc = validate(p);
  if (rc != ATTN_OK) return rc;
  if (!q_host || !k_host || !v_host || !o_host || !lse_host || chunk_heads < 1)
    return ATTN_ERR_INVALID;
  if (p->qk_dtype != ATTN_QK_BF16) return ATTN_ERR_UNSUPPORTED;
  const int64_t Hkv = p->Hkv > 0 ? p->Hkv : p->H;
  const int64_t G = p->H / Hkv;  // query heads per K/V head
  const int64_t dv = p->dv > 0 ? p->dv : p->d;
  // Chunks of whole K/V head groups of one batch entry: contiguous in every
  // tensor, and independent of each other.
  const int64_t hc = std::max<int64_t>(G, (std::min<int64_t>(chunk_heads, p->H) / G) * G);
  const size_t e2 = 2;  // bf16
  const size_t q_head = static_cast<size_t>(p->Nq) * p->d * e2;
  const size_t k_head = static_cast<size_t>(p->Nk) * p->d * e2;
  const size_t v_head = static_cast<size_t>(p->Nk) * dv * e2;
  const size_t o_head = static_cast<size_t>(p->Nq) * dv * e2;
  const size_t l_head = static_cast<size_t>(p->Nq) * sizeof(float);
  auto at = [](const void* base, size_t off) {
    return static_cast<const char*>(base) + off;
  };
  auto at_w = [](void* base, size_t off) { return static_cast<char*>(base) + off; };

  // The side streams start after the work already queued on `stream` (the
  // device buffers may still be in use there).
  cudaEvent_t ev = nullptr;
  if (record_new_event(&ev, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  bool fail = cudaStreamWaitEvent(upload_stream, ev, 0) != cudaSuccess ||
              cudaStreamWaitEvent(download_stream, ev, 0) != cudaSuccess;
  cudaEventDestroy(ev);
  for (int64_t b = 0; b < p->B && !fail; ++b) {
    for (int64_t h0 = 0; h0 < p->H && !fail; h0 += hc) {
      const int64_t h1 = std::min(p->H, h0 + hc);
      const int64_t g0 = h0 / G, g1 = (h1 + G - 1) / G;
      const size_t qo = static_cast<size_t>(b * p->H + h0) * q_head;
      const size_t ko = static_cast<size_t>(b * Hkv + g0) * k_head;
      const size_t vo = static_cast<size_t>(b * Hkv + g0) * v_head;
      const size_t oo = static_cast<size_t>(b * p->H + h0) * o_head;
      const size_t lo = static_cast<size_t>(b * p->H + h0) * l_head;
      const size_t nh = static_cast<size_t>(h1 - h0), nkv = static_cast<size_t>(g1 - g0);
      // Upload the chunk, then compute it on `stream` once it has landed.
      fail = cudaMemcpyAsync(at_w(const_cast<void*>(p->q), qo), at(q_host, qo), nh * q_head,
                             cudaMemcpyHostToDevice, upload_stream) != cudaSuccess ||
             cudaMemcpyAsync(at_w(const_cast<void*>(p->k), ko), at(k_host, ko), nkv * k_head,
                             cudaMemcpyHostToDevice, upload_stream) != cudaSuccess ||
             cudaMemcpyAsync(at_w(const_cast<void*>(p->v), vo), at(v_host, vo), nkv * v_head,
                             cudaMemcpyHostToDevice, upload_stream) != cudaSuccess;
      if (fail) break;
      fail = record_new_event(&ev, upload_stream) != cudaSuccess ||
             cudaStreamWaitEvent(stream, ev, 0) != cudaSuccess;
      cudaEventDestroy(ev);
      if (fail) break;
      attn_params c = *p;
      c.q = at(p->q, qo);
      c.k = at(p->k, ko);
      c.v = at(p->v, vo);
      c.o = at_w(p->o, oo);
      c.lse = reinterpret_cast<float*>(at_w(p->lse, lo));
      c.B = 1;
      c.H = h1 - h0;
      c.Hkv = p->Hkv > 0 ? g1 - g0 : 0;
      rc = attn_fwd_ex(&c, stream);
      if (rc != ATTN_OK) return rc;
      // Download the chunk's O and LSE once it is computed.
      fail = record_new_event(&ev, stream) != cudaSuccess ||
             cudaStreamWaitEvent(download_stream, ev, 0) != cudaSuccess;
      cudaEventDestroy(ev);
      if (fail) break;
      fail = cudaMemcpyAsync(at_w(o_host, oo), at(p->o, oo), nh * o_head,
                             cudaMemcpyDeviceToHost, download_stream) != cudaSuccess ||
             cudaMemcpyAsync(at_w(lse_host, lo), at(p->lse, lo), nh * l_head,
                             cudaMemcpyDeviceToHost, download_stream) != cudaSuccess;
    }
  }
  // `stream` waits for the last download: the host buffers are complete
  // once `stream` is.
  if (record_new_event(&ev, download_stream) != cudaSuccess) return ATTN_ERR_CUDA;
  const bool joined = cudaStreamWaitEvent(stream, ev, 0) == cudaSuccess;
  cudaEventDestroy(ev);
  return fail || !joined ? ATTN_ERR_CUDA : ATTN_OK;
}

extern "C" size_t attn_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t d,
                                               int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || !head_dim_supported(d)) return 0;
  if (num_splits < 1 || num_splits > kMaxSplits) return 0;
  if (B > kMaxDim || H > kMaxDim || Nq > kMaxDim || B * H > kMaxDim) return 0;
  const unsigned __int128 rows =
      static_cast<unsigned __int128>(B * H) * static_cast<unsigned>(num_splits) *
      static_cast<uint64_t>(Nq);
  const unsigned __int128 bytes = rows * static_cast<uint64_t>(d) * 4u + 256u + rows * 4u;
  if (bytes > (static_cast<unsigned __int128>(1) << 62)) return 0;
  const size_t r = static_cast<size_t>(rows);
  return align256(r * static_cast<size_t>(d) * 4) + r * 4;
}

extern "C" int attn_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                            int64_t B, int64_t H, int64_t Nq, int64_t d, int num_splits,
                            cudaStream_t stream) {
  if (!o_part || !lse_part || !o || !lse) return ATTN_ERR_INVALID;
  if (B < 1 || H < 1 || Nq < 1 || num_splits < 1 || num_splits > kMaxSplits)
    return ATTN_ERR_INVALID;
  if (!head_dim_supported(d)) return ATTN_ERR_UNSUPPORTED;
  if (B > kMaxDim || H > kMaxDim || Nq > kMaxDim || B * H > kMaxDim ||
      (B * H * Nq + 7) / 8 > kMaxDim)
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  return launch_combine(o_part, lse_part, o, lse, B * H, Nq, static_cast<int>(d), num_splits,
                        stream) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

extern "C" int attn_fwd_splitkv_ex(const attn_params* p, int num_splits, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  int rc = validate(p);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID;
  if (p->qk_dtype != ATTN_QK_BF16) return ATTN_ERR_UNSUPPORTED;
  const int64_t dv = p->dv > 0 ? p->dv : p->d;  // width of V, O and the partials
  const size_t need = attn_splitkv_workspace_bytes(p->B, p->H, p->Nq, dv, num_splits);
  if (need == 0) return ATTN_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return ATTN_ERR_ALIGN;
  const int64_t BH = p->B * p->H;
  const int64_t Hkv = p->Hkv > 0 ? p->Hkv : p->H;
  const int64_t rows = (p->H / Hkv) * p->Nq;  // query rows sharing one K/V head
  // Several rows per K/V head (and dv = d): the tensor-core partial kernel,
  // one CTA per block of up to 128 rows.  dv != d: the register-streaming
  // kernel, one query row per CTA.  Otherwise the CUDA-core kernels.
  // Head dims 96 and 256 always run on the tensor cores (the CUDA-core
  // kernels' lane layouts cover 64 and 128 only).
  const int64_t tc_min_rows = p->d == 128  ? ATTN_SPLITKV_TC_MIN_ROWS_D128
                              : p->d == 64 ? ATTN_SPLITKV_TC_MIN_ROWS_D64
                                           : 1;
  const bool tc = dv == p->d && rows >= tc_min_rows;
  const int64_t qb = tc ? 128 : (dv != p->d ? 1 : splitkv_rows_per_cta(rows));
  if (p->B * Hkv * ((rows + qb - 1) / qb) * num_splits > kMaxDim) return ATTN_ERR_UNSUPPORTED;
  if (tc && p->B * p->H * p->Nq > kMaxDim) return ATTN_ERR_UNSUPPORTED;

  const size_t part_rows = static_cast<size_t>(BH) * num_splits * static_cast<size_t>(p->Nq);
  SplitArgs a;
  a.q = p->q;
  a.k = p->k;
  a.v = p->v;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        align256(part_rows * static_cast<size_t>(dv) * 4));
  a.BH = BH;
  a.H = p->H;
  a.Hkv = Hkv;
  a.Nq = p->Nq;
  a.Nk = p->Nk;
  a.query_offset = p->query_offset;
  a.keys_per_split = keys_per_split(p->Nk, num_splits);
  a.d = static_cast<int>(p->d);
  a.dv = static_cast<int>(dv);
  a.splits = num_splits;
  a.causal = p->causal ? 1 : 0;
  a.scale = p->scale;
  a.status = p->dev_status;
  if (a.status == nullptr && default_status_word(&a.status) != cudaSuccess) return ATTN_ERR_CUDA;
  a.timeout_ns = 1000ull * (p->wait_timeout_us ? p->wait_timeout_us : 1000000u);
  if (tc) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return ATTN_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!encode_map(enc, &tq, p->q, BH * p->Nq, 1, p->d) ||
        !encode_map(enc, &tk, p->k, p->Nk, p->B * Hkv, p->d) ||
        !encode_map(enc, &tv, p->v, p->Nk, p->B * Hkv, p->d))
      return ATTN_ERR_CUDA;
    if (launch_splitkv_partial_tc(a, tq, tk, tv, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  } else if (launch_splitkv_partial(a, stream) != cudaSuccess) {
    return ATTN_ERR_CUDA;
  }
  if (launch_combine(a.o_part, a.lse_part, p->o, p->lse, BH, p->Nq, a.dv, num_splits, stream) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                                int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                                int causal, float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
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
  return attn_fwd_splitkv_ex(&p, num_splits, workspace, workspace_bytes, stream);
}

extern "C" size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq) {
  if (B < 1 || H < 1 || Nq < 1 || B > kMaxDim || H > kMaxDim || Nq > kMaxDim ||
      B * H > kMaxDim)
    return 0;
  return align256(static_cast<size_t>(B * H) * static_cast<size_t>(Nq) * 4);
}

extern "C" int attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (p == nullptr) return ATTN_ERR_INVALID;
  if (!p->q || !p->k || !p->v || !p->o || !p->dout || !p->lse || !p->dq || !p->dk || !p->dv)
    return ATTN_ERR_INVALID;
  if (p->B < 1 || p->H < 1 || p->Nq < 1 || p->Nk < 1) return ATTN_ERR_INVALID;
  if (!std::isfinite(p->scale) || !(p->scale > 0.0f)) return ATTN_ERR_INVALID;
  if (p->query_offset < -kMaxOffset || p->query_offset > kMaxOffset) return ATTN_ERR_INVALID;
  if (p->query_offset < 0 && !(p->flags & ATTN_FLAG_ALLOW_NEG_OFFSET)) return ATTN_ERR_INVALID;
  if (p->Hkv < 0 || p->Hkv > p->H || (p->Hkv > 0 && p->H % p->Hkv != 0)) return ATTN_ERR_INVALID;
  if (p->d != 64 && p->d != 96 && p->d != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->value_dim < 0) return ATTN_ERR_INVALID;
  const int64_t dv = p->value_dim > 0 ? p->value_dim : p->d;
  // d and dv in {64, 128} in any pair; 96 with 96 only.
  if ((p->d == 96) != (dv == 96) || (dv != 64 && dv != 96 && dv != 128))
    return ATTN_ERR_UNSUPPORTED;
  if (p->B > kMaxDim || p->H > kMaxDim || p->B * p->H > kMaxDim || p->Nq > kMaxDim ||
      p->Nk > kMaxDim)
    return ATTN_ERR_UNSUPPORTED;
  const void* ptrs16[] = {p->q, p->k, p->v, p->o, p->dout, p->dq, p->dk, p->dv};
  for (const void* ptr : ptrs16)
    if (!aligned(ptr, 16)) return ATTN_ERR_ALIGN;
  if (!aligned(p->lse, 4)) return ATTN_ERR_ALIGN;
  const size_t need = attn_bwd_workspace_bytes(p->B, p->H, p->Nq);
  if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return ATTN_ERR_ALIGN;
  const int64_t Hkv = p->Hkv > 0 ? p->Hkv : p->H;
  const int64_t BH = p->B * p->H, BHkv = p->B * Hkv;
  if (BHkv * ((p->Nk + 127) / 128) > kMaxDim || BH * ((p->Nq + 127) / 128) > kMaxDim)
    return ATTN_ERR_UNSUPPORTED;

  int* status = p->dev_status;
  if (status == nullptr && default_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_map(enc, &tq, p->q, p->Nq, BH, p->d) ||
      !encode_map(enc, &tdo, p->dout, p->Nq, BH, dv) ||
      !encode_map(enc, &tk, p->k, p->Nk, BHkv, p->d) ||
      !encode_map(enc, &tv, p->v, p->Nk, BHkv, dv))
    return ATTN_ERR_CUDA;
  BwdArgs a;
  a.o = p->o;
  a.dout = p->dout;
  a.lse = p->lse;
  a.delta = static_cast<float*>(workspace);
  a.dq = p->dq;
  a.dk = p->dk;
  a.dv = p->dv;
  a.status = status;
  a.B = p->B;
  a.H = p->H;
  a.Hkv = Hkv;
  a.Nq = p->Nq;
  a.Nk = p->Nk;
  a.query_offset = p->query_offset;
  a.causal = p->causal ? 1 : 0;
  a.scale = p->scale;
  a.timeout_ns = 1000ull * (p->wait_timeout_us ? p->wait_timeout_us : 1000000u);
  cudaError_t err;
  if (p->d == 96)
    err = launch_bwd<96, 96>(a, tq, tk, tv, tdo, stream);
  else if (p->d == 64)
    err = dv == 64 ? launch_bwd<64, 64>(a, tq, tk, tv, tdo, stream)
                   : launch_bwd<64, 128>(a, tq, tk, tv, tdo, stream);
  else
    err = dv == 64 ? launch_bwd<128, 64>(a, tq, tk, tv, tdo, stream)
                   : launch_bwd<128, 128>(a, tq, tk, tv, tdo, stream);
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_get_device_status(int* dev_status_host, cudaStream_t stream) {
  if (dev_status_host == nullptr) return ATTN_ERR_INVALID;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int* word = nullptr;
  if (default_status_word(&word) != cudaSuccess) return ATTN_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return ATTN_ERR_CUDA;
  *dev_status_host = value;
  return ATTN_OK;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported head dim or size";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: misaligned pointer";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT: a kernel gave up a wait";
    default: return "unknown attn status";
  }
}
