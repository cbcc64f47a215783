/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * Operation (all entry points): for every batch b, head h and query row i,
 *
 *   s_j  = scale * <q[b,h,i,:], k[b,h,j,:]>                 j = 0 .. Nk-1
 *   s_j  = -inf  when causal and j > i + query_offset
 *   o[b,h,i,:] = sum_j softmax(s)_j * v[b,h,j,:]
 *   lse[b,h,i] = ln sum_j exp(s_j)                           (natural log)
 *
 * computed tile by tile with the online-softmax recurrence (running maximum
 * m, normaliser l and unnormalised accumulator o, old state rescaled by
 * exp(m - m_new)), so the Nq x Nk score matrix never reaches device memory.
 * Definitions follow "GPU Engineering: Correctness, Throughput, and
 * Attention": section 22.5 (the recurrence and its rescaling; causal masking
 * before maxima and sums; fully masked rows need explicit semantics) and
 * section 22.7 (the worked lab: scores scaled after the dot product; key j
 * excluded when j > i + query_offset; a row with no admissible key has output
 * 0 and log-normaliser -inf; the log-normaliser is m + ln(l)).  The split-KV
 * merge is the same rescaling applied to whole partial states.
 *
 * Conventions shared by every entry point
 *  - Q, K, V, O are bfloat16, contiguous [B][H][N][d] (N = Nq for Q and O,
 *    Nk for K and V); each (b,h) slice is a row-major [N][d] matrix.  LSE is
 *    float32 [B][H][Nq].  All tensor pointers are DEVICE pointers owned by the
 *    caller; the library keeps no pointer after a call returns.
 *  - Q, K, V, O and workspaces must be 16-byte aligned; LSE 4-byte aligned.
 *  - Head dims: d in {64, 96, 128, 256} for the forward entry points (the
 *    lab of "GPU Engineering" section 22.5 asks for several head
 *    dimensions); 96 and 256 take dv = d; the backward and
 *    attn_fwd_splitkv_noalloc take 64 and 128 (ATTN_ERR_UNSUPPORTED
 *    otherwise).
 *  - B, H, Nq, Nk >= 1 (ATTN_ERR_INVALID otherwise); scale must be finite
 *    and > 0.  Inputs must be finite (a documented precondition, not checked:
 *    a check would cost a full pass over the data).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *    return value reports argument validation and launch errors only.  Device
 *    side wait timeouts are reported through attn_get_device_status().
 *  - Rows >= Nq of O/LSE and any byte outside [B,H,Nq,d] / [B,H,Nq] are never
 *    written.  A fully masked row is written as O = +0.0, LSE = -inf.
 *  - No entry point allocates device memory; the split-KV workspace is the
 *    caller's.  Entry points are thread-safe.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point (0 = success). */
typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = -1,        /* null pointer, size < 1, bad scale, ...   */
  ATTN_ERR_UNSUPPORTED = -2,    /* head dim not supported, size limits      */
  ATTN_ERR_ALIGN = -3,          /* pointer misaligned                       */
  ATTN_ERR_WORKSPACE = -4,      /* split-KV workspace missing or too small  */
  ATTN_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed        */
  ATTN_ERR_DEVICE_TIMEOUT = -6  /* a kernel gave up a bounded wait          */
} attn_status;

/* attn_params.flags */
enum {
  /* Accept query_offset < 0 so that leading rows see no key at all (fully
   * masked rows).  The pages require query_offset >= 0; this flag exists to
   * exercise the fully-masked-row policy. */
  ATTN_FLAG_ALLOW_NEG_OFFSET = 1u << 0,
  /* Fault injection for the timeout path: the prefill kernel's loader skips
   * one K/V tile load so that its consumers' bounded waits expire.  The
   * kernel then records ATTN_ERR_DEVICE_TIMEOUT and returns; no GPU fault. */
  ATTN_FLAG_TEST_SKIP_LOAD = 1u << 1
};

/* Full argument set of the prefill entry point (attn_fwd_ex) and of the
 * split-KV entry point (attn_fwd_splitkv_ex).  Grouped K/V heads (GQA/MQA,
 * among FlashAttention's production features in "GPU Kernels: CUDA, HIP &
 * Triton", section 7.6) are available through these two entry points, and
 * so is FP8 Q K^T (the same section's FP8 mode) for the prefill kernel. */
typedef struct attn_params {
  const void* q;          /* bf16 [B][H][Nq][d], device                    */
  const void* k;          /* bf16 [B][Hkv][Nk][d], device                  */
  const void* v;          /* bf16 [B][Hkv][Nk][dv], device                 */
  void* o;                /* bf16 [B][H][Nq][dv], device, written          */
  float* lse;             /* f32  [B][H][Nq],    device, written           */
  int64_t B, H, Nq, Nk, d;
  int causal;             /* nonzero: key j visible to row i iff j <= i + query_offset */
  float scale;            /* multiplies q.k before masking; finite, > 0    */
  int64_t query_offset;   /* absolute position of query row 0; >= 0        */
  int* dev_status;        /* optional device int; timeouts are OR-ed into it
                             as bit 0; NULL = the library's own status word */
  uint32_t flags;         /* ATTN_FLAG_* */
  uint32_t wait_timeout_us; /* per-wait device timeout; 0 = 1,000,000 us   */
  int64_t Hkv;            /* K/V heads (grouped-query / multi-query attention):
                             K and V are [B][Hkv][Nk][d] and query head h reads
                             K/V head h / (H / Hkv); H % Hkv == 0.  0 = H.  */
  int qk_dtype;           /* ATTN_QK_BF16 (0) or ATTN_QK_E4M3 (prefill only,
                             d = 128): Q and K are FP8 e4m3 (1 byte each) and
                             the scores are scale * q_descale * k_descale *
                             <q, k>; V stays bf16.                          */
  float q_descale;        /* per-tensor factors of the FP8 Q and K; finite, */
  float k_descale;        /* > 0 (ignored for bf16)                         */
  int64_t dv;             /* head dim of V and O; 0 = d.  dv may differ from d
                             in attn_fwd_ex (d and dv in {64, 128}; FP8: d =
                             128, dv in {64, 128}) and attn_fwd_splitkv_ex
                             (bf16, d and dv in {64, 128}); head dims 96 and
                             256, and every other entry point, need dv = d
                             (ATTN_ERR_UNSUPPORTED otherwise).              */
} attn_params;

/* attn_params.qk_dtype */
enum { ATTN_QK_BF16 = 0, ATTN_QK_E4M3 = 1 };

/*
 * Prefill / general forward: O and LSE for all rows, query_offset = 0.
 * tcgen05 (TMEM accumulators) + TMA kernels; any Nq, Nk >= 1; d in
 * {64, 96, 128, 256}.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
             int causal, float scale, cudaStream_t stream);

/* attn_fwd with every option (query_offset, flags, status word, timeout). */
int attn_fwd_ex(const attn_params* p, cudaStream_t stream);

/*
 * End-to-end forward from host memory: copies Q, K and V from the host
 * buffers into the device buffers of `p` (p->q, p->k, p->v, which must not
 * be in use by other work), computes O and LSE into p->o and p->lse as
 * attn_fwd_ex does, and copies them back into o_host and lse_host.  The
 * work is cut into chunks of whole K/V head groups (chunk_heads query heads,
 * rounded to whole groups) of one batch entry -- every (b, h) slice is
 * independent -- and the chunks are pipelined over three caller-owned
 * streams: uploads on upload_stream, the kernels on `stream` once their
 * chunk has landed, downloads on download_stream once it is computed; the
 * side streams first wait for the work already queued on `stream`, and
 * `stream` waits for the last download before this returns, so the host
 * buffers hold the result once `stream` has completed.  Host buffers should
 * be page-locked for the copies to overlap.  Layouts as in attn_params
 * (bf16 Q, K, V, O; f32 LSE; same shapes on host and device).  Nothing is
 * allocated on the device; the call creates and releases timing-free events
 * (two per chunk, two more per call).  Returns the argument checks of attn_fwd_ex, ATTN_ERR_INVALID for a
 * null host pointer or chunk_heads < 1, ATTN_ERR_UNSUPPORTED for FP8 Q/K, and
 * ATTN_ERR_CUDA if a copy, event or launch fails.
 */
int attn_fwd_from_host(const attn_params* p, const void* q_host, const void* k_host,
                       const void* v_host, void* o_host, float* lse_host, int chunk_heads,
                       cudaStream_t stream, cudaStream_t upload_stream,
                       cudaStream_t download_stream);

/*
 * Bytes of workspace attn_fwd_splitkv needs: float32 partial outputs
 * [B][H][num_splits][Nq][d] followed (at a 256-byte boundary) by float32
 * partial log-sum-exps [B][H][num_splits][Nq].  `d` is the width of the
 * partials, i.e. the head dim of V and O (dv when attn_fwd_splitkv_ex is
 * given dv != d).  Returns 0 for invalid sizes.
 */
size_t attn_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t d,
                                    int num_splits);

/*
 * Split-KV forward for short queries (decode): the keys of every (b,h) are
 * cut into num_splits contiguous ranges of L = ceil(Nk/num_splits) keys
 * rounded up to a multiple of 128 (trailing ranges may be empty); each range
 * yields a partial (normalised o, lse) in `workspace`, then attn_combine
 * merges them into O and LSE.  When several query rows share a K/V head
 * (grouped K/V heads through attn_fwd_splitkv_ex, or Nq > 1) they are served
 * together -- up to 128 rows per CTA on the tensor cores, or in blocks of
 * four on the CUDA cores at d = 64 with at most four rows -- so each K/V byte
 * is read about once per group; head dims 96 and 256 always run on the
 * tensor cores, one row per K/V head included.  1 <= num_splits <= 256.  Two launches on
 * `stream`; `workspace` (device, 16-byte aligned, caller-owned) must hold
 * attn_splitkv_workspace_bytes(...) bytes (ATTN_ERR_WORKSPACE otherwise).
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                     int causal, float scale, int num_splits, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/* attn_fwd_splitkv with query_offset, Hkv, dv, flags, dev_status and
 * wait_timeout_us from `p` (the latter two apply to the partial kernels
 * used when several query rows share a K/V head; ATTN_FLAG_TEST_SKIP_LOAD
 * applies to the prefill kernel only).  With dv != d every query row gets
 * its own partial CTAs, so a K/V head shared by several rows is read once
 * per row; the workspace holds dv-wide partials. */
int attn_fwd_splitkv_ex(const attn_params* p, int num_splits, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/*
 * Log-sum-exp merge of num_splits partial states per row:
 *   M = max_s lse_part[s];  if M = -inf: O = +0.0, LSE = -inf;  otherwise
 *   w_s = exp(lse_part[s] - M),  LSE = M + ln sum_s w_s,
 *   O = sum_s (w_s / sum_s w_s) * o_part[s]   (rounded to bf16).
 * o_part: f32 [B][H][num_splits][Nq][d], lse_part: f32 [B][H][num_splits][Nq]
 * (device, 16-byte aligned); o: bf16 [B][H][Nq][d]; lse: f32 [B][H][Nq].
 * 1 <= num_splits <= 256.
 */
int attn_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                 int64_t B, int64_t H, int64_t Nq, int64_t d, int num_splits,
                 cudaStream_t stream);

/* Arguments of the backward pass (attn_bwd). */
typedef struct attn_bwd_params {
  const void* q;          /* bf16 [B][H][Nq][d], the forward's inputs         */
  const void* k;          /* bf16 [B][Hkv][Nk][d]                             */
  const void* v;          /* bf16 [B][Hkv][Nk][dv]                            */
  const void* o;          /* bf16 [B][H][Nq][dv], the forward's output        */
  const void* dout;       /* bf16 [B][H][Nq][dv], loss gradient on O          */
  const float* lse;       /* f32  [B][H][Nq], the forward's log-sum-exp       */
  void* dq;               /* bf16 [B][H][Nq][d], written                      */
  void* dk;               /* bf16 [B][Hkv][Nk][d], written                    */
  void* dv;               /* bf16 [B][Hkv][Nk][dv], written                   */
  int64_t B, H, Hkv, Nq, Nk, d;  /* Hkv = 0 means H; d is 64 or 128          */
  int causal;
  float scale;
  int64_t query_offset;
  int* dev_status;        /* as in attn_params; bit 1 is set (and nothing is
                             computed) if a kernel finds its shared memory
                             not 1024-byte aligned                          */
  uint32_t flags;         /* ATTN_FLAG_ALLOW_NEG_OFFSET only                  */
  uint32_t wait_timeout_us;
  int64_t value_dim;      /* dv, the head dim of V, O, dO and dV: 64 or 128;
                             0 = d                                          */
} attn_bwd_params;

/* Bytes of workspace attn_bwd needs: f32 [B][H][Nq] (the row corrections
 * rowsum(dO * O)).  Returns 0 for invalid sizes. */
size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq);

/*
 * Gradients of the forward above for the loss gradient dout on O
 * ("GPU Engineering: Correctness, Throughput, and Attention", sections 22.5
 * and 22.7): dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)),
 * dQ = scale * dS K, dK = scale * dS^T Q, with P recomputed tile by tile
 * from `lse` (never stored).  Rows with no admissible key get zero dQ; keys no
 * row can see get zero dK and dV.  Grouped K/V heads sum their group's
 * contributions.  Three launches on `stream` (row corrections, a dK/dV kernel
 * per 128-key tile, a dQ kernel per 128-query tile); no atomics, so the
 * result is deterministic.  d and dv in {64, 128} (dv may differ from d), or
 * d = dv = 96; ATTN_ERR_UNSUPPORTED otherwise (head dim 256 has no
 * backward).
 * `workspace` (device, 16-byte aligned, caller-owned) must hold
 * attn_bwd_workspace_bytes(B, H, Nq) bytes.
 */
int attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
             cudaStream_t stream);

/* Size of the library-owned scratch array used by attn_fwd_splitkv_noalloc
 * (one per GPU that loads the library, kept until the process exits). */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * attn_fwd_splitkv without a caller-provided workspace, for callers that
 * cannot allocate device memory: code whose device memory is all planned by
 * an outer arena that forbids further allocation, plug-ins whose host
 * program offers no allocator, or latency-critical loops that cannot afford
 * the device synchronisation cudaMalloc/cudaFree may cause.  The pages have
 * no counterpart to this entry point; it is a deployment convenience.
 *
 * Same arguments, argument checks and results as attn_fwd_splitkv
 * (query_offset 0), with one difference in how the partials are computed:
 * this entry point always runs the CUDA-core partial kernels, also for
 * shapes where attn_fwd_splitkv switches to the tensor-core partial kernel
 * (several query rows per head).  There the two agree within the library's
 * tolerances but may differ in the last bits, and this one is slower.
 * The scratch lives in a fixed device array of ATTN_NOALLOC_SCRATCH_BYTES
 * inside the library; calls whose attn_splitkv_workspace_bytes(...) exceed it
 * return ATTN_ERR_WORKSPACE before launching anything.  Nothing is allocated.
 * Every call looks up the array's device address on the current device (a
 * host-side lookup; the first one on a device may load the library's module
 * there), so make the first call on each device before any stream capture.
 * All calls share the array: calls that overlap on the GPU (other streams or
 * host threads on the same device) race and must be serialised by the
 * caller.  The array keeps the previous call's contents; no call needs it
 * cleared.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                             int causal, float scale, int num_splits, cudaStream_t stream);

/*
 * Synchronises `stream`, copies the library's own device status word (the
 * one kernels use when attn_params.dev_status is NULL) on the current device
 * to *dev_status_host, and clears it.  Bit 0 set = some kernel gave up a
 * bounded wait (ATTN_ERR_DEVICE_TIMEOUT); its outputs are undefined.
 */
int attn_get_device_status(int* dev_status_host, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
