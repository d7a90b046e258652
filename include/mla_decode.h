/*
 * libmla_decode — decode step of DeepSeek-R1-style Multi-head Latent Attention
 * (forward_absorb path) over an FP8 per-tensor-scaled latent cache, for sm_103a.
 *
 * What one call computes (kernelbot-amd-mixed-mla submission 738050, comment
 * block above its mla_decode_fwd call; constants of submission 663509):
 *
 *     out[t, h, :] = softmax_j( q[t, h, :] . K[j, :] / sqrt(576) ) @ V[j, :]
 *
 * for every batch row b with its single query token t = qo_indptr[b], over the
 * cached tokens j of that row.  q has 16 heads of 576 dims (512 latent + 64
 * rope); the one shared KV head stores 576 e4m3fn codes per token with a single
 * float32 scale (value = code * scale); K is all 576 dims of a cache row and V
 * its first 512.  The output is bf16 [T, 16, 512].  The *_bf16kv entry points
 * compute the same step over a bf16 cache (the values themselves, no scale).
 *
 * All pointers named "device" are CUDA device pointers; every buffer is owned
 * and allocated by the caller.  The library never allocates, frees or
 * synchronises on the forward path: all work is ordered on `stream`.
 * Functions return MLA_OK or an mla_status_t describing a host-detected error,
 * in which case nothing was launched.  Errors that need the data to detect are
 * recorded as bits in the workspace error word (MLA_DERR_*), readable with
 * mla_decode_read_error.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 16
#define MLA_QK_HEAD_DIM 576
#define MLA_V_HEAD_DIM 512
#define MLA_TILE_TOKENS 128
#define MLA_ABI_VERSION 5

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,         /* null / misaligned pointer, bad size, plan mismatch  */
  MLA_ERR_UNSUPPORTED = 2,         /* device is not sm_103 / lacks the shared memory      */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < plan->ws_bytes                    */
  MLA_ERR_CUDA = 4                 /* a CUDA runtime or driver call failed                */
} mla_status_t;

/* Bits of the device-side error word (sticky until cleared). */
#define MLA_DERR_QO_INDPTR 1  /* a row does not hold exactly plan->qo_len query tokens in range */
#define MLA_DERR_KV_INDPTR 2  /* kv_indptr decreases, or its end exceeds kv_rows / kv_indices_len */
#define MLA_DERR_KV_INDEX 4   /* a page-table entry lies outside [0, kv_rows)                */
#define MLA_DERR_TIMEOUT 8    /* a pipeline wait ran past its time limit; the call gave up  */
#define MLA_DERR_MX_SCALE 16  /* MXFP4 cache: a block holding a nonzero element has a scale
                                 outside the exact window of mla_decode_fwd_mxfp4 (or NaN)  */
#define MLA_DERR_DEBUG_BOUNDS 32 /* debug builds only: an index failed its bounds check and the
                                    access was skipped (never set by release builds)        */

/*
 * Launch plan for a batch shape.  The split-KV schedule (flash-decoding split,
 * submission 722089 `_mla_multihead_stage1`; the persistent work maps of
 * submissions 663509 and 738050) is fixed analytically here: rows are cut into
 * tiles of 128 tokens; the rows form one sequence of T units, each row with
 * tiles contributing S start units and then its tiles, and `grid` persistent
 * workers take equal contiguous ranges of it.  S = 3 when the batch's N tiles
 * give ranges of at least 8 tiles (ceil(N / grid) >= 8), else 0: a worker
 * whose range takes on a row start also prepares that row's query and writes
 * the previous segment's output, and gets S fewer tiles for it.  (A bf16 cache,
 * whose tiles take twice as long, uses S = 0.)  A row covered
 * by more than one worker is combined by the second stage.
 *
 * Small batches instead take the cluster split (`cluster` = s > 0): row b is
 * shared by a thread-block cluster of s CTAs, the CTA of rank r taking the
 * row's tiles [r k, min((r + 1) k, nt)) with nt = ceil(L_b / 128) and
 * k = ceil(nt / s); each CTA writes its partial result to the workspace, the
 * cluster meets at one barrier, and its CTAs then combine the row's s partials
 * (read back through L2) into the output, each CTA a slice of it: no second
 * kernel runs.  The plan
 * chooses s as the largest of 8, 4, 2 with s <= ceil(max_kv_len / 128) whose
 * clusters for the whole batch fit the GPU at once (at most num_sms / 10
 * clusters of 8, 7 num_sms / 32 of 4, num_sms / 2 of 2), and only when its
 * longest share ceil(ceil(max_kv_len / 128) / s) is at most two tiles longer
 * than the persistent split's longest range; rows of one query token only.
 * The cluster split serves the contiguous e4m3 and bf16 caches; with a page
 * table or an MXFP4 cache the same plan runs the persistent split.  A caller
 * may set `cluster` to 0 to force the persistent split.
 */
typedef struct {
  int32_t batch;       /* B, rows (one query token each)                          */
  int32_t max_kv_len;  /* upper bound on any row's cached tokens (sizes the grid)  */
  int32_t num_sms;     /* SMs the grid is sized for                               */
  int32_t grid;        /* persistent stage-1 workers: with U = B*ceil(max_kv_len/128) and
                        * S = num_sms (num_sms/2 for qo_len >= 3: two CTAs per worker),
                        * k = ceil(U / min(S, U)) tiles for the longest range and
                        * grid = max(1, ceil(U / k)): the fewest workers that keep it */
  int32_t tile_tokens; /* 128                                                      */
  int32_t abi_version; /* MLA_ABI_VERSION                                          */
  int32_t qo_len;      /* query tokens per row: 1 (decode) to 4 (multi-token decode) */
  int32_t cluster;     /* CTAs per row of the cluster split (2, 4 or 8), or 0: the
                        * persistent split (see above)                            */
  uint64_t ws_bytes;   /* workspace bytes mla_decode_fwd needs                      */
  uint64_t ws_prefix_offset;  /* int32[B+1]   tile prefix over rows                 */
  uint64_t ws_workers_offset; /* int32[grid*8] per worker: (t0, t1, first_row, last_row)
                               * then the combine job of the split row whose first
                               * worker boundary is t0: (output row or -1, first
                               * worker, last worker, first worker's partial slot) */
  uint64_t ws_lse_offset;     /* float[2*grid*qo_len*16] base-2 log-sum-exp of partials */
  uint64_t ws_partial_offset; /* bf16[2*grid*qo_len*16*512] normalised split partials,
                               * stored [slot][token][dim/128][head/8][dim%128][head%8] */
} mla_plan_t;

/*
 * mla_decode_plan — pure host function, re-entrant.
 *   batch >= 1, max_kv_len >= 0.  num_sms > 0 sizes the grid for that many SMs;
 *   num_sms <= 0 queries the current device's SM count.
 *   Fills *plan.  Returns MLA_ERR_INVALID_ARG for bad sizes / null plan.
 */
mla_status_t mla_decode_plan(int32_t batch, int32_t max_kv_len, int32_t num_sms, mla_plan_t* plan);

/*
 * mla_decode_plan_mtp — as mla_decode_plan, for rows of qo_len query tokens
 * (multi-token decode, e.g. speculative / multi-token-prediction draft tokens:
 * qo_len = 2 to 4).  qo_indptr[b+1] - qo_indptr[b] must then be qo_len for
 * every row; q is [B*qo_len, 16, 576] and out [B*qo_len, 16, 512].  Query token
 * i of a row with L cached tokens attends to the row's first L - qo_len + 1 + i
 * tokens (its own entry and those before it: the row's last qo_len cached
 * tokens are the query tokens'); a token that sees none outputs zeros.  A
 * stage-1 CTA loads each KV tile once for up to two query tokens x 16 heads;
 * rows of three or four tokens are shared by two sibling CTAs per worker
 * (tokens 0-1 and 2-3), which stream the same tiles at the same time, so the
 * second one's copies mostly come from L2.  qo_len must be 1 to 4.
 */
mla_status_t mla_decode_plan_mtp(int32_t batch, int32_t qo_len, int32_t max_kv_len, int32_t num_sms,
                                 mla_plan_t* plan);


/*
 * mla_decode_fwd — the decode step: stage 1 (split attention) then stage 2
 * (log-sum-exp combine of split rows), both on `stream`.
 *   q_bf16     device, bf16 [B, 16, 576] row-major, 16-byte aligned.
 *   kv_fp8     device, e4m3fn codes [kv_rows, 576] (= [kv_rows, 1, 576]), 16-byte aligned.
 *              Codes must be finite (0x7F / 0xFF never appear).
 *   kv_scale   device, float[1]; a code's value is code * (*kv_scale).
 *   qo_indptr  device, int32 [B+1]; row b's query token is qo_indptr[b], and
 *              qo_indptr[b+1] - qo_indptr[b] must be 1 (decode, qseqlen 1).
 *   kv_indptr  device, int32 [B+1], non-decreasing; row b owns the flattened
 *              tokens [kv_indptr[b], kv_indptr[b+1]).  A row with no token
 *              yields an all-zero output row.
 *   out_bf16   device, bf16 [B, 16, 512], 16-byte aligned.  Fully overwritten.
 *   stream     CUDA stream (0 = legacy default stream).
 *   plan       from mla_decode_plan for this batch size.
 *   kv_indices device int32 page table (page size 1): flattened token j lives in
 *              cache row kv_indices[j].  NULL means row j (identity).
 *   kv_indices_len  entries in kv_indices (ignored when it is NULL).
 *   kv_rows    rows in the cache pool kv_fp8 (>= 1).
 *   workspace  device scratch of at least plan->ws_bytes, 256-byte aligned.
 *              Zero it once after allocating (mla_decode_workspace_init) so the
 *              error word starts clear.  Calls sharing a workspace must not
 *              overlap on the GPU.
 * Output is deterministic for a given plan.  Returns MLA_OK after launching.
 * Calls with their own workspaces may run concurrently on different streams.
 * The call allocates nothing and never synchronises, so it can be captured into
 * a CUDA graph (make one call on the device outside capture first).  The split
 * schedule is derived on the device from kv_indptr, so a replayed graph follows
 * new values in the same buffers (query, cache, kv_indptr, page table) as long
 * as every row stays within plan->max_kv_len, kv_indptr[B] within
 * kv_indices_len (page table) or kv_rows (contiguous rows).
 */
mla_status_t mla_decode_fwd(const void* q_bf16, const void* kv_fp8, const float* kv_scale,
                            const int32_t* qo_indptr, const int32_t* kv_indptr, void* out_bf16,
                            cudaStream_t stream, const mla_plan_t* plan,
                            const int32_t* kv_indices, int64_t kv_indices_len, int64_t kv_rows,
                            void* workspace, size_t workspace_bytes);

/*
 * mla_decode_fwd_static_scratch — mla_decode_fwd without a caller workspace.
 * The pages have no counterpart: this entry exists for callers that must not
 * allocate device memory, such as a plugin inside a host application that owns
 * every device allocation and passes the plugin only its inputs and outputs, or
 * a serving loop where an allocation (which can synchronise the device) is not
 * allowed.  The scratch is a static array of MLA_STATIC_SCRATCH_BYTES that the
 * library reserves on every GPU it is loaded on and keeps until the process
 * exits; nothing is allocated per call.
 *   Arguments as mla_decode_fwd, minus workspace / workspace_bytes.
 *   Returns MLA_ERR_WORKSPACE_TOO_SMALL when plan->ws_bytes exceeds
 *   MLA_STATIC_SCRATCH_BYTES (on a 152-SM GB300 every batch of up to ~600,000
 *   rows fits).
 *   The first call on a device looks up that device's copy of the array; make
 *   that first call before any stream capture.  A device other than sm_103
 *   returns MLA_ERR_UNSUPPORTED.
 *   All calls share the one array: calls that may overlap on the GPU (different
 *   streams, or different host threads on the same device) race and must be
 *   ordered by the caller.  The array's error word collects the MLA_DERR_*
 *   bits of every call (it starts clear when the library is loaded); read and
 *   clear it with mla_decode_static_scratch_read_error, e.g. to learn that a
 *   call gave up on a wait (MLA_DERR_TIMEOUT) and its output is not valid.
 */
#define MLA_STATIC_SCRATCH_BYTES (12u * 1024u * 1024u)
mla_status_t mla_decode_fwd_static_scratch(const void* q_bf16, const void* kv_fp8,
                                           const float* kv_scale, const int32_t* qo_indptr,
                                           const int32_t* kv_indptr, void* out_bf16,
                                           cudaStream_t stream, const mla_plan_t* plan,
                                           const int32_t* kv_indices, int64_t kv_indices_len,
                                           int64_t kv_rows);

/* Read (and, when clear != 0, reset) the error word of the current device's
 * static scratch, as mla_decode_read_error does for a workspace.  Synchronises
 * `stream` (order it after the calls to be checked); off the hot path.  Copies
 * four bytes to the host and allocates nothing. */
mla_status_t mla_decode_static_scratch_read_error(int32_t* err_host, int32_t clear,
                                                  cudaStream_t stream);

/*
 * mla_decode_fwd_bf16kv — the decode step over a bf16 latent cache, as the
 * pages do for batches of at most 131072 cached tokens (submission 722089,
 * AITER PATH section: `_aiter_path` passes the bf16 copy of the cache and the
 * unquantised bf16 query; submission 738050's `custom_kernel` docstring lists
 * that copy among the harness's inputs).  K and V are the cache's bf16 values;
 * q . K and P . V run on bf16 tensor-core operands with float32 accumulation
 * (P rounded to bf16), so each cached token moves 1152 bytes instead of 576.
 *   kv_bf16  device, bf16 [kv_rows, 576] (= [kv_rows, 1, 576]), 16-byte aligned.
 *   kv_indices must be NULL (the cache rows of the batch contiguous, as in the
 *   pages' benchmark); a page table returns MLA_ERR_UNSUPPORTED.
 *   Every other argument, the plan (either qo_len), the workspace, the error
 *   word and the status codes are those of mla_decode_fwd; there is no scale.
 */
mla_status_t mla_decode_fwd_bf16kv(const void* q_bf16, const void* kv_bf16,
                                   const int32_t* qo_indptr, const int32_t* kv_indptr,
                                   void* out_bf16, cudaStream_t stream, const mla_plan_t* plan,
                                   const int32_t* kv_indices, int64_t kv_indices_len,
                                   int64_t kv_rows, void* workspace, size_t workspace_bytes);

/*
 * mla_decode_fwd_mxfp4 — the decode step over an MXFP4 latent cache, the
 * harness's third cache format (submission 738050: `custom_kernel` docstring,
 * `kv_data["mxfp4"]`; `_dequantize_mxfp4_inplace` docstring for the format;
 * submission 722089 `_custom_multihead_path` / `_mla_multihead_stage1` read it).
 * A cached row is 576 E2M1 elements (2 per byte, the even element in the low
 * nibble: 288 bytes) and 18 E8M0 scales, one per 32 consecutive elements; its
 * value is element * 2^(scale - 127).  K is the whole row and V its first 512
 * values, as for mla_decode_fwd.
 *   kv_fp4     device uint8 [kv_rows, 288], 16-byte aligned.
 *   kv_scales  device uint8 [kv_rows, 18] (row stride 18 bytes), 16-byte aligned.
 *   scale_bias each tile is converted in shared memory to the e4m3 codes of
 *              element * 2^(scale - 127 - scale_bias) and attended with the
 *              per-tensor scale 2^scale_bias: exact while every block holding a
 *              nonzero element has scale - 127 - scale_bias in [-8, 6] (block
 *              scales 2^-8 ... 2^6 with the bias 0, which covers blocks whose
 *              largest magnitude lies in [2^-6, 2^9)).  A block outside that
 *              window sets MLA_DERR_MX_SCALE; its values then saturate at
 *              448 * 2^scale_bias or round toward zero.  |scale_bias| <= 100.
 *   kv_rows    rows of the pool, at most 119,304,419.
 *   The rows of the batch are contiguous in the pool (no page table, as in the
 *   pages' MXFP4 kernel); plan->qo_len must be 1 (else MLA_ERR_UNSUPPORTED).
 *   Every other argument, the workspace, the error word and the status codes
 *   are those of mla_decode_fwd.
 */
mla_status_t mla_decode_fwd_mxfp4(const void* q_bf16, const void* kv_fp4, const void* kv_scales,
                                  int32_t scale_bias, const int32_t* qo_indptr,
                                  const int32_t* kv_indptr, void* out_bf16, cudaStream_t stream,
                                  const mla_plan_t* plan, int64_t kv_rows, void* workspace,
                                  size_t workspace_bytes);

/* The two stages of mla_decode_fwd launched separately (same arguments); the
 * pair is equivalent to one mla_decode_fwd call.  Used to time stage 1 alone.
 * mla_decode_stage1_bf16kv is stage 1 of mla_decode_fwd_bf16kv; stage 2 is
 * shared by both caches. */
mla_status_t mla_decode_stage1(const void* q_bf16, const void* kv_fp8, const float* kv_scale,
                               const int32_t* qo_indptr, const int32_t* kv_indptr, void* out_bf16,
                               cudaStream_t stream, const mla_plan_t* plan,
                               const int32_t* kv_indices, int64_t kv_indices_len, int64_t kv_rows,
                               void* workspace, size_t workspace_bytes);
mla_status_t mla_decode_stage1_bf16kv(const void* q_bf16, const void* kv_bf16,
                                      const int32_t* qo_indptr, const int32_t* kv_indptr,
                                      void* out_bf16, cudaStream_t stream, const mla_plan_t* plan,
                                      const int32_t* kv_indices, int64_t kv_indices_len,
                                      int64_t kv_rows, void* workspace, size_t workspace_bytes);
mla_status_t mla_decode_stage1_mxfp4(const void* q_bf16, const void* kv_fp4, const void* kv_scales,
                                     int32_t scale_bias, const int32_t* qo_indptr,
                                     const int32_t* kv_indptr, void* out_bf16, cudaStream_t stream,
                                     const mla_plan_t* plan, int64_t kv_rows, void* workspace,
                                     size_t workspace_bytes);
mla_status_t mla_decode_stage2(const int32_t* qo_indptr, void* out_bf16, cudaStream_t stream,
                               const mla_plan_t* plan, void* workspace, size_t workspace_bytes);

/*
 * mla_decode_fwd_stall_stream — test hook for the bounded waits (no
 * counterpart on the pages).  Same arguments and launches as mla_decode_fwd,
 * but stage 1's producers issue no cache loads, so the waits on them run out
 * after their time limit (about one second of SM cycles); the kernel then sets
 * MLA_DERR_TIMEOUT in the workspace error word, stops issuing work, drains
 * what it issued and returns.  Nothing faults and the context stays usable.
 * The output is not written meaningfully.  Returns MLA_OK after launching.
 */
mla_status_t mla_decode_fwd_stall_stream(const void* q_bf16, const void* kv_fp8,
                                         const float* kv_scale, const int32_t* qo_indptr,
                                         const int32_t* kv_indptr, void* out_bf16,
                                         cudaStream_t stream, const mla_plan_t* plan,
                                         const int32_t* kv_indices, int64_t kv_indices_len,
                                         int64_t kv_rows, void* workspace, size_t workspace_bytes);

/*
 * mla_decode_fwd_mxfp4_stall_stream — test hook for the bounded waits of the
 * MXFP4 kernel (no counterpart on the pages): mla_decode_fwd_mxfp4 with a
 * producer that loads nothing, so the converter warps' and MMA issuers' waits
 * run out; as mla_decode_fwd_stall_stream, the call sets MLA_DERR_TIMEOUT,
 * drains and returns without a fault, and the output is not meaningful.
 * Arguments as mla_decode_fwd_mxfp4.
 */
mla_status_t mla_decode_fwd_mxfp4_stall_stream(const void* q_bf16, const void* kv_fp4,
                                               const void* kv_scales, int32_t scale_bias,
                                               const int32_t* qo_indptr, const int32_t* kv_indptr,
                                               void* out_bf16, cudaStream_t stream,
                                               const mla_plan_t* plan, int64_t kv_rows,
                                               void* workspace, size_t workspace_bytes);

/*
 * mla_debug_q_operand — test hook (no counterpart on the pages): the query
 * operand of the e4m3-cache step exactly as a stage-1 CTA builds it in shared
 * memory, copied out.  The pages hand the tensor cores an FP8 query (submission
 * 722089 `_mla_multihead_stage1` casts each query chunk to float8e4nv;
 * submissions 663509 and 738050 quantise Q per tensor); this library keeps the
 * bf16 query's precision with two e4m3 terms per value.  Per query token:
 * a = max |q| over its 16 x 576 values, k2 the integer with
 * 224 < a * 2^k2 <= 448 (clamped to [-126, 126]; 0 when a = 0),
 * x = float32(q * 2^k2), hi = e4m3(x), lo = e4m3(float32(16 * (x - hi))), both
 * rounded to nearest even and saturating; the QK accumulator of the token is
 * turned into base-2 softmax units by qk_scale = 2^-k2 * kv_scale * log2(e) / 24.
 *   q_bf16         device bf16 [num_tokens, 16, 576], 16-byte aligned.
 *   num_tokens     1 .. 2^24.
 *   tokens_per_cta 1 or 2: run the one- or two-token form of the operand code
 *                  (a stage-1 CTA takes up to two query tokens of a row).
 *   kv_scale       device float[1].
 *   codes_out      device uint8 [num_tokens, 2, 16, 576]: hi codes of the 16
 *                  heads, then lo codes; 16-byte aligned.
 *   qk_scale_out   device float [num_tokens].
 * One kernel on `stream`; returns MLA_OK after launching.
 */
mla_status_t mla_debug_q_operand(const void* q_bf16, int32_t num_tokens, int32_t tokens_per_cta,
                                 const float* kv_scale, void* codes_out, float* qk_scale_out,
                                 cudaStream_t stream);

/*
 * mla_debug_p_split — test hook (no counterpart on the pages): the two-term
 * e4m3 probability operand of the e4m3-cache step, by stage 1's own code.  The
 * pages round P to bf16 before P . V (submission 722089 `_mla_multihead_stage1`);
 * here p16 = float16(p), hi = e4m3(p16), lo = e4m3(float16(16 * (p16 - hi))),
 * every step rounded to nearest even in half precision.
 *   p       device float [n] (0 <= p <= 256 in the kernel), 16-byte aligned.
 *   n       a multiple of 16, >= 16.
 *   hi_out, lo_out  device uint8 [n], 16-byte aligned.
 * One kernel on `stream`; returns MLA_OK after launching.
 */
mla_status_t mla_debug_p_split(const float* p, int64_t n, void* hi_out, void* lo_out,
                               cudaStream_t stream);

/*
 * mla_decode_trace_read — start-up trace of trace builds (no counterpart on the
 * pages): a library compiled with -DMLA_TRACE stamps, for each of the first
 * MLA_TRACE_CTAS stage-1 CTAs, MLA_TRACE_EVENTS events (entry and exit on the
 * global timer in ns; the milestones between them in SM cycles: before and
 * after the wait for the previous kernel, prologue done, first cache copy
 * issued, Q operand ready, first rope panel landed, first QK issued, first
 * scores read, first P published, first PV issued, first epilogue start and
 * end, exit; then the row-pointer loads returned, the prologue's scan barrier,
 * the first query loads returned, the first rope and last latent panel
 * arrived (a lane of the otherwise idle warp 7 watching them); for the
 * cluster split the cluster barrier passed and the combine written; not a
 * clock, segments * 65536 + tiles of the CTA's range; then the boundary into
 * the second segment: the first segment's last P published, the second
 * segment's Q operand published, its first scores read, P published and PV
 * issued, its Q preparation started and its query loads returned; then the
 * cluster combine's weight formed and partials landed, the prologue's totals
 * and first row, the producer's and the softmax's loop starts, the first
 * query loads issued and the producer's first barrier arming; event indices
 * as in the library's kernels.h), and for each of the first
 * MLA_TRACE2_BLOCKS stage-2 blocks
 * (numbered y * grid_x + x) the global timer at entry, after its wait for
 * stage 1 and at exit.  Each call's stamps overwrite the previous call's.
 *   stage1_host  host uint64 [MLA_TRACE_CTAS * MLA_TRACE_EVENTS]
 *   stage2_host  host uint64 [MLA_TRACE2_BLOCKS * 3]
 *   clear        nonzero: zero the device copies after reading.
 * Synchronous.  Release builds return MLA_ERR_UNSUPPORTED.
 */
#define MLA_TRACE_CTAS 320
#define MLA_TRACE_EVENTS 40
#define MLA_TRACE2_BLOCKS 4096
mla_status_t mla_decode_trace_read(uint64_t* stage1_host, uint64_t* stage2_host, int32_t clear);

/*
 * mla_fp8_quantize_per_tensor — per-tensor absmax quantisation of a bf16 tensor
 * to e4m3fn (input preparation; the pages' harness supplies the cache already
 * quantised this way: submission 722089 `quantize_fp8`, submission 738050
 * `_quantize_fp8`):  scale = max(max|x|, 1e-12) / 448 and
 * code = e4m3fn_rn_satfinite(x / scale), both divisions IEEE float32.
 *   src_bf16  device bf16 [n];  dst_fp8 device uint8 [n];
 *   scale_out device float[1];  tmp device scratch of >= 16 bytes.
 * Two kernels and one 4-byte memset on `stream`.
 */
mla_status_t mla_fp8_quantize_per_tensor(const void* src_bf16, int64_t n, void* dst_fp8,
                                         float* scale_out, void* tmp, size_t tmp_bytes,
                                         cudaStream_t stream);

/*
 * mla_mxfp4_quantize — MXFP4 quantisation of bf16 rows of 576 values (input
 * preparation; the pages' harness supplies the cache already quantised, see
 * mla_decode_fwd_mxfp4).  Per block of 32 consecutive values of a row: scale
 * exponent e = floor(log2 max|x|) - 2 clamped to [-127, 127] (-127 for an
 * all-zero block), stored as the byte e + 127; elements x / 2^e rounded to the
 * nearest E2M1 value, ties to even, saturating at +-6 (the OCP Microscaling
 * conversion).
 *   src_bf16   device bf16 [rows, 576], 16-byte aligned (finite values).
 *   dst_fp4    device uint8 [rows, 288], 16-byte aligned.
 *   dst_scales device uint8 [rows, 18].
 * One kernel on `stream`.
 */
mla_status_t mla_mxfp4_quantize(const void* src_bf16, int64_t rows, void* dst_fp4, void* dst_scales,
                                cudaStream_t stream);

/* Zero a workspace (cudaMemsetAsync of ws_bytes on `stream`). */
mla_status_t mla_decode_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Read (and, when clear != 0, reset) the device error word of a workspace.
 * Synchronises `stream`; off the hot path. */
mla_status_t mla_decode_read_error(void* workspace, int32_t* err_host, int32_t clear,
                                   cudaStream_t stream);

/*
 * mla_decode_schedule_host — the stage-1 schedule of an e4m3 (or MXFP4) cache
 * computed on the host from a host copy of kv_indptr, with the same integer
 * formulas the kernel uses.
 *   workers_out int32 [grid*4]: (t0, t1, first_row, last_row) per worker
 *   in schedule units (first_row = last_row = -1 for a range without tiles);
 *   prefix_out int32 [B+1]: units before each row (tiles and start units of
 *   the rows before it).  Pure host; for tests and tools.
 */
mla_status_t mla_decode_schedule_host(const int32_t* kv_indptr_host, int32_t batch, int32_t grid,
                                      int32_t* workers_out, int32_t* prefix_out);

const char* mla_status_string(mla_status_t status);
int32_t mla_decode_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
