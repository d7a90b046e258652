// Kernel parameter blocks and launchers (internal to libmla_decode).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "../../include/mla_decode.h"

namespace mla {

// Debug builds (-DMLA_DEBUG, `build(debug=True)`): every global store of the
// kernels, the query loads, the cache tile coordinates and the converters'
// shared-memory addresses are checked against their buffers first; a failed
// check sets MLA_DERR_DEBUG_BOUNDS in the workspace error word and skips the
// access (a stand-in for a memory checker, which this toolchain's pool does not
// offer).  Release builds compile the checks away.
#ifdef MLA_DEBUG
#define MLA_DCHECK(cond, err) ((cond) ? true : (atomicOr((err), MLA_DERR_DEBUG_BOUNDS), false))
#else
#define MLA_DCHECK(cond, err) true
#endif

// Stage 1 ring: two rope slots (128 tokens x 64 dims); the latent slots and
// every size depend on the cache format (stage1.cu, Geo).
constexpr int kNumRSlots = 2;
// warps 0-3 softmax/epilogue, 4 TMA producer, 5 PV MMA issuer, 6 QK MMA issuer;
// page-table mode with one query token adds TMA producers in warps 7-11 (12
// warps), two query tokens on contiguous rows a second softmax warpgroup in
// warps 8-11 (12 warps), an MXFP4 cache converter warps 8-15 (16 warps);
// registers rebalanced with setmaxnreg in all three.
constexpr int kStage1Threads = 256;
constexpr int kStage1ThreadsGather = 384;
constexpr int kStage1ThreadsMx = 512;  // MXFP4 cache: warps 8-15 convert its panels
constexpr long long kWaitLimitCycles = 2000000000LL;  // ~1 s per pipeline wait at 2 GHz

// Start-up trace of trace builds (-DMLA_TRACE, `build(trace=True)`): per stage-1
// CTA (the first kTraceCtas) kTraceEvents stamps, per stage-2 block (the first
// kTrace2Blocks, numbered y * gridDim.x + x) three global-timer stamps.
constexpr int kTraceCtas = MLA_TRACE_CTAS;
constexpr int kTraceEvents = MLA_TRACE_EVENTS;
constexpr int kTrace2Blocks = MLA_TRACE2_BLOCKS;
constexpr int kTrace2Events = 3;
enum TraceEvent {
  kTrEntryNs = 0,      // global timer at entry (ns)
  kTrEntry = 1,        // the rest: SM cycles (clock64); entry
  kTrPreWait = 2,      // thread 0 before waiting for the previous kernel of the stream
  kTrPostWait = 3,     // ... after it
  kTrPrologue = 4,     // schedule prologue done (after the block barrier)
  kTrFirstCopy = 5,    // producer: first cache copy issued
  kTrQReady = 6,       // softmax: the first segment's Q operand published
  kTrRopeLanded = 7,   // QK issuer: the first rope panel landed
  kTrQkIssued = 8,     // QK issuer: the first tile's QK issued and committed
  kTrSRead = 9,        // softmax: the first tile's scores read out of TMEM
  kTrPReady = 10,      // softmax: the first tile's P published
  kTrPvIssued = 11,    // PV issuer: the first tile's PV issued
  kTrEpilogue = 12,    // softmax: the first segment's epilogue starts (its last PV done)
  kTrEpilogueDone = 13,  // softmax: the first segment's output stores issued
  kTrExit = 14,        // thread 0 after the final block barrier
  kTrExitNs = 15,      // global timer at exit (ns)
  kTrIndptrLoaded = 16,  // thread 0: its rows' kv_indptr entries returned
  kTrScanBarrier = 17,   // thread 0: past the prologue's first block barrier
  kTrQLoaded = 18,       // softmax: the first query loads returned
  kTrRopeArrived = 19,   // observer lane: the first rope panel's copy completed
  kTrTileArrived = 20,   // observer lane: the first tile's last latent panel completed
  kTrClusterBarrier = 21,  // cluster split: thread 0 past the cluster barrier
  kTrCombineDone = 22,     // ... its share of the combine written
  kTrShape = 23,           // not a clock: segments * 65536 + tiles of this CTA's range
  kTrPLast0 = 24,          // softmax: the first segment's last P published
  kTrQReady1 = 25,         // softmax: the second segment's Q operand published
  kTrSRead1 = 26,          // softmax: the second segment's first scores read
  kTrPReady1 = 27,         // softmax: the second segment's first P published
  kTrPvIssued1 = 28,       // PV issuer: the second segment's first PV issued
  kTrQStart1 = 29,         // softmax: the second segment's Q preparation starts
  kTrQLoaded1 = 30,        // softmax: ... its query loads returned
  kTrCombineW = 31,        // cluster split: thread 0's combine weight formed
  kTrCombineLanded = 32,   // ... the partials landed in shared memory
  kTrScanTotals = 33,      // prologue: thread 0 has the batch's totals (after the first barrier)
  kTrFirstRowFound = 34,   // prologue: the first row found and its L2 prefetches issued
  kTrProducerStart = 35,   // producer: its loop starts
  kTrSoftmaxStart = 36,    // softmax: its loop starts
  kTrQIssued = 37,         // softmax: the first query loads issued
  kTrFirstExpect = 38,     // producer: about to arm the first panel's barrier and issue its copy
};
// Copy the trace out (host arrays of kTraceCtas * kTraceEvents and kTrace2Blocks
// * kTrace2Events entries) and zero it; cudaErrorNotSupported without -DMLA_TRACE.
cudaError_t trace_read_stage1(unsigned long long* host, bool clear);
cudaError_t trace_read_stage2(unsigned long long* host, bool clear);

struct Stage1Params {
  const uint16_t* q;          // bf16 bits [B, 16, 576]
  const float* kv_scale;      // [1] (e4m3 cache; unused for a bf16 cache)
  const int32_t* qo_indptr;   // [B+1]
  const int32_t* kv_indptr;   // [B+1]
  const int32_t* kv_indices;  // [kv_indices_len] or null
  uint16_t* out;              // bf16 bits [B, 16, 512]
  int32_t* err;               // workspace error word
  int32_t* prefix;            // [B+1]
  int32_t* workers;           // [grid*8]: worker record + combine job
  float* lse;                 // [2*grid*kQ*16] (kQ: this launch's tokens per row)
  uint16_t* partial;          // bf16 bits [2*grid*kQ*16*512]
  int64_t kv_rows;
  int64_t kv_indices_len;
  int32_t batch;
  int32_t grid;
  int32_t row_tokens;         // query tokens per row (1 to 4)
  int32_t q_off;              // first of the row's tokens this launch handles
  int32_t siblings;           // CTAs per worker (1, or 2 for rows of 3-4 tokens: CTA
                              // 2c + s takes tokens q_off + 2s, up to two of them)
  int32_t slot_tokens;        // query tokens per partial slot (the row's tokens this
                              // launch handles, all siblings together)
  int32_t stall_stream;       // test hook: the producers issue no cache loads, so the
                              // pipeline waits run out (bounded) and the call gives up
  int32_t mx_bias;            // MXFP4 cache: e4m3 panels hold e2m1 * 2^(e - 127 - mx_bias)
  const uint8_t* kv_bytes;    // contiguous rows: the cache (or MXFP4 elements) for an L2
                              // prefetch of the first tile; null with a page table
  int32_t kv_row_bytes;       // bytes per cached row in kv_bytes (576, 1152 or 288)
  int32_t cluster;            // CTAs per row of the cluster split (2, 4, 8), or 0: persistent
};

enum class CacheFormat { kE4m3, kBf16, kMxfp4 };

// TMA descriptors of one call: the cache's latent and rope boxes (e4m3: 128-
// and 64-byte wide; bf16: both 64 dims; MXFP4 elements: 64 and 32 bytes) and,
// for an MXFP4 cache, the flat scale array in 256-byte boxes (else a copy of v).
struct Stage1Maps {
  CUtensorMap v, r, s;
};

struct Stage2Params {
  const int32_t* qo_indptr;
  uint16_t* out;
  int32_t* err;
  const int32_t* prefix;
  const int32_t* workers;  // [grid*8] (t0, t1, first_row, last_row, job tq, job first
                           // worker, job last worker, job first slot), written by stage 1
  const float* lse;
  const uint16_t* partial;  // bf16 bits
  int32_t batch;
  int32_t grid;
  int32_t qo_len;  // query tokens per row (1 to 4), all in one partial slot
};

size_t stage1_smem_bytes();
cudaError_t stage1_prepare(int device);  // sets the dynamic shared memory limit once
cudaError_t launch_stage1(const Stage1Params& p, const Stage1Maps& maps, bool gather,
                          CacheFormat format, cudaStream_t stream);
cudaError_t launch_stage2(const Stage2Params& p, bool programmatic, cudaStream_t stream);
// Test hooks: stage 1's own two-term operand code run on caller buffers.
cudaError_t launch_debug_q_operand(const uint16_t* q, int32_t tokens, int32_t per_cta,
                                   const float* kv_scale, uint8_t* codes, float* qk_scale,
                                   cudaStream_t stream);
cudaError_t launch_debug_p_split(const float* p, int64_t groups, uint8_t* hi, uint8_t* lo,
                                 cudaStream_t stream);
cudaError_t launch_mxfp4_quantize(const uint16_t* src, int64_t rows, uint8_t* dst, uint8_t* scales,
                                  cudaStream_t stream);
cudaError_t launch_fp8_quantize(const uint16_t* src, int64_t n, uint8_t* dst, float* scale_out,
                                uint32_t* amax_bits, cudaStream_t stream);

}  // namespace mla
