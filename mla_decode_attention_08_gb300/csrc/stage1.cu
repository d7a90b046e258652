// Stage 1 of the MLA forward_absorb decode step on sm_103a: split attention.
//
// One persistent CTA per worker of the token-balanced schedule walks its tile
// range (two sibling CTAs for rows of three or four query tokens, each taking
// up to two of them).  Per 128-token tile of the latent cache:
//   * warp 4 streams the tile once through TMA into a ring of swizzled panels
//     (four 128-dim latent panels + one 64-dim rope panel; page-table rows are
//     fetched with tile::gather4, the panels spread over several producer
//     warps),
//   * warp 6 issues the tcgen05 MMAs S^T[128 tok x N] = K_tile . Q_op^T and
//     warp 5 the MMAs O^T[512 x N] += V_tile^T . P^T, accumulators in TMEM,
//   * warps 0-3 run the exp2 online softmax on S read from TMEM, write P, and
//     at the end of a segment write either the bf16 output (row fully inside
//     this worker) or a normalised partial plus its base-2 log-sum-exp.
// The same shared-memory tile feeds both products and all 16 heads (of every
// query token of the row), which is the pages' multi-head KV reuse
// (kernelbot-amd-mixed-mla submission 722089, module docstring and
// `_mla_multihead_stage1`).
//
// Two cache formats (Kv).  An e4m3 cache (codes with one per-tensor scale):
// both operands of each product are FP8 e4m3 (kind::f8f6f4), and Q and P keep
// bf16-level precision by a two-term split x ~= hi + lo / 16 with both terms
// e4m3: per query token the 16 "hi" and 16 "lo" heads, so N = 32 per token of
// the row.  A bf16 cache (the pages' choice for small batches, submission
// 722089 `_aiter_path`): bf16 Q and P operands (kind::f16), N = 16 per token,
// and every tile moves twice the bytes.  An MXFP4 cache (submission 738050,
// `_dequantize_mxfp4_inplace`; submission 722089 `_mla_multihead_stage1`):
// E2M1 elements with one E8M0 scale per 32; the tile streams in at 306 bytes a
// token and eight converter warps rewrite each panel in place as the e4m3 panel
// the e4m3 path reads (exact while the block scales stay in a 15-binade
// window), so the MMAs and the softmax are the e4m3 ones.  A CTA takes one or
// two of the row's query tokens (Geo<kQ, kFmt>); an MXFP4 cache takes one.
#include <cstddef>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/mla_decode.h"
#include "kernels.h"
#include "ptx.cuh"
#include "schedule.h"

namespace mla {
namespace {

// ------------------------------------------------------------ layout
// Operand descriptors (layout codes: 2 = 128B swizzle, 4 = 64B, 6 = 32B).
constexpr uint32_t kLayoutSw128 = 2, kLayoutSw64 = 4, kLayoutSw32 = 6;

constexpr int kMaxQ = 2;          // query tokens per row handled by one CTA tile
constexpr int kMaxCluster = 8;    // CTAs per row of the cluster split
constexpr int kMaxVSlots = 11;    // latent ring slots (e4m3, kQ = 1)

// Latent cache formats.
enum class Kv { kE4m3, kBf16, kMx4 };

// MXFP4 cache: each tile's 128 x 18 scale bytes land, by ten 256-byte boxes of
// the flat scale array starting at the 16-byte boundary at or below the tile's
// first byte, in one of four scale slots.
constexpr int kNumSclSlots = 4;
constexpr int kSclBoxes = 10;
constexpr int kSclSlotBytes = 256 * kSclBoxes;
static_assert(kSclSlotBytes >= 15 + kTileTokens * 18, "a tile's scale bytes fit a slot");
constexpr int kConverterWarps = 8;
constexpr int kFirstConverterWarp = 8;

// Everything that depends on the cache format and on the number kQ of query
// tokens per row.  The MMA N dimension holds, for each query token, the 16
// "hi" then the 16 "lo" heads (e4m3: column n = 32 qi + 16 lo + head) or the 16
// heads (bf16: column n = 16 qi + head).
template <int kQ, Kv kFmt>
struct Geo {
  static_assert(kQ == 1 || kQ == 2, "one or two query tokens per row");
  static_assert(kFmt != Kv::kMx4 || kQ == 1, "an MXFP4 cache takes one query token per row");
  static constexpr bool kMx = kFmt == Kv::kMx4;        // elements converted in shared memory
  static constexpr bool kSplit = kFmt != Kv::kBf16;  // two-term Q and P operands
  static constexpr int kElem = kSplit ? 1 : 2;         // bytes per cache / operand element
  static constexpr int kTokCols = kSplit ? 32 : 16;    // operand columns per query token
  static constexpr int kN = kTokCols * kQ;             // MMA N / operand rows of Q and P
  // Ring slots: a latent slot holds 128 tokens x 128 dims (16 or 32 KB), a rope
  // slot 128 tokens x 64 dims.  A 128-byte-wide swizzled panel holds 128 e4m3 or
  // 64 bf16 dims, so a bf16 latent slot is two panels 16 KB apart.
  static constexpr int kVSlotBytes = 128 * 128 * kElem;
  static constexpr int kRSlotBytes = 128 * 64 * kElem;
  static constexpr int kNumV = kMx ? 10 : (kSplit ? (kQ == 1 ? 11 : 9) : (kQ == 1 ? 5 : 4));
  static constexpr int kPanelDims = 128 / kElem;
  // Q operand: kN rows; the 512 latent dims in 128-byte-wide panels, the 64
  // rope dims in one more (64 bytes wide, swizzle 64B, for e4m3; 128 for bf16).
  static constexpr int kQPanelBytes = kN * 128;
  static constexpr int kQLatentPanels = 512 / kPanelDims;
  static constexpr int kQRopeBytes = kN * 64 * kElem;
  static constexpr int kRopeWidth = 64 * kElem;        // bytes per row of a rope panel
  static constexpr uint32_t kRopeLayout = kSplit ? kLayoutSw64 : kLayoutSw128;
  static constexpr int kPRowBytes = kN * kElem;        // P: one row per token (32 kQ bytes)
  static constexpr int kPBytes = 128 * kPRowBytes;
  static constexpr uint32_t kPLayout = kPRowBytes == 32 ? kLayoutSw32 : kLayoutSw64;  // one atom = one P row

  static constexpr int kOffV = 0;
  static constexpr int kOffR = kOffV + kNumV * kVSlotBytes;
  static constexpr int kOffQ = kOffR + kNumRSlots * kRSlotBytes;
  static constexpr int kOffQRope = kOffQ + kQLatentPanels * kQPanelBytes;
  static constexpr int kOffP = kOffQRope + kQRopeBytes;
  static constexpr int kOffScl = kOffP + 2 * kPBytes;  // MXFP4 scale slots
  static constexpr int kOffMisc = kOffScl + (kMx ? kNumSclSlots * kSclSlotBytes : 0);
  // MXFP4: a panel's elements land in the upper half of its slot (a latent row
  // is 64 bytes of elements, a rope row 32), below the e4m3 panel they become.
  static constexpr int kVRawOff = kVSlotBytes / 2;
  static constexpr int kRRawOff = kRSlotBytes / 2;
  static_assert(kOffP - kOffQ >= kQ * kNumHeads * kVDim * 2, "the Q region stages a bf16 output row");

  // TMEM columns: two S buffers (kN each) then O (4 chunks x kN).
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 2 * kN;
  static constexpr uint32_t kTmemCols = 6 * kN <= 128 ? 128 : (6 * kN <= 256 ? 256 : 512);
  static_assert(kColO + 4 * kN <= kTmemCols, "TMEM columns");

  // K-major A and B for QK; MN-major A and B for PV.
  static constexpr uint32_t kIdescQK = kSplit ? idesc_e4m3(128, kN, false, false)
                                              : idesc_bf16(128, kN, false, false);
  static constexpr uint32_t kIdescPV = kSplit ? idesc_e4m3(128, kN, true, true)
                                              : idesc_bf16(128, kN, true, true);
};

constexpr int kQParts = 5;  // parts of the Q operand, each with a barrier (see q_job)
// The chunk order of the Q preparation (q_job): by parts on contiguous rows.
// And whether the operand is published part by part (q_part_done), which
// needs that order: also only with the QK issuer's loops rolled.  The softmax
// and the issuer both decide by these.
__device__ __forceinline__ bool q_panel_order(bool gather, const Stage1Params&) { return !gather; }
__device__ __forceinline__ bool q_split(bool rolled, bool gather, const Stage1Params& p) {
  return rolled && q_panel_order(gather, p);
}

struct Misc {
  uint64_t v_full[kMaxVSlots];
  uint64_t v_empty[kMaxVSlots];
  uint64_t r_full[kNumRSlots];
  uint64_t raw_full[kMaxVSlots];   // MXFP4: a latent panel's elements landed
  uint64_t rraw_full[kNumRSlots];  // MXFP4: a rope panel's elements and its tile's scales landed
  uint64_t s_full[2];   // QK of tile i landed in S[i & 1]
  uint64_t pv_done[2];  // PV of tile i completed (P[i & 1] free again)
  uint64_t q_empty;     // the segment's last QK completed (Q operand free)
  uint64_t q_part[kQParts];  // a part of the segment's Q operand is written (one phase per segment)
  uint64_t mma_done;
  // Monotonic counters the MMA issuers poll (st.release, then relaxed loads
  // followed by fence.acq_rel once a condition holds), one per softmax
  // warpgroup (the two-token kernels on contiguous rows run two).
  uint32_t s_read[2];   // tiles whose S has been read out by every softmax warp
  uint32_t p_ready[2];  // tiles whose P is published (and O rescaled)
  uint32_t o_free[2];   // segments whose epilogue has read O out of TMEM
  alignas(16) float red_max[2][4][16 * kMaxQ];  // read and written as float4
  alignas(16) float red_sum[4][16 * kMaxQ];
  uint32_t red_u32[16];  // [4 token + warp]: a query token's |q| maxima; [8 + group]: abort flag
  int32_t scan[kStage1ThreadsMx / 32];       // per warp of the prologue's block scan (largest block):
  int32_t scan_rows[kStage1ThreadsMx / 32];  // tiles, and rows with tiles
  int32_t row_start;    // schedule units before each row's tiles (row_start_units)
  uint32_t tmem_base;
  volatile int32_t abort_flag;
  int32_t total_tiles;
  int32_t t0, t1;
  int32_t first_row, first_prefix, first_tiles, last_row;
  // The first row's cached tokens and this launch's first query token of it
  // (-1: malformed row), found by the prologue so that no role loads them
  // again before its first tile.
  int32_t first_kb, first_len, first_tq;
  int32_t bad;
  int32_t tile0_issued;    // the prologue issued the first tile's copies (contiguous rows)
  alignas(16) float cl_w[kMaxCluster][16];    // cluster split: combine weights [rank][head]
  alignas(16) float cl_lse[kMaxCluster][16];  // ... and the partials' log-sum-exps
  uint32_t next_panel[6];  // per producer warp: one past its last issued panel
  alignas(16) float alpha_stage[16 * kMaxQ];  // O rescale factors of the current tile (thread 0 writes)
};

static_assert(offsetof(Misc, red_max) % 16 == 0 && offsetof(Misc, red_sum) % 16 == 0,
              "vector accesses to the reduction scratch need 16-byte alignment");
static_assert(kNumRSlots == 2, "rope slots are released through s_full, which has two phases in flight");

template <int kQ, Kv kFmt>
constexpr int smem_alloc() {
  // + 1024: room to align the base to 1024 B
  return Geo<kQ, kFmt>::kOffMisc + static_cast<int>(sizeof(Misc)) + 1024;
}
template <int kQ, Kv kFmt>
constexpr bool geo_fits() {
  using G = Geo<kQ, kFmt>;
  return G::kOffMisc % 16 == 0 && smem_alloc<kQ, kFmt>() <= 232448 && G::kNumV <= kMaxVSlots;
}
static_assert(geo_fits<1, Kv::kE4m3>() && geo_fits<2, Kv::kE4m3>() && geo_fits<1, Kv::kBf16>() &&
                  geo_fits<2, Kv::kBf16>() && geo_fits<1, Kv::kMx4>(),
              "stage-1 shared memory: per-CTA limit, 16-byte aligned barrier block, ring slots");

constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;    // PV issuer; owns the TMEM allocation
constexpr int kMmaQkWarp = 6;  // QK issuer
constexpr int kIdleWarp = 7;   // contiguous rows: writes the worker record for stage 2
constexpr uint32_t kBarSoftmax = 1;  // named barrier id of warps 0-3
constexpr uint32_t kBarProducers = 2;  // named barrier id of the page-table producers
constexpr uint32_t kBarConverters = 3;  // named barrier id of the MXFP4 converter warps
constexpr uint32_t kBarSoftmaxB = 4;     // named barrier id of the second softmax warpgroup (warps 8-11)
constexpr uint32_t kBarSoftmaxPair = 5;  // ... of both softmax warpgroups together

// A softmax warpgroup: its threads' index within it, the first of the query-
// token columns it owns, its own named barrier, and the barrier it takes
// before it writes the Q region (both warpgroups' when there are two: the
// other's output staging must have been read first).
struct SoftmaxGroup {
  int t;
  int q0;
  uint32_t bar, pair, pair_threads;
};
__device__ __forceinline__ SoftmaxGroup single_softmax_group() {
  return SoftmaxGroup{static_cast<int>(threadIdx.x), 0, kBarSoftmax, kBarSoftmax, 128u};
}
// Page-table mode with one query token: 12 warps, six producer warps (4, 7,
// 8, 9, 10, 11) taking panels round-robin; the softmax warpgroup gets 240
// registers and the other two 128 (launched with 168 each: 128 x 240 + 256 x 128
// <= 384 x 168).
// With two query tokens the softmax needs more than 240 registers, so that
// kernel keeps 8 warps and two producers (warps 4 and 7).
// An MXFP4 cache runs 16 warps: warps 8-15 convert its panels.
template <bool kGather, int kQ, Kv kFmt>
__host__ __device__ constexpr bool wide_block() { return (kGather && kQ == 1) || kFmt == Kv::kMx4; }
// Two query tokens on contiguous rows: two softmax warpgroups, one token
// each (warps 0-3 and 8-11), 12 warps: a warpgroup of 128 threads then does
// the softmax of one token per tile, as in the one-token kernels, instead of
// one warpgroup doing both tokens' (each warp the only one of its scheduler,
// whose latencies nothing covered).
// (Trace builds keep one warpgroup: with the stamps, ptxas finds no register
// allocation for the two-warpgroup split at any softmax count up to 224.)
template <bool kGather, int kQ, Kv kFmt>
__host__ __device__ constexpr bool dual_softmax() {
#ifdef MLA_TRACE
  return false;
#else
  return !kGather && kQ == 2 && kFmt != Kv::kMx4;
#endif
}
template <bool kGather, int kQ, Kv kFmt>
__host__ __device__ constexpr int stage1_threads() {
  return kFmt == Kv::kMx4 ? kStage1ThreadsMx
                          : (wide_block<kGather, kQ, kFmt>() || dual_softmax<kGather, kQ, kFmt>()
                                 ? kStage1ThreadsGather : kStage1Threads);
}
template <bool kGather, int kQ>
__host__ __device__ constexpr uint32_t num_producers() { return !kGather ? 1 : (kQ == 1 ? 6 : 2); }
// Producer index of a warp in page-table mode (warps 4, 7, 8, ...), or -1.
__device__ __forceinline__ int gather_producer_of_warp(int warp, uint32_t producers) {
  const int who = warp == 4 ? 0 : (warp >= 7 ? warp - 6 : -1);
  return who < static_cast<int>(producers) ? who : -1;
}
constexpr int kSoftmaxRegs = 240, kOtherRegs = 128;
static_assert(128 * kSoftmaxRegs + 256 * kOtherRegs <= kStage1ThreadsGather * 168,
              "register split exceeds the launch allocation");
// Two softmax warpgroups (12 warps, launched with 168 registers a thread):
// 200 for each, 104 for the producer and MMA warpgroup (192 / 120 spilled
// three times as many bytes in the softmax).
constexpr int kDualSoftmaxRegs = 200, kDualOtherRegs = 104;
static_assert(2 * 128 * kDualSoftmaxRegs + 128 * kDualOtherRegs <= kStage1ThreadsGather * 168,
              "two-warpgroup register split exceeds the launch allocation");
// MXFP4 (16 warps, launched with 128 registers a thread): 240 for the softmax
// warpgroup, 88 for the other twelve warps.
constexpr int kOtherRegsMx = 88;
static_assert(128 * kSoftmaxRegs + 384 * kOtherRegsMx <= kStage1ThreadsMx * 128,
              "MXFP4 register split exceeds the launch allocation");

// log2(e) / sqrt(576): converts a dot product to base-2 softmax exponent units.
constexpr float kSmScaleLog2 = 1.4426950408889634f / 24.0f;
// A new row maximum above the running reference by more than this many base-2
// units triggers a rescale; below it, P values up to 2^8 still fit e4m3.
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ int32_t ldg_i32(const int32_t* p) { return __ldg(p); }

// ------------------------------------------------------------ start-up trace (-DMLA_TRACE only)
// Clock stamps of one CTA's way to its first output, per role, in SM cycles
// (clock64), plus the global timer at entry and exit; read back with
// mla_decode_trace_read.  Release builds compile the stamps away.
#ifdef MLA_TRACE
__device__ unsigned long long g_trace_stage1[kTraceCtas * kTraceEvents];
__device__ __forceinline__ void trace_put(int ev, unsigned long long v) {
  if (blockIdx.x < static_cast<unsigned>(kTraceCtas)) g_trace_stage1[blockIdx.x * kTraceEvents + ev] = v;
}
#define MLA_TRACE_CLK(ev) trace_put((ev), static_cast<unsigned long long>(clock64()))
#define MLA_TRACE_NS(ev) trace_put((ev), global_timer_ns())
__device__ __forceinline__ void trace_shape(int32_t segments, int32_t tiles) {
  trace_put(kTrShape, static_cast<unsigned long long>(segments) * 65536ull + static_cast<uint32_t>(tiles));
}
#else
#define MLA_TRACE_CLK(ev) ((void)0)
#define MLA_TRACE_NS(ev) ((void)0)
__device__ __forceinline__ void trace_shape(int32_t, int32_t) {}
#endif

__device__ __forceinline__ void set_error(int32_t* err, int32_t bits) { atomicOr(err, bits); }

// Bounded wait on an mbarrier phase.  Returns false when the call is being
// abandoned (this or another role timed out); never spins without limit.  The
// limit is counted in SM cycles (clock64 is cheap to read, unlike the global
// timer): kWaitLimitCycles is about one second at the maximum SM clock.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, Misc* ms, int32_t* err) {
  if (ms->abort_flag) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (ms->abort_flag) return false;
      if (clock64() - start > kWaitLimitCycles) {
        ms->abort_flag = 1;
        set_error(err, MLA_DERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Misc* ms, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;  // the common case: already complete
  return wait_phase_slow(bar, parity, ms, err);
}

// The same wait with its slow path inlined, for the softmax warpgroup: a call
// out of a region whose register count setmaxnreg raised does not compile.
__device__ __forceinline__ bool wait_phase_inl(uint32_t bar, uint32_t parity, Misc* ms, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (ms->abort_flag) return false;
      if (clock64() - start > kWaitLimitCycles) {
        ms->abort_flag = 1;
        set_error(err, MLA_DERR_TIMEOUT);
        return false;
      }
    }
  }
}

template <bool kInline>
__device__ __forceinline__ bool softmax_wait(uint32_t bar, uint32_t parity, Misc* ms, int32_t* err) {
  return kInline ? wait_phase_inl(bar, parity, ms, err) : wait_phase(bar, parity, ms, err);
}

// ------------------------------------------------------------ segment cursor
// Walks the rows intersecting this worker's tile range [t0, t1).
struct Cursor {
  int32_t b;        // current row
  int32_t next_a;   // prefix of row b + 1
  int32_t row_a;    // prefix of row b
  int32_t kb, len;  // first flattened token and token count of row b
  int32_t j, j0, j1;  // current tile and this worker's tile range inside row b
  int32_t seg;      // segment counter (0-based)
  int32_t start;    // schedule units before each row's tiles
  bool whole;       // row b lies entirely inside this worker
  bool live;
};

// Advance to the next row holding tiles of [t0, t1).
__device__ __forceinline__ bool cursor_next_segment(Cursor& c, const int32_t* kv_indptr, int32_t batch,
                                    int32_t t0, int32_t t1) {
  while (c.next_a < t1) {
    const int32_t b = ++c.b;
    if (b >= batch) return false;
    const int32_t kb = ldg_i32(kv_indptr + b);
    const int32_t ke = ldg_i32(kv_indptr + b + 1);
    const int32_t len = ke > kb ? ke - kb : 0;
    const int32_t nt = tiles_of_length(len);
    if (nt == 0) continue;
    const int32_t a = c.next_a + c.start;  // the row's first tile, after its start units
    c.next_a = a + nt;
    if (a >= t1) return false;  // the range ends among the row's start units
    c.row_a = a;
    c.kb = kb;
    c.len = len;
    c.j0 = (t0 > a ? t0 : a) - a;
    c.j1 = (t1 < a + nt ? t1 : a + nt) - a;
    c.j = c.j0;
    c.whole = a >= t0 && a + nt <= t1;
    ++c.seg;
    return true;
  }
  return false;
}

// The first segment comes from the prologue's record of the first row (the
// same values cursor_next_segment would load).
__device__ __forceinline__ void cursor_start(Cursor& c, const Misc* ms) {
  c.seg = -1;
  c.start = ms->row_start;
  c.live = ms->t1 > ms->t0 && ms->first_row >= 0;
  if (!c.live) return;
  const int32_t a = ms->first_prefix, nt = ms->first_tiles, t0 = ms->t0, t1 = ms->t1;
  c.b = ms->first_row;
  c.next_a = a + nt;
  c.row_a = a;
  c.kb = ms->first_kb;
  c.len = ms->first_len;
  c.j0 = (t0 > a ? t0 : a) - a;  // (t0 may lie among the row's start units)
  c.j1 = (t1 < a + nt ? t1 : a + nt) - a;
  c.j = c.j0;
  c.whole = a >= t0 && a + nt <= t1;
  c.seg = 0;
}

// Step to the next tile; returns false when the worker's range is exhausted.
__device__ __forceinline__ bool cursor_next_tile(Cursor& c, const Misc* ms, const int32_t* kv_indptr,
                                 int32_t batch) {
  if (++c.j < c.j1) return true;
  c.live = cursor_next_segment(c, kv_indptr, batch, ms->t0, ms->t1);
  return c.live;
}

// The same step with the segment change out of line, for the roles of the
// MXFP4 kernel other than the softmax (whose raised register count admits no
// calls).  That kernel runs sixteen warps of four roles, each with its own
// copy of the segment change inlined, and it is bound by instruction issue
// with instruction-fetch stalls: one shared copy measured 302 -> 276 us at
// bs256.  (The e4m3 kernels measured the same or slower with it.)
__device__ __noinline__ bool cursor_next_segment_call(Cursor& c, const int32_t* kv_indptr, int32_t batch,
                                                      int32_t t0, int32_t t1) {
  return cursor_next_segment(c, kv_indptr, batch, t0, t1);
}
template <bool kOutOfLine>
__device__ __forceinline__ bool cursor_step(Cursor& c, const Misc* ms, const int32_t* kv_indptr,
                                            int32_t batch) {
  if (!kOutOfLine) return cursor_next_tile(c, ms, kv_indptr, batch);
  if (++c.j < c.j1) return true;
  c.live = cursor_next_segment_call(c, kv_indptr, batch, ms->t0, ms->t1);
  return c.live;
}

// Bounded wait used only while draining at the end of a call.
__device__ __noinline__ bool drain_phase(uint32_t bar, uint32_t parity) {
  const long long start = clock64();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 15 && clock64() - start > kWaitLimitCycles) return false;
  }
}

// ------------------------------------------------------------ this CTA's share
// A worker's tile range is covered by `siblings` CTAs (2c, 2c + 1 with two):
// each takes up to kQ of the row's query tokens, from q_off on, and the
// siblings stream the same tiles (the second one's copies mostly hit L2).
__device__ __forceinline__ int32_t cta_worker(const Stage1Params& p) {
  return static_cast<int32_t>(p.siblings == 2 ? blockIdx.x >> 1 : blockIdx.x);
}
__device__ __forceinline__ int32_t cta_sibling(const Stage1Params& p) {
  return p.siblings == 2 ? static_cast<int32_t>(blockIdx.x & 1) : 0;
}
__device__ __forceinline__ int32_t cta_q_off(const Stage1Params& p) { return p.q_off + 2 * cta_sibling(p); }
template <int kQ>
__device__ __forceinline__ int32_t cta_tokens(const Stage1Params& p) {
  const int32_t left = p.row_tokens - cta_q_off(p);
  return left < kQ ? left : kQ;
}

// The first query token at q_off of a row whose query tokens span
// [q_lo, q_hi), or -1 when that span is not the row_tokens tokens it must be.
__device__ __forceinline__ int32_t row_token(const Stage1Params& p, int32_t q_off, int32_t q_lo,
                                             int32_t q_hi) {
  const int32_t n = p.row_tokens;
  const bool ok = q_hi - q_lo == n && q_lo >= 0 && q_lo <= p.batch * n - n;
  return ok ? q_lo + q_off : -1;
}

// Query tokens of the batch (rows x tokens per row), the bound of q and out.
__device__ __forceinline__ int64_t total_tokens(const Stage1Params& p) {
  return static_cast<int64_t>(p.batch) * p.row_tokens;
}
// bf16 elements of the split partials (2 slots per worker).
__device__ __forceinline__ int64_t partial_elems(const Stage1Params& p) {
  return 2LL * p.grid * p.slot_tokens * kNumHeads * kVDim;
}

// ------------------------------------------------------------ schedule prologue

// All threads.  Tile counts of every row, their prefix, this worker's range
// [t0, t1) and the rows holding its first and last tile.  Worker 0 also stores
// the prefix for stage 2 (every worker's record for stage 2 follows later, in
// write_worker_record).  Zero output for row b (a row without cached tokens, or
// every row when kv_indptr is invalid), written by the one prologue thread that
// finds it.
template <int kQ>
__device__ __forceinline__ void zero_row(const Stage1Params& p, int32_t b) {
  const int32_t tq = row_token(p, cta_q_off(p), ldg_i32(p.qo_indptr + b), ldg_i32(p.qo_indptr + b + 1));
  if (tq < 0) return;
  if (!MLA_DCHECK(tq + cta_tokens<kQ>(p) <= total_tokens(p), p.err)) return;
  uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(tq) * kNumHeads * kVDim);
  const int n = cta_tokens<kQ>(p) * kNumHeads * kVDim * 2 / 16;
  for (int i = 0; i < n; ++i) dst[i] = make_uint4(0, 0, 0, 0);
}

// Contiguous rows: the worker's first tile, issued by the prologue thread that
// finds the worker's first row (tile 0's ring slots start empty), so that its
// copies are in flight while the roles start; the producer begins with the
// second tile.  Not used for an MXFP4 cache or the stall test hook.
// L2 policy of the cache copies.  Every cached element is read once per call
// (by one CTA, or by two siblings a few tiles apart), so its copies leave L2
// first, before the code, query, index and partial lines that every call
// touches again; siblings keep the normal priority, so that the second one's
// copies still find the first one's lines.
__device__ __forceinline__ uint64_t cache_policy(const Stage1Params& p) {
  return p.siblings == 2 ? l2_policy_evict_normal() : l2_policy_evict_first();
}

template <int kQ, Kv kFmt>
__device__ __forceinline__ void issue_first_tile(const Stage1Params& p, const CUtensorMap* map_v,
                                                 const CUtensorMap* map_r, Misc* ms, uint32_t sbase,
                                                 int32_t tok0) {
  using G = Geo<kQ, kFmt>;
  static_assert(G::kNumV >= 4, "tile 0 takes latent slots 0-3");
  if (!MLA_DCHECK(tok0 >= 0 && tok0 < p.kv_rows, p.err)) return;  // the producer then aborts
  const uint64_t pol = cache_policy(p);
  const uint32_t rfull = smem_u32(&ms->r_full[0]);
  mbar_arrive_expect_tx(rfull, G::kRSlotBytes);
  tma_load_2d(sbase + G::kOffR, map_r, kVDim * G::kElem, tok0, rfull, pol);
  constexpr int kBoxes = G::kSplit ? 1 : 2;  // 128-byte-wide boxes per latent slot
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t full = smem_u32(&ms->v_full[c]);
    mbar_arrive_expect_tx(full, G::kVSlotBytes);
#pragma unroll
    for (int i = 0; i < kBoxes; ++i)
      tma_load_2d(sbase + G::kOffV + c * G::kVSlotBytes + i * kTileTokens * 128, map_v,
                  128 * c * G::kElem + 128 * i, tok0, full, pol);
  }
  ms->tile0_issued = 1;
}

template <int kQ, Kv kFmt>
__device__ void schedule_prologue(const Stage1Params& p, const CUtensorMap* map_v,
                                  const CUtensorMap* map_r, Misc* ms, uint32_t sbase) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int32_t batch = p.batch;
  const int32_t per = (batch + nthreads - 1) / nthreads;
  const int32_t r0 = min(tid * per, batch), r1 = min(r0 + per, batch);

  int32_t local = 0, local_rows = 0;  // tiles and rows with tiles of this thread's rows
  int bad = 0;
  // A thread owning a single row also loads its query-token bounds here, in the
  // same round trip (used if that row turns out to be the worker's first).
  int32_t q_lo = 0, q_hi = 0;
  if (r1 - r0 == 1) {
    q_lo = ldg_i32(p.qo_indptr + r0);
    q_hi = ldg_i32(p.qo_indptr + r0 + 1);
  }
  // The row pointers of up to kKeep rows per thread stay in registers for the
  // second pass (batches of up to kKeep x the block's threads need one round
  // trip to global memory); beyond that they are loaded again.
  constexpr int kKeep = 4;
  int32_t keep[kKeep + 1];
  if (r0 < r1) {
    int32_t prev = ldg_i32(p.kv_indptr + r0);
    keep[0] = prev;
#pragma unroll
    for (int i = 0; i < kKeep; ++i) {
      if (r0 + i < r1) {
        keep[i + 1] = ldg_i32(p.kv_indptr + r0 + i + 1);
      }
    }
#pragma unroll
    for (int i = 0; i < kKeep; ++i) {
      if (r0 + i < r1) {
        const int32_t next = keep[i + 1];
        if (next < prev) bad = 1;
        const int32_t nt = tiles_of_length(static_cast<int64_t>(next) - prev);
        local += nt;
        local_rows += nt > 0;
        prev = next;
      }
    }
    for (int32_t b = r0 + kKeep; b < r1; ++b) {
      const int32_t next = ldg_i32(p.kv_indptr + b + 1);
      if (next < prev) bad = 1;
      const int32_t nt = tiles_of_length(static_cast<int64_t>(next) - prev);
      local += nt;
      local_rows += nt > 0;
      prev = next;
    }
  }
  if (tid == 0) {
    const int64_t limit = p.kv_indices != nullptr ? p.kv_indices_len : p.kv_rows;
    const int32_t e0 = ldg_i32(p.kv_indptr), e1 = ldg_i32(p.kv_indptr + batch);
    if (e0 < 0 || e1 > limit) bad = 1;
    // (the stamp depends on the loaded values, so it follows their arrival)
    if (e0 != INT32_MIN && local != INT32_MIN) MLA_TRACE_CLK(kTrIndptrLoaded);
  }
  int32_t incl = local, incl_rows = local_rows;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    const int32_t r = __shfl_up_sync(0xffffffffu, incl_rows, off);
    if (lane >= off) {
      incl += v;
      incl_rows += r;
    }
  }
  if (lane == 31) {
    ms->scan[warp] = incl;
    ms->scan_rows[warp] = incl_rows;
  }
  // (first_row / last_row were set to -1 before the wait for the previous
  // kernel; this barrier orders that before the second pass below.)
  bad = __syncthreads_or(bad);
  if (tid == 0) MLA_TRACE_CLK(kTrScanBarrier);

  int32_t warp_off = 0, tiles = 0, warp_off_rows = 0, rows = 0;
  for (int w = 0; w < nwarps; ++w) {
    const int32_t s = ms->scan[w], r = ms->scan_rows[w];
    if (w < warp) {
      warp_off += s;
      warp_off_rows += r;
    }
    tiles += s;
    rows += r;
  }
  if (bad) tiles = rows = 0;
  // Schedule units: every row with tiles is preceded by `start` units (none
  // for a bf16 cache, whose tiles carry twice the bytes: there a row start
  // costs little against them, and units measured slower).
  const int32_t start = kFmt == Kv::kBf16 ? 0 : row_start_units(tiles, p.grid);
  const int32_t total = tiles + start * rows;
  if (tid == 0) MLA_TRACE_CLK(kTrScanTotals);
  const int32_t c = cta_worker(p);
  const int32_t t0 = worker_begin(c, total, p.grid);
  const int32_t t1 = worker_begin(c + 1, total, p.grid);
  if (tid == 0) {
    ms->total_tiles = total;
    ms->t0 = t0;
    ms->t1 = t1;
    ms->bad = bad;
    ms->row_start = start;
    if (bad) set_error(p.err, MLA_DERR_KV_INDPTR);
  }

  // units before this thread's first row
  int32_t a = bad ? 0 : (warp_off + incl - local) + start * (warp_off_rows + incl_rows - local_rows);
  if (r0 < r1) {
    int32_t prev = keep[0];
    for (int32_t b = r0; b < r1; ++b) {
      int32_t next = 0;
#pragma unroll
      for (int i = 0; i < kKeep; ++i)
        if (b - r0 == i) next = keep[i + 1];
      if (b - r0 >= kKeep) next = ldg_i32(p.kv_indptr + b + 1);
      const int32_t nt = bad ? 0 : tiles_of_length(static_cast<int64_t>(next) - prev);
      const int32_t ra = nt > 0 ? a + start : a;  // the row's first tile, after its start units
      if (c == 0) p.prefix[b] = a;
      if (nt == 0 && b % p.grid == c) zero_row<kQ>(p, b);  // no cached token: zero output
      if (nt > 0 && t1 > t0) {
        if (a <= t0 && t0 < ra + nt && ra < t1) {
          ms->first_row = b;
          ms->first_prefix = ra;
          ms->first_tiles = nt;
          ms->first_kb = prev;
          ms->first_len = next - prev;
          if (r1 - r0 != 1) {
            q_lo = ldg_i32(p.qo_indptr + b);
            q_hi = ldg_i32(p.qo_indptr + b + 1);
          }
          const int32_t tq = row_token(p, cta_q_off(p), q_lo, q_hi);
          ms->first_tq = tq;
          // Warm L2 with what the pipeline reads first: this CTA's query
          // tokens of the row and (contiguous rows) the worker's first tile,
          // while the roles are still starting up.  (Issuing the tile's copies
          // or a bulk copy of the query from here instead measured slower: the
          // block barrier after the prologue, which every role waits for, then
          // ends later, and the query copy lands after the tile.)
          if (tq >= 0)
            prefetch_bulk_l2(p.q + static_cast<size_t>(tq) * kNumHeads * kQkDim,
                             static_cast<uint32_t>(cta_tokens<kQ>(p)) * kNumHeads * kQkDim * 2);
          if (p.kv_bytes != nullptr) {
            const int32_t j0 = t0 > ra ? t0 - ra : 0;
            const int32_t rows = min(kTileTokens, (next - prev) - j0 * kTileTokens);
            prefetch_bulk_l2(p.kv_bytes + (static_cast<int64_t>(prev) + j0 * kTileTokens) * p.kv_row_bytes,
                             static_cast<uint32_t>(rows * p.kv_row_bytes));
          }
          MLA_TRACE_CLK(kTrFirstRowFound);
        }
        // (the next row with tiles has its first tile at ra + nt + start)
        if (ra < t1 && t0 < ra + nt && t1 <= ra + nt + start) ms->last_row = b;
      }
      a = nt > 0 ? ra + nt : a;
      prev = next;
    }
  }
  if (c == 0 && tid == 0) p.prefix[batch] = total;
}

// ------------------------------------------------------------ cluster split prologue
// Row b = blockIdx.x / s is shared by the s CTAs of one cluster (blockIdx.x =
// s b + rank); the CTA of rank r takes the row's tiles [r k, min((r + 1) k, nt)),
// k = ceil(nt / s).  Every CTA checks the whole kv_indptr, as the persistent
// prologue does (a bad one empties every row), in one round trip: thread i
// loads the pointers of row i (the plan keeps the batch within the block), the
// owner of row b also its query bounds.  The roles then see the CTA's share as
// a one-segment tile range starting at prefix 0.  With contiguous rows thread 0
// also issues the share's first tile, so that its copies fly while the roles
// start.  The persistent split's worker records are marked empty so that a
// separately launched stage 2 finds no combine job.
template <int kQ, Kv kFmt>
__device__ void cluster_prologue(const Stage1Params& p, const CUtensorMap* map_v,
                                 const CUtensorMap* map_r, Misc* ms, uint32_t sbase) {
  const int tid = threadIdx.x;
  const int32_t batch = p.batch, s = p.cluster;
  const int32_t b = static_cast<int32_t>(blockIdx.x) / s, rank = static_cast<int32_t>(blockIdx.x) % s;
  int bad = 0;
  for (int32_t r = tid; r < batch; r += blockDim.x) {
    const int32_t x0 = ldg_i32(p.kv_indptr + r), x1 = ldg_i32(p.kv_indptr + r + 1);
    if (x1 < x0) bad = 1;
    if (r == b) {
      const int32_t q_lo = ldg_i32(p.qo_indptr + b), q_hi = ldg_i32(p.qo_indptr + b + 1);
      ms->first_kb = x0;
      ms->first_len = x1 - x0;
      ms->first_tq = row_token(p, cta_q_off(p), q_lo, q_hi);
    }
  }
  if (tid == 0) {
    const int64_t limit = p.kv_indices != nullptr ? p.kv_indices_len : p.kv_rows;
    if (ldg_i32(p.kv_indptr) < 0 || ldg_i32(p.kv_indptr + batch) > limit) bad = 1;
  }
  if (blockIdx.x == 0)
    for (int32_t c = tid; c < p.grid; c += blockDim.x) p.workers[8 * c + 4] = -1;
  bad = __syncthreads_or(bad);
  if (tid == 0) MLA_TRACE_CLK(kTrScanBarrier);
  if (tid == 0) {
    const int32_t nt = bad ? 0 : tiles_of_length(ms->first_len);
    const int32_t k = (nt + s - 1) / s;
    const int32_t j0 = min(rank * k, nt), j1 = min(j0 + k, nt);
    ms->total_tiles = nt;
    ms->t0 = j0;
    ms->t1 = j1;
    ms->first_prefix = 0;
    ms->row_start = 0;
    ms->first_tiles = nt;
    ms->first_row = j1 > j0 ? b : -1;
    ms->last_row = ms->first_row;
    ms->bad = bad;
    if (bad) set_error(p.err, MLA_DERR_KV_INDPTR);
    if (j1 > j0) {
      const int32_t tq = ms->first_tq;
      if (tq >= 0)
        prefetch_bulk_l2(p.q + static_cast<size_t>(tq) * kNumHeads * kQkDim,
                         static_cast<uint32_t>(cta_tokens<kQ>(p)) * kNumHeads * kQkDim * 2);
      if (kFmt != Kv::kMx4 && p.kv_bytes != nullptr && !p.stall_stream)
        issue_first_tile<kQ, kFmt>(p, map_v, map_r, ms, sbase, ms->first_kb + j0 * kTileTokens);
    }
  }
}

// ------------------------------------------------------------ cluster split combine
// Every thread of the CTA of rank r, after the cluster barrier that publishes
// the cluster's partials: the output dims [r D, (r + 1) D), D = 512 / s, of all
// 16 heads of the row's query token, combined from the s CTAs' partials (the
// workspace's partial slots s b .. s b + s - 1: normalised bf16 outputs and
// base-2 log-sum-exps, written by the epilogues) with the weights
// w_i = 2^(lse_i - M) / sum_j 2^(lse_j - M), M = max_i lse_i (submission 722089,
// `_mla_reduce`).  A CTA without tokens (lse = -inf) weighs 0; a row with none
// outputs zeros.
//
// Item (head half, dim): 8 heads of one output dim, a 16-byte piece of each
// slot's partial ([dim / 128][head / 8][dim % 128][head % 8] per slot); a
// thread copies its items' pieces into the ring's first latent slot (free once
// every role has finished) with asynchronous copies, all in flight at once,
// and combines them from there.  The loops over slots are unrolled so that
// their shared-memory loads are all in flight at once: this step is a chain of
// latencies, not of throughput.
template <int kQ, Kv kFmt>
__device__ __forceinline__ void cluster_combine(const Stage1Params& p, Misc* ms, const uint8_t* smem) {
  using G = Geo<kQ, kFmt>;
  static_assert(G::kVSlotBytes >= kNumHeads * kVDim * 2, "the pieces land in one latent slot");
  const int tid = threadIdx.x;
  const int32_t s = p.cluster;
  const int32_t rank = static_cast<int32_t>(cluster_ctarank());
  const int32_t slot0 = static_cast<int32_t>(blockIdx.x) - rank;  // the row's first slot
  const int32_t dims = kVDim / s, items = 2 * dims;
  const size_t slot_elems = static_cast<size_t>(p.slot_tokens) * kNumHeads * kVDim;
  const uint4* land = reinterpret_cast<const uint4*>(smem + G::kOffV);  // [slot][item]
  const int32_t tq = ms->first_tq;
  if (tq < 0) {  // the row's query tokens are malformed: the row is not written
    if (tid == 0 && rank == 0) set_error(p.err, MLA_DERR_QO_INDPTR);
    return;
  }
  if (MLA_DCHECK(static_cast<int64_t>(slot0 + s) * static_cast<int64_t>(slot_elems) <= partial_elems(p),
                 p.err)) {
#pragma unroll 1
    for (int32_t it = tid; it < items; it += static_cast<int32_t>(blockDim.x)) {
      const int32_t hh = it / dims, d = rank * dims + it % dims;
      const uint16_t* src = p.partial + static_cast<size_t>(slot0) * slot_elems +
                            (static_cast<size_t>(d >> 7) * 2 + hh) * (128 * 8) + (d & 127) * 8;
#pragma unroll 1
      for (int32_t i = 0; i < s; ++i)
        cp_async_16(smem_u32(land + i * items + it), src + static_cast<size_t>(i) * slot_elems);
    }
    if (tid < 4 * s)  // 16 bytes (4 heads) of slot tid / 4's log-sum-exps
      cp_async_16(smem_u32(&ms->cl_lse[tid >> 2][4 * (tid & 3)]),
                  p.lse + static_cast<size_t>(slot0 + (tid >> 2)) * p.slot_tokens * kNumHeads + 4 * (tid & 3));
  }
  cp_async_wait_all();
  __syncthreads();
  if (tid == 0) MLA_TRACE_CLK(kTrCombineLanded);
  // Weights of (slot, head), one thread each: w = 2^(lse - M) / sum over the
  // row's slots, M the largest; a slot without tokens (lse = -inf) weighs 0.
  if (tid < 16 * s) {
    const int i = tid >> 4, h = tid & 15;
    float l[kMaxCluster];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      l[j] = j < s ? ms->cl_lse[j][h] : -INFINITY;
      m = fmaxf(m, l[j]);
    }
    float sum = 0.0f, mine = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      const float e = l[j] != -INFINITY ? exp2f(l[j] - m) : 0.0f;
      sum += e;
      mine = j == i ? e : mine;
    }
    ms->cl_w[i][h] = sum > 0.0f ? mine / sum : 0.0f;
    if (tid == 0) MLA_TRACE_CLK(kTrCombineW);
  }
  __syncthreads();
#pragma unroll 1
  for (int32_t it = tid; it < items; it += static_cast<int32_t>(blockDim.x)) {
    const int32_t hh = it / dims, dl = it % dims;
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    uint4 xs[kMaxCluster];
#pragma unroll
    for (int i = 0; i < kMaxCluster; ++i) xs[i] = i < s ? land[i * items + it] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kMaxCluster; ++i) {
      if (i >= s) break;
      const uint4 x = xs[i];
      const float4 w0 = *reinterpret_cast<const float4*>(&ms->cl_w[i][8 * hh]);
      const float4 w1 = *reinterpret_cast<const float4*>(&ms->cl_w[i][8 * hh + 4]);
      const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
      // (an empty or abandoned piece is never written: its weight 0 keeps it out)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xe = __uint_as_float((e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16));
        acc[e] = w[e] != 0.0f ? fmaf(w[e], xe, acc[e]) : acc[e];
      }
    }
    if (MLA_DCHECK(tq < total_tokens(p), p.err)) {
      uint16_t* dst = p.out + (static_cast<size_t>(tq) * kNumHeads + 8 * hh) * kVDim + rank * dims + dl;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat16 y = __float2bfloat16_rn(acc[e]);
        dst[e * kVDim] = *reinterpret_cast<const uint16_t*>(&y);
      }
    }
  }
}

template <int kQ>
__device__ __forceinline__ void write_worker_record(const Stage1Params& p, const Misc* ms);

// The worker record, then the combine job of the split row (if any) whose
// first worker boundary is this worker's start: output row, first and last
// worker of the row, partial slot of the first worker (the others use 2c).
// Only stage 2 reads them, so they are written off the start-up path while the
// pipeline starts: by the otherwise idle warp 7 with contiguous rows, by an
// idle lane of the PV issuer's warp in the page-table kernels (whose warp 7
// produces).
template <int kQ>
__device__ __forceinline__ void write_worker_record(const Stage1Params& p, const Misc* ms) {
  const int32_t c = cta_worker(p);
  const int32_t total = ms->total_tiles, t0 = ms->t0, t1 = ms->t1;
  int32_t job[4] = {-1, 0, 0, 0};
  const int32_t b = ms->first_row, a0 = ms->first_prefix;
  if (t1 > t0 && b >= 0 && a0 < t0) {
    const int32_t c_first = worker_of_tile(a0, total, p.grid);
    if (worker_of_tile(t0 - 1, total, p.grid) == c_first) {
      job[0] = row_token(p, p.q_off, ldg_i32(p.qo_indptr + b), ldg_i32(p.qo_indptr + b + 1));
      job[1] = c_first;
      job[2] = worker_of_tile(a0 + ms->first_tiles - 1, total, p.grid);
      job[3] = partial_slot(c_first, worker_begin(c_first, total, p.grid), a0);
    }
  }
  int4* w = reinterpret_cast<int4*>(p.workers) + 2 * c;
  w[0] = make_int4(t0, t1, ms->first_row, ms->last_row);
  w[1] = make_int4(job[0], job[1], job[2], job[3]);
}

// Trace builds: lane 1 of the otherwise idle warp 7 (contiguous rows) watches
// the first tile's copies land (bounded waits).
template <int kQ, Kv kFmt>
__device__ __forceinline__ void trace_observer(const Stage1Params& p, Misc* ms) {
#ifdef MLA_TRACE
  using G = Geo<kQ, kFmt>;
  if (G::kNumV >= 8 && !p.stall_stream && ms->t1 > ms->t0 && ms->first_row >= 0) {
    if (drain_phase(smem_u32(&ms->r_full[0]), 0)) MLA_TRACE_CLK(kTrRopeArrived);
    if (drain_phase(smem_u32(&ms->v_full[3 % G::kNumV]), 0)) MLA_TRACE_CLK(kTrTileArrived);
  }
#endif
}

// ------------------------------------------------------------ producers (warp 4; page-table mode also 7-11)
constexpr uint32_t kStartGateTile = 2;
// Stream each tile once: the rope slot (64 dims) then four latent slots (128
// dims each), slot fill k = 5 * tile + 1 + c in one sequence over the worker's
// tiles (called "panels" below; a bf16 latent slot takes two boxes of 64 dims).
// Contiguous rows: lane 0 of warp 4 alone issues one tiled box per panel.
// Page table: every lane gathers four rows (tile::gather4) per panel, and the
// panels go round-robin to the producer warps (panel k to producer k % n; n = 6
// with one query token, 2 with two): a warp issues its gathers one lane after
// another, so more issuing warps raise the rate at which row fetches enter the
// copy engine (measured pure-load rates 1.79, 3.53, 4.51, 4.93 and 5.02 TB/s
// with one, two, four, six and eight warps).
//
// Every fill of a slot is issued only after the previous fill of that slot has
// been consumed, so a producer can never be more than one phase ahead on a
// barrier: of its two previous panels at least one is a latent slot, and the
// consumption that panel waited for lies at most two ring laps back.
template <bool kGather, int kQ, Kv kFmt>
__device__ void run_producer(const Stage1Params& p, const CUtensorMap* map_v,
                             const CUtensorMap* map_r, Misc* ms, uint32_t sbase, uint32_t who) {
  using G = Geo<kQ, kFmt>;
  static_assert(!kGather || G::kSplit, "a bf16 cache is read through tiled boxes only");
  constexpr uint32_t kProducers = num_producers<kGather, kQ>();
  static_assert(kProducers <= sizeof(Misc::next_panel) / sizeof(uint32_t), "producer slots");
  const int lane = threadIdx.x & 31;
  if (!kGather && lane != 0) return;
  MLA_TRACE_CLK(kTrProducerStart);
  Cursor cur;
  cursor_start(cur, ms);
  if (p.stall_stream) cur.live = false;  // test hook: nothing is ever loaded
  uint32_t tile = 0;
  uint32_t next_k = 0;  // one past the last panel this warp issued
  const bool tile0_issued = !kGather && ms->tile0_issued;  // by the prologue
  const uint64_t pol = cache_policy(p);
  bool ok = true;
  while (cur.live && ok) {
    if (G::kNumV >= 8 && tile == kStartGateTile) {
      // Start-up: every CTA starts at once, and a ring filled at once puts a
      // few tiles per SM in flight, through which each CTA's first tile (which
      // the pipeline waits for) lands only late.  Tiles from this one on are
      // issued once the first tile's last latent panel has landed.  (Phase 0
      // of that slot is the first tile's only while the second tile fits in
      // other slots: a ring of 8 or more latent slots.  A shallower ring
      // bounds the look-ahead by itself.)
      // (with a page table every lane of the warp waits: a wait run by lane 0
      // alone leaves the warp diverged into the lanes' copies that follow)
      const int w = wait_phase(smem_u32(&ms->v_full[3 % G::kNumV]), 0, ms, p.err);
      ok = kGather ? __all_sync(0xffffffffu, w != 0) : w != 0;
      if (!ok) break;
    }
    const int32_t tok0 = cur.kb + cur.j * kTileTokens;
    const int32_t valid = min(kTileTokens, cur.len - cur.j * kTileTokens);
    int32_t rows[4] = {0, 0, 0, 0};
    if (kGather) {
      // Lane l gathers tokens 4l..4l+3; tokens past the end repeat the last one.
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int32_t t = min(4 * lane + k, valid - 1);
        int32_t idx = ldg_i32(p.kv_indices + tok0 + t);
        if (idx < 0 || static_cast<int64_t>(idx) >= p.kv_rows) {
          set_error(p.err, MLA_DERR_KV_INDEX);
          idx = 0;
        }
        rows[k] = idx;
      }
    }
#pragma unroll 1
    for (int c = -1; c < 4 && ok; ++c) {  // c = -1: rope panel, 0..3: latent panels
      const uint32_t k = tile * 5 + 1 + c;
      if (kProducers > 1 && k % kProducers != who) continue;
      if (tile == 0 && tile0_issued) {
        next_k = k + 1;
        continue;
      }
      uint32_t slot, use, bytes, dst, full, empty;
      int32_t x;
      const CUtensorMap* map;
      if (c < 0) {
        slot = tile % kNumRSlots;
        use = tile / kNumRSlots;
        bytes = G::kRSlotBytes;
        dst = sbase + G::kOffR + slot * G::kRSlotBytes;
        full = smem_u32(&ms->r_full[slot]);
        // With two rope slots and two S buffers, rope slot (tile & 1) is free
        // exactly when the QK of the tile before last has completed, which is
        // the phase of s_full[tile & 1] for that tile.
        empty = smem_u32(&ms->s_full[slot]);
        x = kVDim * G::kElem;
        map = map_r;
      } else {
        const uint32_t g = tile * 4 + c;
        slot = g % G::kNumV;
        use = g / G::kNumV;
        bytes = G::kVSlotBytes;
        dst = sbase + G::kOffV + slot * G::kVSlotBytes;
        full = smem_u32(&ms->v_full[slot]);
        empty = smem_u32(&ms->v_empty[slot]);
        x = 128 * c * G::kElem;
        map = map_v;
      }
      // The maps address the cache as bytes, so x is a byte offset into the row.
      if (kGather) {  // e4m3 only: one 128- or 64-byte-wide panel per slot
        int w = 1;  // every lane waits (see the start gate above)
        if (use > 0) w = wait_phase(empty, (use - 1) & 1, ms, p.err);
        ok = __all_sync(0xffffffffu, w != 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(full, bytes);
        __syncwarp();
        tma_gather4(dst + lane * 4 * (bytes / kTileTokens), map, x, rows[0], rows[1], rows[2],
                    rows[3], full, pol);
      } else {
        // Boxes of one 128-byte-wide panel each: the whole slot for e4m3; for
        // bf16 64 dims, two per latent slot, 16 KB apart.
        const int boxes = G::kSplit || c < 0 ? 1 : 2;
        if (use > 0) ok = wait_phase(empty, (use - 1) & 1, ms, p.err);
        if (!ok) break;
        if (!MLA_DCHECK(tok0 >= 0 && tok0 < p.kv_rows && (x & 15) == 0, p.err)) {
          ms->abort_flag = 1;  // the waiters on this panel see it and give up
          ok = false;
          break;
        }
        if (k == 0) MLA_TRACE_CLK(kTrFirstExpect);
        mbar_arrive_expect_tx(full, bytes);
        for (int i = 0; i < boxes; ++i)
          tma_load_2d(dst + i * kTileTokens * 128, map, x + 128 * i, tok0, full, pol);
      }
      next_k = k + 1;
      if (k == 0 && lane == 0) MLA_TRACE_CLK(kTrFirstCopy);
    }
    if (!ok) break;
    ++tile;
    if (!cursor_next_tile(cur, ms, p.kv_indptr, p.batch)) break;
  }
  // An abandoned call must not leave copies landing in shared memory after
  // exit: wait (bounded) for the last fill issued into every slot; every
  // earlier fill of a slot was consumed before the next one was issued.
  if (lane == 0) ms->next_panel[who] = next_k;
  if (kGather) named_bar_sync(kBarProducers, 32 * kProducers);
  if (who != 0 || lane != 0 || !ms->abort_flag) return;
  uint32_t issued[kProducers];
  uint32_t kmax = 0;
#pragma unroll
  for (uint32_t w = 0; w < kProducers; ++w) {
    issued[w] = ms->next_panel[w];
    kmax = max(kmax, issued[w]);
  }
  uint32_t need_v = (1u << G::kNumV) - 1, need_r = (1u << kNumRSlots) - 1;
  // Holes in the issued set lie within the last ring's worth of panels.
  for (uint32_t n = 0; n < 64 && n < kmax && (need_v | need_r); ++n) {
    const uint32_t k = kmax - 1 - n;
    uint32_t upto = issued[0];
#pragma unroll
    for (uint32_t w = 1; w < kProducers; ++w) upto = k % kProducers == w ? issued[w] : upto;
    if (k >= upto) continue;  // never issued
    const uint32_t t = k / 5;
    const int c = static_cast<int>(k % 5) - 1;
    if (c < 0) {
      const uint32_t slot = t % kNumRSlots;
      if (need_r & (1u << slot)) {
        drain_phase(smem_u32(&ms->r_full[slot]), (t / kNumRSlots) & 1);
        need_r &= ~(1u << slot);
      }
    } else {
      const uint32_t g = t * 4 + c, slot = g % G::kNumV;
      if (need_v & (1u << slot)) {
        drain_phase(smem_u32(&ms->v_full[slot]), (g / G::kNumV) & 1);
        need_v &= ~(1u << slot);
      }
    }
  }
}

// ------------------------------------------------------------ MXFP4 cache (warp 4 producer, warps 8-15 converters)
// Producer (lane 0 of warp 4; contiguous rows only).  Per tile: the rope
// panel's elements (32 bytes a row, 32-byte swizzle) into the upper half of its
// rope slot together with the tile's scale bytes (scale slot tile % 4), then
// each latent panel's elements (64 bytes a row, 64-byte swizzle) into the upper
// half of its latent slot.  A slot is refilled only after the MMAs consumed the
// e4m3 panel converted from its previous fill (which the converters read before
// writing it), exactly as for the e4m3 cache; a scale slot is refilled four
// tiles later, after the QK of two tiles later, so the converters have long
// finished with it.
template <int kQ>
__device__ void run_producer_mx(const Stage1Params& p, const CUtensorMap* map_v,
                                const CUtensorMap* map_r, const CUtensorMap* map_s, Misc* ms,
                                uint32_t sbase) {
  using G = Geo<kQ, Kv::kMx4>;
  if ((threadIdx.x & 31) != 0) return;
  Cursor cur;
  cursor_start(cur, ms);
  if (p.stall_stream) cur.live = false;  // test hook: nothing is ever loaded
  uint32_t tile = 0;
  uint32_t v_fills = 0, r_fills = 0;  // latent / rope panels issued
  const uint64_t pol = cache_policy(p);  // the elements' copies (the scale boxes overlap: unhinted)
  bool ok = true;
  while (cur.live && ok) {
    const int32_t tok0 = cur.kb + cur.j * kTileTokens;
    {
      const uint32_t slot = tile % kNumRSlots, use = tile / kNumRSlots;
      if (use > 0) ok = wait_phase(smem_u32(&ms->s_full[slot]), (use - 1) & 1, ms, p.err);
      if (!ok) break;
      if (!MLA_DCHECK(tok0 >= 0 && tok0 < p.kv_rows, p.err)) {
        ms->abort_flag = 1;
        ok = false;
        break;
      }
      const uint32_t full = smem_u32(&ms->rraw_full[slot]);
      mbar_arrive_expect_tx(full, kTileTokens * 32 + kSclSlotBytes);
      tma_load_2d(sbase + G::kOffR + slot * G::kRSlotBytes + G::kRRawOff, map_r, kVDim / 2, tok0,
                  full, pol);
      const uint32_t sdst = sbase + G::kOffScl + (tile % kNumSclSlots) * kSclSlotBytes;
      const int32_t x0 = (18 * tok0) & ~15;  // the host bounds 18 * kv_rows well below 2^31
#pragma unroll 1
      for (int i = 0; i < kSclBoxes; ++i) tma_load_1d(sdst + 256 * i, map_s, x0 + 256 * i, full);
      r_fills = tile + 1;
      if (tile == 0) MLA_TRACE_CLK(kTrFirstCopy);
    }
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const uint32_t g = tile * 4 + c, slot = g % G::kNumV, use = g / G::kNumV;
      if (use > 0) ok = wait_phase(smem_u32(&ms->v_empty[slot]), (use - 1) & 1, ms, p.err);
      if (!ok) break;
      const uint32_t full = smem_u32(&ms->raw_full[slot]);
      mbar_arrive_expect_tx(full, kTileTokens * 64);
      tma_load_2d(sbase + G::kOffV + slot * G::kVSlotBytes + G::kVRawOff, map_v, 64 * c, tok0, full,
                  pol);
      v_fills = g + 1;
    }
    if (!ok) break;
    ++tile;
    if (!cursor_step<true>(cur, ms, p.kv_indptr, p.batch)) break;
  }
  if (!ms->abort_flag) return;
  // An abandoned call: only the last fill of each slot can still be in flight.
  for (uint32_t n = 0; n < static_cast<uint32_t>(G::kNumV) && n < v_fills; ++n) {
    const uint32_t g = v_fills - 1 - n;
    drain_phase(smem_u32(&ms->raw_full[g % G::kNumV]), (g / G::kNumV) & 1);
  }
  for (uint32_t n = 0; n < static_cast<uint32_t>(kNumRSlots) && n < r_fills; ++n) {
    const uint32_t t = r_fills - 1 - n;
    drain_phase(smem_u32(&ms->rraw_full[t % kNumRSlots]), (t / kNumRSlots) & 1);
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

// Eight E2M1 elements (a 32-bit word, element 0 in the low nibble) times the
// power of two f2 (a half2 pair) -> eight e4m3 codes (element 0 in the low byte).
// Both conversions are the hardware's; the product is exact in half precision.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8(uint32_t w, uint32_t f2) {
  uint32_t h0, h1, h2, h3;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
  asm("mul.rn.f16x2 %0, %0, %4;\n mul.rn.f16x2 %1, %1, %4;\n"
      " mul.rn.f16x2 %2, %2, %4;\n mul.rn.f16x2 %3, %3, %4;"
      : "+r"(h0), "+r"(h1), "+r"(h2), "+r"(h3) : "r"(f2));
  const uint32_t e0 = cvt_f16x2_to_e4m3x2(h0), e1 = cvt_f16x2_to_e4m3x2(h1);
  const uint32_t e2 = cvt_f16x2_to_e4m3x2(h2), e3 = cvt_f16x2_to_e4m3x2(h3);
  return make_uint2(e0 | (e1 << 16), e2 | (e3 << 16));
}

// One 32-element block (16 bytes of elements, scale byte sb) -> 32 e4m3 codes
// e2m1 * 2^(sb - 127 - bias), stored as 16-byte chunks at a0 and a1.  Exact
// while the shift lies in [-8, 6]: e2m1 magnitudes 0.5 ... 6 times 2^shift then
// lie on the e4m3 grid (2^-9 ... 384).  Outside it (or for the NaN scale 0xFF)
// a block holding a nonzero element raises *bad; the codes then saturate at 448
// or round toward zero (a shift below -14 rounds every element to zero, as the
// exact value would).
__device__ __forceinline__ void mx_block_store(uint4 raw, uint32_t sb, int32_t bias, uint32_t a0,
                                               uint32_t a1, int32_t& bad) {
  const int32_t shift = static_cast<int32_t>(sb) - 127 - bias;
  if ((shift < -8 || shift > 6) && (raw.x | raw.y | raw.z | raw.w) != 0) bad = 1;
  const uint32_t f = static_cast<uint32_t>(min(max(shift, -14), 15) + 15) << 10;  // half 2^shift
  const uint32_t f2 = f | (f << 16);
  const uint2 c0 = e2m1x8_to_e4m3x8(raw.x, f2), c1 = e2m1x8_to_e4m3x8(raw.y, f2);
  const uint2 c2 = e2m1x8_to_e4m3x8(raw.z, f2), c3 = e2m1x8_to_e4m3x8(raw.w, f2);
  st_shared_v4(a0, c0.x, c0.y, c1.x, c1.y);
  st_shared_v4(a1, c2.x, c2.y, c3.x, c3.y);
}

// Named-barrier arrival of the converter warps that also ORs a predicate.
__device__ __forceinline__ bool converters_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, %3, pi;"
      " selp.u32 %0, 1, 0, po; }"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)), "r"(kBarConverters), "r"(kConverterWarps * 32)
      : "memory");
  return r != 0;
}

// Converters (warps 8-15): thread t owns row (token) i = t % 128 of every
// panel and its half h = t / 128 (blocks 2h, 2h + 1 of a latent panel, block
// 16 + h of the rope panel).  For each panel, in fill order: wait for its
// elements, load the thread's blocks (and the scale bytes they need), then meet
// the other converters (the vote also ends the call for all of them together
// when a wait gave up); only then write the e4m3 codes over the slot, in the
// swizzled layouts the e4m3 cache's TMA boxes produce (latent rows 128 bytes,
// 128-byte swizzle; rope rows 64 bytes, 64-byte swizzle), and arrive, one lane
// per warp, on the panel's full barrier that the QK issuer waits on.
template <int kQ>
__device__ void run_converter(const Stage1Params& p, Misc* ms, uint32_t sbase) {
  using G = Geo<kQ, Kv::kMx4>;
  const int t = static_cast<int>(threadIdx.x) - kFirstConverterWarp * 32;
  const int i = t & (kTileTokens - 1), h = t >> 7;
  const int lane = threadIdx.x & 31;
  const int32_t bias = p.mx_bias;
  Cursor cur;
  cursor_start(cur, ms);
  uint32_t tile = 0;
  int32_t bad = 0;
  bool stop = !cur.live;
  while (!stop) {
    const int32_t tok0 = cur.kb + cur.j * kTileTokens;
    const uint32_t rslot = tile % kNumRSlots;
    const uint32_t rs = sbase + G::kOffR + rslot * G::kRSlotBytes;
    bool ok = wait_phase(smem_u32(&ms->rraw_full[rslot]), (tile / kNumRSlots) & 1, ms, p.err);
    // The token's scale bytes (the slot stays put until the tile's panels are done).
    const uint32_t sb = sbase + G::kOffScl + (tile % kNumSclSlots) * kSclSlotBytes +
                        ((18 * tok0) & 15) + 18 * i;
    uint32_t sc_rope = 0;
    uint4 rr;
    if (ok) {
      sc_rope = ld_shared_u16(sb + 16);  // blocks 16, 17
      rr = ld_shared_v4(rs + G::kRRawOff + 32 * i + 16 * (h ^ ((i >> 2) & 1)));
    }
    if (converters_bar_or(!ok)) break;
    {  // rope dims 512 + 32 h ... (block 16 + h)
      const uint32_t sw = (i >> 1) & 3;
      mx_block_store(rr, (sc_rope >> (8 * h)) & 0xFFu, bias, rs + 64 * i + 16 * ((2 * h) ^ sw),
                     rs + 64 * i + 16 * ((2 * h + 1) ^ sw), bad);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ms->r_full[rslot]));
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const uint32_t g = tile * 4 + c, slot = g % G::kNumV;
      const uint32_t vs = sbase + G::kOffV + slot * G::kVSlotBytes;
      ok = wait_phase(smem_u32(&ms->raw_full[slot]), (g / G::kNumV) & 1, ms, p.err);
      uint4 lr[2];
      uint32_t sc = 0;  // blocks 4c + 2h, 4c + 2h + 1
      if (ok) {
        sc = ld_shared_u16(sb + 4 * c + 2 * h);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = 2 * h + k;
          lr[k] = ld_shared_v4(vs + G::kVRawOff + 64 * i + 16 * (j ^ ((i >> 1) & 3)));
        }
      }
      if (converters_bar_or(!ok)) {
        stop = true;
        break;
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {  // dims 128 c + 32 j ... (block 4 c + j)
        const int j = 2 * h + k;
        const uint32_t sw = i & 7;
        mx_block_store(lr[k], (sc >> (8 * k)) & 0xFFu, bias, vs + 128 * i + 16 * ((2 * j) ^ sw),
                       vs + 128 * i + 16 * ((2 * j + 1) ^ sw), bad);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms->v_full[slot]));
    }
    if (stop) break;
    ++tile;
    stop = !cursor_step<true>(cur, ms, p.kv_indptr, p.batch);
  }
  if (bad) set_error(p.err, MLA_DERR_MX_SCALE);
}

// ------------------------------------------------------------ MMA issuers (warp 6: QK, warp 5: PV; lane 0)
template <Kv kFmt>
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  if constexpr (kFmt != Kv::kBf16)
    umma_f8(d, a, b, idesc, accumulate);
  else
    umma_f16(d, a, b, idesc, accumulate);
}

// S^T[tile & 1] = K_tile . Q_op^T (Q_op: kN rows, per query token the hi then
// lo heads, or the heads), issued slot by slot as the slots land: first the
// rope slot (64-byte swizzle for e4m3, 128-byte for bf16; it starts the sum),
// then latent slot p (128-byte-swizzled panels), in k-steps of 32 bytes
// (32 e4m3 or 16 bf16 dims).
template <int kQ, Kv kFmt>
__device__ __forceinline__ void issue_qk_rope(uint32_t tmem, uint32_t sbase, uint32_t tile) {
  using G = Geo<kQ, kFmt>;
  const uint32_t d = tmem + G::kColS + G::kN * (tile & 1);
  const uint32_t rs = sbase + G::kOffR + (tile % kNumRSlots) * G::kRSlotBytes;
  constexpr uint32_t kRopeSbo = 8 * G::kRopeWidth;
#pragma unroll
  for (int kk = 0; kk < G::kRopeWidth / 32; ++kk) {
    umma<kFmt>(d, smem_desc(rs + 32 * kk, kRopeSbo, kRopeSbo, G::kRopeLayout),
               smem_desc(sbase + G::kOffQRope + 32 * kk, kRopeSbo, kRopeSbo, G::kRopeLayout),
               G::kIdescQK, kk != 0);
  }
}

template <int kQ, Kv kFmt>
__device__ __forceinline__ void issue_qk_latent(uint32_t tmem, uint32_t sbase, uint32_t tile,
                                                int p) {
  using G = Geo<kQ, kFmt>;
  const uint32_t d = tmem + G::kColS + G::kN * (tile & 1);
  const uint32_t qb = sbase + G::kOffQ;
  const uint32_t vs = sbase + G::kOffV + ((tile * 4 + p) % G::kNumV) * G::kVSlotBytes;
#pragma unroll
  for (int h = 0; h < G::kElem; ++h) {  // 128-byte-wide panels of the slot
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      umma<kFmt>(d, smem_desc(vs + h * kTileTokens * 128 + 32 * kk, 1024, 1024, kLayoutSw128),
                 smem_desc(qb + (p * G::kElem + h) * G::kQPanelBytes + 32 * kk, 1024, 1024,
                           kLayoutSw128),
                 G::kIdescQK, 1);
    }
  }
}

// O^T[chunk c] (+)= V_c^T . P^T over the tile's 128 tokens: latent slot c read
// MN-major (dims contiguous; M = 128 dims is one 128-byte atom of e4m3, or the
// slot's two bf16 panels, 16 KB apart), P read MN-major (a token's P row
// contiguous, one swizzle atom: 32 or 64 bytes), k-steps of 32 e4m3 or 16 bf16
// tokens.  Each latent slot is released as soon as its MMAs complete.
//
// kRolled keeps the loop over latent slots rolled (one copy of a slot's MMAs):
// the issue runs at the MMAs' pace either way, and when the code is not in the
// SM's instruction cache (the first tile of a call whose code left L2) a
// quarter of it is fetched.  Measured: the two-token kernels 3-4 % faster
// throughout, the cluster split's calls 2-3 µs faster with L2 flushed and
// 0.3 µs slower back to back, the one-token persistent kernel 1 % slower at
// bs256, which therefore keeps the unrolled form.
template <int kQ, Kv kFmt, bool kRolled>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t sbase, uint32_t tile, bool first,
                                         Misc* ms) {
  using G = Geo<kQ, kFmt>;
  constexpr int kStepTokens = 32 / G::kElem;
  constexpr uint32_t kLbo = G::kSplit ? 1024 : kTileTokens * 128;
  const uint32_t pb = sbase + G::kOffP + (tile & 1) * G::kPBytes;
  if constexpr (!kRolled) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t g = tile * 4 + c;
      const uint32_t slot = g % G::kNumV;
      const uint32_t vs = sbase + G::kOffV + slot * G::kVSlotBytes;
#pragma unroll
      for (int kk = 0; kk < kTileTokens / kStepTokens; ++kk) {
        umma<kFmt>(tmem + G::kColO + G::kN * c,
                   smem_desc(vs + kk * kStepTokens * 128, kLbo, 1024, kLayoutSw128),
                   smem_desc(pb + kk * kStepTokens * G::kPRowBytes, 8 * G::kPRowBytes,
                             8 * G::kPRowBytes, G::kPLayout),
                   G::kIdescPV, !(first && kk == 0));
      }
      umma_commit(smem_u32(&ms->v_empty[slot]));
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const uint32_t g = tile * 4 + c;
      const uint32_t slot = g % G::kNumV;
      const uint32_t vs = sbase + G::kOffV + slot * G::kVSlotBytes;
#pragma unroll
      for (int kk = 0; kk < kTileTokens / kStepTokens; ++kk) {
        umma<kFmt>(tmem + G::kColO + G::kN * c,
                   smem_desc(vs + kk * kStepTokens * 128, kLbo, 1024, kLayoutSw128),
                   smem_desc(pb + kk * kStepTokens * G::kPRowBytes, 8 * G::kPRowBytes,
                             8 * G::kPRowBytes, G::kPLayout),
                   G::kIdescPV, !(first && kk == 0));
      }
      umma_commit(smem_u32(&ms->v_empty[slot]));
    }
  }
}

// Bounded spin until a monotonic shared counter reaches `target`; false when
// the call is being abandoned.  The caller follows a true return with
// fence_acquire_cta, which orders what the counter's writer published.
__device__ __noinline__ bool spin_counter_slow(const uint32_t* ctr, uint32_t target, Misc* ms,
                                               int32_t* err) {
  const long long start = clock64();
  for (uint32_t n = 1;; ++n) {
    if (ld_relaxed_u32(ctr) >= target) return true;
    if ((n & 15) == 0) {
      if (ms->abort_flag) return false;
      if (clock64() - start > kWaitLimitCycles) {
        ms->abort_flag = 1;
        set_error(err, MLA_DERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool spin_counter(const uint32_t* ctr, uint32_t target, Misc* ms,
                                             int32_t* err) {
  if (ld_relaxed_u32(ctr) >= target) return true;
  return spin_counter_slow(ctr, target, ms, err);
}

// The same wait on a counter of every softmax warpgroup (two in the
// two-token kernels on contiguous rows).
template <bool kDual>
__device__ __forceinline__ bool spin_groups(const uint32_t (&ctr)[2], uint32_t target, Misc* ms,
                                            int32_t* err) {
  return spin_counter(&ctr[0], target, ms, err) && (!kDual || spin_counter(&ctr[1], target, ms, err));
}

// Two threads issue tcgen05.mma, each for one product, so that neither
// product's issue waits behind the other's (issuing one product blocks the
// issuing thread for about its execution time, ~1200 cycles).
//
// QK issuer (warp 6, lane 0): QK of tile i needs S[i & 1] read out by the
// softmax of tile i - 2; then each of its five slots is multiplied as soon as
// its copy has landed (the issuer waits on the TMA barriers itself), so that
// the products overlap the copies still in flight, and, on the first tile of a
// segment, as soon as the matching part of the segment's Q operand is written.
template <bool kGather, int kQ, Kv kFmt, bool kRolled, bool kDual>
__device__ void run_mma_qk(const Stage1Params& p, Misc* ms, uint32_t sbase, uint32_t tmem) {
  using G = Geo<kQ, kFmt>;
  Cursor qc;
  cursor_start(qc, ms);
  uint32_t qk_n = 0;  // tiles whose QK has been issued
  const uint32_t qbars = smem_u32(&ms->q_part[0]);
  while (qc.live) {
    bool ok = true;
    // The segment's Q operand (one barrier phase per segment), on its first
    // tile: part by part with the rolled issue loops (each part just before
    // its products), whole otherwise (the last part's phase).
    const bool qwait = qc.j == qc.j0;
    const uint32_t qpar = static_cast<uint32_t>(qc.seg) & 1;
    const bool by_part = q_split(kRolled, kGather, p);
    if (!by_part && qwait) ok = wait_phase(qbars + 8 * (kQParts - 1), qpar, ms, p.err);
    if (ok && qk_n >= 2) ok = spin_groups<kDual>(ms->s_read, qk_n - 1, ms, p.err);
    if (ok) fence_acquire_cta();
    if (ok) ok = wait_phase(smem_u32(&ms->r_full[qk_n % kNumRSlots]), (qk_n / kNumRSlots) & 1, ms,
                            p.err);
    if (by_part && ok && qwait) ok = wait_phase(qbars, qpar, ms, p.err);
    if (!ok) break;
    if (qk_n == 0) MLA_TRACE_CLK(kTrRopeLanded);
    tc_fence_after();
    issue_qk_rope<kQ, kFmt>(tmem, sbase, qk_n);
    // each latent slot as soon as its copy has landed (rolled: see issue_pv)
    auto latent = [&](int c) {
      const uint32_t g = qk_n * 4 + c;
      if (!wait_phase(smem_u32(&ms->v_full[g % G::kNumV]), (g / G::kNumV) & 1, ms, p.err)) return false;
      if (by_part && qwait && !wait_phase(qbars + 8 * (1 + c), qpar, ms, p.err)) return false;
      tc_fence_after();
      issue_qk_latent<kQ, kFmt>(tmem, sbase, qk_n, c);
      return true;
    };
    if constexpr (kRolled) {
#pragma unroll 1
      for (int c = 0; c < 4 && ok; ++c) ok = latent(c);
    } else {
      for (int c = 0; c < 4 && ok; ++c) {
        const uint32_t g = qk_n * 4 + c;
        ok = wait_phase(smem_u32(&ms->v_full[g % G::kNumV]), (g / G::kNumV) & 1, ms, p.err);
        if (!ok) break;
        tc_fence_after();
        issue_qk_latent<kQ, kFmt>(tmem, sbase, qk_n, c);
      }
    }
    if (!ok) break;
    umma_commit(smem_u32(&ms->s_full[qk_n & 1]));  // also frees rope slot qk_n & 1
    if (qc.j + 1 == qc.j1) umma_commit(smem_u32(&ms->q_empty));
    if (qk_n == 0) MLA_TRACE_CLK(kTrQkIssued);
    ++qk_n;
    cursor_step<kFmt == Kv::kMx4>(qc, ms, p.kv_indptr, p.batch);
  }
  // Every MMA issued by this thread completes before TMEM is released.
  umma_commit(smem_u32(&ms->mma_done));
}

// PV issuer (warp 5, lane 0): PV of tile i needs P[i & 1] published and, on
// the first tile of a later segment, O read out by the previous segment's
// epilogue.
template <int kQ, Kv kFmt, bool kRolled, bool kDual>
__device__ void run_mma_pv(const Stage1Params& p, Misc* ms, uint32_t sbase, uint32_t tmem) {
  Cursor pc;
  cursor_start(pc, ms);
  uint32_t pv_n = 0;  // tiles whose PV has been issued
  while (pc.live) {
    const bool first = pc.j == pc.j0;
    bool ok = spin_groups<kDual>(ms->p_ready, pv_n + 1, ms, p.err);
    if (ok && first && pc.seg > 0) ok = spin_groups<kDual>(ms->o_free, static_cast<uint32_t>(pc.seg), ms, p.err);
    if (!ok) break;
    fence_acquire_cta();
    tc_fence_after();
    issue_pv<kQ, kFmt, kRolled>(tmem, sbase, pv_n, first, ms);
    umma_commit(smem_u32(&ms->pv_done[pv_n & 1]));
    if (pv_n == 0) MLA_TRACE_CLK(kTrPvIssued);
    if (first && pc.seg == 1) MLA_TRACE_CLK(kTrPvIssued1);
    ++pv_n;
    cursor_step<kFmt == Kv::kMx4>(pc, ms, p.kv_indptr, p.batch);
  }
  umma_commit(smem_u32(&ms->mma_done));
}

// ------------------------------------------------------------ softmax warps (0-3)
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Sum of v[h] over the 32 lanes of the warp, returned for head (lane >> 1) & 15:
// four halving exchanges move half of the heads to the partner lane each time.
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 8, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? v[k] : v[k + half];
      const float keep = up ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Byte address of 16-byte chunk `ch` of operand row `row` in the Q operand:
// latent dims in 128-byte-swizzled panels, rope dims in one more panel (64-byte
// swizzle for e4m3; for bf16 it is the ninth 128-byte panel).
template <int kQ, Kv kFmt>
__device__ __forceinline__ uint32_t q_chunk_addr(uint32_t sq, int row, int ch) {
  using G = Geo<kQ, kFmt>;
  if (!G::kSplit || ch < 32) {
    const int panel = ch >> 3, cc = ch & 7;
    return sq + panel * G::kQPanelBytes + row * 128 + ((cc ^ (row & 7)) << 4);
  }
  const int cc = ch - 32;
  return sq + 4 * G::kQPanelBytes + row * 64 + ((cc ^ ((row >> 1) & 3)) << 4);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// The Q operand is written in parts, in the order the QK issuer multiplies
// them: part 0 the rope dims 512..575, part 1 + c the latent dims 128c ..
// 128c + 127.  Each part has an mbarrier (Misc::q_part, one phase per segment)
// that every softmax thread arrives on once its share of the part is written
// and made visible to the tensor core's proxy, so that the first MMAs of a
// segment run while later parts are still being converted.  In round r thread
// t (of 128) takes one 16-dim chunk (ch) of one head of each of its tokens.
// By parts (`panel`): rope chunk 32 + t % 4 of head t / 4 (threads 0-63), or
// latent chunk 8 (r - 1) + t % 8 of head t / 8.  Otherwise the 16 x 36 chunks
// in order, t + 128 r, which measured faster for the page-table kernel (the
// ragged step 76.5 -> 74.4 us).
__device__ __forceinline__ bool q_job(int t, int r, bool panel, int& head, int& ch) {
  if (!panel) {
    const int job = t + 128 * r;
    head = job / 36;
    ch = job % 36;
    return job < 576;
  }
  if (r == 0) {
    head = t >> 2;
    ch = 32 + (t & 3);
    return t < 64;
  }
  head = t >> 3;
  ch = 8 * (r - 1) + (t & 7);
  return true;
}
// Arrive on part r's barrier (bars: the first of Misc::q_part, or 0 for none).
// Without `split` a thread arrives once, on the last part, after all of its
// share, and the issuer waits for the whole operand: where the issue loops are
// unrolled (one proxy fence per segment instead of five measured faster
// there) and with a page table.  A thread arrives on the parts in order, so the
// last part's phase completes only after every part's.  q_split is the one
// rule both sides apply.
__device__ __forceinline__ void q_part_done(uint32_t bars, int r, bool split) {
  if (bars == 0 || (!split && r != kQParts - 1)) return;
  fence_proxy_async_smem();
  mbar_arrive(bars + 8 * r);
}

// Two-term e4m3 split of 16 floats x (|x| <= 448): hi = e4m3(x), lo = e4m3(16 (x - hi)),
// so x ~= hi + lo / 16 with about 8 significant bits.  Packs codes 4 per word.
__device__ __forceinline__ void split_e4m3_16(const float (&x)[16], uint32_t (&hi)[4],
                                              uint32_t (&lo)[4]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint16_t h2 = cvt_e4m3x2(x[2 * k], x[2 * k + 1]);
    const uint32_t hf = cvt_e4m3x2_to_f16x2(h2);
    const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hf));
    const uint16_t l2 = cvt_e4m3x2((x[2 * k] - hv.x) * 16.0f, (x[2 * k + 1] - hv.y) * 16.0f);
    if (k & 1) {
      hi[k >> 1] |= static_cast<uint32_t>(h2) << 16;
      lo[k >> 1] |= static_cast<uint32_t>(l2) << 16;
    } else {
      hi[k >> 1] = h2;
      lo[k >> 1] = l2;
    }
  }
}

// Q operand rows of a bf16 cache: the bf16 values themselves, row 16 qi + head.
template <int kQ, int kQt>
__device__ __forceinline__ void store_q_bf16(uint32_t sq, const uint4 (&raw)[kQt][5][2],
                                             float (&qk_scale)[kQt], const SoftmaxGroup& sg,
                                             uint32_t bars, bool panel, bool split) {
  const int t = sg.t;
  named_bar_sync(sg.pair, sg.pair_threads);
#pragma unroll
  for (int i = 0; i < kQt; ++i) qk_scale[i] = kSmScaleLog2;
#pragma unroll
  for (int r = 0; r < kQParts; ++r) {
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
      const int qi = sg.q0 + i;
      int head, ch;  // ch: 16 dims = two 16-byte chunks
      if (q_job(t, r, panel, head, ch)) {
        const uint4 a = raw[i][r][0], b = raw[i][r][1];
        st_shared_v4(q_chunk_addr<kQ, Kv::kBf16>(sq, 16 * qi + head, 2 * ch), a.x, a.y, a.z, a.w);
        st_shared_v4(q_chunk_addr<kQ, Kv::kBf16>(sq, 16 * qi + head, 2 * ch + 1), b.x, b.y, b.z, b.w);
      }
    }
    q_part_done(bars, r, split);
  }
  fence_proxy_async_smem();
  named_bar_sync(sg.bar, kSoftmaxThreads);
}

// Q operand rows of an e4m3 cache: each query token scaled by a power of two so
// its largest magnitude lands in (224, 448], then split into hi / lo e4m3 rows
// (32 qi + head for hi, 32 qi + 16 + head for lo).
template <int kQ, int kQt>
__device__ __forceinline__ void store_q_e4m3(Misc* ms, uint32_t sq, const uint4 (&raw)[kQt][5][2],
                                             float kv_scale, float (&qk_scale)[kQt],
                                             const SoftmaxGroup& sg, uint32_t bars, int seg, bool panel,
                                             bool split) {
  const int t = sg.t, warp = t >> 5, lane = t & 31;
#pragma unroll
  for (int i = 0; i < kQt; ++i) {
    const int qi = sg.q0 + i;
    uint32_t amax = 0;
    auto fold = [&](uint32_t w) { amax = max(amax, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu)); };
#pragma unroll
    for (int r = 0; r < 5; ++r) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        fold(raw[i][r][k].x);
        fold(raw[i][r][k].y);
        fold(raw[i][r][k].z);
        fold(raw[i][r][k].w);
      }
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    if (t == 0 && qi == 0 && seg == 0 && amax != 0xFFFFFFFFu) MLA_TRACE_CLK(kTrQLoaded);
    if (t == 0 && qi == 0 && seg == 1 && amax != 0xFFFFFFFFu) MLA_TRACE_CLK(kTrQLoaded1);
    if (lane == 0) ms->red_u32[4 * qi + warp] = amax;
  }
  named_bar_sync(sg.pair, sg.pair_threads);
  float up[kQt];
#pragma unroll
  for (int i = 0; i < kQt; ++i) {
    const int qi = sg.q0 + i;
    const uint32_t amax = max(max(ms->red_u32[4 * qi], ms->red_u32[4 * qi + 1]),
                              max(ms->red_u32[4 * qi + 2], ms->red_u32[4 * qi + 3]));
    const float a = __uint_as_float(amax << 16);
    int k2 = 0;
    if (a > 0.0f) {
      int e;
      const float f = frexpf(a, &e);  // a = f * 2^e, f in [0.5, 1)
      k2 = (f <= 0.875f) ? 9 - e : 8 - e;
      k2 = min(max(k2, -126), 126);
    }
    up[i] = __int_as_float((k2 + 127) << 23);
    qk_scale[i] = __int_as_float((127 - k2) << 23) * kv_scale * kSmScaleLog2;
  }
#pragma unroll
  for (int r = 0; r < kQParts; ++r) {
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
      const int qi = sg.q0 + i;
      int head, ch;
      if (q_job(t, r, panel, head, ch)) {
        float x[16];
        auto unpack = [&](uint32_t w, int k) {
          x[2 * k] = u2f(w << 16) * up[i];
          x[2 * k + 1] = u2f(w & 0xFFFF0000u) * up[i];
        };
        unpack(raw[i][r][0].x, 0); unpack(raw[i][r][0].y, 1);
        unpack(raw[i][r][0].z, 2); unpack(raw[i][r][0].w, 3);
        unpack(raw[i][r][1].x, 4); unpack(raw[i][r][1].y, 5);
        unpack(raw[i][r][1].z, 6); unpack(raw[i][r][1].w, 7);
        uint32_t hi[4], lo[4];
        split_e4m3_16(x, hi, lo);
        st_shared_v4(q_chunk_addr<kQ, Kv::kE4m3>(sq, 32 * qi + head, ch), hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(q_chunk_addr<kQ, Kv::kE4m3>(sq, 32 * qi + 16 + head, ch), lo[0], lo[1], lo[2], lo[3]);
      }
    }
    q_part_done(bars, r, split);
  }
  // (every thread has read the |q| maxima before red_u32 is used again)
  fence_proxy_async_smem();
  named_bar_sync(sg.bar, kSoftmaxThreads);
}

// Loads the row's query tokens tq + q0 .. tq + q0 + kQt - 1 of the nq this CTA
// takes (16 heads x 576 bf16 each; tokens past nq give zero operand rows) and
// writes their rows of the Q operand of the cache format (kQ token columns).
// Sets qk_scale[i], the factor turning the QK accumulator of token q0 + i into
// base-2 softmax exponent units.  tq < 0 writes a zero query.  This thread's
// share of each token goes into registers first: in round r (q_job) one
// 16-dim chunk of one head.
template <int kQt>
__device__ __forceinline__ void load_q(const Stage1Params& p, int t, int32_t tq, int32_t nq, int q0,
                                       bool panel, uint4 (&raw)[kQt][5][2]) {
#pragma unroll
  for (int i = 0; i < kQt; ++i) {
    const int qi = q0 + i;
#pragma unroll
    for (int r = 0; r < kQParts; ++r) {
      raw[i][r][0] = raw[i][r][1] = make_uint4(0, 0, 0, 0);
      int head, ch;
      if (q_job(t, r, panel, head, ch) && tq >= 0 && qi < nq && MLA_DCHECK(tq + qi < total_tokens(p), p.err)) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<size_t>(tq + qi) * kNumHeads + head) * kQkDim + ch * 16);
        raw[i][r][0] = __ldg(src);
        raw[i][r][1] = __ldg(src + 1);
      }
    }
  }
}

// bars: the first of the Q part barriers to arrive on (0: none); seg: the
// segment this operand serves (for the trace stamps); panel / split: the chunk
// order and the publication by parts (q_job, q_part_done).
template <int kQ, int kQt, Kv kFmt>
__device__ void prepare_q(const Stage1Params& p, Misc* ms, uint32_t sq, int32_t tq, int32_t nq,
                          float kv_scale, float (&qk_scale)[kQt], const SoftmaxGroup& sg,
                          uint32_t bars, int seg, bool panel, bool split) {
  const bool lead = sg.t == 0 && sg.q0 == 0;
  if (lead && seg == 1) MLA_TRACE_CLK(kTrQStart1);
  uint4 raw[kQt][5][2];
  load_q<kQt>(p, sg.t, tq, nq, sg.q0, panel, raw);
  if (lead && seg == 0) MLA_TRACE_CLK(kTrQIssued);
  // The previous segment's output rows may still be leaving the Q region
  // through bulk stores (the loads above are already in flight); the barrier
  // in the store below (both warpgroups', when there are two) orders every
  // write to it after these waits.
  if (sg.t == 0) bulk_wait_read<0>();
  if constexpr (kFmt == Kv::kBf16)
    store_q_bf16<kQ, kQt>(sq, raw, qk_scale, sg, bars, panel, split);
  else
    store_q_e4m3<kQ, kQt>(ms, sq, raw, kv_scale, qk_scale, sg, bars, seg, panel, split);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named-barrier arrival of the softmax warpgroup that also ORs a predicate.
__device__ __forceinline__ bool softmax_bar_or(bool v, uint32_t bar) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, %3, pi;"
      " selp.u32 %0, 1, 0, po; }"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)), "r"(bar), "r"(kSoftmaxThreads) : "memory");
  return r != 0;
}

// Two-term e4m3 split of 16 probabilities (0 <= p <= 256) via packed half2:
// hi = e4m3(p), lo = e4m3(16 (p - hi)).
__device__ __forceinline__ void split_p_16(const float (&x)[16], uint32_t (&hi)[4],
                                           uint32_t (&lo)[4]) {
  const __half2 sixteen = __float2half2_rn(16.0f);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __half2 p2 = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
    const uint16_t h8 = cvt_f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t*>(&p2));
    const uint32_t hb = cvt_e4m3x2_to_f16x2(h8);
    const __half2 r = __hmul2(__hsub2(p2, *reinterpret_cast<const __half2*>(&hb)), sixteen);
    const uint16_t l8 = cvt_f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t*>(&r));
    if (k & 1) {
      hi[k >> 1] |= static_cast<uint32_t>(h8) << 16;
      lo[k >> 1] |= static_cast<uint32_t>(l8) << 16;
    } else {
      hi[k >> 1] = h8;
      lo[k >> 1] = l8;
    }
  }
}

// The 16 heads' accumulator values of query token qi in TMEM columns `col`
// onward: e4m3 operands give hi and lo columns, combined as hi + lo / 16; bf16
// operands one column per head.
template <Kv kFmt>
__device__ __forceinline__ void tmem_ld_heads(uint32_t addr, float (&v)[16]) {
  if constexpr (kFmt != Kv::kBf16) {
    uint32_t r[32];
    tmem_ld32(addr, r);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 16; ++h) v[h] = fmaf(u2f(r[16 + h]), 0.0625f, u2f(r[h]));
  } else {
    uint32_t r[16];
    tmem_ld16(addr, r);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 16; ++h) v[h] = u2f(r[h]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// kInlineWaits: the waits' slow paths inlined (required where setmaxnreg raised
// the register count: a call out of such a region does not compile).
// kGroups softmax warpgroups share the CTA's query tokens: warpgroup g (warps
// 0-3, and 8-11 for g = 1) owns token columns g kQt .. g kQt + kQt - 1 of the
// kQ, reads their S columns, writes their P chunks and Q rows and their O
// columns, and publishes its own progress counters; the MMA issuers wait for
// every warpgroup's.
template <bool kGather, int kQ, Kv kFmt, bool kInlineWaits, bool kCluster, int kGroups>
__device__ void run_softmax(const Stage1Params& p, Misc* ms, uint32_t sbase, uint32_t tmem,
                            float kv_scale, int g) {
  using G = Geo<kQ, kFmt>;
  static_assert(kGroups == 1 || (kGroups == 2 && kQ == 2 && !kCluster), "two warpgroups take one token each");
  constexpr int kQt = kQ / kGroups;  // token columns of this warpgroup
  // The Q operand is published part by part where the QK issuer's loops are
  // rolled (two tokens, or the cluster split) on contiguous rows, whole
  // otherwise; its chunks go by parts except with a page table (q_job,
  // q_part_done).
  const bool q_panel = q_panel_order(kGather, p);
  const bool q_by_part = q_split(kQ == 2 || kCluster, kGather, p);
  const SoftmaxGroup sg{static_cast<int>(threadIdx.x) - 256 * g, g * kQt,
                        g ? kBarSoftmaxB : kBarSoftmax, kGroups == 2 ? kBarSoftmaxPair : kBarSoftmax,
                        kGroups == 2 ? 2u * kSoftmaxThreads : kSoftmaxThreads};
  const int t = sg.t, warp = t >> 5, lane = t & 31, q0 = sg.q0;
  const bool lead = t == 0 && g == 0;  // trace stamps
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;  // TMEM lane quarter
  const int token = warp * 32 + lane;  // S row (token) / O row (dim within a chunk) of this thread
  const int32_t c = cta_worker(p);
  const int32_t q_off = cta_q_off(p);   // the row's first query token this CTA handles
  const int32_t nq = kQ == 1 ? 1 : cta_tokens<kQ>(p);  // and how many (the rest of the kQ columns idle)
  const int32_t slot_q = q_off - p.q_off;  // their first index within a partial slot

  if (lead) MLA_TRACE_CLK(kTrSoftmaxStart);
  Cursor cur;
  cursor_start(cur, ms);
  uint32_t tile = 0;                 // tiles processed by this CTA
  uint32_t pv_seen[2] = {0, 0};      // pv_done[b] phases consumed

  // Wait until the PV of tile k has completed (phases are consumed in order).
  auto wait_pv = [&](uint32_t k) {
    const uint32_t b = k & 1;
    while (pv_seen[b] <= (k >> 1)) {
      softmax_wait<kInlineWaits>(smem_u32(&ms->pv_done[b]), pv_seen[b] & 1, ms, p.err);
      ++pv_seen[b];
    }
  };

  // A segment's Q operand is normally prepared at its start; with one query
  // token per CTA, after a split piece (whose epilogue uses no shared memory)
  // the next segment's is prepared before that epilogue instead, so that its
  // first QKs overlap the epilogue.
  bool q_early = false;
  int32_t tq_early = -1;
  float qk_scale[kQt];
  while (cur.live) {
    // ------------------------------------------------ segment start
    const int32_t b = cur.b;
    // This launch's first query token of the row.
    const int32_t tq = q_early ? tq_early
                               : (cur.seg == 0 ? ms->first_tq
                                               : row_token(p, q_off, ldg_i32(p.qo_indptr + b),
                                                           ldg_i32(p.qo_indptr + b + 1)));
    const bool row_ok = tq >= 0;
    if (!row_ok && t == 0) set_error(p.err, MLA_DERR_QO_INDPTR);
    if (!q_early) {
      if (cur.seg > 0) softmax_wait<kInlineWaits>(smem_u32(&ms->q_empty), (cur.seg - 1) & 1, ms, p.err);
      prepare_q<kQ, kQt, kFmt>(p, ms, sbase + G::kOffQ, row_ok ? tq : -1, nq, kv_scale, qk_scale, sg,
                               smem_u32(&ms->q_part[0]), cur.seg, q_panel, q_by_part);
      if (lead && cur.seg == 0) MLA_TRACE_CLK(kTrQReady);
      if (lead && cur.seg == 1) MLA_TRACE_CLK(kTrQReady1);
    }
    q_early = false;

    float m_ref[kQt][16], l[kQt][16];
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m_ref[i][h] = -INFINITY;
        l[i][h] = 0.0f;
      }
    }
    const uint32_t seg_first_tile = tile;
    // Query token i of the row's n sees its first len - n + 1 + i tokens
    // (causal, aligned to the end of the row; for n = 1 the whole row); this
    // launch's token qi is token q_off + qi and sees vis0 + qi of them.
    const int32_t vis0 = cur.len - p.row_tokens + 1 + q_off;

    // ------------------------------------------------ tiles
    for (;;) {
      const uint32_t sb = tile & 1;
      softmax_wait<kInlineWaits>(smem_u32(&ms->s_full[sb]), (tile >> 1) & 1, ms, p.err);
      tc_fence_after();
      const int32_t pos = cur.j * kTileTokens + token;  // row-local token of this thread
      bool tok_ok[kQt];
      float s[kQt][16];
      bool exceed = false;
#pragma unroll
      for (int i = 0; i < kQt; ++i) {
        const int qi = q0 + i;
        const uint32_t addr = tmem + lane_base + G::kColS + G::kN * sb + G::kTokCols * qi;
        tok_ok[i] = qi < nq && pos < vis0 + qi;
        const float sc = qk_scale[i];
        if constexpr (G::kSplit) {
          uint32_t r[32];
          tmem_ld32(addr, r);
          tmem_wait_ld();
          const float sc_lo = sc * 0.0625f;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            s[i][h] = tok_ok[i] ? fmaf(u2f(r[16 + h]), sc_lo, u2f(r[h]) * sc) : -INFINITY;
            exceed |= s[i][h] > m_ref[i][h] + kRescaleThreshold;
          }
        } else {
          uint32_t r[16];
          tmem_ld16(addr, r);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            s[i][h] = tok_ok[i] ? u2f(r[h]) * sc : -INFINITY;
            exceed |= s[i][h] > m_ref[i][h] + kRescaleThreshold;
          }
        }
      }
      tc_fence_before();
      if (lead && tile == 0) MLA_TRACE_CLK(kTrSRead);
      if (lead && cur.seg == 1 && tile == seg_first_tile) MLA_TRACE_CLK(kTrSRead1);

      // The reference maximum moves only when some score exceeds it by more
      // than the threshold (always on a segment's first tile); then the tile
      // maximum per column is reduced over the 128 tokens.
      bool moved = false;
      const bool any_exceed = softmax_bar_or(exceed, sg.bar);
      // Every warp of this warpgroup has read S[sb] (its tcgen05.ld completed before the barrier).
      if (t == 0) st_release_u32(&ms->s_read[g], tile + 1);
      if (any_exceed) {
        float mx[kQt][16];
#pragma unroll
        for (int i = 0; i < kQt; ++i) {
#pragma unroll
          for (int h = 0; h < 16; ++h) mx[i][h] = warp_max(s[i][h]);
        }
        if (lane == 0) {
          float4* dst = reinterpret_cast<float4*>(&ms->red_max[sb][warp][0]);
#pragma unroll
          for (int i = 0; i < kQt; ++i) {
            const int qi = q0 + i;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[4 * qi + k] = make_float4(mx[i][4 * k], mx[i][4 * k + 1], mx[i][4 * k + 2],
                                            mx[i][4 * k + 3]);
          }
        }
        named_bar_sync(sg.bar, kSoftmaxThreads);
#pragma unroll
        for (int i = 0; i < kQt; ++i) {
          const int qi = q0 + i;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float4 m4 = reinterpret_cast<const float4*>(&ms->red_max[sb][0][0])[4 * qi + k];
#pragma unroll
            for (int w = 1; w < 4; ++w) {
              const float4 o4 = reinterpret_cast<const float4*>(&ms->red_max[sb][w][0])[4 * qi + k];
              m4.x = fmaxf(m4.x, o4.x); m4.y = fmaxf(m4.y, o4.y);
              m4.z = fmaxf(m4.z, o4.z); m4.w = fmaxf(m4.w, o4.w);
            }
            mx[i][4 * k] = m4.x; mx[i][4 * k + 1] = m4.y;
            mx[i][4 * k + 2] = m4.z; mx[i][4 * k + 3] = m4.w;
          }
          // The O rescale factors go to shared memory (every thread computes
          // the same ones), so that they hold no registers across the P work.
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            float alpha = 1.0f;
            if (mx[i][h] > m_ref[i][h] + kRescaleThreshold) {
              alpha = fast_exp2(m_ref[i][h] - mx[i][h]);  // 0 on a segment's first tile
              m_ref[i][h] = mx[i][h];
              l[i][h] *= alpha;
              moved = true;
            }
            if (t == 0) ms->alpha_stage[16 * qi + h] = alpha;
          }
        }
      }
      const bool rescale_o = moved && tile != seg_first_tile;

      // P row chunks of query token qi: e4m3 hi then lo (16 bytes each), or the
      // bf16 values of heads 0-7 then 8-15.
      uint32_t phi[kQt][4], plo[kQt][4];
#pragma unroll
      for (int i = 0; i < kQt; ++i) {
        float pr[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          pr[h] = tok_ok[i] ? fast_exp2(s[i][h] - m_ref[i][h]) : 0.0f;
          l[i][h] += pr[h];
        }
        if constexpr (G::kSplit) {
          split_p_16(pr, phi[i], plo[i]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            phi[i][k] = pack_bf16x2(pr[2 * k], pr[2 * k + 1]);
            plo[i][k] = pack_bf16x2(pr[8 + 2 * k], pr[9 + 2 * k]);
          }
        }
      }

      // P[sb] was last read by the PV of tile - 2.
      if (tile >= 2) wait_pv(tile - 2);
      {
        // One P row per token: 32 kQ bytes, two 16-byte chunks per query token
        // swizzled as the 32- or 64-byte atom requires.
        const uint32_t pa = sbase + G::kOffP + sb * G::kPBytes + token * G::kPRowBytes;
        const uint32_t sw = kQ == 1 ? (token >> 2) & 1 : (token >> 1) & 3;
#pragma unroll
        for (int i = 0; i < kQt; ++i) {
          const int qi = q0 + i;
          st_shared_v4(pa + (((2 * qi) ^ sw) << 4), phi[i][0], phi[i][1], phi[i][2], phi[i][3]);
          st_shared_v4(pa + (((2 * qi + 1) ^ sw) << 4), plo[i][0], plo[i][1], plo[i][2], plo[i][3]);
        }
      }
      fence_proxy_async_smem();
      if (rescale_o) {  // the same for every softmax thread
        // O must hold every earlier tile before it is rescaled.
        wait_pv(tile - 1);
        named_bar_sync(sg.bar, kSoftmaxThreads);  // thread 0's alpha_stage is written
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int i = 0; i < kQt; ++i) {
            const int qi = q0 + i;
            const uint32_t addr = tmem + lane_base + G::kColO + G::kN * cc + G::kTokCols * qi;
            if constexpr (G::kSplit) {
              uint32_t o[32];
              tmem_ld32(addr, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(u2f(o[j]) * ms->alpha_stage[16 * qi + (j & 15)]);
              tmem_st32(addr, o);
            } else {
              uint32_t o[16];
              tmem_ld16(addr, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(u2f(o[j]) * ms->alpha_stage[16 * qi + j]);
              tmem_st16(addr, o);
            }
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      named_bar_sync(sg.bar, kSoftmaxThreads);
      if (t == 0) st_release_u32(&ms->p_ready[g], tile + 1);
      if (lead && tile == 0) MLA_TRACE_CLK(kTrPReady);
      if (lead && cur.seg == 1 && tile == seg_first_tile) MLA_TRACE_CLK(kTrPReady1);
      if (lead && cur.seg == 0 && cur.j + 1 == cur.j1) MLA_TRACE_CLK(kTrPLast0);
      ++tile;
      if (cur.j + 1 == cur.j1) break;
      ++cur.j;
    }

    // ------------------------------------------------ next segment's Q, early
    // (one query token per CTA: with two, the early preparation measured slower,
    // 70.8 -> 82.9 us of stage 1 on bs64 with two tokens per row)
    if (kQ == 1 && !cur.whole) {
      Cursor nxt = cur;
      if (cursor_next_tile(nxt, ms, p.kv_indptr, p.batch)) {
        tq_early = row_token(p, q_off, ldg_i32(p.qo_indptr + nxt.b), ldg_i32(p.qo_indptr + nxt.b + 1));
        // the QK of this segment's last tile has released the Q region
        softmax_wait<kInlineWaits>(smem_u32(&ms->q_empty), cur.seg & 1, ms, p.err);
        prepare_q<kQ, kQt, kFmt>(p, ms, sbase + G::kOffQ, tq_early, nq, kv_scale, qk_scale, sg,
                                 smem_u32(&ms->q_part[0]), cur.seg + 1, q_panel, q_by_part);
        if (lead && cur.seg == 0) MLA_TRACE_CLK(kTrQReady1);
        q_early = true;
      }
    }

    // ------------------------------------------------ segment epilogue
    // A row held whole leaves through the TMA engine (staged in the Q region,
    // free once the segment's last PV has completed; one bulk store); a split
    // piece leaves through every thread's own global stores.  Neither waits
    // for its stores to drain before the next segment.
    if ((kQ > 1 || cur.whole) && cur.next_a < ms->t1 && b + 1 < p.batch) {
      // More segments follow: bring the next row's query into L2 now, so that
      // its Q preparation after this epilogue reads it from there.
      const int32_t tq_next = ldg_i32(p.qo_indptr + b + 1) + q_off;
      if (tq_next >= 0 && tq_next <= p.batch * p.row_tokens - kQ) {
        const char* qn = reinterpret_cast<const char*>(p.q + static_cast<size_t>(tq_next) * kNumHeads * kQkDim);
        for (int i = t; i < kQ * kNumHeads * kQkDim * 2 / 128; i += kSoftmaxThreads) prefetch_l2(qn + 128 * i);
      }
    }
    if (t == 0) ms->red_u32[8 + g] = static_cast<uint32_t>(ms->abort_flag);
    float l_tot[kQt][16];
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
      float v[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) v[h] = l[i][h];
      const float ws = warp_transpose_sum16(v);
      if ((lane & 1) == 0) ms->red_sum[warp][16 * (q0 + i) + (lane >> 1)] = ws;
    }
    named_bar_sync(sg.bar, kSoftmaxThreads);
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
      const int qi = q0 + i;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        l_tot[i][h] = (ms->red_sum[0][16 * qi + h] + ms->red_sum[1][16 * qi + h]) +
                      (ms->red_sum[2][16 * qi + h] + ms->red_sum[3][16 * qi + h]);
    }
    const bool write = row_ok && ms->red_u32[8 + g] == 0;  // the same for every thread of the warpgroup
    // l >= 1 when the token saw a cached token here (its reference maximum
    // contributes 1): a fast divide suffices; l = 0 (nothing visible) gives 0.
    float inv[kQt][16];
#pragma unroll
    for (int i = 0; i < kQt; ++i) {
#pragma unroll
      for (int h = 0; h < 16; ++h) inv[i][h] = l_tot[i][h] > 0.0f ? __fdividef(kv_scale, l_tot[i][h]) : 0.0f;
    }
    // this warpgroup's tokens that the CTA takes: q0 .. q0 + gn - 1
    const int32_t gn = max(0, min(nq - q0, kQt));
    wait_pv(tile - 1);  // PV of the segment's last tile (and so of all before it)
    tc_fence_after();
    if (lead && cur.seg == 0) MLA_TRACE_CLK(kTrEpilogue);
    const uint32_t stage_q = sbase + G::kOffQ;
    if (!kCluster && cur.whole) {
      // bf16 rows [token][16 heads][512 dims] (16 KB each), staged in the Q region.
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int i = 0; i < kQt; ++i) {
          const int qi = q0 + i;
          if (qi >= nq) continue;  // the same for every softmax thread
          float o[16];
          tmem_ld_heads<kFmt>(tmem + lane_base + G::kColO + G::kN * cc + G::kTokCols * qi, o);
          const int dim = 128 * cc + token;
          if (write) {
#pragma unroll
            for (int h = 0; h < 16; ++h)
              st_shared_u16(stage_q + ((16 * qi + h) * kVDim + dim) * 2, bf16_bits(o[h] * inv[i][h]));
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(sg.bar, kSoftmaxThreads);
      if (t == 0 && write && gn > 0 && MLA_DCHECK(tq + q0 + gn <= total_tokens(p), p.err)) {
        bulk_store(p.out + static_cast<size_t>(tq + q0) * kNumHeads * kVDim,
                   stage_q + q0 * kNumHeads * kVDim * 2, gn * kNumHeads * kVDim * 2);
        bulk_commit();
      }
    } else {
      // bf16 partial of query token qi (as the pages keep their split
      // outputs), stored [slot][slot_q + qi][dim / 128][head / 8][dim % 128][head % 8]:
      // each 128-dim chunk is 4 KB of contiguous memory, in which this thread's
      // dim owns two 16-byte pieces (heads 0-7 and 8-15), so every thread
      // stores its own values straight from registers (a warp's stores are
      // 512 contiguous bytes) and nothing waits for them to drain.  The float
      // base-2 log-sum-exps follow, one per (token, head).
      // (the cluster split: CTA i's piece goes to slot i, combined in this kernel)
      const int32_t slot = kCluster ? static_cast<int32_t>(blockIdx.x) : partial_slot(c, ms->t0, cur.row_a);
      const size_t piece = static_cast<size_t>(slot) * p.slot_tokens + slot_q;  // (slot, token)
#pragma unroll 1
      for (int k = 0; k < 4 * gn; ++k) {
        const int i = kQt == 1 ? 0 : k >> 2, qi = q0 + i, cc = k & 3;
        float o[16];
        tmem_ld_heads<kFmt>(tmem + lane_base + G::kColO + G::kN * cc + G::kTokCols * qi, o);
        if (write) {
          float v[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) v[h] = o[h] * inv[i][h];
          uint4* dst = reinterpret_cast<uint4*>(p.partial + ((piece + qi) * 4 + cc) * (kNumHeads * 128));
          const int64_t last = static_cast<int64_t>(((piece + qi) * 4 + cc) * (kNumHeads * 128)) +
                               (128 + token) * 8 + 8;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (MLA_DCHECK(last <= partial_elems(p), p.err)) dst[j * 128 + token] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                              pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                              pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                              pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        }
      }
      if ((write || kCluster) && t < 16 * gn) {
        // thread t writes the LSE of (token q0 + t / 16, head t % 16); -inf when
        // it saw nothing (or, for the cluster split, when the call gave up: the
        // piece is then not written and weighs 0)
        float mm = m_ref[0][0], ll = l_tot[0][0];
#pragma unroll
        for (int e = 1; e < 16 * kQt; ++e) {
          mm = t == e ? m_ref[e >> 4][e & 15] : mm;
          ll = t == e ? l_tot[e >> 4][e & 15] : ll;
        }
        const size_t at = (piece + q0) * kNumHeads + t;
        if (MLA_DCHECK(static_cast<int64_t>(at) < partial_elems(p) / kVDim, p.err))
          p.lse[at] = write ? mm + log2f(ll) : -INFINITY;
      }
    }
    // O has been read out (tcgen05.wait::ld above): the next segment's PV may
    // overwrite it.  Nothing else is published, so the flag is stored relaxed
    // and does not wait for the output stores to drain.
    tc_fence_before();
    named_bar_sync(sg.bar, kSoftmaxThreads);
    if (t == 0) st_relaxed_u32(&ms->o_free[g], static_cast<uint32_t>(cur.seg + 1));
    if (lead && cur.seg == 0) MLA_TRACE_CLK(kTrEpilogueDone);
    cursor_next_tile(cur, ms, p.kv_indptr, p.batch);
  }
  // The bulk stores have read their staging and written global memory before
  // the CTA exits.
  if (t == 0) bulk_wait_all();
  if (lead) trace_shape(cur.seg + 1, static_cast<int32_t>(tile));
}

// ------------------------------------------------------------ test hooks: the two-term operands
// The Q operand of an e4m3 cache exactly as a stage-1 CTA prepares it: CTA i
// runs prepare_q for query tokens kQ i .. kQ i + kQ - 1 (one 128-thread
// warpgroup, as the softmax warps do) and copies the swizzled operand back out
// as codes [token][hi, lo][head][576] with the token's qk_scale.  The query
// bounds check of prepare_q always holds here (nq stops at the last token), so
// p.err is never written.
template <int kQ>
__global__ void __launch_bounds__(kSoftmaxThreads) debug_q_operand_kernel(const Stage1Params p,
                                                                          uint8_t* codes,
                                                                          float* qk_scale_out) {
  using G = Geo<kQ, Kv::kE4m3>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sq = smem_u32(smem);
  Misc* ms = reinterpret_cast<Misc*>(smem + (G::kOffP - G::kOffQ));
  const int32_t tokens = p.batch;
  const int32_t tq = static_cast<int32_t>(blockIdx.x) * kQ;
  const int32_t nq = min(kQ, tokens - tq);
  float qk_scale[kQ];
  prepare_q<kQ, kQ, Kv::kE4m3>(p, ms, sq, tq, nq, __ldg(p.kv_scale), qk_scale, single_softmax_group(), 0, 0,
                               true, false);
  constexpr int kChunks = kQkDim / 16;  // 16-byte chunks of an operand row
  for (int job = threadIdx.x; job < nq * 32 * kChunks; job += kSoftmaxThreads) {
    const int row = job / kChunks, ch = job % kChunks;  // row = 32 qi + 16 lo + head
    const uint4 v = ld_shared_v4(q_chunk_addr<kQ, Kv::kE4m3>(sq, row, ch));
    *reinterpret_cast<uint4*>(codes + (static_cast<size_t>(tq) * 32 + row) * kQkDim + 16 * ch) = v;
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int qi = 0; qi < kQ; ++qi)
      if (qi < nq) qk_scale_out[tq + qi] = qk_scale[qi];
  }
}

constexpr int debug_q_smem(int q) {
  return (q == 1 ? Geo<1, Kv::kE4m3>::kOffP - Geo<1, Kv::kE4m3>::kOffQ
                 : Geo<2, Kv::kE4m3>::kOffP - Geo<2, Kv::kE4m3>::kOffQ) +
         static_cast<int>(sizeof(Misc)) + 1024;
}
static_assert(debug_q_smem(2) <= 48 * 1024, "the Q-operand hook runs without a shared-memory opt-in");
static_assert((Geo<1, Kv::kE4m3>::kOffP - Geo<1, Kv::kE4m3>::kOffQ) % 16 == 0 &&
                  (Geo<2, Kv::kE4m3>::kOffP - Geo<2, Kv::kE4m3>::kOffQ) % 16 == 0,
              "the hook's barrier block follows the Q region 16-byte aligned");

// The P operand split of the softmax warps: each thread takes 16 consecutive
// probabilities and writes their hi and lo e4m3 codes (16 bytes each).
__global__ void debug_p_split_kernel(const float* p, int64_t groups, uint8_t* hi, uint8_t* lo) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  float x[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) x[k] = p[16 * g + k];
  uint32_t h[4], l[4];
  split_p_16(x, h, l);
  reinterpret_cast<uint4*>(hi)[g] = make_uint4(h[0], h[1], h[2], h[3]);
  reinterpret_cast<uint4*>(lo)[g] = make_uint4(l[0], l[1], l[2], l[3]);
}

// ------------------------------------------------------------ kernel
template <bool kGather, int kQ, Kv kFmt, bool kCluster>
__global__ void __launch_bounds__((stage1_threads<kGather, kQ, kFmt>()), 1)
    mla_decode_stage1_kernel(const __grid_constant__ CUtensorMap map_v,
                             const __grid_constant__ CUtensorMap map_r,
                             const __grid_constant__ CUtensorMap map_s, const Stage1Params p) {
  using G = Geo<kQ, kFmt>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + G::kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    MLA_TRACE_NS(kTrEntryNs);
    MLA_TRACE_CLK(kTrEntry);
  }

  if (warp == kMmaWarp) tmem_alloc(smem_u32(&ms->tmem_base), G::kTmemCols);
  if (tid == kProducerWarp * 32) {
    // The e4m3 panels are complete when their copy lands, or (MXFP4) when
    // every converter warp has written its rows.
    constexpr uint32_t kFullArrivals = G::kMx ? kConverterWarps : 1;
    for (int s = 0; s < G::kNumV; ++s) {
      mbar_init(smem_u32(&ms->v_full[s]), kFullArrivals);
      mbar_init(smem_u32(&ms->v_empty[s]), 1);
      if (G::kMx) mbar_init(smem_u32(&ms->raw_full[s]), 1);
    }
    for (int s = 0; s < kNumRSlots; ++s) {
      mbar_init(smem_u32(&ms->r_full[s]), kFullArrivals);
      if (G::kMx) mbar_init(smem_u32(&ms->rraw_full[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ms->s_full[i]), 1);
      mbar_init(smem_u32(&ms->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&ms->q_empty), 1);
    // every thread of each softmax warpgroup arrives on every part
    for (int i = 0; i < kQParts; ++i)
      mbar_init(smem_u32(&ms->q_part[i]), kSoftmaxThreads * (dual_softmax<kGather, kQ, kFmt>() ? 2 : 1));
    for (int g = 0; g < 2; ++g) ms->s_read[g] = ms->p_ready[g] = ms->o_free[g] = 0;
    mbar_init(smem_u32(&ms->mma_done), 2);  // one commit from each MMA issuer
    ms->abort_flag = 0;
    ms->first_row = -1;
    ms->last_row = -1;
    ms->first_prefix = 0;
    ms->tile0_issued = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_r);
    if (G::kMx) prefetch_tensormap(&map_s);
  }
  // Launched as a programmatic dependent, this grid may start while the
  // previous kernel of the stream is finishing: everything above touches only
  // this CTA's own resources, everything below may read that kernel's results
  // or write what it reads.  (Without the launch attribute the wait is a no-op.)
  if (tid == 0) MLA_TRACE_CLK(kTrPreWait);
  pdl_wait_primary();
  if (tid == 0) MLA_TRACE_CLK(kTrPostWait);
  // Stage 2 may start launching now; it waits for this grid's completion
  // before it reads anything this grid writes.
  pdl_launch_dependents();
  if constexpr (kCluster)
    cluster_prologue<kQ, kFmt>(p, &map_v, &map_r, ms, sbase);
  else
    schedule_prologue<kQ, kFmt>(p, &map_v, &map_r, ms, sbase);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) MLA_TRACE_CLK(kTrPrologue);
  const uint32_t tmem = ms->tmem_base;

  // Page-table mode and the MXFP4 cache run 12 warps: registers move from the
  // producers, MMA issuers and converters to the softmax warpgroup, inside the
  // role branches so that each role's code is compiled under its own count.
  // An MXFP4 cache's e4m3 panels hold e2m1 * 2^(e - 127 - bias): its scale is
  // 2^bias.
  constexpr bool kWide = wide_block<kGather, kQ, kFmt>();
  constexpr bool kDual = dual_softmax<kGather, kQ, kFmt>();
  if (warp < 4 || (kDual && warp >= 8)) {
    if constexpr (kWide) setmaxnreg_inc<kSoftmaxRegs>();
    if constexpr (kDual) setmaxnreg_inc<kDualSoftmaxRegs>();
    const float kv_scale = G::kMx ? __int_as_float((127 + p.mx_bias) << 23)
                                  : (G::kSplit ? __ldg(p.kv_scale) : 1.0f);
    run_softmax<kGather, kQ, kFmt, kWide || kQ == 2, kCluster, kDual ? 2 : 1>(p, ms, sbase, tmem, kv_scale,
                                                                      warp >= 8 ? 1 : 0);
  } else {
    if constexpr (G::kMx)
      setmaxnreg_dec<kOtherRegsMx>();
    else if constexpr (kWide)
      setmaxnreg_dec<kOtherRegs>();
    else if constexpr (kDual)
      setmaxnreg_dec<kDualOtherRegs>();
    const int who = kGather ? gather_producer_of_warp(warp, num_producers<kGather, kQ>())
                            : (warp == kProducerWarp ? 0 : -1);
    if (who >= 0) {
      if constexpr (G::kMx)
        run_producer_mx<kQ>(p, &map_v, &map_r, &map_s, ms, sbase);
      else
        run_producer<kGather, kQ, kFmt>(p, &map_v, &map_r, ms, sbase, static_cast<uint32_t>(who));
    } else if (G::kMx && warp >= kFirstConverterWarp) {
      if constexpr (G::kMx) run_converter<kQ>(p, ms, sbase);
    } else if (warp == kMmaWarp && lane == 0) {
      run_mma_pv<kQ, kFmt, kQ == 2 || kCluster, kDual>(p, ms, sbase, tmem);
    } else if (warp == kMmaQkWarp && lane == 0) {
      run_mma_qk<kGather, kQ, kFmt, kQ == 2 || kCluster, kDual>(p, ms, sbase, tmem);
    } else if (!kCluster && cta_sibling(p) == 0 &&
               (kGather ? warp == kMmaWarp && lane == 1 : warp == kIdleWarp && lane == 0)) {
      write_worker_record<kQ>(p, ms);
    } else if (!kGather && !G::kMx && warp == kIdleWarp && lane == 1) {
      trace_observer<kQ, kFmt>(p, ms);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (kCluster) {
    // A CTA without tokens marks its slot empty; then the barrier publishes
    // every CTA's partial (its global writes, released at cluster scope) and
    // the row is combined.
    if (ms->first_row < 0 && tid < 16 &&
        MLA_DCHECK(static_cast<int64_t>(blockIdx.x) * p.slot_tokens < 2LL * p.grid * p.slot_tokens, p.err))
      p.lse[static_cast<size_t>(blockIdx.x) * p.slot_tokens * kNumHeads + tid] = -INFINITY;
    cluster_sync_all();
    if (tid == 0) MLA_TRACE_CLK(kTrClusterBarrier);
    cluster_combine<kQ, kFmt>(p, ms, smem);
    if (tid == 0) MLA_TRACE_CLK(kTrCombineDone);
  }
  if (tid == 0) {
    MLA_TRACE_CLK(kTrExit);
    MLA_TRACE_NS(kTrExitNs);
  }
  if (warp == kMmaWarp) {
    if (lane == 0) drain_phase(smem_u32(&ms->mma_done), 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

template <bool kGather, int kQ, Kv kFmt, bool kCluster = false>
cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(mla_decode_stage1_kernel<kGather, kQ, kFmt, kCluster>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_alloc<kQ, kFmt>());
}

cudaError_t set_smem_limits() {
  cudaError_t e = set_smem_limit<false, 1, Kv::kE4m3>();
  if (e == cudaSuccess) e = set_smem_limit<true, 1, Kv::kE4m3>();
  if (e == cudaSuccess) e = set_smem_limit<false, 2, Kv::kE4m3>();
  if (e == cudaSuccess) e = set_smem_limit<true, 2, Kv::kE4m3>();
  if (e == cudaSuccess) e = set_smem_limit<false, 1, Kv::kBf16>();
  if (e == cudaSuccess) e = set_smem_limit<false, 2, Kv::kBf16>();
  if (e == cudaSuccess) e = set_smem_limit<false, 1, Kv::kMx4>();
  if (e == cudaSuccess) e = set_smem_limit<false, 1, Kv::kE4m3, true>();
  if (e == cudaSuccess) e = set_smem_limit<false, 1, Kv::kBf16, true>();
  return e;
}

template <bool kGather, int kQ, Kv kFmt, bool kCluster = false>
cudaError_t launch(const Stage1Params& p, const Stage1Maps& maps, cudaStream_t stream) {
  // A programmatic dependent of the previous kernel in the stream: its CTAs
  // may be scheduled while that kernel finishes, and wait for it (griddepcontrol
  // .wait) before touching global memory.  The cluster split launches one
  // cluster of p.cluster CTAs per row.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(kCluster ? p.batch * p.cluster : p.grid * p.siblings));
  cfg.blockDim = dim3(stage1_threads<kGather, kQ, kFmt>());
  cfg.dynamicSmemBytes = smem_alloc<kQ, kFmt>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster ? static_cast<unsigned>(p.cluster) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kCluster ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_stage1_kernel<kGather, kQ, kFmt, kCluster>, maps.v,
                            maps.r, maps.s, p);
}


constexpr int cmax(int a, int b) { return a > b ? a : b; }

}  // namespace

size_t stage1_smem_bytes() {
  return static_cast<size_t>(cmax(cmax(cmax(smem_alloc<1, Kv::kE4m3>(), smem_alloc<2, Kv::kE4m3>()),
                                       cmax(smem_alloc<1, Kv::kBf16>(), smem_alloc<2, Kv::kBf16>())),
                                  smem_alloc<1, Kv::kMx4>()));
}

cudaError_t stage1_prepare(int device) {
  (void)device;
  return set_smem_limits();
}

cudaError_t launch_stage1(const Stage1Params& p, const Stage1Maps& maps, bool gather,
                          CacheFormat format, cudaStream_t stream) {
  const bool two = p.row_tokens - p.q_off >= 2;  // each CTA takes up to two tokens
  if (format == CacheFormat::kMxfp4) {
    if (gather || two) return cudaErrorNotSupported;  // the host rejects these before launching
    return launch<false, 1, Kv::kMx4>(p, maps, stream);
  }
  if (p.cluster > 0) {  // contiguous rows, one query token (the host checks)
    if (gather || two || p.cluster > kMaxCluster || (p.cluster & (p.cluster - 1)) != 0)
      return cudaErrorNotSupported;
    return format == CacheFormat::kBf16 ? launch<false, 1, Kv::kBf16, true>(p, maps, stream)
                                        : launch<false, 1, Kv::kE4m3, true>(p, maps, stream);
  }
  if (format == CacheFormat::kBf16) {
    if (gather) return cudaErrorNotSupported;  // the host rejects this before launching
    return two ? launch<false, 2, Kv::kBf16>(p, maps, stream)
               : launch<false, 1, Kv::kBf16>(p, maps, stream);
  }
  if (two)
    return gather ? launch<true, 2, Kv::kE4m3>(p, maps, stream)
                  : launch<false, 2, Kv::kE4m3>(p, maps, stream);
  return gather ? launch<true, 1, Kv::kE4m3>(p, maps, stream)
                : launch<false, 1, Kv::kE4m3>(p, maps, stream);
}

#ifdef MLA_TRACE
cudaError_t trace_read_stage1(unsigned long long* host, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(host, g_trace_stage1, sizeof(g_trace_stage1));
  if (e == cudaSuccess && clear) {
    static const unsigned long long zeros[kTraceCtas * kTraceEvents] = {};
    e = cudaMemcpyToSymbol(g_trace_stage1, zeros, sizeof(zeros));
  }
  return e;
}
#else
cudaError_t trace_read_stage1(unsigned long long*, bool) { return cudaErrorNotSupported; }
#endif

cudaError_t launch_debug_q_operand(const uint16_t* q, int32_t tokens, int32_t per_cta,
                                   const float* kv_scale, uint8_t* codes, float* qk_scale,
                                   cudaStream_t stream) {
  Stage1Params p = {};
  p.q = q;
  p.kv_scale = kv_scale;
  p.batch = tokens;
  p.row_tokens = 1;
  const unsigned grid = static_cast<unsigned>((tokens + per_cta - 1) / per_cta);
  if (per_cta == 2)
    debug_q_operand_kernel<2><<<grid, kSoftmaxThreads, debug_q_smem(2), stream>>>(p, codes, qk_scale);
  else
    debug_q_operand_kernel<1><<<grid, kSoftmaxThreads, debug_q_smem(1), stream>>>(p, codes, qk_scale);
  return cudaGetLastError();
}

cudaError_t launch_debug_p_split(const float* p, int64_t groups, uint8_t* hi, uint8_t* lo,
                                 cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((groups + 255) / 256);
  debug_p_split_kernel<<<grid, 256, 0, stream>>>(p, groups, hi, lo);
  return cudaGetLastError();
}

}  // namespace mla
