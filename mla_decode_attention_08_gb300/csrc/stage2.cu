// Stage 2 of the decode step: log-sum-exp combine of the rows that stage 1
// split across workers (kernelbot-amd-mixed-mla submission 722089, `_mla_reduce`:
// M = max_s lse_s, w_s = 2^(lse_s - M), out = sum_s w_s partial_s / sum_s w_s),
// done here in one online pass.
//
// A split row contains at least one worker boundary, so the grid is sized by
// the workers, not the rows: stage 1 records in worker c's entry the combine
// job of the split row whose first boundary is worker c's start (output row,
// first and last worker, first worker's partial slot; the others use slot 2c),
// and block (c, 16 qi + 4 cc + j) combines dims 128cc..128cc+127 of heads
// 4j..4j+3 of query token qi of that row, one dim per thread.  Rows held whole
// by one worker, and rows without cached tokens, are written by stage 1.
// Partials are bf16, stored [slot][token][dim / 128][head / 8][dim % 128][head % 8]
// (stage 1's epilogue): a thread reads its four heads as one 8-byte load, and
// the blocks of heads 8k..8k+3 and 8k+4..8k+7 read the two halves of the same
// 512-byte spans.  The partials of a row are visited four at a time, their
// loads in flight together.
#include <cuda_bf16.h>

#include "../../include/mla_decode.h"
#include "kernels.h"
#include "ptx.cuh"
#include "schedule.h"

namespace mla {
namespace {

constexpr int kStage2Threads = 128;  // one thread per dim of a 128-dim chunk
constexpr int kStage2Unroll = 4;     // partials loaded together

// Start-up trace (-DMLA_TRACE only): global-timer stamps of each block at entry,
// after the wait for stage 1 and at exit (see kernels.h).
#ifdef MLA_TRACE
__device__ unsigned long long g_trace_stage2[kTrace2Blocks * kTrace2Events];
__device__ __forceinline__ void trace2_put(int ev) {
  const unsigned blk = blockIdx.y * gridDim.x + blockIdx.x;
  if (threadIdx.x == 0 && blk < static_cast<unsigned>(kTrace2Blocks))
    g_trace_stage2[blk * kTrace2Events + ev] = global_timer_ns();
}
#define MLA_TRACE2(ev) trace2_put(ev)
#else
#define MLA_TRACE2(ev) ((void)0)
#endif

__global__ void __launch_bounds__(kStage2Threads) mla_decode_stage2_kernel(const Stage2Params p) {
  __shared__ __align__(16) uint16_t blk[4 * kStage2Threads];  // bf16 [4 heads][128 dims]
  MLA_TRACE2(0);
  // The next kernel of the stream may start launching; it waits for this
  // grid's completion before it touches global memory.
  pdl_launch_dependents();
  // Everything read below is written by stage 1.
  pdl_wait_primary();
  MLA_TRACE2(1);

  const int32_t c = blockIdx.x;
  const int qi = blockIdx.y >> 4, cc = (blockIdx.y >> 2) & 3, j = blockIdx.y & 3, dd = threadIdx.x;
  const int32_t nq = p.qo_len;
  const int4* rec = reinterpret_cast<const int4*>(p.workers);
  const int4 job = rec[2 * c + 1];  // (output row, first worker, last worker, first slot)
  if (job.x < 0) {
    MLA_TRACE2(2);
    return;
  }
  const int32_t tq = job.x + qi;  // output row: query token qi of the row
  if (!MLA_DCHECK(tq < p.batch * nq && job.y >= 0 && job.z < p.grid && job.w < 2 * p.grid, p.err))
    return;

  const float4* lse4 = reinterpret_cast<const float4*>(p.lse);
  const uint2* part8 = reinterpret_cast<const uint2*>(p.partial);
  // One online pass: m_h is the running maximum of lse_s,h, and the weights of
  // the partials seen so far are rescaled when it grows.
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float wsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int32_t w0 = job.y; w0 <= job.z; w0 += kStage2Unroll) {
    // Issue every load of the group first; a worker with no tiles (possible
    // only when the grid exceeds the tile count) wrote no partial, and its
    // values are dropped.
    int4 wr[kStage2Unroll];
    float4 x[kStage2Unroll];
    uint2 v[kStage2Unroll];
#pragma unroll
    for (int u = 0; u < kStage2Unroll; ++u) {
      const int32_t cu = w0 + u;
      wr[u] = make_int4(0, 0, 0, 0);  // an empty record: the slot is skipped below
      if (cu <= job.z) {
        const int32_t piece = (cu == job.y ? job.w : 2 * cu) * nq + qi;  // (slot, token)
        if (!MLA_DCHECK(piece < 2 * p.grid * nq, p.err)) continue;
        wr[u] = rec[2 * cu];
        x[u] = lse4[piece * 4 + j];
        v[u] = part8[(((static_cast<size_t>(piece) * 4 + cc) * 2 + (j >> 1)) * kStage2Threads + dd) * 2 +
                     (j & 1)];
      }
    }
#pragma unroll
    for (int u = 0; u < kStage2Unroll; ++u) {
      if (w0 + u > job.z || wr[u].y <= wr[u].x) continue;
      const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      const float vs[4] = {__uint_as_float(v[u].x << 16), __uint_as_float(v[u].x & 0xFFFF0000u),
                           __uint_as_float(v[u].y << 16), __uint_as_float(v[u].y & 0xFFFF0000u)};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (xs[h] == -INFINITY) continue;  // the token saw no cached token in this piece
        const float mn = fmaxf(m[h], xs[h]);
        const float f = exp2f(m[h] - mn), w = exp2f(xs[h] - mn);
        wsum[h] = wsum[h] * f + w;
        acc[h] = acc[h] * f + w * vs[h];
        m[h] = mn;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __nv_bfloat16 y = __float2bfloat16_rn(wsum[h] > 0.0f ? acc[h] / wsum[h] : 0.0f);
    blk[h * kStage2Threads + dd] = *reinterpret_cast<const uint16_t*>(&y);
  }
  __syncthreads();
  // 4 heads x 16 vectors of 8 dims.
  if (dd < 64) {
    const int h = dd >> 4, part = dd & 15;
    uint16_t* dst = p.out + (static_cast<size_t>(tq) * kNumHeads + 4 * j + h) * kVDim + 128 * cc + part * 8;
    *reinterpret_cast<uint4*>(dst) = reinterpret_cast<const uint4*>(blk)[dd];
  }
  MLA_TRACE2(2);
}

// Two or more query tokens per row: eight heads a thread, block
// (c, 8 qi + 2 cc + hh) combining dims 128cc..128cc+127 of heads 8hh..8hh+7,
// so that the grid (8 blocks per worker and token) is half as large.  A
// thread reads its eight heads as one 16-byte load; the group's log-sum-exps,
// the same for every thread of the block, go through shared memory (32
// threads load one each, with the worker's record), which keeps the thread
// within the 64 registers that allow 8 blocks per SM.  Measured against the
// four-head kernel: two-token bs64 65.9 -> 65.3 us back to back, 76.5 -> 75.4
// with L2 flushed; one-token workloads were slower with it (bs64 68.3 -> 70.3
// flushed) and keep the four-head kernel.
template <int kHeads>
__global__ void __launch_bounds__(kStage2Threads, 8) mla_decode_stage2_wide_kernel(const Stage2Params p) {
  static_assert(kHeads == 8, "eight heads a thread");
  static_assert(kStage2Unroll * kHeads <= kStage2Threads, "a thread per group log-sum-exp");
  constexpr int kHalves = kNumHeads / kHeads;  // blocks per 128-dim chunk
  __shared__ __align__(16) uint16_t blk[kHeads * kStage2Threads];  // bf16 [heads][128 dims]
  __shared__ float grp_lse[kStage2Unroll][kHeads];  // the group's log-sum-exps (-inf: skip)
  MLA_TRACE2(0);
  // The next kernel of the stream may start launching; it waits for this
  // grid's completion before it touches global memory.
  pdl_launch_dependents();
  // Everything read below is written by stage 1.
  pdl_wait_primary();
  MLA_TRACE2(1);

  const int32_t c = blockIdx.x;
  const int qi = blockIdx.y / (4 * kHalves), cc = (blockIdx.y / kHalves) & 3, hh = blockIdx.y % kHalves;
  const int dd = threadIdx.x;
  const int32_t nq = p.qo_len;
  const int4* rec = reinterpret_cast<const int4*>(p.workers);
  const int4 job = rec[2 * c + 1];  // (output row, first worker, last worker, first slot)
  if (job.x < 0) {
    MLA_TRACE2(2);
    return;
  }
  const int32_t tq = job.x + qi;  // output row: query token qi of the row
  if (!MLA_DCHECK(tq < p.batch * nq && job.y >= 0 && job.z < p.grid && job.w < 2 * p.grid, p.err))
    return;

  const uint4* part = reinterpret_cast<const uint4*>(p.partial);  // a thread's 8 heads of a dim
  // One online pass: m_h is the running maximum of lse_s,h, and the weights of
  // the partials seen so far are rescaled when it grows.
  float m[kHeads], wsum[kHeads], acc[kHeads];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) {
    m[h] = -INFINITY;
    wsum[h] = acc[h] = 0.0f;
  }
  for (int32_t w0 = job.y; w0 <= job.z; w0 += kStage2Unroll) {
    // Issue every load of the group first.  Thread 8u + k (k < 8) brings head
    // 8hh + k's log-sum-exp of the group's partial u, or -inf when there is
    // none: past the row's last worker, or a worker with no tiles (possible
    // only when the grid exceeds the tile count), which wrote no partial.
    uint4 v[kStage2Unroll];
#pragma unroll
    for (int u = 0; u < kStage2Unroll; ++u) {
      const int32_t cu = w0 + u;
      v[u] = make_uint4(0, 0, 0, 0);
      if (cu <= job.z) {
        const int32_t piece = (cu == job.y ? job.w : 2 * cu) * nq + qi;  // (slot, token)
        if (MLA_DCHECK(piece < 2 * p.grid * nq, p.err)) {
          // [piece][dim / 128][head / 8][dim % 128][head % 8], in 16-byte units
          v[u] = part[((static_cast<size_t>(piece) * 4 + cc) * 2 + hh) * kStage2Threads + dd];
        }
      }
    }
    if (dd < kStage2Unroll * kHeads) {
      const int u = dd / kHeads, k = dd % kHeads;
      const int32_t cu = w0 + u;
      float x = -INFINITY;
      if (cu <= job.z) {
        const int32_t piece = (cu == job.y ? job.w : 2 * cu) * nq + qi;
        if (MLA_DCHECK(piece < 2 * p.grid * nq, p.err)) {
          const int4 wr = rec[2 * cu];
          const float l = p.lse[piece * kNumHeads + kHeads * hh + k];
          x = wr.y > wr.x ? l : -INFINITY;
        }
      }
      grp_lse[u][k] = x;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kStage2Unroll; ++u) {
      const uint32_t vw[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        const float xh = grp_lse[u][h];
        if (xh == -INFINITY) continue;  // no partial, or the token saw no cached token in it
        const float vh = __uint_as_float((h & 1) ? (vw[h >> 1] & 0xFFFF0000u) : (vw[h >> 1] << 16));
        const float mn = fmaxf(m[h], xh);
        const float f = exp2f(m[h] - mn), w = exp2f(xh - mn);
        wsum[h] = wsum[h] * f + w;
        acc[h] = acc[h] * f + w * vh;
        m[h] = mn;
      }
    }
    __syncthreads();  // the group's log-sum-exps are read before the next group's are written
  }
#pragma unroll
  for (int h = 0; h < kHeads; ++h) {
    const __nv_bfloat16 y = __float2bfloat16_rn(wsum[h] > 0.0f ? acc[h] / wsum[h] : 0.0f);
    blk[h * kStage2Threads + dd] = *reinterpret_cast<const uint16_t*>(&y);
  }
  __syncthreads();
  // 8 heads x 16 vectors of 8 dims: one 16-byte store a thread.
  {
    const int h = dd >> 4, q8 = dd & 15;
    uint16_t* dst = p.out + (static_cast<size_t>(tq) * kNumHeads + kHeads * hh + h) * kVDim + 128 * cc + q8 * 8;
    *reinterpret_cast<uint4*>(dst) = reinterpret_cast<const uint4*>(blk)[dd];
  }
  MLA_TRACE2(2);
}

}  // namespace

#ifdef MLA_TRACE
cudaError_t trace_read_stage2(unsigned long long* host, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(host, g_trace_stage2, sizeof(g_trace_stage2));
  if (e == cudaSuccess && clear) {
    static const unsigned long long zeros[kTrace2Blocks * kTrace2Events] = {};
    e = cudaMemcpyToSymbol(g_trace_stage2, zeros, sizeof(zeros));
  }
  return e;
}
#else
cudaError_t trace_read_stage2(unsigned long long*, bool) { return cudaErrorNotSupported; }
#endif

cudaError_t launch_stage2(const Stage2Params& p, bool programmatic, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const bool wide = p.qo_len >= 2;  // eight heads a thread (see the wide kernel)
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid), (wide ? 8 : 16) * p.qo_len);
  cfg.blockDim = dim3(kStage2Threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return wide ? cudaLaunchKernelEx(&cfg, mla_decode_stage2_wide_kernel<8>, p)
              : cudaLaunchKernelEx(&cfg, mla_decode_stage2_kernel, p);
}

}  // namespace mla
