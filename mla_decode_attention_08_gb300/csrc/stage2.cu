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
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 16 * p.qo_len);
  cfg.blockDim = dim3(kStage2Threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mla_decode_stage2_kernel, p);
}

}  // namespace mla
