// Stage 2 of the decode step: log-sum-exp combine of the rows that stage 1
// split across workers (kernelbot-amd-mixed-mla submission 722089, `_mla_reduce`:
// M = max_s lse_s, w_s = 2^(lse_s - M), out = sum_s w_s partial_s / sum_s w_s),
// done here in one online pass.  Rows held whole by one worker were written by
// stage 1 and are skipped; rows without cached tokens are written as zeros.
//
// Grid (B, 4) x 256 threads: block (b, g) covers heads 4g..4g+3 of row b, each
// thread 8 consecutive dims, loaded as two float4 per partial and stored as one
// 128-bit bf16 vector.
#include <cuda_bf16.h>

#include "../../include/mla_decode.h"
#include "kernels.h"
#include "ptx.cuh"
#include "schedule.h"

namespace mla {
namespace {

__global__ void __launch_bounds__(256) mla_decode_stage2_kernel(const Stage2Params p) {
  // Everything read below is written by stage 1.
  pdl_wait_primary();

  const int32_t b = blockIdx.x;
  const int head = blockIdx.y * 4 + (threadIdx.x >> 6);
  const int d0 = (threadIdx.x & 63) * 8;
  const int32_t tq = __ldg(p.qo_indptr + b);
  if (__ldg(p.qo_indptr + b + 1) - tq != 1 || tq < 0 || tq >= p.batch) return;

  const int32_t a_begin = p.prefix[b];
  const int32_t a_end = p.prefix[b + 1];
  const int32_t total = p.prefix[p.batch];
  uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(tq) * kNumHeads + head) * kVDim + d0);

  if (a_end <= a_begin) {  // no cached token: zero output
    *dst = make_uint4(0, 0, 0, 0);
    return;
  }
  const int32_t c_first = worker_of_tile(a_begin, total, p.grid);
  const int32_t c_last = worker_of_tile(a_end - 1, total, p.grid);
  if (c_first == c_last) return;  // written whole by stage 1

  float m = -INFINITY, wsum = 0.0f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int32_t c = c_first; c <= c_last; ++c) {
    const int32_t t0 = worker_begin(c, total, p.grid);
    if (worker_begin(c + 1, total, p.grid) == t0) continue;  // empty worker
    const int32_t slot = partial_slot(c, t0, a_begin);
    const float lse = p.lse[slot * kNumHeads + head];
    const float4* src = reinterpret_cast<const float4*>(
        p.partial + (static_cast<size_t>(slot) * kNumHeads + head) * kVDim + d0);
    const float4 v0 = src[0], v1 = src[1];
    if (lse > m) {
      const float f = exp2f(m - lse);
      wsum *= f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= f;
      m = lse;
    }
    const float w = exp2f(lse - m);
    wsum += w;
    acc[0] += w * v0.x; acc[1] += w * v0.y; acc[2] += w * v0.z; acc[3] += w * v0.w;
    acc[4] += w * v1.x; acc[5] += w * v1.y; acc[6] += w * v1.z; acc[7] += w * v1.w;
  }
  const float inv = 1.0f / wsum;
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    ow[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  *dst = o;
}

}  // namespace

cudaError_t launch_stage2(const Stage2Params& p, bool programmatic, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch), 4);
  cfg.blockDim = dim3(256);
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
