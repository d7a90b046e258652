// MXFP4 quantisation of bf16 latent rows (input preparation): per block of 32
// consecutive elements of a 576-element row, one E8M0 scale 2^e with
// e = clamp(floor(log2 max|x|) - 2, -127, 127) (e = -127 for an all-zero block)
// and 32 E2M1 elements x / 2^e rounded to nearest even, saturating at +-6; two
// elements per byte, the even one in the low nibble.  The format is the one
// kernelbot-amd-mixed-mla submission 738050 documents in
// `_dequantize_mxfp4_inplace` (32-element blocks, E2M1 elements, E8M0 scales,
// two elements per byte); the scale rule is the OCP Microscaling one.
#include "kernels.h"
#include "schedule.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerRow = kQkDim / 32;  // 18

// Two floats -> two E2M1 codes in one byte, `lo` in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One thread per 32-element block: 64 bytes of bf16 in, 16 bytes of elements
// and one scale byte out.
__global__ void __launch_bounds__(kThreads) mxfp4_quantize_kernel(const uint16_t* __restrict__ src,
                                                                  int64_t rows,
                                                                  uint8_t* __restrict__ dst,
                                                                  uint8_t* __restrict__ scales) {
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= rows * kBlocksPerRow) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + blk * 32);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = __ldg(s4 + i);
    w[4 * i + 0] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
  uint32_t amax_bits = 0;  // bf16 magnitude bits, monotone in the value
#pragma unroll
  for (int i = 0; i < 16; ++i) amax_bits = max(amax_bits, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  int e = -127;
  if (amax_bits != 0) e = max(-127, min(127, ilogbf(__uint_as_float(amax_bits << 16)) - 2));
  uint32_t out[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // word i holds elements 2i (low half) and 2i + 1
    const float lo = ldexpf(__uint_as_float(w[i] << 16), -e);
    const float hi = ldexpf(__uint_as_float(w[i] & 0xFFFF0000u), -e);
    out[i >> 2] |= cvt_e2m1x2(lo, hi) << (8 * (i & 3));
  }
  reinterpret_cast<uint4*>(dst)[blk] = make_uint4(out[0], out[1], out[2], out[3]);
  scales[blk] = static_cast<uint8_t>(e + 127);
}

}  // namespace

cudaError_t launch_mxfp4_quantize(const uint16_t* src, int64_t rows, uint8_t* dst, uint8_t* scales,
                                  cudaStream_t stream) {
  const int64_t blocks = (rows * kBlocksPerRow + kThreads - 1) / kThreads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  mxfp4_quantize_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(src, rows, dst,
                                                                                scales);
  return cudaGetLastError();
}

}  // namespace mla
