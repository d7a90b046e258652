// Host side of libmla_decode: plan, argument checks, TMA descriptors, launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/mla_decode.h"
#include "kernels.h"
#include "schedule.h"

namespace {

using mla::kNumHeads;
using mla::kQkDim;
using mla::kTileTokens;
using mla::kVDim;

constexpr uint64_t kAlign = 256;
uint64_t round_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The cache addressed as bytes: [kv_rows, 576 * elem] uint8 (elem = 1 for
// e4m3 codes, 2 for bf16, whose boxes are plain copies), box_w bytes wide and
// box_h rows high.
bool encode_kv_map(CUtensorMap* map, const void* kv, int64_t rows, bool bf16, uint32_t box_w,
                   uint32_t box_h, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(kQkDim) * (bf16 ? 2 : 1);
  const cuuint64_t gdim[2] = {row_bytes, static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {row_bytes};
  const cuuint32_t box[2] = {box_w, box_h};
  const cuuint32_t estride[2] = {1, 1};
  // Page-table rows (boxes one row high) sit at random places in the pool: a
  // 64-byte promotion fetches exactly a row (576 = 9 x 64 bytes, rows 64-byte
  // aligned), where 128- and 256-byte promotions also fetch parts of
  // neighbouring rows (DRAM reads measured 313.5 MB against 341.6 MB with 256
  // bytes for the ragged 128-row workload, whose algorithmic bytes are 313.9 MB).
  const CUtensorMapL2promotion promo =
      box_h == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small per-thread cache of encoded descriptors: the same cache pool is
// normally decoded step after step.
struct MapEntry {
  const void* kv = nullptr;
  int64_t rows = 0;
  bool gather = false;
  bool bf16 = false;
  int device = -1;
  CUtensorMap v, r;
};

// Latent and rope boxes (tiles of 128 rows, or single rows for tile::gather4):
// e4m3 128 and 64 bytes wide; bf16 128 bytes (64 dims) for both.
bool kv_maps(const void* kv, int64_t rows, bool gather, bool bf16, int device, CUtensorMap* v,
             CUtensorMap* r) {
  constexpr int kEntries = 8;
  thread_local MapEntry cache[kEntries];
  thread_local int next = 0;
  for (auto& e : cache) {
    if (e.kv == kv && e.rows == rows && e.gather == gather && e.bf16 == bf16 &&
        e.device == device) {
      *v = e.v;
      *r = e.r;
      return true;
    }
  }
  MapEntry e;
  e.kv = kv;
  e.rows = rows;
  e.gather = gather;
  e.bf16 = bf16;
  e.device = device;
  const uint32_t h = gather ? 1u : static_cast<uint32_t>(kTileTokens);
  if (!encode_kv_map(&e.v, kv, rows, bf16, 128, h, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
  if (!encode_kv_map(&e.r, kv, rows, bf16, bf16 ? 128 : 64, h,
                     bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
    return false;
  cache[next] = e;
  next = (next + 1) % kEntries;
  *v = e.v;
  *r = e.r;
  return true;
}

// MXFP4 cache: the elements [kv_rows, 288] uint8 in boxes of 128 rows, 64 bytes
// wide (64-byte swizzle) and 32 bytes wide (32-byte swizzle), and the scale
// bytes [kv_rows * 18] as one flat array in 256-byte boxes (zero fill past its
// end, so a tile's boxes never read beyond the caller's array).
bool encode_mx_maps(const void* fp4, const void* scales, int64_t rows, mla::Stage1Maps* m) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t row_bytes = kQkDim / 2;
  const cuuint64_t gdim[2] = {row_bytes, static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {row_bytes};
  const cuuint32_t estride[2] = {1, 1};
  const cuuint32_t box_v[2] = {64, static_cast<cuuint32_t>(kTileTokens)};
  const cuuint32_t box_r[2] = {32, static_cast<cuuint32_t>(kTileTokens)};
  if (fn(&m->v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(fp4), gdim, gstride, box_v,
         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (fn(&m->r, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(fp4), gdim, gstride, box_r,
         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t sdim[1] = {static_cast<cuuint64_t>(rows) * (kQkDim / 32)};
  // A rank-1 map has no strides, but the encoder rejects a null array.
  const cuuint64_t sstride[1] = {16};
  const cuuint32_t sbox[1] = {256};
  const cuuint32_t sestride[1] = {1};
  return fn(&m->s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, const_cast<void*>(scales), sdim, sstride,
            sbox, sestride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MxMapEntry {
  const void* fp4 = nullptr;
  const void* scales = nullptr;
  int64_t rows = 0;
  int device = -1;
  mla::Stage1Maps maps;
};

bool mx_maps(const void* fp4, const void* scales, int64_t rows, int device, mla::Stage1Maps* m) {
  constexpr int kEntries = 4;
  thread_local MxMapEntry cache[kEntries];
  thread_local int next = 0;
  for (auto& e : cache) {
    if (e.fp4 == fp4 && e.scales == scales && e.rows == rows && e.device == device) {
      *m = e.maps;
      return true;
    }
  }
  MxMapEntry e;
  e.fp4 = fp4;
  e.scales = scales;
  e.rows = rows;
  e.device = device;
  if (!encode_mx_maps(fp4, scales, rows, &e.maps)) return false;
  cache[next] = e;
  next = (next + 1) % kEntries;
  *m = e.maps;
  return true;
}

// Checks the current device is an sm_103 part and sets the kernels' shared
// memory limit once per device.
mla_status_t prepare_device(int* device_out) {
  static std::atomic<int> ready[64];
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  if (device < 0 || device >= 64) return MLA_ERR_UNSUPPORTED;
  *device_out = device;
  if (ready[device].load(std::memory_order_acquire) == 1) return MLA_OK;
  int major = 0, minor = 0, smem = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major != 10 || minor != 3) return MLA_ERR_UNSUPPORTED;
  if (static_cast<size_t>(smem) < mla::stage1_smem_bytes()) return MLA_ERR_UNSUPPORTED;
  if (mla::stage1_prepare(device) != cudaSuccess) return MLA_ERR_CUDA;
  ready[device].store(1, std::memory_order_release);
  return MLA_OK;
}

mla_status_t check_plan(const mla_plan_t* plan) {
  if (plan == nullptr || plan->abi_version != MLA_ABI_VERSION || plan->batch < 1 ||
      plan->grid < 1 || plan->tile_tokens != kTileTokens || plan->max_kv_len < 0 ||
      plan->qo_len < 1 || plan->qo_len > 4 || plan->num_sms < 1)
    return MLA_ERR_INVALID_ARG;
  // The cluster split: the planned size, or 0 (the caller forced the persistent split).
  if (plan->cluster != 0 &&
      plan->cluster != mla::plan_cluster(plan->batch, plan->qo_len, plan->max_kv_len, plan->num_sms))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// CTAs per row of the cluster split for this call, or 0 for the persistent split:
// the cluster split takes contiguous e4m3 and bf16 caches.
int32_t cluster_of(const mla_plan_t* plan, mla::CacheFormat fmt, const int32_t* kv_indices) {
  return kv_indices == nullptr && fmt != mla::CacheFormat::kMxfp4 ? plan->cluster : 0;
}

mla_status_t check_workspace(const mla_plan_t* plan, void* workspace, size_t workspace_bytes) {
  if (workspace == nullptr || !aligned(workspace, kAlign)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->ws_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return MLA_OK;
}

// One CTA holds the accumulators of up to two query tokens per row (TMEM);
// rows of three or four are shared by two sibling CTAs per worker.
constexpr int32_t kCtaTokens = 2;
int32_t siblings_of(const mla_plan_t* plan) { return plan->qo_len > kCtaTokens ? 2 : 1; }

mla::Stage2Params stage2_params(const int32_t* qo_indptr, void* out, const mla_plan_t* plan,
                                void* workspace) {
  auto* ws = static_cast<uint8_t*>(workspace);
  mla::Stage2Params s;
  s.qo_indptr = qo_indptr;
  s.out = static_cast<uint16_t*>(out);
  s.err = reinterpret_cast<int32_t*>(ws);
  s.prefix = reinterpret_cast<const int32_t*>(ws + plan->ws_prefix_offset);
  s.workers = reinterpret_cast<const int32_t*>(ws + plan->ws_workers_offset);
  s.lse = reinterpret_cast<const float*>(ws + plan->ws_lse_offset);
  s.partial = reinterpret_cast<const uint16_t*>(ws + plan->ws_partial_offset);
  s.batch = plan->batch;
  s.grid = plan->grid;
  s.qo_len = plan->qo_len;
  return s;
}

// The largest MXFP4 pool: the kernel addresses the flat scale array (18 bytes a
// row) with 32-bit box coordinates.
constexpr int64_t kMaxMxRows = (INT32_MAX - 4096) / (kQkDim / 32);

// kv_scale is required for an e4m3 cache and ignored for the others; an MXFP4
// cache passes its elements as kv, its scale bytes as mx_scales and the bias.
mla_status_t run_stage1(const void* q, const void* kv, const float* kv_scale,
                        const int32_t* qo_indptr, const int32_t* kv_indptr, void* out,
                        cudaStream_t stream, const mla_plan_t* plan, const int32_t* kv_indices,
                        int64_t kv_indices_len, int64_t kv_rows, void* workspace,
                        size_t workspace_bytes, mla::CacheFormat fmt, bool stall_stream = false,
                        const void* mx_scales = nullptr, int32_t mx_bias = 0) {
  using mla::CacheFormat;
  mla_status_t st = check_plan(plan);
  if (st != MLA_OK) return st;
  if (q == nullptr || kv == nullptr || (kv_scale == nullptr && fmt == CacheFormat::kE4m3) ||
      (mx_scales == nullptr && fmt == CacheFormat::kMxfp4) || qo_indptr == nullptr ||
      kv_indptr == nullptr || out == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  if (kv_rows < 1 || kv_rows > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (kv_indices != nullptr && (kv_indices_len < 0 || kv_indices_len > INT32_MAX))
    return MLA_ERR_INVALID_ARG;
  if (fmt != CacheFormat::kE4m3 && kv_indices != nullptr) return MLA_ERR_UNSUPPORTED;
  if (fmt == CacheFormat::kMxfp4) {
    if (kv_rows > kMaxMxRows || mx_bias < -100 || mx_bias > 100 || !aligned(mx_scales, 16))
      return MLA_ERR_INVALID_ARG;
    if (plan->qo_len != 1) return MLA_ERR_UNSUPPORTED;
  }
  st = check_workspace(plan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  int device = 0;
  st = prepare_device(&device);
  if (st != MLA_OK) return st;

  const bool gather = kv_indices != nullptr;
  mla::Stage1Maps maps;
  if (fmt == CacheFormat::kMxfp4) {
    if (!mx_maps(kv, mx_scales, kv_rows, device, &maps)) return MLA_ERR_CUDA;
  } else {
    if (!kv_maps(kv, kv_rows, gather, fmt == CacheFormat::kBf16, device, &maps.v, &maps.r))
      return MLA_ERR_CUDA;
    maps.s = maps.v;
  }

  auto* ws = static_cast<uint8_t*>(workspace);
  mla::Stage1Params p;
  p.q = static_cast<const uint16_t*>(q);
  p.kv_scale = fmt == CacheFormat::kE4m3 ? kv_scale : nullptr;
  p.qo_indptr = qo_indptr;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.out = static_cast<uint16_t*>(out);
  p.err = reinterpret_cast<int32_t*>(ws);
  p.prefix = reinterpret_cast<int32_t*>(ws + plan->ws_prefix_offset);
  p.workers = reinterpret_cast<int32_t*>(ws + plan->ws_workers_offset);
  p.lse = reinterpret_cast<float*>(ws + plan->ws_lse_offset);
  p.partial = reinterpret_cast<uint16_t*>(ws + plan->ws_partial_offset);
  p.kv_rows = kv_rows;
  p.kv_indices_len = gather ? kv_indices_len : 0;
  p.batch = plan->batch;
  p.grid = plan->grid;
  p.row_tokens = plan->qo_len;
  p.q_off = 0;
  p.siblings = siblings_of(plan);
  p.slot_tokens = plan->qo_len;
  p.stall_stream = stall_stream ? 1 : 0;
  p.mx_bias = mx_bias;
  p.kv_bytes = gather ? nullptr : static_cast<const uint8_t*>(kv);
  p.cluster = cluster_of(plan, fmt, kv_indices);
  p.kv_row_bytes = fmt == CacheFormat::kMxfp4 ? kQkDim / 2 : (fmt == CacheFormat::kBf16 ? 2 * kQkDim : kQkDim);
  return mla::launch_stage1(p, maps, gather, fmt, stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t run_stage2(const int32_t* qo_indptr, void* out, cudaStream_t stream,
                        const mla_plan_t* plan, void* workspace, bool programmatic) {
  return mla::launch_stage2(stage2_params(qo_indptr, out, plan, workspace), programmatic,
                            stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

// The whole step: stage 1 then stage 2 on `stream`, both programmatic dependents.
mla_status_t run_decode(const void* q, const void* kv, const float* kv_scale,
                        const int32_t* qo_indptr, const int32_t* kv_indptr, void* out,
                        cudaStream_t stream, const mla_plan_t* plan, const int32_t* kv_indices,
                        int64_t kv_indices_len, int64_t kv_rows, void* workspace,
                        size_t workspace_bytes, mla::CacheFormat fmt, bool stall_stream = false,
                        const void* mx_scales = nullptr, int32_t mx_bias = 0) {
  mla_status_t st = run_stage1(q, kv, kv_scale, qo_indptr, kv_indptr, out, stream, plan,
                               kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                               fmt, stall_stream, mx_scales, mx_bias);
  // The cluster split combines inside stage 1: no second kernel.
  if (st == MLA_OK && cluster_of(plan, fmt, kv_indices) == 0)
    st = run_stage2(qo_indptr, out, stream, plan, workspace, true);
  return st;
}

}  // namespace

extern "C" {

const char* mla_status_string(mla_status_t status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported device (needs sm_103 with 227 KB shared memory per block)";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA call failed";
  }
  return "unknown status";
}

int32_t mla_decode_abi_version(void) { return MLA_ABI_VERSION; }

mla_status_t mla_decode_plan(int32_t batch, int32_t max_kv_len, int32_t num_sms, mla_plan_t* plan) {
  return mla_decode_plan_mtp(batch, 1, max_kv_len, num_sms, plan);
}

mla_status_t mla_decode_plan_mtp(int32_t batch, int32_t qo_len, int32_t max_kv_len, int32_t num_sms,
                                 mla_plan_t* plan) {
  if (plan == nullptr || batch < 1 || max_kv_len < 0 || qo_len < 1 || qo_len > 4)
    return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * qo_len > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  mla_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.batch = batch;
  p.max_kv_len = max_kv_len;
  p.num_sms = num_sms;
  // Rows of three or four query tokens run two sibling CTAs per worker: one
  // worker per pair of SMs.
  p.grid = mla::plan_grid(batch, max_kv_len,
                          qo_len > kCtaTokens ? (num_sms > 1 ? num_sms / 2 : 1) : num_sms);
  p.tile_tokens = kTileTokens;
  p.abi_version = MLA_ABI_VERSION;
  p.qo_len = qo_len;
  p.cluster = mla::plan_cluster(batch, qo_len, max_kv_len, num_sms);
  const uint64_t g = static_cast<uint64_t>(p.grid);
  const uint64_t nq = static_cast<uint64_t>(qo_len);
  uint64_t off = kAlign;  // error word + reserved header
  p.ws_prefix_offset = off;
  off += round_up((static_cast<uint64_t>(batch) + 1) * sizeof(int32_t));
  p.ws_workers_offset = off;
  off += round_up(g * 8 * sizeof(int32_t));
  p.ws_lse_offset = off;
  off += round_up(2 * g * nq * kNumHeads * sizeof(float));
  p.ws_partial_offset = off;
  off += round_up(2 * g * nq * kNumHeads * kVDim * sizeof(uint16_t));
  p.ws_bytes = off;
  *plan = p;
  return MLA_OK;
}

mla_status_t mla_decode_stage1(const void* q_bf16, const void* kv_fp8, const float* kv_scale,
                               const int32_t* qo_indptr, const int32_t* kv_indptr, void* out_bf16,
                               cudaStream_t stream, const mla_plan_t* plan,
                               const int32_t* kv_indices, int64_t kv_indices_len, int64_t kv_rows,
                               void* workspace, size_t workspace_bytes) {
  return run_stage1(q_bf16, kv_fp8, kv_scale, qo_indptr, kv_indptr, out_bf16, stream, plan,
                    kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                    mla::CacheFormat::kE4m3);
}

mla_status_t mla_decode_stage1_bf16kv(const void* q_bf16, const void* kv_bf16,
                                      const int32_t* qo_indptr, const int32_t* kv_indptr,
                                      void* out_bf16, cudaStream_t stream, const mla_plan_t* plan,
                                      const int32_t* kv_indices, int64_t kv_indices_len,
                                      int64_t kv_rows, void* workspace, size_t workspace_bytes) {
  return run_stage1(q_bf16, kv_bf16, nullptr, qo_indptr, kv_indptr, out_bf16, stream, plan,
                    kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                    mla::CacheFormat::kBf16);
}

mla_status_t mla_decode_stage2(const int32_t* qo_indptr, void* out_bf16, cudaStream_t stream,
                               const mla_plan_t* plan, void* workspace, size_t workspace_bytes) {
  mla_status_t st = check_plan(plan);
  if (st != MLA_OK) return st;
  if (qo_indptr == nullptr || out_bf16 == nullptr || !aligned(out_bf16, 16))
    return MLA_ERR_INVALID_ARG;
  st = check_workspace(plan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  return run_stage2(qo_indptr, out_bf16, stream, plan, workspace, false);
}

mla_status_t mla_decode_fwd(const void* q_bf16, const void* kv_fp8, const float* kv_scale,
                            const int32_t* qo_indptr, const int32_t* kv_indptr, void* out_bf16,
                            cudaStream_t stream, const mla_plan_t* plan,
                            const int32_t* kv_indices, int64_t kv_indices_len, int64_t kv_rows,
                            void* workspace, size_t workspace_bytes) {
  return run_decode(q_bf16, kv_fp8, kv_scale, qo_indptr, kv_indptr, out_bf16, stream, plan,
                    kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                    mla::CacheFormat::kE4m3);
}

mla_status_t mla_decode_fwd_bf16kv(const void* q_bf16, const void* kv_bf16,
                                   const int32_t* qo_indptr, const int32_t* kv_indptr,
                                   void* out_bf16, cudaStream_t stream, const mla_plan_t* plan,
                                   const int32_t* kv_indices, int64_t kv_indices_len,
                                   int64_t kv_rows, void* workspace, size_t workspace_bytes) {
  return run_decode(q_bf16, kv_bf16, nullptr, qo_indptr, kv_indptr, out_bf16, stream, plan,
                    kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                    mla::CacheFormat::kBf16);
}

mla_status_t mla_decode_fwd_stall_stream(const void* q_bf16, const void* kv_fp8,
                                         const float* kv_scale, const int32_t* qo_indptr,
                                         const int32_t* kv_indptr, void* out_bf16,
                                         cudaStream_t stream, const mla_plan_t* plan,
                                         const int32_t* kv_indices, int64_t kv_indices_len,
                                         int64_t kv_rows, void* workspace, size_t workspace_bytes) {
  return run_decode(q_bf16, kv_fp8, kv_scale, qo_indptr, kv_indptr, out_bf16, stream, plan,
                    kv_indices, kv_indices_len, kv_rows, workspace, workspace_bytes,
                    mla::CacheFormat::kE4m3, true);
}

mla_status_t mla_decode_fwd_mxfp4(const void* q_bf16, const void* kv_fp4, const void* kv_scales,
                                  int32_t scale_bias, const int32_t* qo_indptr,
                                  const int32_t* kv_indptr, void* out_bf16, cudaStream_t stream,
                                  const mla_plan_t* plan, int64_t kv_rows, void* workspace,
                                  size_t workspace_bytes) {
  return run_decode(q_bf16, kv_fp4, nullptr, qo_indptr, kv_indptr, out_bf16, stream, plan, nullptr,
                    0, kv_rows, workspace, workspace_bytes, mla::CacheFormat::kMxfp4, false,
                    kv_scales, scale_bias);
}

mla_status_t mla_decode_fwd_mxfp4_stall_stream(const void* q_bf16, const void* kv_fp4,
                                               const void* kv_scales, int32_t scale_bias,
                                               const int32_t* qo_indptr, const int32_t* kv_indptr,
                                               void* out_bf16, cudaStream_t stream,
                                               const mla_plan_t* plan, int64_t kv_rows,
                                               void* workspace, size_t workspace_bytes) {
  return run_decode(q_bf16, kv_fp4, nullptr, qo_indptr, kv_indptr, out_bf16, stream, plan, nullptr,
                    0, kv_rows, workspace, workspace_bytes, mla::CacheFormat::kMxfp4, true,
                    kv_scales, scale_bias);
}

mla_status_t mla_debug_q_operand(const void* q_bf16, int32_t num_tokens, int32_t tokens_per_cta,
                                 const float* kv_scale, void* codes_out, float* qk_scale_out,
                                 cudaStream_t stream) {
  if (q_bf16 == nullptr || kv_scale == nullptr || codes_out == nullptr || qk_scale_out == nullptr ||
      num_tokens < 1 || num_tokens > (1 << 24) || (tokens_per_cta != 1 && tokens_per_cta != 2) ||
      !aligned(q_bf16, 16) || !aligned(codes_out, 16))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  mla_status_t st = prepare_device(&device);
  if (st != MLA_OK) return st;
  return mla::launch_debug_q_operand(static_cast<const uint16_t*>(q_bf16), num_tokens,
                                     tokens_per_cta, kv_scale, static_cast<uint8_t*>(codes_out),
                                     qk_scale_out, stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_decode_trace_read(uint64_t* stage1_host, uint64_t* stage2_host, int32_t clear) {
  if (stage1_host == nullptr || stage2_host == nullptr) return MLA_ERR_INVALID_ARG;
  static_assert(sizeof(uint64_t) == sizeof(unsigned long long), "trace stamps are 64-bit");
  cudaError_t e = mla::trace_read_stage1(reinterpret_cast<unsigned long long*>(stage1_host), clear != 0);
  if (e == cudaSuccess)
    e = mla::trace_read_stage2(reinterpret_cast<unsigned long long*>(stage2_host), clear != 0);
  if (e == cudaErrorNotSupported) return MLA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status_t mla_debug_p_split(const float* p, int64_t n, void* hi_out, void* lo_out,
                               cudaStream_t stream) {
  if (p == nullptr || hi_out == nullptr || lo_out == nullptr || n < 16 || n % 16 != 0 ||
      n > (INT64_C(1) << 34) || !aligned(p, 16) || !aligned(hi_out, 16) || !aligned(lo_out, 16))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  mla_status_t st = prepare_device(&device);
  if (st != MLA_OK) return st;
  return mla::launch_debug_p_split(p, n / 16, static_cast<uint8_t*>(hi_out),
                                   static_cast<uint8_t*>(lo_out), stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_decode_stage1_mxfp4(const void* q_bf16, const void* kv_fp4, const void* kv_scales,
                                     int32_t scale_bias, const int32_t* qo_indptr,
                                     const int32_t* kv_indptr, void* out_bf16, cudaStream_t stream,
                                     const mla_plan_t* plan, int64_t kv_rows, void* workspace,
                                     size_t workspace_bytes) {
  return run_stage1(q_bf16, kv_fp4, nullptr, qo_indptr, kv_indptr, out_bf16, stream, plan, nullptr,
                    0, kv_rows, workspace, workspace_bytes, mla::CacheFormat::kMxfp4, false,
                    kv_scales, scale_bias);
}

mla_status_t mla_mxfp4_quantize(const void* src_bf16, int64_t rows, void* dst_fp4, void* dst_scales,
                                cudaStream_t stream) {
  if (src_bf16 == nullptr || dst_fp4 == nullptr || dst_scales == nullptr || rows < 1 ||
      rows > (INT64_C(1) << 36) || !aligned(src_bf16, 16) || !aligned(dst_fp4, 16))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  mla_status_t st = prepare_device(&device);
  if (st != MLA_OK) return st;
  return mla::launch_mxfp4_quantize(static_cast<const uint16_t*>(src_bf16), rows,
                                    static_cast<uint8_t*>(dst_fp4),
                                    static_cast<uint8_t*>(dst_scales), stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_fp8_quantize_per_tensor(const void* src_bf16, int64_t n, void* dst_fp8,
                                         float* scale_out, void* tmp, size_t tmp_bytes,
                                         cudaStream_t stream) {
  if (src_bf16 == nullptr || dst_fp8 == nullptr || scale_out == nullptr || tmp == nullptr ||
      n < 1 || tmp_bytes < 16 || !aligned(tmp, 4) || !aligned(src_bf16, 2))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  mla_status_t st = prepare_device(&device);
  if (st != MLA_OK) return st;
  return mla::launch_fp8_quantize(static_cast<const uint16_t*>(src_bf16), n,
                                  static_cast<uint8_t*>(dst_fp8), scale_out,
                                  static_cast<uint32_t*>(tmp), stream) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_decode_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (workspace == nullptr || workspace_bytes < sizeof(int32_t)) return MLA_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, stream) == cudaSuccess ? MLA_OK
                                                                               : MLA_ERR_CUDA;
}

mla_status_t mla_decode_read_error(void* workspace, int32_t* err_host, int32_t clear,
                                   cudaStream_t stream) {
  if (workspace == nullptr || err_host == nullptr) return MLA_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  *err_host = v;
  if (clear && cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_decode_schedule_host(const int32_t* kv_indptr_host, int32_t batch, int32_t grid,
                                      int32_t* workers_out, int32_t* prefix_out) {
  if (kv_indptr_host == nullptr || workers_out == nullptr || prefix_out == nullptr || batch < 1 ||
      grid < 1)
    return MLA_ERR_INVALID_ARG;
  bool bad = kv_indptr_host[0] < 0;
  for (int32_t b = 0; b < batch; ++b)
    if (kv_indptr_host[b + 1] < kv_indptr_host[b]) bad = true;
  auto row_tiles = [&](int32_t b) {
    return bad ? 0 : mla::tiles_of_length(static_cast<int64_t>(kv_indptr_host[b + 1]) - kv_indptr_host[b]);
  };
  int32_t tiles = 0;
  for (int32_t b = 0; b < batch; ++b) tiles += row_tiles(b);
  // every row with tiles is preceded by `start` schedule units
  const int32_t start = mla::row_start_units(tiles, grid);
  int32_t a = 0;
  for (int32_t b = 0; b < batch; ++b) {
    prefix_out[b] = a;
    const int32_t nt = row_tiles(b);
    if (nt > 0) a += start + nt;
  }
  prefix_out[batch] = a;
  const int32_t total = a;
  for (int32_t c = 0; c < grid; ++c) {
    const int32_t t0 = mla::worker_begin(c, total, grid);
    const int32_t t1 = mla::worker_begin(c + 1, total, grid);
    int32_t first = -1, last = -1;
    if (t1 > t0) {
      for (int32_t b = 0; b < batch; ++b) {
        const int32_t nt = row_tiles(b);
        if (nt <= 0) continue;
        const int32_t ra = prefix_out[b] + start;  // the row's first tile
        if (ra < t1 && t0 < ra + nt) {  // the worker holds tiles of row b
          if (first < 0) first = b;
          last = b;
        }
      }
    }
    workers_out[4 * c + 0] = t0;
    workers_out[4 * c + 1] = t1;
    workers_out[4 * c + 2] = first;
    workers_out[4 * c + 3] = last;
  }
  return MLA_OK;
}

}  // extern "C"
