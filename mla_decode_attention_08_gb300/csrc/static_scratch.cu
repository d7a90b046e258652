// mla_decode_fwd_static_scratch: the decode step for callers that must not
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a plugin loaded into a
// host application that owns every device allocation and hands the plugin only
// its input and output buffers, or a latency-critical serving loop in which an
// allocation (which may synchronise the device) is not allowed.  For them the
// split partials, tile prefix and error word live in the array below, which the
// library reserves in each GPU's memory when the library is loaded on that GPU
// and keeps until the process exits.
#include <mutex>

#include "../../include/mla_decode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  std::mutex lock;
  void* ptr = nullptr;
};
ScratchAddress g_scratch_address[kMaxDevices];

// Device address of this GPU's copy of the array.  Host code cannot use the
// array's name as a pointer (it is a host-side stand-in), so it is looked up
// once per device, with that device current.  A device this library has no
// kernels for is refused first: the lookup would fail there with a
// missing-image error.
mla_status_t scratch_on_current_device(void** out) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  ScratchAddress& a = g_scratch_address[device];
  std::lock_guard<std::mutex> guard(a.lock);
  if (a.ptr == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
      return MLA_ERR_CUDA;
    if (major != 10 || minor != 3) return MLA_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      (void)cudaGetLastError();  // leave no runtime error behind for the caller
      return MLA_ERR_CUDA;
    }
    a.ptr = ptr;
  }
  *out = a.ptr;
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_fwd_static_scratch(
    const void* q_bf16, const void* kv_fp8, const float* kv_scale, const int32_t* qo_indptr,
    const int32_t* kv_indptr, void* out_bf16, cudaStream_t stream, const mla_plan_t* plan,
    const int32_t* kv_indices, int64_t kv_indices_len, int64_t kv_rows) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->ws_bytes > MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const mla_status_t st = scratch_on_current_device(&scratch);
  if (st != MLA_OK) return st;
  // Nothing in the scratch has to start at zero: every region a call reads is
  // written earlier in the same call.  The error word only accumulates bits;
  // mla_decode_static_scratch_read_error reads and clears it.
  return mla_decode_fwd(q_bf16, kv_fp8, kv_scale, qo_indptr, kv_indptr, out_bf16, stream, plan,
                        kv_indices, kv_indices_len, kv_rows, scratch, MLA_STATIC_SCRATCH_BYTES);
}

extern "C" mla_status_t mla_decode_static_scratch_read_error(int32_t* err_host, int32_t clear,
                                                             cudaStream_t stream) {
  if (err_host == nullptr) return MLA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const mla_status_t st = scratch_on_current_device(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode_read_error(scratch, err_host, clear, stream);
}
