/*
 * A plain C caller of libmla_decode (no Python, no torch): reads a decode
 * problem from a binary file, runs the e4m3 step through the C ABI with device
 * memory from the CUDA runtime, and writes the bf16 output and the device error
 * word.  Built and run by tests/test_gpu_c_abi.py.
 *
 * Input file (little endian): int32 batch, int32 n_tokens, int32 max_kv_len,
 * int32 has_page_table; int32 qo_indptr[batch + 1]; int32 kv_indptr[batch + 1];
 * if has_page_table, int32 kv_indices[n_tokens]; uint16 q[batch][16][576] (bf16
 * bits); uint16 kv[n_tokens][576] (bf16 bits of the cache source).
 * Output file: int32 status, int32 error word, uint16 out[batch][16][512].
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "mla_decode.h"

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input.bin output.bin\n", argv[0]);
    return 2;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 2;
  int32_t hdr[4];
  if (!read_all(f, hdr, sizeof(hdr))) return 2;
  const int32_t batch = hdr[0], n_tokens = hdr[1], max_kv_len = hdr[2], paged = hdr[3];
  const size_t q_elems = (size_t)batch * MLA_NUM_HEADS * MLA_QK_HEAD_DIM;
  const size_t kv_elems = (size_t)(n_tokens > 0 ? n_tokens : 1) * MLA_QK_HEAD_DIM;
  const size_t out_elems = (size_t)batch * MLA_NUM_HEADS * MLA_V_HEAD_DIM;
  int32_t* qo = malloc((size_t)(batch + 1) * 4);
  int32_t* kvp = malloc((size_t)(batch + 1) * 4);
  int32_t* idx = paged ? malloc((size_t)n_tokens * 4) : NULL;
  uint16_t* q = malloc(q_elems * 2);
  uint16_t* kv = calloc(kv_elems, 2);
  uint16_t* out = malloc(out_elems * 2);
  if (!qo || !kvp || !q || !kv || !out || (paged && !idx)) return 2;
  if (!read_all(f, qo, (size_t)(batch + 1) * 4) || !read_all(f, kvp, (size_t)(batch + 1) * 4) ||
      (paged && !read_all(f, idx, (size_t)n_tokens * 4)) || !read_all(f, q, q_elems * 2) ||
      !read_all(f, kv, (size_t)n_tokens * MLA_QK_HEAD_DIM * 2))
    return 2;
  fclose(f);

  void* d_q = to_device(q, q_elems * 2);
  void* d_kv_src = to_device(kv, kv_elems * 2);
  void* d_qo = to_device(qo, (size_t)(batch + 1) * 4);
  void* d_kvp = to_device(kvp, (size_t)(batch + 1) * 4);
  void* d_idx = paged ? to_device(idx, (size_t)n_tokens * 4) : NULL;
  void *d_codes = NULL, *d_scale = NULL, *d_tmp = NULL, *d_out = NULL, *d_ws = NULL;
  if (!d_q || !d_kv_src || !d_qo || !d_kvp || (paged && !d_idx) ||
      cudaMalloc(&d_codes, kv_elems) != cudaSuccess || cudaMalloc(&d_scale, 4) != cudaSuccess ||
      cudaMalloc(&d_tmp, 16) != cudaSuccess || cudaMalloc(&d_out, out_elems * 2) != cudaSuccess)
    return 3;

  mla_status_t st = mla_fp8_quantize_per_tensor(d_kv_src, (int64_t)kv_elems, d_codes, d_scale, d_tmp,
                                                16, (cudaStream_t)0);
  mla_plan_t plan;
  if (st == MLA_OK) st = mla_decode_plan(batch, max_kv_len, 0, &plan);
  if (st == MLA_OK && cudaMalloc(&d_ws, plan.ws_bytes) != cudaSuccess) st = MLA_ERR_CUDA;
  if (st == MLA_OK) st = mla_decode_workspace_init(d_ws, plan.ws_bytes, (cudaStream_t)0);
  if (st == MLA_OK)
    st = mla_decode_fwd(d_q, d_codes, (const float*)d_scale, (const int32_t*)d_qo,
                        (const int32_t*)d_kvp, d_out, (cudaStream_t)0, &plan,
                        (const int32_t*)d_idx, paged ? n_tokens : 0,
                        n_tokens > 0 ? n_tokens : 1, d_ws, plan.ws_bytes);
  int32_t err = -1;
  if (st == MLA_OK) st = mla_decode_read_error(d_ws, &err, 1, (cudaStream_t)0);
  if (st == MLA_OK && cudaMemcpy(out, d_out, out_elems * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
    st = MLA_ERR_CUDA;
  if (st != MLA_OK) fprintf(stderr, "mla: %s\n", mla_status_string(st));

  FILE* o = fopen(argv[2], "wb");
  if (!o) return 2;
  const int32_t res[2] = {(int32_t)st, err};
  fwrite(res, 4, 2, o);
  fwrite(out, 2, out_elems, o);
  fclose(o);
  cudaFree(d_q); cudaFree(d_kv_src); cudaFree(d_qo); cudaFree(d_kvp); cudaFree(d_idx);
  cudaFree(d_codes); cudaFree(d_scale); cudaFree(d_tmp); cudaFree(d_out); cudaFree(d_ws);
  free(qo); free(kvp); free(idx); free(q); free(kv); free(out);
  return st == MLA_OK ? 0 : 1;
}
