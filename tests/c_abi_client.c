/* A plain C11 client of libh3attn.so: tagged RoPE with the continuation shift, then packed varlen
 * attention, called through include/h3attn.h alone (no Python, no torch).  Used by
 * tests/test_c_abi_client.py, which writes the inputs, runs this program and compares its
 * outputs with the Python binding's and with the oracle.
 *
 * usage: c_abi_client <input file> <output file>
 *
 * Input (little-endian): int32 C, H, D, N, S, R, max_seqlen, then
 *   q, k, v    bf16 [C, H, D] each (uint16 bit patterns)
 *   pos        fp32 [N, 3]      tag   uint8 [N]
 *   cu_seqlens int32 [S + 1]    cu_requests int32 [R + 1]    start_frames fp32 [R]
 * Output: int32 status of h3_rope_apply, of h3_varlen_attn_fwd and of h3_get_device_error, then
 *   o bf16 [C, H, D] and lse fp32 [H, C].
 * The pad rows [N, C) of o and lse are preset to bf16 3.0 / fp32 5.0, so the caller can check
 * that the library left them untouched.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "h3attn.h"

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }

#define CHECK_CUDA(call)                                                   \
  do {                                                                     \
    cudaError_t e_ = (call);                                               \
    if (e_ != cudaSuccess) {                                               \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));   \
      return 2;                                                            \
    }                                                                      \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s <input> <output>\n", argv[0]);
    return 1;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t hdr[7];
  if (!read_all(in, hdr, sizeof(hdr))) return 1;
  const int32_t C = hdr[0], H = hdr[1], D = hdr[2], N = hdr[3], S = hdr[4], R = hdr[5];
  const int32_t max_seqlen = hdr[6];
  const size_t elems = (size_t)C * H * D;
  uint16_t* host_qkv = malloc(3 * elems * sizeof(uint16_t));
  float* host_pos = malloc((size_t)N * 3 * sizeof(float) + 4);
  uint8_t* host_tag = malloc((size_t)N + 1);
  int32_t* host_cu = malloc((size_t)(S + 1) * sizeof(int32_t));
  int32_t* host_req = malloc((size_t)(R + 1) * sizeof(int32_t));
  float* host_start = malloc((size_t)R * sizeof(float) + 4);
  if (!host_qkv || !host_pos || !host_tag || !host_cu || !host_req || !host_start) return 1;
  if (!read_all(in, host_qkv, 3 * elems * sizeof(uint16_t)) ||
      !read_all(in, host_pos, (size_t)N * 3 * sizeof(float)) || !read_all(in, host_tag, (size_t)N) ||
      !read_all(in, host_cu, (size_t)(S + 1) * sizeof(int32_t)) ||
      !read_all(in, host_req, (size_t)(R + 1) * sizeof(int32_t)) ||
      !read_all(in, host_start, (size_t)R * sizeof(float)))
    return 1;
  fclose(in);

  /* device buffers: Q, K, V as given; rotated Q and K; O and LSE preset to sentinels */
  void *q, *k, *v, *qr, *kr, *o, *ws;
  float *lse, *pos, *start;
  uint8_t* tag;
  int32_t *cu, *req;
  CHECK_CUDA(cudaMalloc(&q, elems * 2));
  CHECK_CUDA(cudaMalloc(&k, elems * 2));
  CHECK_CUDA(cudaMalloc(&v, elems * 2));
  CHECK_CUDA(cudaMalloc(&qr, elems * 2));
  CHECK_CUDA(cudaMalloc(&kr, elems * 2));
  CHECK_CUDA(cudaMalloc(&o, elems * 2));
  CHECK_CUDA(cudaMalloc((void**)&lse, (size_t)H * C * sizeof(float)));
  CHECK_CUDA(cudaMalloc((void**)&pos, (size_t)N * 3 * sizeof(float) + 4));
  CHECK_CUDA(cudaMalloc((void**)&tag, (size_t)N + 1));
  CHECK_CUDA(cudaMalloc((void**)&cu, (size_t)(S + 1) * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&req, (size_t)(R + 1) * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&start, (size_t)R * sizeof(float) + 4));
  CHECK_CUDA(cudaMemcpy(q, host_qkv, elems * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k, host_qkv + elems, elems * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v, host_qkv + 2 * elems, elems * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(pos, host_pos, (size_t)N * 3 * sizeof(float), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(tag, host_tag, (size_t)N, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(cu, host_cu, (size_t)(S + 1) * sizeof(int32_t), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(req, host_req, (size_t)(R + 1) * sizeof(int32_t), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(start, host_start, (size_t)R * sizeof(float), cudaMemcpyHostToDevice));
  /* rotated Q/K start as copies, so their pad rows [N, C) hold the inputs' bytes */
  CHECK_CUDA(cudaMemcpy(qr, q, elems * 2, cudaMemcpyDeviceToDevice));
  CHECK_CUDA(cudaMemcpy(kr, k, elems * 2, cudaMemcpyDeviceToDevice));

  uint16_t* host_o = malloc(elems * sizeof(uint16_t));
  float* host_lse = malloc((size_t)H * C * sizeof(float));
  if (!host_o || !host_lse) return 1;
  for (size_t i = 0; i < elems; ++i) host_o[i] = 0x4040; /* bf16 3.0 */
  for (size_t i = 0; i < (size_t)H * C; ++i) host_lse[i] = 5.0f;
  CHECK_CUDA(cudaMemcpy(o, host_o, elems * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(lse, host_lse, (size_t)H * C * sizeof(float), cudaMemcpyHostToDevice));

  const size_t ws_bytes = h3_varlen_attn_workspace_size(S, H, max_seqlen, D);
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes > 16 ? ws_bytes : 16));

  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));
  int32_t st[3];
  st[0] = (int32_t)h3_rope_apply(q, qr, k, kr, N, H, D, pos, tag, req, R, start, NULL,
                                 (h3_stream_t)stream);
  st[1] = (int32_t)h3_varlen_attn_fwd(qr, kr, v, o, lse, cu, S, max_seqlen, C, H, D, 0.0f, ws,
                                      ws_bytes, (h3_stream_t)stream);
  st[2] = (int32_t)h3_get_device_error((h3_stream_t)stream);
  CHECK_CUDA(cudaStreamSynchronize(stream));
  CHECK_CUDA(cudaMemcpy(host_o, o, elems * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(host_lse, lse, (size_t)H * C * sizeof(float), cudaMemcpyDeviceToHost));

  FILE* out = fopen(argv[2], "wb");
  if (!out) return 1;
  if (fwrite(st, sizeof(st), 1, out) != 1 || fwrite(host_o, 2, elems, out) != elems ||
      fwrite(host_lse, sizeof(float), (size_t)H * C, out) != (size_t)H * C)
    return 1;
  fclose(out);
  printf("statuses %d %d %d (%s)\n", st[0], st[1], st[2], h3_status_string((h3_status)st[1]));
  cudaStreamDestroy(stream);
  cudaFree(q); cudaFree(k); cudaFree(v); cudaFree(qr); cudaFree(kr); cudaFree(o); cudaFree(lse);
  cudaFree(pos); cudaFree(tag); cudaFree(cu); cudaFree(req); cudaFree(start); cudaFree(ws);
  free(host_qkv); free(host_pos); free(host_tag); free(host_cu); free(host_req); free(host_start);
  free(host_o); free(host_lse);
  return 0;
}
