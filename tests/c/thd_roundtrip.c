/*
 * The C ABI from plain C11: no Python, no torch.  Builds both routes of the
 * tiny workload (cp=2, documents [8, 12, 4]), swaps zigzag -> contiguous and
 * back, and checks against zigzag positions derived by hand from the
 * partition rule ("Packed Sequence 与上下文并行", section 2.4): rank 0 holds
 * chunks 0 and 3 of every document, rank 1 chunks 1 and 2.
 * Exit status 0 and "ok" on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "thd.h"

#define CHECK_CUDA(x)                                                  \
  do {                                                                 \
    cudaError_t e_ = (x);                                              \
    if (e_ != cudaSuccess) {                                           \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));         \
      return 2;                                                        \
    }                                                                  \
  } while (0)
#define CHECK_THD(x)                                                   \
  do {                                                                 \
    thd_status_t s_ = (x);                                             \
    if (s_ != THD_OK) {                                                \
      fprintf(stderr, "%s: %s\n", #x, thd_status_string(s_));          \
      return 3;                                                        \
    }                                                                  \
  } while (0)

enum { T = 24, CP = 2, S = T / CP, ROW = 32 };

/* global rows held by each zigzag slot: rank 0 then rank 1 */
static const int32_t zz[T] = {0, 1, 6, 7, 8, 9, 10, 17, 18, 19, 20, 23,
                              2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 21, 22};

int main(void) {
  const int32_t cu_h[4] = {0, 8, 20, 24};
  int32_t *cu = NULL, *status = NULL, *idx = NULL;
  unsigned char *x = NULL, *y = NULL, *z = NULL, *blob_f = NULL, *blob_b = NULL;
  unsigned char host_x[T * ROW], host_y[T * ROW], host_z[T * ROW];
  int32_t idx_h[T];
  thd_route_t fwd, bwd;
  int32_t code = -1;
  size_t rb = thd_route_bytes(T, CP);

  CHECK_CUDA(cudaMalloc((void **)&cu, sizeof cu_h));
  CHECK_CUDA(cudaMalloc((void **)&status, sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void **)&idx, sizeof idx_h));
  CHECK_CUDA(cudaMalloc((void **)&x, sizeof host_x));
  CHECK_CUDA(cudaMalloc((void **)&y, sizeof host_y));
  CHECK_CUDA(cudaMalloc((void **)&z, sizeof host_z));
  CHECK_CUDA(cudaMalloc((void **)&blob_f, rb));
  CHECK_CUDA(cudaMalloc((void **)&blob_b, rb));
  CHECK_CUDA(cudaMemcpy(cu, cu_h, sizeof cu_h, cudaMemcpyHostToDevice));
  /* row p of the zigzag buffer: every byte = p */
  for (int p = 0; p < T; ++p) memset(host_x + p * ROW, p, ROW);
  CHECK_CUDA(cudaMemcpy(x, host_x, sizeof host_x, cudaMemcpyHostToDevice));

  CHECK_THD(thd_status_clear(status, 0));
  CHECK_THD(thd_route_bind(&fwd, blob_f, rb, T, CP, THD_ZIGZAG_TO_CONTIGUOUS));
  CHECK_THD(thd_route_bind(&bwd, blob_b, rb, T, CP, THD_CONTIGUOUS_TO_ZIGZAG));
  CHECK_THD(thd_route_build_pair(cu, 3, T, CP, &fwd, &bwd, status, 0));
  CHECK_THD(thd_partition_indices(cu, 3, T, CP, -1, idx, status, 0));
  CHECK_THD(thd_swap(x, y, ROW, &fwd, status, 0));
  CHECK_THD(thd_swap(y, z, ROW, &bwd, status, 0));
  CHECK_THD(thd_status_read(status, &code, 0));
  if (code != THD_OK) {
    fprintf(stderr, "device status %d\n", code);
    return 4;
  }
  CHECK_CUDA(cudaMemcpy(idx_h, idx, sizeof idx_h, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(host_y, y, sizeof host_y, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(host_z, z, sizeof host_z, cudaMemcpyDeviceToHost));

  for (int p = 0; p < T; ++p)
    if (idx_h[p] != zz[p]) {
      fprintf(stderr, "partition slot %d: %d, want %d\n", p, idx_h[p], zz[p]);
      return 5;
    }
  /* after z->c, global row zz[p] holds the bytes of zigzag position p */
  for (int p = 0; p < T; ++p)
    for (int b = 0; b < ROW; ++b)
      if (host_y[zz[p] * ROW + b] != (unsigned char)p) {
        fprintf(stderr, "contiguous row %d byte %d: %d, want %d\n", zz[p], b, host_y[zz[p] * ROW + b], p);
        return 6;
      }
  if (memcmp(host_z, host_x, sizeof host_x) != 0) {
    fprintf(stderr, "round trip differs\n");
    return 7;
  }
  /* a bad direction is refused on the host */
  if (thd_route_build(cu, 3, T, CP, (thd_dir_t)7, &fwd, status, 0) != THD_ERR_BAD_DIRECTION) return 8;

  cudaFree(cu); cudaFree(status); cudaFree(idx); cudaFree(x); cudaFree(y); cudaFree(z);
  cudaFree(blob_f); cudaFree(blob_b);
  printf("ok\n");
  return 0;
}
