/*
 * The C ABI from plain C11: no Python, no torch.  Builds both routes of the
 * tiny workload (cp=2, documents [8, 12, 4]), swaps zigzag -> contiguous and
 * back, and checks against zigzag positions derived by hand from the
 * partition rule ("Packed Sequence 与上下文并行", section 2.4): rank 0 holds
 * chunks 0 and 3 of every document, rank 1 chunks 1 and 2.  Then the same
 * conversion through both routes bound into one shared buffer, as a batched
 * swap of two [T][ROW] blocks, and as every rank's pack -> exchange ->
 * scatter on its own shard (the exchange done here by copies, with the split
 * sizes and offsets read back from the route).
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

  /* both routes in one shared buffer; two [T][ROW] blocks in one batched swap */
  {
    thd_route_t pf, pb;
    unsigned char *blob = NULL, *x2 = NULL, *y2 = NULL, *send = NULL, *recv = NULL, *w = NULL;
    unsigned char host_y2[2 * T * ROW], host_w[T * ROW];
    int32_t in_split[CP * CP], send_off[CP * (CP + 1)], recv_off[CP * (CP + 1)];
    size_t pbytes = thd_route_pair_bytes(T, CP);
    CHECK_CUDA(cudaMalloc((void **)&blob, pbytes));
    CHECK_CUDA(cudaMalloc((void **)&x2, 2 * sizeof host_x));
    CHECK_CUDA(cudaMalloc((void **)&y2, 2 * sizeof host_x));
    CHECK_CUDA(cudaMalloc((void **)&send, sizeof host_x));
    CHECK_CUDA(cudaMalloc((void **)&recv, sizeof host_x));
    CHECK_CUDA(cudaMalloc((void **)&w, sizeof host_x));
    CHECK_THD(thd_route_bind_pair(&pf, &pb, blob, pbytes, T, CP));
    if (pf.recv_rows != pb.send_rows || pf.send_rows != pb.recv_rows) return 9;
    CHECK_THD(thd_route_build_pair(cu, 3, T, CP, &pf, &pb, status, 0));
    CHECK_CUDA(cudaMemcpy(x2, x, sizeof host_x, cudaMemcpyDeviceToDevice));
    CHECK_CUDA(cudaMemcpy(x2 + sizeof host_x, x, sizeof host_x, cudaMemcpyDeviceToDevice));
    CHECK_THD(thd_swap_batched(x2, y2, 2, ROW, &pf, status, 0));
    /* every rank packs its own shard, the blocks go to their ranks, every rank scatters */
    for (int r = 0; r < CP; ++r) CHECK_THD(thd_pack_rank(x + r * S * ROW, send + r * S * ROW, r, ROW, &pf, status, 0));
    CHECK_CUDA(cudaMemcpy(in_split, pf.input_split_sizes, sizeof in_split, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(send_off, pf.send_offsets, sizeof send_off, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(recv_off, pf.recv_offsets, sizeof recv_off, cudaMemcpyDeviceToHost));
    for (int s = 0; s < CP; ++s)
      for (int d = 0; d < CP; ++d)
        CHECK_CUDA(cudaMemcpy(recv + (d * S + recv_off[d * (CP + 1) + s]) * ROW,
                              send + (s * S + send_off[s * (CP + 1) + d]) * ROW,
                              (size_t)in_split[s * CP + d] * ROW, cudaMemcpyDeviceToDevice));
    for (int r = 0; r < CP; ++r)
      CHECK_THD(thd_scatter_rank(recv + r * S * ROW, w + r * S * ROW, r, ROW, &pf, status, 0));
    CHECK_THD(thd_status_read(status, &code, 0));
    if (code != THD_OK) {
      fprintf(stderr, "device status %d\n", code);
      return 10;
    }
    CHECK_CUDA(cudaMemcpy(host_y2, y2, sizeof host_y2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(host_w, w, sizeof host_w, cudaMemcpyDeviceToHost));
    if (memcmp(host_y2, host_y, sizeof host_y) != 0 || memcmp(host_y2 + sizeof host_y, host_y, sizeof host_y) != 0) {
      fprintf(stderr, "batched swap differs from the swap\n");
      return 11;
    }
    if (memcmp(host_w, host_y, sizeof host_y) != 0) {
      fprintf(stderr, "per-rank pack / exchange / scatter differs from the swap\n");
      return 12;
    }
    cudaFree(blob); cudaFree(x2); cudaFree(y2); cudaFree(send); cudaFree(recv); cudaFree(w);
  }

  cudaFree(cu); cudaFree(status); cudaFree(idx); cudaFree(x); cudaFree(y); cudaFree(z);
  cudaFree(blob_f); cudaFree(blob_b);
  printf("ok\n");
  return 0;
}
