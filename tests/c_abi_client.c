/*
 * A plain C client of libserac_gb300.so (no Python, no torch): the C ABI of
 * include/serac.h used as a C program would use it.
 *
 *   c_abi_client A.u8 nA B.u8 nB out.bin
 *
 * reads nA x 128 and nB x 128 raw uint8 descriptors, matches them with match_pair
 * (device buffers from cudaMalloc, the default stream) and with match_pair_noalloc,
 * checks the argument-error path, runs the row top-3 (serac_topk_pair), and writes to
 * out.bin:
 *   int32 count, int32 matches[count][2], int32 row_top2[nA][4], int32 col_top2[nB][4],
 *   int32 top3_scores[nA][3], int32 top3_index[nA][3].
 * Exit status 0 on success; the caller compares out.bin with the oracle.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "serac.h"

#define CHECK_CUDA(x)                                                      \
  do {                                                                     \
    cudaError_t e_ = (x);                                                  \
    if (e_ != cudaSuccess) {                                               \
      fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));      \
      return 2;                                                            \
    }                                                                      \
  } while (0)

static uint8_t* read_file(const char* path, size_t bytes) {
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  uint8_t* p = (uint8_t*)malloc(bytes ? bytes : 1);
  if (p && bytes && fread(p, 1, bytes, f) != bytes) {
    free(p);
    p = NULL;
  }
  fclose(f);
  return p;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s A.u8 nA B.u8 nB out.bin\n", argv[0]);
    return 1;
  }
  const int32_t na = atoi(argv[2]), nb = atoi(argv[4]);
  uint8_t* ha = read_file(argv[1], (size_t)na * SERAC_DIM);
  uint8_t* hb = read_file(argv[3], (size_t)nb * SERAC_DIM);
  if (!ha || !hb) {
    fprintf(stderr, "cannot read the descriptor files\n");
    return 1;
  }
  if (serac_device_check() != SERAC_OK) {
    fprintf(stderr, "device check: %s\n", serac_status_str(serac_device_check()));
    return 3;
  }
  serac_params prm;
  if (serac_default_params(&prm, 0.8f, 0.7f) != SERAC_OK) return 4;

  uint8_t *da = NULL, *db = NULL;
  int32_t *matches = NULL, *count = NULL, *row_top2 = NULL, *col_top2 = NULL;
  void* ws = NULL;
  const size_t ws_bytes = serac_pair_workspace_size(na, nb);
  const int32_t cap = na > 0 ? na : 1;
  CHECK_CUDA(cudaMalloc((void**)&da, (size_t)(na ? na : 1) * SERAC_DIM));
  CHECK_CUDA(cudaMalloc((void**)&db, (size_t)(nb ? nb : 1) * SERAC_DIM));
  CHECK_CUDA(cudaMalloc((void**)&matches, (size_t)cap * 2 * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&count, sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&row_top2, (size_t)(na ? na : 1) * 4 * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&col_top2, (size_t)(nb ? nb : 1) * 4 * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemcpy(da, ha, (size_t)na * SERAC_DIM, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(db, hb, (size_t)nb * SERAC_DIM, cudaMemcpyHostToDevice));

  serac_out out;
  out.matches = matches;
  out.capacity = cap;
  out.count = count;
  out.row_top2 = row_top2;
  out.col_top2 = col_top2;

  /* argument errors are reported before anything is enqueued */
  if (match_pair(da, na, db, nb, NULL, &out, ws, ws_bytes, NULL) != SERAC_EINVAL) return 5;
  if (match_pair(da, na, db, nb, &prm, &out, ws, 16, NULL) != SERAC_EWORKSPACE) return 6;

  int st = match_pair(da, na, db, nb, &prm, &out, ws, ws_bytes, NULL);
  if (st != SERAC_OK) {
    fprintf(stderr, "match_pair: %s\n", serac_status_str(st));
    return 7;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  int32_t n = 0;
  CHECK_CUDA(cudaMemcpy(&n, count, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (n < 0 || n > cap) {
    fprintf(stderr, "count %d\n", n);
    return 8;
  }
  int32_t* hm = (int32_t*)malloc((size_t)(n ? n : 1) * 2 * sizeof(int32_t));
  int32_t* hr = (int32_t*)malloc((size_t)(na ? na : 1) * 4 * sizeof(int32_t));
  int32_t* hc = (int32_t*)malloc((size_t)(nb ? nb : 1) * 4 * sizeof(int32_t));
  CHECK_CUDA(cudaMemcpy(hm, matches, (size_t)n * 2 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hr, row_top2, (size_t)na * 4 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hc, col_top2, (size_t)nb * 4 * sizeof(int32_t), cudaMemcpyDeviceToHost));

  /* the same pair through the entry point that allocates nothing: identical list */
  CHECK_CUDA(cudaMemset(count, 0xFF, sizeof(int32_t)));
  out.row_top2 = NULL;
  out.col_top2 = NULL;
  st = match_pair_noalloc(da, na, db, nb, &prm, &out, NULL);
  if (st != SERAC_OK) {
    fprintf(stderr, "match_pair_noalloc: %s\n", serac_status_str(st));
    return 9;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  int32_t n2 = -1;
  CHECK_CUDA(cudaMemcpy(&n2, count, sizeof(int32_t), cudaMemcpyDeviceToHost));
  int32_t* hm2 = (int32_t*)malloc((size_t)(n2 > 0 ? n2 : 1) * 2 * sizeof(int32_t));
  if (n2 != n) return 10;
  CHECK_CUDA(cudaMemcpy(hm2, matches, (size_t)n * 2 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (n && memcmp(hm, hm2, (size_t)n * 2 * sizeof(int32_t)) != 0) return 11;

  /* the row top-3 of the same pair */
  int32_t *tks = NULL, *tki = NULL, *tst = NULL;
  void* tws = NULL;
  const size_t tws_bytes = serac_topk_workspace_size(na, nb, 3);
  if (tws_bytes == 0) return 13;
  CHECK_CUDA(cudaMalloc((void**)&tks, (size_t)(na ? na : 1) * 3 * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&tki, (size_t)(na ? na : 1) * 3 * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&tst, sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc(&tws, tws_bytes));
  if (serac_topk_pair(da, na, db, nb, 9, tks, tki, tst, tws, tws_bytes, NULL) != SERAC_EINVAL) return 14;
  st = serac_topk_pair(da, na, db, nb, 3, tks, tki, tst, tws, tws_bytes, NULL);
  if (st != SERAC_OK) {
    fprintf(stderr, "serac_topk_pair: %s\n", serac_status_str(st));
    return 15;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  int32_t tstatus = -99;
  CHECK_CUDA(cudaMemcpy(&tstatus, tst, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (tstatus != SERAC_OK) return 16;
  int32_t* hks = (int32_t*)malloc((size_t)(na ? na : 1) * 3 * sizeof(int32_t));
  int32_t* hki = (int32_t*)malloc((size_t)(na ? na : 1) * 3 * sizeof(int32_t));
  CHECK_CUDA(cudaMemcpy(hks, tks, (size_t)na * 3 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hki, tki, (size_t)na * 3 * sizeof(int32_t), cudaMemcpyDeviceToHost));

  FILE* f = fopen(argv[5], "wb");
  if (!f) return 12;
  fwrite(&n, sizeof(int32_t), 1, f);
  fwrite(hm, sizeof(int32_t), (size_t)n * 2, f);
  fwrite(hr, sizeof(int32_t), (size_t)na * 4, f);
  fwrite(hc, sizeof(int32_t), (size_t)nb * 4, f);
  fwrite(hks, sizeof(int32_t), (size_t)na * 3, f);
  fwrite(hki, sizeof(int32_t), (size_t)na * 3, f);
  fclose(f);
  printf("%d matches\n", n);
  cudaFree(da);
  cudaFree(db);
  cudaFree(matches);
  cudaFree(count);
  cudaFree(row_top2);
  cudaFree(col_top2);
  cudaFree(ws);
  cudaFree(tks);
  cudaFree(tki);
  cudaFree(tst);
  cudaFree(tws);
  free(hks);
  free(hki);
  free(ha);
  free(hb);
  free(hm);
  free(hm2);
  free(hr);
  free(hc);
  return 0;
}
