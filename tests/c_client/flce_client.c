/* A plain C11 client of the FLCE C ABI (include/flce.h), with no PyTorch:
 *
 *   flce_client plan N H V chunk budget_bytes dlogits_mode cta
 *       prints the plan fields flce_make_plan returns (host only);
 *   flce_client run DIR N H V chunk dlogits_mode
 *       reads DIR/x.bin (N x H bf16), DIR/W.bin (V x H bf16) and DIR/t.bin
 *       (N int64), runs flce_forward_backward on cuda:0 with buffers from
 *       cudaMalloc, and writes DIR/dx.bin (N x H bf16), DIR/dW.bin (V x H
 *       fp32) and the loss on stdout.
 *
 * Exit status 0 on success; any library or CUDA error is printed. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "flce.h"

static int read_file(const char* dir, const char* name, void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return 1;
  const size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  return got != bytes;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

#define CUDA_OK(expr)                                                        \
  do {                                                                       \
    cudaError_t e_ = (expr);                                                 \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s: %s\n", #expr, cudaGetErrorString(e_));           \
      return 2;                                                              \
    }                                                                        \
  } while (0)

static int plan(int argc, char** argv) {
  if (argc != 9) return 64;
  flce_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.dtype = FLCE_DTYPE_BF16;
  cfg.hbm_budget_bytes = strtoull(argv[6], NULL, 10);
  cfg.dlogits_mode = atoi(argv[7]);
  cfg.cta_pair = atoi(argv[8]);
  flce_plan p;
  const flce_status st = flce_make_plan(&cfg, atoll(argv[2]), atoll(argv[3]), atoll(argv[4]),
                                        atoll(argv[5]), 0, &p);
  if (st != FLCE_OK) {
    printf("status %s\n", flce_status_string(st));
    return 1;
  }
  printf("chunk %lld num_chunks %lld vocab_tiles %lld ldv %lld dx_splits %lld workspace_bytes %llu "
         "logits_bytes %llu tile_m %lld tile_n %lld vocab_slab %lld dlogits_mode %lld tile_n_dx %lld "
         "tile_n_dw %lld dw_beside_dx %lld backward_one_launch %lld\n",
         (long long)p.chunk, (long long)p.num_chunks, (long long)p.vocab_tiles, (long long)p.ldv,
         (long long)p.dx_splits, (unsigned long long)p.workspace_bytes,
         (unsigned long long)p.logits_bytes, (long long)p.tile_m, (long long)p.tile_n,
         (long long)p.vocab_slab, (long long)p.dlogits_mode, (long long)p.tile_n_dx,
         (long long)p.tile_n_dw, (long long)p.dw_beside_dx, (long long)p.backward_one_launch);
  return 0;
}

static int run(int argc, char** argv) {
  if (argc != 8) return 64;
  const char* dir = argv[2];
  const int64_t N = atoll(argv[3]), H = atoll(argv[4]), V = atoll(argv[5]), chunk = atoll(argv[6]);
  const size_t xb = (size_t)N * H * 2, wb = (size_t)V * H * 2, tb = (size_t)N * 8;
  const size_t dwb = (size_t)V * H * 4;
  void* xh = malloc(xb);
  void* wh = malloc(wb);
  void* th = malloc(tb);
  void* dxh = malloc(xb);
  void* dwh = malloc(dwb);
  if (!xh || !wh || !th || !dxh || !dwh) return 3;
  if (read_file(dir, "x.bin", xh, xb) || read_file(dir, "W.bin", wh, wb) ||
      read_file(dir, "t.bin", th, tb)) {
    fprintf(stderr, "cannot read the inputs in %s\n", dir);
    return 4;
  }
  void *x, *W, *t, *dx;
  float* dW;
  CUDA_OK(cudaMalloc(&x, xb));
  CUDA_OK(cudaMalloc(&W, wb));
  CUDA_OK(cudaMalloc(&t, tb));
  CUDA_OK(cudaMalloc(&dx, xb));
  CUDA_OK(cudaMalloc((void**)&dW, dwb));
  CUDA_OK(cudaMemcpy(x, xh, xb, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(W, wh, wb, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(t, th, tb, cudaMemcpyHostToDevice));

  flce_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.dtype = FLCE_DTYPE_BF16;
  cfg.dlogits_mode = atoi(argv[7]);
  flce_handle_t h = NULL;
  flce_status st = flce_create(&h, &cfg);
  if (st != FLCE_OK) {
    fprintf(stderr, "flce_create: %s\n", flce_status_string(st));
    return 5;
  }
  float loss = 0.f;
  st = flce_forward_backward(h, x, W, (const int64_t*)t, N, H, V, -100, chunk, &loss, dx, dW, NULL);
  if (st != FLCE_OK) {
    fprintf(stderr, "flce_forward_backward: %s: %s\n", flce_status_string(st), flce_last_error(h));
    flce_destroy(h);
    return 6;
  }
  flce_destroy(h);
  CUDA_OK(cudaMemcpy(dxh, dx, xb, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(dwh, dW, dwb, cudaMemcpyDeviceToHost));
  if (write_file(dir, "dx.bin", dxh, xb) || write_file(dir, "dW.bin", dwh, dwb)) return 7;
  printf("loss %.9g\n", (double)loss);
  cudaFree(x);
  cudaFree(W);
  cudaFree(t);
  cudaFree(dx);
  cudaFree(dW);
  free(xh);
  free(wh);
  free(th);
  free(dxh);
  free(dwh);
  return 0;
}

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "plan") == 0) return plan(argc, argv);
  if (argc >= 2 && strcmp(argv[1], "run") == 0) return run(argc, argv);
  fprintf(stderr, "usage: flce_client plan N H V chunk budget mode cta | run DIR N H V chunk mode\n");
  return 64;
}
