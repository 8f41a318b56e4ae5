// A forward pass driven from host code through the C ABI alone: raw device
// buffers from the CUDA runtime, attn_fwd on the default stream, results
// written to files for the test to compare with the oracle.
//   usage: fwd_from_c <out_dir>
// Inputs: bf16 q/k/v [1, 200, 2, 64] from a 64-bit linear congruential
// generator (values in [-1, 1)), causal, scale 1/8.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "attn.h"

static uint16_t to_bf16(float f) {  // round to nearest even
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int write_file(const char* dir, const char* name, const void* p, size_t n) {
  char path[1024];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t w = fwrite(p, 1, n, f);
  fclose(f);
  return w == n ? 0 : 1;
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  const int B = 1, L = 200, H = 2, d = 64;
  const size_t n = (size_t)B * L * H * d;
  uint16_t* h[3];
  uint64_t s = 12345u;
  for (int t = 0; t < 3; ++t) {
    h[t] = (uint16_t*)malloc(n * 2);
    for (size_t i = 0; i < n; ++i) {
      s = s * 6364136223846793005ull + 1442695040888963407ull;
      h[t][i] = to_bf16((float)((double)(s >> 11) / 9007199254740992.0 * 2.0 - 1.0));
    }
  }
  void *q, *k, *v, *o;
  float* lse;
  if (cudaMalloc(&q, n * 2) || cudaMalloc(&k, n * 2) || cudaMalloc(&v, n * 2) || cudaMalloc(&o, n * 2) ||
      cudaMalloc((void**)&lse, (size_t)B * H * L * 4))
    return 3;
  cudaMemcpy(q, h[0], n * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(k, h[1], n * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(v, h[2], n * 2, cudaMemcpyHostToDevice);
  const attn_status st = attn_fwd(q, k, v, o, lse, B, L, L, H, H, d, 0.125f, 1, NULL, ATTN_BF16, NULL);
  if (st != ATTN_OK) {
    printf("attn_fwd: %s %s\n", attn_status_string(st), attn_last_error());
    return 4;
  }
  uint16_t* ho = (uint16_t*)malloc(n * 2);
  float* hl = (float*)malloc((size_t)B * H * L * 4);
  if (cudaMemcpy(ho, o, n * 2, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(hl, lse, (size_t)B * H * L * 4, cudaMemcpyDeviceToHost))
    return 5;
  if (write_file(argv[1], "q.bin", h[0], n * 2) || write_file(argv[1], "k.bin", h[1], n * 2) ||
      write_file(argv[1], "v.bin", h[2], n * 2) || write_file(argv[1], "o.bin", ho, n * 2) ||
      write_file(argv[1], "lse.bin", hl, (size_t)B * H * L * 4))
    return 6;
  printf("OK\n");
  return 0;
}
