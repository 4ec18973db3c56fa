/*
 * A plain C client of libmosaic.so: no Python, no torch. It allocates device memory with the
 * CUDA runtime, uploads integer-valued bf16 inputs, runs mask-only logits with lazy chunking
 * (a C callback copies each chunk out on the same stream) and checks every output element
 * against the exact integer dot product computed here: the inputs lie in {-2..2} and d is small,
 * so every partial sum is an integer below 2^24 and the fp32 output must be exact. It also
 * checks one argument error and the launch count. Exit status 0 = all checks passed.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mosaic.h"

#define CHECK_CUDA(x)                                                          \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                 \
      return 2;                                                                \
    }                                                                          \
  } while (0)

#define CHECK_MOSAIC(x)                                                        \
  do {                                                                         \
    mosaic_status s_ = (x);                                                    \
    if (s_ != MOSAIC_OK) {                                                     \
      fprintf(stderr, "%s: status %d: %s\n", #x, (int)s_, mosaic_last_error_string()); \
      return 3;                                                                \
    }                                                                          \
  } while (0)

/* bf16 bit pattern of a small integer (exact: the upper half of its fp32 encoding). */
static uint16_t bf16_of_int(int v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  return (uint16_t)(u >> 16);
}

static int h_val(int64_t r, int64_t k) { return (int)((r * 7 + k * 3) % 5) - 2; }
static int w_val(int64_t v, int64_t k) { return (int)((v * 5 + k * 11 + 1) % 5) - 2; }

struct sink {
  float* host;  /* [M, V] */
  int64_t V;
  cudaStream_t stream;
  int calls;
};

/* Runs after each chunk is enqueued: the copy is ordered after the chunk and before the next
   chunk overwrites the buffer, because it is enqueued on the same stream. */
static void on_chunk(int64_t chunk, int64_t row_begin, int64_t rows, void* out, void* user) {
  struct sink* s = (struct sink*)user;
  (void)chunk;
  cudaMemcpyAsync(s->host + row_begin * s->V, out, (size_t)(rows * s->V) * sizeof(float),
                  cudaMemcpyDeviceToHost, s->stream);
  s->calls++;
}

int main(void) {
  const int64_t L = 700, d = 192, V = 1040, M = 300, chunk_rows = 128;
  uint16_t* H = malloc((size_t)(L * d) * sizeof(uint16_t));
  uint16_t* W = malloc((size_t)(V * d) * sizeof(uint16_t));
  int32_t* idx = malloc((size_t)M * sizeof(int32_t));
  float* out_host = malloc((size_t)(M * V) * sizeof(float));
  if (!H || !W || !idx || !out_host) return 4;
  for (int64_t r = 0; r < L; ++r)
    for (int64_t k = 0; k < d; ++k) H[r * d + k] = bf16_of_int(h_val(r, k));
  for (int64_t v = 0; v < V; ++v)
    for (int64_t k = 0; k < d; ++k) W[v * d + k] = bf16_of_int(w_val(v, k));
  for (int64_t i = 0; i < M; ++i) idx[i] = (int32_t)((i * 37 + 11) % L); /* unsorted */
  idx[M - 1] = idx[0];                                                  /* a duplicate */

  void *dH, *dW, *dout;
  int32_t* didx;
  CHECK_CUDA(cudaSetDevice(0));
  CHECK_CUDA(cudaMalloc(&dH, (size_t)(L * d) * sizeof(uint16_t)));
  CHECK_CUDA(cudaMalloc(&dW, (size_t)(V * d) * sizeof(uint16_t)));
  CHECK_CUDA(cudaMalloc((void**)&didx, (size_t)M * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc(&dout, (size_t)(chunk_rows * V) * sizeof(float)));
  CHECK_CUDA(cudaMemcpy(dH, H, (size_t)(L * d) * sizeof(uint16_t), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dW, W, (size_t)(V * d) * sizeof(uint16_t), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(didx, idx, (size_t)M * sizeof(int32_t), cudaMemcpyHostToDevice));

  mosaic_handle* h = NULL;
  CHECK_MOSAIC(mosaic_create(&h, 0));
  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));
  struct sink s = {out_host, V, stream, 0};

  /* an argument error is reported before anything is enqueued */
  if (mosaic_masked_logits(h, dH, L, 7, didx, M, NULL, NULL, 0, dW, V, dout, MOSAIC_F32,
                           chunk_rows, on_chunk, &s, stream) != MOSAIC_ERR_UNSUPPORTED ||
      mosaic_last_error_string()[0] == '\0' || mosaic_launch_count(h) != 0 || s.calls != 0) {
    fprintf(stderr, "d = 7 was not rejected as unsupported\n");
    return 5;
  }

  CHECK_MOSAIC(mosaic_masked_logits(h, dH, L, d, didx, M, NULL, NULL, 0, dW, V, dout,
                                    MOSAIC_F32, chunk_rows, on_chunk, &s, stream));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  CHECK_MOSAIC(mosaic_check(h, stream));
  const int64_t chunks = (M + chunk_rows - 1) / chunk_rows;
  if (s.calls != chunks || mosaic_launch_count(h) != chunks) {
    fprintf(stderr, "expected %lld chunks, got %d callbacks and %lld launches\n",
            (long long)chunks, s.calls, (long long)mosaic_launch_count(h));
    return 6;
  }

  int64_t bad = 0;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t v = 0; v < V; ++v) {
      int64_t exact = 0;
      for (int64_t k = 0; k < d; ++k) exact += (int64_t)h_val(idx[i], k) * w_val(v, k);
      if (out_host[i * V + v] != (float)exact) {
        if (bad < 5)
          fprintf(stderr, "out[%lld, %lld] = %g, exact %lld\n", (long long)i, (long long)v,
                  out_host[i * V + v], (long long)exact);
        ++bad;
      }
    }
  CHECK_MOSAIC(mosaic_destroy(h));
  cudaStreamDestroy(stream);
  cudaFree(dH);
  cudaFree(dW);
  cudaFree(didx);
  cudaFree(dout);
  free(H);
  free(W);
  free(idx);
  free(out_host);
  if (bad) {
    fprintf(stderr, "%lld of %lld elements differ from the exact values\n", (long long)bad,
            (long long)(M * V));
    return 1;
  }
  printf("mosaic_client: %lld elements exact over %lld chunks\n", (long long)(M * V),
         (long long)chunks);
  return 0;
}
