/*
 * A plain C client of libmosaic.so: no Python, no torch. It allocates device memory with the
 * CUDA runtime, uploads integer-valued bf16 inputs, runs mask-only logits with lazy chunking
 * (a C callback copies each chunk out on the same stream) and checks every output element
 * against the exact integer dot product computed here: the inputs lie in {-2..2} and d is small,
 * so every partial sum is an integer below 2^24 and the fp32 output must be exact. It also
 * checks one argument error and the launch count. Then, on a CSR batch with an empty sequence
 * and M = 300 rows (the CTA-pair kernel): bf16 logits (each element the round-to-nearest-even
 * bf16 of the exact integer), fused greedy sampling (the token is the first maximal column of
 * the exact integer logits, the confidence 1 / sum exp(l - max) within 1e-4), the same logits
 * through the allocation-free entry point in chunks (bit for bit, per-chunk status words 0), and
 * the minimum-chunk helper. Exit status 0 = all checks passed.
 */
#include <cuda_runtime_api.h>
#include <math.h>
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

/* Round-to-nearest-even bf16 of a finite float (ties to the even upper half). */
static uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  u += 0x7FFFu + ((u >> 16) & 1u);
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

/* bf16 chunks into a host [M, V] array of bit patterns. */
struct sink16 {
  uint16_t* host;
  int64_t V;
  cudaStream_t stream;
  int calls;
};

static void on_chunk16(int64_t chunk, int64_t row_begin, int64_t rows, void* out, void* user) {
  struct sink16* s = (struct sink16*)user;
  (void)chunk;
  cudaMemcpyAsync(s->host + row_begin * s->V, out, (size_t)(rows * s->V) * sizeof(uint16_t),
                  cudaMemcpyDeviceToHost, s->stream);
  s->calls++;
}

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
  if (bad) {
    fprintf(stderr, "%lld of %lld elements differ from the exact values\n", (long long)bad,
            (long long)(M * V));
    return 1;
  }
  printf("mosaic_client: %lld elements exact over %lld chunks\n", (long long)(M * V),
         (long long)chunks);

  /* ---- CSR batch (sequence 1 empty), M = 300 rows: the CTA-pair kernel, bf16 logits */
  const int32_t B = 3;
  const int32_t seq_off[4] = {0, 250, 250, 700};   /* rows of hidden per sequence */
  const int32_t mask_off[4] = {0, 180, 180, 300};  /* masked positions per sequence */
  int32_t* lidx = malloc((size_t)M * sizeof(int32_t));
  int64_t* grow = malloc((size_t)M * sizeof(int64_t));
  uint16_t* out16 = malloc((size_t)(M * V) * sizeof(uint16_t));
  uint16_t* out16b = malloc((size_t)(M * V) * sizeof(uint16_t));
  int32_t* tok = malloc((size_t)M * sizeof(int32_t));
  float* conf = malloc((size_t)M * sizeof(float));
  int64_t* exact = malloc((size_t)(M * V) * sizeof(int64_t));
  if (!lidx || !grow || !out16 || !out16b || !tok || !conf || !exact) return 4;
  for (int32_t b = 0; b < B; ++b)
    for (int32_t i = mask_off[b]; i < mask_off[b + 1]; ++i) {
      const int32_t len = seq_off[b + 1] - seq_off[b];
      lidx[i] = (int32_t)((i * 53 + 7) % len); /* local to its sequence, unsorted */
      grow[i] = seq_off[b] + lidx[i];
    }
  for (int64_t i = 0; i < M; ++i)
    for (int64_t v = 0; v < V; ++v) {
      int64_t e = 0;
      for (int64_t k = 0; k < d; ++k) e += (int64_t)h_val(grow[i], k) * w_val(v, k);
      exact[i * V + v] = e;
    }
  int32_t *dlidx, *dso, *dmo, *dtok;
  float* dconf;
  void *dout16, *dws;
  CHECK_CUDA(cudaMalloc((void**)&dlidx, (size_t)M * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&dso, sizeof(seq_off)));
  CHECK_CUDA(cudaMalloc((void**)&dmo, sizeof(mask_off)));
  CHECK_CUDA(cudaMalloc(&dout16, (size_t)(M * V) * sizeof(uint16_t)));
  CHECK_CUDA(cudaMalloc((void**)&dtok, (size_t)M * sizeof(int32_t)));
  CHECK_CUDA(cudaMalloc((void**)&dconf, (size_t)M * sizeof(float)));
  CHECK_CUDA(cudaMemcpy(dlidx, lidx, (size_t)M * sizeof(int32_t), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dso, seq_off, sizeof(seq_off), cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dmo, mask_off, sizeof(mask_off), cudaMemcpyHostToDevice));

  CHECK_MOSAIC(mosaic_masked_logits(h, dH, L, d, dlidx, M, dso, dmo, B, dW, V, dout16,
                                    MOSAIC_BF16, 0, NULL, NULL, stream));
  CHECK_MOSAIC(mosaic_check(h, stream));
  CHECK_CUDA(cudaMemcpy(out16, dout16, (size_t)(M * V) * sizeof(uint16_t),
                        cudaMemcpyDeviceToHost));
  for (int64_t e = 0; e < M * V; ++e)
    if (out16[e] != bf16_rne((float)exact[e])) {
      fprintf(stderr, "CSR bf16 out[%lld] = 0x%04x, expected 0x%04x\n", (long long)e, out16[e],
              bf16_rne((float)exact[e]));
      return 7;
    }
  printf("csr bf16: %lld elements exact\n", (long long)(M * V));

  /* ---- fused greedy sampling on the same batch */
  const int64_t ws_bytes = mosaic_masked_sample_workspace_bytes(M, V, 0);
  if (ws_bytes <= 0) return 8;
  CHECK_CUDA(cudaMalloc(&dws, (size_t)ws_bytes));
  CHECK_MOSAIC(mosaic_masked_sample(h, dH, L, d, dlidx, M, dso, dmo, B, dW, V, dtok, dconf, dws,
                                    ws_bytes, 0, stream));
  CHECK_MOSAIC(mosaic_check(h, stream));
  CHECK_CUDA(cudaMemcpy(tok, dtok, (size_t)M * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(conf, dconf, (size_t)M * sizeof(float), cudaMemcpyDeviceToHost));
  for (int64_t i = 0; i < M; ++i) {
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (exact[i * V + v] > exact[i * V + best]) best = v;
    double sum = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      sum += exp((double)(exact[i * V + v] - exact[i * V + best]));
    }
    const double c = 1.0 / sum;
    if (tok[i] != (int32_t)best || conf[i] < c * (1.0 - 1e-4) || conf[i] > c * (1.0 + 1e-4)) {
      fprintf(stderr, "sample row %lld: token %d confidence %.7g, expected %lld %.7g\n",
              (long long)i, tok[i], conf[i], (long long)best, c);
      return 9;
    }
  }
  printf("sampling: %lld tokens exact\n", (long long)M);

  /* ---- the allocation-free entry point, chunked, on the same batch */
  uint32_t cstat[3] = {7u, 7u, 7u};
  struct sink16 s16 = {out16b, V, stream, 0};
  CHECK_MOSAIC(mosaic_masked_logits_noalloc(dH, L, d, dlidx, M, dso, dmo, B, dW, V, dout16,
                                            MOSAIC_BF16, chunk_rows, on_chunk16, &s16, cstat,
                                            stream));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  if (s16.calls != 3 || cstat[0] || cstat[1] || cstat[2] ||
      memcmp(out16, out16b, (size_t)(M * V) * sizeof(uint16_t)) != 0) {
    fprintf(stderr, "noalloc: %d chunks, status %u %u %u, or results differ\n", s16.calls,
            cstat[0], cstat[1], cstat[2]);
    return 10;
  }
  printf("noalloc: bit for bit over 3 chunks\n");

  /* ---- minimum sufficient chunk count for a 100-row bf16 budget */
  int64_t cr = -1, nc = -1;
  CHECK_MOSAIC(mosaic_min_chunk_rows(M, V, MOSAIC_BF16, 100 * V * 2, &cr, &nc));
  if (cr != 100 || nc != 3) {
    fprintf(stderr, "min_chunk_rows: %lld rows x %lld chunks, expected 100 x 3\n",
            (long long)cr, (long long)nc);
    return 11;
  }
  printf("min_chunk_rows: 100 x 3\n");

  CHECK_MOSAIC(mosaic_destroy(h));
  cudaStreamDestroy(stream);
  cudaFree(dH);
  cudaFree(dW);
  cudaFree(didx);
  cudaFree(dout);
  cudaFree(dlidx);
  cudaFree(dso);
  cudaFree(dmo);
  cudaFree(dout16);
  cudaFree(dtok);
  cudaFree(dconf);
  cudaFree(dws);
  free(H);
  free(W);
  free(idx);
  free(out_host);
  free(lidx);
  free(grow);
  free(out16);
  free(out16b);
  free(tok);
  free(conf);
  free(exact);
  return 0;
}
