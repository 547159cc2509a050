/* A plain C caller of the library's C ABI (no Python, no C++): reads a tiny problem from
 * a binary file, runs lp_forward on the GPU with cudaMalloc'd buffers and a caller-owned
 * workspace, and writes logp, LSE and entropy to a second binary file.
 *
 * Input file layout (little endian): int64 T, int64 H, int64 V, float tau,
 *   uint16 X[T*H] (bf16 bits), uint16 W[V*H], int32 y[T].
 * Output file: float logp[T], lse[T], entropy[T].
 * Exit status 0 on success; otherwise the lp_status or CUDA error is printed. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "lp.h"

static int fail(const char* what, int code) {
  fprintf(stderr, "%s failed: %d\n", what, code);
  return 1;
}

int main(int argc, char** argv) {
  if (argc != 3) return fail("usage: c_abi_forward <in> <out>", 2);
  FILE* f = fopen(argv[1], "rb");
  if (!f) return fail("open input", 2);
  int64_t T = 0, H = 0, V = 0;
  float tau = 0.f;
  if (fread(&T, 8, 1, f) != 1 || fread(&H, 8, 1, f) != 1 || fread(&V, 8, 1, f) != 1 || fread(&tau, 4, 1, f) != 1)
    return fail("read header", 2);
  if (T <= 0 || H <= 0 || V <= 0 || T > 4096 || H > 4096 || V > 65536) return fail("sizes", 2);
  uint16_t* X = (uint16_t*)malloc((size_t)(T * H) * 2);
  uint16_t* W = (uint16_t*)malloc((size_t)(V * H) * 2);
  int32_t* y = (int32_t*)malloc((size_t)T * 4);
  float* host_out = (float*)malloc((size_t)T * 12);
  if (!X || !W || !y || !host_out) return fail("malloc", 2);
  if (fread(X, 2, (size_t)(T * H), f) != (size_t)(T * H) || fread(W, 2, (size_t)(V * H), f) != (size_t)(V * H) ||
      fread(y, 4, (size_t)T, f) != (size_t)T)
    return fail("read arrays", 2);
  fclose(f);

  lp_shard_range shard = {0, V};
  lp_vocab_partition part = {V, V, 1, &shard};
  size_t ws_bytes = lp_workspace_size(LP_OP_FORWARD, T, H, &part);

  void *dX = NULL, *dW = NULL, *dy = NULL, *dout = NULL, *ws = NULL;
  cudaError_t e;
  if ((e = cudaMalloc(&dX, (size_t)(T * H) * 2)) != cudaSuccess) return fail("cudaMalloc", (int)e);
  if ((e = cudaMalloc(&dW, (size_t)(V * H) * 2)) != cudaSuccess) return fail("cudaMalloc", (int)e);
  if ((e = cudaMalloc(&dy, (size_t)T * 4)) != cudaSuccess) return fail("cudaMalloc", (int)e);
  if ((e = cudaMalloc(&dout, (size_t)T * 12)) != cudaSuccess) return fail("cudaMalloc", (int)e);
  if (ws_bytes > 0 && (e = cudaMalloc(&ws, ws_bytes)) != cudaSuccess) return fail("cudaMalloc", (int)e);
  cudaMemcpy(dX, X, (size_t)(T * H) * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dW, W, (size_t)(V * H) * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dy, y, (size_t)T * 4, cudaMemcpyHostToDevice);

  cudaStream_t stream;
  if ((e = cudaStreamCreate(&stream)) != cudaSuccess) return fail("cudaStreamCreate", (int)e);
  const void* Wk[1] = {dW};
  lp_outputs out = {(float*)dout, (float*)dout + T, (float*)dout + 2 * T, NULL};
  lp_status st = lp_forward(dX, T, H, Wk, NULL, &part, (const int32_t*)dy, tau, &out, ws, ws_bytes,
                            (lp_stream_t)stream);
  if (st != LP_OK) {
    fprintf(stderr, "lp_forward: %s\n", lp_status_string(st));
    return 1;
  }
  st = lp_get_device_error((lp_stream_t)stream);
  if (st != LP_OK) {
    fprintf(stderr, "device error: %s\n", lp_status_string(st));
    return 1;
  }
  if ((e = cudaMemcpy(host_out, dout, (size_t)T * 12, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail("cudaMemcpy", (int)e);

  FILE* o = fopen(argv[2], "wb");
  if (!o || fwrite(host_out, 4, (size_t)(3 * T), o) != (size_t)(3 * T)) return fail("write output", 2);
  fclose(o);
  cudaStreamDestroy(stream);
  cudaFree(dX);
  cudaFree(dW);
  cudaFree(dy);
  cudaFree(dout);
  cudaFree(ws);
  free(X);
  free(W);
  free(y);
  free(host_out);
  return 0;
}
