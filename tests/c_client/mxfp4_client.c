/*
 * mxfp4_client.c -- a plain C client of libmxfp4.so, with no Python or
 * PyTorch in the loop: it reads bf16 X [T, D] and W [F, D] from files,
 * quantizes both row-wise through mxfp4_quantize (tensor-core scale layout,
 * the parameters given on the command line), multiplies them with mxfp4_gemm
 * (the Fprop product C [T, F] = Xq Wq^T of "Pretraining large language models
 * with MXFP4", Abstract) and writes codes, scales and C to files for the test
 * that compares them with the oracle and with the Python binding's results.
 *
 * usage: mxfp4_client T D F x.bin w.bin out_prefix block scale_mode rounding
 *                     wht sign_mask seed
 * Writes out_prefix.{qx,sx,qw,sw,c}. Exit status 0 on success; otherwise the
 * failing call and the library's error detail go to stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "mxfp4.h"

static int read_file(const char* path, void* buf, size_t n) {
  FILE* f = fopen(path, "rb");
  if (!f) return -1;
  const size_t got = fread(buf, 1, n, f);
  fclose(f);
  return got == n ? 0 : -1;
}

static int write_file(const char* prefix, const char* ext, const void* buf, size_t n) {
  char path[4096];
  snprintf(path, sizeof(path), "%s.%s", prefix, ext);
  FILE* f = fopen(path, "wb");
  if (!f) return -1;
  const size_t put = fwrite(buf, 1, n, f);
  fclose(f);
  return put == n ? 0 : -1;
}

#define CUDA_OK(call)                                                              \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                  \
      return 2;                                                                    \
    }                                                                              \
  } while (0)

#define MX_OK(call)                                                                \
  do {                                                                             \
    mxfp4_status s_ = (call);                                                      \
    if (s_ != MXFP4_OK) {                                                          \
      fprintf(stderr, "%s: %s (%s)\n", #call, mxfp4_status_string(s_),             \
              mxfp4_last_error());                                                 \
      return 3;                                                                    \
    }                                                                              \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 13) {
    fprintf(stderr,
            "usage: %s T D F x.bin w.bin out_prefix block scale_mode rounding wht sign_mask seed\n",
            argv[0]);
    return 1;
  }
  const int64_t T = atoll(argv[1]), D = atoll(argv[2]), F = atoll(argv[3]);
  const char* prefix = argv[6];
  mxfp4_quant_params p = {0};
  p.block = atoi(argv[7]);
  p.scale_mode = atoi(argv[8]);
  p.rounding = atoi(argv[9]);
  p.scale_layout = MXFP4_LAYOUT_MMA;
  p.wht = atoi(argv[10]);
  p.wht_sign_mask = (uint32_t)strtoul(argv[11], NULL, 0);
  p.seed = strtoull(argv[12], NULL, 0);
  p.elem_format = MXFP4_FORMAT_E2M1;
  mxfp4_quant_params px = p, pw = p;
  px.sr_stream = 0;
  pw.sr_stream = 1;

  const size_t nx = (size_t)(T * D), nw = (size_t)(F * D), nc = (size_t)(T * F);
  const size_t qx_b = nx / 2, sx_b = nx / 32, qw_b = nw / 2, sw_b = nw / 32;
  uint16_t* hx = (uint16_t*)malloc(nx * 2);
  uint16_t* hw = (uint16_t*)malloc(nw * 2);
  uint8_t* hq = (uint8_t*)malloc(qx_b > qw_b ? qx_b : qw_b);
  float* hc = (float*)malloc(nc * 4);
  if (!hx || !hw || !hq || !hc) return 4;
  if (read_file(argv[4], hx, nx * 2) || read_file(argv[5], hw, nw * 2)) {
    fprintf(stderr, "cannot read the input files\n");
    return 1;
  }

  void *dx, *dw, *dc;
  uint8_t *qx, *sx, *qw, *sw;
  CUDA_OK(cudaMalloc(&dx, nx * 2));
  CUDA_OK(cudaMalloc(&dw, nw * 2));
  CUDA_OK(cudaMalloc(&dc, nc * 4));
  CUDA_OK(cudaMalloc((void**)&qx, qx_b));
  CUDA_OK(cudaMalloc((void**)&sx, sx_b));
  CUDA_OK(cudaMalloc((void**)&qw, qw_b));
  CUDA_OK(cudaMalloc((void**)&sw, sw_b));
  CUDA_OK(cudaMemcpy(dx, hx, nx * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dw, hw, nw * 2, cudaMemcpyHostToDevice));

  /* NULL stream: the calls are ordered on the context's default stream. */
  MX_OK(mxfp4_quantize(dx, MXFP4_DTYPE_BF16, T, D, D, &px, qx, sx, NULL, NULL, NULL, NULL));
  MX_OK(mxfp4_quantize(dw, MXFP4_DTYPE_BF16, F, D, D, &pw, qw, sw, NULL, NULL, NULL, NULL));
  MX_OK(mxfp4_gemm(qx, sx, qw, sw, T, F, D, (float*)dc, F, NULL));
  CUDA_OK(cudaDeviceSynchronize());
  MX_OK(mxfp4_device_status(NULL));

  int bad = 0;
  CUDA_OK(cudaMemcpy(hq, qx, qx_b, cudaMemcpyDeviceToHost));
  bad |= write_file(prefix, "qx", hq, qx_b);
  CUDA_OK(cudaMemcpy(hq, sx, sx_b, cudaMemcpyDeviceToHost));
  bad |= write_file(prefix, "sx", hq, sx_b);
  CUDA_OK(cudaMemcpy(hq, qw, qw_b, cudaMemcpyDeviceToHost));
  bad |= write_file(prefix, "qw", hq, qw_b);
  CUDA_OK(cudaMemcpy(hq, sw, sw_b, cudaMemcpyDeviceToHost));
  bad |= write_file(prefix, "sw", hq, sw_b);
  CUDA_OK(cudaMemcpy(hc, dc, nc * 4, cudaMemcpyDeviceToHost));
  bad |= write_file(prefix, "c", hc, nc * 4);
  if (bad) {
    fprintf(stderr, "cannot write the output files\n");
    return 1;
  }

  cudaFree(dx);
  cudaFree(dw);
  cudaFree(dc);
  cudaFree(qx);
  cudaFree(sx);
  cudaFree(qw);
  cudaFree(sw);
  free(hx);
  free(hw);
  free(hq);
  free(hc);
  return 0;
}
