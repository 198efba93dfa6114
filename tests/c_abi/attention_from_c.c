/*
 * The joint RoPE attention called from plain C through include/flux_attn.h,
 * with no Python and no torch: device buffers from cudaMalloc, the one-call
 * entry point, its status word read back with flux_query_status.
 *
 * Usage: attention_from_c <dir> B S_txt S_img H
 * Reads <dir>/q.bin, k.bin, v.bin (bf16 [B, S, H, 128] raw), txt_ids.bin and
 * img_ids.bin (int32 [S_txt, 4] and [S_img, 4]); writes <dir>/out.bin (bf16
 * [B, S, H, 128]). Exit status 0 on success; on any failure a message on
 * stderr and a non-zero status.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "flux_attn.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (f == NULL) return NULL;
  void *buf = malloc(bytes > 0 ? bytes : 1);
  const size_t got = buf != NULL ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int check_cuda(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return 0;
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 1;
}

int main(int argc, char **argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s dir B S_txt S_img H\n", argv[0]);
    return 2;
  }
  const char *dir = argv[1];
  const int B = atoi(argv[2]), H = atoi(argv[5]), D = 128;
  const int64_t S_txt = atoll(argv[3]), S_img = atoll(argv[4]), S = S_txt + S_img;
  const size_t tensor = (size_t)B * (size_t)S * (size_t)H * D * 2;
  const size_t txt_bytes = (size_t)S_txt * 4 * sizeof(int32_t);
  const size_t img_bytes = (size_t)S_img * 4 * sizeof(int32_t);
  void *hq = read_file(dir, "q.bin", tensor), *hk = read_file(dir, "k.bin", tensor);
  void *hv = read_file(dir, "v.bin", tensor);
  void *htxt = read_file(dir, "txt_ids.bin", txt_bytes);
  void *himg = read_file(dir, "img_ids.bin", img_bytes);
  if (hq == NULL || hk == NULL || hv == NULL || htxt == NULL || himg == NULL) {
    fprintf(stderr, "cannot read the inputs in %s\n", dir);
    return 3;
  }
  const int32_t axes[4] = {32, 32, 32, 32};
  const size_t ws_bytes = flux_joint_rope_attention_workspace_shared(B, S, H, D);
  void *q = NULL, *k = NULL, *v = NULL, *out = NULL, *ws = NULL, *txt = NULL, *img = NULL;
  cudaStream_t stream = NULL;
  int rc = 0;
  rc |= check_cuda(cudaStreamCreate(&stream), "cudaStreamCreate");
  rc |= check_cuda(cudaMalloc(&q, tensor), "cudaMalloc q");
  rc |= check_cuda(cudaMalloc(&k, tensor), "cudaMalloc k");
  rc |= check_cuda(cudaMalloc(&v, tensor), "cudaMalloc v");
  rc |= check_cuda(cudaMalloc(&out, tensor), "cudaMalloc out");
  rc |= check_cuda(cudaMalloc(&ws, ws_bytes), "cudaMalloc workspace");
  rc |= check_cuda(cudaMalloc(&txt, txt_bytes > 0 ? txt_bytes : 16), "cudaMalloc txt");
  rc |= check_cuda(cudaMalloc(&img, img_bytes > 0 ? img_bytes : 16), "cudaMalloc img");
  if (rc) return 4;
  rc |= check_cuda(cudaMemcpy(q, hq, tensor, cudaMemcpyHostToDevice), "copy q");
  rc |= check_cuda(cudaMemcpy(k, hk, tensor, cudaMemcpyHostToDevice), "copy k");
  rc |= check_cuda(cudaMemcpy(v, hv, tensor, cudaMemcpyHostToDevice), "copy v");
  if (txt_bytes > 0) rc |= check_cuda(cudaMemcpy(txt, htxt, txt_bytes, cudaMemcpyHostToDevice), "copy txt");
  if (img_bytes > 0) rc |= check_cuda(cudaMemcpy(img, himg, img_bytes, cudaMemcpyHostToDevice), "copy img");
  if (rc) return 5;

  int st = flux_joint_rope_attention(q, k, v, txt, S_txt, img, S_img, B, H, D, axes, 4, 2000.0,
                                     out, ws, ws_bytes, (void *)stream);
  if (st != FLUX_OK) {
    fprintf(stderr, "flux_joint_rope_attention: %s\n", flux_status_string(st));
    return 6;
  }
  st = flux_query_status(ws, (void *)stream);
  if (st != FLUX_OK) {
    fprintf(stderr, "device status: %s\n", flux_status_string(st));
    return 7;
  }
  /* a bad argument is refused on the host with its documented status */
  if (flux_joint_rope_attention(q, k, v, txt, S_txt, img, S_img, B, H, 64, axes, 4, 2000.0, out,
                                ws, ws_bytes, (void *)stream) != FLUX_ERR_SHAPE) {
    fprintf(stderr, "D = 64 was not refused with FLUX_ERR_SHAPE\n");
    return 8;
  }
  void *hout = malloc(tensor);
  if (hout == NULL || check_cuda(cudaMemcpy(hout, out, tensor, cudaMemcpyDeviceToHost), "copy out"))
    return 9;
  char path[4096];
  snprintf(path, sizeof path, "%s/out.bin", dir);
  FILE *f = fopen(path, "wb");
  if (f == NULL || fwrite(hout, 1, tensor, f) != tensor) {
    fprintf(stderr, "cannot write %s\n", path);
    return 10;
  }
  fclose(f);
  cudaFree(q);
  cudaFree(k);
  cudaFree(v);
  cudaFree(out);
  cudaFree(ws);
  cudaFree(txt);
  cudaFree(img);
  cudaStreamDestroy(stream);
  free(hq);
  free(hk);
  free(hv);
  free(htxt);
  free(himg);
  free(hout);
  return 0;
}
